"""ctypes binding of libpagedattn.so: argument marshalling only.

Every function checks the tensors' device, dtype and contiguity, passes raw
device pointers, sizes and the current CUDA stream to the C ABI declared in
include/pagedattn.h, and raises on a non-zero return code.  All arithmetic
runs in the library's CUDA kernels; there is no other implementation here, and
a missing library is an error, never a fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

_LIB = None

PKV_STATUS_BITS = {
    1 << 0: "SLOT_OUT_OF_RANGE",
    1 << 1: "BAD_BLOCK_ID",
    1 << 2: "BAD_CONTEXT_LEN",
    1 << 3: "BAD_SEQLENS",
    1 << 4: "BAD_TEMPERATURE",
    1 << 5: "NO_FINITE_KEY",
    1 << 6: "WORKSPACE_OVERFLOW",
    1 << 7: "WAIT_TIMEOUT",
}
STATUS = {v: k for k, v in PKV_STATUS_BITS.items()}

C_FUNCTIONS = ["pkv_version", "pkv_error_string", "pkv_status_string", "pkv_kv_store",
               "pkv_paged_decode_workspace_bytes", "pkv_paged_decode",
               "pkv_paged_prefill_workspace_bytes", "pkv_paged_prefill_varlen", "pkv_sample",
               "pkv_paged_decode_static_workspace", "pkv_kv_store_paged_decode",
               "pkv_kv_store_paged_prefill_varlen", "pkv_paged_decode_plan",
               "pkv_paged_decode_run", "pkv_paged_attention_varlen_workspace_bytes",
               "pkv_kv_store_paged_attention_varlen",
               "pkv_layer_cache", "pkv_sample_philox", "pkv_set_wait_poll_limit"]

# Size of the scratch array compiled into the library for
# pkv_paged_decode_static_workspace (PKV_STATIC_DECODE_WORKSPACE_BYTES).
STATIC_DECODE_WORKSPACE_BYTES = 16 * 1024 * 1024


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads libpagedattn.so (built by __graft_entry__.build() or
    paged_kv_attention_scatter_gb300._build.build()).  Raises if it is missing."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run paged_kv_attention_scatter_gb300._build."
                           "build() (or __graft_entry__.build()) first")
    lib = ctypes.CDLL(path)
    P, I32, SZ, F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    lib.pkv_version.restype = ctypes.c_int
    lib.pkv_version.argtypes = []
    lib.pkv_error_string.restype = ctypes.c_char_p
    lib.pkv_error_string.argtypes = [ctypes.c_int]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_status_string.argtypes = [ctypes.c_uint32]
    lib.pkv_kv_store.restype = ctypes.c_int
    lib.pkv_kv_store.argtypes = [P, P, P, P, P, I32, CacheDesc, P, P]
    lib.pkv_paged_decode_workspace_bytes.restype = SZ
    lib.pkv_paged_decode_workspace_bytes.argtypes = [I32, I32, I32, CacheDesc]
    lib.pkv_paged_decode.restype = ctypes.c_int
    lib.pkv_paged_decode.argtypes = [P, P, P, P, I32, P, I32, I32, I32, F32, P, P, SZ,
                                     CacheDesc, P, P]
    lib.pkv_paged_decode_plan.restype = ctypes.c_int
    lib.pkv_paged_decode_plan.argtypes = [P, I32, I32, I32, I32, P, SZ, CacheDesc, P, P]
    lib.pkv_paged_decode_run.restype = ctypes.c_int
    lib.pkv_paged_decode_run.argtypes = [P, P, P, P, I32, P, I32, I32, I32, F32, P, P, SZ,
                                         CacheDesc, P, P]
    lib.pkv_paged_prefill_workspace_bytes.restype = SZ
    lib.pkv_paged_prefill_workspace_bytes.argtypes = [I32, I32, I32, CacheDesc]
    lib.pkv_paged_prefill_varlen.restype = ctypes.c_int
    lib.pkv_paged_prefill_varlen.argtypes = [P, P, P, P, P, P, P, I32, I32, I32, I32, I32, P,
                                             I32, F32, P, P, SZ, CacheDesc, P, P]
    lib.pkv_sample.restype = ctypes.c_int
    lib.pkv_sample.argtypes = [P, P, P, I32, I32, P, P, P]
    lib.pkv_kv_store_paged_decode.restype = ctypes.c_int
    lib.pkv_kv_store_paged_decode.argtypes = [P, P, P, I32, P, P, P, P, I32, P, I32, I32, I32,
                                              F32, P, P, SZ, CacheDesc, P, P]
    lib.pkv_kv_store_paged_prefill_varlen.restype = ctypes.c_int
    lib.pkv_kv_store_paged_prefill_varlen.argtypes = [P, P, P, P, P, P, P, P, I32, I32, I32,
                                                      I32, I32, P, I32, F32, P, P, SZ,
                                                      CacheDesc, P, P]
    lib.pkv_paged_attention_varlen_workspace_bytes.restype = ctypes.c_size_t
    lib.pkv_paged_attention_varlen_workspace_bytes.argtypes = [I32, I32, I32, I32, CacheDesc]
    lib.pkv_kv_store_paged_attention_varlen.restype = ctypes.c_int
    lib.pkv_kv_store_paged_attention_varlen.argtypes = [P, P, P, P, P, P, P, P, I32, I32, I32,
                                                        I32, I32, P, I32, F32, P, P, SZ,
                                                        CacheDesc, P, P]
    lib.pkv_sample_philox.restype = ctypes.c_int
    lib.pkv_sample_philox.argtypes = [P, P, ctypes.c_uint64, ctypes.c_uint64, I32, I32, P, P, P]
    lib.pkv_layer_cache.restype = ctypes.c_int
    lib.pkv_layer_cache.argtypes = [P, I32, I32, CacheDesc, ctypes.POINTER(ctypes.c_void_p),
                                    ctypes.POINTER(ctypes.c_void_p)]
    lib.pkv_set_wait_poll_limit.restype = ctypes.c_int
    lib.pkv_set_wait_poll_limit.argtypes = [ctypes.c_uint32]
    _LIB = lib
    return lib


# ----------------------------------------------------------------------------
def _check(rc: int, what: str) -> None:
    if rc != 0:
        msg = load().pkv_error_string(rc).decode()
        raise RuntimeError(f"{what}: {msg} (code {rc})")


def _dev(t: torch.Tensor, name: str, dtype, device=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t.data_ptr()


def _ptr_or_null(t, name, dtype, device):
    return None if t is None else _dev(t, name, dtype, device)


def _stream(device, stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    nb, bs, hkv, d = k_cache.shape
    return CacheDesc(nb, bs, hkv, d)


def new_status(device) -> torch.Tensor:
    """A zeroed device status word for the `status=` argument."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def status_names(word: int) -> list[str]:
    return [n for b, n in PKV_STATUS_BITS.items() if word & b]


# ----------------------------------------------------------------------------
def kv_store(k, v, k_cache, v_cache, slot_mapping, status=None, stream=None) -> None:
    """Writes row i of k / v into slot slot_mapping[i] of k_cache / v_cache
    (in place).  k, v: [N, Hkv, D] bf16; caches [NB, bs, Hkv, D] bf16;
    slot_mapping [N] int32 (negative = skip)."""
    lib = load()
    dev = k_cache.device
    n = slot_mapping.numel()
    if k.shape != (n,) + tuple(k_cache.shape[2:]) or v.shape != k.shape:
        raise ValueError("k/v must be [num_tokens, num_kv_heads, head_dim] matching the cache")
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    rc = lib.pkv_kv_store(_dev(k, "k", torch.bfloat16, dev), _dev(v, "v", torch.bfloat16, dev),
                          _dev(k_cache, "k_cache", torch.bfloat16, dev),
                          _dev(v_cache, "v_cache", torch.bfloat16, dev),
                          _dev(slot_mapping, "slot_mapping", torch.int32, dev), n,
                          cache_desc(k_cache), _ptr_or_null(status, "status", torch.int32, dev),
                          _stream(dev, stream))
    _check(rc, "pkv_kv_store")


def paged_decode_workspace_bytes(batch, num_q_heads, max_context_len, k_cache) -> int:
    return int(load().pkv_paged_decode_workspace_bytes(batch, num_q_heads, max_context_len,
                                                       cache_desc(k_cache)))


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale, max_context_len,
                 out=None, workspace=None, status=None, stream=None) -> torch.Tensor:
    """Decode attention: q [B, Hq, D] bf16 -> out [B, Hq, D] bf16.
    block_tables [B, MB] int32, context_lens [B] int32, max_context_len a host
    upper bound of context_lens."""
    lib = load()
    dev = k_cache.device
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    need = paged_decode_workspace_bytes(B, Hq, max_context_len, k_cache)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    rc = lib.pkv_paged_decode(_dev(q, "q", torch.bfloat16, dev),
                              _dev(k_cache, "k_cache", torch.bfloat16, dev),
                              _dev(v_cache, "v_cache", torch.bfloat16, dev),
                              _dev(block_tables, "block_tables", torch.int32, dev),
                              block_tables.shape[1],
                              _dev(context_lens, "context_lens", torch.int32, dev), B, Hq,
                              int(max_context_len), float(scale),
                              _dev(out, "out", torch.bfloat16, dev),
                              _dev(workspace, "workspace", torch.uint8, dev), workspace.numel(),
                              cache_desc(k_cache),
                              _ptr_or_null(status, "status", torch.int32, dev),
                              _stream(dev, stream))
    _check(rc, "pkv_paged_decode")
    return out


def paged_decode_plan(context_lens, num_q_heads, max_context_len, max_blocks_per_seq, k_cache,
                      workspace=None, status=None, stream=None) -> torch.Tensor:
    """The chunk schedule of a decode batch, written into `workspace` (made
    here when None), for any number of paged_decode_run calls over layers that
    share these context lengths.  Returns the workspace."""
    lib = load()
    dev = k_cache.device
    B = context_lens.numel()
    need = paged_decode_workspace_bytes(B, num_q_heads, max_context_len, k_cache)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    rc = lib.pkv_paged_decode_plan(_dev(context_lens, "context_lens", torch.int32, dev), B,
                                   int(num_q_heads), int(max_context_len),
                                   int(max_blocks_per_seq),
                                   _dev(workspace, "workspace", torch.uint8, dev),
                                   workspace.numel(), cache_desc(k_cache),
                                   _ptr_or_null(status, "status", torch.int32, dev),
                                   _stream(dev, stream))
    _check(rc, "pkv_paged_decode_plan")
    return workspace


def paged_decode_run(q, k_cache, v_cache, block_tables, context_lens, scale, max_context_len,
                     workspace, out=None, status=None, stream=None) -> torch.Tensor:
    """paged_decode with the schedule a paged_decode_plan call wrote into
    `workspace` (same context lengths and sizes)."""
    lib = load()
    dev = k_cache.device
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    rc = lib.pkv_paged_decode_run(_dev(q, "q", torch.bfloat16, dev),
                                  _dev(k_cache, "k_cache", torch.bfloat16, dev),
                                  _dev(v_cache, "v_cache", torch.bfloat16, dev),
                                  _dev(block_tables, "block_tables", torch.int32, dev),
                                  block_tables.shape[1],
                                  _dev(context_lens, "context_lens", torch.int32, dev), B, Hq,
                                  int(max_context_len), float(scale),
                                  _dev(out, "out", torch.bfloat16, dev),
                                  _dev(workspace, "workspace", torch.uint8, dev),
                                  workspace.numel(), cache_desc(k_cache),
                                  _ptr_or_null(status, "status", torch.int32, dev),
                                  _stream(dev, stream))
    _check(rc, "pkv_paged_decode_run")
    return out


def paged_prefill_workspace_bytes(batch, total_q, num_q_heads, k_cache_shape) -> int:
    nb, bs, hkv, d = k_cache_shape
    return int(load().pkv_paged_prefill_workspace_bytes(batch, total_q, num_q_heads,
                                                        CacheDesc(nb, bs, hkv, d)))


def paged_prefill_varlen(q, k, v, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                         max_seqlen_k, block_tables, scale, out=None, workspace=None,
                         status=None, stream=None) -> torch.Tensor:
    """Causal varlen prefill: q [Tq, Hq, D], k/v [Tq, Hkv, D] bf16 -> out
    [Tq, Hq, D] bf16.  k_cache/v_cache and block_tables may be None when no
    sequence has a cached prefix."""
    lib = load()
    dev = q.device
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    B = cu_seqlens_q.numel() - 1
    shape = tuple(k_cache.shape) if k_cache is not None else (1, 1, Hkv, D)
    if out is None:
        out = torch.empty_like(q)
    need = paged_prefill_workspace_bytes(B, T, Hq, shape)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    desc = CacheDesc(*shape)
    rc = lib.pkv_paged_prefill_varlen(
        _dev(q, "q", torch.bfloat16, dev), _dev(k, "k", torch.bfloat16, dev),
        _dev(v, "v", torch.bfloat16, dev),
        _ptr_or_null(k_cache, "k_cache", torch.bfloat16, dev),
        _ptr_or_null(v_cache, "v_cache", torch.bfloat16, dev),
        _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32, dev),
        _dev(cu_seqlens_k, "cu_seqlens_k", torch.int32, dev), B, T, int(max_seqlen_q),
        int(max_seqlen_k), Hq, _ptr_or_null(block_tables, "block_tables", torch.int32, dev),
        block_tables.shape[1] if block_tables is not None else 0, float(scale),
        _dev(out, "out", torch.bfloat16, dev), _dev(workspace, "workspace", torch.uint8, dev),
        workspace.numel(), desc, _ptr_or_null(status, "status", torch.int32, dev),
        _stream(dev, stream))
    _check(rc, "pkv_paged_prefill_varlen")
    return out


def kv_store_paged_prefill_varlen(q, k, v, k_cache, v_cache, slot_mapping, cu_seqlens_q,
                                  cu_seqlens_k, max_seqlen_q, max_seqlen_k, block_tables, scale,
                                  out=None, workspace=None, status=None,
                                  stream=None) -> torch.Tensor:
    """kv_store of the chunk's k/v rows (slot_mapping [Tq] int32) followed by
    paged_prefill_varlen, in one call.  block_tables may be None when no
    sequence has a cached prefix; the cache is always written."""
    lib = load()
    dev = q.device
    T, Hq, D = q.shape
    B = cu_seqlens_q.numel() - 1
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must hold one slot per query token")
    if out is None:
        out = torch.empty_like(q)
    need = paged_prefill_workspace_bytes(B, T, Hq, tuple(k_cache.shape))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    rc = lib.pkv_kv_store_paged_prefill_varlen(
        _dev(q, "q", torch.bfloat16, dev), _dev(k, "k", torch.bfloat16, dev),
        _dev(v, "v", torch.bfloat16, dev), _dev(k_cache, "k_cache", torch.bfloat16, dev),
        _dev(v_cache, "v_cache", torch.bfloat16, dev),
        _dev(slot_mapping, "slot_mapping", torch.int32, dev),
        _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32, dev),
        _dev(cu_seqlens_k, "cu_seqlens_k", torch.int32, dev), B, T, int(max_seqlen_q),
        int(max_seqlen_k), Hq, _ptr_or_null(block_tables, "block_tables", torch.int32, dev),
        block_tables.shape[1] if block_tables is not None else 0, float(scale),
        _dev(out, "out", torch.bfloat16, dev), _dev(workspace, "workspace", torch.uint8, dev),
        workspace.numel(), cache_desc(k_cache), _ptr_or_null(status, "status", torch.int32, dev),
        _stream(dev, stream))
    _check(rc, "pkv_kv_store_paged_prefill_varlen")
    return out


def paged_attention_varlen_workspace_bytes(batch, total_q, num_q_heads, max_seqlen_k,
                                           k_cache_shape) -> int:
    nb, bs, hkv, d = k_cache_shape
    return int(load().pkv_paged_attention_varlen_workspace_bytes(
        batch, total_q, num_q_heads, int(max_seqlen_k), CacheDesc(nb, bs, hkv, d)))


def kv_store_paged_attention_varlen(q, k, v, k_cache, v_cache, slot_mapping, cu_seqlens_q,
                                    cu_seqlens_k, max_seqlen_q, max_seqlen_k, block_tables,
                                    scale, out=None, workspace=None, status=None,
                                    stream=None) -> torch.Tensor:
    """kv_store then attention over a batch mixing prefill chunks and decode
    rows: the result of kv_store_paged_prefill_varlen, with one-query
    sequences run by the split-KV decode kernels (they read their own new key
    back from the cache, so slot_mapping must place it in their block table).
    block_tables is required."""
    lib = load()
    dev = q.device
    T, Hq, D = q.shape
    B = cu_seqlens_q.numel() - 1
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must hold one slot per query token")
    if block_tables is None:
        raise ValueError("block_tables is required")
    if out is None:
        out = torch.empty_like(q)
    need = paged_attention_varlen_workspace_bytes(B, T, Hq, max_seqlen_k, tuple(k_cache.shape))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    rc = lib.pkv_kv_store_paged_attention_varlen(
        _dev(q, "q", torch.bfloat16, dev), _dev(k, "k", torch.bfloat16, dev),
        _dev(v, "v", torch.bfloat16, dev), _dev(k_cache, "k_cache", torch.bfloat16, dev),
        _dev(v_cache, "v_cache", torch.bfloat16, dev),
        _dev(slot_mapping, "slot_mapping", torch.int32, dev),
        _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32, dev),
        _dev(cu_seqlens_k, "cu_seqlens_k", torch.int32, dev), B, T, int(max_seqlen_q),
        int(max_seqlen_k), Hq, _dev(block_tables, "block_tables", torch.int32, dev),
        block_tables.shape[1], float(scale),
        _dev(out, "out", torch.bfloat16, dev), _dev(workspace, "workspace", torch.uint8, dev),
        workspace.numel(), cache_desc(k_cache), _ptr_or_null(status, "status", torch.int32, dev),
        _stream(dev, stream))
    _check(rc, "pkv_kv_store_paged_attention_varlen")
    return out


def sample(logits, temperatures, exp_noise, out=None, status=None, stream=None) -> torch.Tensor:
    """Gumbel-max sampling: logits, exp_noise [B, V] fp32, temperatures [B]
    fp32 -> token ids [B] int32."""
    lib = load()
    dev = logits.device
    B, V = logits.shape
    if exp_noise.shape != logits.shape or temperatures.shape != (B,):
        raise ValueError("shape mismatch between logits, temperatures and exp_noise")
    if out is None:
        out = torch.empty(B, dtype=torch.int32, device=dev)
    rc = lib.pkv_sample(_dev(logits, "logits", torch.float32, dev),
                        _dev(temperatures, "temperatures", torch.float32, dev),
                        _dev(exp_noise, "exp_noise", torch.float32, dev), B, V,
                        _dev(out, "out", torch.int32, dev),
                        _ptr_or_null(status, "status", torch.int32, dev), _stream(dev, stream))
    _check(rc, "pkv_sample")
    return out


def paged_decode_static_workspace(q, k_cache, v_cache, block_tables, context_lens, scale,
                                  max_context_len, out=None, status=None,
                                  stream=None) -> torch.Tensor:
    """paged_decode for callers that cannot allocate device memory where they
    call (e.g. a plugin whose host engine owns all device memory, or a loop
    that must not pay for cudaMalloc's implicit synchronisation): the split-KV
    scratch is the library's own fixed array of STATIC_DECODE_WORKSPACE_BYTES,
    so apart from `out` (pass it to avoid the one allocation here) nothing is
    allocated.  Calls share that array: do not let two of them overlap on the
    GPU.  The first call on a device resolves the array's address; make it
    before any stream capture."""
    lib = load()
    fn = lib.pkv_paged_decode_static_workspace
    if fn.restype is not ctypes.c_int or not fn.argtypes:
        P, I32, F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
        fn.restype = ctypes.c_int
        fn.argtypes = [P, P, P, P, I32, P, I32, I32, I32, F32, P, CacheDesc, P, P]
    dev = k_cache.device
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    rc = fn(_dev(q, "q", torch.bfloat16, dev), _dev(k_cache, "k_cache", torch.bfloat16, dev),
            _dev(v_cache, "v_cache", torch.bfloat16, dev),
            _dev(block_tables, "block_tables", torch.int32, dev), block_tables.shape[1],
            _dev(context_lens, "context_lens", torch.int32, dev), B, Hq, int(max_context_len),
            float(scale), _dev(out, "out", torch.bfloat16, dev), cache_desc(k_cache),
            _ptr_or_null(status, "status", torch.int32, dev), _stream(dev, stream))
    _check(rc, "pkv_paged_decode_static_workspace")
    return out


def kv_store_paged_decode(k, v, slot_mapping, q, k_cache, v_cache, block_tables, context_lens,
                          scale, max_context_len, out=None, workspace=None, status=None,
                          stream=None) -> torch.Tensor:
    """kv_store of the new tokens followed by paged_decode, in one call."""
    lib = load()
    dev = k_cache.device
    B, Hq, D = q.shape
    n = slot_mapping.numel()
    if k.shape != (n,) + tuple(k_cache.shape[2:]) or v.shape != k.shape:
        raise ValueError("k/v must be [num_tokens, num_kv_heads, head_dim] matching the cache")
    if out is None:
        out = torch.empty_like(q)
    need = paged_decode_workspace_bytes(B, Hq, max_context_len, k_cache)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    rc = lib.pkv_kv_store_paged_decode(
        _dev(k, "k", torch.bfloat16, dev), _dev(v, "v", torch.bfloat16, dev),
        _dev(slot_mapping, "slot_mapping", torch.int32, dev), n,
        _dev(q, "q", torch.bfloat16, dev), _dev(k_cache, "k_cache", torch.bfloat16, dev),
        _dev(v_cache, "v_cache", torch.bfloat16, dev),
        _dev(block_tables, "block_tables", torch.int32, dev), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32, dev), B, Hq, int(max_context_len),
        float(scale), _dev(out, "out", torch.bfloat16, dev),
        _dev(workspace, "workspace", torch.uint8, dev), workspace.numel(), cache_desc(k_cache),
        _ptr_or_null(status, "status", torch.int32, dev), _stream(dev, stream))
    _check(rc, "pkv_kv_store_paged_decode")
    return out


def layer_cache(kv_pool: torch.Tensor, layer: int):
    """(k_cache, v_cache) views of one layer of a [2, L, NB, bs, Hkv, D] bf16 pool.
    The layer's addresses come from pkv_layer_cache (checked against the views)."""
    if kv_pool.dim() != 6 or kv_pool.shape[0] != 2 or not kv_pool.is_contiguous():
        raise ValueError("kv_pool must be a contiguous [2, L, NB, bs, Hkv, D] tensor")
    L, nb, bs, hkv, d = kv_pool.shape[1:]
    kp, vp = ctypes.c_void_p(), ctypes.c_void_p()
    rc = load().pkv_layer_cache(kv_pool.data_ptr(), L, int(layer), CacheDesc(nb, bs, hkv, d),
                                ctypes.byref(kp), ctypes.byref(vp))
    _check(rc, "pkv_layer_cache")
    kc, vc = kv_pool[0, layer], kv_pool[1, layer]
    if kc.data_ptr() != kp.value or vc.data_ptr() != vp.value:
        raise RuntimeError("pkv_layer_cache disagrees with the tensor layout")
    return kc, vc


def sample_philox(logits, temperatures, seed: int, offset: int, out=None, status=None,
                  stream=None) -> torch.Tensor:
    """Gumbel-max sampling with in-kernel Philox4x32-10 Exp(1) noise: logits
    [B, V] fp32, temperatures [B] fp32 -> token ids [B] int32."""
    lib = load()
    dev = logits.device
    B, V = logits.shape
    if temperatures.shape != (B,):
        raise ValueError("temperatures must be [batch]")
    if out is None:
        out = torch.empty(B, dtype=torch.int32, device=dev)
    rc = lib.pkv_sample_philox(_dev(logits, "logits", torch.float32, dev),
                               _dev(temperatures, "temperatures", torch.float32, dev),
                               int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), B, V,
                               _dev(out, "out", torch.int32, dev),
                               _ptr_or_null(status, "status", torch.int32, dev),
                               _stream(dev, stream))
    _check(rc, "pkv_sample_philox")
    return out


DEFAULT_WAIT_POLLS = 1 << 20            # PKV_DEFAULT_WAIT_POLLS


def set_wait_poll_limit(polls: int = DEFAULT_WAIT_POLLS) -> None:
    """Polls a bounded in-kernel wait makes before it gives up, for calls
    enqueued afterwards (default DEFAULT_WAIT_POLLS).  A diagnostic: 0 makes
    every such wait give up at once, which exercises the kernels' unwinding."""
    _check(load().pkv_set_wait_poll_limit(int(polls) & 0xFFFFFFFF), "pkv_set_wait_poll_limit")
