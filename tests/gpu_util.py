"""Helpers of the GPU parity tests (no arithmetic of the method here)."""
from __future__ import annotations

import numpy as np
import torch

# attention tolerance over a compared tensor: max-abs and relative L2 against
# the float64 oracle
MAX_ABS = 2e-2
REL_L2 = 5e-3


def f64(t) -> np.ndarray:
    return t.detach().to("cpu").double().numpy()


def bits(t) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy()


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = "") -> tuple[float, float]:
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite outputs"
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))
    assert err <= MAX_ABS and rel <= REL_L2, f"{what}: max abs {err:.3g}, rel L2 {rel:.3g}"
    return err, rel


def lib():
    import paged_kv_attention_scatter_gb300 as pkv
    pkv.build()
    pkv.load()
    return pkv


def status_word(s: torch.Tensor) -> int:
    torch.cuda.synchronize()
    return int(s.item()) & 0xFFFFFFFF


def bf16_case(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def build_paged_cache(K_seqs, V_seqs, block_size, num_blocks, gen, extra_blocks_per_seq=None):
    """Scatter per-sequence logical K/V (bf16, [n, Hkv, D]) into a NaN pool
    through random block tables; returns (k_cache, v_cache, block_tables)."""
    Hkv, D = K_seqs[0].shape[1], K_seqs[0].shape[2]
    kc = torch.full((num_blocks * block_size, Hkv, D), float("nan"), dtype=torch.bfloat16)
    vc = kc.clone()
    perm = torch.randperm(num_blocks, generator=gen).tolist()
    tables = []
    for i, (K, V) in enumerate(zip(K_seqs, V_seqs)):
        n = K.shape[0]
        nb = -(-n // block_size)
        if extra_blocks_per_seq is not None:
            nb = max(nb, extra_blocks_per_seq[i])
        t = [perm.pop() for _ in range(nb)]
        tables.append(t)
        for p in range(n):
            s = t[p // block_size] * block_size + p % block_size
            kc[s], vc[s] = K[p], V[p]
    width = max(1, max(len(t) for t in tables))
    bt = torch.full((len(tables), width), -1, dtype=torch.int32)
    for i, t in enumerate(tables):
        if t:
            bt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
    shape = (num_blocks, block_size, Hkv, D)
    return kc.reshape(shape), vc.reshape(shape), bt
