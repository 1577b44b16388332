"""The C ABI from C: tests/c/pkv_client.c includes only include/pagedattn.h
(and, in its GPU mode, the CUDA runtime for device memory), is built with gcc
against libpagedattn.so and calls the library directly.  Host mode runs
without a GPU; GPU mode runs one small decode step (kv_store, paged_decode,
sample) and its outputs are compared with the oracle here."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "pkv_client.c")
CUDA = "/usr/local/cuda"


def _build(tmp_path, gpu: bool) -> str:
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    from paged_kv_attention_scatter_gb300 import _build as B
    lib = B.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / ("pkv_client_gpu" if gpu else "pkv_client"))
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1",
           "-I", os.path.join(ROOT, "include"), SRC, "-L", libdir, "-lpagedattn",
           f"-Wl,-rpath,{libdir}", "-o", exe]
    if gpu:
        cmd[1:1] = ["-DPKV_CLIENT_GPU", "-I", os.path.join(CUDA, "include")]
        cmd += ["-L", os.path.join(CUDA, "lib64"), "-lcudart",
                f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_host_calls_from_c(tmp_path):
    exe = _build(tmp_path, gpu=False)
    r = subprocess.run([exe, "host"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_decode_step_from_c_matches_the_oracle(tmp_path, cuda):
    from oracle import attention as oatt
    from oracle import kv_store as okv
    from oracle import sampler as osm
    from paged_kv_attention_scatter_gb300 import workloads as W

    import gpu_util as U
    exe = _build(tmp_path, gpu=True)
    spec = W.DecodeSpec("c client step", seed=91, batch=6, num_q_heads=8, num_kv_heads=2,
                        head_dim=128, block_size=64, ctx_lo=50, ctx_hi=700,
                        store_new_token=True, vocab=2000, logit_sigma=3.0, logit_spikes=4,
                        t_lo=0.3, t_hi=1.1)
    w = W.decode_workload(spec)
    d = tmp_path

    def put(name, t):
        t.contiguous().view(torch.uint8).numpy().tofile(str(d / name))

    put("k_cache.bin", w.k_cache)
    put("v_cache.bin", w.v_cache)
    put("k_new.bin", w.k_new)
    put("v_new.bin", w.v_new)
    put("slots.bin", w.slot_mapping)
    put("q.bin", w.q)
    put("block_tables.bin", w.block_tables)
    put("context_lens.bin", w.context_lens)
    put("logits.bin", w.logits)
    put("temperatures.bin", w.temperatures)
    put("noise.bin", w.exp_noise)
    nb, bs, hkv, dd = w.k_cache.shape
    (d / "sizes.txt").write_text(f"{nb} {bs} {hkv} {dd} {spec.batch} {spec.num_q_heads} "
                                 f"{w.block_tables.shape[1]} {w.max_context_len} {spec.vocab} "
                                 f"{w.scale!r}\n")
    r = subprocess.run([exe, "gpu", str(d)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr

    def get(name, dtype, shape):
        return np.fromfile(str(d / name), dtype=dtype).reshape(shape)

    # the cache after the store, bit for bit
    kc, vc, _ = okv.kv_store(U.bits(w.k_new), U.bits(w.v_new), U.bits(w.k_cache),
                             U.bits(w.v_cache), w.slot_mapping.numpy())
    assert np.array_equal(get("k_cache_out.bin", np.int16, kc.shape), kc)
    assert np.array_equal(get("v_cache_out.bin", np.int16, vc.shape), vc)
    # the attention output against the float64 oracle
    out = torch.from_numpy(get("out.bin", np.int16, tuple(w.q.shape))).view(torch.bfloat16)
    ref = oatt.paged_decode(U.f64(w.q), torch.from_numpy(kc).view(torch.bfloat16),
                            torch.from_numpy(vc).view(torch.bfloat16), w.block_tables.numpy(),
                            w.context_lens.numpy(), w.scale)
    U.assert_close(U.f64(out), ref, "decode from C")
    # the token ids, exact up to float32 near-ties
    ids = get("ids.bin", np.int32, (spec.batch,))
    want, bad = osm.sample(w.logits.numpy(), w.temperatures.numpy(), w.exp_noise.numpy())
    _, keys = osm.sample_key_form(w.logits.numpy(), w.temperatures.numpy(),
                                  w.exp_noise.numpy())
    near = osm.near_ties(keys)
    assert not bad
    for r_ in range(spec.batch):
        assert ids[r_] == want[r_] or (len(near[r_]) > 1 and ids[r_] in near[r_])
