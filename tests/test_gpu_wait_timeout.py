"""Bounded in-kernel waits that run out.

pkv_set_wait_poll_limit(0) makes every shared-memory barrier wait of the TMA
decode kernel and of the tcgen05 prefill kernel give up at once.  The kernels
must report PKV_STATUS_WAIT_TIMEOUT, let the copies and MMAs they already
issued finish, free TMEM and return (no trap, no fault, nothing left waiting);
with the default limit back, the next calls in the same process must match the
oracle.  A limit of a few polls (some waits succeed, some give up) must unwind
as well.  The limit is restored even when a test fails."""
import numpy as np
import pytest

import gpu_util as U
from oracle import attention as oatt
from paged_kv_attention_scatter_gb300 import workloads as W
from test_gpu_prefill import _check_case, _prefill, make_case

pytestmark = pytest.mark.gpu


@pytest.fixture
def wait_limit():
    pkv = U.lib()
    yield pkv.set_wait_poll_limit
    pkv.set_wait_poll_limit()


def _timeout_bit(pkv):
    return pkv.STATUS["WAIT_TIMEOUT"]


def test_decode_gives_up_then_recovers(cuda, wait_limit):
    pkv = U.lib()
    # block size 256: the TMA-fed split kernel
    spec = W.DecodeSpec("wait timeout decode", seed=41, batch=8, num_q_heads=16,
                        num_kv_heads=8, head_dim=128, block_size=256, ctx_lo=300, ctx_hi=3000)
    w = W.decode_workload(spec, device=cuda)
    bt, ctx = w.block_tables.to(cuda), w.context_lens.to(cuda)
    for polls in (0, 2):
        wait_limit(polls)
        st = pkv.new_status(cuda)
        pkv.paged_decode(w.q, w.k_cache, w.v_cache, bt, ctx, w.scale, w.max_context_len,
                         status=st)
        word = U.status_word(st)                 # synchronises: the kernels returned
        if polls == 0:
            assert word & _timeout_bit(pkv)
        assert word & ~_timeout_bit(pkv) == 0
    wait_limit()
    st = pkv.new_status(cuda)
    out = pkv.paged_decode(w.q, w.k_cache, w.v_cache, bt, ctx, w.scale, w.max_context_len,
                           status=st)
    assert U.status_word(st) == 0
    ref = oatt.paged_decode(U.f64(w.q), w.k_cache.cpu(), w.v_cache.cpu(),
                            w.block_tables.numpy(), w.context_lens.numpy(), w.scale)
    U.assert_close(U.f64(out), ref, "decode after the timeouts")


# block size 256: cached tiles as TMA boxes; 64 and 16: per-block boxes for K
# and part of V, the rest of V gathered with cp.async; 48: both gathered
@pytest.mark.parametrize("bs,cached", [(256, [256, 0, 512]), (64, [128, 64, 0]),
                                       (16, [64, 5, 0]), (48, [96, 5, 0])])
def test_prefill_gives_up_then_recovers(cuda, wait_limit, bs, cached):
    pkv = U.lib()
    c = make_case(43 + bs, [300, 700, 129], cached, 8, 2, 128, bs)
    args = (pkv, cuda, c["q"], c["k"], c["v"], c["kc"], c["vc"], c["cu_q"], c["cu_k"], c["bt"],
            0.088, c["max_sq"], c["max_sk"])
    for polls in (0, 3):
        wait_limit(polls)
        st = pkv.new_status(cuda)
        _prefill(*args, status=st)
        word = U.status_word(st)
        if polls == 0:
            assert word & _timeout_bit(pkv)
        assert word & ~_timeout_bit(pkv) == 0
    wait_limit()
    err, rel = _check_case(pkv, cuda, c, 0.088)
    assert np.isfinite(err) and np.isfinite(rel)
