#!/usr/bin/env python3
"""Benchmark of the paged-KV attention hot path on GB300.

Headline: paged decode HBM GB/s on the decode-0.6b workload (B=64, 16/8 heads,
D=128, 256-slot blocks, context U[512,4096]); a step is the decode attention of
a 28-layer Qwen3-0.6B-shaped model: one paged_decode_plan and 28
paged_decode_run calls (split-KV + combine kernels) over a multi-layer pool,
replayed from one CUDA graph so host launch cost does not enter the device
time.  `e2e` is the same step through the public API with pinned host buffers
copied in and out every step.  The same JSON line also carries the prefill-8b
chunked prefill (tokens/s, TFLOP/s, % of the tensor peak), decode-32b, the
step-8b decode step, the mixed-8b continuous-batching step (decode rows and
prefill chunks in one call) and a single call per graph launch as `secondary`.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (float64 NumPy) on a bounded sample of
the same workload.  Under torchrun (N > 1) every rank runs an independent
replica; value = bytes of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode HBM GB/s (% of peak) & prefill tokens/s (% TC peak), 1 GB300"
L2_BYTES = 129e6
LAYERS_0P6B = 28                   # decoder layers of a Qwen3-0.6B-shaped model

# DRAM bytes (read + write) of one decode-0.6b paged_decode_run, summed over
# its split and combine launches, from one ncu capture (profiles/
# decode_tma_kernel_decode-0.6b.md).  Valid only for the decode sources it was
# taken on: the digest below must match, otherwise the traffic is reported null.
DECODE_0P6B_TRAFFIC = {"bytes": 582375168,
                       "sources_sha256": "4f3671be8474468ac0fcfe30a52d3b3b4518c9ca6ecf37f3d0b5debab6d14c9e"}

DECODE_SOURCES = ["paged_decode.cu", "paged_decode_tma.cu", "decode_common.cuh", "common.cuh",
                  "tc_utils.cuh", "tma_host.cuh"]


def decode_sources_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "paged_kv_attention_scatter_gb300", "csrc")
    for f in DECODE_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return dict(hbm=float(d["hbm_gbs"]), tc=float(d["bf16_tflops"]),
                    tc_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured (MEASURED_PEAKS.json)")
    except Exception:
        return dict(hbm=6800.0, tc=1900.0, tc_sustained=1700.0, source="fallback")


# ----------------------------------------------------------------------------
# algorithmic work
# ----------------------------------------------------------------------------
def decode_bytes(ctx, hq, hkv, d, bs) -> float:
    """K and V of every attended key, q read, out written, block-table entries
    and context lengths read."""
    ctx = [int(c) for c in ctx]
    kv = sum(2 * c * hkv * d * 2 for c in ctx)
    qo = 2 * len(ctx) * hq * d * 2
    tables = 4 * sum(-(-c // bs) for c in ctx)
    return float(kv + qo + tables + 4 * len(ctx))


def prefill_flops(cu_q, cu_k, hq, d) -> float:
    """Causal attention FLOPs: query at position p attends p+1 keys; QK^T and PV
    cost 2*D each per (query, key, head)."""
    tot = 0
    for b in range(len(cu_q) - 1):
        lq, lk = cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]
        c = lk - lq
        tot += (lk * (lk + 1) - c * (c + 1)) // 2          # sum_{p=c}^{lk-1} (p+1)
    return 4.0 * d * hq * tot


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = [r.split(",") for r in open(self.file.name).read().strip().splitlines() if r]
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for n, v in zip(names, r[5:9]):
                    if "Active" in v and "Not" not in v:
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# device timing helpers
# ----------------------------------------------------------------------------
def graph_of(fn, torch):
    fn()                                   # warm: attributes, occupancy queries
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_graph(g, iters, torch):
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(iters):
        g.replay()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / iters * 1e-3          # seconds per replay


def flush_l2(buf):
    """Evicts everything from L2: writes the first half of `buf` (larger than
    L2), then reads the second half, so the timed call neither finds its data
    in L2 nor pays for writing back the flush's dirty lines."""
    half = buf.numel() // 2
    buf[:half].add_(1)
    buf[half:].sum()


def slowest_rank_seconds(step_s: float, dist, device=None) -> float:
    """The largest per-step time over all ranks (each rank is a replica; the
    job is as fast as its slowest GPU).  Works with NCCL (CUDA device) and
    gloo (CPU) process groups; returns step_s unchanged without one."""
    if dist is None:
        return step_s
    import torch
    t = torch.tensor([step_s], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: float, world: int, step_s: float) -> float:
    """Whole-job throughput of `world` identical replicas: units of all ranks
    over the slowest rank's time."""
    return units_per_rank * world / step_s


# ----------------------------------------------------------------------------
def run_ours(args, rank, world, dist):
    import torch

    import paged_kv_attention_scatter_gb300 as pkv
    from paged_kv_attention_scatter_gb300 import workloads as W

    pkv.build()
    pkv.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    pk = peaks()

    # ---------------- headline: decode-0.6b ----------------
    # One step is the decode attention of a whole Qwen3-0.6B-shaped model step:
    # one plan (the layers share context lengths and block tables) and 28
    # layer runs back to back in one CUDA graph, layer l reading its own K/V
    # from a [2, 28, NB, bs, Hkv, D] pool (each layer holds the same synthetic
    # cache contents).  Every run streams 569 MB, far more than L2, so no run
    # finds the previous one's data in L2.
    spec = W.DECODE_0P6B
    w = W.decode_workload(spec, device=dev)
    B, hq, hkv, d, bs = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.block_size
    bt, ctx = w.block_tables.to(dev), w.context_lens.to(dev)
    pool = torch.empty((2, LAYERS_0P6B) + tuple(w.k_cache.shape), dtype=torch.bfloat16,
                       device=dev)
    for layer in range(LAYERS_0P6B):
        pool[0, layer].copy_(w.k_cache)
        pool[1, layer].copy_(w.v_cache)
    layers = [pkv.layer_cache(pool, layer) for layer in range(LAYERS_0P6B)]
    q, scale, max_ctx = w.q, w.scale, w.max_context_len
    ctx_list = w.context_lens.tolist()
    del w
    torch.cuda.empty_cache()
    out = torch.empty_like(q)
    ws = torch.empty(pkv.paged_decode_workspace_bytes(B, hq, max_ctx, layers[0][0]),
                     dtype=torch.uint8, device=dev)
    nbytes = LAYERS_0P6B * decode_bytes(ctx_list, hq, hkv, d, bs)

    mb = bt.shape[1]

    def step():
        # the layers share context lengths and block tables: one plan per step
        pkv.paged_decode_plan(ctx, hq, max_ctx, mb, layers[0][0], workspace=ws)
        for kc, vc in layers:
            pkv.paged_decode_run(q, kc, vc, bt, ctx, scale, max_ctx, ws, out=out)

    g = graph_of(step, torch)
    for _ in range(args.warmup):
        g.replay()
    launches_per_step = 1 + 2 * LAYERS_0P6B
    clocks = ClockSampler(dev.index).start()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        g.replay()
    t1.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    step_s = slowest_rank_seconds(t0.elapsed_time(t1) * 1e-3 / args.steps, dist, dev)
    value = replica_throughput(nbytes, world, step_s) / 1e9

    # ---------------- e2e through the C ABI with host buffers ----------------
    # every step: block tables, context lengths and each layer's q copied in
    # from pinned host memory, each layer's output read back.  The copies run
    # on two copy streams, ordered against the attention by events, so layer
    # i+1's q arrives and layer i's output leaves while layer i+1 computes.
    q_h = q.cpu().pin_memory()
    bt_h, ctx_h = bt.cpu().pin_memory(), ctx.cpu().pin_memory()
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in layers]
    q_d = [torch.empty_like(q) for _ in layers]
    out_d = [torch.empty_like(out) for _ in layers]
    bt_d = [torch.empty_like(bt) for _ in range(2)]        # by step parity
    ctx_d = [torch.empty_like(ctx) for _ in range(2)]
    ws_d = [ws, torch.empty_like(ws)]
    e2e_steps = max(10, min(args.steps, 300))
    ms = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    ev_meta, ev_step = ev(), [ev(), ev()]
    ev_q = [ev() for _ in layers]
    ev_run = [ev() for _ in layers]
    ev_d2h = [ev() for _ in layers]
    for e_ in ev_step + ev_run + ev_d2h:
        e_.record(ms)
    counter = [0]

    def e2e_step():
        p = counter[0] & 1
        counter[0] += 1
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(ev_step[p])          # the step two back is done with them
            bt_d[p].copy_(bt_h, non_blocking=True)
            ctx_d[p].copy_(ctx_h, non_blocking=True)
            ev_meta.record(h2d_s)
            for i in range(len(layers)):
                h2d_s.wait_event(ev_run[i])       # the previous step's run i read q_d[i]
                q_d[i].copy_(q_h, non_blocking=True)
                ev_q[i].record(h2d_s)
        ms.wait_event(ev_meta)
        pkv.paged_decode_plan(ctx_d[p], hq, max_ctx, mb, layers[0][0], workspace=ws_d[p])
        for i, (kc, vc) in enumerate(layers):
            ms.wait_event(ev_q[i])
            ms.wait_event(ev_d2h[i])              # out_d[i] of the previous step was read
            pkv.paged_decode_run(q_d[i], kc, vc, bt_d[p], ctx_d[p], scale, max_ctx, ws_d[p],
                                 out=out_d[i])
            ev_run[i].record(ms)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_run[i])
                out_h[i].copy_(out_d[i], non_blocking=True)
                ev_d2h[i].record(d2h_s)
        ev_step[p].record(ms)

    for _ in range(max(3, args.warmup // 10)):
        e2e_step()
    torch.cuda.synchronize()
    t0.record()
    for _ in range(e2e_steps):
        e2e_step()
    ms.wait_stream(d2h_s)                         # the last outputs are on the host
    t1.record()
    torch.cuda.synchronize()
    e2e_s = t0.elapsed_time(t1) * 1e-3 / e2e_steps
    h2d = LAYERS_0P6B * q_h.numel() * 2 + bt_h.numel() * 4 + ctx_h.numel() * 4
    d2h = LAYERS_0P6B * out.numel() * 2
    # parity spot check of the timed output against nothing but itself is
    # meaningless; the tests cover parity.  Keep the buffers alive until here.
    # the same call alone in its graph: includes a graph launch per call
    kc0, vc0 = layers[0]
    g1 = graph_of(lambda: pkv.paged_decode(q, kc0, vc0, bt, ctx, scale, max_ctx, out=out,
                                           workspace=ws), torch)
    for _ in range(5):
        g1.replay()
    single_s = time_graph(g1, 200, torch)
    single = {"workload": spec.name + ", one call per graph launch",
              "us": round(single_s * 1e6, 2),
              "gbs": round(nbytes / LAYERS_0P6B / single_s / 1e9, 1),
              "frac_hbm": round(nbytes / LAYERS_0P6B / single_s / 1e9 / pk["hbm"], 4)}
    del g, g1, q_h, out_h, layers, pool, kc0, vc0
    torch.cuda.empty_cache()

    secondary = {"decode-0.6b-single-call": single}
    if not args.headline_only:
        secondary.update(run_secondary(args, pkv, W, torch, dev, pk))

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": spec.name, "batch": B, "num_q_heads": hq, "num_kv_heads": hkv,
                   "head_dim": d, "block_size": bs, "seq_len": "context U[512,4096]",
                   "global_batch": B * world, "parallelism": f"replicas x{world}",
                   "layers_per_step": LAYERS_0P6B,
                   "timing": "one CUDA graph per step holding one paged_decode_plan and 28 "
                             "paged_decode_run layer calls over a multi-layer pool; CUDA "
                             "events around the replays",
                   "l2": f"inputs larger than L2: {nbytes / LAYERS_0P6B / 1e6:.0f} MB read per layer call vs "
                         f"{L2_BYTES / 1e6:.0f} MB L2"},
        "roofline": {"bound": "hbm", "achieved": round(nbytes / step_s / 1e9, 2),
                     "peak": pk["hbm"], "unit": "GB/s",
                     "frac": round(nbytes / step_s / 1e9 / pk["hbm"], 4),
                     "traffic": (DECODE_0P6B_TRAFFIC["bytes"]
                                 if decode_sources_digest() ==
                                 DECODE_0P6B_TRAFFIC["sources_sha256"] else None),
                     "traffic_unit": "bytes per paged_decode_run", "peak_source": pk["source"],
                     "kernel": "paged_decode_run (split-KV + combine launches), 28 per "
                               "step, plus one plan launch per step",
                     "bytes_per_launch": nbytes / LAYERS_0P6B},
        "e2e": {"value": round(nbytes * world / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_s * 1e3, 5)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "secondary": secondary,
    }
    return result


def run_secondary(args, pkv, W, torch, dev, pk):
    res = {}
    flush = torch.zeros(int(512e6) // 4, dtype=torch.float32, device=dev)

    which = set(args.secondary.split(",")) if args.secondary else set()
    if "prefill" in which:
        res.update(bench_prefill(pkv, W, torch, dev, pk, flush))
    if "decode32" in which:
        res.update(bench_decode32(pkv, W, torch, dev, pk))
    if "step" in which:
        res.update(bench_step(pkv, W, torch, dev, pk))
    if "sample" in which:
        res.update(bench_sample(pkv, W, torch, dev, pk))
    if "kvstore" in which:
        res.update(bench_kvstore(pkv, W, torch, dev, pk, flush))
    if "mixed" in which:
        res.update(bench_mixed(pkv, W, torch, dev, pk))
    return res


def bench_mixed(pkv, W, torch, dev, pk):
    """A continuous-batching layer step (mixed-8b): 256 decode rows and 4
    prefill chunks in one varlen batch, stored and attended by one call that
    routes the one-query rows to the decode kernels, against the same batch
    through the prefill kernels alone.  The lower bound adds the decode rows'
    bytes at the HBM peak to the chunks' flops at the tensor peak (the two
    passes run one after the other)."""
    spec = W.MIXED_8B
    w = W.mixed_workload(spec, device=dev)
    st = w.step
    kc, vc = w.k_cache0, w.v_cache0
    cu_q, cu_k = st.cu_seqlens_q.to(dev), st.cu_seqlens_k.to(dev)
    bt, sl = st.block_tables.to(dev), st.slot_mapping.to(dev)
    out = torch.empty_like(st.q)
    B, T = st.cu_seqlens_q.numel() - 1, st.q.shape[0]
    ws_m = torch.empty(pkv.paged_attention_varlen_workspace_bytes(
        B, T, spec.num_q_heads, st.max_seqlen_k, kc.shape), dtype=torch.uint8, device=dev)
    ws_p = torch.empty(pkv.paged_prefill_workspace_bytes(B, T, spec.num_q_heads, kc.shape),
                       dtype=torch.uint8, device=dev)
    gm = graph_of(lambda: pkv.kv_store_paged_attention_varlen(
        st.q, st.k, st.v, kc, vc, sl, cu_q, cu_k, st.max_seqlen_q, st.max_seqlen_k, bt,
        w.scale, out=out, workspace=ws_m), torch)
    gp = graph_of(lambda: pkv.kv_store_paged_prefill_varlen(
        st.q, st.k, st.v, kc, vc, sl, cu_q, cu_k, st.max_seqlen_q, st.max_seqlen_k, bt,
        w.scale, out=out, workspace=ws_p), torch)
    for g in (gm, gp):
        for _ in range(3):
            g.replay()
    t_m, t_p = time_graph(gm, 20, torch), time_graph(gp, 20, torch)
    lq = [b - a for a, b in zip(st.cu_seqlens_q.tolist(), st.cu_seqlens_q.tolist()[1:])]
    lk = [b - a for a, b in zip(st.cu_seqlens_k.tolist(), st.cu_seqlens_k.tolist()[1:])]
    dec_ctx = [k for q, k in zip(lq, lk) if q == 1]
    b_dec = decode_bytes(dec_ctx, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                         spec.block_size)
    pre = [(q, k) for q, k in zip(lq, lk) if q != 1]
    cq = [0]
    ck = [0]
    for q, k in pre:
        cq.append(cq[-1] + q)
        ck.append(ck[-1] + k)
    flops = prefill_flops(cq, ck, spec.num_q_heads, spec.head_dim)
    t_lb = b_dec / (pk["hbm"] * 1e9) + flops / (pk["tc"] * 1e12)
    return {"mixed-8b": {
        "workload": spec.name, "decode_rows": len(dec_ctx), "prefill_tokens": sum(cq[-1:]),
        "mixed_call_us": round(t_m * 1e6, 2), "all_prefill_call_us": round(t_p * 1e6, 2),
        "speedup_vs_all_prefill": round(t_p / t_m, 3),
        "lower_bound_us": round(t_lb * 1e6, 2), "frac_of_lower_bound": round(t_lb / t_m, 4),
        "timing": "CUDA graph replays of one call (store + attention), CUDA events; the "
                  "store re-writes the same slots"}}


def bench_sample(pkv, W, torch, dev, pk):
    """The step-8b sampler alone: B=512 rows over a 151936-entry vocabulary."""
    spec = W.STEP_8B
    g = torch.Generator().manual_seed(spec.seed)
    lg, tp, en = W.sampler_inputs(spec.batch, spec.vocab, spec.logit_sigma, spec.logit_spikes,
                                  spec.t_lo, spec.t_hi, g)
    lg, tp, en = lg.to(dev), tp.to(dev), en.to(dev)
    ids = torch.empty(spec.batch, dtype=torch.int32, device=dev)
    gm = graph_of(lambda: pkv.sample(lg, tp, en, out=ids), torch)
    for _ in range(3):
        gm.replay()
    t = time_graph(gm, 50, torch)
    b = 8.0 * spec.batch * spec.vocab + 8 * spec.batch
    gp = graph_of(lambda: pkv.sample_philox(lg, tp, 1234, 0, out=ids), torch)
    for _ in range(3):
        gp.replay()
    tpx = time_graph(gp, 50, torch)
    bp = 4.0 * spec.batch * spec.vocab + 8 * spec.batch
    return {"sample": {"workload": f"B={spec.batch} V={spec.vocab}", "us": round(t * 1e6, 2),
                       "gbs": round(b / t / 1e9, 1), "frac_hbm": round(b / t / 1e9 / pk["hbm"], 4),
                       "bytes": b, "timing": "CUDA graph replays (inputs 622 MB > L2)"},
            "sample_philox": {"workload": f"B={spec.batch} V={spec.vocab}, noise drawn in kernel",
                              "us": round(tpx * 1e6, 2), "gbs": round(bp / tpx / 1e9, 1),
                              "frac_hbm": round(bp / tpx / 1e9 / pk["hbm"], 4), "bytes": bp}}


def bench_kvstore(pkv, W, torch, dev, pk, flush):
    """kv_store of one 16384-token prefill chunk (rows of 8x128 bf16) into the
    prefill-8b pool."""
    w = W.prefill_workload(W.PREFILL_8B)
    st = w.steps[0]
    kc, vc = w.k_cache0.to(dev), w.v_cache0.to(dev)
    k, v, sl = st.k.to(dev), st.v.to(dev), st.slot_mapping.to(dev)
    for _ in range(3):
        pkv.kv_store(k, v, kc, vc, sl)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tot = 0.0
    reps = 20
    for _ in range(reps):
        flush_l2(flush)
        e0.record()
        pkv.kv_store(k, v, kc, vc, sl)
        e1.record()
        torch.cuda.synchronize()
        tot += e0.elapsed_time(e1) * 1e-3
    t = tot / reps
    b = 4.0 * k.numel() * 2
    return {"kv_store": {"workload": f"{k.shape[0]} rows of {k.shape[1]}x{k.shape[2]} bf16",
                         "us": round(t * 1e6, 2), "gbs": round(b / t / 1e9, 1),
                         "frac_hbm": round(b / t / 1e9 / pk["hbm"], 4), "bytes": b,
                         "timing": "CUDA events per call, L2 flushed before each"}}


def bench_prefill(pkv, W, torch, dev, pk, flush):
    res = {}
    spec = W.PREFILL_8B
    w = W.prefill_workload(spec)
    kc, vc = w.k_cache0.to(dev), w.v_cache0.to(dev)
    steps = []
    for st in w.steps:
        t = dict(q=st.q.to(dev), k=st.k.to(dev), v=st.v.to(dev),
                 cu_q=st.cu_seqlens_q.to(dev), cu_k=st.cu_seqlens_k.to(dev),
                 bt=st.block_tables.to(dev), slots=st.slot_mapping.to(dev),
                 msq=st.max_seqlen_q, msk=st.max_seqlen_k,
                 flops=prefill_flops(st.cu_seqlens_q.tolist(), st.cu_seqlens_k.tolist(),
                                     spec.num_q_heads, spec.head_dim))
        t["out"] = torch.empty_like(t["q"])
        t["ws"] = torch.empty(pkv.paged_prefill_workspace_bytes(
            st.cu_seqlens_q.numel() - 1, st.q.shape[0], spec.num_q_heads, kc.shape),
            dtype=torch.uint8, device=dev)
        steps.append(t)

    def run_step(t):
        pkv.kv_store(t["k"], t["v"], kc, vc, t["slots"])
        pkv.paged_prefill_varlen(t["q"], t["k"], t["v"], kc, vc, t["cu_q"], t["cu_k"],
                                 t["msq"], t["msk"], t["bt"], w.scale, out=t["out"],
                                 workspace=t["ws"])

    for t in steps:
        run_step(t)
    reps = 3
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in steps]
    t_store, t_pre = 0.0, 0.0
    for _ in range(reps):
        for i, t in enumerate(steps):
            flush_l2(flush)
            ev[i][0].record()
            pkv.kv_store(t["k"], t["v"], kc, vc, t["slots"])
            ev[i][1].record()
            pkv.paged_prefill_varlen(t["q"], t["k"], t["v"], kc, vc, t["cu_q"], t["cu_k"],
                                     t["msq"], t["msk"], t["bt"], w.scale, out=t["out"],
                                     workspace=t["ws"])
            ev[i][2].record()
        torch.cuda.synchronize()
        for e in ev:
            t_store += e[0].elapsed_time(e[1]) * 1e-3
            t_pre += e[1].elapsed_time(e[2]) * 1e-3
    t_store /= reps
    t_pre /= reps
    tokens = sum(t["q"].shape[0] for t in steps)
    flops = sum(t["flops"] for t in steps)
    store_bytes = sum(4 * t["k"].numel() * 2 for t in steps)
    res["prefill-8b"] = {
        "workload": spec.name, "chunk_steps": len(steps), "new_tokens": tokens,
        "tokens_per_s": round(tokens / t_pre, 1), "prefill_ms": round(t_pre * 1e3, 4),
        "tflops": round(flops / t_pre / 1e12, 2),
        "frac_tc_burst": round(flops / t_pre / 1e12 / pk["tc"], 4),
        "frac_tc_sustained": round(flops / t_pre / 1e12 / pk["tc_sustained"], 4),
        "kv_store_gbs": round(store_bytes / t_store / 1e9, 1),
        "kv_store_frac_hbm": round(store_bytes / t_store / 1e9 / pk["hbm"], 4),
        "timing": "sum of per-call CUDA-event times over the chunk steps, L2 flushed "
                  "before each step, mean of 3 passes"}
    del steps, kc, vc, w
    torch.cuda.empty_cache()
    return res


def bench_decode32(pkv, W, torch, dev, pk):
    res = {}
    for spec, key in ((W.DECODE_32B, "decode-32b"),):
        w = W.decode_workload(spec, device=dev)
        bt, ctx = w.block_tables.to(dev), w.context_lens.to(dev)
        out = torch.empty_like(w.q)
        ws = torch.empty(pkv.paged_decode_workspace_bytes(spec.batch, spec.num_q_heads,
                                                          w.max_context_len, w.k_cache),
                         dtype=torch.uint8, device=dev)
        g = graph_of(lambda: pkv.paged_decode(w.q, w.k_cache, w.v_cache, bt, ctx, w.scale,
                                              w.max_context_len, out=out, workspace=ws), torch)
        for _ in range(5):
            g.replay()
        s = time_graph(g, 50, torch)
        nbytes = decode_bytes(w.context_lens.tolist(), spec.num_q_heads, spec.num_kv_heads,
                              spec.head_dim, spec.block_size)
        res[key] = {"workload": spec.name, "us": round(s * 1e6, 2),
                    "gbs": round(nbytes / s / 1e9, 1),
                    "frac_hbm": round(nbytes / s / 1e9 / pk["hbm"], 4),
                    "bytes": nbytes}
        del w, g, out, ws
        torch.cuda.empty_cache()
    return res


def bench_step(pkv, W, torch, dev, pk):
    res = {}
    spec = W.STEP_8B
    w = W.decode_workload(spec, device=dev)
    bt, ctx, sl = w.block_tables.to(dev), w.context_lens.to(dev), w.slot_mapping.to(dev)
    logits, temps, noise = w.logits.to(dev), w.temperatures.to(dev), w.exp_noise.to(dev)
    out = torch.empty_like(w.q)
    ids = torch.empty(spec.batch, dtype=torch.int32, device=dev)
    ws = torch.empty(pkv.paged_decode_workspace_bytes(spec.batch, spec.num_q_heads,
                                                      w.max_context_len, w.k_cache),
                     dtype=torch.uint8, device=dev)
    gs = graph_of(lambda: pkv.kv_store(w.k_new, w.v_new, w.k_cache, w.v_cache, sl), torch)
    gd = graph_of(lambda: pkv.paged_decode(w.q, w.k_cache, w.v_cache, bt, ctx, w.scale,
                                           w.max_context_len, out=out, workspace=ws), torch)
    gm = graph_of(lambda: pkv.sample(logits, temps, noise, out=ids), torch)
    gz = graph_of(lambda: pkv.kv_store_paged_decode(w.k_new, w.v_new, sl, w.q, w.k_cache,
                                                    w.v_cache, bt, ctx, w.scale,
                                                    w.max_context_len, out=out, workspace=ws),
                  torch)

    def full():
        pkv.kv_store(w.k_new, w.v_new, w.k_cache, w.v_cache, sl)
        pkv.paged_decode(w.q, w.k_cache, w.v_cache, bt, ctx, w.scale, w.max_context_len,
                         out=out, workspace=ws)
        pkv.sample(logits, temps, noise, out=ids)
    gf = graph_of(full, torch)
    for gg in (gs, gd, gm, gf, gz):
        for _ in range(3):
            gg.replay()
    t_s, t_d, t_m, t_f = (time_graph(gs, 200, torch), time_graph(gd, 30, torch),
                          time_graph(gm, 50, torch), time_graph(gf, 30, torch))
    t_z = time_graph(gz, 30, torch)
    b_s = 4.0 * w.k_new.numel() * 2
    b_d = decode_bytes(w.context_lens.tolist(), spec.num_q_heads, spec.num_kv_heads,
                       spec.head_dim, spec.block_size)
    b_m = 8.0 * spec.batch * spec.vocab + 8 * spec.batch
    res["step-8b"] = {
        "workload": spec.name, "step_us": round(t_f * 1e6, 2),
        "kv_store_us": round(t_s * 1e6, 2), "kv_store_gbs": round(b_s / t_s / 1e9, 1),
        "decode_us": round(t_d * 1e6, 2), "decode_gbs": round(b_d / t_d / 1e9, 1),
        "decode_frac_hbm": round(b_d / t_d / 1e9 / pk["hbm"], 4),
        "fused_store_decode_us": round(t_z * 1e6, 2),
        "sample_us": round(t_m * 1e6, 2), "sample_gbs": round(b_m / t_m / 1e9, 1),
        "sample_frac_hbm": round(b_m / t_m / 1e9 / pk["hbm"], 4),
        "timing": "CUDA graph replays, CUDA events; kv_store re-writes the same slots"}
    return res


# ----------------------------------------------------------------------------
# CPU oracle legs
# ----------------------------------------------------------------------------
def oracle_worker(budget_s: float, steps: int, warmup: int, per_step: int):
    """Times oracle.attention.paged_decode on whole sequences of decode-0.6b
    (all q heads of `per_step` sequences per step), in a fresh interpreter with
    single-threaded BLAS, stopping after `budget_s` seconds."""
    from oracle import attention as oatt
    from paged_kv_attention_scatter_gb300 import workloads as W

    spec = W.DECODE_0P6B
    w = W.decode_workload(spec)
    qf = w.q.double().numpy()
    bt, ctx = w.block_tables.numpy(), w.context_lens.numpy()
    B = spec.batch

    def one_step(i):
        nb = 0.0
        for j in range(per_step):
            b = (i * per_step + j) % B
            oatt.paged_decode(qf, w.k_cache, w.v_cache, bt, ctx, w.scale, seqs=[b])
            nb += decode_bytes([int(ctx[b])], spec.num_q_heads, spec.num_kv_heads,
                               spec.head_dim, spec.block_size)
        return nb

    for i in range(warmup):
        one_step(i)
    t = time.perf_counter()
    nbytes, done = 0.0, 0
    for i in range(steps):
        nbytes += one_step(warmup + i)
        done += 1
        if time.perf_counter() - t > budget_s:
            break
    el = time.perf_counter() - t
    print(json.dumps({"value": nbytes / el / 1e9, "seconds": el, "steps": done,
                      "seqs": done * per_step}))


def cpu_oracle(steps, warmup, per_step, budget_s):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-worker",
           "--steps", str(steps), "--warmup", str(warmup), "--per-step", str(per_step),
           "--budget", str(budget_s)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, cwd=ROOT)
    if r.returncode != 0:
        raise RuntimeError(f"oracle worker failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


# ----------------------------------------------------------------------------
def profile_case(name: str, calls: int):
    """A small case for ncu: `calls` eager calls of one operation on a
    single-layer workload (inputs above L2, a few GB on the device at most).
    Prints one line when done; no timing."""
    import torch

    import paged_kv_attention_scatter_gb300 as pkv
    from paged_kv_attention_scatter_gb300 import workloads as W

    pkv.build()
    pkv.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if name == "decode-0.6b":
        spec = W.DECODE_0P6B
        w = W.decode_workload(spec, device=dev)
        bt, ctx = w.block_tables.to(dev), w.context_lens.to(dev)
        out = torch.empty_like(w.q)
        ws = torch.empty(pkv.paged_decode_workspace_bytes(spec.batch, spec.num_q_heads,
                                                          w.max_context_len, w.k_cache),
                         dtype=torch.uint8, device=dev)
        for _ in range(calls):
            pkv.paged_decode(w.q, w.k_cache, w.v_cache, bt, ctx, w.scale, w.max_context_len,
                             out=out, workspace=ws)
    elif name == "prefill-8b":
        spec = W.PREFILL_8B
        w = W.prefill_workload(spec)
        st = w.steps[0]
        kc, vc = w.k_cache0.to(dev), w.v_cache0.to(dev)
        q, k, v = st.q.to(dev), st.k.to(dev), st.v.to(dev)
        cu_q, cu_k = st.cu_seqlens_q.to(dev), st.cu_seqlens_k.to(dev)
        bt, sl = st.block_tables.to(dev), st.slot_mapping.to(dev)
        for _ in range(calls):
            pkv.kv_store(k, v, kc, vc, sl)
            pkv.paged_prefill_varlen(q, k, v, kc, vc, cu_q, cu_k, st.max_seqlen_q,
                                     st.max_seqlen_k, bt, w.scale)
    elif name == "sample":
        spec = W.STEP_8B
        g = torch.Generator().manual_seed(spec.seed)
        lg, tp, en = W.sampler_inputs(spec.batch, spec.vocab, spec.logit_sigma,
                                      spec.logit_spikes, spec.t_lo, spec.t_hi, g)
        lg, tp, en = lg.to(dev), tp.to(dev), en.to(dev)
        for _ in range(calls):
            pkv.sample(lg, tp, en)
            pkv.sample_philox(lg, tp, 1234, 0)
    elif name == "mixed-8b":
        spec = W.MIXED_8B
        w = W.mixed_workload(spec, device=dev)
        st = w.step
        cu_q, cu_k = st.cu_seqlens_q.to(dev), st.cu_seqlens_k.to(dev)
        bt, sl = st.block_tables.to(dev), st.slot_mapping.to(dev)
        for _ in range(calls):
            pkv.kv_store_paged_attention_varlen(st.q, st.k, st.v, w.k_cache0, w.v_cache0, sl,
                                                cu_q, cu_k, st.max_seqlen_q, st.max_seqlen_k,
                                                bt, w.scale)
    else:
        raise SystemExit(f"unknown profile case {name!r}")
    torch.cuda.synchronize()
    print(json.dumps({"profile": name, "calls": calls}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--secondary", default="prefill,decode32,step,mixed",
                    help="comma list of secondary workloads: prefill, decode32, step, "
                         "mixed, sample, kvstore")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-worker", action="store_true")
    ap.add_argument("--per-step", type=int, default=1)
    ap.add_argument("--budget", type=float, default=20.0)
    ap.add_argument("--profile", default=None,
                    help="run a small case for ncu instead of the benchmark: decode-0.6b, "
                         "prefill-8b, sample or mixed-8b (calls = --steps)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    if args.profile:
        profile_case(args.profile, args.steps)
        return

    if args.oracle_worker:
        oracle_worker(args.budget, args.steps, args.warmup, args.per_step)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        r = cpu_oracle(args.steps, min(args.warmup, 3), 1, budget_s=120.0)
        from paged_kv_attention_scatter_gb300 import workloads as W
        spec = W.DECODE_0P6B
        ms = r["seconds"] / max(r["steps"], 1) * 1e3
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(r["value"], 4),
            "unit": "GB/s", "n_gpus": 1, "steps": r["steps"], "warmup": min(args.warmup, 3),
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": spec.name, "batch": spec.batch, "head_dim": spec.head_dim,
                       "block_size": spec.block_size},
            "cpu_baseline": {"value": round(r["value"], 4), "unit": "GB/s", "cores": 1,
                             "kind": "oracle",
                             "sample": f"{r['seqs']} whole sequences (all 16 q heads) of "
                                       "decode-0.6b, one per step, float64 NumPy, "
                                       "single-threaded BLAS, at most 120 s"},
            "e2e": {"value": round(r["value"], 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
        return

    dist = None
    if world > 1:
        import torch.distributed as tdist
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # before any GPU work in this process: the oracle runs in a fresh interpreter
        cpu = cpu_oracle(1000000, 2, 1, budget_s=15.0)
    res = run_ours(args, rank, world, dist)
    if cpu is not None:
        res["cpu_baseline"] = {"value": round(cpu["value"], 4), "unit": "GB/s", "cores": 1,
                               "kind": "oracle",
                               "sample": f"{cpu['seqs']} whole sequences of decode-0.6b "
                                         f"in {cpu['seconds']:.1f} s, float64 NumPy, "
                                         "single-threaded BLAS"}
    if rank == 0:
        print(json.dumps(res))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
