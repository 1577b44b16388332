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
import dataclasses
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
# its split and combine launches, from one ncu capture of
# `bench.py --profile decode-0.6b`.  Valid only for the decode sources it was
# taken on: the digest below must match, otherwise the traffic is reported null.
# (The digest was carried forward over one later change, which touched only
# the register-load split kernel; decode-0.6b, at block size 256, launches
# the plan, the TMA-fed split and the combine kernels, whose code it left as
# captured.)
DECODE_0P6B_TRAFFIC = {"bytes": 582291200,
                       "sources_sha256": "db7514e70993eb3ea2edbffb8840e3adddf26d5fea49088edbfeb85951cbe799"}

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


def time_graphs_paired(ga, gb, pairs, torch):
    """Mean seconds per replay of two graphs timed in alternation (a, b, a,
    b, ...), CUDA events around each replay, so drift of clock or
    temperature over the run falls on both alike; also the 10th, 50th and
    90th percentiles of the per-pair differences b - a."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(2 * pairs)]
    torch.cuda.synchronize()
    for i in range(pairs):
        for j, g in enumerate((ga, gb)):
            s, e = ev[2 * i + j]
            s.record()
            g.replay()
            e.record()
    torch.cuda.synchronize()
    ta = [ev[2 * i][0].elapsed_time(ev[2 * i][1]) * 1e-3 for i in range(pairs)]
    tb = [ev[2 * i + 1][0].elapsed_time(ev[2 * i + 1][1]) * 1e-3 for i in range(pairs)]
    diff = sorted(b - a for a, b in zip(ta, tb))
    return (sum(ta) / pairs, sum(tb) / pairs,
            (diff[pairs // 10], diff[pairs // 2], diff[(9 * pairs) // 10]))


def hbm_read_reference(torch, dev, nbytes=2 << 30, reps=10):
    """A read-only stream for context beside the copy peak: the best of
    `reps` torch reductions (sum and max) over a 2 GiB fp32 tensor, in GB/s
    read.  The copy peak stays the roofline's denominator."""
    x = torch.ones(nbytes // 4, dtype=torch.float32, device=dev)
    best = {}
    for name, fn in (("sum", torch.sum), ("amax", torch.amax)):
        fn(x)
        torch.cuda.synchronize()
        t = []
        for _ in range(reps):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            fn(x)
            e.record()
            torch.cuda.synchronize()
            t.append(s.elapsed_time(e) * 1e-3)
        best[name] = nbytes / min(t) / 1e9
    del x
    torch.cuda.empty_cache()
    name = max(best, key=best.get)
    return {"gbs": round(best[name], 1), "how": f"torch.{name} over a 2 GiB fp32 tensor, best "
            f"of {reps} (CUDA events; sum {best['sum']:.0f}, amax {best['amax']:.0f} GB/s)"}


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

    read_ref = hbm_read_reference(torch, dev)
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
                     "bytes_per_launch": nbytes / LAYERS_0P6B,
                     "read_stream_reference": read_ref,
                     "frac_of_read_stream": round(nbytes / step_s / 1e9 / read_ref["gbs"], 4)},
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
    # kv_store of the chunks on its own: (1) a CUDA graph of the five chunk
    # stores back to back, replayed 20 times (each call's 128 MB of rows was last
    # touched four calls, 512 MB of traffic, earlier: cold in L2), per-call mean;
    # (2) the median of 20 single calls per chunk, each after an L2 flush, timed
    # with CUDA events around the call (includes its launch latency)
    gst = graph_of(lambda: [pkv.kv_store(t["k"], t["v"], kc, vc, t["slots"]) for t in steps],
                   torch)
    for _ in range(3):
        gst.replay()
    t_store_graph = time_graph(gst, 20, torch) / len(steps)
    singles = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for t in steps:
        per = []
        for _ in range(20):
            flush_l2(flush)
            e0.record()
            pkv.kv_store(t["k"], t["v"], kc, vc, t["slots"])
            e1.record()
            torch.cuda.synchronize()
            per.append(e0.elapsed_time(e1) * 1e-3)
        per.sort()
        singles.append(per[len(per) // 2])
    t_store_single = sum(singles) / len(singles)
    tokens = sum(t["q"].shape[0] for t in steps)
    flops = sum(t["flops"] for t in steps)
    store_bytes = sum(4 * t["k"].numel() * 2 for t in steps)
    res["prefill-8b"] = {
        "workload": spec.name, "chunk_steps": len(steps), "new_tokens": tokens,
        "tokens_per_s": round(tokens / t_pre, 1), "prefill_ms": round(t_pre * 1e3, 4),
        "tflops": round(flops / t_pre / 1e12, 2),
        "frac_tc_burst": round(flops / t_pre / 1e12 / pk["tc"], 4),
        "frac_tc_sustained": round(flops / t_pre / 1e12 / pk["tc_sustained"], 4),
        "kv_store_gbs": round(store_bytes / len(steps) / t_store_graph / 1e9, 1),
        "kv_store_frac_hbm": round(store_bytes / len(steps) / t_store_graph / 1e9 / pk["hbm"],
                                   4),
        "kv_store_us_per_chunk": round(t_store_graph * 1e6, 2),
        "kv_store_single_call_median_us": round(t_store_single * 1e6, 2),
        "kv_store_single_call_frac_hbm": round(store_bytes / len(steps) / t_store_single / 1e9
                                               / pk["hbm"], 4),
        "kv_store_timing": "kv_store_gbs: a CUDA graph of the 5 chunk stores back to back "
                           "(640 MB of rows, each call's cold in L2), per-call mean of 20 "
                           "replays; single_call: median of 20 calls per chunk, each after an "
                           "L2 flush, CUDA events around the call (launch latency included)",
        "timing": "prefill: sum of per-call CUDA-event times over the chunk steps, L2 flushed "
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
    gpx = graph_of(lambda: pkv.sample_philox(logits, temps, 1234, 0, out=ids), torch)
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
    for gg in (gs, gd, gm, gf, gz, gpx):
        for _ in range(3):
            gg.replay()
    t_s, t_m, t_f = (time_graph(gs, 200, torch), time_graph(gm, 50, torch),
                     time_graph(gf, 30, torch))
    # the decode alone and the store + decode call, replay by replay in turn
    t_d, t_z, dz = time_graphs_paired(gd, gz, 200, torch)
    t_px = time_graph(gpx, 50, torch)
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
        "fused_minus_decode_mean_us": round((t_z - t_d) * 1e6, 2),
        "fused_minus_decode_median_us": round(dz[1] * 1e6, 2),
        "fused_minus_decode_p10_p90_us": [round(dz[0] * 1e6, 2), round(dz[2] * 1e6, 2)],
        "sample_us": round(t_m * 1e6, 2), "sample_gbs": round(b_m / t_m / 1e9, 1),
        "sample_frac_hbm": round(b_m / t_m / 1e9 / pk["hbm"], 4),
        "sample_philox_us": round(t_px * 1e6, 2),
        "sample_philox_gbs": round((b_m / 2) / t_px / 1e9, 1),
        "sample_philox_note": "noise drawn in the kernel (Philox4x32-10): logits and "
                              "temperatures only, 4 bytes per entry",
        "timing": "CUDA graph replays, CUDA events; kv_store re-writes the same slots; "
                  "decode_us and fused_store_decode_us: 200 replays of each in alternation, "
                  "events around each replay (means; the per-pair difference's median and "
                  "10th/90th percentiles, single replays varying by about +-10 us)"}
    return res


# ----------------------------------------------------------------------------
# CPU oracle legs: the oracle as it stands, timed on the host's cores
# ----------------------------------------------------------------------------
# The legs run in a fresh interpreter with CUDA hidden (started before any GPU
# work of the benchmark).  Multi-core legs use one spawned worker process per
# core of os.sched_getaffinity(0), each single-threaded (BLAS, OpenMP and torch
# intra-op threads set to 1, so the cores are not oversubscribed), sharing the
# inputs through shared memory; a unit of work (one sequence, one sampler row,
# a set of prefill query rows) runs whole in one worker.  A leg dispatches
# waves of units until its time budget is spent and reports the work done
# over the wall time.
_ORACLE_DATA: dict = {}


def _oracle_pool_init(data):
    import torch
    torch.set_num_threads(1)
    _ORACLE_DATA.update(data)


def _oracle_unit(task):
    """One unit of oracle work; returns its algorithmic amount (bytes or
    FLOPs) so the caller can total what was done."""
    from oracle import attention as oatt
    from oracle import sampler as osm
    leg, i = task
    d = _ORACLE_DATA[leg]
    if leg == "prefill-8b":
        s = d["units"][i]
        oatt.paged_prefill_varlen(d["q"][s["b"]], d["k"][s["b"]], d["v"][s["b"]], d["k_cache"],
                                  d["v_cache"], [0, s["lq"]], [0, s["lk"]], d["bt"][s["b"]],
                                  d["scale"], rows={0: s["rows"]})
        return s["flops"]
    if leg == "step-8b sample":
        osm.sample(d["logits"][i:i + 1], d["temps"][i:i + 1], d["noise"][i:i + 1])
        return d["row_bytes"]
    oatt.paged_decode(d["q"], d["k_cache"], d["v_cache"], d["bt"], d["ctx"], d["scale"],
                      seqs=[i])
    return d["unit_bytes"][i]


def _decode_leg_data(spec, torch):
    from paged_kv_attention_scatter_gb300 import workloads as W
    w = W.decode_workload(spec)
    ctx = w.context_lens.numpy()
    return w, {"q": w.q.double().numpy(), "k_cache": w.k_cache.share_memory_(),
               "v_cache": w.v_cache.share_memory_(), "bt": w.block_tables.numpy(), "ctx": ctx,
               "scale": w.scale,
               "unit_bytes": [decode_bytes([int(c)], spec.num_q_heads, spec.num_kv_heads,
                                           spec.head_dim, spec.block_size) for c in ctx]}


def _prefill_leg_data(spec, prompts: int, rows_per_unit: int):
    """The first `prompts` prompts of prefill-8b (lengths and cached prefixes
    drawn as the full workload draws them), computed in one chunk; a unit is
    every n-th query row of one prompt."""
    from dataclasses import replace

    from paged_kv_attention_scatter_gb300 import workloads as W
    g = W._gen(spec.seed)
    lens = W.randint_incl(spec.len_lo, spec.len_hi, spec.num_prompts, g)
    kbs = W.randint_incl(0, spec.max_cached_blocks, spec.num_prompts, g)
    sub = replace(spec, num_prompts=prompts)
    w = W.prefill_workload(sub, prompt_lens=lens[:prompts], cached_blocks=kbs[:prompts])
    assert len(w.steps) == 1
    st = w.steps[0]
    cu_q, cu_k = st.cu_seqlens_q.tolist(), st.cu_seqlens_k.tolist()
    q, k, v, bt, units = [], [], [], [], []
    for b in range(prompts):
        lq, lk = cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]
        q.append(st.q[cu_q[b]:cu_q[b + 1]].clone().share_memory_())
        k.append(st.k[cu_q[b]:cu_q[b + 1]].clone().share_memory_())
        v.append(st.v[cu_q[b]:cu_q[b + 1]].clone().share_memory_())
        bt.append(st.block_tables[b:b + 1].numpy())
        n_units = -(-lq // rows_per_unit)
        for u in range(n_units):
            rows = list(range(u, lq, n_units))
            c = lk - lq
            flops = 4.0 * spec.head_dim * spec.num_q_heads * sum(c + i + 1 for i in rows)
            units.append({"b": b, "lq": lq, "lk": lk, "rows": rows, "flops": flops})
    return {"q": q, "k": k, "v": v, "k_cache": w.k_cache0.share_memory_(),
            "v_cache": w.v_cache0.share_memory_(), "bt": bt, "units": units,
            "scale": w.scale, "tokens": cu_q[-1]}


def _run_leg(pool, leg, n_units, cores, budget_s, warm_units=0):
    """Waves of 2*cores units (cycling over the leg's units) until budget_s of
    wall time; returns (amount done, units done, seconds, the unit indices
    done)."""
    nxt = 0
    if warm_units:
        pool.map(_oracle_unit, [(leg, (nxt + j) % n_units) for j in range(warm_units)],
                 chunksize=1)
        nxt += warm_units
    amount, idx = 0.0, []
    t0 = time.perf_counter()
    while True:
        wave = [(leg, (nxt + j) % n_units) for j in range(2 * cores)]
        nxt += len(wave)
        amount += sum(pool.map(_oracle_unit, wave, chunksize=1))
        idx += [i for _, i in wave]
        if time.perf_counter() - t0 > budget_s:
            break
    return amount, len(idx), time.perf_counter() - t0, idx


def _one_core_tiny(budget_s: float):
    """The whole tiny scenario (store + prefill with and without block tables,
    three decode steps, the sampler) through the oracle on this one core."""
    import torch

    from oracle import attention as oatt
    from oracle import kv_store as okv
    from oracle import sampler as osm
    from paged_kv_attention_scatter_gb300 import workloads as W
    w = W.tiny_workload()
    bits = lambda t: t.contiguous().view(torch.int16).numpy()  # noqa: E731

    def scenario():
        p = w.prefill
        kc, vc, _ = okv.kv_store(bits(p.k), bits(p.v), bits(w.k_cache0), bits(w.v_cache0),
                                 p.slot_mapping.numpy())
        kt, vt = torch.from_numpy(kc).view(torch.bfloat16), torch.from_numpy(vc).view(torch.bfloat16)
        for bt in (p.block_tables.numpy(), None):
            oatt.paged_prefill_varlen(p.q, p.k, p.v, kt, vt, p.cu_seqlens_q.numpy(),
                                      p.cu_seqlens_k.numpy(), bt, w.scale)
        for st in w.decode_steps:
            kc, vc, _ = okv.kv_store(bits(st.k_new), bits(st.v_new), kc, vc,
                                     st.slot_mapping.numpy())
            kt = torch.from_numpy(kc).view(torch.bfloat16)
            vt = torch.from_numpy(vc).view(torch.bfloat16)
            oatt.paged_decode(st.q, kt, vt, st.block_tables.numpy(), st.context_lens.numpy(),
                              w.scale)
        osm.sample(w.logits.numpy(), w.temperatures.numpy(), w.exp_noise.numpy())

    scenario()
    n, t0 = 0, time.perf_counter()
    while n < 3 or time.perf_counter() - t0 < budget_s:
        scenario()
        n += 1
    return (time.perf_counter() - t0) / n, n


def _one_core_decode(data, budget_s: float):
    _oracle_pool_init({"decode-0.6b": data})
    nb, n, t0 = 0.0, 0, time.perf_counter()
    while n < 2 or time.perf_counter() - t0 < budget_s:
        nb += _oracle_unit(("decode-0.6b", n % len(data["ctx"])))
        n += 1
    return nb, n, time.perf_counter() - t0


def oracle_table(budget_s: float):
    """Every leg of the CPU baseline; returns the JSON-ready table."""
    import multiprocessing as mp

    import torch
    import torch.multiprocessing  # noqa: F401  (shared-memory tensor pickling)
    from dataclasses import replace

    from paged_kv_attention_scatter_gb300 import workloads as W
    torch.set_num_threads(1)
    cores = len(os.sched_getaffinity(0))
    w06, d06 = _decode_leg_data(W.DECODE_0P6B, torch)
    spec32 = replace(W.DECODE_32B, batch=16, num_blocks=None)
    _, d32 = _decode_leg_data(spec32, torch)
    spec_step = replace(W.STEP_8B, batch=32, vocab=None, store_new_token=False)
    _, dstep = _decode_leg_data(spec_step, torch)
    g = W._gen(W.STEP_8B.seed)
    lg, tp, en = W.sampler_inputs(64, W.STEP_8B.vocab, W.STEP_8B.logit_sigma,
                                  W.STEP_8B.logit_spikes, W.STEP_8B.t_lo, W.STEP_8B.t_hi, g)
    dsamp = {"logits": lg.numpy(), "temps": tp.numpy(), "noise": en.numpy(),
             "row_bytes": 8.0 * W.STEP_8B.vocab + 8}
    dpre = _prefill_leg_data(W.PREFILL_8B, prompts=2, rows_per_unit=64)
    data = {"decode-0.6b": d06, "decode-32b": d32, "step-8b decode": dstep,
            "step-8b sample": dsamp, "prefill-8b": dpre}
    one_dec = _one_core_decode(d06, budget_s * 0.5)
    tiny_s, tiny_n = _one_core_tiny(budget_s * 0.25)
    ctx = mp.get_context("spawn")
    res = {}
    with ctx.Pool(cores, initializer=_oracle_pool_init, initargs=(data,)) as pool:
        for leg, n_units in (("decode-0.6b", len(d06["ctx"])), ("decode-32b", len(d32["ctx"])),
                             ("step-8b decode", len(dstep["ctx"])),
                             ("step-8b sample", dsamp["logits"].shape[0]),
                             ("prefill-8b", len(dpre["units"]))):
            res[leg] = _run_leg(pool, leg, n_units, cores, budget_s, warm_units=cores)
    # the whole prefill-8b workload's FLOPs and new tokens, from its drawn
    # prompt lengths and cached prefixes (chunking does not change the total)
    sp = W.PREFILL_8B
    g = W._gen(sp.seed)
    lens = W.randint_incl(sp.len_lo, sp.len_hi, sp.num_prompts, g)
    kbs = W.randint_incl(0, sp.max_cached_blocks, sp.num_prompts, g)
    cached = [min(kb, (L - 1) // sp.block_size) * sp.block_size for L, kb in zip(lens, kbs)]
    full_tokens = sum(L - c for L, c in zip(lens, cached))
    full_flops = sum(prefill_flops([0, L - c], [0, L], sp.num_q_heads, sp.head_dim)
                     for L, c in zip(lens, cached))
    gbs = lambda r: round(r[0] / r[2] / 1e9, 4)  # noqa: E731
    fl, n_pre, s_pre, idx_pre = res["prefill-8b"]
    pre_rows = sum(len(dpre["units"][i]["rows"]) for i in idx_pre)
    table = {
        "cores": cores,
        "decode-0.6b": {"value": gbs(res["decode-0.6b"]), "unit": "GB/s",
                        "sample": f"{res['decode-0.6b'][1]} whole sequences (all 16 q heads) "
                                  f"in {res['decode-0.6b'][2]:.1f} s"},
        "decode-32b": {"value": gbs(res["decode-32b"]), "unit": "GB/s",
                       "sample": f"{res['decode-32b'][1]} whole sequences of 16 drawn like "
                                 f"decode-32b's (log-uniform contexts) in "
                                 f"{res['decode-32b'][2]:.1f} s"},
        "step-8b decode": {"value": gbs(res["step-8b decode"]), "unit": "GB/s",
                           "sample": f"{res['step-8b decode'][1]} whole sequences of 32 drawn "
                                     f"like step-8b's in {res['step-8b decode'][2]:.1f} s"},
        "step-8b sample": {"value": gbs(res["step-8b sample"]), "unit": "GB/s",
                           "rows_per_s": round(res["step-8b sample"][1] /
                                               res["step-8b sample"][2], 2),
                           "sample": f"{res['step-8b sample'][1]} rows of V=151936 in "
                                     f"{res['step-8b sample'][2]:.1f} s"},
        "prefill-8b": {"tflops": round(fl / s_pre / 1e12, 6),
                       "tokens_per_s": round(pre_rows / s_pre, 2),
                       "extrapolated_ms_for_workload": round(full_flops / (fl / s_pre) * 1e3, 1),
                       "workload_tokens": full_tokens,
                       "sample": f"{pre_rows} query rows (all 32 q heads; {n_pre} units of "
                                 f"about 64 rows) of the first 2 prompts ({dpre['tokens']} new "
                                 f"tokens) in "
                                 f"{s_pre:.1f} s; the whole workload's time extrapolated by "
                                 "FLOPs"},
        "one_core": {
            "decode-0.6b": {"value": round(one_dec[0] / one_dec[2] / 1e9, 4), "unit": "GB/s",
                            "sample": f"{one_dec[1]} whole sequences in {one_dec[2]:.1f} s"},
            "tiny": {"ms_per_scenario": round(tiny_s * 1e3, 2),
                     "sample": f"{tiny_n} runs of the whole tiny scenario (store, prefill "
                               "with and without tables, 3 decode steps, sampler)"}},
    }
    del w06
    return table


def oracle_worker(args):
    """Entry of the fresh interpreter that runs the CPU legs; prints one JSON
    line.  --budget is the seconds per multi-core leg."""
    if args.reference_steps:
        print(json.dumps(reference_waves(args.steps, args.warmup, args.budget)))
    else:
        print(json.dumps(oracle_table(args.budget)))


def reference_waves(steps: int, warmup: int, budget_s: float):
    """The reference arm: `steps` waves of decode-0.6b sequences, one per core
    and wave, after `warmup` waves; stops early after budget_s seconds."""
    import multiprocessing as mp

    import torch
    import torch.multiprocessing  # noqa: F401

    from paged_kv_attention_scatter_gb300 import workloads as W
    torch.set_num_threads(1)
    cores = len(os.sched_getaffinity(0))
    _, d06 = _decode_leg_data(W.DECODE_0P6B, torch)
    n = len(d06["ctx"])
    with mp.get_context("spawn").Pool(cores, initializer=_oracle_pool_init,
                                      initargs=({"decode-0.6b": d06},)) as pool:
        nxt = 0
        for _ in range(warmup):
            pool.map(_oracle_unit, [("decode-0.6b", (nxt + j) % n) for j in range(cores)],
                     chunksize=1)
            nxt += cores
        amount, done = 0.0, 0
        t0 = time.perf_counter()
        for _ in range(steps):
            amount += sum(pool.map(_oracle_unit,
                                   [("decode-0.6b", (nxt + j) % n) for j in range(cores)],
                                   chunksize=1))
            nxt += cores
            done += 1
            if time.perf_counter() - t0 > budget_s:
                break
        el = time.perf_counter() - t0
    return {"value": amount / el / 1e9, "seconds": el, "steps": done, "seqs": done * cores,
            "cores": cores}


def cpu_oracle(budget_s: float, reference_steps: int = 0, warmup: int = 0):
    """Runs the CPU legs in a fresh interpreter (no CUDA, one thread per
    process) and returns its JSON."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-worker",
           "--budget", str(budget_s)]
    if reference_steps:
        cmd += ["--reference-steps", "--steps", str(reference_steps), "--warmup", str(warmup)]
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
    if name in ("decode-0.6b", "decode-0.6b-bs16"):
        spec = W.DECODE_0P6B
        if name == "decode-0.6b-bs16":
            # the same batch on 16-slot cache blocks: the register-load split kernel
            spec = dataclasses.replace(spec, block_size=16)
        w = W.decode_workload(spec, device=dev)
        bt, ctx = w.block_tables.to(dev), w.context_lens.to(dev)
        out = torch.empty_like(w.q)
        ws = torch.empty(pkv.paged_decode_workspace_bytes(spec.batch, spec.num_q_heads,
                                                          w.max_context_len, w.k_cache),
                         dtype=torch.uint8, device=dev)
        for _ in range(calls):
            pkv.paged_decode(w.q, w.k_cache, w.v_cache, bt, ctx, w.scale, w.max_context_len,
                             out=out, workspace=ws)
    elif name in ("prefill-8b", "prefill-8b-bs16"):
        spec = W.PREFILL_8B
        if name == "prefill-8b-bs16":
            # the same prompts on 16-slot cache blocks: cached rows are gathered
            spec = dataclasses.replace(spec, block_size=16, max_cached_blocks=64)
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
    ap.add_argument("--reference-steps", action="store_true")
    ap.add_argument("--budget", type=float, default=6.0,
                    help="seconds of wall time per multi-core CPU oracle leg")
    ap.add_argument("--profile", default=None,
                    help="run a small case for ncu instead of the benchmark: decode-0.6b, "
                         "decode-0.6b-bs16, prefill-8b, prefill-8b-bs16, sample or mixed-8b "
                         "(calls = --steps)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    if args.profile:
        profile_case(args.profile, args.steps)
        return

    if args.oracle_worker:
        oracle_worker(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        warm = min(args.warmup, 3)
        r = cpu_oracle(120.0, reference_steps=max(args.steps, 1), warmup=warm)
        from paged_kv_attention_scatter_gb300 import workloads as W
        spec = W.DECODE_0P6B
        ms = r["seconds"] / max(r["steps"], 1) * 1e3
        sample = (f"{r['seqs']} whole sequences (all 16 q heads) of decode-0.6b, one per core "
                  f"and step on {r['cores']} host cores (one spawned process each, float64 "
                  "NumPy, single-threaded BLAS), at most 120 s")
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(r["value"], 4),
            "unit": "GB/s", "n_gpus": 1, "steps": r["steps"], "warmup": warm,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": spec.name, "batch": spec.batch, "head_dim": spec.head_dim,
                       "block_size": spec.block_size},
            "cpu_baseline": {"value": round(r["value"], 4), "unit": "GB/s",
                             "cores": r["cores"], "kind": "oracle", "sample": sample},
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
        cpu = cpu_oracle(args.budget)
    res = run_ours(args, rank, world, dist)
    if cpu is not None:
        d06 = cpu.pop("decode-0.6b")
        cores = cpu.pop("cores")
        one = cpu.pop("one_core")
        res["cpu_baseline"] = {
            "value": d06["value"], "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": d06["sample"] + f" of decode-0.6b on {cores} host cores (one spawned "
                      "process each, float64 NumPy, single-threaded BLAS)",
            "one_core": one, "workloads": cpu}
    if rank == 0:
        print(json.dumps(res))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
