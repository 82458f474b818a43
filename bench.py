"""Benchmark of the routed-expert MXFP4 MoE layer on GB300.

Default workload: the full-size decode layer (E=896 experts, hidden 7168,
intermediate 1600, top-16), 1000 seeded synthetic tokens decoded one at a time.
One step = route + expert forward of all 1000 tokens (2 library calls, 2 kernels
per token), captured once in a CUDA graph and replayed.  value = layer-tokens/s.

    python bench.py [--steps K] [--warmup W] [--impl ours|reference] [--gpus N]

--impl reference times the fp64 CPU oracle (the only baseline this workload has)
on a bounded sample of the same tokens.  Under torchrun every rank runs an
independent replica (the layer does not shard); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer decode layer-tokens/s and expert-weight HBM GB/s (% of peak); prefill tok/s"
WORKLOAD = "full-size decode layer: E=896, H=7168, I=1600, top-16, M=1, 1000 seeded tokens one at a time"
NTOK = 1000


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def tensor_peak_tflops():
    """Dense bf16 tensor peak (measured burst, else the fallback) and its source."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def expert_bytes(H, I):
    return synth.expert_code_bytes(H, I) + synth.expert_scale_bytes(H, I)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out = ""

    def summary(self):
        rows = [r.split(",") for r in self.out.strip().splitlines() if r.count(",") >= 7]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in rows if r[0].strip().replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[4 + i] and "Not" not in r[4 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------- reference arm


def oracle_sample(ntok, threads=None):
    """Time the fp64 oracle on `ntok` tokens of the workload (route + experts),
    with the experts pre-generated outside the timed region."""
    import oracle
    s = synth.FULL
    xb = synth.tokens_bf16(synth.TOKENS_SEED["full"], 0, ntok, s.H)
    Wrb = synth.router_bf16(synth.router_seed(0), s.E, s.H)
    idx, _, _ = oracle.route(xb, Wrb, s.k)
    pool = oracle.SyntheticPool(synth.pool_seed(0), s.E, s.H, s.I, cache=ntok * s.k)
    for e in sorted(set(int(v) for v in idx.ravel())):
        pool(e)
    t0 = time.perf_counter()
    oracle.decode_layer(pool, xb, Wrb, s.k)
    return time.perf_counter() - t0


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    ntok = args.ref_tokens
    for _ in range(args.warmup if args.warmup < 1 else 1):
        oracle_sample(1)
    times = [oracle_sample(ntok) for _ in range(args.steps)]
    tot = sum(times)
    v = args.steps * ntok / tot
    cb = {"value": v, "unit": "layer-tokens/s", "cores": cores, "kind": "oracle",
          "sample": f"{ntok} tokens of the workload per step (route exact + 16 experts fp64), experts pre-generated"}
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "layer-tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_tokens_per_step": ntok},
        "cpu_baseline": cb,
        "e2e": {"value": v, "unit": "layer-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


# ---------------------------------------------------------------------- ours


def max_over_ranks(ms, dist, device):
    """The slowest rank's time (each rank runs an independent replica): an all-reduce
    MAX over the process group, or ms itself without one."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world, tokens_per_rank, ms_per_step):
    """Layer-tokens/s of the whole job: the tokens all ranks processed per step divided
    by the (max-over-ranks) step time."""
    return world * tokens_per_rank / (ms_per_step / 1000.0)


def measure_prefill(moe, torch, pool, Wr, dev, T, iters=3, act_mode=1):
    """Expert-major prefill of T tokens on the full-size layer: route, sort,
    MXFP8 (act_mode 1) or MXFP4 (2) gather, grouped gate/up and down GEMMs, combine.
    Returns timings."""
    s = synth.FULL
    xb = synth.tokens_bf16(synth.TOKENS_SEED["prefill"], 0, T, s.H)
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    ws_r = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_ROUTE, s.E, s.H, s.I, T, s.k), dev)
    ws_g = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_GROUPED, s.E, s.H, s.I, T, s.k), dev)
    idx = torch.empty((T, s.k), dtype=torch.int32, device=dev)
    w = torch.empty((T, s.k), dtype=torch.float32, device=dev)
    out = {"perm": torch.empty(T * s.k, dtype=torch.int32, device=dev),
           "inv_perm": torch.empty(T * s.k, dtype=torch.int32, device=dev),
           "offsets": torch.empty(s.E + 1, dtype=torch.int32, device=dev),
           "partial": torch.empty((T * s.k, s.H), dtype=torch.float32, device=dev)}
    y = torch.empty((T, s.H), dtype=torch.bfloat16, device=dev)

    def once():
        moe.moe_route_topk(x, Wr, s.k, ws=ws_r, idx=idx, w=w)
        moe.moe_expert_forward_grouped(pool, x, idx, act_mode=act_mode, ws=ws_g, out=out)
        moe.moe_combine(out["partial"], out["inv_perm"], w, y=y)

    once()
    torch.cuda.synchronize()
    assert moe.moe_check_status(ws_g) == 0 and moe.moe_check_status(ws_r) == 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        once()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / iters
    kern = {}
    for name in ("route_logits", "route_select", "gemm_gateup", "gemm_down", "combine", "gather_quant"):
        moe.moe_trace_begin(name)
        once()
        n, tot = moe.moe_trace_end()
        kern[name] = tot / max(n, 1)
    off = out["offsets"].cpu().numpy()
    nexp = int(np.count_nonzero(np.diff(off)))       # experts with at least one pair
    P = T * s.k
    wbytes = nexp * expert_bytes(s.H, s.I)
    flops = 2.0 * 3 * s.H * s.I * P
    gemm_ms = kern["gemm_gateup"] + kern["gemm_down"]
    tflops = flops / (gemm_ms / 1000.0) / 1e12
    bf16, bf16_kind = tensor_peak_tflops()
    hbm, hbm_kind = peaks()
    # Roofline of the two grouped GEMMs together: the MXFP4 weights of every expert with
    # pairs, the activation rows of x read (codes + one scale byte per 32), h written and
    # read again, and the fp32 expert outputs written.  MXFP8 rows: the MMA kind issued
    # (mxf8f6f4: E2M1 x E4M3) runs at the FP8 rate, the nominal 2x of the measured bf16
    # peak; MXFP4 rows: kind::mxf4 at the FP4 rate, the nominal 6x.
    eb = 1.0 if act_mode == 1 else 0.5           # bytes per activation element
    act_bytes = P * s.H * (eb + 1 / 32) + 2 * P * s.I * (eb + 1 / 32) + P * s.H * 4
    gbytes = wbytes + act_bytes
    kind_ratio = 2.0 if act_mode == 1 else 6.0
    t_bytes = gbytes / (hbm * 1e9) * 1e3
    t_flops = flops / (kind_ratio * bf16 * 1e12) * 1e3
    attainable = max(t_bytes, t_flops)
    return {"tok_s": T / (ms / 1000.0), "ms": ms, "kernel_ms": kern,
            "gemm_weight_gbs": wbytes / (gemm_ms / 1000.0) / 1e9,
            "gemm_tflops": tflops,
            "tensor_frac": {"of_fp8_rate": tflops / (2.0 * bf16), "of_fp4_rate": tflops / (6.0 * bf16),
                            "bf16_peak_tflops": bf16, "peak_kind": bf16_kind},
            "roofline": {"kernels": "gemm_gateup + gemm_down", "bound": "hbm" if t_bytes >= t_flops else "tensor",
                         "mma_kind": "mxf8f6f4" if act_mode == 1 else "mxf4",
                         "algorithmic_bytes": gbytes, "weight_bytes": wbytes, "flops": flops,
                         "peak_hbm_gbs": hbm, "peak_tflops": kind_ratio * bf16,
                         "peak_kind": f"{hbm_kind} hbm; {bf16_kind} bf16 x {kind_ratio:g} (nominal "
                         f"{'fp8' if act_mode == 1 else 'fp4'} ratio)", "attainable_ms": attainable,
                         "measured_ms": gemm_ms, "frac": attainable / gemm_ms}}


def measure_verify(moe, torch, pool, Wr, dev, M, nbatch=50, iters=3):
    """Multi-token verify on the full-size layer: nbatch seeded batches of M correlated
    rows, each routed and run through the experts (every distinct selected expert
    read once and applied to all its rows).  One CUDA graph over all batches."""
    s = synth.FULL
    xb = np.stack([synth.verify_batch_bf16(synth.TOKENS_SEED["verify"], b, M, s.H) for b in range(nbatch)])
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    idx = torch.empty((nbatch, M, s.k), dtype=torch.int32, device=dev)
    w = torch.empty((nbatch, M, s.k), dtype=torch.float32, device=dev)
    y = torch.empty((nbatch, M, s.H), dtype=torch.bfloat16, device=dev)
    ws_r = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_ROUTE, s.E, s.H, s.I, M, s.k), dev)
    ws_d = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_DECODE, s.E, s.H, s.I, M, s.k), dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        for b in range(nbatch):
            moe.moe_route_topk(x[b], Wr, s.k, ws=ws_r, idx=idx[b], w=w[b])
            moe.moe_expert_forward_decode(pool, x[b], idx[b], w[b], ws=ws_d, y=y[b])

    with torch.cuda.stream(stream):
        step()
        torch.cuda.synchronize()
        sd, sr = moe.moe_check_status(ws_d), moe.moe_check_status(ws_r)
        if sd != 0 or sr != 0:
            raise RuntimeError(f"verify M={M}: decode status {moe.status_string(sd)}, route status {moe.status_string(sr)}")
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
    torch.cuda.synchronize()
    union = float(np.mean([len(np.unique(a)) for a in idx.cpu().numpy().reshape(nbatch, -1)]))
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(iters):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / (iters * nbatch)
    kern = {}
    for name in ("route_logits", "route_select", "sort_small", "gather_split", "gemm_gateup", "gemm_down",
                 "combine"):
        moe.moe_trace_begin(name)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(50_000_000)
            step()
        n, tot = moe.moe_trace_end()
        torch.cuda.synchronize()  # the side stream's work is done before its tensors are freed
        if n:
            kern[name] = tot / n
    nbytes = union * expert_bytes(s.H, s.I) + s.E * s.H * 2
    hbm, _ = peaks()
    return {"us_per_batch": us, "rows_per_s": M / (us * 1e-6), "mean_union_experts": union,
            "bytes_per_batch": nbytes, "hbm_gbs": nbytes / (us * 1e-6) / 1e9,
            "hbm_frac": nbytes / (us * 1e-6) / 1e9 / hbm, "kernel_ms": kern}


def measure_stacked(moe, torch, pool0, dev, ntok=64, L=8, iters=2):
    """Eight stacked layers (each its own pool, router and Zipf skew), one token at a
    time: per layer x_hat = prescale(x) and route(x_hat) in one router launch, then
    x = x + MoE(x_hat).  Reports layer-tokens/s.  Allocates L - 1 more full-size pools."""
    s = synth.FULL
    pools = [pool0]
    for l in range(1, L):
        p = moe.Pool(s.E, s.H, s.I, device=dev)
        moe.moe_pool_fill_synthetic(p, synth.pool_seed(l))
        pools.append(p)
    Wrs = [torch.from_numpy(synth.router_bf16(synth.router_seed(l), s.E, s.H).view(np.int16)).to(dev)
           .view(torch.bfloat16) for l in range(L)]
    skews = [torch.from_numpy(synth.zipf_skew_f32(synth.skew_seed(l), s.E)).to(dev) for l in range(L)]
    xb = synth.tokens_bf16(synth.TOKENS_SEED["stacked"], 0, ntok, s.H)
    xs = [torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)]
    xs += [torch.empty_like(xs[0]) for _ in range(L)]
    xh = torch.empty((1, s.H), dtype=torch.bfloat16, device=dev)
    idx = torch.empty((1, s.k), dtype=torch.int32, device=dev)
    w = torch.empty((1, s.k), dtype=torch.float32, device=dev)
    ws_r = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_ROUTE, s.E, s.H, s.I, 1, s.k), dev)
    ws_d = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_DECODE, s.E, s.H, s.I, 1, s.k), dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        for t in range(ntok):
            for l in range(L):
                # pre-scale folded into the single-token router, which writes x_hat
                moe.moe_route_topk_prescaled(xs[l][t:t + 1], Wrs[l], s.k, skews[l], ws=ws_r, idx=idx, w=w, xhat=xh)
                moe.moe_expert_forward_decode(pools[l], xh, idx, w, residual=xs[l][t:t + 1], ws=ws_d,
                                              y=xs[l + 1][t:t + 1])

    with torch.cuda.stream(stream):
        step()
        torch.cuda.synchronize()
        assert moe.moe_check_status(ws_d) == 0 and moe.moe_check_status(ws_r) == 0
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(iters):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1000.0 / iters
    per_layer = s.k * expert_bytes(s.H, s.I) + s.E * s.H * 2
    del pools[1:]
    return {"tokens": ntok, "layers": L, "layer_tokens_per_s": ntok * L / sec,
            "us_per_layer_token": sec * 1e6 / (ntok * L), "hbm_gbs": ntok * L * per_layer / sec / 1e9}


def measure_tiny_l2(moe, torch, dev, ntok=1000, iters=3):
    """The small decode case (E = 64, H = 1024, I = 512, top-16, one token at a time):
    its 53.5 MB pool fits in L2, so this is a latency figure, not an HBM fraction.
    Route + decode per token, 1000 seeded tokens in one CUDA graph; reports
    layer-tokens/s, microseconds per token and the effective GB/s of the expert bytes
    and W_r, flagged L2-resident."""
    s = synth.TINY
    pool = moe.Pool(s.E, s.H, s.I, device=dev)
    moe.moe_pool_fill_synthetic(pool, synth.pool_seed(0))
    Wr = torch.from_numpy(synth.router_bf16(synth.router_seed(0), s.E, s.H).view(np.int16)).to(dev).view(torch.bfloat16)
    xb = synth.tokens_bf16(synth.TOKENS_SEED["tiny"], 0, ntok, s.H)
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty_like(x)
    idx = torch.empty((ntok, s.k), dtype=torch.int32, device=dev)
    w = torch.empty((ntok, s.k), dtype=torch.float32, device=dev)
    ws_r = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_ROUTE, s.E, s.H, s.I, 1, s.k), dev)
    ws_d = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_DECODE, s.E, s.H, s.I, 1, s.k), dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        for t in range(ntok):
            moe.moe_route_topk(x[t:t + 1], Wr, s.k, ws=ws_r, idx=idx[t:t + 1], w=w[t:t + 1])
            moe.moe_expert_forward_decode(pool, x[t:t + 1], idx[t:t + 1], w[t:t + 1], ws=ws_d, y=y[t:t + 1])

    with torch.cuda.stream(stream):
        step()
        torch.cuda.synchronize()
        assert moe.moe_check_status(ws_d) == 0 and moe.moe_check_status(ws_r) == 0
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(iters):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1000.0 / iters
    per_token = s.k * expert_bytes(s.H, s.I) + s.E * s.H * 2
    return {"shape": "E=64, H=1024, I=512, top-16, M=1", "tokens": ntok, "layer_tokens_per_s": ntok / sec,
            "us_per_token": sec * 1e6 / ntok, "bytes_per_token": per_token,
            "effective_gbs": per_token * ntok / sec / 1e9, "residency": "L2 (pool 53.5 MB < L2)"}


def measure_streamed(moe, torch, pool0, dev, ntok=48, warm=16, L=8, slots=128):
    """Eight stacked layers decoded one token at a time with the experts streamed: the
    records live in pinned host memory (one host copy of the pool shared by the
    layers, each layer with its own router, Zipf skew and HBM cache of `slots`
    records), and per layer-token the router's indices are read back, the missing
    records copied over NVLink-C2C (one cudaMemcpyAsync each) and the layer run on the
    cache.  Reports layer-tokens/s, the cache hit rate and the copy rate."""
    s = synth.FULL
    rec = moe.moe_pool_record_bytes(s.H, s.I)
    hb = moe.HostBuffer(s.E * rec, dev)  # pinned, on the GPU's own host NUMA node
    host = hb.tensor
    host.copy_(pool0.mem)
    sps = [moe.StreamPool(host, s.E, s.H, s.I, slots, device=dev) for _ in range(L)]
    Wrs = [torch.from_numpy(synth.router_bf16(synth.router_seed(l), s.E, s.H).view(np.int16)).to(dev)
           .view(torch.bfloat16) for l in range(L)]
    skews = [torch.from_numpy(synth.zipf_skew_f32(synth.skew_seed(l), s.E)).to(dev) for l in range(L)]
    xb = synth.tokens_bf16(synth.TOKENS_SEED["stacked"], 0, warm + ntok, s.H)
    x_all = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    xs = [torch.empty((1, s.H), dtype=torch.bfloat16, device=dev) for _ in range(L + 1)]
    xh = torch.empty((1, s.H), dtype=torch.bfloat16, device=dev)
    idx = torch.empty((1, s.k), dtype=torch.int32, device=dev)
    w = torch.empty((1, s.k), dtype=torch.float32, device=dev)
    idx_h = torch.empty((1, s.k), dtype=torch.int32).pin_memory()
    slot_h = torch.empty((1, s.k), dtype=torch.int32).pin_memory()
    slot_d = torch.empty((1, s.k), dtype=torch.int32, device=dev)
    ws_r = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_ROUTE, s.E, s.H, s.I, 1, s.k), dev)
    ws_d = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_DECODE, slots, s.H, s.I, 1, s.k), dev)
    stream = torch.cuda.current_stream(dev)

    def token(t):
        xs[0].copy_(x_all[t:t + 1])
        for l in range(L):
            moe.moe_route_topk_prescaled(xs[l], Wrs[l], s.k, skews[l], ws=ws_r, idx=idx, w=w, xhat=xh)
            idx_h.copy_(idx, non_blocking=True)
            stream.synchronize()
            slot_h.numpy()[:] = sps[l].map(idx_h.numpy(), stream)
            slot_d.copy_(slot_h, non_blocking=True)
            moe.moe_expert_forward_decode(sps[l].cache, xh, slot_d, w, residual=xs[l], ws=ws_d, y=xs[l + 1])

    for t in range(warm):
        token(t)
    torch.cuda.synchronize()
    st0 = [sp.stats() for sp in sps]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for t in range(warm, warm + ntok):
        token(t)
    e1.record(stream)
    torch.cuda.synchronize()
    assert moe.moe_check_status(ws_d) == 0 and moe.moe_check_status(ws_r) == 0
    sec = e0.elapsed_time(e1) / 1000.0
    st1 = [sp.stats() for sp in sps]
    hits = sum(b[0] - a[0] for a, b in zip(st0, st1))
    misses = sum(b[1] - a[1] for a, b in zip(st0, st1))
    copied = sum(b[2] - a[2] for a, b in zip(st0, st1))
    node = hb.numa_node
    del sps, host
    hb.close()
    return {"tokens": ntok, "layers": L, "slots_per_layer": slots, "slot_fraction": slots / s.E,
            "host_numa_node": node, "gpu_host_numa_node": moe.moe_host_numa_node(dev),
            "layer_tokens_per_s": ntok * L / sec, "us_per_layer_token": sec * 1e6 / (ntok * L),
            "hit_rate": hits / max(hits + misses, 1), "misses_per_layer_token": misses / (ntok * L),
            "copy_gbs": copied / sec / 1e9,
            "note": "one pinned host copy of the pool, on the GPU's own NUMA node, shared by the layers"}


def run_ours(args):
    import torch
    import mxfp4_routed_expert_topk_gb300 as moe

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    moe.build()

    s = synth.FULL
    pool = moe.Pool(s.E, s.H, s.I, device=dev)
    moe.moe_pool_fill_synthetic(pool, synth.pool_seed(0))
    Wrb = synth.router_bf16(synth.router_seed(0), s.E, s.H)
    Wr = torch.from_numpy(Wrb.view(np.int16)).to(dev).view(torch.bfloat16)
    xb = synth.tokens_bf16(synth.TOKENS_SEED["full"], 0, NTOK, s.H)
    x_host = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).pin_memory()
    x = x_host.to(dev)
    y = torch.empty((NTOK, s.H), dtype=torch.bfloat16, device=dev)
    y_host = torch.empty((NTOK, s.H), dtype=torch.bfloat16).pin_memory()
    idx = torch.empty((NTOK, s.k), dtype=torch.int32, device=dev)
    w = torch.empty((NTOK, s.k), dtype=torch.float32, device=dev)
    ws_r = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_ROUTE, s.E, s.H, s.I, 1, s.k), dev)
    ws_d = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_DECODE, s.E, s.H, s.I, 1, s.k), dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        for t in range(NTOK):
            moe.moe_route_topk(x[t:t + 1], Wr, s.k, ws=ws_r, idx=idx[t:t + 1], w=w[t:t + 1])
            moe.moe_expert_forward_decode(pool, x[t:t + 1], idx[t:t + 1], w[t:t + 1], ws=ws_d, y=y[t:t + 1])

    with torch.cuda.stream(stream):
        step()                                   # eager once (sets kernel attributes)
        torch.cuda.synchronize()
        assert moe.moe_check_status(ws_d) == 0 and moe.moe_check_status(ws_r) == 0
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
    torch.cuda.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        graph.replay()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            e1.record(stream)
        barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    ms_step = ms / args.steps
    value = whole_job_value(world, NTOK, ms_step)

    # end to end through the public API: pinned host x in, host y out, every step
    with torch.cuda.stream(stream):
        for _ in range(2):
            x.copy_(x_host, non_blocking=True)
            graph.replay()
            y_host.copy_(y, non_blocking=True)
        barrier()
        e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2.record(stream)
        for _ in range(args.steps):
            x.copy_(x_host, non_blocking=True)
            graph.replay()
            y_host.copy_(y, non_blocking=True)
        e3.record(stream)
        barrier()
    e2e_ms = e2.elapsed_time(e3) / args.steps
    h2d = x_host.numel() * 2
    d2h = y_host.numel() * 2

    # per-kernel device time over one more pass of the timed region (eager launches
    # queued behind a bounded sleep kernel, so the GPU never waits on the host)
    kern = {}
    for name in ("decode_fused", "route_single"):
        moe.moe_trace_begin(name)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(200_000_000)
            step()
        n, tot = moe.moe_trace_end()
        kern[name] = tot / max(n, 1)
    hbm, peak_kind = peaks()
    # dominant kernel: the fused expert kernel streams the 16 selected experts' MXFP4
    # codes and scales (18,278,400 B each at this shape)
    kern_bytes = s.k * expert_bytes(s.H, s.I)
    layer_bytes = s.k * expert_bytes(s.H, s.I) + s.E * s.H * 2
    achieved = kern_bytes / (kern["decode_fused"] / 1000.0) / 1e9
    layer_gbs = layer_bytes / (ms_step / 1000.0 / NTOK) / 1e9
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "decode_fused_traffic.json")
    if os.path.exists(tfile):
        traffic = json.load(open(tfile)).get("bytes_per_launch")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        prev = oracle.set_threads(cores)
        secs = oracle_sample(args.ref_tokens)
        oracle.set_threads(1)
        n1 = max(1, args.ref_tokens // 8)
        secs1 = oracle_sample(n1)
        oracle.set_threads(prev)
        cpu = {"value": args.ref_tokens / secs, "unit": "layer-tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{args.ref_tokens} tokens of the workload (exact route + 16 experts, fp64), "
                         "experts pre-generated outside the timing",
               "single_thread": {"value": n1 / secs1, "unit": "layer-tokens/s", "cores": 1,
                                 "sample": f"{n1} tokens of the same workload on one thread"}}
    launches = 2 * NTOK * args.steps      # route_single + decode_fused per token
    prefill, prefill4, pairs = {}, {}, {}
    if not args.no_prefill:
        for T in synth.PREFILL_T:
            prefill[str(T)] = measure_prefill(moe, torch, pool, Wr, dev, T)
        for T in synth.PREFILL_T + synth.PREFILL_T_LARGE:
            prefill4[str(T)] = measure_prefill(moe, torch, pool, Wr, dev, T, act_mode=2)
            torch.cuda.empty_cache()
        # the other tile shape of each row format: MXFP8 on one CTA per tile (the default
        # runs it on paired-SM tiles, tcgen05 cta_group::2), MXFP4 on paired-SM tiles
        for mode, cases in ((moe.CTA_PAIRS_NEVER, ((8192, 1),)), (moe.CTA_PAIRS_ALWAYS, ((8192, 2), (32768, 2)))):
            moe.moe_grouped_set_cta_pairs(mode)
            try:
                for T, act in cases:
                    key = f"{T}_{'mxfp8' if act == 1 else 'mxfp4'}_{'one_cta' if mode == moe.CTA_PAIRS_NEVER else 'pairs'}"
                    pairs[key] = measure_prefill(moe, torch, pool, Wr, dev, T, act_mode=act)["kernel_ms"]
            finally:
                moe.moe_grouped_set_cta_pairs(moe.CTA_PAIRS_MXFP8)
        torch.cuda.empty_cache()
    verify, stacked, streamed, tiny = {}, None, None, None
    if not args.no_extra:
        tiny = measure_tiny_l2(moe, torch, dev)
        for M in synth.VERIFY_M:
            verify[str(M)] = measure_verify(moe, torch, pool, Wr, dev, M)
        stacked = measure_stacked(moe, torch, pool, dev)
        torch.cuda.empty_cache()
        streamed = {str(c): measure_streamed(moe, torch, pool, dev, slots=c) for c in (128, 256)}
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "layer-tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "mxfp4(e2m1)xbf16, f16x2 block MAC, fp32 accumulate",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2: 17.6 GB resident pool, 16 fresh experts per token",
                       "graph": "one CUDA graph per step (1000 tokens)"},
            "expert_weight_hbm_gbs": layer_gbs, "hbm_frac_layer": layer_gbs / hbm,
            "roofline": {"bound": "hbm", "kernel": "decode_fused", "achieved": achieved, "peak": hbm,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                         "algorithmic_bytes_per_launch": kern_bytes},
            "kernel_ms": kern,
            "cpu_baseline": cpu,
            "e2e": {"value": NTOK / (e2e_ms / 1000.0) * world, "unit": "layer-tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "prefill": prefill,
            "prefill_mxfp4": prefill4,
            "prefill_other_tile_shape": pairs,
            "verify": verify,
            "stacked_8_layers": stacked,
            "tiny_l2": tiny,
            "streamed_8_layers": streamed,
            "clocks": clk.summary(),
        }))
    if dist is not None:
        dist.destroy_process_group()


def run_profile_case(args):
    """A small case of the same kernels for ncu captures: full H and I, a 64-expert
    pool (1.2 GB, larger than L2); a few single-token calls (decode) or one
    expert-major call of --profile-tokens tokens (prefill; 585 tokens give the 146
    rows per expert of 8192 tokens over 896 experts)."""
    import torch
    import mxfp4_routed_expert_topk_gb300 as moe
    moe.build()
    if args.profile == "route":
        # the router alone at the full shape (E=896, H=7168): 12.8 MB of W_r; four
        # single-token calls, or (--profile-tokens > 64) one call on that many tokens,
        # which takes the tiled logit kernel
        s = synth.FULL
        Wr = torch.from_numpy(synth.router_bf16(synth.router_seed(0), s.E, s.H).view(np.int16)).cuda()
        Wr = Wr.view(torch.bfloat16)
        n = args.profile_tokens if args.profile_tokens > 64 else 4
        xb = synth.tokens_bf16(synth.TOKENS_SEED["full"], 0, n, s.H)
        x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
        if n > 64:
            for _ in range(2):
                moe.moe_route_topk(x, Wr, s.k)
        else:
            for t in range(4):
                moe.moe_route_topk(x[t:t + 1], Wr, s.k)
        torch.cuda.synchronize()
        print("profile case done")
        return
    s = synth.Shape(E=64, H=synth.FULL.H, I=synth.FULL.I, k=16)
    pool = moe.Pool(s.E, s.H, s.I)
    moe.moe_pool_fill_synthetic(pool, synth.pool_seed(0))
    Wr = torch.from_numpy(synth.router_bf16(synth.router_seed(0), s.E, s.H).view(np.int16)).cuda().view(torch.bfloat16)
    if args.profile == "verify":
        # four verify batches of --profile-tokens correlated rows (router, sort, split,
        # grouped GEMMs, combine); the router at the full E = 896
        Wr_full = torch.from_numpy(synth.router_bf16(synth.router_seed(0), synth.FULL.E, s.H).view(np.int16)).cuda()
        Wr_full = Wr_full.view(torch.bfloat16)
        M = args.profile_tokens
        for b in range(4):
            xb = synth.verify_batch_bf16(synth.TOKENS_SEED["verify"], b, M, s.H)
            x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
            moe.moe_route_topk(x, Wr_full, s.k)
            idx, w = moe.moe_route_topk(x, Wr, s.k)
            moe.moe_expert_forward_decode(pool, x, idx, w)
        torch.cuda.synchronize()
        print("profile case done")
        return
    if args.profile == "prefill":
        xb = synth.tokens_bf16(synth.TOKENS_SEED["prefill"], 0, args.profile_tokens, s.H)
        x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
        for _ in range(2):
            idx, w = moe.moe_route_topk(x, Wr, s.k)
            out = moe.moe_expert_forward_grouped(pool, x, idx, act_mode=args.profile_act)
            moe.moe_combine(out["partial"], out["inv_perm"], w)
        torch.cuda.synchronize()
        print("profile case done")
        return
    xb = synth.tokens_bf16(synth.TOKENS_SEED["full"], 0, 4, s.H)
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    for t in range(4):
        idx, w = moe.moe_route_topk(x[t:t + 1], Wr, s.k)
        moe.moe_expert_forward_decode(pool, x[t:t + 1], idx, w)
    torch.cuda.synchronize()
    print("profile case done")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the expert-major prefill measurements")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the multi-token verify and 8-layer stacked measurements")
    ap.add_argument("--profile", choices=["decode", "prefill", "route", "verify"], default=None,
                    help="run a small case of the kernels for an ncu capture (no JSON line)")
    ap.add_argument("--profile-tokens", type=int, default=64,
                    help="tokens of the prefill profile case (64-expert pool)")
    ap.add_argument("--profile-act", type=int, default=1, choices=[1, 2],
                    help="activation format of the prefill profile case: 1 MXFP8, 2 MXFP4")
    args = ap.parse_args()
    if args.profile:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
