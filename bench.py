#!/usr/bin/env python
"""MiTA forward pass on GB300: queries/s and the roofline fraction.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mita|reference]
                    [--config long1m] [--no-sweep] [--no-cpu] [--no-e2e]
                    [--only backward]

One step = one full forward pass (landmark pooling, landmark scan with expert
selection, routing, grouping, expert attention) over one synthetic batch
already resident in HBM. value = B*H*N queries / device time per step. With
N GPUs (torchrun) every rank runs an independent replica on its own inputs
(the heads are independent problems; there is no exchange step), the time is
the max over ranks, and value counts the queries of all ranks (weak scaling).

--impl reference times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MiTA fwd queries/s at N=4K-1M, d=64; achieved fraction of roofline"
DEFAULT_CONFIG = "long1m"
# every other workload of the metric, each timed as its own entry of the line
SWEEP = ("tiny", "deit", "seg1024", "seg1600", "lra", "long64k", "long256k")
L2_BYTES = 129 * 1000 * 1000  # GB300 L2
L2_FLUSH_BYTES = 512 << 20     # written between passes whose inputs would stay in L2
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
STAGES = ("pool", "pilot", "scan", "select", "route", "group", "expert")
# the source file of the kernel that runs each stage on the long-sequence workloads
KERNEL_SOURCES = {"pool": "pool.cu", "pilot": "scan_tc.cu", "scan": "scan_tc.cu", "select": "select.cu",
                  "route": "route_tc.cu", "group": "group.cu", "expert": "expert_tc.cu"}


def describe(name):
    c = synth.CONFIGS[name]
    grid = f"{c['grid_h']}x{c['grid_w']} grid" if c["grid_h"] else f"1-D windows of {c['N'] // c['m']}"
    rec = {"iid": "Q,K,V i.i.d. N(0,1)",
           "outliers": "Q,K,V i.i.d. N(0,1), 1% of key rows x4",
           "clusters": f"K,Q from {c.get('clusters')} Gaussian clusters (sigma 0.3), V N(0,1)",
           "runs": f"K,Q from {c.get('clusters')} clusters in runs of 16-256 tokens, V N(0,1)"}[c["recipe"]]
    return f"{name}: B={c['B']} H={c['H']} N={c['N']} d=64 m={c['m']} k={c['k']}, {grid}; {rec}; seed 0"


# ---------------------------------------------------------------------------
# Algorithmic work per stage (the roofline numerators), per call.
# Whole pass: FLOPs = B*H*(4 m N d + 4 N (m+k) d); bytes = B*H*(3 N d + N d)*2
# + B*H*m*k*2*d*2 (Q,K,V read once, gathered expert rows, output written).
# ---------------------------------------------------------------------------
def work(c, shared=True, s=1):
    """shared=False: the routing-only ablation, whose scan forms only the
    logits (no shared-expert values) and whose experts hold k keys alone.
    s > 1: s routed experts per query; the attention counts m + s k keys per
    query (an upper bound: shared keys of two experts are attended once) and
    reads s expert row sets per query group."""
    BH, N, d, m, k = c["B"] * c["H"], c["N"], 64, c["m"], c["k"]
    row = N * d * 2
    if s > 1:
        return {
            "total": {"flops": BH * (4 * m * N * d + 4 * N * (m + s * k) * d),
                      "bytes": BH * (4 * row + m * k * 2 * d * 2)},
            "pool": {"flops": 0, "bytes": BH * row},
            "scan": {"flops": BH * 4 * m * N * d, "bytes": BH * 2 * row},
            "route": {"flops": BH * 2 * N * m * d, "bytes": BH * row},
            "expert": {"flops": BH * 4 * N * (m + s * k) * d, "bytes": BH * (s * 2 * row + s * m * k * 2 * d * 2)},
        }
    if not shared:
        return {
            "total": {"flops": BH * (2 * m * N * d + 4 * N * k * d), "bytes": BH * (4 * row + m * k * 2 * d * 2)},
            "pool": {"flops": 0, "bytes": BH * row},
            "scan": {"flops": BH * 2 * m * N * d, "bytes": BH * row},
            "route": {"flops": BH * 2 * N * m * d, "bytes": BH * row},
            "expert": {"flops": BH * 4 * N * k * d, "bytes": BH * (2 * row + m * k * 2 * d * 2)},
        }
    return {
        "total": {"flops": BH * (4 * m * N * d + 4 * N * (m + k) * d),
                  "bytes": BH * (4 * row + m * k * 2 * d * 2)},
        "pool": {"flops": 0, "bytes": BH * row},
        "scan": {"flops": BH * 4 * m * N * d, "bytes": BH * 2 * row},
        "route": {"flops": BH * 2 * N * m * d, "bytes": BH * row},
        "expert": {"flops": BH * 4 * N * (m + k) * d, "bytes": BH * (2 * row + m * k * 2 * d * 2)},
    }


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return {k: float(j[k]) for k in PEAKS_FALLBACK}, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def roofline_time(w, peaks, sustained):
    tf = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"] * 1e12
    return max(w["flops"] / tf, w["bytes"] / (peaks["hbm_gbs"] * 1e9))


def dominant_roofline(w, stage_ms, peaks, sustained=False):
    """The roofline object of the stage kernel (pool, scan, route or expert)
    with the largest time: its algorithmic FLOPs or bytes per launch over its
    CUDA-event time, against the peak of the resource that bounds it (the
    burst bf16 figure for these sub-second loops unless `sustained`)."""
    dom = max(("pool", "scan", "route", "expert"), key=lambda x: stage_ms[x])
    wd = w[dom]
    t = stage_ms[dom] / 1e3
    pk = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    tensor = wd["flops"] / (pk * 1e12) >= wd["bytes"] / (peaks["hbm_gbs"] * 1e9)
    if tensor:
        r = {"bound": "tensor", "achieved": wd["flops"] / t / 1e12, "peak": pk, "unit": "TFLOP/s"}
    else:
        r = {"bound": "hbm", "achieved": wd["bytes"] / t / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r["kernel"] = dom
    r["scope"] = f"dominant kernel of the pass ({dom}), not the whole pass"
    return r


def whole_pass_roofline(w, ms_step, peaks, peak_src):
    """The metric's own fraction: t_roof / t_measured for the whole pass,
    t_roof = max(FLOPs / bf16 peak, bytes / HBM bandwidth), with the burst
    bf16 peak (the timed loops run well under a second) and, labelled, the
    sustained one."""
    t_b = roofline_time(w["total"], peaks, sustained=False)
    t_s = roofline_time(w["total"], peaks, sustained=True)
    t = ms_step / 1e3
    bound = "tensor" if w["total"]["flops"] / (peaks["bf16_tflops"] * 1e12) >= \
        w["total"]["bytes"] / (peaks["hbm_gbs"] * 1e9) else "hbm"
    return {"t_roof_us": t_b * 1e6, "t_us": t * 1e6, "frac": t_b / t, "bound": bound,
            "frac_vs_sustained_peak": t_s / t, "flops": w["total"]["flops"], "bytes": w["total"]["bytes"],
            "peak_source": f"{peak_src}: burst bf16 {peaks['bf16_tflops']} TFLOP/s, copy {peaks['hbm_gbs']} GB/s "
                           f"(sustained bf16 {peaks['bf16_tflops_sustained']} TFLOP/s for frac_vs_sustained_peak)"}


def kernel_traffic(stage, workload):
    """DRAM bytes per launch of a stage's kernel from a committed ncu summary,
    or None when absent or taken on a different version of the kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    t = json.load(open(p)).get(stage)
    if not t or t.get("workload") != workload:
        return None
    src = os.path.join(ROOT, "mixture_top_forward_gb300", "csrc", KERNEL_SOURCES[stage])
    if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != t.get("source_sha"):
        return None
    return t.get("bytes_per_launch")


# ---------------------------------------------------------------------------
# Clock sampling during the timed region.
# ---------------------------------------------------------------------------
class Clocks:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.path = tempfile.mktemp(prefix="clocks", suffix=".csv")
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                rows.append((float(f[0]), float(f[1]), f[3:7]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle timing on a bounded sample of one head.
# ---------------------------------------------------------------------------
def oracle_head_time(name, q, k, v, n_landmarks, n_queries, seed=1, head=0):
    """Seconds the oracle needs for one whole head, estimated from a sample:
    pooling of the head in full, the scan of `n_landmarks` landmarks (values
    and expert selection) and routing + attention of `n_queries` queries,
    each scaled to the full head (m landmarks, N queries). The attention of
    the sampled queries runs on the scanned landmarks' experts and values,
    with same-shaped stand-ins for the rest (the work does not depend on the
    values)."""
    import oracle

    c = synth.CONFIGS[name]
    N, m, kk, gh, gw = c["N"], c["m"], c["k"], c["grid_h"], c["grid_w"]
    rng = np.random.default_rng(seed)
    b, h = divmod(head, q.shape[1])
    qs, ks, vs = q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1]
    t0 = time.perf_counter()
    lq = oracle.landmarks(qs, gh, gw, m)
    t1 = time.perf_counter()
    nl = min(m, n_landmarks)
    which_l = np.sort(rng.choice(m, size=nl, replace=False))
    lv_s, e_s, _ = oracle.scan(lq, ks, vs, kk, which=which_l)
    t2 = time.perf_counter()
    lv = np.zeros((1, 1, m, 64))
    e = np.tile(np.arange(kk, dtype=np.int32), (1, 1, m, 1))
    lv[0, 0, which_l] = lv_s
    e[0, 0, which_l] = e_s
    nq = min(N, n_queries)
    which_q = np.sort(rng.choice(N, size=nq, replace=False))
    r_s, _ = oracle.route(qs, lq, which=which_q)
    route = np.zeros((1, 1, N), np.int32)
    route[0, 0, which_q] = r_s
    t3 = time.perf_counter()
    oracle.attend(qs, lq, lv, ks, vs, e, route, which=which_q)
    t4 = time.perf_counter()
    t_head = (t1 - t0) + (t2 - t1) * m / nl + (t4 - t2) * N / nq
    if nl == m and nq == N:
        sample = f"1 whole head of {name} (N={N}, m={m}, k={kk})"
    else:
        sample = (f"1 head of {name}: pooling of all {N} tokens, scan of {nl}/{m} landmarks, routing+attention of "
                  f"{nq}/{N} queries, scaled to the head")
    return t_head, sample, t4 - t0


def cpu_baseline(name, q, k, v, heads=2):
    """The oracle on `heads` whole heads of the workload (about ten seconds
    of host work at N = 1M), as queries per second."""
    import oracle

    c = synth.CONFIGS[name]
    nh = min(heads, q.shape[0] * q.shape[1])
    t_sum, wall = 0.0, 0.0
    for h in range(nh):
        t_head, sample, w = oracle_head_time(name, q, k, v, c["m"], c["N"], head=h)
        t_sum += t_head
        wall += w
    sample = f"{nh} whole heads of {name} (N={c['N']}, m={c['m']}, k={c['k']}), run one after the other"
    return {"value": nh * c["N"] / t_sum, "unit": "queries/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": sample, "wall_s": round(wall, 2)}


# ---------------------------------------------------------------------------
# GPU arm.
# ---------------------------------------------------------------------------
def rank_barrier(world):
    """All ranks meet here (N > 1 only)."""
    if world > 1:
        import torch

        torch.distributed.barrier()


def max_over_ranks(ms, world, device=None):
    """The slowest rank's time; every rank gets it. The replicas are
    independent, so the job is done when the last one is."""
    if world == 1:
        return ms
    import torch

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(queries_per_rank, world, ms_step):
    """Queries of all ranks per second (weak scaling: each rank has its own
    full problem), over the slowest rank's step time."""
    return queries_per_rank * world / (ms_step / 1e3)


def run_gpu(args, rank, world):
    import torch

    import mixture_top_forward_gb300 as M

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    M.load(build_if_missing=False)
    name = args.config
    c = synth.CONFIGS[name]
    B, H, N, m, kk, gh, gw = c["B"], c["H"], c["N"], c["m"], c["k"], c["grid_h"], c["grid_w"]
    q, k, v = synth.make_inputs(c, seed=rank)

    def dev_bf16(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    Q, K, V = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    out = torch.empty_like(Q)
    eidx = torch.empty((B, H, m, kk), dtype=torch.int32, device=dev)
    sr = args.s_route
    route = torch.empty((B, H, N) if sr == 1 else (B, H, N, sr), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        if sr == 1:
            M.mita_forward(Q, K, V, gh, gw, m, kk, out=out, expert_idx=eidx, route=route, stream=stream)
        else:
            M.mita_forward_multi(Q, K, V, gh, gw, m, kk, sr, out=out, expert_idx=eidx, route=route, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert M.mita_sync_status(stream) == 0, M.mita_last_error()
    M.mita_profile_read(stream)  # discard
    clocks = Clocks(dev.index) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)
    M.mita_profile_enable(True)
    rank_barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    rank_barrier(world)
    M.mita_profile_enable(False)
    ms = ev0.elapsed_time(ev1)
    stages = M.mita_profile_read(stream)
    clk = clocks.stop() if clocks else None
    assert M.mita_sync_status(stream) == 0, M.mita_last_error()
    ms = max_over_ranks(ms, world, dev)
    ms_step = ms / args.steps
    queries = B * H * N
    value = job_throughput(queries, world, ms_step)

    peaks, peak_src = load_peaks()
    w = work(c, s=sr)
    stage_ms = {s: stages[s][0] / args.steps for s in STAGES}
    launches = sum(stages[s][1] for s in STAGES)
    roof = dominant_roofline(w, stage_ms, peaks)
    dom = roof["kernel"]
    roof["traffic"] = kernel_traffic(dom, name) if sr == 1 else None  # the counters are the one-expert kernels'
    roof["peak_source"] = f"{peak_src} ({'burst bf16' if roof['bound'] == 'tensor' else 'copy bandwidth'})"

    res = {
        "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": describe(name) + (f"; s={sr} routed experts per query" if sr > 1 else ""),
                   "B": B, "H": H, "N": N, "d": 64, "m": m, "k": kk, "s": sr,
                   "l2": f"inputs ({3 * Q.numel() * 2 / 1e9:.2f} GB) larger than L2, no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof,
        "roofline_whole_pass": whole_pass_roofline(w, ms_step, peaks, peak_src),
        "stage_ms": stage_ms,
        "gpu_launches": launches,
        "clocks": clk,
    }
    del Q, K, V, out
    torch.cuda.empty_cache()

    if not args.no_e2e and sr == 1:  # every rank: the job's end-to-end rate (the host entry point is s = 1)
        e = e2e(args, M, q, k, v, c, stream, world, dev)
        if rank == 0:
            res["e2e"] = e
    if rank == 0 and not args.no_sweep:
        # the side measurements: a failure is recorded in the line, never
        # loses the headline numbers above
        def leg(key, fn):
            try:
                res[key] = fn()
            except Exception as ex:  # noqa: BLE001 (reported, not hidden)
                res[key] = {"error": f"{type(ex).__name__}: {ex}"[:400]}

        leg("sweep", lambda: sweep(args, M, dev, stream, peaks, peak_src, with_cpu=not args.no_cpu))
        leg("routed_only", lambda: routed_only(args, M, dev, stream, peaks))
        leg("split_shared", lambda: split_shared(args, M, dev, stream, peaks))
        leg("multi_expert", lambda: multi_expert(args, M, dev, stream, peaks))
        leg("backward", lambda: backward(args, M, dev, stream, peaks))
        mita_ms = {n: r["ms_per_step"] for n, r in res["sweep"].items()} if "error" not in res["sweep"] else {}
        mita_ms[name] = ms_step
        leg("full_attention", lambda: full_attention(args, dev, stream, mita_ms))
    if rank == 0 and not args.no_cpu and world == 1 and sr == 1:
        res["cpu_baseline"] = cpu_baseline(name, q, k, v)
    return res


def e2e(args, M, q, k, v, c, stream, world=1, dev=None):
    """Same metric through the host-buffer entry point: each step copies the
    inputs from pinned host memory and the results back. With N ranks each
    runs its replica; the time is the slowest rank's."""
    import torch

    pin = lambda a: torch.from_numpy(a).pin_memory().numpy()
    qh, kh, vh = pin(q), pin(k), pin(v)
    out = pin(np.empty_like(q))
    eidx = pin(np.empty((c["B"], c["H"], c["m"], c["k"]), np.int32))
    route = pin(np.empty((c["B"], c["H"], c["N"]), np.int32))
    args_ = (c["grid_h"], c["grid_w"], c["m"], c["k"])
    for _ in range(max(1, min(args.warmup, 3))):
        M.mita_forward_host(qh, kh, vh, *args_, out=out, expert_idx=eidx, route=route, stream=stream.cuda_stream)
    n = max(3, min(args.steps, 10))
    rank_barrier(world)
    t0 = time.perf_counter()
    for _ in range(n):
        M.mita_forward_host(qh, kh, vh, *args_, out=out, expert_idx=eidx, route=route, stream=stream.cuda_stream)
    dt = max_over_ranks((time.perf_counter() - t0) * 1e3, world, dev) / 1e3 / n
    return {"value": job_throughput(c["B"] * c["H"] * c["N"], world, dt * 1e3), "unit": "queries/s",
            "h2d_bytes_per_step": int(qh.nbytes + kh.nbytes + vh.nbytes),
            "d2h_bytes_per_step": int(out.nbytes + eidx.nbytes + route.nbytes), "steps": n,
            "ms_per_step": dt * 1e3}


# host oracle per sweep workload: whole heads where that stays within a few
# seconds of host work, else one head with sampled landmarks and queries
# (scaled to the head; see oracle_head_time)
ORACLE_SAMPLE = {"tiny": None, "deit": None, "seg1024": None, "seg1600": None, "lra": (64, 4096),
                 "long64k": (32, 8192), "long256k": (16, 8192)}


def oracle_rate(name, q, k, v):
    """The fp64 oracle's queries/s on this machine's host cores for a workload:
    the whole batch for the small ViT shapes, one (sampled) head otherwise."""
    import oracle

    c = synth.CONFIGS[name]
    smp = ORACLE_SAMPLE.get(name)
    if smp is None:
        orc = oracle.Oracle()
        t0 = time.perf_counter()
        orc.forward(q, k, v, c["grid_h"], c["grid_w"], c["m"], c["k"])
        t = time.perf_counter() - t0
        return {"value": c["B"] * c["H"] * c["N"] / t, "unit": "queries/s", "cores": oracle.num_threads(),
                "kind": "oracle", "sample": f"the whole batch of {name} ({c['B'] * c['H']} heads), one run",
                "wall_s": round(t, 3)}
    t_head, sample, wall = oracle_head_time(name, q, k, v, smp[0], smp[1])
    return {"value": c["N"] / t_head, "unit": "queries/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": sample, "wall_s": round(wall, 3)}


def sweep(args, M, dev, stream, peaks, peak_src, with_cpu=True):
    """Every other workload of the metric, each timed like the headline one
    (device-resident inputs, CUDA events around n passes after warm-up): its
    queries/s and whole-pass roofline fraction from passes without the
    library's stage events, its stage times and dominant kernel (with its own
    roofline) from a second loop with them, and the oracle's rate on the host
    cores."""
    import torch

    res = {}
    for name in SWEEP:
        if name == args.config:
            continue
        c = synth.CONFIGS[name]
        q, k, v = synth.make_inputs(c)
        to = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        Q, K, V = to(q), to(k), to(v)
        out = torch.empty_like(Q)
        e = torch.empty((c["B"], c["H"], c["m"], c["k"]), dtype=torch.int32, device=dev)
        r = torch.empty((c["B"], c["H"], c["N"]), dtype=torch.int32, device=dev)
        a = (c["grid_h"], c["grid_w"], c["m"], c["k"])
        for _ in range(5):
            M.mita_forward(Q, K, V, *a, out=out, expert_idx=e, route=r, stream=stream)
        torch.cuda.synchronize()
        assert M.mita_sync_status(stream) == 0, M.mita_last_error()
        M.mita_profile_read(stream)  # discard
        n = 20 if c["N"] >= 65536 else 50
        in_bytes = 3 * Q.numel() * 2
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev) if in_bytes < 2 * L2_BYTES else None

        def timed_passes():
            if flush is None:  # inputs larger than L2: one bracket around n passes
                ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                ev0.record(stream)
                for _ in range(n):
                    M.mita_forward(Q, K, V, *a, out=out, expert_idx=e, route=r, stream=stream)
                ev1.record(stream)
                torch.cuda.synchronize()
                return ev0.elapsed_time(ev1) / n
            # L2 flushed before every pass, outside its events
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            for e0, e1 in evs:
                flush.zero_()
                e0.record(stream)
                M.mita_forward(Q, K, V, *a, out=out, expert_idx=e, route=r, stream=stream)
                e1.record(stream)
            torch.cuda.synchronize()
            return sum(e0.elapsed_time(e1) for e0, e1 in evs) / n

        # the pass time without the library's stage events (on short passes
        # their records are a visible share), then the stage breakdown from
        # a second, instrumented loop of the same passes
        ms = timed_passes()
        M.mita_profile_enable(True)
        ms_instrumented = timed_passes()
        M.mita_profile_enable(False)
        stages = M.mita_profile_read(stream)
        assert M.mita_sync_status(stream) == 0, M.mita_last_error()
        w = work(c)
        stage_ms = {x: stages[x][0] / n for x in STAGES}
        wp = whole_pass_roofline(w, ms, peaks, peak_src)
        ent = {"queries_per_s": c["B"] * c["H"] * c["N"] / (ms / 1e3), "ms_per_step": ms, "steps": n,
               "ms_per_step_with_stage_events": ms_instrumented,
               "roofline_frac": wp["frac"], "roofline_bound": wp["bound"], "t_roof_us": wp["t_roof_us"],
               "roofline_frac_vs_sustained_peak": wp["frac_vs_sustained_peak"],
               "stage_ms": stage_ms, "gpu_launches_per_step": sum(stages[x][1] for x in STAGES) / n,
               "dominant": dominant_roofline(w, stage_ms, peaks),
               "l2": "inputs larger than 2x L2, no flush" if flush is None else
                     f"L2 flushed before every timed pass ({L2_FLUSH_BYTES >> 20} MiB written)"}
        del Q, K, V, out, flush
        torch.cuda.empty_cache()
        if with_cpu:
            try:
                ent["cpu_baseline"] = oracle_rate(name, q, k, v)
            except Exception as ex:  # noqa: BLE001 (reported, not hidden)
                ent["cpu_baseline"] = {"error": f"{type(ex).__name__}: {ex}"[:300]}
        res[name] = ent
    return res


def routed_only(args, M, dev, stream, peaks):
    """The routing-only ablation on the timed workload at the same budget:
    no shared pairs, each expert holds k' = m + k keys. Device-resident
    inputs, per-stage times from the library's stage profile."""
    import torch

    c = dict(synth.CONFIGS[args.config])
    q, k, v = synth.make_inputs(c)
    c["k"] = min(c["m"] + c["k"], c["N"])
    to = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    Q, K, V = to(q), to(k), to(v)
    out = torch.empty_like(Q)
    e = torch.empty((c["B"], c["H"], c["m"], c["k"]), dtype=torch.int32, device=dev)
    r = torch.empty((c["B"], c["H"], c["N"]), dtype=torch.int32, device=dev)
    a = (c["grid_h"], c["grid_w"], c["m"], c["k"])
    for _ in range(3):
        M.mita_forward_routed(Q, K, V, *a, out=out, expert_idx=e, route=r, stream=stream)
    torch.cuda.synchronize()
    assert M.mita_sync_status(stream) == 0, M.mita_last_error()
    M.mita_profile_read(stream)
    M.mita_profile_enable(True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 10
    ev0.record(stream)
    for _ in range(n):
        M.mita_forward_routed(Q, K, V, *a, out=out, expert_idx=e, route=r, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    M.mita_profile_enable(False)
    stages = M.mita_profile_read(stream)
    assert M.mita_sync_status(stream) == 0, M.mita_last_error()
    ms = ev0.elapsed_time(ev1) / n
    w = work(c, shared=False)
    stage_ms = {s: stages[s][0] / n for s in STAGES}
    t_exp = stage_ms["expert"] / 1e3
    del Q, K, V, out
    torch.cuda.empty_cache()
    exp_tf = w["expert"]["flops"] / t_exp / 1e12 if t_exp > 0 else None
    return {"k_routed": c["k"], "queries_per_s": c["B"] * c["H"] * c["N"] / (ms / 1e3), "ms_per_step": ms,
            "roofline_frac": roofline_time(w["total"], peaks, sustained=False) / (ms / 1e3),
            "expert_tflops": exp_tf, "expert_frac": exp_tf / peaks["bf16_tflops"] if exp_tf else None,
            "peak": "burst bf16",
            "stage_ms": stage_ms}


def split_shared(args, M, dev, stream, peaks):
    """mita_forward_split on the timed workload: the shared branch folded into
    the routing kernel (the routing stage then also forms each query's
    softmax over its landmark logits, and the expert stage attends to the k
    routed keys alone). Device-resident inputs, stage times from the
    library's profile; the same FLOP count as the headline pass."""
    import torch

    c = synth.CONFIGS[args.config]
    q, k, v = synth.make_inputs(c)
    to = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    Q, K, V = to(q), to(k), to(v)
    out = torch.empty_like(Q)
    e = torch.empty((c["B"], c["H"], c["m"], c["k"]), dtype=torch.int32, device=dev)
    r = torch.empty((c["B"], c["H"], c["N"]), dtype=torch.int32, device=dev)
    a = (c["grid_h"], c["grid_w"], c["m"], c["k"])
    for _ in range(3):
        M.mita_forward_split(Q, K, V, *a, out=out, expert_idx=e, route=r, stream=stream)
    torch.cuda.synchronize()
    assert M.mita_sync_status(stream) == 0, M.mita_last_error()
    M.mita_profile_read(stream)
    M.mita_profile_enable(True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 10
    ev0.record(stream)
    for _ in range(n):
        M.mita_forward_split(Q, K, V, *a, out=out, expert_idx=e, route=r, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    M.mita_profile_enable(False)
    stages = M.mita_profile_read(stream)
    assert M.mita_sync_status(stream) == 0, M.mita_last_error()
    ms = ev0.elapsed_time(ev1) / n
    del Q, K, V, out
    torch.cuda.empty_cache()
    return {"queries_per_s": c["B"] * c["H"] * c["N"] / (ms / 1e3), "ms_per_step": ms,
            "roofline_frac": roofline_time(work(c)["total"], peaks, sustained=False) / (ms / 1e3),
            "stage_ms": {x: stages[x][0] / n for x in STAGES}}




def backward(args, M, dev, stream, peaks):
    """mita_backward on the timed workload (device-resident inputs and dO,
    the forward pass's experts and routes). FLOPs: 2.5x the forward pass's
    (the usual count for an attention backward: recomputed logits, dP, dS
    products for dQ, dK, dV), against the burst bf16 tensor peak (the
    products run on the tensor cores for m <= 256 and expert lists of at most
    512 keys, which the timed workloads are)."""
    import torch

    c = synth.CONFIGS[args.config]
    q, k, v = synth.make_inputs(c)
    to = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    Q, K, V = to(q), to(k), to(v)
    dO = to(synth.normal_bf16(q.shape, 11, 7))
    a = (c["grid_h"], c["grid_w"], c["m"], c["k"])
    _, e, r = M.mita_forward(Q, K, V, *a, stream=stream)
    dq = torch.empty(Q.shape, dtype=torch.float32, device=dev)
    dk, dv = torch.empty_like(dq), torch.empty_like(dq)
    for _ in range(3):
        M.mita_backward(Q, K, V, dO, *a, e, r, dq, dk, dv, stream=stream)
    torch.cuda.synchronize()
    assert M.mita_sync_status(stream) == 0, M.mita_last_error()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 3
    ev0.record(stream)
    for _ in range(n):
        M.mita_backward(Q, K, V, dO, *a, e, r, dq, dk, dv, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    assert M.mita_sync_status(stream) == 0, M.mita_last_error()
    ms = ev0.elapsed_time(ev1) / n
    flops = 2.5 * work(c)["total"]["flops"]
    tf = flops / (ms / 1e3) / 1e12
    del Q, K, V, dO, dq, dk, dv
    torch.cuda.empty_cache()
    pk = peaks["bf16_tflops"]
    return {"queries_per_s": c["B"] * c["H"] * c["N"] / (ms / 1e3), "ms_per_step": ms,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": pk, "unit": "TFLOP/s", "frac": tf / pk,
                         "flops": "2.5 x the forward pass's", "peak_source": "measured burst bf16"}}


def multi_expert(args, M, dev, stream, peaks, s=2):
    """s routed experts per query on the timed workload (device-resident
    inputs; one tensor-core attention pass per rank of the routes). The
    expert stage's FLOPs count s*k routed keys per query, an upper bound (a
    key shared by two chosen experts is attended once)."""
    import torch

    c = synth.CONFIGS[args.config]
    q, k, v = synth.make_inputs(c)
    to = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    Q, K, V = to(q), to(k), to(v)
    out = torch.empty_like(Q)
    e = torch.empty((c["B"], c["H"], c["m"], c["k"]), dtype=torch.int32, device=dev)
    r = torch.empty((c["B"], c["H"], c["N"], s), dtype=torch.int32, device=dev)
    a = (c["grid_h"], c["grid_w"], c["m"], c["k"], s)
    for _ in range(3):
        M.mita_forward_multi(Q, K, V, *a, out=out, expert_idx=e, route=r, stream=stream)
    torch.cuda.synchronize()
    assert M.mita_sync_status(stream) == 0, M.mita_last_error()
    M.mita_profile_read(stream)
    M.mita_profile_enable(True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 5
    ev0.record(stream)
    for _ in range(n):
        M.mita_forward_multi(Q, K, V, *a, out=out, expert_idx=e, route=r, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    M.mita_profile_enable(False)
    stages = M.mita_profile_read(stream)
    assert M.mita_sync_status(stream) == 0, M.mita_last_error()
    ms = ev0.elapsed_time(ev1) / n
    stage_ms = {x: stages[x][0] / n for x in STAGES}
    BH, N, m, kk = c["B"] * c["H"], c["N"], c["m"], c["k"]
    exp_flops = BH * 4 * N * (m + s * kk) * 64
    exp_tf = exp_flops / (stage_ms["expert"] / 1e3) / 1e12
    del Q, K, V, out
    torch.cuda.empty_cache()
    pk = peaks["bf16_tflops"]  # burst: the timed loop runs well under a second
    return {"s": s, "queries_per_s": BH * N / (ms / 1e3), "ms_per_step": ms, "stage_ms": stage_ms,
            "expert": {"bound": "tensor", "achieved": exp_tf, "peak": pk, "unit": "TFLOP/s", "frac": exp_tf / pk,
                       "flops": "4 N (m + s k) d per head (upper bound)"}}


# ---------------------------------------------------------------------------
# Full-attention comparator: plain softmax attention over all N keys by
# PyTorch's fused SDPA (a library kernel, not this library's), the baseline
# the pages' speedups are quoted against.
# ---------------------------------------------------------------------------
SDPA_BACKENDS = ("CUDNN_ATTENTION", "FLASH_ATTENTION", "EFFICIENT_ATTENTION")


def sdpa_full(Q, K, V, backend=None):
    """softmax(Q K^T / sqrt(d)) V on [B,H,N,d] bf16 device tensors through
    the first fused SDPA backend that accepts the shapes (or `backend`).
    Returns (out, backend name)."""
    import torch
    from torch.nn.attention import SDPBackend, sdpa_kernel

    last = None
    for name in ((backend,) if backend else SDPA_BACKENDS):
        try:
            with sdpa_kernel(getattr(SDPBackend, name)):
                return torch.nn.functional.scaled_dot_product_attention(Q, K, V), name
        except RuntimeError as e:  # backend refuses the shape or the device
            last = e
    raise RuntimeError(f"no fused SDPA backend ran: {last}")


def full_attention(args, dev, stream, mita_ms, max_queries=65536):
    """Full attention at the long-sequence workloads. Above max_queries the
    timed call takes the first max_queries queries against all N keys and the
    time is scaled by N / max_queries (each query's cost is the same, so the
    pass is linear in the number of queries)."""
    import torch

    res = {}
    for name in ("long64k", "long256k", args.config):
        if name in res or name not in mita_ms:
            continue
        c = synth.CONFIGS[name]
        q, k, v = synth.make_inputs(c)
        to = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        K, V = to(k), to(v)
        nq = min(c["N"], max_queries)
        Q = to(np.ascontiguousarray(q[:, :, :nq]))
        _, backend = sdpa_full(Q, K, V)
        for _ in range(2):
            sdpa_full(Q, K, V, backend)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = 3
        ev0.record(torch.cuda.current_stream(dev))
        for _ in range(n):
            sdpa_full(Q, K, V, backend)
        ev1.record(torch.cuda.current_stream(dev))
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / n * c["N"] / nq
        flops = 4 * c["B"] * c["H"] * c["N"] * c["N"] * 64
        res[name] = {"backend": backend, "ms_per_pass": ms, "queries_timed": nq * c["B"] * c["H"],
                     "tflops": flops / (ms / 1e3) / 1e12, "mita_speedup": ms / mita_ms[name]}
        del Q, K, V
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# Reference arm: the fp64 oracle on the host cores.
# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    import oracle

    if rank != 0:
        return None
    name = args.config
    c = synth.CONFIGS[name]
    q, k, v = synth.make_inputs(c)
    for _ in range(args.warmup):
        oracle_head_time(name, q, k, v, 2, 512)
    times, walls, sample = [], [], ""
    for s in range(args.steps):
        t_head, sample, wall = oracle_head_time(name, q, k, v, 16, 8192, seed=100 + s)
        times.append(t_head)
        walls.append(wall)
    t = statistics.median(times)
    value = c["N"] / t
    # ms_per_step is the measured wall time of one timed step (one sample);
    # value is the oracle's rate on a whole head, estimated from that sample
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(walls) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(name), "B": c["B"], "H": c["H"], "N": c["N"], "d": 64, "m": c["m"],
                   "k": c["k"]},
        "cpu_baseline": {"value": value, "unit": "queries/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample + "; each timed step is one such sample (ms_per_step: its measured wall "
                                            "time), value from the median over steps",
                         "estimated_ms_per_full_pass": round(t * 1e3 * c["B"] * c["H"], 1)},
        "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("mita", "reference"), default="mita")
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(synth.CONFIGS))
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--s-route", type=int, default=1, help="routed experts per query (1: the pages' configuration)")
    ap.add_argument("--only", choices=("backward",),
                    help="run one side measurement alone on --config and print its JSON (no headline line)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "mita":
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.only == "backward":
        import torch

        import mixture_top_forward_gb300 as M

        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        M.load(build_if_missing=False)
        peaks, _ = load_peaks()
        res = {"only": "backward", "config": args.config,
               "backward": backward(args, M, dev, torch.cuda.current_stream(dev), peaks)}
    elif args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch

            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
            torch.distributed.init_process_group("nccl")
        res = run_gpu(args, rank, world)
        if world > 1:
            import torch

            torch.distributed.destroy_process_group()
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
