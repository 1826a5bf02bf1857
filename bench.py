#!/usr/bin/env python
"""Throughput of GDN chunked prefill (forward; forward + backward) on GB300.

One step = one pass of the whole path over one batch of seeded synthetic
input: the forward (prep, state walk with output, and the intra-card
sequence-parallel maps and scan where the workload uses them) keeping its
per-chunk context, then the backward (reverse gradient walk, chunk-local
gradients) reading that context.  q and k are L2-normalised inside the
library (use_qk_l2norm) unless --no-l2norm is given.

Headline workload: the packed varlen batch (16 sequences of 512-8192 tokens,
H=32, K=V=128, bf16 q/k/v, fp32 g/beta/state), the largest configuration that
fits one GPU.  The training, long-context and edge workloads are reported as
extra entries.  Prints one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the fp64 CPU oracle (the only reference this method
has here) on a bounded sample of the same workload.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN chunked-prefill tokens/s (fwd; fwd+bwd) on 1 GB300 + % of roofline"
HEADLINE = "varlen"
EXTRA_WORKLOADS = ("training", "long", "edge")
WARMUP_WORKLOADS = {"edge": [0, 5], "long": [3]}     # sampled heads for the oracle check
WARMUP_CHUNKS, WARMUP_TAU = 8, 1e-3
CHUNK = 64
GRAD_BYTES = 4          # dq, dk, dv come back in fp32 (the library's default)
L2_BYTES = 129 * 2 ** 20
SUSTAINED_S = 1.2       # length of the sustained block the clocks are sampled over


# ------------------------------------------------------------------ algorithmic work
def flops_per_token_head(K, V, part):
    """Chunk-form FLOPs per token and head (C = 64, masked triangles at half):
    fwd = 3CK + 2CV + C^2/3 + 6KV ; bwd = 12KV + 6CK + 4CV + 2C^2/3."""
    C = CHUNK
    if part == "fwd":
        return 3 * C * K + 2 * C * V + C * C / 3 + 6 * K * V
    return 12 * K * V + 6 * C * K + 4 * C * V + 2 * C * C / 3


def bytes_per_token_head(K, V, e, part, eg=GRAD_BYTES):
    """Inputs read once, outputs written once.  fwd: q, k, v, g, beta in, o out.
    bwd: q, k, v, g, beta, dO in; dq, dk, dv (eg bytes each), dg, dbeta out."""
    if part == "fwd":
        return e * (2 * K + V) + 8 + e * V
    return e * (2 * K + V) + 8 + e * V + eg * (2 * K + V) + 8


# Per-kernel HBM bytes per token-head on the tensor-core path (bf16 inputs, K =
# V = 128, C = 64, gradients of eg bytes), split into ALGORITHMIC bytes (the
# method's own inputs the kernel reads and outputs it writes, each once) and
# OVERHEAD bytes (intermediates of the split design: the within-chunk cumsum
# gam, the bf16 W^T / u^T / dU^T / Qs / Y^T chunk tiles of 2 bytes per feature,
# the bf16 (I + A)^-1 of 2C bytes per token, and bf16 chunk states of 2KV/C
# bytes per token).  The roofline of a kernel counts the algorithmic bytes only.
def kernel_bytes_per_token_head(name, K, V, e=2, eg=GRAD_BYTES):
    C = CHUNK
    t_mat = 2 * C
    state = 2 * K * V / C
    table = {
        "tc_prep": (e * (K + V) + 8, 4 + 2 * (K + V) + t_mat),
        "tc_walk": (e * K, 2 * (K + V) + 4 + state),
        "tc_walk_fused": (2 * e * K + e * V, 2 * (K + V) + 4 + state),
        # the one-kernel forward: q, k, v, g, beta in, O out, nothing in between
        "tc_full_fwd": (e * (2 * K + V) + 8 + e * V, 0),
        "tc_out": (2 * e * K + e * V, 2 * (K + V) + state + 4),
        "tc_bwd_intra": (e * (2 * K + V), 4 + 2 * K + 2 * V),
        "tc_dwalk_out": (e * K + e * V, 2 * K + 2 * K + 2 * V + 4 + state + 2 * V),
        "tc_dwalk_fused": (2 * e * K + e * V, 2 * K + 4 + state + 2 * V),
        "tc_local_grad": (e * (2 * K + 2 * V) + 8 + eg * (2 * K + V) + 8,
                          2 * (K + 2 * V) + 2 * state + t_mat),
    }
    return table.get(name)


# DRAM bytes per token-head (dram__bytes_read.sum + dram__bytes_write.sum of one
# launch, divided by the token-heads it processed) from one ncu capture of the
# named kernel on the named workload; valid while the sources it was built from
# still hash to `sha256` (sha256 over the files in order; otherwise reported as
# null).  The kernels' traffic grows in proportion to the token-heads processed,
# so it is scaled to the benchmarked launch.
NCU_TRAFFIC = {
    # training workload (B=4 T=4096 H=32, 524,288 token-heads): 1,547,845,888 B
    # read + 766,588,928 B written in the captured launch
    "tc_local_grad": {"bytes_per_token_head": 2314434816 / 524288, "workload": "training",
                      "K": 128, "V": 128,
                      "files": ["gdn_tc_local.cu", "tc_ptx.cuh", "gdn_common.cuh"],
                      "sha256": "ea2b22f9082ef2928da13b7f425dda6b30c164c759daf2e0e081a62701062792"},
}


def sources_digest(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "gated_deltanet_linear_bwd_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic_per_th(name, K, V):
    rec = NCU_TRAFFIC.get(name)
    if not rec or (rec["K"], rec["V"]) != (K, V):
        return None, None
    try:
        digest = sources_digest(rec["files"])
    except OSError:
        return None, None
    if digest != rec["sha256"]:
        return None, None
    return rec["bytes_per_token_head"], rec["workload"]


# ------------------------------------------------------------------ statistics
def pct(xs, q):
    """q-th percentile (0..100) by linear interpolation."""
    s = sorted(xs)
    if not s:
        return None
    pos = (len(s) - 1) * q / 100.0
    lo, hi = int(math.floor(pos)), int(math.ceil(pos))
    return s[lo] + (s[hi] - s[lo]) * (pos - lo)


def summary(ms_list):
    return {"median_ms": statistics.median(ms_list), "p5_ms": pct(ms_list, 5),
            "p95_ms": pct(ms_list, 95), "mean_ms": statistics.mean(ms_list),
            "n": len(ms_list)}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None):
        self.rows = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if gpu_id is not None:
            cmd[1:1] = ["-i", str(gpu_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 8:
                self.rows.append(parts)

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if not self.rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in self.rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in self.rows if num(r[1]) is not None]
        pw = [num(r[2]) for r in self.rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in self.rows for n, v in zip(names, r[4:]) if v == "Active"})
        # samples under load: power well above the idle floor
        floor = min(pw) if pw else 0.0
        loaded = [num(r[0]) for r in self.rows
                  if num(r[2]) is not None and num(r[2]) > floor + 100 and num(r[0]) is not None]
        return {"sm_mhz": statistics.median(loaded or sm) if (loaded or sm) else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows), "samples_under_load": len(loaded),
                "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(p, heads, reps_min_s=0.0):
    """fp64 oracle forward + backward on the given heads of problem p (every
    sequence).  Returns (seconds per pass, threads used, token-heads per pass)."""
    import oracle
    sub = p.heads(heads)
    threads = min(oracle.max_threads(), len(heads) * sub.N)
    t0 = time.perf_counter()
    passes = 0
    while True:
        oracle.fwd(sub.q, sub.k, sub.v, sub.g, sub.beta, h0=sub.h0, cu_seqlens=sub.cu_seqlens,
                   nthreads=threads)
        oracle.bwd(sub.q, sub.k, sub.v, sub.g, sub.beta, do=sub.do, h0=sub.h0, dht=sub.dht,
                   cu_seqlens=sub.cu_seqlens, nthreads=threads)
        passes += 1
        if time.perf_counter() - t0 >= reps_min_s:
            break
    dt = (time.perf_counter() - t0) / passes
    return dt, threads, sub.B * sub.T * len(heads)


# ------------------------------------------------------------------ ranks
def max_over_ranks(values, dist=None, device=None):
    """The slowest rank's figure for each entry (max over ranks, which every rank
    receives); the figures themselves when running alone."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_rate(world, units, ms):
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return world * units / (ms / 1e3)


# ------------------------------------------------------------------ the timed calls
def training_step(gdn, x, cp, l2):
    """The benchmarked step: the forward keeps its per-chunk context and the
    backward reuses it.  Returns (o, final_state, dq, dk, dv, dg, dbeta, dh0)."""
    o, fs, saved = gdn.chunk_gated_delta_rule_fwd(x.q, x.k, x.v, x.g, x.beta,
                                                  initial_state=x.h0, output_final_state=True,
                                                  cu_seqlens=x.cu_seqlens, use_qk_l2norm=l2,
                                                  cp=cp, save_ctx=True)
    grads = gdn.chunk_gated_delta_rule_bwd(x.q, x.k, x.v, x.g, x.beta, x.do, dht=x.dht,
                                           initial_state=x.h0, cu_seqlens=x.cu_seqlens,
                                           use_qk_l2norm=l2, cp=cp, ctx=saved)
    return (o, fs) + tuple(grads)


def forward_step(gdn, x, cp, l2, **kw):
    """The benchmarked forward alone (no context kept)."""
    return gdn.chunk_gated_delta_rule_fwd(x.q, x.k, x.v, x.g, x.beta, initial_state=x.h0,
                                          output_final_state=True, cu_seqlens=x.cu_seqlens,
                                          use_qk_l2norm=l2, cp=cp, **kw)


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--extra", default=",".join(EXTRA_WORKLOADS),
                    help="comma-separated extra workloads ('' for none)")
    ap.add_argument("--no-l2norm", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-warmup-check", action="store_true")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world, local)


def workload_problem(name):
    import gdn_synth
    return gdn_synth.make(name)


def config_of(p, name, l2, graph=False):
    m = p.meta
    shape = (f"N={p.N} packed sequences of {min(m['lengths'])}-{max(m['lengths'])} tokens "
             f"({p.T} in all)" if p.cu_seqlens is not None else f"B={p.B} T={p.T}")
    return {"workload": f"{name}: {shape} H={p.H} K={p.K} V={p.V} {m['dtype']} q/k/v, fp32 "
                        f"g/beta/state, cp={m['cp']}, use_qk_l2norm={l2}; step = fwd (keeping "
                        f"its context) + bwd",
            "global_batch": p.N, "seq_len": p.T, "heads": p.H, "parallelism": "replicas",
            "l2_flush_between_steps": True,
            **({"launch": "one CUDA graph per step"} if graph else {})}


def reference_heads(p):
    return [0]


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    p = workload_problem(args.workload)
    heads = reference_heads(p)
    for _ in range(args.warmup):
        oracle_sample(p, heads)
    times = []
    threads = tokens_heads = None
    for _ in range(args.steps):
        dt, threads, tokens_heads = oracle_sample(p, heads)
        times.append(dt)
    ms = 1e3 * statistics.median(times)
    tok = tokens_heads / len(heads)              # tokens of the whole batch per sampled head
    # the whole workload has p.H heads: its tokens/s is the sampled rate / H
    value = tok / p.H / (ms / 1e3) * len(heads)
    sample = (f"fp64 oracle fwd+bwd over head(s) {heads} of the {args.workload} workload "
              f"(all {p.N} sequences, {p.T} tokens) per step; tokens/s scaled to all {p.H} heads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(p, args.workload, not args.no_l2norm),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                             "host_cores": os.cpu_count(), "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


class Timer:
    """Per-step CUDA events on the launching stream, the L2 flushed between steps
    outside the events."""

    def __init__(self, torch, dev, stream, dist):
        self.torch, self.dev, self.stream, self.dist = torch, dev, stream, dist
        self.flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def run(self, fn, steps, profile_gdn=None):
        torch = self.torch
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        torch.cuda.synchronize(self.dev)
        if self.dist:
            self.dist.barrier()
        torch.cuda.synchronize(self.dev)
        if profile_gdn:
            profile_gdn.gdn_profile_begin()
        for i in range(steps):
            self.flush.fill_(float(i))                 # evict the inputs from L2 (untimed)
            starts[i].record(self.stream)
            fn()
            ends[i].record(self.stream)
        torch.cuda.synchronize(self.dev)
        prof = profile_gdn.gdn_profile_end() if profile_gdn else None
        if self.dist:
            self.dist.barrier()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)], prof


def graphed(torch, dev, fn):
    """fn captured once as a CUDA graph: the library launches only on the current
    stream and neither allocates nor synchronises inside a call, so a whole step
    replays as one graph launch (same kernels, no per-launch host work)."""
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(2):
            fn()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    torch.cuda.synchronize(dev)
    return graph.replay, graph


def roofline_terms(p, e_in, peaks):
    th = p.B * p.T * p.H
    hbm = peaks.get("hbm_gbs", 6800.0)
    bf16 = peaks.get("bf16_tflops", 1900.0)
    states = p.N * p.H * p.K * p.V * 4
    fwd_bytes = th * bytes_per_token_head(p.K, p.V, e_in, "fwd") + states * (2 if p.h0 is not None else 1)
    fwd_flops = th * flops_per_token_head(p.K, p.V, "fwd")
    bwd_bytes = th * bytes_per_token_head(p.K, p.V, e_in, "bwd")
    bwd_bytes += states * ((1 if p.dht is not None else 0) + 1)       # dh_T in, dh0 out
    step_bytes = fwd_bytes + bwd_bytes
    step_flops = fwd_flops + th * flops_per_token_head(p.K, p.V, "bwd")
    t_step = max(step_bytes / (hbm * 1e9), step_flops / (bf16 * 1e12))
    t_fwd = max(fwd_bytes / (hbm * 1e9), fwd_flops / (bf16 * 1e12))
    return dict(th=th, hbm=hbm, bf16=bf16, step_bytes=step_bytes, step_flops=step_flops,
                fwd_bytes=fwd_bytes, fwd_flops=fwd_flops, t_step=t_step, t_fwd=t_fwd)


def kernel_table(prof, steps, p, e_in):
    th = p.B * p.T * p.H
    total = sum(s[2] for s in prof)
    out = []
    for name, launches, ms in prof:
        ent = {"name": name, "launches_per_step": launches / steps, "ms_per_step": ms / steps,
               "share": ms / total}
        b = kernel_bytes_per_token_head(name, p.K, p.V, e_in, GRAD_BYTES)
        if b is not None:
            per_launch_s = ms / launches / 1e3
            ent["alg_gbs"] = b[0] * th / per_launch_s / 1e9
            ent["all_gbs"] = (b[0] + b[1]) * th / per_launch_s / 1e9
        out.append(ent)
    return out


def dominant_roofline(prof, p, e_in, rt, peaks_src):
    dom = max(prof, key=lambda s: s[2])
    name, launches, ms = dom
    th = rt["th"]
    avg_s = ms / launches / 1e3
    b = kernel_bytes_per_token_head(name, p.K, p.V, e_in, GRAD_BYTES)
    if b is None:
        return {"kernel": name, "bound": "hbm", "unit": "GB/s", "achieved": None,
                "peak": rt["hbm"], "frac": None, "traffic": None,
                "avg_launch_ms": avg_s * 1e3}
    alg, ovh = b[0] * th, b[1] * th
    tr_th, tr_wl = measured_traffic_per_th(name, p.K, p.V)
    traffic = None if tr_th is None else tr_th * th
    achieved = alg / avg_s / 1e9
    return {"kernel": name, "bound": "hbm", "unit": "GB/s", "achieved": achieved,
            "peak": rt["hbm"], "frac": achieved / rt["hbm"],
            "peak_source": f"{peaks_src} HBM copy bandwidth (MEASURED_PEAKS hbm_gbs)",
            "bytes_per_launch": alg, "overhead_bytes": ovh,
            "achieved_incl_overhead": (alg + ovh) / avg_s / 1e9,
            "traffic": traffic,
            "traffic_ratio": None if traffic is None else traffic / alg,
            "traffic_source": None if tr_wl is None else
            f"ncu DRAM read+write per token-head of one launch on the {tr_wl} workload, "
            f"scaled to this launch's token-heads",
            "avg_launch_ms": avg_s * 1e3, "launches_per_step": None}


def one_kernel_entry(world, tokens, ms, rt, prof, steps, p, e_in):
    """The forward with fuse_prep set: one kernel (prep inside the walk) where it
    applies, else the same two-kernel path as `fwd`."""
    m = statistics.median(ms)
    return {"value": job_rate(world, tokens, m), "unit": "tokens/s", "ms_per_step": m,
            "step_roofline_frac": rt["t_fwd"] * 1e3 / m,
            "kernels": kernel_table(prof, steps, p, e_in),
            "what": "the forward with fuse_prep=1: W, u and gam made and used inside one "
                    "kernel where no context is kept, sequence parallelism is off and the "
                    "(sequence, head) pairs fill the GPU"}


def measure_workload(torch, gdn, name, args, timer, dev, peaks, peaks_src, l2, headline=False):
    """Times the fwd+bwd step and the forward of one workload (graph replays)."""
    p = workload_problem(name)
    cp = p.meta["cp"]
    d = p.to(dev)
    e_in = 2 if p.meta["dtype"] == "bf16" else 4
    tokens = p.B * p.T
    steps = args.steps
    for _ in range(max(args.warmup, 3)):
        training_step(gdn, d, cp, l2)
    torch.cuda.synchronize(dev)
    st = timer.stream
    if gdn.gdn_sync_status(st.cuda_stream) != 0:
        raise RuntimeError(f"{name}: device status after warm-up: " + gdn.gdn_last_error())
    step_g, g1 = graphed(torch, dev, lambda: training_step(gdn, d, cp, l2))
    fwd_g, g2 = graphed(torch, dev, lambda: forward_step(gdn, d, cp, l2))
    # the one-kernel forward (fuse_prep), where it applies; elsewhere the same as fwd_g
    fwd1_g, g3 = graphed(torch, dev, lambda: forward_step(gdn, d, cp, l2, fuse_prep=True))
    for _ in range(max(args.warmup, 3)):
        step_g()
        fwd_g()
        fwd1_g()
    res = {"p": p, "d": d, "cp": cp, "e_in": e_in, "tokens": tokens, "graphs": (g1, g2, g3)}
    clocks = None
    if headline:
        props = torch.cuda.get_device_properties(dev)
        uuid = getattr(props, "uuid", None)
        clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None and
                              not str(uuid).startswith("GPU") else uuid)
    ms_step, _ = timer.run(step_g, steps)
    if headline:
        # the same step repeated for >= SUSTAINED_S, so that the clock samples cover a
        # sustained run; reported beside the K-step figures
        n_s = max(steps, int(math.ceil(SUSTAINED_S * 1e3 / statistics.median(ms_step))))
        ms_sus, _ = timer.run(step_g, n_s)
        res["sustained"] = summary(ms_sus)
        res["clocks"] = clocks.stop()
    ms_fwd, _ = timer.run(fwd_g, steps)
    ms_fwd1, _ = timer.run(fwd1_g, steps)
    # per-kernel times from the library's own CUDA events, in a separate eager pass:
    # events between kernels stop them from overlapping, so they stay out of ms_step
    _, prof = timer.run(lambda: training_step(gdn, d, cp, l2), steps, profile_gdn=gdn)
    _, prof_fwd = timer.run(lambda: forward_step(gdn, d, cp, l2), steps, profile_gdn=gdn)
    _, prof_fwd1 = timer.run(lambda: forward_step(gdn, d, cp, l2, fuse_prep=True), steps,
                             profile_gdn=gdn)
    if gdn.gdn_sync_status(st.cuda_stream) != 0:
        raise RuntimeError(f"{name}: device status after the timed region: " +
                           gdn.gdn_last_error())
    res.update(ms_step=ms_step, ms_fwd=ms_fwd, prof=prof, prof_fwd=prof_fwd, ms_fwd1=ms_fwd1,
               prof_fwd1=prof_fwd1)
    return res


def warmup_report(torch, gdn, name, heads, timer, dev, args, l2):
    """The warmup shortcut (flag): its error against the oracle on sampled heads,
    reported apart from the exact path, the fraction of heads that took it, and
    the forward's time with and without it."""
    import numpy as np
    import oracle
    p = workload_problem(name)
    d = p.to(dev)
    stats = torch.zeros(2, dtype=torch.int32, device=dev)
    kw = dict(cp_warmup_chunks=WARMUP_CHUNKS, cp_warmup_tau=WARMUP_TAU)
    o_w, fs_w = forward_step(gdn, d, "force", l2, cp_stats=stats, **kw)
    o_x, fs_x = forward_step(gdn, d, "force", l2)
    torch.cuda.synchronize(dev)
    took, total = stats.tolist()
    sub = p.heads(heads)
    ro, rfs = oracle.fwd(sub.q, sub.k, sub.v, sub.g, sub.beta, h0=sub.h0,
                         cu_seqlens=sub.cu_seqlens, use_l2norm=l2)

    def err(a, b):
        return float(np.abs(a.float().cpu().numpy().astype(np.float64) - b).max())
    e_w = max(err(o_w[:, :, heads], ro), err(fs_w[:, heads], rfs))
    e_x = max(err(o_x[:, :, heads], ro), err(fs_x[:, heads], rfs))
    fw, _ = graphed(torch, dev, lambda: forward_step(gdn, d, "force", l2, **kw))
    fx, _ = graphed(torch, dev, lambda: forward_step(gdn, d, "force", l2))
    for _ in range(3):
        fw()
        fx()
    t_w, _ = timer.run(fw, args.steps)
    t_x, _ = timer.run(fx, args.steps)
    return {"window_chunks": WARMUP_CHUNKS, "tau": WARMUP_TAU,
            "heads_taking_shortcut": took, "heads_under_cp": total,
            "fraction": took / total if total else None,
            "pages_claim": "6-8 chunks enough for 60-80% of heads",
            "max_abs_err_vs_oracle": e_w, "exact_path_max_abs_err_vs_oracle": e_x,
            "sampled_heads": heads, "fwd_ms_median": statistics.median(t_w),
            "exact_fwd_ms_median": statistics.median(t_x)}


def run_ours(args, rank, world, local):
    import torch
    import gated_deltanet_linear_bwd_gb300 as gdn

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except OSError:
        pass
    peaks_src = "measured" if "hbm_gbs" in peaks else "fallback"
    l2 = not args.no_l2norm
    stream = torch.cuda.current_stream(dev)
    timer = Timer(torch, dev, stream, dist)

    h = measure_workload(torch, gdn, args.workload, args, timer, dev, peaks, peaks_src, l2,
                         headline=True)
    p, d, cp, e_in, tokens = h["p"], h["d"], h["cp"], h["e_in"], h["tokens"]

    # end to end through the public API, called eagerly every step: pinned host
    # inputs in, every result back to pinned host memory
    host_in = {k: getattr(p, k) for k in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens",
                                          "do", "dht")}
    host_in = {k: v.pin_memory() for k, v in host_in.items() if v is not None}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    outs = training_step(gdn, d, cp, l2)
    host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs
                if o is not None]
    d2h = sum(o.numel() * o.element_size() for o in host_out)
    copy_stream = torch.cuda.Stream(dev)
    n_fwd_out = sum(1 for o in outs[:2] if o is not None)

    def e2e_step():
        # The forward's inputs go first; the backward's own inputs (dO, d final
        # state) travel on a second stream while the forward runs, and O and the
        # final state travel back while the backward runs.
        main = torch.cuda.current_stream(dev)
        x = {k: host_in[k].to(dev, non_blocking=True)
             for k in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens") if k in host_in}
        copy_stream.wait_stream(main)
        inputs_in = torch.cuda.Event()
        with torch.cuda.stream(copy_stream):
            xb = {k: host_in[k].to(dev, non_blocking=True) for k in ("do", "dht") if k in host_in}
            inputs_in.record(copy_stream)
        for t in xb.values():
            t.record_stream(main)
        o, fs, saved = gdn.chunk_gated_delta_rule_fwd(
            x["q"], x["k"], x["v"], x["g"], x["beta"], initial_state=x.get("h0"),
            output_final_state=True, cu_seqlens=x.get("cu_seqlens"), use_qk_l2norm=l2, cp=cp,
            save_ctx=True)
        fwd_out = [t for t in (o, fs) if t is not None]
        copy_stream.wait_stream(main)
        with torch.cuda.stream(copy_stream):
            for hbuf, t in zip(host_out[:n_fwd_out], fwd_out):
                hbuf.copy_(t, non_blocking=True)
        for t in fwd_out:
            t.record_stream(copy_stream)
        main.wait_event(inputs_in)
        grads = gdn.chunk_gated_delta_rule_bwd(
            x["q"], x["k"], x["v"], x["g"], x["beta"], xb["do"], dht=xb.get("dht"),
            initial_state=x.get("h0"), cu_seqlens=x.get("cu_seqlens"), use_qk_l2norm=l2,
            cp=cp, ctx=saved)
        for hbuf, t in zip(host_out[n_fwd_out:], [t for t in grads if t is not None]):
            hbuf.copy_(t, non_blocking=True)
        main.wait_stream(copy_stream)

    for _ in range(max(args.warmup, 3)):
        e2e_step()
    ms_e2e, _ = timer.run(e2e_step, args.steps)
    torch.cuda.synchronize(dev)
    for hbuf, t in zip(host_out, [t for t in outs if t is not None]):
        if not torch.equal(hbuf, t.cpu()):
            raise RuntimeError("end-to-end results differ from the device-resident step")
    # The same steps as a user's loop would run them: step k + 1's inputs travel up
    # while step k computes and step k - 1's results travel down (three streams;
    # inputs at most two steps ahead).  Every step's copies are inside the timed
    # region, which spans the whole loop; the per-step figure is that time / steps.
    h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    fwd_keys = [k for k in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens", "do", "dht")
                if k in host_in]

    def e2e_pipeline(n):
        main = torch.cuda.current_stream(dev)
        h2d_stream.wait_stream(main)          # nothing moves before the timed region opens
        computed = []
        for step in range(n):
            if step >= 2:
                h2d_stream.wait_event(computed[step - 2])
            with torch.cuda.stream(h2d_stream):
                x = {k: host_in[k].to(dev, non_blocking=True) for k in fwd_keys}
                arrived = torch.cuda.Event()
                arrived.record(h2d_stream)
            main.wait_event(arrived)
            for t in x.values():
                t.record_stream(main)
            o, fs, saved = gdn.chunk_gated_delta_rule_fwd(
                x["q"], x["k"], x["v"], x["g"], x["beta"], initial_state=x.get("h0"),
                output_final_state=True, cu_seqlens=x.get("cu_seqlens"), use_qk_l2norm=l2,
                cp=cp, save_ctx=True)
            grads = gdn.chunk_gated_delta_rule_bwd(
                x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], dht=x.get("dht"),
                initial_state=x.get("h0"), cu_seqlens=x.get("cu_seqlens"), use_qk_l2norm=l2,
                cp=cp, ctx=saved)
            done = torch.cuda.Event()
            done.record(main)
            computed.append(done)
            res = [t for t in (o, fs) + tuple(grads) if t is not None]
            d2h_stream.wait_event(done)
            with torch.cuda.stream(d2h_stream):
                for hbuf, t in zip(host_out, res):
                    hbuf.copy_(t, non_blocking=True)
            for t in res:
                t.record_stream(d2h_stream)
        main.wait_stream(d2h_stream)

    e2e_pipeline(max(args.warmup, 3))
    ms_pipe = []
    for _ in range(3):
        ms, _ = timer.run(lambda: e2e_pipeline(args.steps), 1)
        ms_pipe.append(ms[0] / args.steps)
    torch.cuda.synchronize(dev)
    for hbuf, t in zip(host_out, [t for t in outs if t is not None]):
        if not torch.equal(hbuf, t.cpu()):
            raise RuntimeError("pipelined end-to-end results differ from the device-resident step")
    # the serial end-to-end step captured once as a CUDA graph (no per-call host work)
    e2e_g, e2e_graph_obj = graphed(torch, dev, e2e_step)
    for _ in range(3):
        e2e_g()
    ms_e2e_graph, _ = timer.run(e2e_g, args.steps)
    torch.cuda.synchronize(dev)

    # the same step with the decay formed inside the library from raw gate logits
    import gdn_synth
    gx, ga = (t.to(dev) for t in gdn_synth.gate_draws(p, seed=0))

    def gated_step():
        o, fs, saved = gdn.chunk_gated_delta_rule_fwd(
            d.q, d.k, d.v, gx, d.beta, initial_state=d.h0, output_final_state=True,
            cu_seqlens=d.cu_seqlens, use_qk_l2norm=l2, cp=cp, save_ctx=True, gate_scale=ga)
        return gdn.chunk_gated_delta_rule_bwd(
            d.q, d.k, d.v, gx, d.beta, d.do, dht=d.dht, initial_state=d.h0,
            cu_seqlens=d.cu_seqlens, use_qk_l2norm=l2, cp=cp, ctx=saved, gate_scale=ga)

    gated_g, gated_graph = graphed(torch, dev, gated_step)
    for _ in range(3):
        gated_g()
    ms_gated, _ = timer.run(gated_g, args.steps)
    del gated_g, gated_graph, gx, ga

    # decode: one token for each of 64 sequences x 32 heads from resident fp32 states
    dn, dh = 64, 32
    dgen = torch.Generator(device="cpu").manual_seed(7)
    dq_ = (torch.randn(dn, dh, p.K, generator=dgen) / p.K ** 0.5).to(dev, d.q.dtype)
    dk_ = (torch.randn(dn, dh, p.K, generator=dgen) / p.K ** 0.5).to(dev, d.q.dtype)
    dv_ = torch.randn(dn, dh, p.V, generator=dgen).to(dev, d.q.dtype)
    dg_ = -torch.rand(dn, dh, generator=dgen).to(dev)
    db_ = torch.rand(dn, dh, generator=dgen).to(dev)
    dst = (0.1 * torch.randn(dn, dh, p.K, p.V, generator=dgen)).to(dev)

    def decode_step():
        gdn.recurrent_step(dq_, dk_, dv_, dg_, db_, dst)

    for _ in range(3):
        decode_step()
    ms_dec, _ = timer.run(decode_step, args.steps)
    dec_bytes = 2 * dst.numel() * 4 + dn * dh * (2 * p.K + 2 * p.V) * e_in + dn * dh * 8
    del dq_, dk_, dv_, dg_, db_, dst

    # everything the headline line needs, before its tensors are released
    rt = roofline_terms(p, e_in, peaks)
    head = {"ms_step": h["ms_step"], "ms_fwd": h["ms_fwd"], "prof": h["prof"],
            "prof_fwd": h["prof_fwd"], "sustained": h["sustained"], "clocks": h["clocks"],
            "ms_fwd1": h["ms_fwd1"], "prof_fwd1": h["prof_fwd1"]}
    del h, outs, host_out, e2e_g, e2e_graph_obj, d
    torch.cuda.empty_cache()

    extra = {}
    for name in [w for w in args.extra.split(",") if w and w != args.workload]:
        x = measure_workload(torch, gdn, name, args, timer, dev, peaks, peaks_src, l2)
        xp = x["p"]
        xrt = roofline_terms(xp, x["e_in"], peaks)
        ms_s, ms_f = statistics.median(x["ms_step"]), statistics.median(x["ms_fwd"])
        extra[name] = {
            "config": config_of(xp, name, l2, True)["workload"],
            "fwd_bwd": {"value": job_rate(world, x["tokens"], ms_s), "unit": "tokens/s",
                        **summary(x["ms_step"]),
                        "step_roofline_frac": xrt["t_step"] * 1e3 / ms_s,
                        "t_roof_ms": xrt["t_step"] * 1e3},
            "fwd": {"value": job_rate(world, x["tokens"], ms_f), "unit": "tokens/s",
                    **summary(x["ms_fwd"]),
                    "step_roofline_frac": xrt["t_fwd"] * 1e3 / ms_f,
                    "t_roof_ms": xrt["t_fwd"] * 1e3},
            "fwd_one_kernel": one_kernel_entry(world, x["tokens"], x["ms_fwd1"], xrt,
                                               x["prof_fwd1"], args.steps, xp, x["e_in"]),
            "roofline": dominant_roofline(x["prof"], xp, x["e_in"], xrt, peaks_src),
            "kernels": kernel_table(x["prof"], args.steps, xp, x["e_in"])}
        del x
        torch.cuda.empty_cache()

    warm = {}
    if not args.no_warmup_check and world == 1:
        for name, heads in WARMUP_WORKLOADS.items():
            warm[name] = warmup_report(torch, gdn, name, heads, timer, dev, args, l2)
            torch.cuda.empty_cache()

    status = gdn.gdn_sync_status(stream.cuda_stream)
    if status != 0:
        raise RuntimeError("device status after the timed regions: " + gdn.gdn_last_error())

    med_step = statistics.median(head["ms_step"])
    med_fwd = statistics.median(head["ms_fwd"])
    med_e2e = statistics.median(ms_e2e)
    med_e2e_g = statistics.median(ms_e2e_graph)
    med_pipe = statistics.median(ms_pipe)
    med_gated, med_dec = statistics.median(ms_gated), statistics.median(ms_dec)
    med_fwd1 = statistics.median(head["ms_fwd1"])
    med_step, med_fwd, med_e2e, med_e2e_g, med_gated, med_dec, med_fwd1, med_pipe = max_over_ranks(
        [med_step, med_fwd, med_e2e, med_e2e_g, med_gated, med_dec, med_fwd1, med_pipe], dist, dev)
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        heads = reference_heads(p)
        dt, threads, th_s = oracle_sample(p, heads, reps_min_s=10.0)
        cpu = {"value": (th_s / p.H) / dt, "unit": "tokens/s", "cores": threads,
               "host_cores": os.cpu_count(), "kind": "oracle",
               "sample": f"fp64 oracle fwd+bwd over head(s) {heads} of the {args.workload} "
                         f"workload (all {p.N} sequences), repeated for >= 10 s; tokens/s "
                         f"scaled to all {p.H} heads"}

    prof = head["prof"]
    roof = dominant_roofline(prof, p, e_in, rt, peaks_src)
    roof["launches_per_step"] = {n: l for n, l, _ in prof}[roof["kernel"]] / args.steps
    launches_per_step = sum(s[1] for s in prof) / args.steps
    line = {"metric": METRIC, "value": job_rate(world, tokens, med_step), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": med_step, "step_stats": summary(head["ms_step"]),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; see gdn_synth.py)",
            "config": config_of(p, args.workload, l2, True),
            "fwd": {"value": job_rate(world, tokens, med_fwd), "unit": "tokens/s",
                    "ms_per_step": med_fwd, "stats": summary(head["ms_fwd"]),
                    "step_roofline": {"t_roof_ms": rt["t_fwd"] * 1e3,
                                      "frac": rt["t_fwd"] * 1e3 / med_fwd,
                                      "bytes": rt["fwd_bytes"], "flops": rt["fwd_flops"]},
                    "kernels": kernel_table(head["prof_fwd"], args.steps, p, e_in)},
            "fwd_one_kernel": one_kernel_entry(world, tokens, [med_fwd1], rt, head["prof_fwd1"],
                                               args.steps, p, e_in),
            "sustained": head["sustained"],
            "step_roofline": {"t_roof_ms": rt["t_step"] * 1e3,
                              "frac": rt["t_step"] * 1e3 / med_step,
                              "bytes": rt["step_bytes"], "flops": rt["step_flops"],
                              "peaks": {"hbm_gbs": rt["hbm"], "bf16_tflops": rt["bf16"],
                                        "source": peaks_src}},
            "roofline": roof,
            "kernels": kernel_table(prof, args.steps, p, e_in),
            "gpu_launches": int(round(launches_per_step * args.steps)),
            "e2e": {"value": job_rate(world, tokens, med_pipe), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": med_pipe, "stats": summary(ms_pipe),
                    "what": f"{args.steps} steps of eager public-API calls (fwd keeping its "
                            "context, bwd), every step's inputs from pinned host memory and every "
                            "result back to it inside the timed region, consecutive steps "
                            "overlapped as a training loop would (step k+1's inputs in while step "
                            "k computes and step k-1's results go out); time of the whole loop / "
                            "steps, three loops"},
            "e2e_serial": {"value": job_rate(world, tokens, med_e2e), "unit": "tokens/s",
                           "ms_per_step": med_e2e, "stats": summary(ms_e2e),
                           "what": "the same step with nothing overlapped across steps: each "
                                   "step timed alone"},
            "e2e_graph": {"value": job_rate(world, tokens, med_e2e_g), "unit": "tokens/s",
                          "ms_per_step": med_e2e_g,
                          "what": "the serial end-to-end step captured once as a CUDA graph"},
            "gated": {"value": job_rate(world, tokens, med_gated), "unit": "tokens/s",
                      "ms_per_step": med_gated,
                      "what": "the same fwd+bwd step with the decay formed inside from gate "
                              "logits (gate_scale), d(logits) and d(gate_scale) returned"},
            "decode": {"value": job_rate(world, dn, med_dec), "unit": "tokens/s",
                       "ms_per_step": med_dec, "batch": f"{dn} sequences x {dh} heads",
                       "hbm_gbs": dec_bytes / (med_dec / 1e3) / 1e9,
                       "frac_of_hbm": dec_bytes / (med_dec / 1e3) / 1e9 / rt["hbm"],
                       "what": "one gdn_recurrent_step: state read and written once"},
            "workloads": extra, "warmup_shortcut": warm,
            "clocks": head["clocks"], "cpu_baseline": cpu}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
