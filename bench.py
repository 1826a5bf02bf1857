#!/usr/bin/env python
"""Throughput of GDN chunked prefill (forward + backward) on GB300.

One step = one pass of the whole path over one batch of seeded synthetic
input: forward (prep, state walk with output, intra-card sequence-parallel
maps and scan) and backward (recomputed states, reverse gradient walk,
chunk-local gradients).  Default workload: the edge / TP8 prefill shape
(B=1, T=8192, H=8, K=V=128, bf16 q/k/v, fp32 g/beta/state, sequence
parallelism forced).  Prints one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the fp64 CPU oracle (the only reference this method
has here) on a bounded sample of the same workload.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN chunked-prefill tokens/s (fwd; fwd+bwd) on 1 GB300 + % of roofline"
CHUNK = 64
GRAD_BYTES = 4          # dq, dk, dv come back in fp32 (the library's default)
L2_BYTES = 129 * 2 ** 20


# ------------------------------------------------------------------ algorithmic work
def flops_per_token_head(K, V, part):
    """Chunk-form FLOPs per token and head (C = 64, masked triangles at half):
    fwd = 3CK + 2CV + C^2/3 + 6KV ; bwd = 12KV + 6CK + 4CV + 2C^2/3."""
    C = CHUNK
    if part == "fwd":
        return 3 * C * K + 2 * C * V + C * C / 3 + 6 * K * V
    return 12 * K * V + 6 * C * K + 4 * C * V + 2 * C * C / 3


def bytes_per_token_head(K, V, e, part):
    """Inputs read once, outputs written once.  fwd: q, k, v, g, beta, o.
    bwd: q, k, v, g, beta, dO in; dq, dk, dv (fp32), dg, dbeta out."""
    if part == "fwd":
        return e * (2 * K + V) + 8 + e * V
    return e * (2 * K + V) + 8 + e * V + 4 * (2 * K + V) + 8


# Per-kernel algorithmic FLOPs per token-head processed (the kernel's share
# of the chunk form) -- used for the roofline of the dominant kernel.
def kernel_flops_per_token_head(name, K, V):
    C = CHUNK
    table = {
        "simt_prep": 2 * C * K + C * V + C * C / 3,
        "simt_walk_out": 6 * K * V + C * K + C * V,
        "simt_walk_states": 4 * K * V,
        "simt_walk_map": 4 * K * (K + V),
        "simt_dwalk_out": 6 * K * V + C * K + C * V,
        "simt_dwalk_map": 4 * K * (K + V) + C * K + C * V,
        "simt_local_grad": 6 * K * V + 6 * C * K + 3 * C * V + 2 * C * C / 3,
    }
    return table.get(name)


FP32_LANES_PER_SM = 128


# Per-kernel algorithmic HBM bytes per token-head for the tensor-core path
# (bf16 q/k/v/dO, K = V = 128, chunk C = 64; gradients of eg bytes): every
# operand the kernel needs read once, every result written once.  W^T, u^T,
# dU^T, Y^T = (dO^T P)^T and Qs are bf16 chunk tiles (2 bytes per feature per
# token); T is the bf16 64 x 64 inverse (128 bytes per token); hc / dhc are
# the bf16 chunk states (K V 2 / C bytes per token).
def kernel_bytes_per_token_head(name, K, V, e=2, eg=4):
    C = CHUNK
    t_mat = C * 2
    state = K * V * 2 / C
    table = {
        "tc_prep": e * (K + V) + 8 + 4 + 2 * (K + V) + t_mat,
        "tc_walk": e * K + 2 * (K + V) + 4 + state,
        "tc_walk_fused": 2 * e * K + 2 * (K + V) + 4 + state + e * V,   # forms O as well
        "tc_out": 2 * e * K + 2 * (K + V) + state + 4 + e * V,
        "tc_bwd_intra": e * (2 * K + V) + 4 + 2 * K + 2 * V,
        "tc_dwalk_out": e * K + 2 * K + e * V + 2 * K + 2 * V + 4 + state + 2 * V,
        "tc_dwalk_fused": 2 * e * K + 2 * K + e * V + 4 + state + 2 * V,   # forms Qs, Y^T itself
        "tc_local_grad": (e * (2 * K + 2 * V) + 2 * (K + 2 * V) + 2 * state + t_mat + 8 +
                          eg * (2 * K + V) + 8),
    }
    return table.get(name)


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture of the named kernel on the named workload, valid while the
# kernel's source file still hashes to `sha256` (otherwise reported as null).
NCU_TRAFFIC = {
    ("tc_local_grad", "edge"): {
        "file": "gdn_tc_local.cu", "bytes": 193560320 + 57232896,
        "sha256": "2b572b435ef3a0a0bf77e87a6e4a458a739daf337dfe2fd966497e9585d25cd2"},
}


def measured_traffic(name, workload):
    import hashlib
    rec = NCU_TRAFFIC.get((name, workload))
    if not rec:
        return None
    src = os.path.join(ROOT, "gated_deltanet_linear_bwd_gb300", "csrc", rec["file"])
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    return rec["bytes"] if digest == rec["sha256"] else None


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
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in self.rows for n, v in zip(names, r[4:]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(p, heads, reps_min_s=0.0):
    """fp64 oracle forward + backward on the given heads of problem p.
    Returns (seconds per pass, threads used, token-heads per pass)."""
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


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="edge")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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


def config_of(p, name, graph=False):
    m = p.meta
    return {"workload": f"{name}: B={p.B} T={p.T} H={p.H} K={p.K} V={p.V} "
                        f"{m['dtype']} q/k/v, fp32 g/beta/state, cp={m['cp']}, "
                        f"fwd (keeping its context) + bwd",
            "global_batch": p.B, "seq_len": p.T, "heads": p.H, "parallelism": "replicas",
            "l2_flush_between_steps": True,
            **({"launch": "one CUDA graph per step"} if graph else {})}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    p = workload_problem(args.workload)
    heads = list(range(p.H))
    for _ in range(args.warmup):
        oracle_sample(p, heads[:1])
    times = []
    threads = tokens_heads = None
    for _ in range(args.steps):
        dt, threads, tokens_heads = oracle_sample(p, heads)
        times.append(dt)
    ms = 1e3 * statistics.mean(times)
    tok = tokens_heads / p.H
    value = tok / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(p, args.workload),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                             "kind": "oracle",
                             "sample": f"fp64 oracle fwd+bwd over all {p.H} heads of the "
                                       f"{args.workload} workload per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def kernel_entry(name, launches, ms, total_ms, p, th, e_in):
    ent = {"name": name, "launches": launches, "ms": ms, "share": ms / total_ms}
    by_th = kernel_bytes_per_token_head(name, p.K, p.V, e_in, GRAD_BYTES)
    if by_th is not None:
        ent["gbs"] = by_th * th / (ms / launches / 1e3) / 1e9
    return ent


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

    p = workload_problem(args.workload)
    cp = p.meta["cp"]
    d = p.to(dev)
    e_in = 2 if p.meta["dtype"] == "bf16" else 4
    tokens = p.B * p.T
    stream = torch.cuda.current_stream(dev)

    def step(x):
        # a training step: the forward keeps its per-chunk context, the backward reuses it
        o, fs, saved = gdn.chunk_gated_delta_rule_fwd(x.q, x.k, x.v, x.g, x.beta,
                                                      initial_state=x.h0, output_final_state=True,
                                                      cu_seqlens=x.cu_seqlens, cp=cp,
                                                      save_ctx=True)
        grads = gdn.chunk_gated_delta_rule_bwd(x.q, x.k, x.v, x.g, x.beta, x.do, dht=x.dht,
                                               initial_state=x.h0, cu_seqlens=x.cu_seqlens, cp=cp,
                                               ctx=saved)
        return (o, fs) + tuple(grads)

    def fwd_only(x):
        return gdn.chunk_gated_delta_rule_fwd(x.q, x.k, x.v, x.g, x.beta, initial_state=x.h0,
                                              output_final_state=True, cu_seqlens=x.cu_seqlens,
                                              cp=cp)

    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def timed(fn, steps, profile=False):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        if profile:
            gdn.gdn_profile_begin()
        for i in range(steps):
            flush.fill_(float(i))                      # evict the inputs from L2 (untimed)
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        prof = gdn.gdn_profile_end() if profile else None
        if dist:
            dist.barrier()
        ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / steps
        return ms, prof

    def graphed(fn):
        # fn captured once as a CUDA graph: the library launches only on the current
        # stream and neither allocates nor synchronises inside a call, so a whole
        # step replays as one graph launch (same kernels, no per-launch host work)
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
        return graph.replay

    for _ in range(max(args.warmup, 3)):
        step(d)
    torch.cuda.synchronize(dev)
    if gdn.gdn_sync_status(stream.cuda_stream) != 0:
        raise RuntimeError("device status after warm-up: " + gdn.gdn_last_error())
    step_g = graphed(lambda: step(d))
    fwd_g = graphed(lambda: fwd_only(d))
    for _ in range(max(args.warmup, 3)):
        step_g()
        fwd_g()

    gpu_index = torch.cuda.get_device_properties(dev)
    uuid = getattr(gpu_index, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU")
                          else uuid)
    ms_step, _ = timed(step_g, args.steps)
    ms_fwd, _ = timed(fwd_g, args.steps)

    # the same step with the gate formed inside the library from raw logits
    import gdn_synth
    gx, ga = (t.to(dev) for t in gdn_synth.gate_draws(p, seed=0))

    def gated_step(x):
        o, fs, saved = gdn.chunk_gated_delta_rule_fwd(x.q, x.k, x.v, gx, x.beta,
                                                      initial_state=x.h0, output_final_state=True,
                                                      cu_seqlens=x.cu_seqlens, cp=cp,
                                                      save_ctx=True, gate_scale=ga)
        return gdn.chunk_gated_delta_rule_bwd(x.q, x.k, x.v, gx, x.beta, x.do, dht=x.dht,
                                              initial_state=x.h0, cu_seqlens=x.cu_seqlens,
                                              cp=cp, ctx=saved, gate_scale=ga)

    gated_g = graphed(lambda: gated_step(d))
    for _ in range(max(args.warmup, 3)):
        gated_g()
    ms_gated, _ = timed(gated_g, args.steps)

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

    for _ in range(max(args.warmup, 3)):
        decode_step()
    ms_dec, _ = timed(decode_step, args.steps)
    dec_bytes = 2 * dst.numel() * 4 + dn * dh * (2 * p.K + 2 * p.V) * e_in + dn * dh * 8
    # per-kernel times from the library's own CUDA events, in a separate pass: the
    # events between kernels stop them from overlapping, so they stay out of ms_step
    _, prof = timed(lambda: step(d), args.steps, profile=True)

    # end to end through the public API: pinned host inputs in, results back out
    host_in = {k: getattr(p, k) for k in ("q", "k", "v", "g", "beta", "h0", "do", "dht")}
    host_in = {k: v.pin_memory() for k, v in host_in.items() if v is not None}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    outs = step(d)
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
             for k in ("q", "k", "v", "g", "beta", "h0") if k in host_in}
        copy_stream.wait_stream(main)
        inputs_in = torch.cuda.Event()
        with torch.cuda.stream(copy_stream):
            xb = {k: host_in[k].to(dev, non_blocking=True) for k in ("do", "dht") if k in host_in}
            inputs_in.record(copy_stream)
        for t in xb.values():
            t.record_stream(main)
        o, fs, saved = gdn.chunk_gated_delta_rule_fwd(
            x["q"], x["k"], x["v"], x["g"], x["beta"], initial_state=x.get("h0"),
            output_final_state=True, cu_seqlens=d.cu_seqlens, cp=cp, save_ctx=True)
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
            initial_state=x.get("h0"), cu_seqlens=d.cu_seqlens, cp=cp, ctx=saved)
        for hbuf, t in zip(host_out[n_fwd_out:], [t for t in grads if t is not None]):
            hbuf.copy_(t, non_blocking=True)
        main.wait_stream(copy_stream)

    e2e_g = graphed(e2e_step)
    for _ in range(max(args.warmup, 3)):
        e2e_g()
    ms_e2e, _ = timed(e2e_g, args.steps)
    torch.cuda.synchronize(dev)
    for hbuf, t in zip(host_out, [t for t in outs if t is not None]):
        if not torch.equal(hbuf, t.cpu()):
            raise RuntimeError("end-to-end results differ from the device-resident step")
    clk = clocks.stop()
    status = gdn.gdn_sync_status(stream.cuda_stream)
    if status != 0:
        raise RuntimeError("device status after the timed region: " + gdn.gdn_last_error())

    ms_step, ms_fwd, ms_e2e, ms_gated, ms_dec = max_over_ranks(
        [ms_step, ms_fwd, ms_e2e, ms_gated, ms_dec], dist, dev)
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    value = job_rate(world, tokens, ms_step)
    th = tokens * p.H
    step_bytes = th * (bytes_per_token_head(p.K, p.V, e_in, "fwd") +
                       bytes_per_token_head(p.K, p.V, e_in, "bwd"))
    step_bytes += p.N * p.H * p.K * p.V * 4 * 5          # h0 (x2), hT, dhT, dh0
    step_flops = th * (flops_per_token_head(p.K, p.V, "fwd") +
                       flops_per_token_head(p.K, p.V, "bwd"))
    hbm = peaks.get("hbm_gbs", 6800.0)
    bf16 = peaks.get("bf16_tflops", 1900.0)
    t_roof = max(step_bytes / (hbm * 1e9), step_flops / (bf16 * 1e12))
    # the forward alone: inputs, O and the states (h0 in, final state out)
    fwd_bytes = th * bytes_per_token_head(p.K, p.V, e_in, "fwd") + p.N * p.H * p.K * p.V * 4 * 2
    fwd_flops = th * flops_per_token_head(p.K, p.V, "fwd")
    t_roof_fwd = max(fwd_bytes / (hbm * 1e9), fwd_flops / (bf16 * 1e12))
    total_launches = sum(s[1] for s in prof)
    dom = max(prof, key=lambda s: s[2])
    dom_name, dom_launches, dom_ms = dom
    avg_s = dom_ms / dom_launches / 1e3
    hbm_src = "measured" if "hbm_gbs" in peaks else "fallback"
    by_th = kernel_bytes_per_token_head(dom_name, p.K, p.V, e_in, GRAD_BYTES)
    if by_th is not None:
        # the tensor-core kernels move more bytes than their few MMAs can hide: HBM roofline
        roof = {"kernel": dom_name, "bound": "hbm", "unit": "GB/s",
                "achieved": by_th * th / avg_s / 1e9, "peak": hbm,
                "peak_source": f"{hbm_src} HBM copy bandwidth",
                "bytes_per_launch": by_th * th,
                "traffic": measured_traffic(dom_name, args.workload),
                "avg_launch_ms": avg_s * 1e3, "launches_per_step": dom_launches / args.steps}
    else:
        per_th = kernel_flops_per_token_head(dom_name, p.K, p.V)
        sm_max = (clk or {}).get("sm_max_mhz") or peaks.get("sm_max_mhz", 2070.0)
        n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
        alu_peak = n_sms * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
        roof = {"kernel": dom_name, "bound": "alu", "unit": "TFLOP/s",
                "achieved": None if per_th is None else per_th * th / avg_s / 1e12,
                "peak": alu_peak, "peak_source": "fp32 FMA: SMs x 128 lanes x 2 x max SM clock",
                "traffic": None, "avg_launch_ms": avg_s * 1e3,
                "launches_per_step": dom_launches / args.steps}
    roof["frac"] = None if roof["achieved"] is None else roof["achieved"] / roof["peak"]

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        dt, threads, th_s = oracle_sample(p, list(range(p.H)), reps_min_s=10.0)
        cpu = {"value": th_s / p.H / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"fp64 oracle fwd+bwd over all {p.H} heads of the {args.workload} "
                         f"workload, repeated for >= 10 s"}

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; see gdn_synth.py)", "config": config_of(p, args.workload, True),
            "fwd": {"value": job_rate(world, tokens, ms_fwd), "unit": "tokens/s",
                    "ms_per_step": ms_fwd,
                    "step_roofline": {"t_roof_ms": t_roof_fwd * 1e3,
                                      "frac": t_roof_fwd * 1e3 / ms_fwd,
                                      "bytes": fwd_bytes, "flops": fwd_flops}},
            "decode": {"value": job_rate(world, dn, ms_dec), "unit": "tokens/s",
                       "ms_per_step": ms_dec, "batch": f"{dn} sequences x {dh} heads",
                       "hbm_gbs": dec_bytes / (ms_dec / 1e3) / 1e9,
                       "frac_of_hbm": dec_bytes / (ms_dec / 1e3) / 1e9 / hbm,
                       "what": "one gdn_recurrent_step: state read and written once"},
            "gated": {"value": job_rate(world, tokens, ms_gated), "unit": "tokens/s",
                      "ms_per_step": ms_gated,
                      "what": "the same fwd+bwd step with the decay formed inside from gate "
                              "logits (gate_scale), d(logits) and d(gate_scale) returned"},
            "step_roofline": {"t_roof_ms": t_roof * 1e3, "frac": t_roof * 1e3 / ms_step,
                              "bytes": step_bytes, "flops": step_flops,
                              "peaks": {"hbm_gbs": hbm, "bf16_tflops": bf16,
                                        "source": "measured" if peaks else "fallback"}},
            "roofline": roof,
            "kernels": [kernel_entry(n, l, m, sum(s[2] for s in prof), p, th, e_in)
                        for n, l, m in prof],
            "gpu_launches": total_launches,
            "e2e": {"value": job_rate(world, tokens, ms_e2e), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "clocks": clk, "cpu_baseline": cpu}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
