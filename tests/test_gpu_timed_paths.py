"""Parity of the exact calls bench.py times, at the full workload sizes.

bench.py's step is a forward that keeps its per-chunk context followed by a
backward that reads it (bench.training_step), with intra-card sequence
parallelism forced on the edge and long-context workloads and chosen by the
library elsewhere.  Here that same step runs on the whole workload on the GPU,
and sampled (sequence, head) units of O, the final state and every gradient
are compared element by element with the fp64 oracle at the bf16 tolerance.
The kernels that ran are read from the library's tracing, so each test also
pins which path it covered (the fused reverse walk on training and varlen,
the sequence-parallel map walks on edge and long).  The gated varlen step
(bench.py's `gated` figure) is checked the same way, d(gate logits) and
d(gate_scale) included."""
import numpy as np
import pytest
import torch

import bench
import gdn_synth
from gpu_helpers import TOL, check, lib, oracle_bwd, oracle_fwd, sub_problem, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("these tests need a CUDA GPU")
    lib()


def timed_step(p, l2):
    gdn = lib()
    d = p.to("cuda")
    gdn.gdn_profile_begin()
    outs = bench.training_step(gdn, d, p.meta["cp"], l2)
    torch.cuda.synchronize()
    names = {n for n, _, _ in gdn.gdn_profile_end()}
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 0
    o, fs, dq, dk, dv, dg, db, dh0 = (to_np(t) for t in outs)
    return dict(o=o, final_state=fs, dq=dq, dk=dk, dv=dv, dg=dg, dbeta=db, dh0=dh0), names


def compare_sampled(name, got, p, heads, batches, l2):
    tol = TOL[p.meta["dtype"]]
    sub = sub_problem(p, heads=heads, batches=batches)
    ro, rfs = oracle_fwd(sub, l2=l2)
    r = oracle_bwd(sub, l2=l2)
    packed = p.cu_seqlens is not None

    def tok(x):          # [B, T, H, ...] -> sampled rows and heads
        x = x if batches is None else x[batches]
        return x[:, :, heads]

    def st(x):           # [N, H, K, V] -> sampled sequences and heads
        x = x if batches is None or packed else x[batches]
        return x[:, heads]
    errs = {"o": check(f"{name} o", tok(got["o"]), ro, tol),
            "final_state": check(f"{name} final_state", st(got["final_state"]), rfs, tol)}
    for k in ("dq", "dk", "dv", "dg", "dbeta"):
        errs[k] = check(f"{name} {k}", tok(got[k]), r[k], tol)
    if got["dh0"] is not None and r["dh0"] is not None:
        errs["dh0"] = check(f"{name} dh0", st(got["dh0"]), r["dh0"], tol)
    print(name, {k: f"{v:.2e}" for k, v in errs.items()})
    return errs


@pytest.mark.parametrize("l2", [False, True])
def test_edge_step_as_timed(l2):
    """B=1 T=8192 H=8: forward keeping its context, sequence parallelism forced,
    backward reading the context (the map walks and both segment scans run)."""
    p = gdn_synth.make("edge")
    got, names = timed_step(p, l2)
    assert {"tc_walk_map", "map_scan", "tc_dwalk_map", "map_rscan"} <= names, names
    compare_sampled("edge", got, p, heads=[0, 5], batches=None, l2=l2)


@pytest.mark.parametrize("l2", [False, True])
def test_training_step_as_timed(l2):
    """B=4 T=4096 H=32: no sequence parallelism; both fused walks with the saved
    context (the reverse walk forms P, Qs and Y^T itself)."""
    p = gdn_synth.make("training")
    got, names = timed_step(p, l2)
    assert "tc_dwalk_fused" in names and "tc_bwd_intra" not in names, names
    assert "tc_walk_fused" in names and "tc_out" not in names, names
    compare_sampled("training", got, p, heads=[1, 20], batches=[2], l2=l2)


@pytest.mark.parametrize("l2", [False, True])
def test_varlen_step_as_timed(l2):
    """16 packed sequences of 512-8192 tokens, H=32: the headline workload."""
    p = gdn_synth.make("varlen")
    got, names = timed_step(p, l2)
    assert "tc_dwalk_fused" in names and "tc_walk_fused" in names, names
    compare_sampled("varlen", got, p, heads=[7, 30], batches=None, l2=l2)


def test_long_context_step_as_timed():
    """B=1 T=65536 H=16 forward + backward with sequence parallelism (the extra
    fwd+bwd row of the long-context workload), one sampled head."""
    p = gdn_synth.make("long")
    got, names = timed_step(p, True)
    assert {"tc_walk_map", "tc_dwalk_map"} <= names, names
    compare_sampled("long", got, p, heads=[3], batches=None, l2=True)


def timed_forward(p, l2, fuse):
    gdn = lib()
    d = p.to("cuda")
    gdn.gdn_profile_begin()
    o, fs = bench.forward_step(gdn, d, p.meta["cp"], l2, fuse_prep=fuse)
    torch.cuda.synchronize()
    names = {n for n, _, _ in gdn.gdn_profile_end()}
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 0
    return to_np(o), to_np(fs), names


@pytest.mark.parametrize("name,heads,batches", [
    ("training", [1, 20], [2]),
    ("varlen", [7, 30], None),
])
@pytest.mark.parametrize("l2", [False, True])
@pytest.mark.parametrize("fuse", [False, True])
def test_forward_as_timed(name, heads, batches, l2, fuse):
    """The forward bench.py times on its own (no context kept): prep and the
    walk that forms O, or (fuse_prep) the one-kernel forward."""
    p = gdn_synth.make(name)
    o, fs, names = timed_forward(p, l2, fuse)
    if fuse:
        assert "tc_full_fwd" in names and not ({"tc_prep", "tc_walk_fused"} & names), names
    else:
        assert {"tc_prep", "tc_walk_fused"} <= names and "tc_full_fwd" not in names, names
    sub = sub_problem(p, heads=heads, batches=batches)
    ro, rfs = oracle_fwd(sub, l2=l2)
    x = o if batches is None else o[batches]
    packed = p.cu_seqlens is not None
    f = fs if batches is None or packed else fs[batches]
    tol = TOL[p.meta["dtype"]]
    e_o = check(f"{name} o", x[:, :, heads], ro, tol)
    e_s = check(f"{name} final_state", f[:, heads], rfs, tol)
    print(name, f"o {e_o:.2e} final_state {e_s:.2e}")


def test_gated_varlen_step_as_timed():
    """The bench's `gated` measurement: the varlen step with the decay formed
    inside the library from gate logits (gate_scale), forward keeping its
    context, q/k normalised inside; sampled heads of O, the final state, every
    gradient, d(logits) and d(gate_scale) against the oracle's gate followed by
    its recurrence."""
    import oracle
    p = gdn_synth.make("varlen")
    x, a = gdn_synth.gate_draws(p, seed=0)
    d = p.to("cuda")
    xg, ag = x.cuda(), a.cuda()
    gdn = lib()
    gdn.gdn_profile_begin()
    o, fs, saved = gdn.chunk_gated_delta_rule_fwd(
        d.q, d.k, d.v, xg, d.beta, initial_state=d.h0, output_final_state=True,
        cu_seqlens=d.cu_seqlens, use_qk_l2norm=True, cp=p.meta["cp"], save_ctx=True,
        gate_scale=ag)
    dq, dk, dv, dx, db, dh0, da = gdn.chunk_gated_delta_rule_bwd(
        d.q, d.k, d.v, xg, d.beta, d.do, dht=d.dht, initial_state=d.h0,
        cu_seqlens=d.cu_seqlens, use_qk_l2norm=True, cp=p.meta["cp"], ctx=saved, gate_scale=ag)
    torch.cuda.synchronize()
    names = {n for n, _, _ in gdn.gdn_profile_end()}
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 0
    assert {"tc_walk_fused", "tc_dwalk_fused", "tc_local_grad"} <= names, names
    heads = [5, 22]
    sub = sub_problem(p, heads=heads)
    xs, as_ = x[:, :, heads].contiguous(), a[heads].contiguous()
    g = oracle.gate(xs, as_)
    ro, rfs = oracle.fwd(sub.q, sub.k, sub.v, g, sub.beta, h0=sub.h0, cu_seqlens=sub.cu_seqlens,
                         use_l2norm=True)
    r = oracle.bwd(sub.q, sub.k, sub.v, g, sub.beta, do=sub.do, h0=sub.h0, dht=sub.dht,
                   cu_seqlens=sub.cu_seqlens, use_l2norm=True)
    dx_ref, da_ref = oracle.gate_bwd(xs, as_, r["dg"])
    tol = TOL["bf16"]
    tok = lambda t: to_np(t)[:, :, heads]
    check("gated o", tok(o), ro, tol)
    check("gated final_state", to_np(fs)[:, heads], rfs, tol)
    for nm, got in (("dq", dq), ("dk", dk), ("dv", dv), ("dbeta", db)):
        check(f"gated {nm}", tok(got), r[nm], tol)
    check("gated dh0", to_np(dh0)[:, heads], r["dh0"], tol)
    check("gated d(logits)", tok(dx), dx_ref, tol)
    # d a_h sums one head's per-token terms over n tokens: the per-element
    # tolerance times sqrt(n)
    check("gated d(gate_scale)", to_np(da)[heads], da_ref, tol * np.sqrt(x.shape[1]))
