"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle,
element by element, on seeded inputs.  Small cases span several chunks and a
ragged tail; the full-size workloads compare sampled (sequence, head) units
in the same launch configuration the benchmark times."""
import numpy as np
import pytest
import torch

import gdn_synth
import oracle
from gpu_helpers import (TOL, check, gpu_bwd, gpu_fwd, lib, oracle_bwd, oracle_fwd,
                         sub_problem, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("these tests need a CUDA GPU")
    lib()


def full_check(p, cp="off", l2=False, seg=0, bwd=True):
    tol = TOL[p.meta["dtype"]]
    o, fs = gpu_fwd(p, cp=cp, l2=l2, seg=seg)
    ro, rfs = oracle_fwd(p, l2=l2)
    errs = dict(o=check("o", o, ro, tol), final=check("final_state", fs, rfs, tol))
    if bwd:
        g = gpu_bwd(p, cp=cp, l2=l2, seg=seg)
        r = oracle_bwd(p, l2=l2)
        for k in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
            errs[k] = check(k, g[k], r[k], tol)
    return errs


# ------------------------------------------------------------- tiny workload (fp32)
@pytest.mark.parametrize("cp", ["off", "force"])
@pytest.mark.parametrize("l2", [False, True])
def test_tiny_workload(cp, l2):
    p = gdn_synth.make("tiny", normalise=not l2)
    full_check(p, cp=cp, l2=l2, seg=1)


def test_tiny_with_states_and_gradient_in():
    p = gdn_synth.make("tiny", h0_std=0.1, dht_std=0.1)
    full_check(p)


@pytest.mark.parametrize("K,V", [(128, 64), (64, 128), (128, 128)])
def test_ragged_tail_and_mixed_dims(K, V):
    p = gdn_synth.make("tiny", B=2, T=200, H=3, K=K, V=V, h0_std=0.1, dht_std=0.1)
    full_check(p)
    full_check(p, cp="force", seg=2)


@pytest.mark.parametrize("T", [0, 1, 63, 64, 65])
def test_short_sequences(T):
    p = gdn_synth.make("tiny", B=2, T=T, H=2, h0_std=0.1, dht_std=0.1)
    full_check(p)


@pytest.mark.parametrize("cp", ["off", "force"])
def test_varlen_with_empty_and_ragged_sequences(cp):
    p = gdn_synth.make("tiny", lengths=[0, 1, 63, 64, 65, 130, 7, 0], H=2, h0_std=0.1,
                       dht_std=0.1)
    full_check(p, cp=cp, seg=1)


def test_null_initial_state_equals_explicit_zeros():
    p = gdn_synth.make("tiny", T=150, h0_std=0.1)
    o_null, fs_null = gpu_fwd(p, h0=False)
    p.h0 = torch.zeros_like(p.h0)
    o_zero, fs_zero = gpu_fwd(p)
    np.testing.assert_array_equal(o_null, o_zero)
    np.testing.assert_array_equal(fs_null, fs_zero)


# ------------------------------------------------------------- bf16, several tiles
@pytest.mark.parametrize("cp,seg", [("off", 0), ("force", 0), ("force", 3), ("force", 1)])
def test_bf16_multi_chunk(cp, seg):
    p = gdn_synth.make("training", B=2, T=700, H=2, h0_std=0.1, dht_std=0.01)
    full_check(p, cp=cp, seg=seg)


def test_bf16_l2norm_and_bf16_grads():
    p = gdn_synth.make("training", B=1, T=300, H=2, normalise=False, h0_std=0.1, dht_std=0.01)
    full_check(p, l2=True)
    g = gpu_bwd(p, l2=True, grad_dtype=torch.bfloat16)
    r = oracle_bwd(p, l2=True)
    for k in ("dq", "dk", "dv"):
        check(k, g[k], r[k], TOL["bf16"])


def test_cp_result_does_not_depend_on_segmenting():
    p = gdn_synth.make("edge", T=2048, H=2)
    ref, ref_fs = gpu_fwd(p, cp="off")
    for seg in (1, 2, 5, 32):
        o, fs = gpu_fwd(p, cp="force", seg=seg)
        assert np.abs(o - ref).max() <= 1e-2
        assert np.abs(fs - ref_fs).max() <= 1e-3


# ------------------------------------------------------------- saved forward context
@pytest.mark.parametrize("kw,cp", [
    (dict(B=2, T=300, H=2), "off"),
    (dict(B=1, T=700, H=2), "force"),
    (dict(lengths=[130, 0, 64, 257], H=2), "auto"),
])
def test_backward_with_saved_context_matches_recompute_and_oracle(kw, cp):
    gdn = lib()
    p = gdn_synth.make("training", h0_std=0.1, dht_std=0.01, **kw)
    d = p.to("cuda")
    o, fs, saved = gdn.chunk_gated_delta_rule_fwd(d.q, d.k, d.v, d.g, d.beta, initial_state=d.h0,
                                                  cu_seqlens=d.cu_seqlens, cp=cp, save_ctx=True)
    assert saved is not None and saved.numel() > 0
    with_ctx = gdn.chunk_gated_delta_rule_bwd(d.q, d.k, d.v, d.g, d.beta, d.do, dht=d.dht,
                                              initial_state=d.h0, cu_seqlens=d.cu_seqlens, cp=cp,
                                              ctx=saved)
    torch.cuda.synchronize()
    r = oracle_bwd(p)
    ro, rfs = oracle_fwd(p)
    check("o (saving)", to_np(o), ro, TOL["bf16"])
    check("final_state (saving)", to_np(fs), rfs, TOL["bf16"])
    g = gpu_bwd(p, cp=cp)
    for name, x in zip(["dq", "dk", "dv", "dg", "dbeta", "dh0"], with_ctx):
        check(f"{name} with ctx", to_np(x), r[name], TOL["bf16"])
        assert np.abs(to_np(x) - g[name]).max() <= 1e-3, name   # same arithmetic either way


def test_fp32_path_keeps_no_context_and_warmup_refuses_one():
    gdn = lib()
    p = gdn_synth.make("tiny", T=100).to("cuda")
    o, fs, saved = gdn.chunk_gated_delta_rule_fwd(p.q, p.k, p.v, p.g, p.beta, save_ctx=True)
    assert saved is None
    pb = gdn_synth.make("edge", T=1024, H=2).to("cuda")
    with pytest.raises(gdn.GdnError, match="warmup"):
        gdn.chunk_gated_delta_rule_fwd(pb.q, pb.k, pb.v, pb.g, pb.beta, cp="force",
                                       cp_warmup_chunks=4, save_ctx=True)


# ------------------------------------------------------------- warmup shortcut (flag)
def test_warmup_shortcut_error_is_reported_separately():
    # strongly decaying heads: the 6-chunk window forgets all but ~e^-40 of the state
    p = gdn_synth.make("edge", T=2048, H=4, a_lo=0.5)
    stats = torch.zeros(2, dtype=torch.int32, device="cuda")
    o_w, fs_w = gpu_fwd(p, cp="force", seg=4, warm=6, tau=1e-6, stats=stats)
    ro, rfs = oracle_fwd(p)
    err = max(np.abs(o_w - ro).max(), np.abs(fs_w - rfs).max())
    took, total = stats.tolist()
    print(f"warmup shortcut: {took}/{total} heads, max abs error vs oracle {err:.3e}")
    assert total == 4 and took >= 1
    assert err <= TOL["bf16"]


# ------------------------------------------------------------- device-side checks
def test_bad_cu_seqlens_sets_the_status_word():
    gdn = lib()
    p = gdn_synth.make("tiny", lengths=[100, 50, 50], H=2)
    p.cu_seqlens = torch.tensor([0, 100, 60, 200], dtype=torch.int32)   # not monotone
    gpu_fwd(p)
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 6
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 0  # cleared


@pytest.mark.parametrize("kw,fuse", [
    (dict(B=1, T=300, H=2), False),          # prep, state walk, output pass
    (dict(B=2, T=200, H=64), False),         # the walk that forms O
    (dict(B=2, T=200, H=64), True),          # the one-kernel forward
])
def test_bounded_wait_gives_up_and_reports_timeout(kw, fuse):
    """Spin limit 0: every bounded wait of the tensor-core kernels gives up at
    once; the status word reports GDN_ERR_TIMEOUT and the context stays usable."""
    gdn = lib()
    p = gdn_synth.make("training", h0_std=0.1, **kw)
    stream = torch.cuda.current_stream().cuda_stream
    assert gdn.gdn_sync_status(stream) == 0
    gdn.gdn_set_spin_limit(0)
    try:
        gpu_fwd(p, fuse=fuse)
        assert gdn.gdn_sync_status(stream) == 5
    finally:
        gdn.gdn_set_spin_limit(-1)
    o, fs = gpu_fwd(p, fuse=fuse)
    ro, rfs = oracle_fwd(p)
    check("o after timeout", o, ro, TOL["bf16"])
    check("final_state after timeout", fs, rfs, TOL["bf16"])
    assert gdn.gdn_sync_status(stream) == 0


@pytest.mark.parametrize("kw,cp", [
    (dict(B=1, T=300, H=2), "off"),          # intra pass, reverse walk, local gradients
    (dict(B=2, T=200, H=64), "off"),         # the reverse walk that forms the intra terms
    (dict(B=1, T=640, H=2), "force"),        # segment-map walks and scans
])
def test_backward_bounded_waits_give_up_and_report_timeout(kw, cp):
    """The same for every backward kernel: with spin limit 0 each gives up at its
    first wait, the status word reports GDN_ERR_TIMEOUT, and a backward run
    afterwards matches the oracle."""
    gdn = lib()
    p = gdn_synth.make("training", h0_std=0.1, dht_std=0.01, **kw)
    stream = torch.cuda.current_stream().cuda_stream
    assert gdn.gdn_sync_status(stream) == 0
    gdn.gdn_set_spin_limit(0)
    try:
        gpu_bwd(p, cp=cp)
        assert gdn.gdn_sync_status(stream) == 5
    finally:
        gdn.gdn_set_spin_limit(-1)
    g = gpu_bwd(p, cp=cp)
    assert gdn.gdn_sync_status(stream) == 0
    r = oracle_bwd(p)
    for k in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        check(k + " after timeout", g[k], r[k], TOL["bf16"])


def test_autograd_wrapper_matches_low_level_backward():
    gdn = lib()
    p = gdn_synth.make("tiny", T=130, h0_std=0.1).to("cuda")
    leaves = [x.clone().requires_grad_(True) for x in (p.q, p.k, p.v, p.g, p.beta, p.h0)]
    o, fs = gdn.chunk_gated_delta_rule(*leaves[:5], initial_state=leaves[5],
                                       output_final_state=True)
    dfs = torch.randn_like(fs)
    (o * p.do).sum().backward(retain_graph=True)
    grads1 = [x.grad.clone() for x in leaves]
    for x in leaves:
        x.grad = None
    ((o * p.do).sum() + (fs * dfs).sum()).backward()
    dq, dk, dv, dg, db, dh0 = gdn.chunk_gated_delta_rule_bwd(p.q, p.k, p.v, p.g, p.beta, p.do,
                                                             dht=dfs, initial_state=p.h0)
    for got, want in zip([x.grad for x in leaves], [dq, dk, dv, dg, db, dh0]):
        torch.testing.assert_close(got, want, atol=1e-5, rtol=1e-5)
    assert grads1[0].abs().sum() > 0


def test_profiler_reports_every_launch():
    gdn = lib()
    p = gdn_synth.make("tiny", T=130)
    gdn.gdn_profile_begin()
    gpu_fwd(p)
    stats = gdn.gdn_profile_end()
    names = [s[0] for s in stats]
    assert any("prep" in n for n in names) and any("walk" in n for n in names)
    assert all(s[1] >= 1 and s[2] > 0 for s in stats)


# ------------------------------------------------------------- full-size workloads
def sampled_units_check(name, heads, batches=None, bwd=False):
    p = gdn_synth.make(name)
    cp = p.meta["cp"]
    tol = TOL[p.meta["dtype"]]
    o, fs = gpu_fwd(p, cp=cp)
    sub = sub_problem(p, heads=heads, batches=batches)
    ro, rfs = oracle_fwd(sub)
    o_s = o[:, :, heads] if batches is None else o[batches][:, :, heads]
    fs_s = fs[:, heads] if batches is None or p.cu_seqlens is not None else fs[batches][:, heads]
    check(f"{name} o", o_s, ro, tol)
    check(f"{name} final_state", fs_s, rfs, tol)
    if bwd:
        g = gpu_bwd(p, cp=cp)
        r = oracle_bwd(sub)
        for k in ("dq", "dk", "dv", "dg", "dbeta"):
            x = g[k][batches] if batches is not None else g[k]
            check(f"{name} {k}", x[:, :, heads], r[k], tol)
        x = g["dh0"][batches] if batches is not None else g["dh0"]
        check(f"{name} dh0", x[:, heads], r["dh0"], tol)


def test_full_edge_workload_sampled():
    sampled_units_check("edge", heads=[0, 5], bwd=True)


def test_full_long_workload_sampled():
    sampled_units_check("long", heads=[3])


def test_full_varlen_workload_sampled():
    sampled_units_check("varlen", heads=[7, 30])


def test_full_training_workload_sampled():
    sampled_units_check("training", heads=[1, 20], batches=[2], bwd=True)


@pytest.mark.parametrize("name,kw,cp", [
    ("tiny", dict(T=130, H=2), "off"),                   # CUDA-core path, fp32
    ("training", dict(B=1, T=300, H=2), "off"),          # tensor cores: output and intra passes
    ("training", dict(B=2, T=200, H=64), "off"),         # the fused walks
    ("training", dict(B=1, T=640, H=2), "force"),        # sequence parallelism
])
def test_explicit_scale_matches_oracle(name, kw, cp):
    """A caller's own `scale` (here 0.3 instead of K^-1/2) reaches every
    product that carries it, forward and backward, with and without q/k
    normalisation inside."""
    gdn = lib()
    p = gdn_synth.make(name, h0_std=0.1, dht_std=0.01, **kw)
    d = p.to("cuda")
    tol = TOL[gdn_synth.WORKLOADS[name]["dtype"]]
    for l2 in (False, True):
        o, fs = gdn.chunk_gated_delta_rule_fwd(d.q, d.k, d.v, d.g, d.beta, scale=0.3,
                                               initial_state=d.h0, output_final_state=True,
                                               use_qk_l2norm=l2, cp=cp)
        dq, dk, dv, dg, db, dh0 = gdn.chunk_gated_delta_rule_bwd(
            d.q, d.k, d.v, d.g, d.beta, d.do, dht=d.dht, scale=0.3, initial_state=d.h0,
            use_qk_l2norm=l2, cp=cp)
        torch.cuda.synchronize()
        ro, rfs = oracle.fwd(p.q, p.k, p.v, p.g, p.beta, h0=p.h0, scale=0.3, use_l2norm=l2)
        r = oracle.bwd(p.q, p.k, p.v, p.g, p.beta, do=p.do, h0=p.h0, dht=p.dht, scale=0.3,
                       use_l2norm=l2)
        check(f"o l2={l2}", to_np(o), ro, tol)
        check(f"final_state l2={l2}", to_np(fs), rfs, tol)
        for k, x in (("dq", dq), ("dk", dk), ("dv", dv), ("dg", dg), ("dbeta", db), ("dh0", dh0)):
            check(f"{k} l2={l2}", to_np(x), r[k], tol)
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 0


@pytest.mark.parametrize("kw,cp", [
    (dict(B=1, T=300, H=2), "off"),
    (dict(B=2, T=200, H=64), "off"),         # fused walks
    (dict(B=1, T=640, H=2), "force"),        # sequence parallelism
])
def test_optional_outputs_left_out(kw, cp):
    """No final state asked of the forward, no d(initial state) of the backward,
    no initial state and no d(final state) given: the outputs that are asked
    for still match the oracle (which takes the missing states as zeros)."""
    gdn = lib()
    p = gdn_synth.make("training", **kw)
    d = p.to("cuda")
    o, fs = gdn.chunk_gated_delta_rule_fwd(d.q, d.k, d.v, d.g, d.beta, output_final_state=False,
                                           cp=cp)
    assert fs is None
    dq, dk, dv, dg, db, dh0 = gdn.chunk_gated_delta_rule_bwd(
        d.q, d.k, d.v, d.g, d.beta, d.do, cp=cp, want_dh0=False)
    assert dh0 is None
    torch.cuda.synchronize()
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 0
    ro, _ = oracle.fwd(p.q, p.k, p.v, p.g, p.beta)
    r = oracle.bwd(p.q, p.k, p.v, p.g, p.beta, do=p.do)
    check("o", to_np(o), ro, TOL["bf16"])
    for k, x in (("dq", dq), ("dk", dk), ("dv", dv), ("dg", dg), ("dbeta", db)):
        check(k, to_np(x), r[k], TOL["bf16"])
