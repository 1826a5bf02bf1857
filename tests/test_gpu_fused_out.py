"""The walks that absorb a chunk-parallel pass when their CTAs fill most of
the SMs: the state walk that forms O (with intra-card sequence parallelism, or
with a context kept for the backward), the one-kernel forward that also does
each chunk's preparation (without either), and the reverse walk that forms P,
Qs and Y^T itself (without sequence parallelism).  Results match the oracle,
the absorbed passes do not run, and with few walk CTAs they do."""
import pytest
import torch

import gdn_synth
from gpu_helpers import TOL, check, gpu_bwd, gpu_fwd, lib, oracle_bwd, oracle_fwd, to_np

pytestmark = pytest.mark.gpu


def _kernels(p, cp, seg=0, l2=False, save_ctx=False, fuse=False):
    gdn = lib()
    d = p.to("cuda")
    gdn.gdn_profile_begin()
    res = gdn.chunk_gated_delta_rule_fwd(
        d.q, d.k, d.v, d.g, d.beta, initial_state=d.h0, output_final_state=True,
        cu_seqlens=d.cu_seqlens, use_qk_l2norm=l2, cp=cp, cp_segment_chunks=seg,
        save_ctx=save_ctx, fuse_prep=fuse)
    torch.cuda.synchronize()
    names = {n for n, _, _ in gdn.gdn_profile_end()}
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 0
    return to_np(res[0]), to_np(res[1]), names


FULL = {"tc_full_fwd"}                       # the one-kernel forward
SPLIT = {"tc_prep", "tc_walk_fused"}         # prep, then the walk that forms O


@pytest.mark.parametrize("kw,cp,seg,ctx,fuse,l2,path", [
    # 128 walk CTAs, ragged last chunk
    (dict(B=2, T=200, H=64), "off", 0, False, False, True, SPLIT),
    (dict(B=2, T=200, H=64), "off", 0, False, True, False, FULL),
    (dict(B=2, T=200, H=64), "off", 0, False, True, True, FULL),
    (dict(B=2, T=200, H=64), "off", 0, True, True, True, SPLIT),      # a context: split
    # 10 segments x 12 heads = 120 walk CTAs (sequence parallelism: split)
    (dict(B=1, T=640, H=12), "force", 1, False, True, False, SPLIT),
    # varlen, 5 x 32 walk CTAs (one sequence empty, one of a single token)
    (dict(lengths=[130, 0, 64, 257, 1], H=32), "off", 0, False, False, False, SPLIT),
    (dict(lengths=[130, 0, 64, 257, 1], H=32), "off", 0, False, True, False, FULL),
    (dict(lengths=[130, 0, 64, 257, 1], H=32), "off", 0, False, True, True, FULL),
    (dict(lengths=[130, 0, 64, 257, 1], H=32), "off", 0, True, False, False, SPLIT),
])
def test_fused_output_walk_matches_oracle(kw, cp, seg, ctx, fuse, l2, path):
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = gdn_synth.make("training", h0_std=0.1, **kw)
    o, fs, names = _kernels(p, cp, seg, l2, ctx, fuse)
    walk_ctas = (p.T // 64 if cp == "force" and seg == 1 else p.N) * p.H
    assert 4 * walk_ctas >= 3 * n_sms, "problem too small to take the fused walk"
    assert path <= names and "tc_out" not in names, names
    if path is FULL:
        assert not (SPLIT & names), names
    ro, rfs = oracle_fwd(p, l2=l2)
    check("o", o, ro, TOL["bf16"])
    check("final_state", fs, rfs, TOL["bf16"])


def test_one_kernel_forward_without_initial_state():
    p = gdn_synth.make("training", B=1, T=1000, H=128)
    d = p.to("cuda")
    gdn = lib()
    gdn.gdn_profile_begin()
    o, fs = gdn.chunk_gated_delta_rule_fwd(d.q, d.k, d.v, d.g, d.beta, output_final_state=True,
                                           fuse_prep=True)
    torch.cuda.synchronize()
    assert FULL <= {n for n, _, _ in gdn.gdn_profile_end()}
    ro, rfs = oracle_fwd(p, h0=False)
    check("o", to_np(o), ro, TOL["bf16"])
    check("final_state", to_np(fs), rfs, TOL["bf16"])


def test_few_walk_ctas_use_the_output_pass():
    p = gdn_synth.make("training", B=1, T=300, H=2, h0_std=0.1)
    o, fs, names = _kernels(p, "off", fuse=True)
    assert not (FULL & names), names
    assert "tc_out" in names and "tc_walk" in names, names
    ro, rfs = oracle_fwd(p)
    check("o", o, ro, TOL["bf16"])


def _bwd_kernels(p, cp, seg=0, l2=False):
    gdn = lib()
    gdn.gdn_profile_begin()
    g = gpu_bwd(p, cp=cp, seg=seg, l2=l2)
    torch.cuda.synchronize()
    names = {n for n, _, _ in gdn.gdn_profile_end()}
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 0
    return g, names


@pytest.mark.parametrize("kw,cp,seg,l2", [
    (dict(B=2, T=200, H=64), "off", 0, False),       # 128 reverse-walk CTAs, ragged last chunk
    (dict(B=2, T=200, H=64), "off", 0, True),
    (dict(lengths=[130, 0, 64, 257, 1], H=32), "off", 0, False),   # varlen, one sequence empty
])
def test_fused_reverse_walk_matches_oracle(kw, cp, seg, l2):
    p = gdn_synth.make("training", h0_std=0.1, dht_std=0.01, **kw)
    g, names = _bwd_kernels(p, cp, seg, l2)
    assert "tc_dwalk_fused" in names and "tc_bwd_intra" not in names, names
    r = oracle_bwd(p, l2=l2)
    for k in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        check(k, g[k], r[k], TOL["bf16"])


@pytest.mark.parametrize("kw,cp,seg", [
    (dict(B=1, T=300, H=2), "off", 0),
    (dict(B=1, T=300, H=2), "force", 1),
    # with sequence parallelism the segment-map walk reads the intra pass's Qs and
    # Y^T, so the intra pass runs however many segment walks there are
    (dict(B=1, T=630, H=12), "force", 1),
])
def test_few_reverse_walk_ctas_or_segments_use_the_intra_pass(kw, cp, seg):
    p = gdn_synth.make("training", h0_std=0.1, dht_std=0.01, **kw)
    g, names = _bwd_kernels(p, cp, seg)
    assert "tc_bwd_intra" in names and "tc_dwalk_out" in names, names
    r = oracle_bwd(p)
    for k in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        check(k, g[k], r[k], TOL["bf16"])
