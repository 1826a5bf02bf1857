"""The walks that absorb a chunk-parallel pass when their CTAs fill most of
the SMs (q and k not L2-normalised): the state walk that forms O (with and
without intra-card sequence parallelism) and the reverse walk that forms P, Qs
and Y^T itself (without it).  Results match the oracle, the absorbed pass does
not run, and with few walk CTAs it does."""
import pytest
import torch

import gdn_synth
from gpu_helpers import TOL, check, gpu_bwd, gpu_fwd, lib, oracle_bwd, oracle_fwd

pytestmark = pytest.mark.gpu


def _kernels(p, cp, seg=0):
    gdn = lib()
    gdn.gdn_profile_begin()
    o, fs = gpu_fwd(p, cp=cp, seg=seg)
    torch.cuda.synchronize()
    names = {n for n, _, _ in gdn.gdn_profile_end()}
    return o, fs, names


@pytest.mark.parametrize("kw,cp,seg", [
    (dict(B=2, T=200, H=64), "off", 0),             # 128 walk CTAs, ragged last chunk
    (dict(B=1, T=640, H=12), "force", 1),           # 10 segments x 12 heads = 120 walk CTAs
    (dict(lengths=[130, 0, 64, 257, 1], H=32), "off", 0),   # varlen, 5 x 32 walk CTAs (one sequence empty)
])
def test_fused_output_walk_matches_oracle(kw, cp, seg):
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = gdn_synth.make("training", h0_std=0.1, **kw)
    o, fs, names = _kernels(p, cp, seg)
    walk_ctas = (p.T // 64 if cp == "force" and seg == 1 else p.N) * p.H
    assert 4 * walk_ctas >= 3 * n_sms, "problem too small to take the fused walk"
    assert "tc_out" not in names and "tc_walk_fused" in names, names
    ro, rfs = oracle_fwd(p)
    check("o", o, ro, TOL["bf16"])
    check("final_state", fs, rfs, TOL["bf16"])


def test_few_walk_ctas_use_the_output_pass():
    p = gdn_synth.make("training", B=1, T=300, H=2, h0_std=0.1)
    o, fs, names = _kernels(p, "off")
    assert "tc_out" in names and "tc_walk" in names, names
    ro, rfs = oracle_fwd(p)
    check("o", o, ro, TOL["bf16"])


def _bwd_kernels(p, cp):
    gdn = lib()
    gdn.gdn_profile_begin()
    g = gpu_bwd(p, cp=cp)
    torch.cuda.synchronize()
    names = {n for n, _, _ in gdn.gdn_profile_end()}
    return g, names


@pytest.mark.parametrize("kw", [
    dict(B=2, T=200, H=64),                          # 128 reverse-walk CTAs, ragged last chunk
    dict(lengths=[130, 0, 64, 257, 1], H=32),        # varlen, one sequence empty
])
def test_fused_reverse_walk_matches_oracle(kw):
    p = gdn_synth.make("training", h0_std=0.1, dht_std=0.01, **kw)
    g, names = _bwd_kernels(p, "off")
    assert "tc_dwalk_fused" in names and "tc_bwd_intra" not in names, names
    r = oracle_bwd(p)
    for k in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        check(k, g[k], r[k], TOL["bf16"])


def test_few_reverse_walk_ctas_use_the_intra_pass():
    p = gdn_synth.make("training", B=1, T=300, H=2, h0_std=0.1, dht_std=0.01)
    g, names = _bwd_kernels(p, "off")
    assert "tc_bwd_intra" in names and "tc_dwalk_out" in names, names
