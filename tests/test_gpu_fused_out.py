"""The state walk that forms O inside its chunk loop (used when the walk's CTAs
fill most of the SMs, q and k not L2-normalised): O and the final state match
the oracle, with and without intra-card sequence parallelism, and the separate
output pass does not run; with few walk CTAs the output pass does run."""
import pytest
import torch

import gdn_synth
from gpu_helpers import TOL, check, gpu_fwd, lib, oracle_fwd

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
