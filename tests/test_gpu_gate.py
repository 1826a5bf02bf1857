"""Gate preprocessing on the GPU: g holds raw gate logits x and the library
forms the log decay -a_h softplus(x) itself (the pages' "gate preprocessing",
aivizor, FLA-flow paragraph); the backward returns the gradient with respect
to x in dg and the gradient with respect to a_h.  Compared element by element
with the oracle's gate followed by its recurrence, on the CUDA-core path
(fp32) and the tensor-core path (bf16, with and without sequence
parallelism, with a saved forward context, and the one-kernel forward)."""
import numpy as np
import pytest
import torch

import gdn_synth
import oracle
from gpu_helpers import TOL, check, lib, to_np

pytestmark = pytest.mark.gpu

CASES = [
    ("tiny", dict(T=200, H=2), "off", False, False),
    ("training", dict(B=2, T=700, H=2, h0_std=0.1), "off", False, False),
    ("training", dict(B=1, T=1500, H=2, h0_std=0.1), "force", True, False),
    # 128 (sequence, head) pairs, no context: the one-kernel forward
    ("training", dict(B=2, T=300, H=64, h0_std=0.1), "off", False, True),
]


@pytest.mark.parametrize("name,kw,cp,ctx,fuse", CASES)
def test_gated_forward_and_backward_match_the_oracle(name, kw, cp, ctx, fuse):
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA GPU")
    p = gdn_synth.make(name, **kw)
    x, a = gdn_synth.gate_draws(p, seed=3)
    tol = TOL[gdn_synth.WORKLOADS[name]["dtype"]]
    # oracle: the gate, then the recurrence, then the gate's backward
    g = oracle.gate(x, a)
    o_ref, ht_ref = oracle.fwd(p.q, p.k, p.v, g, p.beta, h0=p.h0)
    ref = oracle.bwd(p.q, p.k, p.v, g, p.beta, do=p.do, h0=p.h0, dht=p.dht)
    dx_ref, da_ref = oracle.gate_bwd(x, a, ref["dg"])
    # library: logits in, gate formed inside
    d = p.to("cuda")
    xg, ag = x.cuda(), a.cuda()
    gdn = lib()
    res = gdn.chunk_gated_delta_rule_fwd(d.q, d.k, d.v, xg, d.beta, initial_state=d.h0,
                                         output_final_state=True, cp=cp, save_ctx=ctx,
                                         gate_scale=ag, fuse_prep=fuse)
    o, fs = res[0], res[1]
    saved = res[2] if ctx else None
    dq, dk, dv, dx, db, dh0, da = gdn.chunk_gated_delta_rule_bwd(
        d.q, d.k, d.v, xg, d.beta, d.do, dht=d.dht, initial_state=d.h0, cp=cp, ctx=saved,
        gate_scale=ag)
    torch.cuda.synchronize()
    check("o", to_np(o), o_ref, tol)
    check("final_state", to_np(fs), ht_ref, tol)
    for nm, got in (("dq", dq), ("dk", dk), ("dv", dv), ("dbeta", db), ("dh0", dh0)):
        check(nm, to_np(got), ref[nm if nm != "dbeta" else "dbeta"], tol)
    check("dx (gate logits)", to_np(dx), dx_ref, tol)
    # d a_h sums the per-token gradients of one head over n tokens; with each
    # term within the per-element tolerance and independent rounding, its
    # bound is the per-element tolerance times sqrt(n)
    check("d gate_scale", to_np(da), da_ref, tol * np.sqrt(x[..., 0].numel()))
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 0


def test_autograd_gradient_of_gate_scale():
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA GPU")
    p = gdn_synth.make("tiny", T=130, H=2)
    x, a = gdn_synth.gate_draws(p, seed=4)
    g = oracle.gate(x, a)
    ref = oracle.bwd(p.q, p.k, p.v, g, p.beta, do=p.do, h0=p.h0, dht=p.dht)
    dx_ref, da_ref = oracle.gate_bwd(x, a, ref["dg"])
    d = p.to("cuda")
    xg = x.cuda().requires_grad_(True)
    ag = a.cuda().requires_grad_(True)
    o, fs = lib().chunk_gated_delta_rule(d.q, d.k, d.v, xg, d.beta, initial_state=d.h0,
                                         output_final_state=True, gate_scale=ag)
    loss = (o * d.do).sum() + (fs * d.dht).sum() if d.dht is not None else (o * d.do).sum()
    loss.backward()
    check("dx", to_np(xg.grad), dx_ref, TOL["fp32"])
    check("d gate_scale", to_np(ag.grad), da_ref, TOL["fp32"] * np.sqrt(x[..., 0].numel()))
