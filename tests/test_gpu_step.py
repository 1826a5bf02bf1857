"""The decode step (gdn_recurrent_step): token-by-token steps from an initial
state must reproduce the oracle's sequential recurrence over the same tokens
(outputs of every step and the state after the last one), on fp32 and bf16,
K, V in {64, 128}, with and without q/k normalisation and the gate; one step
over enough (sequence, head) pairs that every persistent CTA cycles its
state stages several times; and a chunked prefill followed by decode steps
must continue the same recurrence."""
import numpy as np
import pytest
import torch

import gdn_synth
import oracle
from gpu_helpers import TOL, check, lib, to_np

pytestmark = pytest.mark.gpu


def _steps(p, l2=False, gate=None, scale=None):
    d = p.to("cuda")
    state = (d.h0.clone() if d.h0 is not None
             else torch.zeros(p.B, p.H, p.K, p.V, device="cuda"))
    xg, ag = (None, None) if gate is None else (gate[0].cuda(), gate[1].cuda())
    outs = []
    for t in range(p.T):
        g = (xg if xg is not None else d.g)[:, t].contiguous()
        o = lib().recurrent_step(d.q[:, t].contiguous(), d.k[:, t].contiguous(),
                                 d.v[:, t].contiguous(), g, d.beta[:, t].contiguous(), state,
                                 use_qk_l2norm=l2, gate_scale=ag, scale=scale)
        outs.append(o)
    torch.cuda.synchronize()
    return to_np(torch.stack(outs, 1)), to_np(state)


@pytest.mark.parametrize("name,K,V,l2,gated", [
    ("tiny", 64, 64, False, False), ("tiny", 64, 64, True, True),
    ("tiny", 128, 64, False, False), ("tiny", 64, 128, True, False),
    ("training", 128, 128, False, False), ("training", 128, 128, True, False),
    ("training", 128, 128, False, True),
    ("training", 128, 64, True, False), ("training", 64, 128, False, True),
])
def test_steps_reproduce_the_recurrence(name, K, V, l2, gated):
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA GPU")
    p = gdn_synth.make(name, B=3, T=7, H=2, K=K, V=V, h0_std=0.3, normalise=not l2)
    gate = gdn_synth.gate_draws(p, seed=9) if gated else None
    g = oracle.gate(*gate) if gated else p.g
    o_ref, ht_ref = oracle.fwd(p.q, p.k, p.v, g, p.beta, h0=p.h0, use_l2norm=l2)
    o, st = _steps(p, l2, gate)
    tol = TOL[gdn_synth.WORKLOADS[name]["dtype"]]
    check("o (every step)", o, o_ref, tol)
    check("state after the last step", st, ht_ref, tol)


@pytest.mark.parametrize("name,K,V,l2", [
    ("training", 128, 128, False),     # 4096 half-state items, 27 per CTA
    ("training", 128, 128, True),
    ("tiny", 128, 128, False),         # fp32 inputs
    ("training", 64, 64, False),       # whole-state items of 16 KB
])
def test_one_step_over_many_units(name, K, V, l2):
    """One step for 64 sequences x 32 heads (the bench's decode batch) against
    the oracle's recurrence over one token from the same state."""
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA GPU")
    p = gdn_synth.make(name, B=64, T=1, H=32, K=K, V=V, h0_std=0.3, normalise=not l2)
    o_ref, ht_ref = oracle.fwd(p.q, p.k, p.v, p.g, p.beta, h0=p.h0, use_l2norm=l2)
    o, st = _steps(p, l2)
    tol = TOL[gdn_synth.WORKLOADS[name]["dtype"]]
    check("o", o, o_ref, tol)
    check("state", st, ht_ref, tol)


def test_prefill_then_decode_continues_the_recurrence():
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA GPU")
    p = gdn_synth.make("training", B=2, T=200, H=2, h0_std=0.1)
    n_pre = 195
    d = p.to("cuda")
    o_pre, fs = lib().chunk_gated_delta_rule_fwd(
        d.q[:, :n_pre].contiguous(), d.k[:, :n_pre].contiguous(), d.v[:, :n_pre].contiguous(),
        d.g[:, :n_pre].contiguous(), d.beta[:, :n_pre].contiguous(), initial_state=d.h0,
        output_final_state=True)
    outs = []
    for t in range(n_pre, p.T):
        outs.append(lib().recurrent_step(d.q[:, t].contiguous(), d.k[:, t].contiguous(),
                                         d.v[:, t].contiguous(), d.g[:, t].contiguous(),
                                         d.beta[:, t].contiguous(), fs))
    torch.cuda.synchronize()
    o_ref, ht_ref = oracle.fwd(p.q, p.k, p.v, p.g, p.beta, h0=p.h0)
    tol = TOL["bf16"]
    check("prefill o", to_np(o_pre), o_ref[:, :n_pre], tol)
    check("decode o", to_np(torch.stack(outs, 1)), o_ref[:, n_pre:], tol)
    check("state", to_np(fs), ht_ref, tol)


def test_empty_batch_is_a_no_op():
    gdn = lib()
    from gated_deltanet_linear_bwd_gb300 import _abi
    a = _abi.gdn_step_args()
    a.N, a.H, a.K, a.V, a.dtype = 0, 4, 128, 128, _abi.GDN_BF16
    assert _abi.load().gdn_recurrent_step(a, None) == _abi.GDN_OK
    a.N, a.K = 2, 96
    assert _abi.load().gdn_recurrent_step(a, None) == _abi.GDN_ERR_UNSUPPORTED
    assert "96" in gdn.gdn_last_error()


def test_steps_with_an_explicit_scale():
    p = gdn_synth.make("training", B=3, T=5, H=4, h0_std=0.3)
    o_ref, ht_ref = oracle.fwd(p.q, p.k, p.v, p.g, p.beta, h0=p.h0, scale=0.3, use_l2norm=True)
    o, st = _steps(p, True, scale=0.3)
    check("o (every step)", o, o_ref, TOL["bf16"])
    check("state after the last step", st, ht_ref, TOL["bf16"])
