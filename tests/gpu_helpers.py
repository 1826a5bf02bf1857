"""Shared helpers of the GPU tests: run the CUDA path through the C ABI and the
fp64 oracle on the same seeded inputs, and compare them element by element."""
import numpy as np
import torch

import gdn_synth
import oracle

# Max-abs tolerances: fp32 inputs 1e-4, bf16 inputs 2e-2 (on O, the final
# state and every gradient).
TOL = {"fp32": 1e-4, "bf16": 2e-2}


def lib():
    import gated_deltanet_linear_bwd_gb300 as gdn
    return gdn


def to_np(t):
    return None if t is None else t.detach().float().cpu().numpy().astype(np.float64)


def gpu_fwd(p, cp="off", l2=False, seg=0, warm=0, tau=1e-3, stats=None, h0=True, fuse=False):
    d = p.to("cuda")
    o, fs = lib().chunk_gated_delta_rule_fwd(
        d.q, d.k, d.v, d.g, d.beta, initial_state=d.h0 if h0 else None,
        output_final_state=True, cu_seqlens=d.cu_seqlens, use_qk_l2norm=l2, cp=cp,
        cp_segment_chunks=seg, cp_warmup_chunks=warm, cp_warmup_tau=tau, cp_stats=stats,
        fuse_prep=fuse)
    torch.cuda.synchronize()
    return to_np(o), to_np(fs)


def gpu_bwd(p, cp="off", l2=False, seg=0, grad_dtype=torch.float32):
    d = p.to("cuda")
    dq, dk, dv, dg, db, dh0 = lib().chunk_gated_delta_rule_bwd(
        d.q, d.k, d.v, d.g, d.beta, d.do, dht=d.dht, initial_state=d.h0,
        cu_seqlens=d.cu_seqlens, use_qk_l2norm=l2, cp=cp, cp_segment_chunks=seg,
        grad_dtype=grad_dtype)
    torch.cuda.synchronize()
    return dict(dq=to_np(dq), dk=to_np(dk), dv=to_np(dv), dg=to_np(dg), dbeta=to_np(db),
                dh0=to_np(dh0))


def sub_problem(p, heads=None, batches=None):
    return p.heads(range(p.H) if heads is None else heads, batches)


def oracle_fwd(p, l2=False, h0=True):
    return oracle.fwd(p.q, p.k, p.v, p.g, p.beta, h0=p.h0 if h0 else None,
                      cu_seqlens=p.cu_seqlens, use_l2norm=l2)


def oracle_bwd(p, l2=False):
    return oracle.bwd(p.q, p.k, p.v, p.g, p.beta, do=p.do, h0=p.h0, dht=p.dht,
                      cu_seqlens=p.cu_seqlens, use_l2norm=l2)


def max_err(a, b):
    assert a.shape == b.shape, (a.shape, b.shape)
    if a.size == 0:
        return 0.0
    assert np.isfinite(a).all()
    return float(np.abs(a - b).max())


def check(name, got, want, tol):
    e = max_err(got, want)
    assert e <= tol, f"{name}: max abs error {e:.3e} > {tol:.1e}"
    return e
