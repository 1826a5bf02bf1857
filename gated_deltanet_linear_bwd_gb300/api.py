"""Torch-facing wrappers over the C ABI: they allocate outputs and workspace
with torch on the tensors' device and pass raw pointers on the current
stream.  Every step of the computation runs in libgdn.so's CUDA kernels.

The call follows the pages' statement of the interface (ollai.cn page,
"如何使用FlashQLA": chunk_gated_delta_rule(q, k, v, g, beta) returning O and
the final state, with optional cu_seqlens and initial_state; "FlashQLA的主要
功能": a high-level API plus low-level fwd / bwd entry points).
"""
from typing import Optional

import torch

from . import _abi

_DT = {torch.float32: _abi.GDN_FP32, torch.bfloat16: _abi.GDN_BF16}
_CP = {"auto": _abi.GDN_CP_AUTO, "off": _abi.GDN_CP_OFF, "force": _abi.GDN_CP_FORCE}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _check(name, t, dtype=None, shape=None, device=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _common(args, q, k, v, g, beta, initial_state, cu_seqlens, scale, use_qk_l2norm, cp,
            cp_segment_chunks, gate_scale=None):
    if q.dtype not in _DT:
        raise ValueError(f"unsupported dtype {q.dtype}")
    B, T, H, K = q.shape
    V = v.shape[-1]
    dev = q.device
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    _check("q", q, q.dtype, (B, T, H, K), dev)
    _check("k", k, q.dtype, (B, T, H, K), dev)
    _check("v", v, q.dtype, (B, T, H, V), dev)
    _check("g", g, torch.float32, (B, T, H), dev)
    _check("beta", beta, torch.float32, (B, T, H), dev)
    _check("initial_state", initial_state, torch.float32, (N, H, K, V), dev)
    _check("cu_seqlens", cu_seqlens, torch.int32, None, dev)
    _check("gate_scale", gate_scale, torch.float32, (H,), dev)
    args.q, args.k, args.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    args.g, args.beta = g.data_ptr(), beta.data_ptr()
    args.initial_state = _ptr(initial_state)
    args.cu_seqlens = _ptr(cu_seqlens)
    args.B, args.T, args.H, args.K, args.V, args.N = B, T, H, K, V, N
    args.dtype = _DT[q.dtype]
    args.scale = float(scale) if scale is not None else 0.0
    args.use_qk_l2norm = int(bool(use_qk_l2norm))
    args.cp_mode = _CP[cp]
    args.cp_segment_chunks = int(cp_segment_chunks)
    args.gate_scale = _ptr(gate_scale)
    return B, T, H, K, V, N, dev


def chunk_gated_delta_rule_fwd(q, k, v, g, beta, scale=None, initial_state=None,
                               output_final_state=True, cu_seqlens=None, use_qk_l2norm=False,
                               cp="auto", cp_segment_chunks=0, cp_warmup_chunks=0,
                               cp_warmup_tau=1e-3, cp_stats=None, save_ctx=False,
                               gate_scale=None, fuse_prep=False):
    """Low-level forward: returns (o, final_state or None), or
    (o, final_state, ctx) with save_ctx=True, where ctx is the saved-context
    buffer for chunk_gated_delta_rule_bwd (None when the path keeps none).
    With `gate_scale` ([H] fp32, a_h > 0), g holds raw gate logits x and the
    log decay is -a_h * softplus(x).  fuse_prep=True asks for the one-kernel
    forward where it applies (no ctx kept, no sequence parallelism, enough
    (sequence, head) pairs to fill the GPU)."""
    a = _abi.gdn_fwd_args()
    B, T, H, K, V, N, dev = _common(a, q, k, v, g, beta, initial_state, cu_seqlens, scale,
                                    use_qk_l2norm, cp, cp_segment_chunks, gate_scale)
    o = torch.empty(B, T, H, V, dtype=q.dtype, device=dev)
    fs = torch.empty(N, H, K, V, dtype=torch.float32, device=dev) if output_final_state else None
    a.o, a.final_state = o.data_ptr(), _ptr(fs)
    a.cp_warmup_chunks = int(cp_warmup_chunks)
    a.cp_warmup_tau = float(cp_warmup_tau)
    a.cp_stats = _ptr(cp_stats)
    a.fuse_prep = int(bool(fuse_prep))
    ctx = None
    if save_ctx:
        nc = _abi.gdn_fwd_ctx_size(a)
        if nc > 0:
            ctx = torch.empty(nc, dtype=torch.uint8, device=dev)
            a.ctx = ctx.data_ptr()
    n = _abi.gdn_fwd_workspace_size(a)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    _abi.gdn_chunk_fwd(a, ws.data_ptr(), n, torch.cuda.current_stream(dev).cuda_stream)
    return (o, fs, ctx) if save_ctx else (o, fs)


def chunk_gated_delta_rule_bwd(q, k, v, g, beta, do, dht=None, scale=None, initial_state=None,
                               cu_seqlens=None, use_qk_l2norm=False, cp="auto",
                               cp_segment_chunks=0, grad_dtype=torch.float32,
                               want_dh0=True, ctx=None, gate_scale=None):
    """Low-level backward: returns (dq, dk, dv, dg, dbeta, dh0 or None), plus
    d(gate_scale) when `gate_scale` is given (dg is then the gradient with
    respect to the gate logits).  `ctx` (optional) is the buffer a forward with
    the same inputs saved."""
    a = _abi.gdn_bwd_args()
    B, T, H, K, V, N, dev = _common(a, q, k, v, g, beta, initial_state, cu_seqlens, scale,
                                    use_qk_l2norm, cp, cp_segment_chunks, gate_scale)
    _check("do", do, q.dtype, (B, T, H, V), dev)
    _check("dht", dht, torch.float32, (N, H, K, V), dev)
    if grad_dtype not in _DT:
        raise ValueError(f"unsupported grad dtype {grad_dtype}")
    dq = torch.empty(B, T, H, K, dtype=grad_dtype, device=dev)
    dk = torch.empty(B, T, H, K, dtype=grad_dtype, device=dev)
    dv = torch.empty(B, T, H, V, dtype=grad_dtype, device=dev)
    dg = torch.empty(B, T, H, dtype=torch.float32, device=dev)
    db = torch.empty(B, T, H, dtype=torch.float32, device=dev)
    dh0 = torch.empty(N, H, K, V, dtype=torch.float32, device=dev) if want_dh0 else None
    a.d_o, a.d_final_state = do.data_ptr(), _ptr(dht)
    a.grad_dtype = _DT[grad_dtype]
    a.dq, a.dk, a.dv, a.dg, a.dbeta = (t.data_ptr() for t in (dq, dk, dv, dg, db))
    a.d_initial_state = _ptr(dh0)
    a.ctx = _ptr(ctx)
    dgs = torch.empty(H, dtype=torch.float32, device=dev) if gate_scale is not None else None
    a.d_gate_scale = _ptr(dgs)
    n = _abi.gdn_bwd_workspace_size(a)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    _abi.gdn_chunk_bwd(a, ws.data_ptr(), n, torch.cuda.current_stream(dev).cuda_stream)
    if gate_scale is not None:
        return dq, dk, dv, dg, db, dh0, dgs
    return dq, dk, dv, dg, db, dh0


class _ChunkGatedDeltaRule(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, beta, initial_state, gate_scale, scale, cu_seqlens,
                use_qk_l2norm, cp):
        o, fs, saved = chunk_gated_delta_rule_fwd(q, k, v, g, beta, scale=scale,
                                                  initial_state=initial_state,
                                                  output_final_state=True,
                                                  cu_seqlens=cu_seqlens,
                                                  use_qk_l2norm=use_qk_l2norm, cp=cp,
                                                  save_ctx=True, gate_scale=gate_scale)
        ctx.save_for_backward(q, k, v, g, beta, initial_state, cu_seqlens, saved, gate_scale)
        ctx.cfg = (scale, use_qk_l2norm, cp)
        return o, fs

    @staticmethod
    def backward(ctx, do, dht):
        q, k, v, g, beta, h0, cu, saved, gs = ctx.saved_tensors
        scale, l2, cp = ctx.cfg
        out = chunk_gated_delta_rule_bwd(
            q, k, v, g, beta, do.contiguous().to(q.dtype),
            dht=None if dht is None else dht.contiguous(), scale=scale, initial_state=h0,
            cu_seqlens=cu, use_qk_l2norm=l2, cp=cp, want_dh0=h0 is not None, ctx=saved,
            gate_scale=gs)
        dq, dk, dv, dg, db, dh0 = out[:6]
        dgs = out[6] if gs is not None else None
        return (dq.to(q.dtype), dk.to(k.dtype), dv.to(v.dtype), dg, db, dh0, dgs, None, None,
                None, None)


def chunk_gated_delta_rule(q, k, v, g, beta, scale=None, initial_state=None,
                           output_final_state=False, cu_seqlens=None, use_qk_l2norm=False,
                           cp="auto", gate_scale=None):
    """High-level call: (o, final_state or None), differentiable in q, k, v, g,
    beta, initial_state and gate_scale.  With `gate_scale` ([H], a_h > 0), g
    holds raw gate logits x and the log decay is -a_h * softplus(x).  Gradients
    are cast to the inputs' dtypes only at this autograd boundary."""
    o, fs = _ChunkGatedDeltaRule.apply(q, k, v, g, beta, initial_state, gate_scale, scale,
                                       cu_seqlens, use_qk_l2norm, cp)
    return o, (fs if output_final_state else None)


def recurrent_step(q, k, v, g, beta, state, scale=None, use_qk_l2norm=False, gate_scale=None):
    """One decode step per (sequence, head): q, k [N, H, K], v [N, H, V], g, beta
    [N, H], state [N, H, K, V] fp32 (updated in place).  Returns o [N, H, V].
    With `gate_scale`, g holds gate logits as in the chunked forward."""
    N, H, K = q.shape
    V = v.shape[-1]
    dev = q.device
    if q.dtype not in _DT:
        raise ValueError(f"unsupported dtype {q.dtype}")
    _check("q", q, q.dtype, (N, H, K), dev)
    _check("k", k, q.dtype, (N, H, K), dev)
    _check("v", v, q.dtype, (N, H, V), dev)
    _check("g", g, torch.float32, (N, H), dev)
    _check("beta", beta, torch.float32, (N, H), dev)
    _check("state", state, torch.float32, (N, H, K, V), dev)
    _check("gate_scale", gate_scale, torch.float32, (H,), dev)
    o = torch.empty(N, H, V, dtype=q.dtype, device=dev)
    a = _abi.gdn_step_args()
    a.q, a.k, a.v, a.g, a.beta = (t.data_ptr() for t in (q, k, v, g, beta))
    a.gate_scale = _ptr(gate_scale)
    a.state, a.o = state.data_ptr(), o.data_ptr()
    a.N, a.H, a.K, a.V = N, H, K, V
    a.dtype = _DT[q.dtype]
    a.scale = float(scale) if scale is not None else 0.0
    a.use_qk_l2norm = int(bool(use_qk_l2norm))
    _abi.gdn_recurrent_step(a, torch.cuda.current_stream(dev).cuda_stream)
    return o
