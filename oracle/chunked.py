"""Chunk-wise restatement of the gated delta rule forward, in torch fp64 (CPU).

TEST INFRASTRUCTURE ONLY: it exists to pin the sequential oracle in
gdn_oracle.c, never to check the CUDA path directly.  Agreement of the two
for every chunk size C (1, 16, 64, T, with a partial last chunk) is one pin;
torch autograd through this form is an independent check of the oracle's
hand-derived reverse recurrence.

The pages ("FlashQLA是什么", ollai.cn, sections "FlashQLA的主要功能" and
"FlashQLA的技术原理") describe the method as GDN *chunked* prefill without
writing the chunk form.  The form below follows from unrolling the
recurrence over one chunk of L rows with state H at its start (H = S^T,
K x V), gamma_r = g_1 + ... + g_r and D_rs = exp(gamma_r - gamma_s):

  A  = strict_lower( diag(beta) K K^T  (.)  D )
  T  = (I + A)^-1                     (the UT / WY transform)
  w  = T diag(beta * exp(gamma)) K,   u = T diag(beta) V
  U  = u - w H                        (the chunk's effective values)
  O  = scale * ( diag(exp(gamma)) Q H + (Q K^T (.) lower_incl (.) D) U )
  H' = exp(gamma_L) H + K^T diag(exp(gamma_L - gamma)) U
"""
import torch


def _decay(gam, strict):
    """D_rs = exp(gamma_r - gamma_s) on (strictly) lower entries, 0 above."""
    n = gam.shape[0]
    mask = torch.ones(n, n, dtype=torch.bool).tril(-1 if strict else 0)
    diff = gam[:, None] - gam[None, :]
    return torch.exp(torch.where(mask, diff, torch.full_like(diff, float("-inf"))))


def forward_unit(q, k, v, g, beta, h0, scale, C):
    """One (sequence, head): q, k [L, K]; v [L, V]; g, beta [L]; h0 [K, V].

    Returns (o [L, V], hT [K, V]).  Differentiable with torch autograd.
    """
    L = q.shape[0]
    H = h0
    outs = []
    for c0 in range(0, L, C):
        sl = slice(c0, min(c0 + C, L))
        Q, Kc, Vc, gc, bc = q[sl], k[sl], v[sl], g[sl], beta[sl]
        n = Q.shape[0]
        gam = torch.cumsum(gc, 0)
        A = bc[:, None] * (Kc @ Kc.T) * _decay(gam, strict=True)
        T = torch.linalg.inv(torch.eye(n, dtype=q.dtype) + A)
        w = T @ ((bc * torch.exp(gam))[:, None] * Kc)
        u = T @ (bc[:, None] * Vc)
        U = u - w @ H
        P = (Q @ Kc.T) * _decay(gam, strict=False)
        outs.append(scale * (torch.exp(gam)[:, None] * (Q @ H) + P @ U))
        H = torch.exp(gam[-1]) * H + Kc.T @ (torch.exp(gam[-1] - gam)[:, None] * U)
    o = torch.cat(outs, 0) if outs else torch.zeros(0, v.shape[1], dtype=q.dtype)
    return o, H


def l2norm(x, eps):
    return x / torch.sqrt((x * x).sum(-1, keepdim=True) + eps)


def forward(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None, C=64, use_l2norm=False,
            eps=1e-6):
    """Whole problem in the oracle's layouts (torch fp64 tensors); returns (o, hT)."""
    B, T, Hh, K = q.shape
    V = v.shape[-1]
    scale = K ** -0.5 if scale is None else scale
    if use_l2norm:
        q, k = l2norm(q, eps), l2norm(k, eps)
    if cu_seqlens is None:
        ranges = [(b, 0, T) for b in range(B)]
    else:
        cu = [int(x) for x in cu_seqlens]
        ranges = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    N = len(ranges)
    o = torch.zeros(B, T, Hh, V, dtype=q.dtype)
    hts = []
    for n, (b, t0, t1) in enumerate(ranges):
        per_head = []
        for h in range(Hh):
            s0 = h0[n, h] if h0 is not None else torch.zeros(K, V, dtype=q.dtype)
            oo, ht = forward_unit(q[b, t0:t1, h], k[b, t0:t1, h], v[b, t0:t1, h],
                                  g[b, t0:t1, h], beta[b, t0:t1, h], s0, scale, C)
            o[b, t0:t1, h] = oo
            per_head.append(ht)
        hts.append(torch.stack(per_head))
    return o, torch.stack(hts) if N else torch.zeros(0, Hh, K, V, dtype=q.dtype)
