"""fp64 CPU oracle for Gated DeltaNet prefill -- TEST INFRASTRUCTURE ONLY.

Only tests/, the smoke check in __graft_entry__ and the benchmark's
cpu_baseline / reference leg may import this package.  The CUDA library never
does, and this package never imports the CUDA library: the two share no code.

`fwd` and `bwd` wrap the plain sequential recurrence in gdn_oracle.c (the
gated delta rule, Yang et al. "Gated Delta Networks", ICLR 2025, which the
pages name as the computation of "GDN Chunked Prefill": "FlashQLA是什么" on
ollai.cn, section "FlashQLA的主要功能").  `chunked` holds an independent
chunk-wise restatement of the same forward, used only to pin this one.

Every array argument is converted to contiguous float64.  Layouts:
  q, k [B, T, H, K];  v, do [B, T, H, V];  g, beta [B, T, H];
  states [N, H, K, V];  cu_seqlens int32 [N+1] (then B == 1).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _configure(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    i, d = ctypes.c_int, ctypes.c_double
    lib.gdn_oracle_fwd.argtypes = [dp, dp, dp, dp, dp, dp, ip, i, i, i, i, i, i, d, i, d,
                                   dp, dp, ip, i, i]
    lib.gdn_oracle_fwd.restype = ctypes.c_int
    lib.gdn_oracle_bwd.argtypes = [dp, dp, dp, dp, dp, dp, ip, i, i, i, i, i, i, d, i, d,
                                   dp, dp, dp, dp, dp, dp, dp, dp, ip, i, i]
    lib.gdn_oracle_bwd.restype = ctypes.c_int
    lib.gdn_oracle_max_threads.restype = ctypes.c_int
    lib.gdn_oracle_gate.argtypes = [dp, dp, ctypes.c_long, i, dp]
    lib.gdn_oracle_gate.restype = ctypes.c_int
    lib.gdn_oracle_gate_bwd.argtypes = [dp, dp, dp, ctypes.c_long, i, dp, dp]
    lib.gdn_oracle_gate_bwd.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(_build.build()))
    return _lib


def open_library(path):
    """Opens another build of gdn_oracle.c (the mutation tests plant bugs in
    copies of the source); pass the result as `lib=` to fwd / bwd."""
    return _configure(ctypes.CDLL(path))


def max_threads() -> int:
    return int(_load().gdn_oracle_max_threads())


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a, t=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(t))


def _dims(q, v, cu_seqlens):
    B, T, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        N = int(cu.shape[0] - 1)
    else:
        cu, N = None, B
    return B, T, H, K, V, N, cu


def _units(units):
    if units is None:
        return None, 0
    u = np.ascontiguousarray(np.asarray(units, dtype=np.int32))
    return u, int(u.shape[0])


def fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None, use_l2norm=False, eps=1e-6,
        units=None, nthreads=0, lib=None):
    """Returns (o [B,T,H,V], hT [N,H,K,V]) in float64.

    `units` (optional list of n*H + h) restricts the work to those
    (sequence, head) pairs; the other entries of o and hT are left as NaN.
    """
    lib = lib or _load()
    q, k, v, g, beta, h0 = (_f64(x) for x in (q, k, v, g, beta, h0))
    B, T, H, K, V, N, cu = _dims(q, v, cu_seqlens)
    if scale is None:
        scale = K ** -0.5
    o = np.full((B, T, H, V), np.nan)
    ht = np.full((N, H, K, V), np.nan)
    ul, nu = _units(units)
    rc = lib.gdn_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                            _ptr(cu, ctypes.c_int32), N, B, T, H, K, V, float(scale),
                            int(bool(use_l2norm)), float(eps), _ptr(o), _ptr(ht),
                            _ptr(ul, ctypes.c_int32), nu, int(nthreads))
    if rc != 0:
        raise ValueError("oracle fwd rejected its arguments")
    return o, ht


def bwd(q, k, v, g, beta, do, h0=None, dht=None, cu_seqlens=None, scale=None,
        use_l2norm=False, eps=1e-6, units=None, nthreads=0, lib=None):
    """Returns dict(dq, dk, dv, dg, dbeta, dh0) in float64 (NaN outside `units`)."""
    lib = lib or _load()
    q, k, v, g, beta, h0, do, dht = (_f64(x) for x in (q, k, v, g, beta, h0, do, dht))
    B, T, H, K, V, N, cu = _dims(q, v, cu_seqlens)
    if scale is None:
        scale = K ** -0.5
    out = dict(dq=np.full((B, T, H, K), np.nan), dk=np.full((B, T, H, K), np.nan),
               dv=np.full((B, T, H, V), np.nan), dg=np.full((B, T, H), np.nan),
               dbeta=np.full((B, T, H), np.nan), dh0=np.full((N, H, K, V), np.nan))
    ul, nu = _units(units)
    rc = lib.gdn_oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                            _ptr(cu, ctypes.c_int32), N, B, T, H, K, V, float(scale),
                            int(bool(use_l2norm)), float(eps), _ptr(do), _ptr(dht),
                            _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]),
                            _ptr(out["dbeta"]), _ptr(out["dh0"]), _ptr(ul, ctypes.c_int32), nu,
                            int(nthreads))
    if rc != 0:
        raise ValueError("oracle bwd rejected its arguments")
    return out


def gate(x, a, lib=None):
    """Log decay g = -a_h * softplus(x) from gate logits x [..., H] and a [H] (float64)."""
    lib = lib or _load()
    x, a = _f64(x), _f64(a)
    H = int(a.shape[0])
    g = np.empty_like(x)
    if lib.gdn_oracle_gate(_ptr(x), _ptr(a), int(x.size // H), H, _ptr(g)) != 0:
        raise ValueError("oracle gate rejected its arguments")
    return g


def gate_bwd(x, a, dg, lib=None):
    """Gradients (dx, da) of the gate from dg = dL/dg (float64)."""
    lib = lib or _load()
    x, a, dg = _f64(x), _f64(a), _f64(dg)
    H = int(a.shape[0])
    dx = np.empty_like(x)
    da = np.empty(H)
    if lib.gdn_oracle_gate_bwd(_ptr(x), _ptr(a), _ptr(dg), int(x.size // H), H, _ptr(dx),
                               _ptr(da)) != 0:
        raise ValueError("oracle gate_bwd rejected its arguments")
    return dx, da
