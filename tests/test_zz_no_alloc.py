"""The allocation-free forward, gdn_chunk_fwd_static.

Some callers cannot call cudaMalloc (a plugin inside a host framework that
owns all device memory, or a latency-critical thread that must not hit
cudaMalloc's implicit device synchronisation), so they cannot hand
gdn_chunk_fwd a workspace.  gdn_chunk_fwd_static takes its scratch from a
fixed area built into the library instead.  These tests call it through the
C ABI and check it against the ordinary workspace-taking entry point on two
calls in a row (the second call finds the first call's leftovers in the
shared scratch area), and that an oversized problem is refused up front.

This file is named to be collected last, so that a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import gdn_synth
from gpu_helpers import TOL, check, gpu_fwd, lib, to_np

pytestmark = pytest.mark.gpu


def static_fwd(p, cp):
    lib()
    from gated_deltanet_linear_bwd_gb300 import _abi
    from gated_deltanet_linear_bwd_gb300.api import _common
    d = p.to("cuda")
    a = _abi.gdn_fwd_args()
    B, T, H, K, V, N, dev = _common(a, d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, None,
                                    False, cp, 0)
    o = torch.empty(B, T, H, V, dtype=d.q.dtype, device=dev)
    fs = torch.empty(N, H, K, V, dtype=torch.float32, device=dev)
    a.o, a.final_state = o.data_ptr(), fs.data_ptr()
    _abi.gdn_chunk_fwd_static(a, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return to_np(o), to_np(fs)


@pytest.mark.parametrize("name,kw,cp", [
    ("training", dict(B=2, T=700, H=2, h0_std=0.1), "force"),     # tensor-core path
    ("tiny", dict(T=200, H=2, h0_std=0.1), "off"),                 # CUDA-core path
])
def test_static_scratch_forward_matches_workspace_forward(name, kw, cp):
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA GPU")
    tol = TOL[gdn_synth.WORKLOADS[name]["dtype"]]
    for seed in (11, 12):                      # two calls in a row, different inputs
        p = gdn_synth.make(name, seed=seed, **kw)
        o_s, fs_s = static_fwd(p, cp)
        o_w, fs_w = gpu_fwd(p, cp=cp)
        check(f"o (call seed {seed})", o_s, o_w, tol)
        check(f"final_state (call seed {seed})", fs_s, fs_w, tol)
    gdn = lib()
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 0


def test_oversized_problem_is_refused_before_any_work():
    gdn = lib()
    from gated_deltanet_linear_bwd_gb300 import _abi
    a = _abi.gdn_fwd_args()
    a.q = a.k = a.v = a.g = a.beta = a.o = 4096          # never dereferenced: refused first
    a.B, a.T, a.H, a.K, a.V = 1, 65536, 16, 128, 128
    a.dtype = _abi.GDN_BF16
    rc = _abi.load().gdn_chunk_fwd_static(ctypes.byref(a), None)
    assert rc == _abi.GDN_ERR_WORKSPACE
    msg = gdn.gdn_last_error()
    assert "static scratch" in msg and str(_abi.GDN_STATIC_SCRATCH_BYTES) in msg
