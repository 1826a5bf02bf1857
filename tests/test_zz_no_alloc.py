"""The allocation-free forward, gdn_chunk_fwd_static.

Some callers cannot call cudaMalloc (a plugin inside a host framework that
owns all device memory, or a latency-critical thread that must not hit
cudaMalloc's implicit device synchronisation), so they cannot hand
gdn_chunk_fwd a workspace.  gdn_chunk_fwd_static takes its scratch from a
fixed area built into the library instead.  These tests call it through the
C ABI and check:

- that it matches the ordinary workspace-taking entry point bit for bit (both
  run the same kernels under the same plan), on two calls in a row with
  different inputs, after a first call of the same shape has filled every
  scratch region it uses with NaN (so a region read before it is written
  would show up in the outputs), and that it matches the oracle;
- the varlen sequence tables, the sequence-parallel maps and the warmup
  decision regions as well (a packed batch with sequence parallelism and the
  warmup shortcut on);
- that a call after the first one changes the device's free memory by nothing;
- that an oversized problem is refused up front.

This file is named to be collected last, so that a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import gdn_synth
from gpu_helpers import TOL, check, lib, oracle_fwd, to_np

pytestmark = pytest.mark.gpu


def _args(d, cp, warm=0, tau=1e-3):
    from gated_deltanet_linear_bwd_gb300 import _abi
    from gated_deltanet_linear_bwd_gb300.api import _common
    a = _abi.gdn_fwd_args()
    B, T, H, K, V, N, dev = _common(a, d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, None,
                                    False, cp, 0)
    a.cp_warmup_chunks, a.cp_warmup_tau = warm, tau
    o = torch.empty(B, T, H, V, dtype=d.q.dtype, device=dev)
    fs = torch.empty(N, H, K, V, dtype=torch.float32, device=dev)
    a.o, a.final_state = o.data_ptr(), fs.data_ptr()
    return a, o, fs


def static_fwd(d, cp, **kw):
    from gated_deltanet_linear_bwd_gb300 import _abi
    a, o, fs = _args(d, cp, **kw)
    _abi.gdn_chunk_fwd_static(a, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return o, fs


def workspace_fwd(d, cp, **kw):
    from gated_deltanet_linear_bwd_gb300 import _abi
    a, o, fs = _args(d, cp, **kw)
    n = _abi.gdn_fwd_workspace_size(a)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    _abi.gdn_chunk_fwd(a, ws.data_ptr(), n, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return o, fs


def poisoned(p):
    """The same shapes with NaN q, k, v, g and beta: a forward over them leaves
    NaN in every floating-point scratch region it writes."""
    d = p.to("cuda")
    for name in ("q", "k", "v", "g", "beta"):
        setattr(d, name, torch.full_like(getattr(d, name), float("nan")))
    return d


CASES = [
    ("training", dict(B=2, T=700, H=2, h0_std=0.1), dict(cp="force")),    # tensor-core path
    ("tiny", dict(T=200, H=2, h0_std=0.1), dict(cp="off")),                # CUDA-core path
    ("training", dict(lengths=[700, 0, 64, 333, 1], H=2, h0_std=0.1),     # varlen + CP + warmup
     dict(cp="force", warm=2, tau=0.5)),
]


@pytest.mark.parametrize("name,kw,call", CASES)
def test_static_scratch_forward_matches_workspace_forward(name, kw, call):
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA GPU")
    gdn = lib()
    tol = TOL[gdn_synth.WORKLOADS[name]["dtype"]]
    first = gdn_synth.make(name, seed=10, **kw)
    o_p, _ = static_fwd(poisoned(first), **call)
    assert torch.isnan(o_p.float()).any(), "the poisoning call left no NaN behind"
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 0
    for seed in (11, 12):                      # two calls in a row, different inputs
        p = gdn_synth.make(name, seed=seed, **kw)
        d = p.to("cuda")
        o_s, fs_s = (to_np(t) for t in static_fwd(d, **call))
        o_w, fs_w = (to_np(t) for t in workspace_fwd(d, **call))
        assert np.isfinite(o_s).all() and np.isfinite(fs_s).all()
        np.testing.assert_array_equal(o_s, o_w)
        np.testing.assert_array_equal(fs_s, fs_w)
        if not call.get("warm"):
            ro, rfs = oracle_fwd(p)
            check(f"o vs oracle (seed {seed})", o_s, ro, tol)
            check(f"final_state vs oracle (seed {seed})", fs_s, rfs, tol)
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 0


def test_static_forward_takes_no_device_memory():
    lib()
    d = gdn_synth.make("training", B=2, T=700, H=2, h0_std=0.1).to("cuda")
    from gated_deltanet_linear_bwd_gb300 import _abi
    a, o, fs = _args(d, "force")
    stream = torch.cuda.current_stream().cuda_stream
    _abi.gdn_chunk_fwd_static(a, stream)          # first call: per-device set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _abi.gdn_chunk_fwd_static(a, stream)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


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


def test_bad_arguments_get_the_workspace_entry_points_status():
    """An unsupported dtype is GDN_ERR_UNSUPPORTED from both entry points."""
    lib()
    from gated_deltanet_linear_bwd_gb300 import _abi
    a = _abi.gdn_fwd_args()
    a.q = a.k = a.v = a.g = a.beta = a.o = 4096
    a.B, a.T, a.H, a.K, a.V = 1, 64, 1, 128, 128
    a.dtype = 7
    L = _abi.load()
    rc_static = L.gdn_chunk_fwd_static(ctypes.byref(a), None)
    rc_ws = L.gdn_chunk_fwd(ctypes.byref(a), None, 0, None)
    assert rc_static == rc_ws == _abi.GDN_ERR_UNSUPPORTED
