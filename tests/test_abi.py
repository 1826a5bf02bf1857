"""The C ABI without a GPU: libgdn.so loads, exports every function that
include/gdn.h declares, the ctypes structs match the C layout, and host-side
validation rejects bad arguments before touching a device."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def abi():
    import __graft_entry__
    __graft_entry__.build()
    from gated_deltanet_linear_bwd_gb300 import _abi
    _abi.load()
    return _abi


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_function_is_exported(abi):
    names = declared_functions()
    assert set(names) == set(abi.EXPORTS), names
    lib = abi.load()
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", abi.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}\b", out), n


def test_struct_layout_matches_header(abi):
    probe = r"""
#include <stdio.h>
#include <stddef.h>
#include "gdn.h"
#define F(S, f) printf(#S " " #f " %zu\n", offsetof(S, f));
int main(void) {
  printf("gdn_fwd_args sizeof %zu\n", sizeof(gdn_fwd_args));
  printf("gdn_bwd_args sizeof %zu\n", sizeof(gdn_bwd_args));
  printf("gdn_kernel_stat sizeof %zu\n", sizeof(gdn_kernel_stat));
%s
  return 0;
}
"""
    lines = []
    for cls in (abi.gdn_fwd_args, abi.gdn_bwd_args, abi.gdn_kernel_stat):
        for name, _ in cls._fields_:
            lines.append(f"  F({cls.__name__}, {name})")
    src = probe.replace("%s", "\n".join(lines))
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "probe.c")
        exe = os.path.join(d, "probe")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), c, "-o", exe],
                       check=True)
        got = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    for line in filter(None, got):
        sname, field, val = line.split()
        cls = getattr(abi, sname)
        if field == "sizeof":
            assert ctypes.sizeof(cls) == int(val), sname
        else:
            assert getattr(cls, field).offset == int(val), (sname, field)


def _fwd_args(abi, **kw):
    a = abi.gdn_fwd_args()
    a.q = a.k = a.v = a.g = a.beta = a.o = 4096
    a.B, a.T, a.H, a.K, a.V = 1, 256, 2, 64, 64
    a.dtype = abi.GDN_FP32
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_abi_version_and_workspace_query_need_no_gpu(abi):
    assert abi.gdn_abi_version() == 4
    n_off = abi.gdn_fwd_workspace_size(_fwd_args(abi, cp_mode=abi.GDN_CP_OFF))
    n_cp = abi.gdn_fwd_workspace_size(_fwd_args(abi, cp_mode=abi.GDN_CP_FORCE))
    assert 0 < n_off < n_cp
    b = abi.gdn_bwd_args()
    b.q = b.k = b.v = b.g = b.beta = 4096
    b.B, b.T, b.H, b.K, b.V = 2, 100, 3, 128, 64
    assert abi.gdn_bwd_workspace_size(b) > n_off


@pytest.mark.parametrize("bad, msg", [
    (dict(K=96), "K and V"),
    (dict(V=32), "K and V"),
    (dict(q=None), "required"),
    (dict(B=0), "bad sizes"),
    (dict(dtype=7), "dtype"),
    (dict(cp_mode=9), "cp_mode"),
    (dict(q=4097), "aligned"),
    (dict(cu_seqlens=4096, B=2, N=2), "cu_seqlens"),
])
def test_bad_arguments_are_rejected_on_the_host(abi, bad, msg):
    a = _fwd_args(abi, **bad)
    assert abi.load().gdn_fwd_workspace_size(ctypes.byref(a)) == 0
    assert msg in abi.gdn_last_error()
    rc = abi.load().gdn_chunk_fwd(ctypes.byref(a), ctypes.c_void_p(4096), 1 << 30, None)
    assert rc in (abi.GDN_ERR_INVALID_ARG, abi.GDN_ERR_UNSUPPORTED)
    assert msg in abi.gdn_last_error()


def test_bad_fuse_prep_is_rejected_on_the_host(abi):
    a = _fwd_args(abi, fuse_prep=2)
    rc = abi.load().gdn_chunk_fwd(ctypes.byref(a), ctypes.c_void_p(4096), 1 << 30, None)
    assert rc == abi.GDN_ERR_INVALID_ARG
    assert "fuse_prep" in abi.gdn_last_error()


def test_missing_outputs_are_rejected(abi):
    a = _fwd_args(abi, o=None)
    rc = abi.load().gdn_chunk_fwd(ctypes.byref(a), ctypes.c_void_p(4096), 1 << 30, None)
    assert rc == abi.GDN_ERR_INVALID_ARG
    b = abi.gdn_bwd_args()
    b.B, b.T = 1, 5
    rc = abi.load().gdn_chunk_bwd(ctypes.byref(b), ctypes.c_void_p(4096), 1 << 30, None)
    assert rc == abi.GDN_ERR_INVALID_ARG
    assert "required" in abi.gdn_last_error()


def _step_args(abi, **kw):
    a = abi.gdn_step_args()
    a.q = a.k = a.v = a.g = a.beta = a.state = a.o = 4096
    a.N, a.H, a.K, a.V = 2, 3, 128, 128
    a.dtype = abi.GDN_BF16
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("bad, rc_name, msg", [
    (dict(K=96), "GDN_ERR_UNSUPPORTED", "K = 96"),
    (dict(V=32), "GDN_ERR_UNSUPPORTED", "V = 32"),
    (dict(dtype=5), "GDN_ERR_UNSUPPORTED", "dtype"),
    (dict(state=None), "GDN_ERR_INVALID_ARG", "required"),
    (dict(o=None), "GDN_ERR_INVALID_ARG", "required"),
    (dict(beta=4100), "GDN_ERR_INVALID_ARG", "aligned"),
    (dict(N=-1), "GDN_ERR_INVALID_ARG", ">= 0"),
])
def test_decode_step_rejects_bad_arguments_on_the_host(abi, bad, rc_name, msg):
    rc = abi.load().gdn_recurrent_step(ctypes.byref(_step_args(abi, **bad)), None)
    assert rc == getattr(abi, rc_name)
    assert msg in abi.gdn_last_error()


def test_decode_step_with_no_sequences_is_a_host_side_no_op(abi):
    assert abi.load().gdn_recurrent_step(ctypes.byref(_step_args(abi, N=0)), None) == abi.GDN_OK


def test_saved_context_exists_only_on_the_tensor_core_path(abi):
    bf = _fwd_args(abi, dtype=abi.GDN_BF16, K=128, V=128, T=1000)
    n = abi.gdn_fwd_ctx_size(bf)
    assert n > 0
    # bf16 T, W, u and chunk start states, about 2KV/C + 2(K+V) + 132 bytes per token-head
    per = (2 * 128 * 128 / 64 + 2 * 256 + 132) * 1000 * 2
    assert 0.5 * per < n < 2 * per
    assert abi.gdn_fwd_ctx_size(_fwd_args(abi, dtype=abi.GDN_FP32, K=128, V=128)) == 0
    assert abi.gdn_fwd_ctx_size(_fwd_args(abi, dtype=abi.GDN_BF16, K=64, V=64)) == 0


def test_saved_context_keeps_the_forward_maps_under_forced_sequence_parallelism(abi):
    """Fixed-length batches with sequence parallelism forced also keep the A
    parts of the forward's segment maps (fp32 K x K per segment and head), sized
    for the most segments the forward can choose: 64 per sequence, or the count
    cp_segment_chunks fixes.  The size depends on the arguments only."""
    base = dict(dtype=abi.GDN_BF16, K=128, V=128, B=2, T=8192, H=4)
    off = abi.gdn_fwd_ctx_size(_fwd_args(abi, cp_mode=abi.GDN_CP_OFF, **base))
    auto = abi.gdn_fwd_ctx_size(_fwd_args(abi, cp_mode=abi.GDN_CP_AUTO, **base))
    force = abi.gdn_fwd_ctx_size(_fwd_args(abi, cp_mode=abi.GDN_CP_FORCE, **base))
    fixed = abi.gdn_fwd_ctx_size(_fwd_args(abi, cp_mode=abi.GDN_CP_FORCE, cp_segment_chunks=16,
                                           **base))
    maps = lambda segs: base["B"] * segs * base["H"] * 128 * 128 * 4
    assert off == auto
    assert force - off == maps(64)
    assert fixed - off == maps(8192 // 64 // 16)


def test_tensor_core_path_only_where_its_tma_coordinates_fit(abi):
    """The tensor-core path addresses the per-(chunk, head) state tiles with 32-bit
    TMA row coordinates up to 2 (chunk * H + head) * 128 + 128; a problem whose
    coordinates would not fit takes the CUDA-core path (which keeps no saved
    context), one chunk-head below the limit still takes the tensor cores."""
    limit = (2 ** 31 - 128) // 256          # chunk-heads the coordinates allow
    below = _fwd_args(abi, dtype=abi.GDN_BF16, K=128, V=128, B=1, H=1, T=64 * (limit - 1))
    above = _fwd_args(abi, dtype=abi.GDN_BF16, K=128, V=128, B=1, H=1, T=64 * (limit + 1))
    assert abi.gdn_fwd_ctx_size(below) > 0
    assert abi.gdn_fwd_ctx_size(above) == 0
