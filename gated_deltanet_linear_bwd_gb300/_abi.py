"""ctypes binding of libgdn.so (include/gdn.h).  Argument marshalling only.

The names mirror the C entry points.  The library must have been built
(gated_deltanet_linear_bwd_gb300/build.py, or __graft_entry__.build()); there
is no fallback of any kind when it is missing.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgdn.so")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_WORKSPACE, GDN_ERR_CUDA, \
    GDN_ERR_TIMEOUT, GDN_ERR_BAD_SEQLENS = range(7)
GDN_FP32, GDN_BF16 = 0, 1
GDN_CP_AUTO, GDN_CP_OFF, GDN_CP_FORCE = 0, 1, 2

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_f32 = ctypes.c_float


class gdn_fwd_args(ctypes.Structure):
    _fields_ = [("q", _vp), ("k", _vp), ("v", _vp), ("g", _vp), ("beta", _vp),
                ("initial_state", _vp), ("cu_seqlens", _vp),
                ("B", _i32), ("T", _i32), ("H", _i32), ("K", _i32), ("V", _i32), ("N", _i32),
                ("dtype", _i32), ("scale", _f32), ("use_qk_l2norm", _i32), ("cp_mode", _i32),
                ("cp_segment_chunks", _i32), ("cp_warmup_chunks", _i32), ("cp_warmup_tau", _f32),
                ("o", _vp), ("final_state", _vp), ("cp_stats", _vp), ("ctx", _vp),
                ("gate_scale", _vp), ("fuse_prep", _i32)]


class gdn_bwd_args(ctypes.Structure):
    _fields_ = [("q", _vp), ("k", _vp), ("v", _vp), ("g", _vp), ("beta", _vp),
                ("initial_state", _vp), ("cu_seqlens", _vp),
                ("B", _i32), ("T", _i32), ("H", _i32), ("K", _i32), ("V", _i32), ("N", _i32),
                ("dtype", _i32), ("scale", _f32), ("use_qk_l2norm", _i32), ("cp_mode", _i32),
                ("cp_segment_chunks", _i32),
                ("d_o", _vp), ("d_final_state", _vp),
                ("grad_dtype", _i32), ("dq", _vp), ("dk", _vp), ("dv", _vp), ("dg", _vp),
                ("dbeta", _vp), ("d_initial_state", _vp), ("ctx", _vp),
                ("gate_scale", _vp), ("d_gate_scale", _vp)]


class gdn_step_args(ctypes.Structure):
    _fields_ = [("q", _vp), ("k", _vp), ("v", _vp), ("g", _vp), ("beta", _vp),
                ("gate_scale", _vp), ("state", _vp),
                ("N", _i32), ("H", _i32), ("K", _i32), ("V", _i32), ("dtype", _i32),
                ("scale", _f32), ("use_qk_l2norm", _i32), ("o", _vp)]


class gdn_kernel_stat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 64), ("launches", _i32), ("total_ms", ctypes.c_double)]


EXPORTS = ("gdn_abi_version", "gdn_fwd_workspace_size", "gdn_chunk_fwd", "gdn_bwd_workspace_size",
           "gdn_chunk_bwd", "gdn_sync_status", "gdn_last_error", "gdn_set_spin_limit",
           "gdn_profile_begin", "gdn_profile_end", "gdn_chunk_fwd_static", "gdn_fwd_ctx_size",
           "gdn_recurrent_step")
GDN_STATIC_SCRATCH_BYTES = 64 << 20

_lib = None


def load(path: str = LIB_PATH):
    """Opens libgdn.so and declares every exported signature."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libgdn.so is not built ({path}); run "
                          "`python gated_deltanet_linear_bwd_gb300/build.py`")
    lib = ctypes.CDLL(path)
    lib.gdn_abi_version.restype = _i32
    lib.gdn_abi_version.argtypes = []
    lib.gdn_fwd_workspace_size.restype = ctypes.c_size_t
    lib.gdn_fwd_workspace_size.argtypes = [ctypes.POINTER(gdn_fwd_args)]
    lib.gdn_chunk_fwd.restype = _i32
    lib.gdn_chunk_fwd.argtypes = [ctypes.POINTER(gdn_fwd_args), _vp, ctypes.c_size_t, _vp]
    lib.gdn_bwd_workspace_size.restype = ctypes.c_size_t
    lib.gdn_bwd_workspace_size.argtypes = [ctypes.POINTER(gdn_bwd_args)]
    lib.gdn_chunk_bwd.restype = _i32
    lib.gdn_chunk_bwd.argtypes = [ctypes.POINTER(gdn_bwd_args), _vp, ctypes.c_size_t, _vp]
    lib.gdn_sync_status.restype = _i32
    lib.gdn_sync_status.argtypes = [_vp]
    lib.gdn_last_error.restype = ctypes.c_char_p
    lib.gdn_last_error.argtypes = []
    lib.gdn_set_spin_limit.restype = None
    lib.gdn_set_spin_limit.argtypes = [ctypes.c_int64]
    lib.gdn_fwd_ctx_size.restype = ctypes.c_size_t
    lib.gdn_fwd_ctx_size.argtypes = [ctypes.POINTER(gdn_fwd_args)]
    lib.gdn_chunk_fwd_static.restype = _i32
    lib.gdn_chunk_fwd_static.argtypes = [ctypes.POINTER(gdn_fwd_args), _vp]
    lib.gdn_recurrent_step.restype = _i32
    lib.gdn_recurrent_step.argtypes = [ctypes.POINTER(gdn_step_args), _vp]
    lib.gdn_profile_begin.restype = _i32
    lib.gdn_profile_begin.argtypes = []
    lib.gdn_profile_end.restype = _i32
    lib.gdn_profile_end.argtypes = [ctypes.POINTER(gdn_kernel_stat), _i32]
    _lib = lib
    return lib


class GdnError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn} returned {code}: {gdn_last_error()}")


def gdn_abi_version() -> int:
    return int(load().gdn_abi_version())


def gdn_last_error() -> str:
    return load().gdn_last_error().decode()


def gdn_set_spin_limit(polls: int) -> None:
    load().gdn_set_spin_limit(int(polls))


def gdn_fwd_workspace_size(args: gdn_fwd_args) -> int:
    n = int(load().gdn_fwd_workspace_size(ctypes.byref(args)))
    if n == 0:
        raise GdnError("gdn_fwd_workspace_size", GDN_ERR_INVALID_ARG)
    return n


def gdn_fwd_ctx_size(args: gdn_fwd_args) -> int:
    """Bytes of the saved forward context (0: this path keeps none)."""
    return int(load().gdn_fwd_ctx_size(ctypes.byref(args)))


def gdn_bwd_workspace_size(args: gdn_bwd_args) -> int:
    n = int(load().gdn_bwd_workspace_size(ctypes.byref(args)))
    if n == 0:
        raise GdnError("gdn_bwd_workspace_size", GDN_ERR_INVALID_ARG)
    return n


def gdn_chunk_fwd(args: gdn_fwd_args, workspace: int, ws_bytes: int, stream: int) -> None:
    rc = load().gdn_chunk_fwd(ctypes.byref(args), _vp(workspace), ws_bytes, _vp(stream))
    if rc != GDN_OK:
        raise GdnError("gdn_chunk_fwd", rc)


def gdn_chunk_bwd(args: gdn_bwd_args, workspace: int, ws_bytes: int, stream: int) -> None:
    rc = load().gdn_chunk_bwd(ctypes.byref(args), _vp(workspace), ws_bytes, _vp(stream))
    if rc != GDN_OK:
        raise GdnError("gdn_chunk_bwd", rc)


def gdn_sync_status(stream: int) -> int:
    """Returns the device status code (GDN_OK, GDN_ERR_BAD_SEQLENS, GDN_ERR_TIMEOUT, ...)."""
    return int(load().gdn_sync_status(_vp(stream)))


def gdn_profile_begin() -> None:
    load().gdn_profile_begin()


def gdn_profile_end(max_kernels: int = 64):
    """Returns [(kernel name, launches, total ms)] for launches since gdn_profile_begin."""
    buf = (gdn_kernel_stat * max_kernels)()
    n = int(load().gdn_profile_end(buf, max_kernels))
    return [(buf[i].name.decode(), int(buf[i].launches), float(buf[i].total_ms))
            for i in range(min(n, max_kernels))]


def gdn_chunk_fwd_static(args: gdn_fwd_args, stream: int) -> None:
    """Forward without a workspace: scratch comes from the library's fixed
    GDN_STATIC_SCRATCH_BYTES device area (see include/gdn.h)."""
    rc = load().gdn_chunk_fwd_static(ctypes.byref(args), _vp(stream))
    if rc != GDN_OK:
        raise GdnError("gdn_chunk_fwd_static", rc)


def gdn_recurrent_step(args: gdn_step_args, stream: int) -> None:
    rc = load().gdn_recurrent_step(ctypes.byref(args), _vp(stream))
    if rc != GDN_OK:
        raise GdnError("gdn_recurrent_step", rc)
