"""ctypes binding of the C ABI in include/la.h (liblagb300.so, built in-tree).

Loading fails loudly: there is no fallback implementation anywhere in this
package.  Build the library with `python linear_attention_head_gb300/build.py`
or `__graft_entry__.build()`.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# LA_LIBRARY in the environment names another build of the same library (the
# bounds-checking one, liblagb300_checked.so) to load instead
LIB_PATH = os.environ.get("LA_LIBRARY") or os.path.join(HERE, "liblagb300.so")

LA_OK = 0
LA_ERR_INVALID_ARG = 1
LA_ERR_UNSUPPORTED = 2
LA_ERR_CUDA = 3
LA_ERR_TIMEOUT = 4
LA_ERR_BOUNDS = 5

LA_DTYPE_BF16 = 0
LA_DTYPE_F32 = 1

LA_FWD_NOALLOC_MAX_SEQS = 16384   # include/la.h
LA_BUILD_BOUNDS_CHECKED = 1       # include/la.h


class LaDims(ctypes.Structure):
    """Mirror of `la_dims` (include/la.h)."""
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("seq_len", ctypes.c_int32),
        ("heads", ctypes.c_int32),
        ("dim_qk", ctypes.c_int32),
        ("dim_v", ctypes.c_int32),
        ("num_seqs", ctypes.c_int32),
        ("qk_strides", ctypes.c_int64 * 3),
        ("v_strides", ctypes.c_int64 * 3),
        ("kv_heads", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("k_strides", ctypes.c_int64 * 3),
        ("kv_v_strides", ctypes.c_int64 * 3),
    ]


class LaError(RuntimeError):
    def __init__(self, status, detail):
        self.status = status
        super().__init__("%s (status %d): %s" % (strerror(status), status, detail))


class LaInvalidArgument(LaError, ValueError):
    pass


class LaUnsupported(LaError, NotImplementedError):
    pass


_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_f32 = ctypes.c_float
_sz = ctypes.c_size_t
_dims_p = ctypes.POINTER(LaDims)

# name -> (restype, argtypes); mirrors include/la.h exactly (float* are passed
# as void* addresses).
PROTOTYPES = {
    "la_fwd": (_i32, [_dims_p, _i32, _vp, _vp, _vp, _vp, _f32, _vp, _i32, _vp, _vp,
                      _vp, _vp, _vp, _sz, _vp]),
    "la_bwd": (_i32, [_dims_p, _i32, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _vp, _i32,
                      _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "la_bwd_dq": (_i32, [_dims_p, _i32, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _i32,
                         _vp, _vp, _vp, _vp, _sz, _vp]),
    "la_bwd_dkdv": (_i32, [_dims_p, _i32, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _i32,
                           _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "la_workspace_size": (_sz, [_i32]),
    "la_workspace_size_for": (_sz, [_dims_p, _i32, _vp]),
    "la_set_sequence_split": (_i32, [_i32, _i32]),
    "la_gla_fwd": (_i32, [_dims_p, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _i32, _vp,
                          _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "la_gla_fwd_workspace_size": (_sz, [_dims_p, _i32, _vp]),
    "la_gla_bwd": (_i32, [_dims_p, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _vp,
                          _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _sz, _vp]),
    "la_gla_workspace_size": (_sz, [_dims_p, _i32, _vp, _i32]),
    "la_debug_withhold_next_handoff": (_i32, [_i32]),
    "la_debug_split_segments": (_i32, [_dims_p, _i32, _vp, _i32]),
    "la_fwd_noalloc": (_i32, [_dims_p, _i32, _vp, _vp, _vp, _vp, _f32, _vp, _i32, _vp, _vp,
                              _vp, _vp, _vp]),
    "la_get_device_error": (_i32, [_vp]),
    "la_strerror": (ctypes.c_char_p, [_i32]),
    "la_last_error": (ctypes.c_char_p, []),
    "la_kernel_family": (_i32, [_dims_p, _i32]),
    "la_launch_count": (ctypes.c_uint64, []),
    "la_version": (_i32, []),
    "la_build_flags": (_i32, []),
}

_lib = None


def lib():
    """The loaded library (raises ImportError when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("%s is not built (run linear_attention_head_gb300/build.py); "
                              "this package has no fallback path" % os.path.basename(LIB_PATH))
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in PROTOTYPES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def strerror(status):
    return lib().la_strerror(int(status)).decode()


def last_error():
    return lib().la_last_error().decode()


def check(status):
    if status == LA_OK:
        return
    detail = last_error()
    if status == LA_ERR_INVALID_ARG:
        raise LaInvalidArgument(status, detail)
    if status == LA_ERR_UNSUPPORTED:
        raise LaUnsupported(status, detail)
    raise LaError(status, detail)
