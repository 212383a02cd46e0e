"""ctypes loader and signatures of libdiffattn.so (include/diffattn.h)."""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdiffattn.so")

DIFFATTN_OK = 0
DIFFATTN_ERR_INVALID = -1
DIFFATTN_ERR_UNSUPPORTED = -2
DIFFATTN_ERR_CUDA = -3
DIFFATTN_ERR_TIMEOUT = -4

DIFFATTN_BF16 = 0
DIFFATTN_F32 = 1

DIFFATTN_KERNEL_TCGEN05 = 1
DIFFATTN_KERNEL_SIMT = 2

DIFFATTN_NORM_NONE = 0
DIFFATTN_NORM_RMS = 1
DIFFATTN_NORM_GROUP = 2

# Every symbol include/diffattn.h declares.
EXPORTED = (
    "diffattn_lambda",
    "diffattn_lambda_backward",
    "diffattn_fwd",
    "diffattn_fwd_ex",
    "diffattn_fwd_host",
    "diffattn_fwd_train",
    "diffattn_bwd",
    "diffattn_bwd_saved",
    "diffattn_bwd_workspace_bytes",
    "diffattn_decode",
    "diffattn_decode_workspace_bytes",
    "diffattn_decode_noalloc",
    "diffattn_workspace_bytes",
    "diffattn_select_kernel",
    "diffattn_get_device_error",
    "diffattn_selftest_timeout",
    "diffattn_strerror",
    "diffattn_version",
)


class DiffattnDesc(ctypes.Structure):
    """Mirror of diffattn_desc."""
    _fields_ = [
        ("B", ctypes.c_int64), ("H", ctypes.c_int64), ("T", ctypes.c_int64), ("D", ctypes.c_int64),
        ("dtype", ctypes.c_int32), ("kv_group", ctypes.c_int32),
        ("q1_stride", ctypes.c_int64 * 3), ("k1_stride", ctypes.c_int64 * 3),
        ("q2_stride", ctypes.c_int64 * 3), ("k2_stride", ctypes.c_int64 * 3),
        ("v_stride", ctypes.c_int64 * 3), ("o_stride", ctypes.c_int64 * 3),
        ("Dv", ctypes.c_int64),
    ]


class DiffattnKvDesc(ctypes.Structure):
    """Mirror of diffattn_kv_desc."""
    _fields_ = [
        ("B", ctypes.c_int64), ("H", ctypes.c_int64), ("Tq", ctypes.c_int64), ("Tk", ctypes.c_int64),
        ("D", ctypes.c_int64), ("dtype", ctypes.c_int32), ("kv_group", ctypes.c_int32),
        ("q1_stride", ctypes.c_int64 * 3), ("k1_stride", ctypes.c_int64 * 3),
        ("q2_stride", ctypes.c_int64 * 3), ("k2_stride", ctypes.c_int64 * 3),
        ("v_stride", ctypes.c_int64 * 3), ("o_stride", ctypes.c_int64 * 3),
        ("Dv", ctypes.c_int64),
    ]


class DiffattnEpilogue(ctypes.Structure):
    """Mirror of diffattn_epilogue."""
    _fields_ = [
        ("norm", ctypes.c_int32), ("eps", ctypes.c_float), ("weight", ctypes.c_void_p),
        ("bias", ctypes.c_void_p), ("out_scale", ctypes.c_float), ("reserved", ctypes.c_int32),
    ]


class DiffattnError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.diffattn_lambda.argtypes = [vp, vp, vp, vp, i64, ctypes.c_double, vp, vp]
    lib.diffattn_lambda.restype = ctypes.c_int
    lib.diffattn_lambda_backward.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, vp, vp, vp]
    lib.diffattn_lambda_backward.restype = ctypes.c_int
    lib.diffattn_fwd.argtypes = [ctypes.POINTER(DiffattnDesc), vp, vp, vp, vp, vp, ctypes.c_float,
                                 vp, ctypes.c_int, vp, vp, ctypes.c_size_t, vp]
    lib.diffattn_fwd_ex.argtypes = [ctypes.POINTER(DiffattnDesc), vp, vp, vp, vp, vp, ctypes.c_float,
                                    vp, ctypes.c_int, ctypes.POINTER(DiffattnEpilogue), vp, vp,
                                    ctypes.c_size_t, vp]
    lib.diffattn_fwd_ex.restype = ctypes.c_int
    lib.diffattn_decode.argtypes = [ctypes.POINTER(DiffattnKvDesc), vp, vp, vp, vp, vp, ctypes.c_float,
                                    vp, ctypes.c_int, ctypes.POINTER(DiffattnEpilogue), vp, vp,
                                    ctypes.c_size_t, vp]
    lib.diffattn_decode.restype = ctypes.c_int
    lib.diffattn_decode_noalloc.argtypes = [ctypes.POINTER(DiffattnKvDesc), vp, vp, vp, vp, vp,
                                            ctypes.c_float, vp, ctypes.c_int,
                                            ctypes.POINTER(DiffattnEpilogue), vp, vp]
    lib.diffattn_decode_noalloc.restype = ctypes.c_int
    lib.diffattn_bwd.argtypes = [ctypes.POINTER(DiffattnDesc), vp, vp, vp, vp, vp, ctypes.c_float,
                                 vp, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.diffattn_bwd.restype = ctypes.c_int
    lib.diffattn_fwd_host.argtypes = [ctypes.POINTER(DiffattnDesc), vp, vp, vp, vp, vp,
                                      ctypes.c_float, vp, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp,
                                      vp, ctypes.c_size_t, vp]
    lib.diffattn_fwd_host.restype = ctypes.c_int
    lib.diffattn_fwd_train.argtypes = [ctypes.POINTER(DiffattnDesc), vp, vp, vp, vp, vp,
                                       ctypes.c_float, vp, ctypes.c_int, vp, vp, vp, vp,
                                       ctypes.c_size_t, vp]
    lib.diffattn_fwd_train.restype = ctypes.c_int
    lib.diffattn_bwd_saved.argtypes = [ctypes.POINTER(DiffattnDesc), vp, vp, vp, vp, vp,
                                       ctypes.c_float, vp, ctypes.c_int, vp, vp, vp, vp, vp, vp,
                                       vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.diffattn_bwd_saved.restype = ctypes.c_int
    lib.diffattn_bwd_workspace_bytes.argtypes = [ctypes.POINTER(DiffattnDesc)]
    lib.diffattn_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.diffattn_decode_workspace_bytes.argtypes = [ctypes.POINTER(DiffattnKvDesc)]
    lib.diffattn_decode_workspace_bytes.restype = ctypes.c_size_t
    lib.diffattn_workspace_bytes.argtypes = []
    lib.diffattn_workspace_bytes.restype = ctypes.c_size_t
    lib.diffattn_fwd.restype = ctypes.c_int
    lib.diffattn_select_kernel.argtypes = [ctypes.POINTER(DiffattnDesc), vp, vp, vp, vp, vp, vp]
    lib.diffattn_select_kernel.restype = ctypes.c_int
    lib.diffattn_get_device_error.argtypes = [vp]
    lib.diffattn_get_device_error.restype = ctypes.c_int
    lib.diffattn_selftest_timeout.argtypes = [vp]
    lib.diffattn_selftest_timeout.restype = ctypes.c_int
    lib.diffattn_strerror.argtypes = [ctypes.c_int]
    lib.diffattn_strerror.restype = ctypes.c_char_p
    lib.diffattn_version.argtypes = []
    lib.diffattn_version.restype = ctypes.c_int
    _lib = lib
    return lib


def strerror(code: int) -> str:
    try:
        return load().diffattn_strerror(code).decode()
    except RuntimeError:
        return f"error {code}"


def check(code: int, what: str) -> None:
    if code != DIFFATTN_OK:
        raise DiffattnError(code, what)
