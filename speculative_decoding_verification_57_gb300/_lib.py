"""ctypes declarations of the C ABI in include/specv.h (argument marshalling
only; every step of the verify path runs in the library's CUDA kernels)."""
import ctypes
import os

from . import build as _build

SPECV_OK = 0
SPECV_ERR_INVALID_ARGUMENT = 1
SPECV_ERR_UNSUPPORTED = 2
SPECV_ERR_CUDA = 3
SPECV_ERR_TIMEOUT = 4
SPECV_F32 = 0
SPECV_BF16 = 1

# row_status bits
ST_NONFINITE = 1
ST_TOKEN_RANGE = 2
ST_UNIFORM_RANGE = 4
ST_TEMPERATURE = 8
ST_ZERO_RESIDUAL = 16
ST_Q_INVALID = 32
ST_TIMEOUT = 64
ST_PARENT = 512
ST_FILTER = 1024
ST_ERROR_MASK = (ST_NONFINITE | ST_TOKEN_RANGE | ST_UNIFORM_RANGE | ST_TEMPERATURE | ST_Q_INVALID | ST_TIMEOUT
                 | ST_PARENT | ST_FILTER)


class SpecvDebug(ctypes.Structure):
    _fields_ = [
        ("p_at_draft", ctypes.c_void_p),
        ("q_at_draft", ctypes.c_void_p),
        ("row_max", ctypes.c_void_p),
        ("row_sumexp", ctypes.c_void_p),
        ("residual_mass", ctypes.c_void_p),
    ]


_lib = None


def load(build_if_missing=True):
    """Load libspecv.so (building it in-tree first when it is missing and
    nvcc is available).  Raises if the library cannot be had: there is no
    fallback implementation."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing and (not os.path.exists(path)):
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run __graft_entry__.build() to compile the CUDA library")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.specv_create.restype = i32
    lib.specv_create.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i64]
    lib.specv_verify_sample.restype = i32
    lib.specv_verify_sample.argtypes = [vp, i32, vp, vp, vp, vp, vp, i32, i32, i64, vp, vp, vp,
                                        ctypes.POINTER(SpecvDebug), vp]
    lib.specv_verify_greedy.restype = i32
    lib.specv_verify_greedy.argtypes = [vp, i32, vp, vp, i32, i32, i64, vp, vp, vp, vp]
    lib.specv_verify_sample_host.restype = i32
    lib.specv_verify_sample_host.argtypes = [vp, i32, vp, vp, vp, vp, vp, i32, i32, i64, vp, vp, vp, vp]
    lib.specv_verify_sample_filtered.restype = i32
    lib.specv_verify_sample_filtered.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp, i32, i32, i64, vp, vp, vp, vp]
    lib.specv_verify_tree_greedy.restype = i32
    lib.specv_verify_tree_greedy.argtypes = [vp, i32, vp, vp, vp, i32, i32, i64, vp, vp, vp, vp, vp]
    lib.specv_rollback.restype = i32
    lib.specv_rollback.argtypes = [vp, vp, i32, i32, vp, vp, i32, vp, i32, vp, i64, vp, vp, vp]
    lib.specv_plan_cluster.restype = i32
    lib.specv_plan_cluster.argtypes = [vp, i32, i32, i32, i64]
    lib.specv_test_withhold_stage.restype = i32
    lib.specv_test_withhold_stage.argtypes = [vp, i32, i32]
    lib.specv_launch_count.restype = i64
    lib.specv_launch_count.argtypes = [vp]
    lib.specv_destroy.restype = None
    lib.specv_destroy.argtypes = [vp]
    lib.specv_status_string.restype = ctypes.c_char_p
    lib.specv_status_string.argtypes = [i32]
    lib.specv_last_cuda_error.restype = ctypes.c_char_p
    lib.specv_last_cuda_error.argtypes = []
    _lib = lib
    return lib
