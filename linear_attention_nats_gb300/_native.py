"""ctypes view of libnats.so (the C ABI declared in include/nats.h).

Argument marshalling only: every step of the layer runs in the CUDA kernels
behind this library.  There is no fallback: if the library is missing the
import fails.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnats.so")

NATS_BF16 = 0
NATS_F32 = 1

STATUS = {
    0: "NATS_OK", 1: "NATS_ERR_NULL", 2: "NATS_ERR_SHAPE", 3: "NATS_ERR_DTYPE",
    4: "NATS_ERR_ALIGN", 5: "NATS_ERR_WORKSPACE", 6: "NATS_ERR_UNSUPPORTED", 7: "NATS_ERR_CUDA",
    8: "NATS_ERR_INTERNAL", 9: "NATS_ERR_VALUE",
}

# Every symbol include/nats.h declares.
EXPORTS = ("nats_status_string", "nats_last_cuda_error", "nats_workspace_size", "nats_workspace_check", "nats_select",
           "nats_hybrid_fwd", "nats_hybrid_fwd_profiled", "nats_hybrid_fwd_streams", "nats_hybrid_fwd_noalloc",
           "nats_noalloc_check",
           "nats_x_workspace_size", "nats_x_workspace_check",
           "nats_hybrid_fwd_x_profiled",
           "nats_hybrid_fwd_x", "nats_debug_fail_stage", "nats_debug_bounded_wait", "nats_decode_step",
           "nats_bwd_workspace_size", "nats_hybrid_bwd", "nats_hybrid_bwd_profiled", "nats_hybrid_bwd_streams",
           "nats_score_bwd",
           "nats_nha_workspace_size", "nats_nha_fwd",
           "nats_nha_workspace_check", "nats_nha_fwd_profiled")

NOALLOC_SCRATCH_BYTES = 64 << 20

NUM_STAGES = 8
STAGES = ("score", "compact", "softmax", "gdn_prep", "gdn_scan", "merge", "proj_in", "proj_out")
BWD_STAGES = ("merge_bwd", "softmax_bwd", "gdn_bwd", "gdn_products")


class Profile(ctypes.Structure):
    _fields_ = [("start", ctypes.c_void_p * NUM_STAGES), ("stop", ctypes.c_void_p * NUM_STAGES),
                ("launches", ctypes.c_int32), ("stage_launches", ctypes.c_int32 * NUM_STAGES)]


class Streams(ctypes.Structure):
    """nats_streams: the caller's second stream and fork / join events."""
    _fields_ = [("side", ctypes.c_void_p), ("fork", ctypes.c_void_p), ("join", ctypes.c_void_p)]


class DecodeState(ctypes.Structure):
    _fields_ = [("S", ctypes.c_void_p), ("S0", ctypes.c_void_p), ("ck", ctypes.c_void_p), ("cv", ctypes.c_void_p),
                ("psum", ctypes.c_void_p), ("kv_k", ctypes.c_void_p), ("kv_v", ctypes.c_void_p),
                ("n_kv", ctypes.c_void_p), ("cap", ctypes.c_int64),
                ("err", ctypes.c_void_p)]


class Dims(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("L", ctypes.c_int32),
        ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("chunk", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("scale", ctypes.c_float), ("eps", ctypes.c_float),
    ]


class NhaDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("L", ctypes.c_int32), ("d", ctypes.c_int32),
                ("slots", ctypes.c_int32), ("window", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("scale", ctypes.c_float)]


def nha_dims(B, H, L, d=128, slots=64, window=512, dtype=NATS_BF16, scale=0.0) -> NhaDims:
    return NhaDims(int(B), int(H), int(L), int(d), int(slots), int(window), int(dtype), float(scale))


class NatsError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {STATUS.get(code, code)}"
        if code == 7 and _lib is not None:  # NATS_ERR_CUDA: add the CUDA runtime's reason
            msg += f" ({_lib.nats_last_cuda_error().decode()})"
        super().__init__(msg)


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libnats.so is not built ({LIB_PATH}); run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    lib.nats_last_cuda_error.argtypes = []
    lib.nats_last_cuda_error.restype = ctypes.c_char_p
    lib.nats_status_string.argtypes = [ctypes.c_int]
    lib.nats_status_string.restype = ctypes.c_char_p
    lib.nats_workspace_size.argtypes = [ctypes.POINTER(Dims)]
    lib.nats_workspace_size.restype = ctypes.c_size_t
    lib.nats_workspace_check.argtypes = [ctypes.POINTER(Dims), P, P]
    lib.nats_workspace_check.restype = ctypes.c_int
    lib.nats_select.argtypes = [ctypes.POINTER(Dims), P, P, P, P, P, P, P]
    lib.nats_select.restype = ctypes.c_int
    lib.nats_hybrid_fwd.argtypes = [ctypes.POINTER(Dims)] + [P] * 18 + [ctypes.c_size_t, P]
    lib.nats_hybrid_fwd.restype = ctypes.c_int
    lib.nats_hybrid_fwd_profiled.argtypes = [ctypes.POINTER(Dims)] + [P] * 18 + [
        ctypes.c_size_t, P, ctypes.POINTER(Profile)]
    lib.nats_hybrid_fwd_profiled.restype = ctypes.c_int
    lib.nats_hybrid_fwd_streams.argtypes = [ctypes.POINTER(Dims)] + [P] * 19 + [
        ctypes.c_size_t, P, ctypes.POINTER(Streams), ctypes.POINTER(Profile)]
    lib.nats_hybrid_fwd_streams.restype = ctypes.c_int
    lib.nats_hybrid_fwd_noalloc.argtypes = [ctypes.POINTER(Dims)] + [P] * 17 + [P]
    lib.nats_hybrid_fwd_noalloc.restype = ctypes.c_int
    lib.nats_noalloc_check.argtypes = [ctypes.POINTER(Dims), P]
    lib.nats_noalloc_check.restype = ctypes.c_int
    lib.nats_x_workspace_size.argtypes = [ctypes.POINTER(Dims), ctypes.c_int32]
    lib.nats_x_workspace_size.restype = ctypes.c_size_t
    lib.nats_hybrid_fwd_x.argtypes = [ctypes.POINTER(Dims), ctypes.c_int32] + [P] * 14 + [ctypes.c_size_t, P]
    lib.nats_hybrid_fwd_x.restype = ctypes.c_int
    lib.nats_hybrid_fwd_x_profiled.argtypes = [ctypes.POINTER(Dims), ctypes.c_int32] + [P] * 14 + [
        ctypes.c_size_t, P, ctypes.POINTER(Profile)]
    lib.nats_hybrid_fwd_x_profiled.restype = ctypes.c_int
    lib.nats_x_workspace_check.argtypes = [ctypes.POINTER(Dims), ctypes.c_int32, P, P]
    lib.nats_x_workspace_check.restype = ctypes.c_int
    lib.nats_debug_fail_stage.argtypes = [ctypes.c_int32]
    lib.nats_debug_fail_stage.restype = None
    lib.nats_debug_bounded_wait.argtypes = [P, ctypes.c_int64, P]
    lib.nats_debug_bounded_wait.restype = ctypes.c_int
    lib.nats_decode_step.argtypes = [ctypes.POINTER(Dims), ctypes.c_int64] + [P] * 11 + [
        ctypes.POINTER(DecodeState)] + [P] * 4 + [P]
    lib.nats_decode_step.restype = ctypes.c_int
    lib.nats_bwd_workspace_size.argtypes = [ctypes.POINTER(Dims)]
    lib.nats_bwd_workspace_size.restype = ctypes.c_size_t
    lib.nats_hybrid_bwd.argtypes = [ctypes.POINTER(Dims)] + [P] * 23 + [ctypes.c_size_t, P]
    lib.nats_hybrid_bwd.restype = ctypes.c_int
    lib.nats_hybrid_bwd_profiled.argtypes = [ctypes.POINTER(Dims)] + [P] * 23 + [ctypes.c_size_t, P,
                                                                               ctypes.POINTER(Profile)]
    lib.nats_hybrid_bwd_profiled.restype = ctypes.c_int
    lib.nats_hybrid_bwd_streams.argtypes = [ctypes.POINTER(Dims)] + [P] * 24 + [
        ctypes.c_size_t, P, ctypes.POINTER(Streams), ctypes.POINTER(Profile)]
    lib.nats_hybrid_bwd_streams.restype = ctypes.c_int
    lib.nats_score_bwd.argtypes = [ctypes.POINTER(Dims)] + [P] * 11 + [P]
    lib.nats_score_bwd.restype = ctypes.c_int
    lib.nats_nha_workspace_size.argtypes = [ctypes.POINTER(NhaDims)]
    lib.nats_nha_workspace_size.restype = ctypes.c_size_t
    lib.nats_nha_fwd.argtypes = [ctypes.POINTER(NhaDims)] + [P] * 6 + [ctypes.c_size_t, P]
    lib.nats_nha_fwd.restype = ctypes.c_int
    lib.nats_nha_workspace_check.argtypes = [ctypes.POINTER(NhaDims), P, P]
    lib.nats_nha_workspace_check.restype = ctypes.c_int
    lib.nats_nha_fwd_profiled.argtypes = [ctypes.POINTER(NhaDims)] + [P] * 6 + [ctypes.c_size_t, P,
                                                                                ctypes.POINTER(Profile)]
    lib.nats_nha_fwd_profiled.restype = ctypes.c_int
    return lib


_lib = None


def __getattr__(name):
    # `lib` loads on first use, so that the build helper in this package can
    # be imported before the library exists.
    global _lib
    if name == "lib":
        if _lib is None:
            _lib = _load()
        return _lib
    raise AttributeError(name)


def dims(B, H, L, d, dtype=NATS_BF16, scale=0.0, eps=1e-6, chunk=64) -> Dims:
    return Dims(int(B), int(H), int(L), int(d), int(d), int(chunk), int(dtype), float(scale), float(eps))


def check(code: int, where: str) -> None:
    if code != 0:
        raise NatsError(code, where)
