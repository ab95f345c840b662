"""ctypes view of libmoe.so (the C ABI in include/moe.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation of any stage.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")
CHECK_LIB_PATH = os.path.join(_HERE, "libmoe_check.so")   # bounds-checked build

MOE_OK = 0
MOE_ERR_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE = 6
MOE_ERR_BOUNDS = 7

MOE_F32, MOE_BF16 = 0, 1
MOE_ACT_GELU, MOE_ACT_RELU, MOE_ACT_SWIGLU = 0, 1, 2
MOE_GATE_SOFTMAX_TOPK, MOE_GATE_SIGMOID_RENORM, MOE_GATE_SOFTMAX_FULL = 0, 1, 2
MOE_NUM_STAGES = 6
MOE_TUNE_ROUTER, MOE_TUNE_GATHER, MOE_TUNE_TILE_N_UP, MOE_TUNE_TILE_N_DOWN = 0, 1, 2, 3
MOE_TUNE_PARTIAL_A_ROWS, MOE_TUNE_MMA_M64, MOE_TUNE_FUSED_COMBINE = 4, 5, 6
MOE_TUNE_CLUSTER, MOE_TUNE_FUSED_PROJ, MOE_TUNE_F8_DOWN_FORM = 7, 8, 9
MOE_PLAN_ROUTE_ONE_LAUNCH, MOE_PLAN_ROUTE_CLUSTER, MOE_PLAN_ROUTE_DECODE = 1, 2, 4
MOE_PLAN_GATHER_ROWS, MOE_PLAN_COMBINE_IN_DOWN, MOE_PLAN_FUSED_PROJECTIONS = 8, 16, 32
MOE_ROUTER_SIMT, MOE_ROUTER_FUSED, MOE_ROUTER_TC = 1, 2, 3
STAGE_NAMES = ("router", "topk", "permute", "up", "down", "combine")

EXPORTS = (
    "moe_workspace_size", "moe_forward", "moe_route_workspace_size", "moe_route",
    "moe_host_io_workspace_size", "moe_forward_host_io", "moe_check_status",
    "moe_error_string", "moe_forward_timed", "moe_launch_count", "moe_selftest_wait_timeout",
    "moe_router_scores", "moe_router_scores_noalloc", "moe_router_z_loss", "moe_bias_update",
    "moe_workspace_size_fp8", "moe_forward_fp8", "moe_forward_fp8_timed", "moe_launch_count_fp8",
    "moe_set_tuning", "moe_host_io_workspace_size_fp8", "moe_forward_fp8_host_io",
    "moe_forward_host_io_batches", "moe_forward_fp8_host_io_batches", "moe_plan_flags",
    "moe_forward_fp8_all", "moe_forward_fp8_all_timed", "moe_forward_fp8_all_host_io_batches",
    "moe_plan_flags_fp8",
)


class MoeConfig(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
        ("k", ctypes.c_int32), ("f", ctypes.c_int32), ("n_shared", ctypes.c_int32),
        ("f_shared", ctypes.c_int32), ("dtype", ctypes.c_int32), ("act", ctypes.c_int32),
        ("gate", ctypes.c_int32), ("capacity_factor", ctypes.c_double),
        ("alpha", ctypes.c_float), ("reserved", ctypes.c_int32),
    ]


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {error_string(code)} (code {code})")


_lib = None
_libs = {}
P = ctypes.c_void_p
SZ = ctypes.c_size_t
I32P = ctypes.POINTER(ctypes.c_int32)


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _load(LIB_PATH)
    return _lib


def use_library(variant: str) -> None:
    """Routes every later call to `variant`: "default" (libmoe.so) or "check"
    (libmoe_check.so, the bounds-checked build; tests only)."""
    global _lib
    _lib = _load(CHECK_LIB_PATH if variant == "check" else LIB_PATH)


def _load(path: str) -> ctypes.CDLL:
    if path in _libs:
        return _libs[path]
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m sparse_mixture_experts_65_b300.build`"
            " (or __graft_entry__.build()); this package has no non-CUDA fallback")
    L = ctypes.CDLL(path)
    cfgp = ctypes.POINTER(MoeConfig)
    for name in ("moe_workspace_size", "moe_route_workspace_size", "moe_host_io_workspace_size",
                 "moe_workspace_size_fp8", "moe_host_io_workspace_size_fp8"):
        f = getattr(L, name)
        f.argtypes = [cfgp, ctypes.POINTER(SZ)]
        f.restype = ctypes.c_int
    fwd_args = [cfgp, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]
    L.moe_forward.argtypes = fwd_args
    L.moe_forward.restype = ctypes.c_int
    L.moe_forward_timed.argtypes = fwd_args + [ctypes.POINTER(P)]
    L.moe_forward_timed.restype = ctypes.c_int
    L.moe_route.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]
    L.moe_route.restype = ctypes.c_int
    L.moe_forward_host_io.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]
    L.moe_forward_host_io.restype = ctypes.c_int
    L.moe_forward_fp8_host_io.argtypes = [cfgp] + [P] * 12 + [SZ, P]
    L.moe_forward_fp8_host_io.restype = ctypes.c_int
    L.moe_forward_host_io_batches.argtypes = [cfgp, ctypes.c_int32] + [P] * 13 + [SZ, P, P, P]
    L.moe_forward_host_io_batches.restype = ctypes.c_int
    L.moe_forward_fp8_host_io_batches.argtypes = [cfgp, ctypes.c_int32] + [P] * 12 + [SZ, P, P, P]
    L.moe_forward_fp8_host_io_batches.restype = ctypes.c_int
    L.moe_router_scores.argtypes = [cfgp, P, P, P, P, P, SZ, P]
    L.moe_router_scores.restype = ctypes.c_int
    fp8_args = [cfgp] + [P] * 20 + [SZ, P]
    L.moe_forward_fp8.argtypes = fp8_args
    L.moe_forward_fp8.restype = ctypes.c_int
    L.moe_forward_fp8_timed.argtypes = fp8_args + [ctypes.POINTER(P)]
    L.moe_forward_fp8_timed.restype = ctypes.c_int
    fp8_all_args = [cfgp] + [P] * 21 + [SZ, P]
    L.moe_forward_fp8_all.argtypes = fp8_all_args
    L.moe_forward_fp8_all.restype = ctypes.c_int
    L.moe_forward_fp8_all_timed.argtypes = fp8_all_args + [ctypes.POINTER(P)]
    L.moe_forward_fp8_all_timed.restype = ctypes.c_int
    L.moe_forward_fp8_all_host_io_batches.argtypes = ([cfgp, ctypes.c_int32] + [P] * 13
                                                      + [SZ, P, P, P])
    L.moe_forward_fp8_all_host_io_batches.restype = ctypes.c_int
    L.moe_launch_count_fp8.argtypes = [cfgp, I32P]
    L.moe_launch_count_fp8.restype = ctypes.c_int
    L.moe_router_z_loss.argtypes = [P, ctypes.c_int32, ctypes.c_int32, P, P]
    L.moe_router_z_loss.restype = ctypes.c_int
    L.moe_bias_update.argtypes = [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.c_float, P, P]
    L.moe_bias_update.restype = ctypes.c_int
    L.moe_check_status.argtypes = [P, P]
    L.moe_check_status.restype = ctypes.c_int
    L.moe_error_string.argtypes = [ctypes.c_int]
    L.moe_error_string.restype = ctypes.c_char_p
    L.moe_launch_count.argtypes = [cfgp, I32P]
    L.moe_launch_count.restype = ctypes.c_int
    L.moe_plan_flags.argtypes = [cfgp, ctypes.POINTER(ctypes.c_uint32)]
    L.moe_plan_flags.restype = ctypes.c_int
    L.moe_plan_flags_fp8.argtypes = [cfgp, ctypes.POINTER(ctypes.c_uint32)]
    L.moe_plan_flags_fp8.restype = ctypes.c_int
    L.moe_set_tuning.argtypes = [ctypes.c_int32, ctypes.c_int32]
    L.moe_set_tuning.restype = ctypes.c_int
    L.moe_selftest_wait_timeout.argtypes = [P, SZ, ctypes.c_uint64, P]
    L.moe_selftest_wait_timeout.restype = ctypes.c_int
    _libs[path] = L
    return L


def error_string(code: int) -> str:
    try:
        return lib().moe_error_string(code).decode()
    except Exception:  # pragma: no cover - only when the library itself is missing
        return f"code {code}"


def check(code: int, what: str) -> None:
    if code != MOE_OK:
        raise MoeError(code, what)
