"""ctypes loader for libmoe.so: the C ABI declared in include/moe.h and include/moe_adamw.h.

Argument marshalling only.  There is no fallback: if the library has not been
built (``__graft_entry__.build()`` or ``python -m top_softmax_router_gb300.build``)
loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED_SHAPE = -2
MOE_ERR_WORKSPACE_TOO_SMALL = -3
MOE_ERR_CUDA = -4
MOE_ERR_TIMEOUT = -5
MOE_ERR_DEVICE_CHECK = -6
MOE_ERR_NOT_BUILT = -7

KERNEL_CLASSES = ["router_logits", "router_topk", "plan", "gather", "gemm_gateup", "gemm_down", "combine",
                  "gemm_dact", "gemm_dw", "gemm_dx", "unpermute", "router_dw", "zero", "hop_plan", "finalize",
                  "adamw", "ce_logits", "ce_merge", "ce_dlogit", "ce_dx", "ce_dw", "route_grad"]

# Every symbol include/*.h declares.
EXPORTS = ["moe_workspace_bytes", "moe_route", "moe_plan", "moe_chunk_plan", "moe_forward", "moe_backward",
           "moe_check_status", "moe_set_wait_limit_ns", "moe_last_stats", "moe_strerror", "moe_profile_enable",
           "moe_profile_read", "moe_profile_reset", "moe_diag_wait_timeout", "moe_diag_gemm_wait_stats",
           "moe_route_noalloc",
           "moe_hop_rows_worst_case", "moe_hops_workspace_bytes", "moe_forward_hops", "moe_backward_hops",
           "moe_set_gemm_form", "moe_set_launch_chaining", "moe_set_dispatch", "moe_adamw_staging_bytes", "moe_adamw_offload_step", "moe_adamw_step",
           "moe_ce_workspace_bytes", "moe_ce_forward", "moe_ce_backward", "moe_ce_last_stats"]

MOE_GEMM_AUTO, MOE_GEMM_SINGLE, MOE_GEMM_PAIR = 0, 1, 2
MOE_DISPATCH_GATHER, MOE_DISPATCH_ON_LOAD = 0, 1
MOE_CHAIN_NONE, MOE_CHAIN_EARLY, MOE_CHAIN_LATE = 0, 1, 2
MOE_GRAD_F32, MOE_GRAD_BF16 = 0, 1
MOE_ADAMW_MAX_SLOTS = 16
MOE_GEMM_WAIT_CLASSES, MOE_GEMM_WAIT_FIELDS = 32, 8


class MoeConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("N", "H", "E", "k", "I", "c", "K_max")]


class AdamwHparams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in ("lr", "beta1", "beta2", "eps", "weight_decay")] + \
        [("step", ctypes.c_int64)]


class CeConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("N", "H", "V", "P")]


class CeStats(ctypes.Structure):
    _fields_ = [("strips", ctypes.c_int32), ("strip_classes", ctypes.c_int32), ("strip_bytes", ctypes.c_int64),
                ("strip_bound_bytes", ctypes.c_int64), ("partial_bytes", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("kernel_launches", ctypes.c_int32)]


class MoeStats(ctypes.Structure):
    _fields_ = [("K", ctypes.c_int32), ("c_eff", ctypes.c_int32), ("routed_rows", ctypes.c_int64),
                ("routed_bytes_peak", ctypes.c_int64), ("routed_bytes_bound", ctypes.c_int64),
                ("inter_bytes_peak", ctypes.c_int64), ("inter_bytes_bound", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("kernel_launches", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmoe.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        cfgp = ctypes.POINTER(MoeConfig)
        hpp = ctypes.POINTER(AdamwHparams)
        cep = ctypes.POINTER(CeConfig)
        sig = {
            "moe_workspace_bytes": [cfgp, ctypes.POINTER(SZ), ctypes.POINTER(SZ), ctypes.POINTER(SZ)],
            "moe_route": [cfgp, P, P, P, P, P, P, SZ, P],
            "moe_plan": [cfgp, P, P, P, P, P, SZ, P],
            "moe_chunk_plan": [cfgp, ctypes.POINTER(I32), ctypes.POINTER(I32)],
            "moe_forward": [cfgp, P, P, P, P, P, P, P, P, SZ, P],
            "moe_backward": [cfgp, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P],
            "moe_check_status": [P, P],
            "moe_set_wait_limit_ns": [I64],
            "moe_last_stats": [ctypes.POINTER(MoeStats)],
            "moe_strerror": [ctypes.c_int],
            "moe_profile_enable": [ctypes.c_int],
            "moe_profile_read": [ctypes.POINTER(I32), ctypes.POINTER(ctypes.c_double),
                                 ctypes.POINTER(ctypes.c_char_p)],
            "moe_profile_reset": [],
            "moe_diag_wait_timeout": [I64, P, SZ, P],
            "moe_diag_gemm_wait_stats": [P, ctypes.c_int],
            "moe_route_noalloc": [cfgp, P, P, P, P, P, P],
            "moe_hop_rows_worst_case": [cfgp, I32, ctypes.POINTER(I32)],
            "moe_set_gemm_form": [ctypes.c_int],
            "moe_set_launch_chaining": [ctypes.c_int],
            "moe_set_dispatch": [ctypes.c_int],
            "moe_hops_workspace_bytes": [cfgp, I32, I32, ctypes.POINTER(SZ), ctypes.POINTER(SZ)],
            "moe_forward_hops": [cfgp, I32, I32, P, P, P, P, P, P, P, P, SZ, P],
            "moe_backward_hops": [cfgp, I32, I32, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P],
            "moe_adamw_staging_bytes": [I64, I32, ctypes.POINTER(SZ)],
            "moe_adamw_offload_step": [hpp, I64, I64, I32, P, P, P, P, I32, P, P, SZ, P],
            "moe_adamw_step": [hpp, I64, P, P, P, P, I32, P, P],
            "moe_ce_workspace_bytes": [cep, ctypes.POINTER(SZ), ctypes.POINTER(SZ)],
            "moe_ce_forward": [cep, P, P, P, P, P, P, P, SZ, P],
            "moe_ce_backward": [cep, P, P, P, P, P, P, P, P, SZ, P],
            "moe_ce_last_stats": [ctypes.POINTER(CeStats)],
        }
        for name, args in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ctypes.c_char_p if name == "moe_strerror" else ctypes.c_int
        _lib = lib
        return lib


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = load().moe_strerror(code)
        super().__init__(f"{where}: {msg.decode() if msg else code}")


def check(code: int, where: str) -> None:
    if code != MOE_OK:
        raise MoeError(code, where)
