"""ctypes view of libmoe_b300.so (the C ABI declared in include/moe.h)."""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_b300.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT",
                6: "MOE_ERR_NO_DEVICE"}
MOE_TRACE_MAX_EVENTS = 32

# every symbol include/moe.h declares
EXPORTED = ["moe_workspace_size", "moe_max_rows", "moe_capacity", "moe_forward_num_launches",
            "moe_forward_launch_name", "moe_route", "moe_expert_choice", "moe_update_sel_bias", "moe_permute",
            "moe_expert_ffn", "moe_combine", "moe_forward", "moe_forward_host",
            "moe_permute_static", "moe_workspace_status", "moe_debug_suppress_gemm_producer",
            "moe_status_string", "moe_version"]
MOE_STATIC_MAX_ASSIGNMENTS = 65536
MOE_STATIC_MAX_EXPERTS = 256


ROUTING = {"token": 0, "expert": 1}
ACTIVATION = {"gelu": 0, "silu": 1, "swiglu": 2}
DROP_ORDER = {"token": 0, "slot": 1}
WEIGHT_DTYPE = {"bf16": 0, "e4m3": 1}


class MoeConfig(C.Structure):
    _fields_ = [("T", C.c_int32), ("H", C.c_int32), ("F", C.c_int32), ("N", C.c_int32),
                ("k", C.c_int32), ("capacity_factor", C.c_float), ("F_shared", C.c_int32),
                ("aux_alpha", C.c_float), ("routing", C.c_int32), ("activation", C.c_int32),
                ("min_capacity", C.c_int32), ("drop_order", C.c_int32),
                ("weight_dtype", C.c_int32)]


class MoeWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in
                ("Wg", "bg", "sel_bias", "W1", "b1", "W2", "b2", "W1s", "b1s", "W2s", "b2s",
                 "s1", "s2", "s1s", "s2s")]


class MoeOutputs(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in
                ("topk_idx", "topk_w", "probs", "p_mean", "counts", "offsets", "perm", "inv",
                 "f", "l_aux", "z_loss", "logits")]


_lib = None


def load() -> C.CDLL:
    """Loads the in-tree library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python sparse_mixture_experts_72_b300/build.py`")
    lib = C.CDLL(LIB_PATH)
    P = C.c_void_p
    cfgp = C.POINTER(MoeConfig)
    lib.moe_workspace_size.argtypes = [cfgp]
    lib.moe_workspace_size.restype = C.c_size_t
    lib.moe_max_rows.argtypes = [cfgp]
    lib.moe_max_rows.restype = C.c_int64
    lib.moe_capacity.argtypes = [cfgp]
    lib.moe_capacity.restype = C.c_int64
    lib.moe_forward_num_launches.argtypes = [cfgp]
    lib.moe_forward_num_launches.restype = C.c_int32
    lib.moe_forward_launch_name.argtypes = [cfgp, C.c_int32]
    lib.moe_forward_launch_name.restype = C.c_char_p
    lib.moe_route.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, P, P, C.c_size_t, P]
    lib.moe_route.restype = C.c_int
    lib.moe_expert_choice.argtypes = [cfgp, P, P, P, P, P, P, P, P, P]
    lib.moe_expert_choice.restype = C.c_int
    lib.moe_update_sel_bias.argtypes = [cfgp, P, P, C.c_float, P]
    lib.moe_update_sel_bias.restype = C.c_int
    lib.moe_permute.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, C.c_size_t, P]
    lib.moe_permute.restype = C.c_int
    lib.moe_expert_ffn.argtypes = [cfgp, P, P, P, P, C.POINTER(MoeWeights), P, P, P, C.c_size_t, P]
    lib.moe_expert_ffn.restype = C.c_int
    lib.moe_combine.argtypes = [cfgp, P, P, P, P, P]
    lib.moe_combine.restype = C.c_int
    lib.moe_forward.argtypes = [cfgp, C.POINTER(MoeWeights), P, P, C.POINTER(MoeOutputs), P,
                                C.c_size_t, P, P]
    lib.moe_forward.restype = C.c_int
    lib.moe_forward_host.argtypes = [cfgp, C.POINTER(MoeWeights), P, P, P, P,
                                     C.POINTER(MoeOutputs), P, C.c_size_t, P, P, P]
    lib.moe_forward_host.restype = C.c_int
    lib.moe_permute_static.argtypes = [cfgp, P, P, P, P, P, P, P, P, P]
    lib.moe_permute_static.restype = C.c_int
    lib.moe_workspace_status.argtypes = [P, P]
    lib.moe_workspace_status.restype = C.c_int
    lib.moe_debug_suppress_gemm_producer.argtypes = [C.c_int]
    lib.moe_debug_suppress_gemm_producer.restype = C.c_int
    lib.moe_status_string.argtypes = [C.c_int]
    lib.moe_status_string.restype = C.c_char_p
    lib.moe_version.argtypes = []
    lib.moe_version.restype = C.c_char_p
    _lib = lib
    return lib


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = load().moe_status_string(status).decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({msg})")


def check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)
