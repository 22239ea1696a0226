"""ctypes view of the C ABI in include/moe_layer.h (no compute here).

The shared library is built in-tree by ``moe_expert_layer_router_gb300.build``
into ``moe_expert_layer_router_gb300/lib/libmoe_gb300.so``.  Loading fails
loudly when it is missing: there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libmoe_gb300.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "moe_layer.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, \
    MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_BOUNDS = range(7)
MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID = 0, 1
MOE_DTYPE_BF16, MOE_DTYPE_FP8_E4M3, MOE_DTYPE_NVFP4 = 0, 1, 2
MOE_OP_ROUTE, MOE_OP_PERMUTE, MOE_OP_GROUPED_FFN, MOE_OP_COMBINE, MOE_OP_FORWARD = range(5)
MOE_FORWARD_FUSED_DISPATCH = 0x1


class MoeConfig(C.Structure):
    _fields_ = [("T", C.c_int64), ("H", C.c_int32), ("E", C.c_int32), ("k", C.c_int32),
                ("I", C.c_int32), ("I_shared", C.c_int32), ("score", C.c_int32),
                ("renormalize", C.c_int32), ("route_scale", C.c_float), ("wtype", C.c_int32)]


class MoeWeightList(C.Structure):
    _fields_ = [("gate", C.POINTER(C.c_void_p)), ("up", C.POINTER(C.c_void_p)),
                ("down", C.POINTER(C.c_void_p)), ("gate_scales", C.POINTER(C.c_void_p)),
                ("up_scales", C.POINTER(C.c_void_p)), ("down_scales", C.POINTER(C.c_void_p)),
                ("shared_gate", C.c_void_p), ("shared_up", C.c_void_p),
                ("shared_down", C.c_void_p), ("shared_gate_scales", C.c_void_p),
                ("shared_up_scales", C.c_void_p), ("shared_down_scales", C.c_void_p),
                ("gate_sf", C.POINTER(C.c_void_p)), ("down_sf", C.POINTER(C.c_void_p)),
                ("gate_tscale", C.POINTER(C.c_void_p)), ("down_tscale", C.POINTER(C.c_void_p)),
                ("shared_gate_sf", C.c_void_p), ("shared_down_sf", C.c_void_p),
                ("shared_gate_tscale", C.c_void_p), ("shared_down_tscale", C.c_void_p),
                ("input_scale", C.c_float), ("hidden_scale", C.c_float)]


class MoeTrace(C.Structure):
    _fields_ = [("events", C.POINTER(C.c_void_p)), ("kernel_ids", C.POINTER(C.c_int32)),
                ("capacity", C.c_int32), ("count", C.c_int32), ("kernel_mask", C.c_uint32)]


KERNEL_NAMES = ["router", "hist", "scan", "scatter", "plan", "gemm1_gate_up_swiglu",
                "gemm2_down", "combine", "quant"]

_P = C.c_void_p
_CFG = C.POINTER(MoeConfig)
_SIG = {
    "moe_abi_version": (C.c_int32, []),
    "moe_status_string": (C.c_char_p, [C.c_int]),
    "moe_last_error_message": (C.c_char_p, []),
    "moe_workspace_size": (C.c_int, [_CFG, C.c_int32, C.POINTER(C.c_size_t)]),
    "moe_workspace_init": (C.c_int, [_P, C.c_size_t, _P]),
    "moe_get_device_error": (C.c_int, [_P, _P, C.POINTER(C.c_int32)]),
    "moe_weights_create": (C.c_int, [_CFG, C.POINTER(MoeWeightList), C.POINTER(_P)]),
    "moe_weights_destroy": (None, [_P]),
    "moe_stack_create": (C.c_int, [_CFG, C.c_int32, C.POINTER(MoeWeightList), _P, _P,
                                   C.POINTER(_P)]),
    "moe_stack_destroy": (None, [_P]),
    "moe_forward_stack": (C.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "moe_route": (C.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "moe_permute": (C.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "moe_grouped_ffn": (C.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "moe_combine": (C.c_int, [_CFG, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "moe_forward": (C.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "moe_forward_ex": (C.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, C.c_uint32, _P, C.c_size_t, _P]),
    "moe_quantize_weight_fp8": (C.c_int, [_P, C.c_int64, C.c_int64, _P, _P, _P]),
    "moe_quantize_act_fp8": (C.c_int, [_P, C.c_int64, C.c_int64, _P, _P, _P]),
    "moe_quantize_weight_nvfp4": (C.c_int, [_P, _P, C.c_int64, C.c_int64, _P, _P, _P, _P]),
    "moe_quantize_act_nvfp4": (C.c_int, [_P, C.c_int64, C.c_int64, C.c_float, _P, _P, _P]),
    "moe_set_trace": (C.c_int, [C.POINTER(MoeTrace)]),
    "moe_test_stall_gemm1": (C.c_int, [C.c_int32]),
    "moe_nvfp4_rows": (C.c_int, [_CFG, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
    "moe_permute_nvfp4": (C.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                    _P, C.c_size_t, _P]),
    "moe_grouped_ffn_nvfp4": (C.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                        C.c_size_t, _P]),
    "moe_permute_noalloc": (C.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
}

_lib = None


def lib() -> C.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m moe_expert_layer_router_gb300.build` (or __graft_entry__.build())")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIG.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        L = lib()
        msg = L.moe_last_error_message().decode(errors="replace")
        name = L.moe_status_string(status).decode()
        super().__init__(f"{where}: {name} ({status}): {msg}")
        self.status = status


def check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)
