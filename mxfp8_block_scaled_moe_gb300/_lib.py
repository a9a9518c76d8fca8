"""ctypes loader of libmxmoe.so and the C-ABI prototypes of include/mxmoe.h.

Loading fails loudly if the library has not been built: there is no CPU or
PyTorch fallback for any entry point.
"""

from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmxmoe.so")

# every symbol include/mxmoe.h declares
EXPORTS = (
    "mxmoe_status_string", "mxmoe_version", "mxmoe_get_device_status",
    "mxmoe_set_wait_limit_cycles", "mx_quantize_3d", "moe_route_quant_mxfp8_workspace_size",
    "moe_route_quant_mxfp8", "moe_route_permute_bf16", "grouped_gemm_swiglu_quant_mxfp8",
    "grouped_gemm_mxfp8", "moe_finalize_routing", "moe_forward_mxfp8_workspace_size",
    "moe_forward_mxfp8", "moe_route_quant_mxfp8_noalloc", "mx_scales_to_mma_layout",
    "moe_forward_mxfp8_mma_scales", "mxmoe_layer_profile_enable", "mxmoe_layer_profile_read",
    "mxmoe_set_gemm_2sm", "mxmoe_set_gemm_chain", "moe_forward_mxfp8_host", "moe_forward_mxfp8_host_workspace_size",
    "moe_forward_mxfp8_host_plan", "mx_quantize_fp4_3d", "moe_forward_w4a8_mma_scales",
    "mxfp8_linear_workspace_size", "mxfp8_linear", "mxfp8_linear_mma_scales",
    "moe_forward_w4a4_mma_scales", "mxfp4_linear", "mxfp4_linear_mma_scales",
    "moe_router_gate_topk", "mx_dequantize_bf16_2d", "moe_forward_mxfp8_gated_mma_scales",
)

_P = C.c_void_p
_I = C.c_int
_I64 = C.c_int64
_SZ = C.c_size_t

_PROTOS = {
    "mxmoe_status_string": (C.c_char_p, [_I]),
    "mxmoe_version": (C.c_char_p, []),
    "mxmoe_get_device_status": (_I, [C.POINTER(C.c_int32), _I]),
    "mxmoe_set_wait_limit_cycles": (None, [C.c_longlong]),
    "mx_quantize_3d": (_I, [_P, _I64, _I64, _I64, _P, _P, _P]),
    "moe_route_quant_mxfp8_workspace_size": (_SZ, [_I, _I]),
    "moe_route_quant_mxfp8": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _P, _SZ, _P]),
    "moe_route_quant_mxfp8_noalloc": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                                           _P, _P, _P]),
    "moe_route_permute_bf16": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                    _P, _SZ, _P]),
    "grouped_gemm_swiglu_quant_mxfp8": (_I, [_P, _P, _P, _P, _P, _I64, _I, _I, _I, _P, _P, _P]),
    "grouped_gemm_mxfp8": (_I, [_P, _P, _P, _P, _P, _I64, _I, _I, _I, _P, _P]),
    "moe_finalize_routing": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_forward_mxfp8_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_forward_mxfp8": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "moe_forward_mxfp8_mma_scales": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P,
                                          _SZ, _P]),
    "moe_forward_w4a8_mma_scales": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P,
                                         _SZ, _P]),
    "mx_scales_to_mma_layout": (_I, [_P, _I64, _I64, _I64, _P, _P]),
    "mxmoe_layer_profile_enable": (_I, [_I]),
    "mxmoe_set_gemm_2sm": (None, [_I]),
    "mxmoe_set_gemm_chain": (None, [_I]),
    "moe_forward_mxfp8_host_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moe_forward_mxfp8_host": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _P,
                                    _SZ, _P]),
    "moe_forward_mxfp8_host_plan": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P,
                                         _I, _P, _SZ, _P]),
    "mx_quantize_fp4_3d": (_I, [_P, _I64, _I64, _I64, _P, _P, _P]),
    "mxmoe_layer_profile_read": (_I, [C.POINTER(C.c_float), _I]),
    "mxfp8_linear_workspace_size": (_SZ, [_I64, _I64, _I64]),
    "mxfp8_linear": (_I, [_P, _P, _P, _I64, _I64, _I64, _P, _P, _SZ, _P]),
    "mxfp8_linear_mma_scales": (_I, [_P, _P, _P, _I64, _I64, _I64, _P, _P, _SZ, _P]),
    "moe_forward_w4a4_mma_scales": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P,
                                         _SZ, _P]),
    "mxfp4_linear": (_I, [_P, _P, _P, _I64, _I64, _I64, _P, _P, _SZ, _P]),
    "mxfp4_linear_mma_scales": (_I, [_P, _P, _P, _I64, _I64, _I64, _P, _P, _SZ, _P]),
    "moe_router_gate_topk": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "mx_dequantize_bf16_2d": (_I, [_P, _P, _I64, _I64, _P, _P]),
    "moe_forward_mxfp8_gated_mma_scales": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                                _P, _P, _SZ, _P]),
}

_lib = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load (once) and return the library with its prototypes set."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"libmxmoe.so not found at {path}: build it first "
            "(python -m mxfp8_block_scaled_moe_gb300.build, or __graft_entry__.build())")
    lib = C.CDLL(path)
    for name, (res, args) in _PROTOS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class MXMoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = load().mxmoe_status_string(code).decode()
        super().__init__(f"{fn} failed: {msg} (status {code})")
        self.code = code


def check(fn: str, code: int) -> None:
    if code != 0:
        raise MXMoEError(fn, code)
