"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument validation rejects bad calls before any launch (no GPU needed)."""

import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mxfp8_block_scaled_moe_gb300 import _lib, build
    build.build()
    return _lib.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "mxmoe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_every_declared_symbol_is_exported(lib):
    from mxfp8_block_scaled_moe_gb300 import _lib
    declared = _declared_functions()
    assert len(declared) >= 13
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(_lib.EXPORTS)


def test_status_strings(lib):
    for code in range(9):
        assert lib.mxmoe_status_string(code).decode().startswith("MXMOE_")
    assert b"sm_103a" in lib.mxmoe_version()


def test_workspace_sizes(lib):
    assert lib.moe_route_quant_mxfp8_workspace_size(16384, 128) >= 256 * 128 * 4
    ws = lib.moe_forward_mxfp8_workspace_size(16384, 2048, 128, 8, 768)
    M = 16384 * 8
    assert ws >= M * 2048 * 3 + M * 768
    assert lib.moe_forward_mxfp8_workspace_size(-1, 2048, 128, 8, 768) == 0


def test_host_validation_rejects_bad_arguments(lib):
    p = C.c_void_p(4096)        # never dereferenced: validation fails first
    odd = C.c_void_p(4097)
    nul = C.c_void_p(0)
    # K not a multiple of 32
    assert lib.mx_quantize_3d(p, 1, 4, 33, p, p, nul) == 3
    # misaligned payload pointer
    assert lib.mx_quantize_3d(odd, 1, 4, 64, p, p, nul) == 2
    # null weight pointer
    assert lib.mx_quantize_3d(nul, 1, 4, 64, p, p, nul) == 1
    # empty tensor is a no-op
    assert lib.mx_quantize_3d(nul, 0, 4, 64, nul, nul, nul) == 0
    # k > E
    assert lib.moe_route_quant_mxfp8(p, p, 4, 64, 4, 5, 1, p, p, p, p, p, p, p, p, p, 1 << 20, nul) == 3
    # workspace too small
    assert lib.moe_route_quant_mxfp8(p, p, 4096, 64, 8, 2, 1, p, p, p, p, p, p, p, p, p, 16, nul) == 5
    # GEMM with K % 128 != 0 -> unsupported; E > 256 -> unsupported
    assert lib.grouped_gemm_mxfp8(p, p, p, p, p, 128, 8, 96, 256, p, nul) == 4
    assert lib.grouped_gemm_mxfp8(p, p, p, p, p, 128, 300, 128, 256, p, nul) == 4
    # negative M
    assert lib.grouped_gemm_swiglu_quant_mxfp8(p, p, p, p, p, -1, 8, 256, 128, p, p, nul) == 3
    # finalize: H % 8 != 0
    assert lib.moe_finalize_routing(p, p, p, 4, 2, 12, p, nul) == 3
    # forward: workspace not 256-aligned / too small
    assert lib.moe_forward_mxfp8(p, p, p, p, p, p, 64, 256, 8, 2, 128, 1, p, C.c_void_p(4096 + 16),
                                 1 << 30, nul) == 2
    assert lib.moe_forward_mxfp8(p, p, p, p, p, p, 64, 256, 8, 2, 128, 1, p, p, 1024, nul) == 5
    # T == 0 is a no-op
    assert lib.moe_forward_mxfp8(nul, nul, nul, nul, nul, nul, 0, 256, 8, 2, 128, 1, nul, nul, 0,
                                 nul) == 0
    # host-buffer layer with an explicit chunk plan: sizes must be positive
    # and sum to T (checked before any device work)
    big = 1 << 40
    for plan, ok in (([30, 30], False), ([64, 0], False), ([70, -6], False), ([], False)):
        arr = (C.c_int32 * max(1, len(plan)))(*plan)
        st = lib.moe_forward_mxfp8_host_plan(p, p, p, p, p, p, 64, 256, 8, 2, 128, 1, p,
                                             C.cast(arr, C.c_void_p), len(plan), p, big, nul)
        assert st == 3, (plan, st)
    # the default plan: one chunk up to 4096 tokens, three beyond (slot = largest chunk)
    w1 = lib.moe_forward_mxfp8_host_workspace_size(4096, 2048, 128, 8, 768, 0)
    assert w1 == lib.moe_forward_mxfp8_host_workspace_size(4096, 2048, 128, 8, 768, 1)
    w3 = lib.moe_forward_mxfp8_host_workspace_size(16384, 2048, 128, 8, 768, 0)
    assert w3 == lib.moe_forward_mxfp8_host_workspace_size(10240, 2048, 128, 8, 768, 1)


def test_python_binding_refuses_cpu_tensors():
    import torch
    import mxfp8_block_scaled_moe_gb300 as mm
    with pytest.raises(ValueError, match="CUDA"):
        mm.mx_quantize_3d(torch.zeros(2, 64, dtype=torch.bfloat16))


def test_host_validation_of_the_linear_router_and_fp4_entry_points(lib):
    p = C.c_void_p(4096)
    nul = C.c_void_p(0)
    # dense linear: K % 16 != 0 / N % 16 != 0 -> shape; M == 0 is a no-op
    assert lib.mxfp8_linear(p, p, p, 8, 64, 40, p, p, 1 << 30, nul) == 3
    assert lib.mxfp8_linear(p, p, p, 8, 40, 64, p, p, 1 << 30, nul) == 3
    assert lib.mxfp8_linear(nul, nul, nul, 0, 64, 64, nul, nul, 0, nul) == 0
    # output not 32-byte aligned, workspace too small
    assert lib.mxfp8_linear(p, p, p, 8, 64, 64, C.c_void_p(4096 + 16), p, 1 << 30, nul) == 2
    assert lib.mxfp8_linear(p, p, p, 8, 64, 64, p, p, 16, nul) == 5
    assert lib.mxfp8_linear_workspace_size(8, 64, 40) == 0
    assert lib.mxfp8_linear_workspace_size(128, 4096, 4304) >= 128 * 4304
    # W4A4 linear: K % 128 != 0 -> shape; packed weights must be 32-byte aligned
    assert lib.mxfp4_linear(p, p, p, 8, 64, 192, p, p, 1 << 30, nul) == 3
    assert lib.mxfp4_linear(p, C.c_void_p(4096 + 16), p, 8, 64, 256, p, p, 1 << 30, nul) == 2
    # router: H % 64, E > 256, k > 32 -> unsupported; k > E -> shape
    assert lib.moe_router_gate_topk(p, p, 8, 96, 128, 8, 1, nul, p, p, nul) == 4
    assert lib.moe_router_gate_topk(p, p, 8, 128, 300, 8, 1, nul, p, p, nul) == 4
    assert lib.moe_router_gate_topk(p, p, 8, 128, 128, 33, 1, nul, p, p, nul) == 4
    assert lib.moe_router_gate_topk(p, p, 8, 128, 4, 8, 1, nul, p, p, nul) == 3
    assert lib.moe_router_gate_topk(nul, nul, 0, 128, 16, 2, 1, nul, nul, nul, nul) == 0
    # gate dequant: K % 32 != 0
    assert lib.mx_dequantize_bf16_2d(p, p, 4, 48, p, nul) == 3
    # W4A4 and gated layers share the layer's checks (k > E -> shape)
    assert lib.moe_forward_w4a4_mma_scales(p, p, p, p, p, p, 64, 256, 8, 9, 128, 1, p, p,
                                           1 << 30, nul) == 3
    assert lib.moe_forward_mxfp8_gated_mma_scales(p, p, p, p, p, p, 64, 256, 8, 9, 128, 1, p, p,
                                                  1 << 30, nul) == 3
