"""The routing entry point for callers that cannot allocate device memory.

moe_route_quant_mxfp8_noalloc serves callers that own their inputs and
outputs but may not cudaMalloc a workspace (for instance a serving runtime
that has split all device memory into its own pool).  Its scratch is a fixed
2 MiB array inside the library, shared by every call.  These tests call it
through the C ABI and check that its results equal those of
moe_route_quant_mxfp8 (which takes a caller-provided workspace), bit for bit,
on two calls in a row with different inputs -- the second call must not see
anything the first one left in the shared array.  This file is collected
last so a failure here comes after every other test has run.
"""

import ctypes as C

import pytest
import torch

from mxfp8_block_scaled_moe_gb300 import workloads


@pytest.fixture(scope="module")
def mm():
    import __graft_entry__
    __graft_entry__.build()
    import mxfp8_block_scaled_moe_gb300 as m
    return m


@pytest.mark.gpu
def test_noalloc_route_matches_workspace_entry_point_twice(mm):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    dev = "cuda"
    for cfg in ("qwen3_30b_prefill", "tiny"):      # two calls in a row, different shapes
        shape = workloads.CONFIGS[cfg]
        inp = workloads.make_layer(shape, dev, weights=False)
        got = mm.api.moe_route_quant_mxfp8_noalloc(inp["x"], inp["logits"], shape.k)
        want = mm.moe_route_quant_mxfp8(inp["x"], inp["logits"], shape.k)
        torch.cuda.synchronize()
        assert mm.device_status() == 0
        assert set(got) == set(want)
        for key in want:
            assert torch.equal(got[key], want[key]), (cfg, key)


def test_noalloc_route_rejects_sizes_beyond_its_scratch(mm):
    """ceil(T/64) * E above 262144 is refused before anything is launched."""
    from mxfp8_block_scaled_moe_gb300 import _lib
    lib = _lib.load()
    p = C.c_void_p(4096)          # never dereferenced: the size check comes first
    T, E = 64 * 257, 1024         # 257 * 1024 = 263168 > 262144
    rc = lib.moe_route_quant_mxfp8_noalloc(p, p, T, 256, E, 8, 1, p, p, p, p, p, p, p, p,
                                           C.c_void_p(0))
    assert rc == 5                # MXMOE_ERR_WORKSPACE
    assert "workspace" in lib.mxmoe_status_string(rc).decode()
