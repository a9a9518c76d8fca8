"""GPU parity of the whole layer (moe_forward_mxfp8, one C-ABI call) against
the oracle on the small shapes, the entry points' agreement, the 1-SM / 2-SM
kernel agreement and the host-buffer call (the prefill shapes against the
oracle: test_gpu_full_oracle.py)."""

import numpy as np
import pytest
import torch

from oracle import moe
from mxfp8_block_scaled_moe_gb300 import workloads

from _util import OUT_REL_FROB, bits16, rel_frob, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def mm():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import mxfp8_block_scaled_moe_gb300 as m
    return m


@pytest.mark.parametrize("cfg", ["tiny", "qwen3_30b_decode"])
def test_layer_matches_oracle(mm, cfg):
    shape = workloads.CONFIGS[cfg]
    inp = workloads.make_layer(shape, DEV)
    layer = mm.MXFP8MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    out = layer(inp["x"], inp["logits"])
    out2 = layer(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    assert torch.equal(out, out2)      # deterministic, workspace reuse is clean
    ref = moe.moe_forward(bits16(inp["x"]), inp["logits"].cpu().numpy(), u8(layer.w13q),
                          u8(layer.w13s), u8(layer.w2q), u8(layer.w2s), shape.k, shape.I)
    assert rel_frob(bits16(out), ref["out"]) <= OUT_REL_FROB


@pytest.mark.parametrize("mode", [0, 1])
def test_layer_at_the_expert_limit(mm, mode):
    """E = 256 (the layer's maximum) with top-8 over a ragged batch: many
    experts hold 0-3 rows, the tile schedule spans every lane's 8 experts."""
    T, H, E, k, I = 300, 256, 256, 8, 128
    g = torch.Generator(device=DEV).manual_seed(256)
    x = torch.randn(T, H, generator=g, device=DEV).to(torch.bfloat16)
    logits = torch.randn(T, E, generator=g, device=DEV)
    w13 = (torch.randn(E, 2 * I, H, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    w2 = (torch.randn(E, H, I, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    layer = mm.MXFP8MoELayer.from_bf16(w13, w2, k)
    mm.set_gemm_2sm(mode)
    try:
        out = layer(x, logits)
        torch.cuda.synchronize()
    finally:
        mm.set_gemm_2sm("auto")
    assert mm.device_status() == 0
    ref = moe.moe_forward(bits16(x), logits.cpu().numpy(), u8(layer.w13q), u8(layer.w13s),
                          u8(layer.w2q), u8(layer.w2s), k, I)
    assert rel_frob(bits16(out), ref["out"]) <= OUT_REL_FROB


def _mma_layout_numpy(s, K):
    """Re-index [R, K/32] scales into 512-byte chunks (row block, K slice):
    byte (r % 32) * 16 + (r // 32) * 4 + kb of chunk (row // 128, kt)."""
    R = s.shape[0]
    KT = K // 128
    out = np.zeros(R * K // 32, np.uint8)
    rows = np.arange(R)[:, None]
    j = np.arange(K // 32)[None, :]
    r = rows % 128
    off = ((rows // 128) * KT + j // 4) * 512 + (r % 32) * 16 + (r // 32) * 4 + (j % 4)
    out[off.reshape(-1)] = s.reshape(-1)
    return out


@pytest.mark.parametrize("E,N,K", [(1, 128, 128), (3, 256, 384), (8, 1536, 2048)])
def test_scales_to_mma_layout(mm, E, N, K):
    g = torch.Generator(device=DEV).manual_seed(E + N + K)
    s = torch.randint(0, 255, (E, N, K // 32), generator=g, device=DEV, dtype=torch.int32)
    s = s.to(torch.uint8)
    t = mm.mx_scales_to_mma_layout(s, K)
    torch.cuda.synchronize()
    assert np.array_equal(u8(t).reshape(-1), _mma_layout_numpy(u8(s).reshape(E * N, -1), K))


@pytest.mark.parametrize("cfg", ["tiny", "qwen3_30b_decode", "qwen3_30b_prefill"])
def test_layer_entry_points_agree(mm, cfg):
    """moe_forward_mxfp8 (canonical weight scales), moe_forward_mxfp8_mma_scales
    and the four per-step entry points give the same bytes."""
    shape = workloads.CONFIGS[cfg]
    inp = workloads.make_layer(shape, DEV)
    layer = mm.MXFP8MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    del inp["w13"], inp["w2"]
    a = mm.moe_forward_mxfp8(inp["x"], inp["logits"], layer.w13q, layer.w13s, layer.w2q,
                             layer.w2s, shape.k)
    b = layer(inp["x"], inp["logits"])
    r = mm.moe_route_quant_mxfp8(inp["x"], inp["logits"], shape.k)
    aq, as_ = mm.grouped_gemm_swiglu_quant_mxfp8(r["xq"], r["xs"], layer.w13q, layer.w13s,
                                                 r["expert_offsets"])
    y = mm.grouped_gemm_mxfp8(aq, as_, layer.w2q, layer.w2s, r["expert_offsets"])
    c = mm.moe_finalize_routing(y, r["topk_w"], r["src_to_sorted"], shape.k)
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    assert torch.equal(a, b)
    assert torch.equal(a, c)


def test_layer_profile_segments(mm):
    shape = workloads.CONFIGS["tiny"]
    inp = workloads.make_layer(shape, DEV)
    layer = mm.MXFP8MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    mm.api.layer_profile_enable(True)
    try:
        layer(inp["x"], inp["logits"])
        prof = mm.api.layer_profile_read()
    finally:
        mm.api.layer_profile_enable(False)
    assert prof["weight_scale_layout"] >= 0.0
    for key in ("route_quant", "gemm1_swiglu_quant", "gemm2", "finalize"):
        assert prof[key] > 0.0, key


@pytest.mark.parametrize("cfg", ["tiny", "qwen3_30b_decode", "qwen3_30b_prefill", "qwen3_235b_prefill"])
def test_two_sm_and_one_sm_gemm_kernels_agree(mm, cfg):
    """The 2-SM (cta_group::2) and 1-SM grouped GEMMs give the same layer bytes,
    alone or mixed (the default sends gmm2 to the 2-SM kernel)."""
    shape = workloads.CONFIGS[cfg]
    inp = workloads.make_layer(shape, DEV)
    if shape.offline:
        layer = mm.MXFP8MoELayer.from_quantized(inp["w13q"], inp["w13s"], inp["w2q"], inp["w2s"],
                                                shape.k)
    else:
        layer = mm.MXFP8MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    outs = []
    try:
        for mode in (0, 1, "auto"):  # 1-SM, 2-SM, 2-SM for gmm2 only
            mm.api.set_gemm_2sm(mode)
            outs.append(layer(inp["x"], inp["logits"]))
    finally:
        mm.api.set_gemm_2sm("auto")
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


@pytest.mark.parametrize("shape", [
    workloads.CONFIGS["qwen3_30b_decode"],                       # 32 tokens, ~110 of 128 experts
    workloads.CONFIGS["qwen3_30b_decode"].with_tokens(1),        # 8 experts, one row each
    workloads.CONFIGS["qwen3_30b_decode"].with_tokens(7),
    workloads.CONFIGS["qwen3_30b_skewed"].with_tokens(32),       # Zipf routing: crowded experts
    workloads.LayerShape("chain_e8", T=32, H=512, E=8, k=2, I=256, seed=5, gate_std=0.05),
], ids=lambda s: s.name)
def test_small_batch_gemm_chain_equals_two_kernels(mm, shape):
    """At most 32 tokens: both grouped GEMMs in one persistent kernel (gmm2's
    units of an expert wait for that expert's gmm1 units) give the bytes of one
    kernel per GEMM, on uniform, single-token, skewed and few-expert routing
    (up to 32 rows per expert, gmm2 units waiting on gmm1 units of other CTAs)."""
    inp = workloads.make_layer(shape, DEV)
    layer = mm.MXFP8MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    outs = []
    try:
        for chain in (False, True, True):
            mm.api.set_gemm_chain(chain)
            outs.append(layer(inp["x"], inp["logits"]).clone())
    finally:
        mm.api.set_gemm_chain(True)
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_small_batch_gemm_chain_token_sweep(mm):
    """One set of Qwen3-30B-A3B-shaped weights, token counts 2..31 in turn (the
    per-expert counters are zeroed by every routing step): the one-kernel GEMMs
    give the bytes of one kernel per GEMM at every size."""
    shape = workloads.CONFIGS["qwen3_30b_decode"]
    inp = workloads.make_layer(shape.with_tokens(31), DEV)
    layer = mm.MXFP8MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    try:
        for T in (2, 3, 9, 16, 24, 31):
            x, logits = inp["x"][:T].contiguous(), inp["logits"][:T].contiguous()
            mm.api.set_gemm_chain(False)
            ref = layer(x, logits).clone()
            mm.api.set_gemm_chain(True)
            out = layer(x, logits)
            torch.cuda.synchronize()
            assert torch.equal(out, ref), T
    finally:
        mm.api.set_gemm_chain(True)
    assert mm.device_status() == 0


@pytest.mark.parametrize("cfg,n_chunks", [("tiny", 3), ("qwen3_30b_decode", 0),
                                          ("qwen3_30b_prefill", 0), ("qwen3_30b_prefill", 5)])
def test_host_buffer_layer_matches_device_layer(mm, cfg, n_chunks):
    """Chunked, copy-overlapped layer on host buffers == the on-device layer."""
    shape = workloads.CONFIGS[cfg]
    inp = workloads.make_layer(shape, DEV)
    layer = mm.MXFP8MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    ref = layer(inp["x"], inp["logits"])
    x_h = inp["x"].cpu().pin_memory()
    l_h = inp["logits"].cpu().pin_memory()
    out_h = layer.forward_host(x_h, l_h, n_chunks=n_chunks)
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    assert torch.equal(out_h, ref.cpu())


@pytest.mark.parametrize("cfg,chunks", [("tiny", [5, 50, 9]), ("tiny", [64]),
                                        ("qwen3_30b_prefill", [1000, 15000, 384]),
                                        ("qwen3_30b_prefill", [3072, 10240, 3072])])
def test_host_buffer_layer_explicit_chunk_plan(mm, cfg, chunks):
    """An explicit uneven chunk plan gives the on-device layer's bytes."""
    shape = workloads.CONFIGS[cfg]
    inp = workloads.make_layer(shape, DEV)
    layer = mm.MXFP8MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    ref = layer(inp["x"], inp["logits"])
    x_h = inp["x"].cpu().pin_memory()
    l_h = inp["logits"].cpu().pin_memory()
    out_h = layer.forward_host(x_h, l_h, chunks=chunks)
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    assert torch.equal(out_h, ref.cpu())
