"""GPU parity: MX weight/activation quant, fused route+quant, finalize.

Every kernel runs through the C ABI (the Python binding only marshals
pointers) and is compared with the CPU oracle on the same seeded bytes:
bit-exact for codes, scales, ids, permutation, counts and offsets.
"""

import numpy as np
import pytest
import torch

from oracle import moe, mx
from mxfp8_block_scaled_moe_gb300 import workloads

from _util import OUT_REL_FROB, TOPK_W_RTOL, bits16, finalize_bound_ok, rel_frob, to_bf16_tensor, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mm():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import mxfp8_block_scaled_moe_gb300 as m
    return m


DEV = "cuda"


def _special_rows(rng, K):
    """Rows exercising zero blocks, subnormal amax, huge values, ties and -0."""
    rows = [np.zeros(K), rng.normal(0, 1, K) * 2.0 ** -130, rng.normal(0, 1, K) * 2.0 ** 120,
            np.full(K, -0.0), rng.normal(0, 1, K)]
    tie = np.zeros(K)
    tie[:5] = [1.0, 1.0625, 1.1875, 1.171875, -1.0625]
    rows.append(tie)
    sat = np.zeros(K)
    sat[:3] = [1.9375, 1.796875, -1.9375]
    rows.append(sat)
    under = np.full(K, -2.0 ** -18)
    under[0] = 1.0
    rows.append(under)
    return np.stack(rows)


@pytest.mark.parametrize("E,N,K", [(1, 1, 32), (3, 5, 96), (8, 256, 256), (8, 256, 128),
                                   (2, 37, 2048)])
def test_mx_quantize_3d_bit_exact(mm, E, N, K):
    rng = np.random.default_rng(E * 1000 + N + K)
    x = rng.standard_t(4, (E, N, K)) * np.exp2(rng.integers(-30, 30, (E, N, 1)))
    sp = _special_rows(rng, K)
    n = min(N, sp.shape[0])
    x[0, :n] = sp[:n]
    xb = mx.f64_to_bf16_bits(x)
    q, s = mm.mx_quantize_3d(to_bf16_tensor(xb, DEV))
    torch.cuda.synchronize()
    qr, sr = mx.mx_quantize(mx.bf16_bits_to_f64(xb))
    assert np.array_equal(u8(s), sr)
    assert np.array_equal(u8(q), qr)


def _offset16(t):
    """A copy of t whose data starts 16 bytes past a 32-byte boundary."""
    flat = torch.empty(t.numel() * t.element_size() + 48, dtype=torch.uint8, device=t.device)
    base = (-flat.data_ptr()) % 32 + 16
    v = flat[base:base + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 32 == 16
    return v


def test_mx_quantize_16_byte_aligned_input(mm):
    """A 16-byte (not 32-byte) aligned input takes the 16-byte load path."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 40, 256)) * np.exp2(rng.integers(-8, 8, (3, 40, 1)))
    xb = mx.f64_to_bf16_bits(x)
    q, s = mm.mx_quantize_3d(_offset16(to_bf16_tensor(xb, DEV)))
    torch.cuda.synchronize()
    qr, sr = mx.mx_quantize(mx.bf16_bits_to_f64(xb))
    assert np.array_equal(u8(s), sr) and np.array_equal(u8(q), qr)


@pytest.mark.parametrize("cfg", ["tiny", "qwen3_30b_decode"])
def test_weight_quant_of_config_bit_exact(mm, cfg):
    shape = workloads.CONFIGS[cfg]
    w13, w2 = workloads.make_weights_bf16(shape, DEV)
    for w in (w13, w2):
        q, s = mm.mx_quantize_3d(w)
        torch.cuda.synchronize()
        experts = range(w.shape[0]) if w.shape[0] <= 8 else [0, 17, 63, w.shape[0] - 1]
        for e in experts:
            qr, sr = mx.mx_quantize(mx.bf16_bits_to_f64(bits16(w[e])))
            assert np.array_equal(u8(s[e]), sr)
            assert np.array_equal(u8(q[e]), qr)


def _check_route(r, x_bits, logits, k, E, renorm=True):
    ids, w = moe.route_topk(logits, k, renorm)
    assert np.array_equal(r["topk_ids"].cpu().numpy(), ids)
    wg = r["topk_w"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(wg - w) / np.abs(w)) <= TOPK_W_RTOL
    counts, offsets, s2s, src2s = moe.permute(ids, E)
    assert np.array_equal(r["expert_counts"].cpu().numpy(), counts)
    assert np.array_equal(r["expert_offsets"].cpu().numpy(), offsets)
    assert np.array_equal(r["sorted_to_src"].cpu().numpy(), s2s)
    assert np.array_equal(r["src_to_sorted"].cpu().numpy(), src2s)
    return ids, s2s


@pytest.mark.parametrize("cfg", ["tiny", "qwen3_30b_decode", "qwen3_30b_prefill"])
def test_route_quant_bit_exact(mm, cfg):
    shape = workloads.CONFIGS[cfg]
    inp = workloads.make_layer(shape, DEV, weights=False)
    r = mm.moe_route_quant_mxfp8(inp["x"], inp["logits"], shape.k)
    torch.cuda.synchronize()
    xb = bits16(inp["x"])
    logits = inp["logits"].cpu().numpy()
    ids, s2s = _check_route(r, xb, logits, shape.k, shape.E)
    xq, xs, *_ = moe.route_quant(mx.bf16_bits_to_f64(xb), ids, shape.E)
    assert np.array_equal(u8(r["xs"]), xs)
    assert np.array_equal(u8(r["xq"]), xq)


@pytest.mark.parametrize("T", workloads.SKEW_SWEEP_T)
def test_route_quant_skewed_load(mm, T):
    shape = workloads.CONFIGS["qwen3_30b_skewed"].with_tokens(T)
    inp = workloads.make_layer(shape, DEV, weights=False)
    r = mm.moe_route_quant_mxfp8(inp["x"], inp["logits"], shape.k)
    torch.cuda.synchronize()
    xb = bits16(inp["x"])
    ids, s2s = _check_route(r, xb, inp["logits"].cpu().numpy(), shape.k, shape.E)
    counts = r["expert_counts"].cpu().numpy()
    if T == 16384:
        assert (counts == 0).sum() >= 4
        assert counts.max() > 0.10 * shape.M
    xq, xs, *_ = moe.route_quant(mx.bf16_bits_to_f64(xb), ids, shape.E)
    assert np.array_equal(u8(r["xq"]), xq) and np.array_equal(u8(r["xs"]), xs)


@pytest.mark.parametrize("T,H,E,k,renorm", [(1, 32, 1, 1, True), (65, 96, 5, 3, False),
                                             (130, 512, 40, 8, True), (7, 2048, 128, 8, False),
                                             (300, 64, 256, 32, True), (64, 256, 8, 8, True),
                                             (200, 64, 600, 32, True), (130, 96, 1000, 4, False),
                                             (70, 64, 1024, 8, True), (20001, 64, 128, 8, True),
                                             (9800, 32, 256, 6, False), (9, 4096, 256, 8, True),
                                             (17, 96, 64, 6, False), (33, 2048, 200, 8, True),
                                             (57, 128, 160, 4, True), (40, 64, 300, 8, True),
                                             (64, 96, 1024, 2, False)])
def test_route_quant_edge_shapes(mm, T, H, E, k, renorm):
    """Odd E, E up to 256 at 313 routing blocks with a ragged last one (20001
    tokens) and at 154 (9800), wide E (8+ logits per lane), ties; the
    single-cluster small-batch path at 1, 7, 9, 17, 33, 57 and 64 tokens (one
    to eight tokens per CTA, one to eight CTAs, rows of 1 to 4 chunks); one
    routing block through the three-kernel path (E above the cluster path's
    256: the scan's row and totals CTAs over a single block)."""
    g = torch.Generator(device=DEV).manual_seed(T * 7 + E)
    x = torch.randn(T, H, generator=g, device=DEV).to(torch.bfloat16)
    logits = torch.randn(T, E, generator=g, device=DEV)
    if E >= 8:  # exact ties in the logits: lower expert id wins
        logits[:, 3] = logits[:, 5]
    r = mm.moe_route_quant_mxfp8(x, logits, k, renorm)
    torch.cuda.synchronize()
    xb = bits16(x)
    ids, s2s = _check_route(r, xb, logits.cpu().numpy(), k, E, renorm)
    xq, xs, *_ = moe.route_quant(mx.bf16_bits_to_f64(xb), ids, E)
    assert np.array_equal(u8(r["xq"]), xq) and np.array_equal(u8(r["xs"]), xs)


@pytest.mark.parametrize("quant", [True, False])
def test_route_16_byte_aligned_input(mm, quant):
    """x 16-byte (not 32-byte) aligned: the permutation takes 16-byte accesses."""
    g = torch.Generator(device=DEV).manual_seed(99)
    T, H, E, k = 77, 1024, 16, 4
    x = _offset16(torch.randn(T, H, generator=g, device=DEV).to(torch.bfloat16))
    logits = torch.randn(T, E, generator=g, device=DEV)
    xb = bits16(x)
    if quant:
        r = mm.moe_route_quant_mxfp8(x, logits, k)
        torch.cuda.synchronize()
        ids, _ = _check_route(r, xb, logits.cpu().numpy(), k, E, True)
        xq, xs, *_ = moe.route_quant(mx.bf16_bits_to_f64(xb), ids, E)
        assert np.array_equal(u8(r["xq"]), xq) and np.array_equal(u8(r["xs"]), xs)
    else:
        r = mm.moe_route_permute_bf16(x, logits, k)
        torch.cuda.synchronize()
        ref = moe.permute_rows(xb, r["sorted_to_src"].cpu().numpy(), k)
        assert np.array_equal(bits16(r["xp"]), ref)


def test_route_logits_not_16_byte_aligned_is_rejected(mm):
    """Every input pointer of the routing call must be 16-byte aligned: logits
    at a 4-byte aligned address return MXMOE_ERR_ALIGN before any launch."""
    from mxfp8_block_scaled_moe_gb300._lib import MXMoEError
    T, H, E, k = 100, 128, 128, 8
    x = torch.zeros(T, H, dtype=torch.bfloat16, device=DEV)
    logits = torch.zeros(T * E + 1, device=DEV)[1:].view(T, E)
    assert logits.data_ptr() % 16 == 4
    with pytest.raises(MXMoEError, match="MXMOE_ERR_ALIGN"):
        mm.moe_route_quant_mxfp8(x, logits, k)
    torch.cuda.synchronize()
    assert mm.device_status() == 0


def test_route_empty_batch(mm):
    x = torch.zeros(0, 256, dtype=torch.bfloat16, device=DEV)
    logits = torch.zeros(0, 8, device=DEV)
    r = mm.moe_route_quant_mxfp8(x, logits, 2)
    torch.cuda.synchronize()
    assert r["expert_offsets"].cpu().tolist() == [0] * 9
    assert r["expert_counts"].cpu().tolist() == [0] * 8


@pytest.mark.parametrize("cfg", ["tiny", "qwen3_30b_prefill"])
def test_fused_route_quant_equals_two_step(mm, cfg):
    """quant_mode=3 output is byte-identical to bf16 permute + separate quant."""
    shape = workloads.CONFIGS[cfg]
    inp = workloads.make_layer(shape, DEV, weights=False)
    fused = mm.moe_route_quant_mxfp8(inp["x"], inp["logits"], shape.k)
    two = mm.moe_route_permute_bf16(inp["x"], inp["logits"], shape.k)
    q2, s2 = mm.mx_quantize_3d(two["xp"])
    torch.cuda.synchronize()
    assert torch.equal(fused["sorted_to_src"], two["sorted_to_src"])
    assert torch.equal(fused["xq"], q2) and torch.equal(fused["xs"], s2)
    # the bf16 permute itself is exact
    xp_ref = moe.permute_rows(bits16(inp["x"]), two["sorted_to_src"].cpu().numpy(), shape.k)
    assert np.array_equal(bits16(two["xp"]), xp_ref)


def test_route_is_deterministic(mm):
    shape = workloads.CONFIGS["qwen3_30b_prefill"]
    inp = workloads.make_layer(shape, DEV, weights=False)
    a = mm.moe_route_quant_mxfp8(inp["x"], inp["logits"], shape.k)
    b = mm.moe_route_quant_mxfp8(inp["x"], inp["logits"], shape.k)
    torch.cuda.synchronize()
    for key in a:
        assert torch.equal(a[key], b[key]), key


# ---------------------------------------------------------------- finalize

# 1040 = 1024 + 16: a second column chunk holding one lane; 600 and 40 are not
# multiples of 16 (8-column lanes); offset16 takes the 16-byte access path.
@pytest.mark.parametrize("T,H,k,off", [(64, 256, 2, False), (32, 2048, 8, False),
                                       (1000, 2048, 8, False), (5, 40, 3, False),
                                       (17, 1040, 4, False), (9, 600, 5, False),
                                       (33, 2048, 8, True), (17, 1040, 4, True)])
def test_finalize_matches_oracle(mm, T, H, k, off):
    g = torch.Generator(device=DEV).manual_seed(T + H + k)
    y = torch.randn(T * k, H, generator=g, device=DEV).to(torch.bfloat16)
    if off:
        y = _offset16(y)
    w = torch.rand(T, k, generator=g, device=DEV)
    perm = torch.randperm(T * k, generator=g, device=DEV).to(torch.int32)
    out = mm.moe_finalize_routing(y, w, perm, k)
    torch.cuda.synchronize()
    ref = moe.finalize(bits16(y), w.cpu().numpy(), perm.cpu().numpy(), k)
    assert rel_frob(bits16(out), ref) <= OUT_REL_FROB
    assert finalize_bound_ok(bits16(out), bits16(y), w.cpu().numpy(), perm.cpu().numpy(), k) == 0.0


def test_identity_layer_route_finalize(mm):
    """k=1, weights 1, identity expert: finalize(permute(x)) == x bit-exact."""
    g = torch.Generator(device=DEV).manual_seed(11)
    T, H, E = 513, 256, 16
    x = torch.randn(T, H, generator=g, device=DEV).to(torch.bfloat16)
    logits = torch.randn(T, E, generator=g, device=DEV)
    r = mm.moe_route_permute_bf16(x, logits, 1)
    assert torch.all(r["topk_w"] == 1.0)
    out = mm.moe_finalize_routing(r["xp"], r["topk_w"], r["src_to_sorted"], 1)
    torch.cuda.synchronize()
    assert torch.equal(out, x)
