"""Pins for the oracle's dense MXFP8 linear (CPU only).

Each check ties ``oracle.linear`` to something other than itself:

* inputs that MX-quantize losslessly make the linear the plain fp64 matmul
  of the inputs (numpy's, a library routine), partial last block included;
* a partial last block of 16 gives the same bytes and product as the same
  row padded with 16 zeros to a whole block (the amax of a block is not
  changed by zeros), so the partial-block rule is pinned by the full-block
  one;
* a tiny case rebuilt by brute force: scales from the binary exponent of
  the amax, elements by exhaustive nearest-value search over the e4m3 grid
  built from its bit fields (ties to the even code), exact rational sums;
* the pages' K = 4304 example: 135 scales per row, 68 pairs after padding;
* with one group the linear equals the grouped GEMM2 of the MoE oracle;
* W4A4: MXFP4-lossless inputs give the exact matmul, and the W4A4 linear is
  the (pinned) MXFP8 linear fed the same values as e4m3 codes.
"""

from fractions import Fraction
import math

import numpy as np
import pytest
import torch

from oracle import linear, moe, mx


def _bf16_bits(v: np.ndarray) -> np.ndarray:
    """float64 values exactly representable in bf16 -> bf16 bit patterns (via torch)."""
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float64)).to(torch.bfloat16)
    assert torch.equal(t.to(torch.float64), torch.from_numpy(np.asarray(v, dtype=np.float64)))
    return t.view(torch.int16).numpy().view(np.uint16)


def _lossless_rows(rng, rows, K):
    """Rows whose every block (partial last one included) has amax 256 * 2^s
    and integer multiples of 2^s elsewhere: the MX quant is exact."""
    x = rng.integers(-16, 17, (rows, K)).astype(np.float64)
    nb = -(-K // 32)
    s = rng.integers(-3, 4, (rows, nb))
    for r in range(rows):
        for j in range(nb):
            lo, hi = 32 * j, min(K, 32 * j + 32)
            pos = lo + int(rng.integers(0, hi - lo))
            x[r, pos] = 256.0 * (1 if rng.random() < 0.5 else -1)
            x[r, lo:hi] *= 2.0 ** s[r, j]
    return x


@pytest.mark.parametrize("M,N,K", [(7, 5, 80), (3, 9, 64), (4, 3, 16), (2, 6, 208)])
def test_lossless_inputs_give_the_exact_matmul(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    x = _lossless_rows(rng, M, K)
    w = _lossless_rows(rng, N, K) / 64.0
    wq, ws = mx.mx_quantize(w)
    assert ws.shape == (N, math.ceil(K / 32))
    assert np.array_equal(mx.mx_dequantize(wq, ws), w)
    got = linear.mxfp8_linear(_bf16_bits(x), wq, ws, round_bf16=False)
    assert np.array_equal(got, x @ w.T)


@pytest.mark.parametrize("K", [16, 48, 80, 336, 4304])
def test_partial_block_equals_zero_padded_block(K):
    assert K % 32 == 16
    rng = np.random.default_rng(K)
    M, N = 6, 5
    xb = _bf16_bits(torch.randn(M, K, dtype=torch.float64).to(torch.bfloat16).double().numpy())
    w = rng.normal(0, 0.02, (N, K))
    wq, ws = mx.mx_quantize(w)
    wq_p, ws_p = mx.mx_quantize(np.concatenate([w, np.zeros((N, 16))], axis=1))
    assert np.array_equal(wq_p[:, :K], wq) and np.array_equal(ws_p, ws)
    assert np.all(wq_p[:, K:] == 0)
    xb_p = np.concatenate([xb, np.zeros((M, 16), np.uint16)], axis=1)
    xq, xs = linear.quantize_activations(xb)
    xq_p, xs_p = linear.quantize_activations(xb_p)
    assert np.array_equal(xq_p[:, :K], xq) and np.array_equal(xs_p, xs)
    assert np.array_equal(linear.mxfp8_linear(xb, wq, ws), linear.mxfp8_linear(xb_p, wq_p, ws_p))


def _e4m3_grid():
    """(code, value) for every finite e4m3fn code, from the bit fields:
    sign | 4 exponent bits (bias 7) | 3 mantissa bits; exponent 0 is
    subnormal; S.1111.111 is NaN."""
    out = []
    for c in range(256):
        sgn, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue
        v = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        out.append((c, -v if sgn else v))
    return out


def _brute_quant_row(vals):
    grid = _e4m3_grid()
    codes, scales = [], []
    for j in range(0, len(vals), 32):
        blk = [Fraction(v) for v in vals[j:j + 32]]
        amax = max(abs(v) for v in blk)
        if amax == 0:
            s = -127
        else:
            s = math.frexp(float(amax))[1] - 1 - 8
        scales.append(s)
        for v in blk:
            t = v / Fraction(2) ** s
            t = max(min(t, Fraction(448)), Fraction(-448))
            best = min(abs(t - g) for _, g in grid)
            cands = [c for c, g in grid if abs(t - g) == best]
            even = [c for c in cands if c & 1 == 0]
            c = (even or cands)[0]
            codes.append(dict(grid)[c])
    return codes, scales


def test_tiny_linear_by_brute_force():
    M, N, K = 2, 3, 48
    x = torch.randn(M, K, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    w = torch.randn(N, K, generator=torch.Generator().manual_seed(8)).double().numpy() * 0.05
    xb = x.view(torch.int16).numpy().view(np.uint16)
    xv = x.double().numpy()
    wq, ws = mx.mx_quantize(w)
    got = linear.mxfp8_linear(xb, wq, ws, round_bf16=False)
    for n in range(N):
        wc, wsc = _brute_quant_row(list(w[n]))
        assert [int(b) - 127 for b in ws[n]] == wsc
        for m in range(M):
            xc, xsc = _brute_quant_row(list(xv[m]))
            acc = Fraction(0)
            for k in range(K):
                acc += (xc[k] * Fraction(2) ** xsc[k // 32]) * (wc[k] * Fraction(2) ** wsc[k // 32])
            assert Fraction(got[m, n]) == acc


def test_k4304_scale_count_and_pairs():
    w = np.random.default_rng(1).normal(0, 0.02, (3, 4304))
    _, ws = mx.mx_quantize(w)
    assert ws.shape == (3, 135)
    assert mx.pair_split_scales(ws).shape == (3, 68, 2)


def test_linear_equals_one_group_gmm2():
    rng = np.random.default_rng(5)
    M, N, K = 37, 24, 96
    xb = _bf16_bits(torch.randn(M, K, dtype=torch.float64).to(torch.bfloat16).double().numpy())
    wq, ws = mx.mx_quantize(rng.normal(0, 0.02, (N, K)))
    xq, xs = linear.quantize_activations(xb)
    ref = moe.gmm2(xq, xs, wq[None], ws[None], np.array([0, M]))
    assert np.array_equal(linear.mxfp8_linear(xb, wq, ws), ref)


def _lossless_fp4_rows(rng, rows, K):
    """Rows that MXFP4-quantize exactly: per block one element +-4 * 2^s (it
    fixes the scale at 2^s) and e2m1 grid values * 2^s elsewhere."""
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    x = grid[rng.integers(0, 8, (rows, K))] * np.where(rng.random((rows, K)) < 0.5, -1, 1)
    nb = K // 32
    s = rng.integers(-3, 4, (rows, nb))
    pos = rng.integers(0, 32, (rows, nb))
    for j in range(nb):
        x[np.arange(rows), 32 * j + pos[:, j]] = 4.0 * np.where(rng.random(rows) < 0.5, -1, 1)
    return x * np.exp2(np.repeat(s, 32, axis=1))


@pytest.mark.parametrize("M,N,K", [(5, 3, 64), (2, 7, 32), (4, 4, 160)])
def test_w4a4_lossless_inputs_give_the_exact_matmul(M, N, K):
    rng = np.random.default_rng(M * 31 + N + K)
    x = _lossless_fp4_rows(rng, M, K)
    w = _lossless_fp4_rows(rng, N, K) / 8.0
    wp, ws = mx.mxfp4_quantize(w)
    assert np.array_equal(mx.mxfp4_dequantize(wp, ws), w)
    got = linear.mxfp4_linear(_bf16_bits(x), wp, ws, round_bf16=False)
    assert np.array_equal(got, x @ w.T)


def test_w4a4_linear_equals_mxfp8_linear_on_reencoded_values():
    rng = np.random.default_rng(9)
    M, N, K = 9, 12, 96
    xb = _bf16_bits(torch.randn(M, K, dtype=torch.float64).to(torch.bfloat16).double().numpy())
    wp, ws = mx.mxfp4_quantize(rng.normal(0, 0.02, (N, K)))
    xp, xs = linear.quantize_activations(xb, "e2m1")
    assert xp.shape == (M, K // 2)
    e8 = lambda q: mx.e4m3_encode(mx.e2m1_decode(mx.unpack_fp4(q)))
    assert np.array_equal(linear.mxfp4_linear(xb, wp, ws), linear.linear(e8(xp), xs, e8(wp), ws))
