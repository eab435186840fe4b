"""Pins of the oracle's FP8 and NVFP4 weight formats (rlx-cpu 0.2.13,
src/thunk/ops/quant.rs: fp8_e4m3_to_f32, fp8_e5m2_to_f32, dequant_matmul_fp8,
dequant_matmul_nvfp4).

Decoders are checked against torch's own float8 types, an independent
implementation:
  * e5m2 as the page defines it is IEEE style, exactly torch.float8_e5m2;
  * e4m3 as the page defines it equals torch.float8_e4m3fn on every code
    whose exponent is below 15; exponent 15 is +-infinity (mantissa 0) or
    NaN, the page's rule, where the OCP "fn" format has finite values;
  * the NVFP4 block scale (OCP E4M3) equals torch.float8_e4m3fn on all codes;
  * every FP4 E2M1 value equals the E4M3 value of the code with the same sign
    and mantissa and the exponent moved from bias 1 to bias 7.
The products are checked on one-hot rows (each output is one decoded weight
times its scale), against numpy products of independently decoded weights,
and on a hand-worked NVFP4 example of the page's nibble and scale indexing.
"""
import numpy as np
import pytest
import torch

import oracle

CODES = np.arange(256)


def _torch_decode(codes, dt):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(dt).float().numpy()


def _same(a, b):
    return (a == b) | (np.isnan(a) & np.isnan(b))


def test_e5m2_is_ieee_style_on_every_code():
    assert _same(oracle.fp8_decode(CODES, e5m2=True), _torch_decode(CODES, torch.float8_e5m2)).all()


def test_e4m3_matches_ocp_below_the_top_exponent_and_is_inf_nan_at_it():
    got = oracle.fp8_decode(CODES)
    ref = _torch_decode(CODES, torch.float8_e4m3fn)
    top = ((CODES >> 3) & 0xF) == 15
    assert _same(got[~top], ref[~top]).all()
    assert got[0x78] == np.inf and got[0xF8] == -np.inf
    assert np.isnan(got[top & ((CODES & 7) != 0)]).all()
    # a few values of the page's formula worked by hand: 1.0, 2.0, the smallest subnormal, -1.5
    assert got[0x38] == 1.0 and got[0x40] == 2.0 and got[0x01] == 2.0 ** -9 and got[0xBC] == -1.5


def test_nvfp4_scale_is_ocp_e4m3():
    assert _same(oracle.e4m3fn_scale(CODES), _torch_decode(CODES, torch.float8_e4m3fn)).all()


def test_e2m1_equals_e4m3_with_the_exponent_rebiased():
    nib = np.arange(16)
    s, e, m = nib >> 3, (nib >> 1) & 3, nib & 1
    # normal E2M1 (e > 0): 2^(e-1) (1 + m/2) is E4M3 with exponent field e + 6 and mantissa m << 2;
    # subnormal E2M1 (e = 0): m * 0.5 is E4M3 0.5 (exponent field 6) or zero
    e4 = np.where(e > 0, e + 6, np.where(m == 1, 6, 0))
    m4 = np.where(e > 0, m << 2, 0)
    mapped = (s << 7) | (e4 << 3) | m4
    assert np.array_equal(oracle.e2m1(nib), _torch_decode(mapped, torch.float8_e4m3fn))


def _finite_fp8(rng, shape, e5m2):
    top = 31 if e5m2 else 15
    shift = 2 if e5m2 else 3
    c = rng.integers(0, 256, size=shape)
    bad = ((c >> shift) & top) == top
    c[bad] &= ~(1 << (shift + 1))  # clear one exponent bit: never the all-ones exponent
    return c.astype(np.uint8)


@pytest.mark.parametrize("e5m2", [False, True])
def test_fp8_one_hot_rows_pick_one_scaled_weight(e5m2):
    rng = np.random.default_rng(11)
    K, N = 24, 10
    w8 = _finite_fp8(rng, (K, N), e5m2)
    s = rng.uniform(0.5, 2.0, N).astype(np.float32)
    y, _ = oracle.matmul_fp8(np.eye(K), w8, s, K, N, e5m2=e5m2)
    dec = _torch_decode(w8, torch.float8_e5m2 if e5m2 else torch.float8_e4m3fn).astype(np.float64)
    assert np.array_equal(y, dec * s.astype(np.float64)[None, :])
    y1, _ = oracle.matmul_fp8(np.eye(K), w8, None, K, N, e5m2=e5m2)  # no scales: 1.0
    assert np.array_equal(y1, dec)


@pytest.mark.parametrize("e5m2", [False, True])
def test_fp8_product_equals_numpy_on_decoded_weights(e5m2):
    rng = np.random.default_rng(12)
    M, K, N = 3, 100, 17
    x = rng.standard_normal((M, K))
    w8 = _finite_fp8(rng, (K, N), e5m2)
    s = rng.uniform(0.01, 0.1, N).astype(np.float32)
    y, mag = oracle.matmul_fp8(x, w8, s, K, N, e5m2=e5m2)
    W = _torch_decode(w8, torch.float8_e5m2 if e5m2 else torch.float8_e4m3fn).astype(np.float64)
    ref = x @ (W * s.astype(np.float64)[None, :])
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12 * np.abs(mag).max())
    np.testing.assert_allclose(mag, np.abs(x) @ np.abs(W * s.astype(np.float64)[None, :]), rtol=1e-12)


def test_fp8_infinite_weight_propagates():
    w8 = np.array([[0x38], [0x78]], dtype=np.uint8)  # 1.0, then +inf (the page's exponent-15 rule)
    y, _ = oracle.matmul_fp8(np.array([[1.0, 2.0]]), w8, None, 2, 1)
    assert y[0, 0] == np.inf


def test_nvfp4_hand_worked_indexing():
    # K = 16 (one scale block), N = 2: flat index f = 2p + j, so byte p holds (p, 0) in its low nibble and
    # (p, 1) in its high nibble.  Byte 0x21: w(0, 0) = e2m1(1) = 0.5, w(0, 1) = e2m1(2) = 1.0.  Block scales
    # 0x38 = 1.0 (column 0) and 0x40 = 2.0 (column 1); global scale 0.5.  A one-hot row on p = 0 gives
    # [0.5 * 1.0 * 0.5, 1.0 * 2.0 * 0.5] = [0.25, 1.0].
    K, N = 16, 2
    w4 = np.zeros(K * N // 2, dtype=np.uint8)
    w4[0] = 0x21
    scale8 = np.array([[0x38, 0x40]], dtype=np.uint8)
    x = np.zeros((1, K))
    x[0, 0] = 1.0
    y, _ = oracle.matmul_nvfp4(x, w4, scale8, 0.5, K, N)
    assert np.array_equal(y, np.array([[0.25, 1.0]]))


@pytest.mark.parametrize("K,N", [(32, 6), (40, 5)])  # 40: a partial last scale block; N odd: bytes straddle rows
def test_nvfp4_weights_and_product_against_independent_decoding(K, N):
    rng = np.random.default_rng(13)
    w4 = rng.integers(0, 256, size=(K * N + 1) // 2, dtype=np.uint8)
    scale8 = rng.integers(0x20, 0x50, size=(-(-K // 16), N), dtype=np.uint8)  # positive, finite scales
    g = np.float32(0.75)
    nib = np.stack([w4 & 0x0F, w4 >> 4], axis=1).reshape(-1)[:K * N].reshape(K, N)
    s_, e_, m_ = nib >> 3, (nib >> 1) & 3, nib & 1
    mapped = (s_ << 7) | (np.where(e_ > 0, e_ + 6, np.where(m_ == 1, 6, 0)) << 3) | np.where(e_ > 0, m_ << 2, 0)
    fp4 = _torch_decode(mapped, torch.float8_e4m3fn)
    sc = _torch_decode(scale8, torch.float8_e4m3fn)[np.arange(K) // 16]
    W = (fp4 * sc).astype(np.float32) * g  # in f32, in the page's order
    assert np.array_equal(oracle.nvfp4_weights(w4, scale8, g, K, N), W)
    x = rng.standard_normal((2, K))
    y, _ = oracle.matmul_nvfp4(x, w4, scale8, g, K, N)
    np.testing.assert_allclose(y, x @ W.astype(np.float64), rtol=0, atol=1e-12 * np.abs(x).sum())
