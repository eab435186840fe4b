"""Pins for the CPU oracle: hand-worked values, closed forms, invariants and
exact brute force.  None of these re-types the oracle's own formula: the
brute force decodes through a bit string and sums in exact rationals.

Sources: onnx-runtime-ep-cpu 0.1.0-dev.5, src/kernels/matmul_nbits.rs
(module doc, fn dequantize_nbits_value, MatMulNBitsKernel::execute,
fn quantize_activation_signed, fn int4_dot_row_scalar, fn int8_row);
rlx-cpu 0.2.13, src/thunk/ops/quant.rs (fn dequant_matmul_int4).
"""
from fractions import Fraction

import numpy as np
import pytest

from block_quantized_weight_matmulnbits_gb300 import workloads as wl
from tests._golden import pack_codes_test, pack_matrix_test, pack_zp_test, rows


# ---- hand-worked fixtures -------------------------------------------------

def test_codes_lsb_first_golden(oracle_mod):
    for bits, hexbytes, *codes in rows("codes_lsb_first.txt"):
        bits = int(bits)
        blob = np.frombuffer(bytes.fromhex(hexbytes), dtype=np.uint8)
        bs = len(blob) * 8 // bits
        b = blob.reshape(1, 1, -1)
        got = [oracle_mod.code(b, 1, bs, bits, bs, 0, k) for k in range(bs)]
        assert got == [int(c) for c in codes], (bits, hexbytes)


def test_zero_points_golden(oracle_mod):
    for bits, hexbytes, *zps in rows("zero_points.txt"):
        bits = int(bits)
        nblk = len(zps)
        bs = 16
        K = nblk * bs
        zp = None if hexbytes == "none" else np.frombuffer(bytes.fromhex(hexbytes), np.uint8).reshape(1, -1)
        got = [oracle_mod.zero_point(zp, 1, K, bits, bs, 0, g) for g in range(nblk)]
        assert got == [int(z) for z in zps], (bits, hexbytes)


def test_dequant_values_golden(oracle_mod):
    for q, zp, s, exp in rows("dequant_values.txt"):
        q, zp, s, exp = int(q), int(zp), float(s), float(exp)
        bits = 8 if max(q, zp) > 15 else 4
        bs = 16
        codes = [q] * bs
        b = pack_codes_test(codes, bits).reshape(1, 1, -1)
        z = pack_zp_test(np.array([[zp]]), bits)
        w = oracle_mod.dequantize(b, np.array([[s]], np.float32), z, 1, bs, bits, bs)
        assert np.all(w == np.float32(exp)), (q, zp, s, w[0, :4])


def _case(case):
    if case == "A":
        bits, bs, K = 4, 16, 16
        b = np.full((1, 1, 8), 0x98, np.uint8)
        return bits, bs, K, b, np.array([[0.5]], np.float32), None, np.arange(16, dtype=np.float64)
    if case == "B":
        bits, bs, K = 2, 16, 16
        b = np.full((1, 1, 4), 0xE4, np.uint8)
        return bits, bs, K, b, np.array([[0.25]], np.float32), np.array([[0x01]], np.uint8), np.ones(16)
    if case == "C":
        bits, bs, K = 8, 16, 20
        b = np.full((1, 2, 16), 0xFF, np.uint8)
        for k in range(20):
            b[0, k // 16, k % 16] = 100 + k
        return (bits, bs, K, b, np.array([[1.0, 2.0]], np.float32),
                np.array([[110, 120]], np.uint8), np.ones(20))
    raise ValueError(case)


def test_tiny_matmul_golden(oracle_mod):
    for case, bits, bs, K, exp in rows("tiny_matmul.txt"):
        cb, cbs, cK, b, s, zp, x = _case(case)
        assert (cb, cbs, cK) == (int(bits), int(bs), int(K))
        y, _ = oracle_mod.matmul(x.reshape(1, -1), b, s, zp, 1, cK, cb, cbs)
        assert y[0, 0] == float(exp), (case, y[0, 0])


# ---- exact brute force through an independent decoder ---------------------

def _bitstring_codes(b, N, K, bits, bs):
    """Decode by spelling each blob as a bit string, least significant bit of
    each byte first, and reading consecutive `bits`-wide fields."""
    kb = -(-K // bs)
    q = np.zeros((N, K), dtype=np.int64)
    for n in range(N):
        for blk in range(kb):
            s = "".join(format(int(byte), "08b")[::-1] for byte in b[n, blk])
            for i in range(bs):
                k = blk * bs + i
                if k < K:
                    q[n, k] = int(s[i * bits:(i + 1) * bits][::-1], 2)
    return q


def _bitstring_zps(zp, N, kb, bits):
    if zp is None:
        return np.full((N, kb), 1 << (bits - 1), dtype=np.int64)
    z = np.zeros((N, kb), dtype=np.int64)
    for n in range(N):
        s = "".join(format(int(byte), "08b")[::-1] for byte in zp[n])
        for g in range(kb):
            z[n, g] = int(s[g * bits:(g + 1) * bits][::-1], 2)
    return z


@pytest.mark.parametrize("bits,bs,K,N,M,asym", [
    (4, 16, 40, 3, 2, True), (4, 32, 64, 2, 1, False), (2, 16, 37, 3, 2, True),
    (2, 64, 64, 2, 1, True), (8, 16, 33, 2, 3, True), (8, 32, 32, 3, 1, False),
])
def test_bruteforce_exact_rationals(oracle_mod, bits, bs, K, N, M, asym):
    rng = np.random.default_rng(1000 + bits * 100 + K)
    kb = -(-K // bs)
    b = rng.integers(0, 256, size=(N, kb, bs * bits // 8), dtype=np.uint8)
    zp = rng.integers(0, 256, size=(N, -(-kb * bits // 8)), dtype=np.uint8) if asym else None
    s = rng.uniform(0.01, 0.1, (N, kb)).astype(np.float32)
    x = wl.widen_f64(wl.to_storage(rng.standard_normal((M, K)), wl.BF16), wl.BF16)
    q = _bitstring_codes(b, N, K, bits, bs)
    z = _bitstring_zps(zp, N, kb, bits)
    # weights: exact rational (q - z) * s, then one rounding to f32
    w_exact = np.zeros((N, K), dtype=np.float32)
    for n in range(N):
        for k in range(K):
            w_exact[n, k] = np.float32(float(Fraction(int(q[n, k] - z[n, k // bs])) * Fraction(float(s[n, k // bs]))))
    w = oracle_mod.dequantize(b, s, zp, N, K, bits, bs)
    assert np.array_equal(w.view(np.uint32), w_exact.view(np.uint32))
    y, mag = oracle_mod.matmul(x, b, s, zp, N, K, bits, bs)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(x[m, k])) * Fraction(float(w_exact[n, k])) for k in range(K))
            # f64 accumulation of K products: |err| <= K * 2^-53 * sum|x w|
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(K + 1) * Fraction(2) ** -52 * Fraction(mag[m, n])


# ---- invariants and special cases -----------------------------------------

def _random(bits, bs, K, N, M, asym=True, seed=7):
    rng = np.random.default_rng(seed)
    kb = -(-K // bs)
    b = rng.integers(0, 256, size=(N, kb, bs * bits // 8), dtype=np.uint8)
    zp = rng.integers(0, 256, size=(N, -(-kb * bits // 8)), dtype=np.uint8) if asym else None
    s = rng.uniform(0.01, 0.1, (N, kb)).astype(np.float32)
    x = rng.standard_normal((M, K))
    return b, s, zp, x


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_all_codes_equal_zero_point_gives_zero(oracle_mod, bits):
    bs, K, N = 32, 96, 4
    rng = np.random.default_rng(bits)
    kb = K // bs
    z = rng.integers(0, 1 << bits, size=(N, kb))
    q = np.repeat(z, bs, axis=1)
    b = pack_matrix_test(q, bits, bs)
    zp = pack_zp_test(z, bits)
    s = rng.uniform(0.01, 0.1, (N, kb)).astype(np.float32)
    y, _ = oracle_mod.matmul(rng.standard_normal((3, K)), b, s, zp, N, K, bits, bs)
    assert np.all(y == 0.0)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_one_hot_row_selects_dequantized_column(oracle_mod, bits):
    bs, K, N = 16, 48, 5
    b, s, zp, _ = _random(bits, bs, K, N, 1, seed=bits + 11)
    w = oracle_mod.dequantize(b, s, zp, N, K, bits, bs)
    x = np.eye(K)[[0, 17, 47]]
    y, _ = oracle_mod.matmul(x, b, s, zp, N, K, bits, bs)
    assert np.array_equal(y, w[:, [0, 17, 47]].T.astype(np.float64))


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_exact_scaling_by_two(oracle_mod, bits):
    b, s, zp, x = _random(bits, 32, 128, 6, 2, seed=bits + 21)
    y1, _ = oracle_mod.matmul(x, b, s, zp, 6, 128, bits, 32)
    y2, _ = oracle_mod.matmul(x, b, s * np.float32(2), zp, 6, 128, bits, 32)
    assert np.array_equal(y2, 2.0 * y1)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_absent_zero_points_equal_explicit_midpoint(oracle_mod, bits):
    bs, K, N = 16, 80, 3
    b, s, _, x = _random(bits, bs, K, N, 2, asym=False, seed=bits + 31)
    kb = K // bs
    zp = pack_zp_test(np.full((N, kb), 1 << (bits - 1)), bits)
    ya, _ = oracle_mod.matmul(x, b, s, None, N, K, bits, bs)
    yb, _ = oracle_mod.matmul(x, b, s, zp, N, K, bits, bs)
    assert np.array_equal(ya, yb)


def test_permuting_rows_of_b_permutes_columns_of_y(oracle_mod):
    bits, bs, K, N = 4, 32, 96, 7
    b, s, zp, x = _random(bits, bs, K, N, 3, seed=41)
    perm = np.random.default_rng(5).permutation(N)
    y, _ = oracle_mod.matmul(x, b, s, zp, N, K, bits, bs)
    yp, _ = oracle_mod.matmul(x, b[perm], s[perm], zp[perm], N, K, bits, bs)
    assert np.array_equal(yp, y[:, perm])


def test_linearity_in_x(oracle_mod):
    bits, bs, K, N = 4, 32, 128, 5
    b, s, zp, x1 = _random(bits, bs, K, N, 2, seed=51)
    x2 = np.random.default_rng(52).standard_normal((2, K))
    a = 0.75
    y1, m1 = oracle_mod.matmul(x1, b, s, zp, N, K, bits, bs)
    y2, m2 = oracle_mod.matmul(x2, b, s, zp, N, K, bits, bs)
    y3, m3 = oracle_mod.matmul(a * x1 + x2, b, s, zp, N, K, bits, bs)
    assert np.all(np.abs(y3 - (a * y1 + y2)) <= 1e-12 * (m1 + m2 + m3 + 1))


def test_padding_codes_past_k_are_ignored(oracle_mod):
    bits, bs, K, N = 4, 32, 70, 3   # KB = 3, last block holds 6 valid codes
    b, s, zp, x = _random(bits, bs, K, N, 2, seed=61)
    b2 = b.copy()
    b2[:, -1, 3:] ^= 0xFF           # flip codes 6.. of the last block
    ya, _ = oracle_mod.matmul(x, b, s, zp, N, K, bits, bs)
    yb, _ = oracle_mod.matmul(x, b2, s, zp, N, K, bits, bs)
    assert np.array_equal(ya, yb)


def test_g_idx_identity_equals_plain_blocks_and_bias_adds(oracle_mod):
    bits, bs, K, N = 4, 16, 64, 4
    b, s, zp, x = _random(bits, bs, K, N, 2, seed=71)
    g = (np.arange(K) // bs).astype(np.int32)
    ya, _ = oracle_mod.matmul(x, b, s, zp, N, K, bits, bs)
    yb, _ = oracle_mod.matmul(x, b, s, zp, N, K, bits, bs, g_idx=g)
    assert np.array_equal(ya, yb)
    bias = np.array([1.0, -2.0, 0.5, 0.0])
    yc, _ = oracle_mod.matmul(x, b, s, zp, N, K, bits, bs, bias_f64=bias)
    assert np.allclose(yc, ya + bias, rtol=0, atol=1e-12)


def test_g_idx_selects_scale_and_zero_point_column(oracle_mod):
    """With g_idx, depth k keeps its code (block k//bs) but takes scale and
    zero point from group g_idx[k]."""
    bits, bs, K, N = 4, 16, 32, 2
    b, s, zp, _ = _random(bits, bs, K, N, 1, seed=81)
    g = np.array([1] * 16 + [0] * 16, dtype=np.int32)
    w = oracle_mod.dequantize(b, s, zp, N, K, bits, bs, g_idx=g)
    q = _bitstring_codes(b, N, K, bits, bs)
    z = _bitstring_zps(zp, N, 2, bits)
    for n in range(N):
        for k in range(K):
            assert w[n, k] == np.float32(np.float32(q[n, k] - z[n, g[k]]) * s[n, g[k]])


# ---- int8-activation variant ----------------------------------------------

def test_activation_quant_hand_worked(oracle_mod):
    # amax = 127 -> s_a = 1; 62.5 rounds half away from zero to 63 (an
    # even-rounding mistake would give 62); -62.5 -> -63; tail past K -> 0.
    x = np.zeros((1, 20), np.float32)
    x[0, :5] = [127.0, 62.5, -62.5, 0.49, -127.0]
    qa, sa = oracle_mod.quantize_act(x, 20, 16)
    assert sa[0, 0] == np.float32(1.0)
    assert list(qa[0, :5]) == [127, 63, -63, 0, -127]
    assert sa[0, 1] == 0.0 and np.all(qa[0, 16:] == 0)


def test_activation_quant_range_and_error(oracle_mod):
    rng = np.random.default_rng(3)
    K, bs = 256, 32
    x = (rng.standard_normal((4, K)) * 3).astype(np.float32)
    qa, sa = oracle_mod.quantize_act(x, K, bs)
    assert qa.min() >= -127 and qa.max() <= 127
    xh = qa.astype(np.float64).reshape(4, -1, bs) * sa[:, :, None]
    err = np.abs(xh.reshape(4, K) - x)
    # each code is within half a step of its activation
    assert np.all(err <= 0.5 * np.repeat(sa, bs, axis=1) * (1 + 1e-6))
    # the block maximum maps to +-127 exactly
    amax_idx = np.abs(x.reshape(4, -1, bs)).argmax(axis=2)
    got = np.take_along_axis(np.abs(qa.reshape(4, -1, bs)), amax_idx[:, :, None], 2)
    assert np.all(got == 127)


def test_a8_integer_identity_int4_symmetric(oracle_mod):
    """sum (q-8) a = sum q a - 8 sum a  (the zero-point factorisation used by
    the int4 VNNI kernels), checked through the a8 oracle on integer data."""
    bits, bs, K, N = 4, 32, 128, 3
    rng = np.random.default_rng(9)
    q = rng.integers(0, 16, size=(N, K))
    b = pack_matrix_test(q, bits, bs)
    qa = rng.integers(-127, 128, size=(2, K)).astype(np.int8)
    sa = np.ones((2, K // bs), np.float32)
    s = np.ones((N, K // bs), np.float32)
    y, _ = oracle_mod.matmul_a8(qa, sa, b, s, None, N, K, bits, bs)
    a = qa.astype(np.int64)
    expect = a @ q.T - 8 * a.sum(axis=1, keepdims=True)
    assert np.array_equal(y, expect.astype(np.float64))


def test_a8_equals_fp_oracle_on_exactly_quantizable_x(oracle_mod):
    """When x = qa * s_a exactly, the a8 product and the fp oracle agree to
    f32 rescale rounding."""
    bits, bs, K, N = 8, 32, 96, 4
    b, s, zp, _ = _random(bits, bs, K, N, 1, seed=91)
    rng = np.random.default_rng(92)
    codes = rng.integers(-127, 128, size=(2, K))
    codes[:, ::bs] = 127                       # make amax hit 127 in every block
    x = (codes * 0.0625).astype(np.float32)    # s_a = 0.0625 exactly
    qa, sa = oracle_mod.quantize_act(x, K, bs)
    assert np.all(sa == np.float32(0.0625)) and np.array_equal(qa, codes.astype(np.int8))
    ya, ma = oracle_mod.matmul_a8(qa, sa, b, s, zp, N, K, bits, bs)
    yf, mf = oracle_mod.matmul(x.astype(np.float64), b, s, zp, N, K, bits, bs)
    assert np.all(np.abs(ya - yf) <= 1e-6 * (mf + 1e-30))
