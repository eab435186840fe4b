"""Pins of oracle.matmul_grouped, the grouped (mixture-of-experts) product of
ggml's MUL_MAT_ID (toy 0.8.0, data/vendor/ggml/src/ggml-cpu/spacemit/ime.cpp,
forward_mul_mat_id) and rlx's grouped dequant matmul (rlx-cpu 0.2.13,
src/thunk/ops/quant.rs).

The oracle groups (token, slot) rows by expert and runs one plain product per
group.  These pins check it against things that share none of that
gathering and scattering:
  * a one-hot restatement: y[t, s] = sum over ALL experts e of
    [ids[t, s] == e] * (x_row(t, s) . W_e^T), with W_e from the pinned
    dequantisation and numpy's einsum (a wrong row, slot, expert slab or
    transposition changes the result);
  * relabelling the experts (permuting the weight slabs and the ids alike)
    leaves y unchanged, bit for bit;
  * E = 1 reduces to the plain product of each token's row;
  * per-slot activation rows that all equal the token's row reduce to the
    shared-row form.
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_matmulnbits_gb300 import workloads as wl

F16, BF16, F32 = wl.F16, wl.BF16, wl.F32


def _case(T, S, E, N, K, bits, bs, zp, x_per_slot=False, ids="distinct", seed=0, scale_dtype=F16):
    w = wl.MoeWorkload(f"pin_t{T}_s{S}_e{E}", T, S, E, N, K, bits, bs, F32, F32, scale_dtype,
                       x_per_slot=x_per_slot, ids=ids, scale_lo=0.01, scale_hi=0.05, zp=zp, seed=seed)
    d = wl.generate_moe(w)
    x = wl.widen_f64(d["x"], F32)
    s32 = wl.widen_f32(d["scales"], scale_dtype)
    return w, d, x, s32


def _one_hot_reference(w, d, x, s32):
    W = np.stack([oracle.dequantize(d["b"][e], s32[e], None if d["zp"] is None else d["zp"][e], w.N, w.K, w.bits,
                                    w.bs) for e in range(w.E)]).astype(np.float64)  # [E, N, K]
    xr = x if w.x_per_slot else np.repeat(x[:, None, :], w.S, axis=1)            # [T, S, K]
    every = np.einsum("tsk,enk->tsen", xr, W)                                      # all experts
    mag_every = np.einsum("tsk,enk->tsen", np.abs(xr), np.abs(W))
    onehot = (d["ids"][:, :, None] == np.arange(w.E)[None, None, :]).astype(np.float64)  # [T, S, E]
    return np.einsum("tse,tsen->tsn", onehot, every), np.einsum("tse,tsen->tsn", onehot, mag_every)


CASES = [
    dict(T=3, S=2, E=5, N=20, K=64, bits=4, bs=16, zp=(0, 15), seed=1),
    dict(T=4, S=3, E=4, N=17, K=100, bits=2, bs=32, zp=None, seed=2, ids="repeat"),
    dict(T=2, S=2, E=6, N=9, K=256, bits=8, bs=128, zp=(100, 150), seed=3, x_per_slot=True),
    dict(T=5, S=1, E=3, N=33, K=48, bits=4, bs=16, zp=None, seed=4, scale_dtype=BF16),
]


@pytest.mark.parametrize("c", CASES, ids=lambda c: f"t{c['T']}s{c['S']}e{c['E']}b{c['bits']}")
def test_grouped_equals_one_hot_sum_over_all_experts(c):
    w, d, x, s32 = _case(**c)
    y, mag = oracle.matmul_grouped(x, d["ids"], d["b"], s32, d["zp"], w.E, w.N, w.K, w.bits, w.bs,
                                   x_per_slot=w.x_per_slot)
    y_ref, mag_ref = _one_hot_reference(w, d, x, s32)
    assert y.shape == (w.T, w.S, w.N)
    np.testing.assert_allclose(y, y_ref, rtol=0, atol=1e-12 * max(1.0, np.abs(mag_ref).max()))
    np.testing.assert_allclose(mag, mag_ref, rtol=1e-12)


def test_relabelling_experts_leaves_the_result_unchanged():
    w, d, x, s32 = _case(T=4, S=2, E=6, N=24, K=96, bits=4, bs=32, zp=(0, 15), seed=5)
    y, _ = oracle.matmul_grouped(x, d["ids"], d["b"], s32, d["zp"], w.E, w.N, w.K, w.bits, w.bs)
    perm = np.random.default_rng(6).permutation(w.E)          # expert e becomes perm[e]
    inv = np.argsort(perm)
    y2, _ = oracle.matmul_grouped(x, perm[d["ids"]], d["b"][inv], s32[inv], d["zp"][inv], w.E, w.N, w.K, w.bits,
                                  w.bs)
    assert np.array_equal(y, y2)


def test_single_expert_is_the_plain_product():
    w, d, x, s32 = _case(T=3, S=2, E=1, N=18, K=64, bits=4, bs=16, zp=(0, 15), seed=7, ids="repeat")
    assert np.all(d["ids"] == 0)
    y, _ = oracle.matmul_grouped(x, d["ids"], d["b"], s32, d["zp"], 1, w.N, w.K, w.bits, w.bs)
    y_plain, _ = oracle.matmul(x, d["b"][0], s32[0], d["zp"][0], w.N, w.K, w.bits, w.bs)
    for s in range(w.S):
        assert np.array_equal(y[:, s, :], y_plain)


def test_equal_slot_rows_reduce_to_the_shared_row_form():
    w, d, x, s32 = _case(T=3, S=3, E=4, N=16, K=64, bits=2, bs=16, zp=(0, 3), seed=8)
    y, _ = oracle.matmul_grouped(x, d["ids"], d["b"], s32, d["zp"], w.E, w.N, w.K, w.bits, w.bs)
    x3 = np.repeat(x[:, None, :], w.S, axis=1)
    y3, _ = oracle.matmul_grouped(x3, d["ids"], d["b"], s32, d["zp"], w.E, w.N, w.K, w.bits, w.bs,
                                  x_per_slot=True)
    assert np.array_equal(y, y3)


def test_out_of_range_expert_id_is_an_error():
    w, d, x, s32 = _case(T=2, S=2, E=3, N=16, K=32, bits=4, bs=16, zp=None, seed=9)
    ids = d["ids"].copy()
    ids[1, 0] = w.E
    with pytest.raises(ValueError):
        oracle.matmul_grouped(x, ids, d["b"], s32, None, w.E, w.N, w.K, w.bits, w.bs)
