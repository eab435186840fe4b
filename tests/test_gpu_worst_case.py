"""Worst-case inputs for the per-element bound, on every kernel family, with
f32 outputs so that no output rounding hides an error:

    |y - y_ref| <= 2e-3 * sum_k |x_k * w_k| + 1e-6

* One-hot X rows: y[m, n] is one weight w[n, k0] = (q - zp) * scale
  (onnx-runtime-ep-cpu matmul_nbits.rs, fn dequantize_nbits_value), so a
  kernel that rounds w to bf16 (relative error up to 2^-8) is caught on a
  single element.  q - zp = 3 with a scale of 1 + 2^-7 gives w = 3.0234375,
  a tie in bf16; a scale of 1 + 2^-8 is itself a bf16 tie.
* Rows with every x > 0 and every q > zp: rounding errors of a weight
  representation cannot cancel, so a systematic bias shows up in the sum.
* f32 scales of 1e-6 and 1e5 on the f16-activation path: outside the normal
  range of f16, where a kernel that forms w in f16 would underflow or
  overflow.
The expected values come from the fp64 oracle (the a8 oracle for accuracy
level 4)."""
import numpy as np
import pytest
import torch

from block_quantized_weight_matmulnbits_gb300 import workloads as wl
from tests._golden import pack_matrix_test, pack_zp_test

pytestmark = pytest.mark.gpu

F32, F16, BF16 = wl.F32, wl.F16, wl.BF16

# Scales that a bf16 or f16 weight representation gets wrong, times powers of two.
TIE_SCALES = [1 + 2 ** -7, 1 + 2 ** -8, 1 + 2 ** -8 + 2 ** -9, 1 + 3 * 2 ** -10, 1.0]
F32_EXTRA = [1e-6, 1e5, 0.1234567, 3.3333333e-4]


def build(M, N, K, bits, bs, act, sdt, zp_mode, x_mode, seed, extra_scales=()):
    """Inputs as the workload generator returns them (storage formats)."""
    rng = np.random.default_rng(seed)
    kb = -(-K // bs)
    maxq = (1 << bits) - 1
    if zp_mode == "none":
        z = np.full((N, kb), 1 << (bits - 1), dtype=np.int64)
    elif zp_mode == "low":  # zero points at the bottom so every q can exceed them
        z = rng.integers(0, max(1, maxq // 4) + 1, size=(N, kb))
    else:
        raise ValueError(zp_mode)
    # q - zp = 3 where the range allows, else the largest positive difference
    d = np.minimum(3, maxq - z)
    q = np.repeat(z + d, bs, axis=1)[:, :K]
    if x_mode == "positive":  # random codes above the zero point
        hi = np.repeat(maxq - z, bs, axis=1)[:, :K]
        q = np.repeat(z, bs, axis=1)[:, :K] + 1 + (rng.integers(0, 1 << 16, size=(N, K)) % np.maximum(hi, 1))
        q = np.minimum(q, maxq)
    pool = list(TIE_SCALES) + list(extra_scales)
    s = np.array([pool[(i * 7 + j * 3) % len(pool)] * 2.0 ** ((i + j) % 5 - 2)
                  for i in range(N) for j in range(kb)]).reshape(N, kb)
    if x_mode == "one_hot":
        x = np.zeros((M, K))
        vals = [1.0, 1.5, -3.0, 0.375, 2.0]
        for m in range(M):
            k0 = (m * 37 + (K - 1 if m == M - 1 else 0)) % K  # spans blocks, the last row hits depth K - 1
            x[m, k0] = vals[m % len(vals)]
    else:
        x = rng.uniform(0.5, 1.0, size=(M, K))
    return {
        "x": wl.to_storage(x, act),
        "b": pack_matrix_test(q, bits, bs),
        "scales": wl.to_storage(s, sdt),
        "zp": None if zp_mode == "none" else pack_zp_test(z, bits),
    }


def _wl(M, N, K, bits, bs, act, sdt, zp_mode):
    return wl.Workload(f"worst_m{M}_n{N}_k{K}_b{bits}_bs{bs}", M, N, K, bits, bs, act, F32, sdt,
                       zp=None if zp_mode == "none" else (0, (1 << bits) - 1))


def check(G, w, data, kernel, what, **kw):
    P = G.Problem(w, data)
    y = P.y64(P.run(kernel, **kw))
    ref, mag = P.oracle_full()
    G.assert_within(y, ref, mag, F32, f"{what} {kernel} {w.name}")


# (bits, bs, act, scale dtype, zero points)
SHAPES = [
    (4, 32, BF16, F16, "low"),
    (4, 32, BF16, F32, "none"),
    (8, 128, F16, F32, "low"),
    (2, 64, BF16, F16, "low"),
    (4, 16, F16, F16, "none"),
    (8, 32, BF16, BF16, "low"),
]


@pytest.mark.parametrize("x_mode", ["one_hot", "positive"])
@pytest.mark.parametrize("bits,bs,act,sdt,zpm", SHAPES)
@pytest.mark.parametrize("kernel,M,env", [
    ("gemv_mma", 1, {"MNB_GEMV_SCHED": "xr"}),
    ("gemv_mma", 8, {"MNB_GEMV_SCHED": "xr"}),
    ("gemv_mma", 1, {"MNB_GEMV_SCHED": "stream"}),
    ("gemv_mma", 8, {"MNB_GEMV_SCHED": "stream"}),
    ("gemv_mma", 16, {"MNB_GEMV_SCHED": "stream"}),
    ("gemv_mma", 1, {"MNB_GEMV_SCHED": "tile"}),
    ("gemv_mma", 5, {"MNB_GEMV_SCHED": "pers"}),
    ("gemv_mma", 16, {"MNB_GEMV_SCHED": "tile"}),
    ("gemm_tc", 5, {"MNB_TC_BT": "32"}),
    ("gemm_tc", 70, {"MNB_TC_BT": "64"}),
    ("gemm_tc", 130, {"MNB_TC_BT": "128"}),
    ("generic", 7, {}),
])
def test_worst_case_float_kernels(G, monkeypatch, kernel, M, env, bits, bs, act, sdt, zpm, x_mode):
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    N, K = 150, 4 * bs + 3 * 128 - 8
    extra = F32_EXTRA if sdt == F32 else ()
    data = build(M, N, K, bits, bs, act, sdt, zpm, x_mode, 4000 + M + bits + bs, extra)
    check(G, _wl(M, N, K, bits, bs, act, sdt, zpm), data, kernel, x_mode)


# The k-chunk decode schedule takes K a multiple of 4 packed tiles (1024 /
# bits depths) and at most 32 bytes of scales per row and chunk.
KS_SHAPES = [(4, 32, BF16, BF16, "low"), (4, 16, F16, F16, "none"), (2, 64, BF16, F16, "low"),
             (2, 256, F16, F16, "low"), (8, 32, BF16, BF16, "low"), (8, 128, F16, F32, "none"),
             (4, 256, BF16, F32, "low"), (4, 32, BF16, F32, "low"), (2, 64, F16, F32, "low")]


@pytest.mark.parametrize("x_mode", ["one_hot", "positive"])
@pytest.mark.parametrize("bits,bs,act,sdt,zpm", KS_SHAPES)
@pytest.mark.parametrize("M", [1, 3, 8])
def test_worst_case_gemv_ks(G, monkeypatch, M, bits, bs, act, sdt, zpm, x_mode):
    monkeypatch.setenv("MNB_GEMV_SCHED", "ks")
    N, K = 150, 3 * (1024 // bits)
    extra = F32_EXTRA if sdt == F32 else ()
    data = build(M, N, K, bits, bs, act, sdt, zpm, x_mode, 4300 + M + bits + bs, extra)
    check(G, _wl(M, N, K, bits, bs, act, sdt, zpm), data, "gemv_mma", x_mode)


@pytest.mark.parametrize("x_mode", ["one_hot", "positive"])
@pytest.mark.parametrize("bits,bs,sdt,zpm", [(4, 32, F32, "low"), (8, 128, F32, "none"), (2, 16, F16, "low")])
def test_worst_case_f32_activation_gemv(G, bits, bs, sdt, zpm, x_mode):
    N, K = 200, 6 * bs + 64
    data = build(1, N, K, bits, bs, F32, sdt, zpm, x_mode, 4100 + bits, F32_EXTRA if sdt == F32 else ())
    check(G, _wl(1, N, K, bits, bs, F32, sdt, zpm), data, "gemv", x_mode)


@pytest.mark.parametrize("x_mode", ["one_hot", "positive"])
@pytest.mark.parametrize("bits,bs,act,sdt,zpm", SHAPES[:4])
@pytest.mark.parametrize("M", [3, 40])
def test_worst_case_int8_activations(G, mnb, oracle_mod, M, bits, bs, act, sdt, zpm, x_mode):
    """Accuracy level 4 against the a8 oracle (activations quantised per block
    as the page does): one-hot rows quantise exactly, positive rows do not
    cancel.  M = 3 runs the int8 GEMV, M = 40 the prefill GEMM."""
    N, K = 150, 4 * bs + 3 * 128
    data = build(M, N, K, bits, bs, act, sdt, zpm, x_mode, 4200 + bits + M, F32_EXTRA if sdt == F32 else ())
    w = _wl(M, N, K, bits, bs, act, sdt, zpm)
    P = G.Problem(w, data)
    ws = G.aligned_empty(mnb.mnb_workspace_size(M, N, K, bits, bs, 4))
    y = P.y64(P.run(accuracy_level=4, workspace=ws))
    qa, sa = oracle_mod.quantize_act(P.x64.astype(np.float32), K, bs)
    ref, mag = oracle_mod.matmul_a8(qa, sa, data["b"], P.s32, data["zp"], N, K, bits, bs)
    G.assert_within(y, ref, mag, F32, f"a8 {x_mode} {w.name}")


@pytest.mark.parametrize("x_mode", ["one_hot", "positive"])
def test_worst_case_grouped(G, mnb, oracle_mod, x_mode):
    """The grouped (MoE) GEMV on two experts built from worst-case weights."""
    T, S, E, N, K, bits, bs = 4, 2, 2, 96, 512, 4, 32
    ds = [build(T, N, K, bits, bs, BF16, F16, "low", x_mode, 4300 + e) for e in range(E)]
    x = ds[0]["x"]
    ids = np.array([[0, 1], [1, 0], [0, 1], [1, 0]], dtype=np.int32)
    ps = mnb.mnb_packed_size(N, K, bits, bs)
    packed = G.aligned_empty(E * ps)
    for e in range(E):
        be = torch.from_numpy(np.ascontiguousarray(ds[e]["b"])).cuda()
        mnb.mnb_pack_weights(be, packed[e * ps:(e + 1) * ps], N, K, bits, bs)
    s_all = np.stack([d["scales"] for d in ds])
    z_all = np.stack([d["zp"] for d in ds])
    y = torch.empty((T, S, N), dtype=torch.float32, device="cuda")
    mnb.mnb_matmul_grouped(G.to_dev(x, BF16), torch.from_numpy(ids).cuda(), packed, G.to_dev(s_all, F16),
                           torch.from_numpy(z_all).cuda(), y, T, S, E, N, K, bits, bs, BF16, F32, F16)
    torch.cuda.synchronize()
    ref, mag = oracle_mod.matmul_grouped(wl.widen_f64(x, BF16), ids, np.stack([d["b"] for d in ds]),
                                         wl.widen_f32(s_all, F16), z_all, E, N, K, bits, bs)
    G.assert_within(y.cpu().numpy().astype(np.float64), ref, mag, F32, f"grouped {x_mode}")


@pytest.mark.parametrize("x_mode", ["one_hot", "positive"])
@pytest.mark.parametrize("bits,bs,act,sdt,zpm", [KS_SHAPES[0], KS_SHAPES[2], KS_SHAPES[5], KS_SHAPES[7]])
@pytest.mark.parametrize("M", [1, 5])
def test_worst_case_act_order(G, M, bits, bs, act, sdt, zpm, x_mode):
    """The act-order decode (mnb_pack_weights_gidx + MNB_FLAG_KPERM) on the same inputs, with a seeded act-order
    g_idx: the scale and zero point of each depth follow g_idx, so one-hot rows read single weights of the page's
    act-order dequantisation."""
    import block_quantized_weight_matmulnbits_gb300 as mnb
    N, K = 150, 3 * (1024 // bits)
    extra = F32_EXTRA if sdt == F32 else ()
    data = build(M, N, K, bits, bs, act, sdt, zpm, x_mode, 4600 + M + bits + bs, extra)
    w = _wl(M, N, K, bits, bs, act, sdt, zpm)
    P = G.Problem(w, data)
    order = np.random.default_rng(4700 + K).permutation(K)
    g = np.empty(K, dtype=np.int32)
    g[order] = np.arange(K, dtype=np.int32) // bs
    packed = G.aligned_empty(mnb.mnb_packed_size_gidx(N, K, bits, bs))
    mnb.mnb_pack_weights_gidx(P.b, torch.from_numpy(g).cuda(), packed, N, K, bits, bs)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    mnb.mnb_matmul_ex(P.x, packed, P.s, P.zp, y, M, N, K, bits, bs, act, F32, sdt, flags=mnb.MNB_FLAG_KPERM)
    torch.cuda.synchronize()
    assert mnb.mnb_get_device_error() == mnb.MNB_OK
    ref, mag = P.oracle_full(g_idx=g)
    G.assert_within(P.y64(y), ref, mag, F32, f"act-order {x_mode} {w.name}")

