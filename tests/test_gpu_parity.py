"""GPU parity: the CUDA path against the CPU oracle, through the C ABI.

Bars: the re-tiling round trip and the dequantised weights are bit-exact;
Y is within |y - y_ref| <= 2e-3 * sum_k |x_k w_k| + 1e-6 (+ half an output
ulp for bf16/f16 outputs) of the f64 oracle, element by element on small and
ragged shapes and on sampled outputs of the full-size workloads.
"""
import numpy as np
import pytest
import torch

from block_quantized_weight_matmulnbits_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

F32, F16, BF16 = wl.F32, wl.F16, wl.BF16
BITS_BS = [(4, 32), (4, 16), (4, 64), (4, 128), (2, 16), (2, 64), (2, 128), (8, 16), (8, 32), (8, 128)]
DTYPES = [(BF16, F16, BF16), (F16, F32, F16), (F32, F32, F32), (BF16, BF16, F32), (F16, F16, BF16)]


def _w(M, N, K, bits, bs, dt, asym, seed, x_dist="normal"):
    act, sc, out = dt
    zp = (0, (1 << bits) - 1) if asym else None
    return wl.Workload(f"t{M}x{N}x{K}b{bits}s{bs}", M, N, K, bits, bs, act, out, sc, x_dist=x_dist,
                       scale_lo=0.01, scale_hi=0.05, zp=zp, seed=seed)


@pytest.fixture(scope="module")
def G(mnb):
    from tests import _gpu
    return _gpu


# ---- layout module ---------------------------------------------------------

@pytest.mark.parametrize("bits,bs", BITS_BS)
@pytest.mark.parametrize("N,K", [(37, 40), (16, 256), (300, 389), (1, 16)])
def test_pack_unpack_round_trip(G, mnb, bits, bs, N, K):
    w = _w(1, N, K, bits, bs, DTYPES[0], True, 11)
    P = G.Problem(w)
    back = torch.zeros_like(P.b)
    mnb.mnb_unpack_codes(P.packed, back, N, K, bits, bs)
    torch.cuda.synchronize()
    assert torch.equal(back, P.b)


@pytest.mark.parametrize("bits,bs", BITS_BS)
@pytest.mark.parametrize("sdt", [F32, F16, BF16])
def test_dequantize_bit_exact(G, mnb, oracle_mod, bits, bs, sdt):
    N, K = 45, 3 * bs + 7
    w = _w(1, N, K, bits, bs, (BF16, sdt, BF16), True, 12)
    P = G.Problem(w)
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    mnb.mnb_dequantize(P.packed, P.s, P.zp, out, N, K, bits, bs, sdt)
    torch.cuda.synchronize()
    ref = oracle_mod.dequantize(P.d["b"], P.s32, P.d["zp"], N, K, bits, bs)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_dequantize_symmetric_default_zero_point(G, mnb, oracle_mod):
    for bits in (2, 4, 8):
        w = _w(1, 20, 64, bits, 32, (BF16, F16, BF16), False, 13)
        P = G.Problem(w)
        out = torch.empty((20, 64), dtype=torch.float32, device="cuda")
        mnb.mnb_dequantize(P.packed, P.s, None, out, 20, 64, bits, 32, F16)
        torch.cuda.synchronize()
        ref = oracle_mod.dequantize(P.d["b"], P.s32, None, 20, 64, bits, 32)
        assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


# ---- matmul: each kernel on small and ragged shapes -------------------------

GEMV_CASES = []
for i, (bits, bs) in enumerate(BITS_BS):
    for asym in (True, False):
        dt = DTYPES[(i + asym) % len(DTYPES)]
        GEMV_CASES.append((bits, bs, asym, dt, 300, 3 * bs + 5))
# long rows: every warp slice holds whole chunks, so each block size takes the
# statically unrolled path (1, 2, 4 or 8 k-steps per block)
for bits in (2, 4, 8):
    for bs in (16, 32, 64, 128):
        GEMV_CASES.append((bits, bs, bs != 32, DTYPES[(bits + bs) % len(DTYPES)], 40, 4096 + bs))
GEMV_CASES += [(4, 32, True, DTYPES[0], 64, 4096), (8, 128, True, DTYPES[1], 48, 11008),
               (2, 64, True, DTYPES[0], 33, 4096), (4, 32, False, DTYPES[2], 16, 32),
               (4, 16, True, DTYPES[3], 1, 16), (8, 16, True, DTYPES[4], 7, 1)]


@pytest.mark.parametrize("bits,bs,asym,dt,N,K", GEMV_CASES)
@pytest.mark.parametrize("kernel", ["gemv", "generic"])
def test_matmul_m1(G, bits, bs, asym, dt, N, K, kernel):
    w = _w(1, N, K, bits, bs, dt, asym, 100 + bits * 7 + bs + N)
    P = G.Problem(w)
    y = P.y64(P.run(kernel))
    ref, mag = P.oracle_full()
    G.assert_within(y, ref, mag, w.out_dtype, f"{kernel} {w.name}")


MMA_CASES = []
for i, (bits, bs) in enumerate(BITS_BS):
    for M in (1, 3, 8, 9, 16):
        act = BF16 if (i + M) % 2 else F16
        MMA_CASES.append((M, bits, bs, (act, [F16, F32, BF16][(i + M) % 3], [BF16, F16, F32][i % 3]),
                          (i + M) % 3 != 0, 150 + 16 * (i % 3) + M, 3 * bs + 5))
for bits in (2, 4, 8):
    for bs in (16, 32, 64, 128):
        for M in (1, 8):
            MMA_CASES.append((M, bits, bs, (BF16 if bs != 64 else F16, F16, BF16), bs != 32, 40, 4096 + bs))
MMA_CASES += [(1, 4, 32, (BF16, F16, BF16), True, 64, 4096), (1, 8, 128, (F16, F32, F16), True, 48, 11008),
              (8, 2, 64, (BF16, F16, BF16), True, 33, 4096), (16, 4, 32, (F16, F16, F16), False, 16, 32),
              (2, 4, 16, (BF16, BF16, F32), True, 1, 16), (5, 8, 16, (F16, F16, BF16), True, 7, 1),
              (12, 8, 32, (BF16, F32, BF16), True, 100, 200)]


@pytest.mark.parametrize("M,bits,bs,dt,asym,N,K", MMA_CASES)
def test_matmul_gemv_mma(G, M, bits, bs, dt, asym, N, K):
    w = _w(M, N, K, bits, bs, dt, asym, 700 + M * 13 + bits * 7 + bs + N)
    P = G.Problem(w)
    y = P.y64(P.run("gemv_mma"))
    ref, mag = P.oracle_full()
    G.assert_within(y, ref, mag, w.out_dtype, f"gemv_mma {w.name}")


# Enough row tiles (N >= 2 x 16 x SMs) for every decode schedule (the
# streaming default, the persistent ring, one CTA per row tile); ragged N
# and K, every code width, 1 <= M <= 16.
PERS_CASES = [
    (1, 4, 32, (BF16, F16, BF16), True, 4801, 4096),
    (1, 4, 16, (F16, F32, F16), False, 4800, 1000),
    (8, 2, 64, (BF16, F16, BF16), True, 4900, 4096),
    (3, 8, 32, (BF16, BF16, F32), True, 4850, 2048),
    (16, 4, 128, (F16, F16, BF16), True, 4864, 1024),
    (5, 2, 16, (BF16, F32, BF16), False, 4800, 640),
    (1, 8, 128, (F16, F32, F16), True, 4800, 2048),
    (12, 4, 64, (BF16, F16, F32), True, 4817, 3000),
]


@pytest.mark.parametrize("M,bits,bs,dt,asym,N,K", PERS_CASES)
@pytest.mark.parametrize("sched", ["ks", "xr", "stream", "pers", "tile"])
def test_matmul_gemv_schedules(G, monkeypatch, M, bits, bs, dt, asym, N, K, sched):
    monkeypatch.setenv("MNB_GEMV_SCHED", sched)
    w = _w(M, N, K, bits, bs, dt, asym, 900 + M * 13 + bits * 7 + bs + N)
    P = G.Problem(w)
    y = P.y64(P.run("gemv_mma"))
    ref, mag = P.oracle_full()
    G.assert_within(y, ref, mag, w.out_dtype, f"gemv_mma {sched} {w.name}")


# Shapes the k-chunk schedule takes (K a multiple of 4 packed tiles): every
# code width, block size and scale type it serves, ragged N, a partial last
# CTA, with and without zero points.
KS_CASES = [
    (1, 4, 32, (BF16, BF16, BF16), True, 4801, 4096),
    (1, 4, 128, (F16, F16, F16), False, 1000, 2048),
    (2, 2, 64, (BF16, BF16, F32), True, 333, 1536),
    (8, 2, 32, (BF16, BF16, BF16), True, 3000, 2048),
    (5, 8, 32, (F16, F16, F16), True, 777, 1152),
    (3, 8, 128, (BF16, BF16, BF16), False, 2500, 11008),
    (1, 4, 256, (BF16, BF16, BF16), True, 150, 768),
    (7, 4, 16, (F16, F16, F32), True, 4800, 512),
    (1, 2, 256, (F16, F16, F16), True, 16, 1024),
    (4, 8, 16, (BF16, BF16, BF16), True, 40, 256),
    (1, 4, 32, (BF16, F16, BF16), True, 11008, 4096),
    (1, 8, 128, (F16, F32, F16), True, 1000, 11008),
    (8, 2, 64, (BF16, F16, BF16), True, 2000, 4096),
    (2, 4, 64, (F16, BF16, F32), False, 500, 1024),
    (6, 2, 128, (BF16, F32, F32), True, 700, 2048),
]


@pytest.mark.parametrize("M,bits,bs,dt,asym,N,K", KS_CASES)
def test_matmul_gemv_ks(G, monkeypatch, M, bits, bs, dt, asym, N, K):
    monkeypatch.setenv("MNB_GEMV_SCHED", "ks")
    w = _w(M, N, K, bits, bs, dt, asym, 950 + M * 13 + bits * 7 + bs + N)
    P = G.Problem(w)
    y = P.y64(P.run("gemv_mma"))
    ref, mag = P.oracle_full()
    G.assert_within(y, ref, mag, w.out_dtype, f"gemv_mma ks {w.name}")


TC_CASES = []
for i, (bits, bs) in enumerate(BITS_BS):
    for M in (17, 128, 200):
        act = BF16 if (i + M) % 2 else F16
        TC_CASES.append((M, bits, bs, (act, [F16, F32, BF16][(i + M) % 3], [BF16, F16, F32][i % 3]),
                         (i + M) % 3 != 0, 96 + 16 * (i % 4) + (M % 5), 64 * (2 + i % 3)))
TC_CASES += [(64, 4, 32, (BF16, F16, BF16), False, 4096, 512), (1, 4, 32, (BF16, F16, BF16), True, 300, 256),
             (33, 8, 128, (F16, F32, F16), True, 250, 1000), (130, 2, 64, (BF16, F16, BF16), True, 77, 1024),
             (256, 4, 16, (BF16, BF16, F32), True, 520, 136), (300, 8, 16, (F16, F16, BF16), False, 48, 72)]


# Larger shapes for the tcgen05 GEMM, each run at every token-tile width
# (MNB_TC_BT): every code width, ragged M and N, both activation dtypes, with
# and without zero points.
TA_CASES = [
    (128, 4, 32, (BF16, F16, BF16), True, 256, 1024),
    (200, 4, 32, (F16, F32, F16), False, 300, 2048),
    (64, 2, 64, (BF16, F16, BF16), True, 130, 4096),
    (40, 8, 128, (F16, F32, F16), True, 200, 2048),
    (33, 8, 128, (BF16, F16, BF16), True, 77, 2048),
    (256, 4, 16, (BF16, BF16, F32), True, 520, 1024),
    (300, 4, 64, (F16, F16, BF16), True, 64, 2048),
    (17, 4, 32, (BF16, F16, BF16), True, 1000, 1024),
    (512, 4, 128, (BF16, F16, BF16), False, 384, 4096),
]


@pytest.mark.parametrize("M,bits,bs,dt,asym,N,K", TA_CASES)
@pytest.mark.parametrize("bt", ["32", "64", "128"])
def test_matmul_gemm_token_tiles(G, monkeypatch, M, bits, bs, dt, asym, N, K, bt):
    monkeypatch.setenv("MNB_TC_BT", bt)
    w = _w(M, N, K, bits, bs, dt, asym, 1100 + M * 3 + bits * 7 + bs + N)
    P = G.Problem(w)
    y = P.y64(P.run("gemm_tc"))
    ref, mag = P.oracle_full()
    G.assert_within(y, ref, mag, w.out_dtype, f"gemm_tc bt={bt} {w.name}")


@pytest.mark.parametrize("M,bits,bs,dt,asym,N,K", TC_CASES)
def test_matmul_gemm_tc(G, M, bits, bs, dt, asym, N, K):
    w = _w(M, N, K, bits, bs, dt, asym, 800 + M * 3 + bits * 7 + bs + N)
    P = G.Problem(w)
    y = P.y64(P.run("gemm_tc"))
    ref, mag = P.oracle_full()
    G.assert_within(y, ref, mag, w.out_dtype, f"gemm_tc {w.name}")


@pytest.mark.parametrize("M", [2, 3, 8, 17, 33, 64])
@pytest.mark.parametrize("bits,bs,dt", [(4, 32, DTYPES[0]), (8, 128, DTYPES[1]), (2, 64, DTYPES[2]),
                                        (4, 16, DTYPES[3])])
def test_matmul_generic_batched(G, M, bits, bs, dt):
    w = _w(M, 70, 2 * bs + 9, bits, bs, dt, True, 200 + M)
    P = G.Problem(w)
    y = P.y64(P.run("generic"))
    ref, mag = P.oracle_full()
    G.assert_within(y, ref, mag, w.out_dtype, f"generic {w.name}")


def test_bias_and_g_idx_generic(G, mnb):
    bits, bs, N, K, M = 4, 16, 40, 64, 3
    w = _w(M, N, K, bits, bs, DTYPES[0], True, 300)
    P = G.Problem(w)
    rng = np.random.default_rng(301)
    g = rng.integers(0, K // bs, size=K).astype(np.int32)
    bias = rng.standard_normal(N).astype(np.float32)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    mnb.mnb_matmul_ex(P.x, P.packed, P.s, P.zp, y, M, N, K, bits, bs, w.act_dtype, w.out_dtype, w.scale_dtype,
                      g_idx=torch.from_numpy(g).cuda(), bias=torch.from_numpy(bias).cuda(),
                      bias_dtype=F32, kernel="auto")
    torch.cuda.synchronize()
    ref, mag = P.oracle_full(g_idx=g, bias_f64=bias.astype(np.float64))
    G.assert_within(P.y64(y), ref, mag, w.out_dtype, "g_idx+bias")


@pytest.mark.parametrize("bad", ["one_past_end", "negative"])
def test_g_idx_out_of_range_sets_status_and_writes_nothing(G, mnb, bad):
    """A g_idx value outside [0, KB) is rejected as on the page
    (MatMulNBitsKernel::dequantize_weight): the device status word becomes
    MNB_ERR_INVALID_ARG and Y stays as it was.  The scale and zero-point
    buffers carry one padding row before and after, so even an unchecked read
    at the bad index would stay inside the allocation."""
    bits, bs, N, K, M = 4, 16, 40, 64, 3
    KB = K // bs
    w = _w(M, N, K, bits, bs, DTYPES[0], True, 320)
    P = G.Problem(w)
    zp_row = P.zp.shape[1]
    s_pad = torch.zeros((N + 2) * KB, dtype=P.s.dtype, device="cuda")
    s_pad[KB:(N + 1) * KB] = P.s.reshape(-1)
    z_pad = torch.zeros((N + 2) * zp_row, dtype=torch.uint8, device="cuda")
    z_pad[zp_row:(N + 1) * zp_row] = P.zp.reshape(-1)
    g = np.arange(K, dtype=np.int32) // bs
    g[K // 2] = KB if bad == "one_past_end" else -1
    sentinel = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    y = sentinel.clone()
    assert mnb.mnb_get_device_error() == 0
    mnb.mnb_matmul_ex(P.x, P.packed, s_pad[KB:], z_pad[zp_row:], y, M, N, K, bits, bs, w.act_dtype,
                      w.out_dtype, w.scale_dtype, g_idx=torch.from_numpy(g).cuda(), kernel="auto")
    torch.cuda.synchronize()
    assert mnb.mnb_get_device_error() == mnb.MNB_ERR_INVALID_ARG
    assert torch.equal(y, sentinel)
    # the next valid call is unaffected
    g[K // 2] = (K // 2) // bs
    y2 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    mnb.mnb_matmul_ex(P.x, P.packed, P.s, P.zp, y2, M, N, K, bits, bs, w.act_dtype, w.out_dtype,
                      w.scale_dtype, g_idx=torch.from_numpy(g).cuda(), kernel="auto")
    torch.cuda.synchronize()
    assert mnb.mnb_get_device_error() == 0
    ref, mag = P.oracle_full(g_idx=g)
    G.assert_within(P.y64(y2), ref, mag, w.out_dtype, "g_idx after a rejected call")


@pytest.mark.parametrize("kernel", ["gemv", "gemv_mma", "generic"])
def test_bias_m1(G, mnb, kernel):
    w = _w(1, 100, 96, 4, 32, DTYPES[0], True, 310)
    P = G.Problem(w)
    bias = torch.randn(100, dtype=torch.float16, device="cuda")
    y = torch.empty((1, 100), dtype=torch.bfloat16, device="cuda")
    mnb.mnb_matmul_ex(P.x, P.packed, P.s, P.zp, y, 1, 100, 96, 4, 32, w.act_dtype, w.out_dtype, w.scale_dtype,
                      bias=bias, bias_dtype=F16, kernel=kernel)
    torch.cuda.synchronize()
    b64 = bias.float().cpu().numpy().astype(np.float64)
    ref, mag = P.oracle_full(bias_f64=b64)
    G.assert_within(P.y64(y), ref, mag, w.out_dtype, "bias")


# ---- degenerate cases --------------------------------------------------------

@pytest.mark.parametrize("kernel", ["gemv", "gemv_mma", "gemm_tc", "generic"])
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_all_codes_equal_zero_point_give_zero(G, mnb, kernel, bits):
    from tests._golden import pack_matrix_test, pack_zp_test
    N, K, bs = 48, 128, 32
    rng = np.random.default_rng(bits)
    z = rng.integers(0, 1 << bits, size=(N, K // bs))
    w = _w(1 if kernel != "gemm_tc" else 40, N, K, bits, bs, DTYPES[0], True, 400)
    data = wl.generate(w)
    data["b"] = pack_matrix_test(np.repeat(z, bs, axis=1), bits, bs)
    data["zp"] = pack_zp_test(z, bits)
    P = G.Problem(w, data)
    y = P.y64(P.run(kernel))
    assert np.all(y == 0.0)


@pytest.mark.parametrize("kernel", ["gemv", "generic"])
def test_one_hot_row_selects_weight(G, mnb, oracle_mod, kernel):
    N, K, bits, bs = 64, 256, 4, 32
    w = _w(1, N, K, bits, bs, (F32, F32, F32), True, 410)
    data = wl.generate(w)
    for k0 in (0, 77, 255):
        data = dict(data)
        xv = np.zeros((1, K), np.float32)
        xv[0, k0] = 1.0
        data["x"] = xv
        P = G.Problem(w, data)
        y = P.run(kernel).cpu().numpy()[0]
        wref = oracle_mod.dequantize(data["b"], P.s32, data["zp"], N, K, bits, bs)
        assert np.array_equal(y, wref[:, k0])


@pytest.mark.parametrize("kernel", ["gemv", "gemv_mma", "gemm_tc", "generic"])
def test_deterministic_and_n_split_bit_identical(G, mnb, kernel):
    N, K = 96, 1024
    w = _w(1 if kernel != "gemm_tc" else 70, N, K, 4, 32, DTYPES[0], True, 420)
    P = G.Problem(w)
    y1 = P.run(kernel).clone()
    y2 = P.run(kernel).clone()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    # rows [0, 48) and [48, 96) packed and run on their own (N-sharding)
    parts = []
    for lo, hi in ((0, 48), (48, 96)):
        d = {"x": P.d["x"], "b": P.d["b"][lo:hi], "scales": P.d["scales"][lo:hi], "zp": P.d["zp"][lo:hi]}
        Ps = G.Problem(wl.variant(w, N=hi - lo), d)
        parts.append(Ps.run(kernel))
    assert torch.equal(torch.cat(parts, dim=1).view(torch.int16), y1.view(torch.int16))


def test_m0_and_status_word(G, mnb):
    w = _w(1, 32, 64, 4, 32, DTYPES[0], True, 430)
    P = G.Problem(w)
    y = torch.empty((1, 32), dtype=torch.bfloat16, device="cuda")
    mnb.mnb_matmul(P.x, P.packed, P.s, P.zp, y, 0, 32, 64, 4, 32, BF16, BF16, F16)
    assert mnb.mnb_get_device_error() == 0


def test_forced_kernel_that_cannot_run_is_unsupported(G, mnb):
    w = _w(2, 32, 64, 4, 32, DTYPES[0], True, 440)
    P = G.Problem(w)
    with pytest.raises(mnb.MnbError) as e:
        P.run("gemv")
    assert e.value.status == mnb.MNB_ERR_UNSUPPORTED


def test_injected_launch_failure_reports_cuda_error(G, mnb, monkeypatch):
    w = _w(1, 32, 64, 4, 32, DTYPES[0], True, 450)
    P = G.Problem(w)
    monkeypatch.setenv("MNB_FAIL_LAUNCH", "1")
    with pytest.raises(mnb.MnbError) as e:
        P.run("gemv")
    assert e.value.status == mnb.MNB_ERR_CUDA
    monkeypatch.delenv("MNB_FAIL_LAUNCH")
    P.run("gemv")


# ---- full-size workloads, sampled outputs ----------------------------------

@pytest.mark.parametrize("ci", [0, 1, 2, 3, 4])
def test_full_size_workloads_sampled(G, ci):
    w = wl.config(ci)
    P = G.Problem(w)
    y = P.y64(P.run("auto"))
    rng = np.random.default_rng(500 + ci)
    n_samples = 256
    ms = rng.integers(0, w.M, n_samples)
    ns = rng.integers(0, w.N, n_samples)
    ns[:4] = [0, w.N - 1, w.N // 2, 15]
    ref, mag = P.oracle_points(ms, ns)
    G.assert_within(y[ms, ns], ref, mag, w.out_dtype, w.name)
    assert np.all(np.isfinite(y))


def test_pdl_chain_matches_plain_launches(G, mnb):
    """A chain y1 = f(x), y2 = f(y1), y3 = f(y2) launched with programmatic
    dependent launch must equal the same chain launched plainly, bit for bit:
    each call reads its X only after the previous call has finished."""
    N = K = 1024
    w = _w(1, N, K, 4, 32, (BF16, F16, BF16), True, 900)
    P = G.Problem(w)
    outs = {}
    for flags in (0, mnb.MNB_FLAG_PDL):
        ys = [torch.empty((1, N), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
        src = P.x
        for y in ys:
            mnb.mnb_matmul_ex(src, P.packed, P.s, P.zp, y, 1, N, K, 4, 32, BF16, BF16, F16, kernel="gemv_mma",
                              flags=flags)
            src = y
        torch.cuda.synchronize()
        outs[flags] = [y.clone() for y in ys]
    for a, b in zip(outs[0], outs[mnb.MNB_FLAG_PDL]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
