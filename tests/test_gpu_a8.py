"""GPU parity of the int8-activation path (accuracy level 4) through the C ABI.

Bars: the activation codes and scales of mnb_quantize_activations are
bit-exact against the oracle's per-block quantisation; Y is within
2e-3 * sum_k |x_hat_k w_k| + 1e-6 (+ half an output ulp) of the oracle's
exact-integer block dots rescaled in f64, where x_hat = qa * s_a is the
quantised activation (the tolerance is relative to the quantised product,
not to the float path).
"""
import numpy as np
import pytest
import torch

from block_quantized_weight_matmulnbits_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

F32, F16, BF16 = wl.F32, wl.F16, wl.BF16


@pytest.fixture(scope="module")
def G(mnb):
    from tests import _gpu
    return _gpu


def _w(M, N, K, bits, bs, dt, asym, seed, x_dist="normal"):
    act, sc, out = dt
    zp = (0, (1 << bits) - 1) if asym else None
    return wl.Workload(f"a8_{M}x{N}x{K}b{bits}s{bs}", M, N, K, bits, bs, act, out, sc, x_dist=x_dist,
                       scale_lo=0.01, scale_hi=0.05, zp=zp, seed=seed)


def _quantize_dev(G, mnb, P):
    w = P.w
    kb = -(-w.K // w.bs)
    qa = G.aligned_empty(w.M * kb * w.bs)
    sa = torch.empty((w.M, kb), dtype=torch.float32, device="cuda")
    mnb.mnb_quantize_activations(P.x, qa, sa, w.M, w.K, w.bs, w.act_dtype)
    torch.cuda.synchronize()
    return qa.cpu().numpy().view(np.int8).reshape(w.M, kb * w.bs), sa.cpu().numpy()


def _run_a8(G, mnb, P, bias=None, flags=0, ws=None):
    w = P.w
    if ws is None:
        need = mnb.mnb_workspace_size(w.M, w.N, w.K, w.bits, w.bs, 4)
        ws = G.aligned_empty(need)
    kw = {}
    if bias is not None:
        kw = dict(bias=bias, bias_dtype=F32)
    return P.run(accuracy_level=4, workspace=ws, flags=flags, **kw)


def _oracle_a8(oracle_mod, P, bias=None):
    w = P.w
    qa, sa = oracle_mod.quantize_act(P.x64.astype(np.float32), w.K, w.bs)
    return oracle_mod.matmul_a8(qa, sa, P.d["b"], P.s32, P.d["zp"], w.N, w.K, w.bits, w.bs, bias_f64=bias)


# ---- activation quantisation (bit-exact) -------------------------------------

@pytest.mark.parametrize("dt", [F32, F16, BF16])
@pytest.mark.parametrize("M,K,bs", [(1, 4096, 32), (3, 389, 16), (2, 1000, 128), (5, 77, 64), (16, 512, 256)])
def test_quantize_activations_bit_exact(G, mnb, oracle_mod, dt, M, K, bs):
    w = _w(M, 16, K, 4, bs, (dt, F32, F32), False, 31)
    P = G.Problem(w)
    qa, sa = _quantize_dev(G, mnb, P)
    ref_qa, ref_sa = oracle_mod.quantize_act(P.x64.astype(np.float32), K, bs)
    assert np.array_equal(sa.view(np.uint32), ref_sa.view(np.uint32))
    assert np.array_equal(qa, ref_qa)


def test_quantize_activations_ties_and_zero_block(G, mnb, oracle_mod):
    """amax = 127 gives s_a = 1 exactly, so x = +-2.5, +-3.5 are exact ties
    (rounded away from zero); an all-zero block gives s_a = 0 and zero codes."""
    K, bs = 64, 32
    x = np.zeros((1, K), dtype=np.float32)
    x[0, :8] = [127.0, 2.5, -2.5, 3.5, -3.5, 0.5, -0.5, 126.5]
    x[0, 8:32] = np.linspace(-100, 100, 24, dtype=np.float32)
    w = _w(1, 16, K, 4, bs, (F32, F32, F32), False, 32)
    d = wl.generate(w)
    d["x"] = x
    P = G.Problem(w, data=d)
    qa, sa = _quantize_dev(G, mnb, P)
    ref_qa, ref_sa = oracle_mod.quantize_act(x, K, bs)
    assert list(qa[0, :8]) == [127, 3, -3, 4, -4, 1, -1, 127]
    assert sa[0, 1] == 0.0 and not qa[0, 32:].any()
    assert np.array_equal(qa, ref_qa) and np.array_equal(sa.view(np.uint32), ref_sa.view(np.uint32))


# ---- the int8-activation product ----------------------------------------------

A8_CASES = [
    # M, bits, bs, dtypes (act, scale, out), asym, N, K
    (1, 4, 32, (BF16, F16, BF16), True, 300, 4096),
    (1, 4, 16, (F16, F32, F16), False, 77, 389),
    (1, 4, 64, (F32, F32, F32), True, 128, 1000),
    (1, 2, 16, (BF16, F16, BF16), True, 45, 300),
    (1, 2, 64, (BF16, BF16, F32), True, 200, 4096),
    (1, 2, 128, (F16, F16, BF16), False, 64, 777),
    (1, 8, 128, (F16, F32, F16), True, 160, 11008),
    (1, 8, 16, (BF16, F16, BF16), True, 33, 400),
    (1, 8, 32, (F32, F32, F32), False, 48, 96),
    (2, 4, 32, (BF16, F16, BF16), True, 100, 2048),
    (5, 2, 64, (BF16, F16, BF16), True, 90, 4096),
    (8, 2, 64, (BF16, F16, BF16), True, 256, 4096),
    (8, 8, 128, (F16, F32, F16), True, 70, 1536),
    (16, 4, 32, (BF16, F16, BF16), True, 48, 4096),
    (16, 2, 16, (F16, F16, F32), True, 40, 208),
    (3, 4, 256, (BF16, F16, BF16), True, 50, 1024),
    (1, 4, 512, (BF16, F16, BF16), True, 50, 2048),
]


@pytest.mark.parametrize("M,bits,bs,dt,asym,N,K", A8_CASES)
@pytest.mark.parametrize("hilo", ["1", "0"])
def test_matmul_a8(G, mnb, oracle_mod, monkeypatch, M, bits, bs, dt, asym, N, K, hilo):
    """M <= 4 runs the bf16 K-chunk GEMV over hi / lo activation rows where its shape limits
    allow (hilo=1), else and with MNB_A8_HILO=0 the int8 dp4a kernel."""
    monkeypatch.setenv("MNB_A8_HILO", hilo)
    w = _w(M, N, K, bits, bs, dt, asym, 40 + M + bits + bs)
    P = G.Problem(w)
    assert mnb.mnb_select_kernel(M, N, K, bits, bs, dt[0], 4) == "gemv_i8"
    y = _run_a8(G, mnb, P)
    ref, mag = _oracle_a8(oracle_mod, P)
    G.assert_within(P.y64(y), ref, mag, w.out_dtype, f"a8 {w.name}")


@pytest.mark.parametrize("M,bits,bs,dt,asym,N,K", [c for c in A8_CASES if c[0] <= 4 and 32 <= c[2] <= 256])
def test_matmul_a8_fused_quantisation_bit_identical(G, mnb, monkeypatch, M, bits, bs, dt, asym, N, K):
    """The one-launch form (X quantised while the GEMV stages it) gives the bits of the two-launch form
    (quantised hi / lo rows through the workspace, MNB_A8_HILO=2)."""
    w = _w(M, N, K, bits, bs, dt, asym, 40 + M + bits + bs)
    P = G.Problem(w)
    y1 = _run_a8(G, mnb, P).clone()
    monkeypatch.setenv("MNB_A8_HILO", "2")
    y2 = _run_a8(G, mnb, P)
    assert torch.equal(y1.view(torch.uint8), y2.view(torch.uint8))


@pytest.mark.parametrize("act", [F32, BF16])
def test_matmul_a8_fused_ties_and_zero_block(G, mnb, oracle_mod, monkeypatch, act):
    """The one-launch form on exact quantisation ties (amax = 127 gives s_a = 1, so +-2.5 and +-3.5 round away
    from zero) and an all-zero block (s_a = 0, zero codes): the bits of the two-launch form and the oracle's
    integer result within the bound."""
    M, N, K, bs = 2, 64, 512, 32
    w = _w(M, N, K, 4, bs, (act, F16, F32), True, 77)
    d = wl.generate(w)
    x = wl.widen_f64(d["x"], act).copy()
    x[:, :8] = [127.0, 2.5, -2.5, 3.5, -3.5, 0.5, -0.5, 126.5]
    x[:, 32:64] = 0.0  # block 1: all zero
    x[1, 64:96] = -x[1, 64:96]
    d["x"] = wl.to_storage(x, act)
    P = G.Problem(w, data=d)
    y1 = _run_a8(G, mnb, P).clone()
    monkeypatch.setenv("MNB_A8_HILO", "2")
    y2 = _run_a8(G, mnb, P)
    assert torch.equal(y1.view(torch.uint8), y2.view(torch.uint8))
    ref, mag = _oracle_a8(oracle_mod, P)
    G.assert_within(P.y64(y1), ref, mag, w.out_dtype, "a8 fused ties")


def test_matmul_a8_bias_and_pdl(G, mnb, oracle_mod):
    w = _w(4, 111, 2048, 4, 32, (BF16, F16, BF16), True, 50)
    P = G.Problem(w)
    bias_h = np.random.default_rng(5).uniform(-1, 1, w.N).astype(np.float32)
    bias = torch.from_numpy(bias_h).cuda()
    ref, mag = _oracle_a8(oracle_mod, P, bias=bias_h.astype(np.float64))
    for flags in (0, mnb.MNB_FLAG_PDL):
        y = _run_a8(G, mnb, P, bias=bias, flags=flags)
        G.assert_within(P.y64(y), ref, mag, w.out_dtype, f"a8 bias flags={flags}")


def test_matmul_a8_all_codes_equal_zero_point_give_zero(G, mnb):
    from tests._golden import pack_matrix_test, pack_zp_test
    N, K, bs = 48, 256, 32
    for bits in (2, 4, 8):
        z = np.random.default_rng(bits).integers(0, 1 << bits, size=(N, K // bs))
        w = _w(3, N, K, bits, bs, (BF16, F16, F32), True, 51)
        d = wl.generate(w)
        d["b"] = pack_matrix_test(np.repeat(z, bs, axis=1), bits, bs)
        d["zp"] = pack_zp_test(z, bits)
        P = G.Problem(w, d)
        y = P.y64(_run_a8(G, mnb, P))
        assert np.all(y == 0.0), f"bits {bits}"


def test_matmul_a8_deterministic(G, mnb):
    w = _w(8, 300, 4096, 4, 32, (BF16, F16, BF16), True, 52)
    P = G.Problem(w)
    y1 = _run_a8(G, mnb, P).clone()
    y2 = _run_a8(G, mnb, P)
    assert torch.equal(y1, y2)


def test_matmul_a8_workspace_checks(G, mnb):
    w = _w(2, 64, 512, 4, 32, (BF16, F16, BF16), True, 53)
    P = G.Problem(w)
    need = mnb.mnb_workspace_size(w.M, w.N, w.K, w.bits, w.bs, 4)
    assert need >= w.M * w.K + w.M * (w.K // w.bs) * 4
    assert mnb.mnb_workspace_size(w.M, w.N, w.K, w.bits, w.bs, 0) == 0
    with pytest.raises(mnb.MnbError) as e:
        _run_a8(G, mnb, P, ws=G.aligned_empty(need - 1))
    assert e.value.status == mnb.MNB_ERR_NO_MEM
    raw = G.aligned_empty(need + 256)
    with pytest.raises(mnb.MnbError) as e:
        _run_a8(G, mnb, P, ws=raw[16:16 + need])
    assert e.value.status == mnb.MNB_ERR_INVALID_ARG
    # a float-path kernel cannot be forced with accuracy level 4, nor the int8 one without it
    with pytest.raises(mnb.MnbError):
        P.run(kernel="gemv_mma", accuracy_level=4, workspace=G.aligned_empty(need))
    with pytest.raises(mnb.MnbError):
        P.run(kernel="gemv_i8")


@pytest.mark.parametrize("ci", [1, 2, 3])
def test_full_size_decode_workloads_a8(G, mnb, oracle_mod, ci):
    w = wl.CONFIGS[ci]
    P = G.Problem(w)
    y = _run_a8(G, mnb, P)
    ref, mag = _oracle_a8(oracle_mod, P)
    G.assert_within(P.y64(y), ref, mag, w.out_dtype, f"a8 {w.name}")


# ---- accuracy level 4 above 16 rows: the tensor-core prefill GEMM ----------------

A8_GEMM_CASES = [
    # M, bits, bs, dtypes (act, scale, out), asym, N, K
    (17, 4, 32, (BF16, F16, BF16), True, 300, 4096),
    (64, 2, 64, (F16, F16, F32), True, 257, 2048),
    (512, 4, 32, (BF16, F16, BF16), False, 1024, 4096),
    (40, 8, 128, (F32, F32, F16), True, 200, 1152),
    (100, 4, 16, (BF16, BF16, BF16), True, 130, 1000),
    (33, 2, 256, (F16, F16, F16), True, 64, 1536),
    (20, 4, 512, (BF16, F16, F32), True, 70, 2048),
    (129, 8, 32, (BF16, F16, BF16), False, 129, 640),
]


@pytest.mark.parametrize("M,bits,bs,dt,asym,N,K", A8_GEMM_CASES)
def test_matmul_a8_prefill(G, mnb, oracle_mod, M, bits, bs, dt, asym, N, K):
    w = _w(M, N, K, bits, bs, dt, asym, 60 + M + bits + bs)
    P = G.Problem(w)
    assert mnb.mnb_select_kernel(M, N, K, bits, bs, dt[0], 4) == "gemm_tc"
    y = _run_a8(G, mnb, P)
    assert mnb.mnb_get_device_error() == mnb.MNB_OK
    ref, mag = _oracle_a8(oracle_mod, P)
    G.assert_within(P.y64(y), ref, mag, w.out_dtype, f"a8 prefill {w.name}")


def test_matmul_a8_prefill_forced_at_small_m(G, mnb, oracle_mod):
    """The prefill GEMM also runs below 17 rows when forced, with its own (larger) workspace."""
    w = _w(5, 150, 1024, 4, 32, (BF16, F16, BF16), True, 61)
    P = G.Problem(w)
    kb = -(-w.K // w.bs)
    need = -(-(w.M * kb * w.bs * 4) // 256) * 256  # code * s_a as tf32, [M, Kpad]
    y = P.run(kernel="gemm_tc", accuracy_level=4, workspace=G.aligned_empty(need))
    ref, mag = _oracle_a8(oracle_mod, P)
    G.assert_within(P.y64(y), ref, mag, w.out_dtype, "a8 prefill forced")
    with pytest.raises(mnb.MnbError) as e:
        P.run(kernel="gemm_tc", accuracy_level=4, workspace=G.aligned_empty(need - 256))
    assert e.value.status == mnb.MNB_ERR_NO_MEM


def test_matmul_a8_prefill_bias_pdl_deterministic(G, mnb, oracle_mod):
    w = _w(70, 111, 2048, 4, 32, (BF16, F16, BF16), True, 62)
    P = G.Problem(w)
    bias_h = np.random.default_rng(6).uniform(-1, 1, w.N).astype(np.float32)
    bias = torch.from_numpy(bias_h).cuda()
    ref, mag = _oracle_a8(oracle_mod, P, bias=bias_h.astype(np.float64))
    ys = []
    for flags in (0, mnb.MNB_FLAG_PDL, 0):
        y = _run_a8(G, mnb, P, bias=bias, flags=flags)
        G.assert_within(P.y64(y), ref, mag, w.out_dtype, f"a8 prefill bias flags={flags}")
        ys.append(y.clone())
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])


def test_matmul_a8_prefill_all_codes_equal_zero_point_give_zero(G, mnb):
    from tests._golden import pack_matrix_test, pack_zp_test
    N, K, bs = 150, 512, 32
    for bits in (2, 4, 8):
        z = np.random.default_rng(10 + bits).integers(0, 1 << bits, size=(N, K // bs))
        w = _w(40, N, K, bits, bs, (BF16, F16, F32), True, 63)
        d = wl.generate(w)
        d["b"] = pack_matrix_test(np.repeat(z, bs, axis=1), bits, bs)
        d["zp"] = pack_zp_test(z, bits)
        P = G.Problem(w, d)
        y = P.y64(_run_a8(G, mnb, P))
        assert np.all(y == 0.0), f"bits {bits}"


def test_full_size_prefill_workload_a8(G, mnb, oracle_mod):
    """The 512 x 4096 x 4096 int4 prefill at accuracy level 4, against the oracle on 24 sampled rows
    (rows are independent: the oracle takes those rows' codes and scales)."""
    w = wl.CONFIGS[4]
    P = G.Problem(w)
    y = P.y64(_run_a8(G, mnb, P))
    qa, sa = oracle_mod.quantize_act(P.x64.astype(np.float32), w.K, w.bs)
    rows = np.unique(np.linspace(0, w.M - 1, 24).astype(int))
    ref, mag = oracle_mod.matmul_a8(qa[rows], sa[rows], P.d["b"], P.s32, P.d["zp"], w.N, w.K, w.bits, w.bs)
    G.assert_within(y[rows], ref, mag, w.out_dtype, "a8 prefill full size")
