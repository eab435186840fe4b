"""FP8 (E4M3 / E5M2) and NVFP4 weights on the GPU against the oracle:
dequant_matmul_fp8 and dequant_matmul_nvfp4 of rlx-cpu 0.2.13,
src/thunk/ops/quant.rs.

* One-hot activation rows read single weights, so every one of the 256 FP8
  codes (and every E2M1 nibble under every E4M3 block-scale code) is compared
  bit for bit with the oracle's decode.
* The page's E4M3 rule makes exponent 15 infinite (zero mantissa) or NaN;
  columns holding such codes must come out non-finite exactly where the
  oracle's do.
* Random activations at ragged shapes (partial 16-deep NVFP4 scale blocks,
  N not a multiple of 16) are held to the per-element bound
  |y - y_ref| <= 2e-3 * sum_k |x_k w_k| + 1e-6 (+ half an output ulp)."""
import numpy as np
import pytest
import torch

import block_quantized_weight_matmulnbits_gb300 as mnb
import oracle
from block_quantized_weight_matmulnbits_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

F32, F16, BF16 = wl.F32, wl.F16, wl.BF16


@pytest.fixture(scope="module")
def G(mnb_lib):
    from tests import _gpu
    return _gpu


@pytest.fixture(scope="module")
def mnb_lib():
    return mnb.load()


def _pack(G, w_kn_bytes, N, K, fmt):
    w = torch.from_numpy(np.ascontiguousarray(w_kn_bytes)).cuda()
    packed = G.aligned_empty(mnb.mnb_fp_packed_size(N, K, fmt))
    mnb.mnb_pack_fp_weights(w, packed, N, K, fmt)
    return packed


def _run(G, x_stored, act, packed, scales_t, gs, M, N, K, fmt, out_dtype):
    x = G.to_dev(x_stored, act)
    y = torch.empty((M, N), dtype=G.TORCH_DT[out_dtype], device="cuda")
    mnb.mnb_matmul_fp(x, packed, scales_t, gs, y, M, N, K, fmt, act, out_dtype)
    torch.cuda.synchronize()
    assert mnb.mnb_get_device_error() == mnb.MNB_OK
    return G.to_host_f64(y, out_dtype)


def _nibbles(codes_kn):
    """[K, N] nibble codes to the packed byte stream (flat index k*N + n, low nibble first)."""
    flat = np.asarray(codes_kn, dtype=np.uint8).ravel()
    if flat.size % 2:
        flat = np.concatenate([flat, np.zeros(1, np.uint8)])
    return (flat[0::2] | (flat[1::2] << 4)).astype(np.uint8)


def _same_class(y, ref):
    """Non-finite elements agree in kind (NaN, +inf, -inf); returns the finite mask."""
    assert np.array_equal(np.isnan(y), np.isnan(ref))
    assert np.array_equal(np.isposinf(y), np.isposinf(ref))
    assert np.array_equal(np.isneginf(y), np.isneginf(ref))
    return np.isfinite(ref)


def _finite_fp8_codes(e5m2):
    c = np.arange(256, dtype=np.uint8)
    exp = (c >> 2) & 31 if e5m2 else (c >> 3) & 15
    return c[exp != (31 if e5m2 else 15)]


@pytest.mark.parametrize("fmt", [mnb.MNB_WF_E4M3, mnb.MNB_WF_E5M2])
@pytest.mark.parametrize("with_scales", [False, True])
def test_fp8_every_code_one_hot(G, fmt, with_scales):
    """Y row m = W row m (x one-hot at k = m): each finite code times its column scale, rounded once
    to f32 (the page's acc += x * w * s with x = 1)."""
    e5m2 = fmt == mnb.MNB_WF_E5M2
    codes = _finite_fp8_codes(e5m2)
    N, K = 150, len(codes) // 2 + 7
    rng = np.random.default_rng(61 + fmt)
    w = rng.choice(codes, size=(K, N)).astype(np.uint8)
    w.reshape(-1)[: len(codes)] = codes  # every finite code at least once
    s = rng.uniform(0.25, 4.0, size=N).astype(np.float32) if with_scales else None
    M = K
    x = np.eye(M, K)
    packed = _pack(G, w, N, K, fmt)
    st = None if s is None else torch.from_numpy(s).cuda()
    y = _run(G, wl.to_storage(x, F32), F32, packed, st, 0.0, M, N, K, fmt, F32)
    ref, _ = oracle.matmul_fp8(x, w, s, K, N, e5m2=e5m2)
    # the oracle's product w * s is exact (fp64); a one-hot row returns it rounded once to f32
    assert np.array_equal(y, ref.astype(np.float32).astype(np.float64))


@pytest.mark.parametrize("fmt", [mnb.MNB_WF_E4M3, mnb.MNB_WF_E5M2])
def test_fp8_non_finite_codes(G, fmt):
    """Infinity and NaN codes (exponent all ones) poison exactly the columns that hold them."""
    e5m2 = fmt == mnb.MNB_WF_E5M2
    N, K, M = 40, 33, 3
    rng = np.random.default_rng(7 + fmt)
    w = rng.choice(_finite_fp8_codes(e5m2), size=(K, N)).astype(np.uint8)
    specials = [0x7C, 0xFC, 0x7D, 0x7F] if e5m2 else [0x78, 0xF8, 0x79, 0xFF]  # +inf, -inf, NaN, NaN
    for j, code in enumerate(specials):
        w[5 + j, 3 * j + 1] = code
    x = rng.uniform(0.5, 1.0, size=(M, K))
    packed = _pack(G, w, N, K, fmt)
    y = _run(G, wl.to_storage(x, F32), F32, packed, None, 0.0, M, N, K, fmt, F32)
    ref, mag = oracle.matmul_fp8(x, w, None, K, N, e5m2=e5m2)
    fin = _same_class(y, ref)
    assert (~fin).sum() == M * len(specials)
    G.assert_within(np.where(fin, y, 0), np.where(fin, ref, 0), np.where(fin, mag, 0), F32, "fp8 finite columns")


def test_nvfp4_every_nibble_and_scale_code_one_hot(G):
    """Every E2M1 nibble under every E4M3 block-scale code, formed as the page forms it."""
    N = 256
    K = 16 * 16 + 5  # 17 scale blocks, the last partial
    KB = -(-K // 16)
    rng = np.random.default_rng(404)
    w4 = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
    w4[:16, :] = np.arange(16, dtype=np.uint8)[:, None]  # block 0: all nibbles in every column
    finite_scales = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    s8 = rng.choice(finite_scales, size=(KB, N)).astype(np.uint8)
    s8[0, :] = np.arange(256, dtype=np.uint8)  # block 0: every scale code (NaN ones included), one per column
    gs = np.float32(0.7351)
    M = K
    x = np.eye(M, K)
    packed = _pack(G, _nibbles(w4), N, K, mnb.MNB_WF_NVFP4)
    y = _run(G, wl.to_storage(x, F32), F32, packed, torch.from_numpy(s8).cuda(), float(gs), M, N, K,
             mnb.MNB_WF_NVFP4, F32)
    ref, _ = oracle.matmul_nvfp4(x, _nibbles(w4), s8, float(gs), K, N)
    fin = _same_class(y, ref)
    assert np.array_equal(y[fin], ref[fin])
    # block-0 columns with the scale NaN codes (0x7F, 0xFF) are the only non-finite ones
    assert set(np.nonzero(~fin)[1].tolist()) == {0x7F, 0xFF}


CASES = [
    # (M, N, K, act, out)
    (1, 4096, 4096, BF16, BF16),
    (1, 333, 1000, F16, F16),
    (7, 150, 261, F32, F32),
    (33, 77, 512, BF16, F32),
    (16, 1024, 130, F16, BF16),
]


@pytest.mark.parametrize("M,N,K,act,out", CASES)
@pytest.mark.parametrize("fmt", [mnb.MNB_WF_E4M3, mnb.MNB_WF_E5M2])
def test_fp8_random(G, M, N, K, act, out, fmt):
    e5m2 = fmt == mnb.MNB_WF_E5M2
    rng = np.random.default_rng(M * 131 + N + K + fmt)
    w = rng.choice(_finite_fp8_codes(e5m2), size=(K, N)).astype(np.uint8)
    s = rng.uniform(1e-3, 1e-2, size=N).astype(np.float32)
    x = rng.standard_normal((M, K))
    xs = wl.to_storage(x, act)
    x64 = wl.widen_f64(xs, act) if act != F32 else xs.astype(np.float64)
    packed = _pack(G, w, N, K, fmt)
    y = _run(G, xs, act, packed, torch.from_numpy(s).cuda(), 0.0, M, N, K, fmt, out)
    ref, mag = oracle.matmul_fp8(x64, w, s, K, N, e5m2=e5m2)
    G.assert_within(y, ref, mag, out, f"fp8 fmt={fmt} {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,act,out", CASES)
def test_nvfp4_random(G, M, N, K, act, out):
    rng = np.random.default_rng(M * 17 + N + K)
    KB = -(-K // 16)
    w4 = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
    s8 = rng.choice([c for c in range(256) if (c & 0x7F) != 0x7F], size=(KB, N)).astype(np.uint8)
    gs = float(np.float32(rng.uniform(0.01, 0.1)))
    x = rng.standard_normal((M, K))
    xs = wl.to_storage(x, act)
    x64 = wl.widen_f64(xs, act) if act != F32 else xs.astype(np.float64)
    packed = _pack(G, _nibbles(w4), N, K, mnb.MNB_WF_NVFP4)
    y = _run(G, xs, act, packed, torch.from_numpy(s8).cuda(), gs, M, N, K, mnb.MNB_WF_NVFP4, out)
    ref, mag = oracle.matmul_nvfp4(x64, _nibbles(w4), s8, gs, K, N)
    G.assert_within(y, ref, mag, out, f"nvfp4 {M}x{N}x{K}")


def test_fp_format_mismatch_sets_status(G):
    """A buffer packed as E4M3 called as E5M2 (same N, K) sets MNB_ERR_LAYOUT_MISMATCH."""
    N, K, M = 64, 64, 2
    w = np.zeros((K, N), np.uint8)
    packed = _pack(G, w, N, K, mnb.MNB_WF_E4M3)
    x = G.to_dev(wl.to_storage(np.ones((M, K)), F32), F32)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    mnb.mnb_matmul_fp(x, packed, None, 0.0, y, M, N, K, mnb.MNB_WF_E5M2, F32, F32)
    torch.cuda.synchronize()
    assert mnb.mnb_get_device_error() == mnb.MNB_ERR_LAYOUT_MISMATCH
    assert mnb.mnb_get_device_error() == mnb.MNB_OK  # read and cleared


def test_fp_pack_is_a_permutation(G):
    """Packing FP8 moves codes only: the integer unpack of the same buffer (8-bit codes, 128-deep
    blocks) returns the [N, K] transpose of the source."""
    N, K = 37, 300
    rng = np.random.default_rng(5)
    w = rng.integers(0, 256, size=(K, N)).astype(np.uint8)
    packed = _pack(G, w, N, K, mnb.MNB_WF_E4M3)
    KB = -(-K // 128)
    out = torch.zeros(N * KB * 128, dtype=torch.uint8, device="cuda")
    # the header records the FP format, so the integer unpack flags a mismatch but still moves the bytes
    mnb.mnb_unpack_codes(packed, out, N, K, 8, 128)
    torch.cuda.synchronize()
    mnb.mnb_get_device_error()
    got = out.cpu().numpy().reshape(N, KB * 128)[:, :K]
    assert np.array_equal(got, w.T)


# ---- the decode GEMV (M <= 4, bf16 / f16 X, K a multiple of 128 for FP8 and 256 for NVFP4) ----

FAST_CASES = [
    # (M, N, K, act, out)
    (1, 11008, 4096, BF16, BF16),
    (1, 150, 512, F16, F32),
    (3, 333, 1024, BF16, F32),
    (4, 4096, 2048, F16, F16),
    (2, 17, 256, BF16, BF16),
]


@pytest.mark.parametrize("M,N,K,act,out", FAST_CASES)
@pytest.mark.parametrize("fmt", [mnb.MNB_WF_E4M3, mnb.MNB_WF_E5M2, mnb.MNB_WF_NVFP4])
def test_fp_decode_gemv(G, monkeypatch, M, N, K, act, out, fmt):
    """The decode GEMV against the oracle, and against the exact kernel forced with MNB_FP_KERNEL=generic."""
    rng = np.random.default_rng(M * 7 + N + K + 13 * fmt)
    x = rng.standard_normal((M, K))
    xs = wl.to_storage(x, act)
    x64 = wl.widen_f64(xs, act)
    if fmt == mnb.MNB_WF_NVFP4:
        w4 = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
        s8 = rng.choice([c for c in range(256) if (c & 0x7F) != 0x7F], size=(K // 16, N)).astype(np.uint8)
        gs = float(np.float32(0.0371))
        src, st = _nibbles(w4), torch.from_numpy(s8).cuda()
        ref, mag = oracle.matmul_nvfp4(x64, src, s8, gs, K, N)
    else:
        e5m2 = fmt == mnb.MNB_WF_E5M2
        src = rng.choice(_finite_fp8_codes(e5m2), size=(K, N)).astype(np.uint8)
        s = rng.uniform(1e-3, 1e-2, size=N).astype(np.float32)
        gs, st = 0.0, torch.from_numpy(s).cuda()
        ref, mag = oracle.matmul_fp8(x64, src, s, K, N, e5m2=e5m2)
    packed = _pack(G, src, N, K, fmt)
    y = _run(G, xs, act, packed, st, gs, M, N, K, fmt, out)
    G.assert_within(y, ref, mag, out, f"fp gemv fmt={fmt} {M}x{N}x{K}")
    monkeypatch.setenv("MNB_FP_KERNEL", "generic")
    y2 = _run(G, xs, act, packed, st, gs, M, N, K, fmt, out)
    G.assert_within(y2, ref, mag, out, f"fp generic fmt={fmt} {M}x{N}x{K}")
    if fmt == mnb.MNB_WF_NVFP4:
        # the table kernel, which the tensor-core kernel replaces for these shapes
        monkeypatch.setenv("MNB_FP_KERNEL", "lut")
        y3 = _run(G, xs, act, packed, st, gs, M, N, K, fmt, out)
        G.assert_within(y3, ref, mag, out, f"fp lut fmt={fmt} {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,offset", [(4, 64, 256, 0), (1, 4096, 512, 1), (3, 48, 1024, 3)])
def test_nvfp4_decode_gemv_scale_staging_paths(G, M, N, K, offset):
    """The tensor-core NVFP4 GEMV's two block-scale staging paths: 16 codes per load (N % 16 == 0 and a 16-byte
    aligned scale array) and one code per load (a scale array starting `offset` bytes into an allocation), with one
    K-chunk per row tile (K = 256) among the shapes; both against the oracle."""
    rng = np.random.default_rng(4242 + N + K + offset)
    x = rng.standard_normal((M, K))
    xs = wl.to_storage(x, BF16)
    w4 = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
    s8 = rng.choice([c for c in range(256) if (c & 0x7F) != 0x7F], size=(K // 16, N)).astype(np.uint8)
    gs = float(np.float32(0.0517))
    packed = _pack(G, _nibbles(w4), N, K, mnb.MNB_WF_NVFP4)
    buf = torch.zeros(s8.size + 16, dtype=torch.uint8, device="cuda")
    st = buf[offset:offset + s8.size]
    st.copy_(torch.from_numpy(s8.ravel()).cuda())
    y = _run(G, xs, BF16, packed, st, gs, M, N, K, mnb.MNB_WF_NVFP4, F32)
    ref, mag = oracle.matmul_nvfp4(wl.widen_f64(xs, BF16), _nibbles(w4), s8, gs, K, N)
    G.assert_within(y, ref, mag, F32, f"nvfp4 gemv staging offset={offset} {M}x{N}x{K}")


@pytest.mark.parametrize("act", [BF16, F16])
def test_nvfp4_decode_gemv_every_nibble_and_scale_code(G, act):
    """The tensor-core NVFP4 GEMV on one-hot rows: every E2M1 nibble (the subnormal 0.5 and both zeros
    included) under every E4M3 block-scale code equals the page's f32(f32(e2m1 * e4m3) * global) bit for
    bit, and only the NaN scale codes give NaN."""
    N, K, M = 256, 512, 4
    rng = np.random.default_rng(405 + act)
    w4 = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
    w4[:16, :] = np.arange(16, dtype=np.uint8)[:, None]  # block 0: nibble k at depth k, every column
    s8 = rng.choice([c for c in range(256) if (c & 0x7F) != 0x7F], size=(K // 16, N)).astype(np.uint8)
    s8[0, :] = np.arange(256, dtype=np.uint8)  # block 0: every scale code, one per column
    gs = np.float32(0.7351)
    packed = _pack(G, _nibbles(w4), N, K, mnb.MNB_WF_NVFP4)
    st = torch.from_numpy(s8).cuda()
    for d0 in range(0, 16, M):
        x = np.zeros((M, K))
        x[np.arange(M), d0 + np.arange(M)] = 1.0
        y = _run(G, wl.to_storage(x, act), act, packed, st, float(gs), M, N, K, mnb.MNB_WF_NVFP4, F32)
        ref, _ = oracle.matmul_nvfp4(x, _nibbles(w4), s8, float(gs), K, N)
        fin = _same_class(y, ref)
        assert np.array_equal(y[fin], ref[fin]), f"depths {d0}..{d0 + M - 1}"
        assert set(np.nonzero(~fin)[1].tolist()) == {0x7F, 0xFF}


@pytest.mark.parametrize("fmt", [mnb.MNB_WF_E4M3, mnb.MNB_WF_E5M2])
def test_fp8_decode_gemv_non_finite_codes(G, fmt):
    """The decode GEMV's decode tables keep the page's exponent-all-ones rule: infinity and NaN codes
    poison exactly their columns."""
    e5m2 = fmt == mnb.MNB_WF_E5M2
    N, K, M = 48, 256, 1
    rng = np.random.default_rng(70 + fmt)
    w = rng.choice(_finite_fp8_codes(e5m2), size=(K, N)).astype(np.uint8)
    specials = [0x7C, 0xFC, 0x7D, 0xFF] if e5m2 else [0x78, 0xF8, 0x7A, 0xFF]
    for j, code in enumerate(specials):
        w[40 + 3 * j, 5 * j + 2] = code
    x = rng.uniform(0.5, 1.0, size=(M, K))
    xs = wl.to_storage(x, BF16)
    packed = _pack(G, w, N, K, fmt)
    y = _run(G, xs, BF16, packed, None, 0.0, M, N, K, fmt, F32)
    ref, mag = oracle.matmul_fp8(wl.widen_f64(xs, BF16), w, None, K, N, e5m2=e5m2)
    fin = _same_class(y, ref)
    assert (~fin).sum() == len(specials)
    G.assert_within(np.where(fin, y, 0), np.where(fin, ref, 0), np.where(fin, mag, 0), F32, "fp8 gemv finite")


def test_nvfp4_decode_gemv_nan_scale_codes(G):
    """NaN block-scale codes (0x7F, 0xFF) make their columns NaN; every other column stays within the bound."""
    N, K, M = 64, 512, 2
    rng = np.random.default_rng(77)
    w4 = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
    s8 = rng.choice([c for c in range(256) if (c & 0x7F) != 0x7F], size=(K // 16, N)).astype(np.uint8)
    s8[3, 10] = 0x7F
    s8[30, 41] = 0xFF
    x = rng.uniform(0.5, 1.0, size=(M, K))
    xs = wl.to_storage(x, F16)
    packed = _pack(G, _nibbles(w4), N, K, mnb.MNB_WF_NVFP4)
    y = _run(G, xs, F16, packed, torch.from_numpy(s8).cuda(), 0.5, M, N, K, mnb.MNB_WF_NVFP4, F32)
    ref, mag = oracle.matmul_nvfp4(wl.widen_f64(xs, F16), _nibbles(w4), s8, 0.5, K, N)
    fin = _same_class(y, ref)
    assert set(np.nonzero(~fin)[1].tolist()) == {10, 41}
    G.assert_within(np.where(fin, y, 0), np.where(fin, ref, 0), np.where(fin, mag, 0), F32, "nvfp4 gemv finite")


@pytest.mark.parametrize("fmt,kern", [(mnb.MNB_WF_NVFP4, ""), (mnb.MNB_WF_NVFP4, "lut"), (mnb.MNB_WF_E4M3, "")])
def test_fp_pdl_chain_matches_plain_launches(G, monkeypatch, fmt, kern):
    """y1 = f(x), y2 = f(y1), y3 = f(y2) launched with MNB_FLAG_PDL equals the plain chain bit for bit: each
    call stages its X only after the previous call has finished."""
    if kern:
        monkeypatch.setenv("MNB_FP_KERNEL", kern)
    N = K = 1024
    rng = np.random.default_rng(911 + fmt)
    if fmt == mnb.MNB_WF_NVFP4:
        w4 = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
        s8 = rng.choice(np.arange(0x20, 0x38), size=(K // 16, N)).astype(np.uint8)
        src, st, gs = _nibbles(w4), torch.from_numpy(s8).cuda(), 0.03
    else:
        src = rng.choice(_finite_fp8_codes(False), size=(K, N)).astype(np.uint8)
        st, gs = torch.from_numpy(rng.uniform(1e-3, 1e-2, size=N).astype(np.float32)).cuda(), 0.0
    packed = _pack(G, src, N, K, fmt)
    x0 = G.to_dev(wl.to_storage(rng.standard_normal((1, K)), BF16), BF16)
    outs = {}
    for flags in (0, mnb.MNB_FLAG_PDL):
        ys = [torch.empty((1, N), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
        xin = x0
        for y in ys:
            mnb.mnb_matmul_fp(xin, packed, st, gs, y, 1, N, K, fmt, BF16, BF16, flags=flags)
            xin = y
        torch.cuda.synchronize()
        assert mnb.mnb_get_device_error() == mnb.MNB_OK
        outs[flags] = [y.clone() for y in ys]
    for a, b in zip(outs[0], outs[mnb.MNB_FLAG_PDL]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
