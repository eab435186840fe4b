"""Act-order (g_idx) weights on the fast path: mnb_pack_weights_gidx sorts the
depths by their quantisation block and stores the permutation, and a call with
MNB_FLAG_KPERM runs the K-chunk decode GEMV gathering X through it (the
generic kernel for other shapes).  The reference is the oracle with g_idx,
MatMulNBitsKernel::dequantize_weight of onnx-runtime-ep-cpu 0.1.0-dev.5,
src/kernels/matmul_nbits.rs (the code keeps its place, the scale and zero
point follow g_idx[k])."""
import numpy as np
import pytest
import torch

import block_quantized_weight_matmulnbits_gb300 as mnb_mod
from block_quantized_weight_matmulnbits_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

F32, F16, BF16 = wl.F32, wl.F16, wl.BF16


@pytest.fixture(scope="module")
def mnb():
    mnb_mod.load()
    return mnb_mod


@pytest.fixture(scope="module")
def G(mnb):
    from tests import _gpu
    return _gpu


def _w(M, N, K, bits, bs, dt, asym, seed):
    act, sc, out = dt
    zp = (0, (1 << bits) - 1) if asym else None
    return wl.Workload(f"gidx{M}x{N}x{K}b{bits}s{bs}", M, N, K, bits, bs, act, out, sc, scale_lo=0.01,
                       scale_hi=0.05, zp=zp, seed=seed)


def act_order_gidx(K, bs, seed):
    """g_idx of an act-order quantiser: a random permutation of the depths cut into blocks of bs."""
    order = np.random.default_rng(seed).permutation(K)
    g = np.empty(K, dtype=np.int32)
    g[order] = np.arange(K, dtype=np.int32) // bs
    return g


def _pack_gidx(G, mnb, P, g):
    w = P.w
    packed = G.aligned_empty(mnb.mnb_packed_size_gidx(w.N, w.K, w.bits, w.bs))
    mnb.mnb_pack_weights_gidx(P.b, torch.from_numpy(g).cuda(), packed, w.N, w.K, w.bits, w.bs)
    return packed


def _run(mnb, P, packed, flags, g=None, kernel="auto"):
    w = P.w
    y = torch.empty((w.M, w.N), dtype=wl_torch(w.out_dtype), device="cuda")
    mnb.mnb_matmul_ex(P.x, packed, P.s, P.zp, y, w.M, w.N, w.K, w.bits, w.bs, w.act_dtype, w.out_dtype,
                      w.scale_dtype, kernel=kernel, flags=flags,
                      g_idx=None if g is None else torch.from_numpy(g).cuda())
    torch.cuda.synchronize()
    return y


def wl_torch(dt):
    return {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[dt]


CASES = [
    # M, bits, bs, (act, scale, out), asym, N, K
    (1, 4, 32, (BF16, F16, BF16), True, 4801, 4096),   # decode GEMV
    (3, 2, 64, (F16, F16, F32), True, 333, 1536),      # decode GEMV, ragged N
    (8, 8, 128, (BF16, F32, BF16), True, 700, 2048),   # decode GEMV, 8-bit
    (2, 4, 16, (F16, BF16, F16), False, 150, 256),     # decode GEMV, one chunk per row tile
    (1, 4, 128, (F16, F16, F16), True, 1000, 1000),    # K not a chunk multiple: generic
    (20, 4, 32, (BF16, F16, BF16), True, 300, 512),    # M > 8: generic
    (4, 2, 32, (F32, F32, F32), True, 100, 512),       # f32 X: generic
]


@pytest.mark.parametrize("M,bits,bs,dt,asym,N,K", CASES)
def test_act_order_matches_oracle(G, mnb, M, bits, bs, dt, asym, N, K):
    """Act-order pack + MNB_FLAG_KPERM against the oracle with g_idx, and against the plain pack with g_idx on
    the generic kernel."""
    w = _w(M, N, K, bits, bs, dt, asym, 1500 + M + bits + bs + N)
    P = G.Problem(w)
    g = act_order_gidx(K, bs, 77 + K)
    assert mnb.mnb_get_device_error() == 0
    y = _run(mnb, P, _pack_gidx(G, mnb, P, g), mnb.MNB_FLAG_KPERM)
    assert mnb.mnb_get_device_error() == 0
    ref, mag = P.oracle_full(g_idx=g)
    G.assert_within(P.y64(y), ref, mag, w.out_dtype, f"act-order {w.name}")
    y2 = _run(mnb, P, P.packed, 0, g=g)
    G.assert_within(P.y64(y2), ref, mag, w.out_dtype, f"plain pack + g_idx {w.name}")


@pytest.mark.parametrize("M,bits,bs,dt,asym,N,K", [CASES[0], CASES[2], CASES[3]])
def test_act_order_identity_gidx_is_bit_identical(G, mnb, M, bits, bs, dt, asym, N, K):
    """With g_idx[k] = k / bs the act-order pack stores the plain layout and the identity permutation: the
    decode GEMV's result is bit for bit that of the plain pack."""
    w = _w(M, N, K, bits, bs, dt, asym, 1600 + N)
    P = G.Problem(w)
    g = (np.arange(K) // bs).astype(np.int32)
    y1 = _run(mnb, P, _pack_gidx(G, mnb, P, g), mnb.MNB_FLAG_KPERM)
    y2 = _run(mnb, P, P.packed, 0)
    assert torch.equal(y1.view(torch.uint8), y2.view(torch.uint8))


def test_act_order_forced_kernels(G, mnb):
    """Forced families: the decode GEMV and the generic kernel take an act-order pack; the prefill GEMM needs the
    workspace for the gathered X."""
    w = _w(2, 256, 512, 4, 32, (BF16, F16, BF16), True, 1700)
    P = G.Problem(w)
    g = act_order_gidx(512, 32, 5)
    packed = _pack_gidx(G, mnb, P, g)
    ref, mag = P.oracle_full(g_idx=g)
    for kernel in ("gemv_mma", "generic"):
        y = _run(mnb, P, packed, mnb.MNB_FLAG_KPERM, kernel=kernel)
        G.assert_within(P.y64(y), ref, mag, w.out_dtype, f"act-order {kernel}")
    with pytest.raises(mnb.MnbError):
        _run(mnb, P, packed, mnb.MNB_FLAG_KPERM, kernel="gemm_tc")
    with pytest.raises(mnb.MnbError):  # g_idx together with the flag
        _run(mnb, P, packed, mnb.MNB_FLAG_KPERM, g=g)
    assert mnb.mnb_get_device_error() == 0


def test_act_order_flag_and_pack_must_agree(G, mnb):
    """The header records the act-order pack: the flag on a plain pack, or a plain call on an act-order pack, sets
    MNB_ERR_LAYOUT_MISMATCH; matching calls are unaffected."""
    w = _w(1, 128, 512, 4, 32, (BF16, F16, BF16), True, 1800)
    P = G.Problem(w)
    g = act_order_gidx(512, 32, 9)
    packed = _pack_gidx(G, mnb, P, g)
    assert mnb.mnb_get_device_error() == 0
    plain = G.aligned_empty(mnb.mnb_packed_size_gidx(w.N, w.K, w.bits, w.bs))  # room for the permutation
    mnb.mnb_pack_weights(P.b, plain, w.N, w.K, w.bits, w.bs)
    _run(mnb, P, plain, mnb.MNB_FLAG_KPERM)
    assert mnb.mnb_get_device_error() == mnb.MNB_ERR_LAYOUT_MISMATCH
    _run(mnb, P, packed, 0)
    assert mnb.mnb_get_device_error() == mnb.MNB_ERR_LAYOUT_MISMATCH
    y = _run(mnb, P, packed, mnb.MNB_FLAG_KPERM)
    assert mnb.mnb_get_device_error() == 0
    ref, mag = P.oracle_full(g_idx=g)
    G.assert_within(P.y64(y), ref, mag, w.out_dtype, "act-order after mismatches")


@pytest.mark.parametrize("bad", ["crowded_block", "out_of_range"])
def test_act_order_pack_rejects_bad_gidx(G, mnb, bad):
    """A g_idx that is not a permutation of whole blocks (one block with a depth too many, or a value outside
    [0, KB)) sets MNB_ERR_INVALID_ARG at pack time; a later call on that buffer reads no memory outside X."""
    w = _w(1, 64, 512, 4, 32, (BF16, F16, BF16), True, 1900)
    P = G.Problem(w)
    g = (np.arange(512) // 32).astype(np.int32)
    g[40] = 0 if bad == "crowded_block" else 16
    packed = _pack_gidx(G, mnb, P, g)
    assert mnb.mnb_get_device_error() == mnb.MNB_ERR_INVALID_ARG
    _run(mnb, P, packed, mnb.MNB_FLAG_KPERM)  # permutation entries are clamped before use
    assert mnb.mnb_get_device_error() == 0


PREFILL_CASES = [
    # M, bits, bs, (act, scale, out), asym, N, K
    (64, 4, 32, (BF16, F16, BF16), True, 512, 1024),
    (200, 2, 64, (BF16, BF16, F32), True, 300, 2048),
    (33, 8, 128, (F16, F32, F16), True, 250, 1024),
    (512, 4, 32, (BF16, F16, BF16), False, 256, 4096),
]


@pytest.mark.parametrize("M,bits,bs,dt,asym,N,K", PREFILL_CASES)
def test_act_order_prefill_on_tensor_cores(G, mnb, M, bits, bs, dt, asym, N, K):
    """M > 8 with the workspace of mnb_workspace_size_ex: X gathered into the pack's depth order, then the
    tensor-core prefill GEMM; against the oracle with g_idx. Without the workspace the call takes the generic
    kernel, and a forced GEMM reports MNB_ERR_NO_MEM."""
    w = _w(M, N, K, bits, bs, dt, asym, 2100 + M + bits)
    P = G.Problem(w)
    g = act_order_gidx(K, bs, 31 + K)
    packed = _pack_gidx(G, mnb, P, g)
    need = mnb.mnb_workspace_size_ex(M, N, K, bits, bs, 0, mnb.MNB_FLAG_KPERM)
    assert need == -(-(M * K * 2) // 256) * 256
    ws = G.aligned_empty(need)
    ref, mag = P.oracle_full(g_idx=g)
    for flags in (mnb.MNB_FLAG_KPERM, mnb.MNB_FLAG_KPERM | mnb.MNB_FLAG_PDL):
        y = torch.empty((M, N), dtype=wl_torch(w.out_dtype), device="cuda")
        mnb.mnb_matmul_ex(P.x, packed, P.s, P.zp, y, M, N, K, bits, bs, w.act_dtype, w.out_dtype, w.scale_dtype,
                          workspace=ws, flags=flags)
        torch.cuda.synchronize()
        assert mnb.mnb_get_device_error() == 0
        G.assert_within(P.y64(y), ref, mag, w.out_dtype, f"act-order prefill {w.name} flags={flags}")
    y2 = _run(mnb, P, packed, mnb.MNB_FLAG_KPERM)  # no workspace: generic
    G.assert_within(P.y64(y2), ref, mag, w.out_dtype, f"act-order generic {w.name}")
    with pytest.raises(mnb.MnbError):
        _run(mnb, P, packed, mnb.MNB_FLAG_KPERM, kernel="gemm_tc")

