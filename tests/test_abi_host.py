"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every symbol include/mnb.h declares, sizes the packed
buffer as documented, chooses kernels as documented, and rejects invalid
arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import block_quantized_weight_matmulnbits_gb300 as mnb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return mnb.load()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "mnb.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mnb_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_binding_exports():
    assert declared_symbols() == sorted(mnb.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert getattr(lib, name) is not None


def test_abi_version(lib):
    assert mnb.mnb_abi_version() == 1


@pytest.mark.parametrize("N,K,bits,bs", [(11008, 4096, 4, 32), (4096, 11008, 8, 128), (14336, 4096, 2, 64),
                                         (37, 40, 4, 32), (1, 1, 2, 16), (17, 300, 8, 16)])
def test_packed_size_formula(N, K, bits, bs):
    KB = -(-K // bs)
    KT = 256 // bits
    ktiles = -(-(KB * bs) // KT)
    nt = -(-N // 16)
    assert mnb.mnb_packed_size(N, K, bits, bs) == 256 + nt * ktiles * 512
    # the packed buffer never holds less than the ORT bytes
    assert mnb.mnb_packed_size(N, K, bits, bs) >= N * KB * bs * bits // 8


@pytest.mark.parametrize("bad", [(0, 64, 4, 32), (8, 0, 4, 32), (8, 64, 3, 32), (8, 64, 4, 24), (8, 64, 4, 8),
                                 (8, 64, 16, 32), (-1, 64, 4, 32)])
def test_packed_size_rejects_invalid(bad):
    assert mnb.mnb_packed_size(*bad) == 0


@pytest.mark.parametrize("N,K", [(4096, 4096), (37, 300), (1, 1), (150, 261)])
def test_fp_packed_size_formula(N, K):
    nt = -(-N // 16)
    # FP8: 8-bit codes in 128-deep blocks, 32 depths per tile
    assert mnb.mnb_fp_packed_size(N, K, mnb.MNB_WF_E4M3) == 256 + nt * (-(-K // 128) * 128 // 32) * 512
    assert mnb.mnb_fp_packed_size(N, K, mnb.MNB_WF_E5M2) == mnb.mnb_fp_packed_size(N, K, mnb.MNB_WF_E4M3)
    # NVFP4: 4-bit codes in 16-deep scale blocks, 64 depths per tile
    assert mnb.mnb_fp_packed_size(N, K, mnb.MNB_WF_NVFP4) == 256 + nt * (-(-(-(-K // 16) * 16) // 64)) * 512


@pytest.mark.parametrize("bad", [(0, 64, 1), (8, 0, 1), (8, 64, 0), (8, 64, 4), (-1, 64, 3)])
def test_fp_packed_size_rejects_invalid(bad):
    assert mnb.mnb_fp_packed_size(*bad) == 0


def test_fp_matmul_rejects_invalid_before_cuda():
    """Argument errors come back before any CUDA call (null pointers, NVFP4 without scales)."""
    lib = mnb.load()
    assert lib.mnb_matmul_fp(None, None, None, 1.0, None, 1, 8, 8, 3, 0, 0, None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_matmul_fp(None, None, None, 1.0, None, 0, 8, 8, 1, 0, 0, None) == mnb.MNB_OK  # M == 0
    assert lib.mnb_matmul_fp(None, None, None, 1.0, None, 1, 8, 8, 9, 0, 0, None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_pack_fp_weights(None, None, 0, 8, 8, 1, None) == mnb.MNB_ERR_INVALID_ARG
    # the flags form: an unknown flag bit is an argument error; MNB_FLAG_PDL alone is not
    assert lib.mnb_matmul_fp_ex(None, None, None, 1.0, None, 0, 8, 8, 1, 0, 0, None, 2) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_matmul_fp_ex(None, None, None, 1.0, None, 0, 8, 8, 1, 0, 0, None, mnb.MNB_FLAG_PDL) == mnb.MNB_OK


@pytest.mark.parametrize("M,K,bs", [(17, 4096, 32), (512, 4096, 32), (64, 1000, 128)])
def test_a8_prefill_workspace_size(M, K, bs):
    """Accuracy level 4 above 16 rows: the quantised activations code * s_a as tf32 in f32
    containers, [M, Kpad], 256-byte aligned size."""
    kb = -(-K // bs)
    assert mnb.mnb_workspace_size(M, 4096, K, 4, bs, 4) == -(-(M * kb * bs * 4) // 256) * 256


def test_kernel_selection():
    assert mnb.mnb_select_kernel(1, 11008, 4096, 4, 32, mnb.MNB_BF16) == "gemv_mma"
    assert mnb.mnb_select_kernel(1, 4096, 11008, 8, 128, mnb.MNB_F16) == "gemv_mma"
    assert mnb.mnb_select_kernel(1, 256, 256, 4, 32, mnb.MNB_F32) == "gemv"
    assert mnb.mnb_select_kernel(8, 14336, 4096, 2, 64, mnb.MNB_BF16) == "gemv_mma"
    assert mnb.mnb_select_kernel(16, 4096, 4096, 4, 32, mnb.MNB_F16) == "gemv_mma"
    assert mnb.mnb_select_kernel(17, 4096, 4096, 4, 32, mnb.MNB_BF16) == "gemm_tc"
    assert mnb.mnb_select_kernel(512, 4096, 4096, 4, 32, mnb.MNB_BF16) == "gemm_tc"
    assert mnb.mnb_select_kernel(8, 4096, 4096, 4, 32, mnb.MNB_F32) == "generic"
    assert mnb.mnb_select_kernel(1, 4096, 4096, 4, 32, mnb.MNB_BF16, 4) == "gemv_i8"
    assert mnb.mnb_select_kernel(16, 4096, 4096, 4, 32, mnb.MNB_BF16, 4) == "gemv_i8"
    assert mnb.mnb_select_kernel(17, 4096, 4096, 4, 32, mnb.MNB_BF16, 4) == "gemm_tc"


FAKE = 1 << 20  # aligned, never dereferenced: validation fails before any CUDA call


def _ex(lib, **kw):
    a = mnb.MatmulArgs()
    d = dict(x=FAKE, packed_b=FAKE, scales=FAKE, y=FAKE, M=1, N=64, K=64, bits=4, block_size=32,
             act_dtype=2, out_dtype=2, scale_dtype=1, bias_dtype=0, accuracy_level=0, kernel=0)
    d.update(kw)
    for k, v in d.items():
        setattr(a, k, v)
    return lib.mnb_matmul_ex(ctypes.byref(a))


@pytest.mark.parametrize("kw", [
    dict(bits=3), dict(block_size=48), dict(block_size=8), dict(N=0), dict(K=0), dict(M=-1),
    dict(act_dtype=7), dict(out_dtype=-1), dict(scale_dtype=3), dict(accuracy_level=5),
    dict(x=0), dict(packed_b=0), dict(scales=0), dict(y=0), dict(x=FAKE + 8), dict(y=FAKE + 4),
    dict(packed_b=FAKE + 16), dict(scales=FAKE + 1), dict(g_idx=FAKE + 2),
])
def test_matmul_ex_rejects_invalid_arguments(lib, kw):
    assert _ex(lib, **kw) == mnb.MNB_ERR_INVALID_ARG


def test_matmul_m0_is_noop(lib):
    assert _ex(lib, M=0, x=0, y=0) == mnb.MNB_OK


def test_other_entry_points_reject_invalid(lib):
    assert lib.mnb_pack_weights(FAKE, FAKE, 1 << 30, 64, 64, 5, 32, None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_pack_weights(None, FAKE, 1 << 30, 64, 64, 4, 32, None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_pack_weights(FAKE, FAKE + 16, 1 << 30, 64, 64, 4, 32, None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_pack_weights(FAKE, FAKE, 100, 64, 64, 4, 32, None) == mnb.MNB_ERR_NO_MEM
    assert lib.mnb_unpack_codes(FAKE, None, 64, 64, 4, 32, None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_dequantize(FAKE, FAKE, None, FAKE + 2, 64, 64, 4, 32, 1, None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_quantize_activations(FAKE, FAKE, FAKE, 1, 64, 24, 2, None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_workspace_size(1, 64, 64, 4, 32, 0) == 0


def test_status_strings(lib):
    for s in range(7):
        assert mnb.mnb_status_string(s)
    assert mnb.mnb_kernel_name(3) == "gemm_tc"


def _grouped(lib, **kw):
    d = dict(x=FAKE, ids=FAKE, packed_b=FAKE, scales=FAKE, zp=None, y=FAKE, T=4, S=2, E=8, x_per_slot=0, N=64,
             K=64, bits=4, block_size=32, act=2, out=2, sc=1)
    d.update(kw)
    return lib.mnb_matmul_grouped(d["x"], d["ids"], d["packed_b"], d["scales"], d["zp"], d["y"], d["T"], d["S"],
                                  d["E"], d["x_per_slot"], d["N"], d["K"], d["bits"], d["block_size"], d["act"],
                                  d["out"], d["sc"], None)


@pytest.mark.parametrize("kw,want", [
    (dict(S=0), mnb.MNB_ERR_INVALID_ARG), (dict(E=0), mnb.MNB_ERR_INVALID_ARG), (dict(T=-1), mnb.MNB_ERR_INVALID_ARG),
    (dict(x_per_slot=2), mnb.MNB_ERR_INVALID_ARG), (dict(bits=3), mnb.MNB_ERR_INVALID_ARG),
    (dict(act=5), mnb.MNB_ERR_INVALID_ARG), (dict(ids=0), mnb.MNB_ERR_INVALID_ARG),
    (dict(ids=FAKE + 2), mnb.MNB_ERR_INVALID_ARG), (dict(x=FAKE + 8), mnb.MNB_ERR_INVALID_ARG),
    (dict(packed_b=FAKE + 16), mnb.MNB_ERR_INVALID_ARG), (dict(act=0), mnb.MNB_ERR_UNSUPPORTED),
    (dict(E=1025), mnb.MNB_ERR_UNSUPPORTED), (dict(T=4097, S=1), mnb.MNB_ERR_UNSUPPORTED),
    (dict(T=1 << 40, S=1 << 30), mnb.MNB_ERR_UNSUPPORTED), (dict(T=2048, S=3), mnb.MNB_ERR_UNSUPPORTED),
    (dict(T=0, x=0, y=0), mnb.MNB_OK),
])
def test_grouped_rejects_invalid_arguments_on_the_host(lib, kw, want):
    assert _grouped(lib, **kw) == want


def _host_io(lib, **kw):
    a = mnb.MatmulArgs()
    d = dict(x=FAKE, packed_b=FAKE, scales=FAKE, y=FAKE, M=1, N=64, K=64, bits=4, block_size=32,
             act_dtype=2, out_dtype=2, scale_dtype=1, bias_dtype=0, accuracy_level=0, kernel=0)
    d.update(kw)
    for k, v in d.items():
        setattr(a, k, v)
    return lib.mnb_matmul_host_io(ctypes.byref(a))


@pytest.mark.parametrize("kw,want", [
    (dict(bits=3), mnb.MNB_ERR_INVALID_ARG), (dict(act_dtype=9), mnb.MNB_ERR_INVALID_ARG),
    (dict(M=-1), mnb.MNB_ERR_INVALID_ARG), (dict(x=0), mnb.MNB_ERR_INVALID_ARG), (dict(y=0), mnb.MNB_ERR_INVALID_ARG),
    (dict(x=FAKE + 4), mnb.MNB_ERR_INVALID_ARG), (dict(y=FAKE + 8), mnb.MNB_ERR_INVALID_ARG),
    (dict(M=17, K=1 << 18), mnb.MNB_ERR_NO_MEM),                   # 17 x 256 Ki bf16 > 8 MiB
    (dict(M=9, K=1 << 18, act_dtype=0), mnb.MNB_ERR_NO_MEM),       # f32 X counts 4 bytes per element
    (dict(M=0, x=0, y=0), mnb.MNB_OK),
])
def test_host_io_rejects_invalid_arguments_on_the_host(lib, kw, want):
    assert _host_io(lib, **kw) == want
    assert lib.mnb_matmul_host_io(None) == mnb.MNB_ERR_INVALID_ARG


@pytest.mark.parametrize("N,K,bits,bs", [(4096, 4096, 4, 32), (77, 1000, 2, 64), (300, 11008, 8, 128), (16, 17, 4, 16)])
def test_act_order_packed_size(N, K, bits, bs):
    """The act-order pack adds the permutation, one int32 per padded depth, in whole 256-byte units."""
    kpad = -(-K // bs) * bs
    assert mnb.mnb_packed_size_gidx(N, K, bits, bs) == mnb.mnb_packed_size(N, K, bits, bs) + -(-(4 * kpad) // 256) * 256
    assert mnb.mnb_packed_size_gidx(N, K, 3, bs) == 0


def test_act_order_pack_rejects_invalid_before_cuda():
    """Argument errors of mnb_pack_weights_gidx come back before any CUDA call."""
    lib = mnb.load()
    assert lib.mnb_pack_weights_gidx(None, None, None, 0, 16, 64, 4, 32, None) == mnb.MNB_ERR_INVALID_ARG
    assert lib.mnb_pack_weights_gidx(None, None, None, 0, 16, 64, 5, 32, None) == mnb.MNB_ERR_INVALID_ARG


def test_act_order_workspace_size():
    """The act-order prefill's workspace: X in the pack's depth order (M * K 16-bit values, whole 256-byte units)
    for M > 8 with MNB_FLAG_KPERM; otherwise mnb_workspace_size."""
    assert mnb.mnb_workspace_size_ex(512, 4096, 4096, 4, 32, 0, mnb.MNB_FLAG_KPERM) == 512 * 4096 * 2
    assert mnb.mnb_workspace_size_ex(17, 100, 1000, 4, 128, 0, mnb.MNB_FLAG_KPERM) == -(-(17 * 1000 * 2) // 256) * 256
    assert mnb.mnb_workspace_size_ex(8, 4096, 4096, 4, 32, 0, mnb.MNB_FLAG_KPERM) == 0
    assert mnb.mnb_workspace_size_ex(512, 4096, 4096, 4, 32, 0, 0) == 0
    assert mnb.mnb_workspace_size_ex(512, 4096, 4096, 4, 32, 4, 0) == mnb.mnb_workspace_size(512, 4096, 4096, 4, 32, 4)

