"""Failure paths detected on the device, exercised without faulting the GPU.

* A packed buffer whose header does not match the call (packed for another
  K or N, or a wrong magic word): every kernel that reads packed weights
  compares the header with the call's shape and records
  MNB_ERR_LAYOUT_MISMATCH in the device status word.  The mismatched calls
  here ask for a smaller K or N than the buffer was packed for, so every
  read stays inside the buffers.
* A bounded mbarrier wait that runs out: MNB_WAIT_LIMIT=1 makes each wait of
  the tcgen05 GEMM give up after one poll, so the kernel's first wait that is
  not already satisfied returns MNB_ERR_TIMEOUT; the kernel then lets its
  copies and MMAs finish, frees tensor memory and returns, and the next call
  on the device is correct.
"""
import numpy as np
import pytest
import torch

from block_quantized_weight_matmulnbits_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

F32, F16, BF16 = wl.F32, wl.F16, wl.BF16


def _problem(G, M, N, K, bits=4, bs=32, act=BF16, seed=600):
    w = wl.Workload(f"f_m{M}_n{N}_k{K}", M, N, K, bits, bs, act, BF16, F16, zp=(0, (1 << bits) - 1),
                    scale_lo=0.01, scale_hi=0.05, seed=seed)
    return w, G.Problem(w)


@pytest.mark.parametrize("kernel,M", [("gemv_mma", 1), ("gemv_mma", 8), ("gemm_tc", 64), ("generic", 3)])
@pytest.mark.parametrize("change", ["K", "N"])
def test_header_mismatch_sets_layout_status(G, mnb, kernel, M, change):
    w, P = _problem(G, M, 96, 512)
    assert mnb.mnb_get_device_error() == 0
    N2, K2 = (w.N, w.K // 2) if change == "K" else (w.N // 2, w.K)
    x = P.x if change == "N" else P.x[:, :K2].contiguous()
    y = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    mnb.mnb_matmul_ex(x, P.packed, P.s, P.zp, y, M, N2, K2, w.bits, w.bs, w.act_dtype, w.out_dtype,
                      w.scale_dtype, kernel=kernel)
    torch.cuda.synchronize()
    assert mnb.mnb_get_device_error() == mnb.MNB_ERR_LAYOUT_MISMATCH
    # the matching call is clean
    P.run(kernel)
    assert mnb.mnb_get_device_error() == 0


def test_header_mismatch_on_the_exports_and_a_bad_magic(G, mnb):
    w, P = _problem(G, 1, 64, 256)
    bad = P.packed.clone()
    bad[:4] = 0  # the magic word
    out = torch.empty((w.N, w.K), dtype=torch.float32, device="cuda")
    mnb.mnb_dequantize(bad, P.s, P.zp, out, w.N, w.K, w.bits, w.bs, w.scale_dtype)
    torch.cuda.synchronize()
    assert mnb.mnb_get_device_error() == mnb.MNB_ERR_LAYOUT_MISMATCH
    y = torch.empty((1, w.N), dtype=torch.bfloat16, device="cuda")
    mnb.mnb_matmul(P.x, bad, P.s, P.zp, y, 1, w.N, w.K, w.bits, w.bs, w.act_dtype, w.out_dtype, w.scale_dtype)
    torch.cuda.synchronize()
    assert mnb.mnb_get_device_error() == mnb.MNB_ERR_LAYOUT_MISMATCH
    mnb.mnb_dequantize(P.packed, P.s, P.zp, out, w.N, w.K, w.bits, w.bs, w.scale_dtype)
    torch.cuda.synchronize()
    assert mnb.mnb_get_device_error() == 0


def test_bounded_wait_timeout_reports_and_recovers(G, mnb, monkeypatch):
    w, P = _problem(G, 200, 300, 1024, seed=610)
    ref, mag = P.oracle_full()
    assert mnb.mnb_get_device_error() == 0
    monkeypatch.setenv("MNB_WAIT_LIMIT", "1")
    y = torch.full((w.M, w.N), 5.0, dtype=torch.bfloat16, device="cuda")
    mnb.mnb_matmul_ex(P.x, P.packed, P.s, P.zp, y, w.M, w.N, w.K, w.bits, w.bs, w.act_dtype, w.out_dtype,
                      w.scale_dtype, kernel="gemm_tc")
    torch.cuda.synchronize()
    assert mnb.mnb_get_device_error() == mnb.MNB_ERR_TIMEOUT
    monkeypatch.delenv("MNB_WAIT_LIMIT")
    # tensor memory was freed and the device is usable: the same call, twice, is correct
    for _ in range(2):
        y = P.run("gemm_tc")
        G.assert_within(P.y64(y), ref, mag, w.out_dtype, "after a timed-out call")
    assert mnb.mnb_get_device_error() == 0
