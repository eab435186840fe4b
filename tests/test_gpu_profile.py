"""MNB_PROFILE=1: the per-call timers of the C entry points.  They stand in for
the CPU operator's env-gated phase timers, printed every 512 calls
(onnx-runtime-ep-cpu 0.1.0-dev.5, src/kernels/matmul_nbits.rs, mm_profile).
Each kernel family gets one stderr line every MNB_PROFILE_EVERY calls, carrying
its host and device time per call.  Profiling changes no result."""
import re

import numpy as np
import pytest
import torch

import block_quantized_weight_matmulnbits_gb300 as mnb_mod
from block_quantized_weight_matmulnbits_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

F32, F16, BF16 = wl.F32, wl.F16, wl.BF16
LINE = re.compile(r"\[mnb profile\] kernel=(\S+) calls=(\d+) host_us_per_call=([\d.]+) "
                  r"device_us_per_call=([\d.]+) timed_calls=(\d+)")


@pytest.fixture(scope="module")
def mnb():
    mnb_mod.load()
    return mnb_mod


@pytest.fixture(scope="module")
def G(mnb):
    from tests import _gpu
    return _gpu


def _problem(G, M, N, K):
    w = wl.Workload(f"prof{M}x{N}x{K}", M, N, K, 4, 32, BF16, BF16, F16, scale_lo=0.01, scale_hi=0.05,
                    zp=(0, 15), seed=3100 + M)
    return G.Problem(w)


def _lines(err):
    return [LINE.match(l).groups() for l in err.splitlines() if LINE.match(l)]


def test_profile_reports_each_family(G, mnb, monkeypatch, capfd):
    """Decode (gemv_mma) and prefill (gemm_tc) calls are counted per family. Every 4th call of a family prints a
    line whose counts match, whose times are positive, and whose calls were all timed on the device. Results stay
    bit-identical to unprofiled calls."""
    dec, pre = _problem(G, 1, 512, 1024), _problem(G, 64, 256, 1024)
    y_dec0, y_pre0 = dec.run(), pre.run()
    capfd.readouterr()
    monkeypatch.setenv("MNB_PROFILE", "1")
    monkeypatch.setenv("MNB_PROFILE_EVERY", "4")
    for _ in range(8):
        y_dec = dec.run()
    for _ in range(4):
        y_pre = pre.run()
    monkeypatch.delenv("MNB_PROFILE")
    dec.run()  # not counted
    err = capfd.readouterr().err
    got = _lines(err)
    fams = {}
    for fam, calls, host_us, dev_us, timed in got:
        fams.setdefault(fam, []).append((int(calls), float(host_us), float(dev_us), int(timed)))
    # counts are per process: the lines of this test are 4 calls apart, each of them timed on the device
    dec_rows, pre_rows = fams["gemv_mma"], fams["gemm_tc"]
    assert len(dec_rows) == 2 and dec_rows[1][0] - dec_rows[0][0] == 4, err
    assert dec_rows[1][3] - dec_rows[0][3] == 4, err
    assert len(pre_rows) == 1 and pre_rows[0][0] % 4 == 0, err
    for rows in fams.values():
        for calls, host_us, dev_us, timed in rows:
            assert calls % 4 == 0 and host_us > 0 and dev_us > 0 and 0 < timed <= calls
    assert torch.equal(y_dec.view(torch.int16), y_dec0.view(torch.int16))
    assert torch.equal(y_pre.view(torch.int16), y_pre0.view(torch.int16))


def test_profile_skips_device_timing_under_graph_capture(G, mnb, monkeypatch, capfd):
    """Calls captured into a CUDA graph are counted but not timed on the device (no events are recorded in a
    capture). The replayed graph gives the same result as an eager call."""
    P = _problem(G, 1, 256, 512)
    y_ref = P.run()
    y = torch.empty_like(y_ref)
    capfd.readouterr()
    monkeypatch.setenv("MNB_PROFILE", "1")
    monkeypatch.setenv("MNB_PROFILE_EVERY", "2")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    w = P.w
    with torch.cuda.graph(g, stream=s):
        for _ in range(2):
            mnb.mnb_matmul_ex(P.x, P.packed, P.s, P.zp, y, w.M, w.N, w.K, w.bits, w.bs, w.act_dtype, w.out_dtype,
                              w.scale_dtype, stream=s.cuda_stream)
    monkeypatch.delenv("MNB_PROFILE")
    g.replay()
    torch.cuda.synchronize()
    got = _lines(capfd.readouterr().err)
    assert any(f == "gemv_mma" and int(c) >= 2 and int(t) < int(c) for f, c, _, _, t in got), got
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))


def test_profile_fp_path_and_failed_calls(G, mnb, monkeypatch, capfd):
    """The FP8 decode is counted under its own family; a rejected call (bad alignment) is not counted."""
    N, K = 256, 512
    rng = np.random.default_rng(7)
    codes = torch.from_numpy(rng.integers(0, 256, size=(K, N), dtype=np.uint8)).cuda()
    packed = G.aligned_empty(mnb.mnb_fp_packed_size(N, K, mnb.MNB_WF_E4M3))
    mnb.mnb_pack_fp_weights(codes, packed, N, K, mnb.MNB_WF_E4M3)
    scales = torch.full((N,), 0.01, dtype=torch.float32, device="cuda")
    x = torch.randn((1, K), device="cuda").to(torch.bfloat16)
    y = torch.empty((1, N), dtype=torch.bfloat16, device="cuda")
    monkeypatch.setenv("MNB_PROFILE", "1")
    monkeypatch.setenv("MNB_PROFILE_EVERY", "3")
    capfd.readouterr()
    for _ in range(3):
        mnb.mnb_matmul_fp(x, packed, scales, 1.0, y, 1, N, K, mnb.MNB_WF_E4M3, BF16, BF16)
    torch.cuda.synchronize()
    P = _problem(G, 1, 256, 512)
    bad = torch.empty((1, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mnb.MnbError):  # y 2 bytes past a 16-byte boundary
        mnb.mnb_matmul_ex(P.x, P.packed, P.s, P.zp, bad.view(-1)[1:].view(1, 255), 1, 255, 512, 4, 32, BF16, BF16,
                          F16)
    got = _lines(capfd.readouterr().err)
    assert any(f in ("gemv_fp", "gemv_nv") and c == "3" for f, c, *_ in got), got
    assert not any(c == "0" for _, c, *_ in got)
