"""mnb_matmul_host_io (X and Y in page-locked host memory, moved by the
library's own kernels) through the C ABI: bit-identical to mnb_matmul_ex on
device buffers for every kernel family, within the oracle's tolerance, fresh
host data on every call (also under CUDA-graph replay), and host-side
rejection of pageable memory and of X larger than the staging array."""
import numpy as np
import pytest
import torch

from block_quantized_weight_matmulnbits_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

F16, BF16, F32 = wl.F16, wl.BF16, wl.F32

# (workload, accuracy level); each row reaches a different kernel family
CASES = [
    (wl.Workload("hio_m1_n300_k4096_int4_zp", 1, 300, 4096, 4, 32, BF16, BF16, F16, zp=(0, 15), scale_lo=0.01,
                 scale_hi=0.05, seed=81), 0),                                     # gemv_mma, per-tile
    (wl.Workload("hio_m8_n200_k2048_int2", 8, 200, 2048, 2, 64, F16, F16, F16, zp=None, scale_lo=0.01,
                 scale_hi=0.05, seed=82), 0),                                     # gemv_mma
    (wl.Workload("hio_m1_n96_k1000_int8_f32x", 1, 96, 1000, 8, 128, F32, F32, F32, zp=(120, 136),
                 scale_lo=1e-3, scale_hi=1e-2, seed=83), 0),                      # gemv (f32 X), ragged K
    (wl.Workload("hio_m3_n45_k300_int4_f32x", 3, 45, 300, 4, 16, F32, BF16, BF16, zp=(0, 15), scale_lo=0.01,
                 scale_hi=0.05, seed=84), 0),                                     # generic
    (wl.Workload("hio_m80_n256_k512_int4", 80, 256, 512, 4, 32, BF16, BF16, BF16, zp=(0, 15), scale_lo=0.01,
                 scale_hi=0.05, seed=85), 0),                                     # tcgen05 GEMM
    (wl.Workload("hio_m2_n130_k1536_int4_a8", 2, 130, 1536, 4, 32, F16, F16, F16, zp=(0, 15), scale_lo=0.01,
                 scale_hi=0.05, seed=86), 4),                                     # int8-activation path
]


def _pinned_like(t):
    return torch.empty(t.shape, dtype=t.dtype).pin_memory()


def _bits(t):
    """The raw bit patterns of a host or device tensor, on the host."""
    t = t.detach().cpu()
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


@pytest.mark.parametrize("w,acc", CASES, ids=lambda c: c.name if hasattr(c, "name") else f"acc{c}")
def test_host_io_matches_device_call(mnb, w, acc):
    from tests import _gpu as G
    P = G.Problem(w)
    ws_bytes = mnb.mnb_workspace_size(w.M, w.N, w.K, w.bits, w.bs, acc)
    ws = G.aligned_empty(ws_bytes) if ws_bytes else None
    y_dev = P.run(accuracy_level=acc, workspace=ws)
    xh = _pinned_like(P.x)
    xh.copy_(P.x.cpu())
    yh = torch.full((w.M, w.N), float("nan"), dtype=G.TORCH_DT[w.out_dtype]).pin_memory()
    mnb.mnb_matmul_host_io(xh, P.packed, P.s, P.zp, yh, w.M, w.N, w.K, w.bits, w.bs, w.act_dtype, w.out_dtype,
                           w.scale_dtype, accuracy_level=acc, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(_bits(yh), _bits(y_dev))
    if acc == 0:
        y_ref, mag = P.oracle_full()
        G.assert_within(P.y64(yh), y_ref, mag, w.out_dtype, "host io vs oracle")


def test_host_io_reads_fresh_host_data_each_call_and_under_graph_replay(mnb):
    from tests import _gpu as G
    w = CASES[0][0]
    P = G.Problem(w)
    rng = np.random.default_rng(87)
    xs = [P.x]
    for _ in range(3):
        xs.append(P.x[:, torch.from_numpy(rng.permutation(w.K)).cuda()].contiguous())
    refs = []
    for x in xs:
        y = torch.empty((w.M, w.N), dtype=G.TORCH_DT[w.out_dtype], device="cuda")
        mnb.mnb_matmul_ex(x, P.packed, P.s, P.zp, y, w.M, w.N, w.K, w.bits, w.bs, w.act_dtype, w.out_dtype,
                          w.scale_dtype)
        refs.append(y.cpu())
    torch.cuda.synchronize()
    xh = _pinned_like(P.x)
    yh = torch.empty((w.M, w.N), dtype=G.TORCH_DT[w.out_dtype]).pin_memory()
    stream = torch.cuda.Stream()

    def call():
        mnb.mnb_matmul_host_io(xh, P.packed, P.s, P.zp, yh, w.M, w.N, w.K, w.bits, w.bs, w.act_dtype,
                               w.out_dtype, w.scale_dtype, stream=stream)

    for x, ref in zip(xs, refs):  # eager calls: the host rewrites X between calls
        xh.copy_(x.cpu())
        with torch.cuda.stream(stream):
            call()
        stream.synchronize()
        assert torch.equal(_bits(yh), _bits(ref))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call()
    for x, ref in zip(reversed(xs), reversed(refs)):  # graph replays
        xh.copy_(x.cpu())
        yh.fill_(float("nan"))
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        assert torch.equal(_bits(yh), _bits(ref))


def test_host_io_rejects_pageable_memory_without_launching(mnb):
    from tests import _gpu as G
    w = CASES[0][0]
    P = G.Problem(w)
    x_pageable = P.x.cpu()
    y_pinned = torch.empty((w.M, w.N), dtype=torch.bfloat16).pin_memory()
    y_pageable = torch.empty((w.M, w.N), dtype=torch.bfloat16)
    for x, y in ((x_pageable, y_pinned), (_pinned_like(P.x), y_pageable)):
        with pytest.raises(mnb.MnbError) as e:
            mnb.mnb_matmul_host_io(x, P.packed, P.s, P.zp, y, w.M, w.N, w.K, w.bits, w.bs, w.act_dtype,
                                   w.out_dtype, w.scale_dtype)
        assert e.value.status == mnb.MNB_ERR_INVALID_ARG
    torch.cuda.synchronize()


def test_host_io_rejects_x_beyond_the_staging_array(mnb):
    from tests import _gpu as G
    M, N, K = 16, 32, 1 << 18  # 16 x 256 Ki bf16 = 8 MiB + 0: exactly the limit, then one row more
    assert M * K * 2 == mnb.MNB_HOST_IO_X_BYTES
    xh = torch.empty(16, dtype=torch.uint8).pin_memory()  # never read: the size check comes first
    yh = torch.empty(16, dtype=torch.uint8).pin_memory()
    packed = G.aligned_empty(256)
    s = torch.empty(1, dtype=torch.float16, device="cuda")
    with pytest.raises(mnb.MnbError) as e:
        mnb.mnb_matmul_host_io(xh, packed, s, None, yh, M + 1, N, K, 4, 32, BF16, BF16, F16)
    assert e.value.status == mnb.MNB_ERR_NO_MEM


@pytest.mark.parametrize("case", [0, 5], ids=["gemv_mma", "int8_path"])
def test_host_io_pdl_back_to_back_calls_without_syncs(mnb, case):
    """MNB_FLAG_PDL: each call's X fetch may start before the previous call's
    matmul has finished.  Six calls issued back to back (eager, then twice in
    one captured graph), each with its own host X and Y, must each give the
    device-buffer call's result."""
    from tests import _gpu as G
    w, acc = CASES[case]
    P = G.Problem(w)
    ws_bytes = mnb.mnb_workspace_size(w.M, w.N, w.K, w.bits, w.bs, acc)
    ws = G.aligned_empty(ws_bytes) if ws_bytes else None
    rng = np.random.default_rng(88)
    n = 6
    xs = [P.x] + [P.x[:, torch.from_numpy(rng.permutation(w.K)).cuda()].contiguous() for _ in range(n - 1)]
    refs = []
    for x in xs:
        y = torch.empty((w.M, w.N), dtype=G.TORCH_DT[w.out_dtype], device="cuda")
        mnb.mnb_matmul_ex(x, P.packed, P.s, P.zp, y, w.M, w.N, w.K, w.bits, w.bs, w.act_dtype, w.out_dtype,
                          w.scale_dtype, accuracy_level=acc, workspace=ws)
        refs.append(y.cpu())
    torch.cuda.synchronize()
    xhs = [_pinned_like(P.x) for _ in range(n)]
    for xh, x in zip(xhs, xs):
        xh.copy_(x.cpu())
    yhs = [torch.empty((w.M, w.N), dtype=G.TORCH_DT[w.out_dtype]).pin_memory() for _ in range(n)]
    stream = torch.cuda.Stream()

    def calls():
        for xh, yh in zip(xhs, yhs):
            mnb.mnb_matmul_host_io(xh, P.packed, P.s, P.zp, yh, w.M, w.N, w.K, w.bits, w.bs, w.act_dtype,
                                   w.out_dtype, w.scale_dtype, accuracy_level=acc, workspace=ws, stream=stream,
                                   flags=mnb.MNB_FLAG_PDL)

    def check():
        for i, (yh, ref) in enumerate(zip(yhs, refs)):
            assert torch.equal(_bits(yh), _bits(ref)), f"call {i}"

    for yh in yhs:
        yh.fill_(float("nan"))
    with torch.cuda.stream(stream):
        calls()
    stream.synchronize()
    check()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        calls()
    for _ in range(2):
        for yh in yhs:
            yh.fill_(float("nan"))
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        check()
