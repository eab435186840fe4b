"""mnb_matmul_a8_static (int8-activation matmul on a file-scope device scratch
array, no caller workspace) against mnb_matmul_ex with a caller workspace,
through the C ABI.  Collected last on purpose: it must pass alone and after
every other test has used the device."""
import numpy as np
import pytest
import torch

from block_quantized_weight_matmulnbits_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

F16, BF16, F32 = wl.F16, wl.BF16, wl.F32

CASES = [
    wl.Workload("ns_m1_n300_k4096_int4", 1, 300, 4096, 4, 32, BF16, BF16, F16, zp=(0, 15), scale_lo=0.01,
                scale_hi=0.05, seed=71),
    wl.Workload("ns_m8_n96_k1536_int8", 8, 96, 1536, 8, 128, F16, F16, F32, zp=(120, 136), scale_lo=1e-3,
                scale_hi=1e-2, seed=72),
    wl.Workload("ns_m3_n45_k300_int2", 3, 45, 300, 2, 16, BF16, F32, BF16, zp=(0, 3), scale_lo=0.01,
                scale_hi=0.05, seed=73),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_static_scratch_matches_workspace_entry(mnb, oracle_mod, w):
    from tests import _gpu as G
    P = G.Problem(w)
    ws = G.aligned_empty(mnb.mnb_workspace_size(w.M, w.N, w.K, w.bits, w.bs, 4))
    y_ref = P.y64(P.run(accuracy_level=4, workspace=ws))
    qa, sa = oracle_mod.quantize_act(P.x64.astype(np.float32), w.K, w.bs)
    _, mag = oracle_mod.matmul_a8(qa, sa, P.d["b"], P.s32, P.d["zp"], w.N, w.K, w.bits, w.bs)
    y_ws = P.run(accuracy_level=4, workspace=ws)
    for call in range(2):  # two calls in a row reuse the same scratch
        y = torch.full((w.M, w.N), float("nan"), dtype=G.TORCH_DT[w.out_dtype], device="cuda")
        mnb.mnb_matmul_a8_static(P.x, P.packed, P.s, P.zp, y, w.M, w.N, w.K, w.bits, w.bs, w.act_dtype,
                                 w.out_dtype, w.scale_dtype)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: bit-identical to the workspace call
        assert torch.equal(y.view(torch.int16 if y.element_size() == 2 else torch.int32),
                           y_ws.view(torch.int16 if y_ws.element_size() == 2 else torch.int32)), \
            f"static scratch call {call} differs from the workspace call"
        G.assert_within(P.y64(y), y_ref, mag, w.out_dtype, f"static scratch call {call}")


def test_static_scratch_rejects_sizes_beyond_its_maximum(mnb):
    from tests import _gpu as G
    M, N, K = 16, 32, 1 << 16  # 16 rows x 64 Ki int8 activations = 1 MiB, plus the block scales
    assert mnb.mnb_workspace_size(M, N, K, 4, 32, 4) > mnb.MNB_A8_STATIC_SCRATCH_BYTES
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    packed = G.aligned_empty(mnb.mnb_packed_size(N, K, 4, 32))
    s = torch.ones((N, K // 32), dtype=torch.float16, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mnb.MnbError) as e:
        mnb.mnb_matmul_a8_static(x, packed, s, None, y, M, N, K, 4, 32, BF16, BF16, F16)
    assert e.value.status == mnb.MNB_ERR_NO_MEM
