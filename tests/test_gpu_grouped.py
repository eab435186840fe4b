"""mnb_matmul_grouped (mixture-of-experts grouped GEMV, one launch over all
experts) against oracle.matmul_grouped, element by element, through the C
ABI.  Covers top-k and repeated routing, many mostly idle experts, S = 1
(one expert per row), more rows per expert than one 16-row chunk, K-split
clusters, ragged K, per-slot activation rows, the full-size MoE decode
workload, out-of-range ids (reported, rows left alone) and the host-side
limits."""
import numpy as np
import pytest
import torch

from block_quantized_weight_matmulnbits_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

F16, BF16, F32 = wl.F16, wl.BF16, wl.F32


class Grouped:
    """One grouped instance on the device: E packed experts back to back."""

    def __init__(self, mnb, w: wl.MoeWorkload):
        from tests import _gpu as G
        self.w, self.G, self.mnb = w, G, mnb
        self.d = d = wl.generate_moe(w)
        self.x = G.to_dev(d["x"], w.act_dtype)
        self.ids = torch.from_numpy(d["ids"]).cuda()
        self.s = G.to_dev(d["scales"], w.scale_dtype)
        self.zp = None if d["zp"] is None else torch.from_numpy(np.ascontiguousarray(d["zp"])).cuda()
        self.ps = mnb.mnb_packed_size(w.N, w.K, w.bits, w.bs)
        assert self.ps % 256 == 0
        self.packed = G.aligned_empty(w.E * self.ps)
        for e in range(w.E):
            be = torch.from_numpy(np.ascontiguousarray(d["b"][e])).cuda()
            mnb.mnb_pack_weights(be, self.packed[e * self.ps:(e + 1) * self.ps], w.N, w.K, w.bits, w.bs)
        torch.cuda.synchronize()

    def run(self, ids=None, y=None):
        w = self.w
        if y is None:
            y = torch.empty((w.T, w.S, w.N), dtype=self.G.TORCH_DT[w.out_dtype], device="cuda")
        self.mnb.mnb_matmul_grouped(self.x, self.ids if ids is None else ids, self.packed, self.s, self.zp, y,
                                    w.T, w.S, w.E, w.N, w.K, w.bits, w.bs, w.act_dtype, w.out_dtype,
                                    w.scale_dtype, x_per_slot=w.x_per_slot)
        torch.cuda.synchronize()
        return y

    def oracle(self, oracle_mod, ids=None):
        w, d = self.w, self.d
        return oracle_mod.matmul_grouped(wl.widen_f64(d["x"], w.act_dtype), d["ids"] if ids is None else ids,
                                         d["b"], wl.widen_f32(d["scales"], w.scale_dtype), d["zp"], w.E, w.N, w.K,
                                         w.bits, w.bs, x_per_slot=w.x_per_slot)


def _w(name, T, S, E, N, K, bits, bs, act, out, sd, zp, seed, **kw):
    return wl.MoeWorkload(name, T, S, E, N, K, bits, bs, act, out, sd, zp=zp, scale_lo=0.01, scale_hi=0.05,
                          seed=seed, **kw)


CASES = [
    _w("top2_t4_e8_int4", 4, 2, 8, 300, 4096, 4, 32, BF16, BF16, F16, (0, 15), 91),
    _w("repeat_t16_s4_e8_int2", 16, 4, 8, 200, 1024, 2, 64, F16, F16, F16, None, 92, ids="repeat"),
    _w("idle_t3_s2_e64_int8_ragged_perslot", 3, 2, 64, 130, 1000, 8, 16, F16, F32, F16, (100, 150), 93,
       x_per_slot=True),
    _w("ksplit_t1_s8_e16_int8", 1, 8, 16, 96, 11008, 8, 128, BF16, BF16, F32, (120, 136), 94),
    _w("chunks_t40_s2_e4_int4", 40, 2, 4, 64, 512, 4, 32, BF16, F32, BF16, (0, 15), 95),
    _w("rows_s1_t6_e3_int4", 6, 1, 3, 48, 256, 4, 16, F16, F16, F16, None, 96),
    _w("dupes_t5_s4_e2_int4_perslot", 5, 4, 2, 40, 384, 4, 128, BF16, BF16, F16, (0, 15), 97, ids="repeat",
       x_per_slot=True),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("sched", ["auto", "tile"])
def test_grouped_matches_oracle(mnb, oracle_mod, monkeypatch, w, sched):
    """Both schedules: the K-chunk grouped mode (at most 8 pairs, the default) and the per-tile kernel."""
    if sched == "tile":
        monkeypatch.setenv("MNB_MOE_SCHED", "tile")
    P = Grouped(mnb, w)
    y = P.run()
    y_ref, mag = P.oracle(oracle_mod)
    y64 = P.G.to_host_f64(y, w.out_dtype).reshape(w.T, w.S, w.N)
    P.G.assert_within(y64, y_ref, mag, w.out_dtype, w.name)


def test_grouped_full_size_moe_decode(mnb, oracle_mod):
    w = wl.MOE_CONFIGS[0]
    P = Grouped(mnb, w)
    y = P.run()
    y_ref, mag = P.oracle(oracle_mod)
    P.G.assert_within(P.G.to_host_f64(y, w.out_dtype).reshape(w.T, w.S, w.N), y_ref, mag, w.out_dtype, w.name)


def test_grouped_is_deterministic(mnb):
    P = Grouped(mnb, CASES[1])
    a, b = P.run(), P.run()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_out_of_range_ids_are_reported_and_their_rows_left_alone(mnb, oracle_mod):
    w = CASES[0]
    P = Grouped(mnb, w)
    assert mnb.mnb_get_device_error() == 0
    ids = P.d["ids"].copy()
    ids[1, 0] = w.E
    ids[3, 1] = -1
    y = torch.full((w.T, w.S, w.N), 7.0, dtype=P.G.TORCH_DT[w.out_dtype], device="cuda")
    P.run(ids=torch.from_numpy(ids).cuda(), y=y)
    assert mnb.mnb_get_device_error() == mnb.MNB_ERR_INVALID_ARG
    assert mnb.mnb_get_device_error() == 0  # read and cleared
    y64 = P.G.to_host_f64(y, w.out_dtype).reshape(w.T, w.S, w.N)
    assert np.all(y64[1, 0] == 7.0) and np.all(y64[3, 1] == 7.0)
    keep = np.ones((w.T, w.S), dtype=bool)
    keep[1, 0] = keep[3, 1] = False
    ids_ok = np.where(keep, ids, 0)
    y_ref, mag = P.oracle(oracle_mod, ids=ids_ok)
    P.G.assert_within(y64[keep], y_ref[keep], mag[keep], w.out_dtype, "valid rows")


def test_grouped_host_side_limits(mnb):
    from tests import _gpu as G
    x = torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    packed = G.aligned_empty(mnb.mnb_packed_size(16, 64, 4, 32))
    s = torch.ones((1, 16, 2), dtype=torch.float16, device="cuda")
    y = torch.empty((1, 1, 16), dtype=torch.bfloat16, device="cuda")
    args = (x, ids, packed, s, None, y)
    mnb.mnb_matmul_grouped(*args, 0, 1, 1, 16, 64, 4, 32, BF16, BF16, F16)  # T = 0: nothing to do
    for T, S, E, act, want in ((4097, 1, 1, BF16, mnb.MNB_ERR_UNSUPPORTED),   # T*S beyond the pair list
                               (1, 1, 1025, BF16, mnb.MNB_ERR_UNSUPPORTED),   # E beyond the bitmap
                               (1, 1, 1, F32, mnb.MNB_ERR_UNSUPPORTED),       # f32 activations
                               (1, 0, 1, BF16, mnb.MNB_ERR_INVALID_ARG)):
        with pytest.raises(mnb.MnbError) as e:
            mnb.mnb_matmul_grouped(*args, T, S, E, 16, 64, 4, 32, act, BF16, F16)
        assert e.value.status == want
    torch.cuda.synchronize()
