"""GPU-test helpers: move seeded inputs to the device, run the library through
its binding, and compare with the oracle.  Test code only."""
import numpy as np
import torch

import block_quantized_weight_matmulnbits_gb300 as mnb
import oracle
from block_quantized_weight_matmulnbits_gb300 import workloads as wl
from tests._golden import tolerance

TORCH_DT = {wl.F32: torch.float32, wl.F16: torch.float16, wl.BF16: torch.bfloat16}


def to_dev(stored, dtype):
    a = np.ascontiguousarray(stored)
    if dtype == wl.F32:
        return torch.from_numpy(a.astype(np.float32)).cuda()
    return torch.from_numpy(a.view(np.int16)).cuda().view(TORCH_DT[dtype])


def to_host_f64(t, dtype):
    t = t.detach().cpu()
    if dtype == wl.F32:
        return t.numpy().astype(np.float64)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    return wl.widen_f64(bits, dtype)


def aligned_empty(nbytes, align=256):
    """A uint8 CUDA tensor whose data pointer is `align`-byte aligned."""
    raw = torch.empty(nbytes + align, dtype=torch.uint8, device="cuda")
    off = (-raw.data_ptr()) % align
    return raw[off:off + nbytes]


class Problem:
    """One MatMulNBits instance: host inputs, device tensors and the packed weight."""

    def __init__(self, w: wl.Workload, data=None):
        self.w = w
        self.d = data if data is not None else wl.generate(w)
        d = self.d
        self.x = to_dev(d["x"], w.act_dtype)
        self.b = torch.from_numpy(np.ascontiguousarray(d["b"])).cuda()
        self.s = to_dev(d["scales"], w.scale_dtype)
        self.zp = None if d["zp"] is None else torch.from_numpy(np.ascontiguousarray(d["zp"])).cuda()
        nbytes = mnb.mnb_packed_size(w.N, w.K, w.bits, w.bs)
        self.packed = aligned_empty(nbytes)
        mnb.mnb_pack_weights(self.b, self.packed, w.N, w.K, w.bits, w.bs)
        self.x64 = wl.widen_f64(d["x"], w.act_dtype)
        self.s32 = wl.widen_f32(d["scales"], w.scale_dtype)

    def run(self, kernel="auto", y=None, **kw):
        w = self.w
        if y is None:
            y = torch.empty((w.M, w.N), dtype=TORCH_DT[w.out_dtype], device="cuda")
        mnb.mnb_matmul_ex(self.x, self.packed, self.s, self.zp, y, w.M, w.N, w.K, w.bits, w.bs, w.act_dtype,
                          w.out_dtype, w.scale_dtype, kernel=kernel, **kw)
        torch.cuda.synchronize()
        return y

    def y64(self, y):
        return to_host_f64(y, self.w.out_dtype)

    def oracle_full(self, **kw):
        w = self.w
        return oracle.matmul(self.x64, self.d["b"], self.s32, self.d["zp"], w.N, w.K, w.bits, w.bs, **kw)

    def oracle_points(self, ms, ns, **kw):
        w = self.w
        return oracle.matmul_points(self.x64, self.d["b"], self.s32, self.d["zp"], w.N, w.K, w.bits, w.bs,
                                    ms, ns, **kw)


def assert_within(y, y_ref, absdot, out_dtype, what=""):
    tol = tolerance(y_ref, absdot, out_dtype)
    err = np.abs(y - y_ref)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {idx.tolist()} "
                             f"y={y[bad][:5]} ref={y_ref[bad][:5]} tol={tol[bad][:5]}")
