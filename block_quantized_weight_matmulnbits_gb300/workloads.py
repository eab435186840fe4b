"""Seeded synthetic inputs for MatMulNBits, shared by the tests, the bench and the smoke check.

This module holds no arithmetic of the method: it only draws random numbers,
rounds them to a storage dtype and returns raw buffers.  Both the CUDA path
and the CPU oracle consume what it returns, and neither is imported here.

Weight codes are drawn as raw bytes.  Codes drawn uniformly over
0 .. 2^bits - 1 and packed least-significant-bits first fill every byte with
independent uniform bits, so a uniform random byte *is* a block of uniform
packed codes; the same holds for zero points drawn over their full range.
A zero-point range narrower than the full code range is only used with 8-bit
codes, where one byte holds one zero point, so no packing is ever done here.

Shapes, dtypes and distributions of the five named workloads are LLM-projection
shaped stand-ins (4096x11008, 11008x4096, 4096x14336, 4096x4096); no trained
weights or datasets are used.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

F32, F16, BF16 = 0, 1, 2
DTYPE_NAMES = {F32: "f32", F16: "f16", BF16: "bf16"}
DTYPE_BYTES = {F32: 4, F16: 2, BF16: 2}
SEED_BASE = 20261202


def to_storage(v64: np.ndarray, dtype: int) -> np.ndarray:
    """Round f64 values to a storage dtype with round-to-nearest-even.

    Returns float32 for F32 and the raw 16-bit patterns (uint16) for F16/BF16.
    """
    v32 = np.asarray(v64, dtype=np.float64).astype(np.float32)
    if dtype == F32:
        return v32
    if dtype == F16:
        return np.asarray(v64, dtype=np.float64).astype(np.float16).view(np.uint16)
    if dtype == BF16:
        u = v32.view(np.uint32).astype(np.uint64)
        rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        return rounded.astype(np.uint16)
    raise ValueError(f"unknown dtype {dtype}")


def widen_f32(stored: np.ndarray, dtype: int) -> np.ndarray:
    """Exact widening of stored values to f32."""
    if dtype == F32:
        return np.asarray(stored, dtype=np.float32)
    if dtype == F16:
        return np.asarray(stored, dtype=np.uint16).view(np.float16).astype(np.float32)
    if dtype == BF16:
        return (np.asarray(stored, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    raise ValueError(f"unknown dtype {dtype}")


def widen_f64(stored: np.ndarray, dtype: int) -> np.ndarray:
    return widen_f32(stored, dtype).astype(np.float64)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    bits: int
    bs: int
    act_dtype: int
    out_dtype: int
    scale_dtype: int
    x_dist: str = "normal"            # "normal" = N(0,1), "uniform" = U(-1,1)
    scale_lo: float = 0.001
    scale_hi: float = 0.01
    zp: Optional[tuple] = None        # None = absent (default zero point), else (lo, hi) inclusive
    seed: int = SEED_BASE

    @property
    def kblocks(self) -> int:
        return -(-self.K // self.bs)

    @property
    def blob(self) -> int:
        return self.bs * self.bits // 8

    @property
    def zp_row_bytes(self) -> int:
        return -(-(self.kblocks * self.bits) // 8)

    def algorithmic_bytes(self) -> int:
        """Bytes a matmul must move once: codes, scales, zero points, X and Y."""
        b = self.N * self.kblocks * self.blob
        s = self.N * self.kblocks * DTYPE_BYTES[self.scale_dtype]
        z = self.N * self.zp_row_bytes if self.zp is not None else 0
        x = self.M * self.K * DTYPE_BYTES[self.act_dtype]
        y = self.M * self.N * DTYPE_BYTES[self.out_dtype]
        return b + s + z + x + y

    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


CONFIGS = [
    Workload("m1_k256_n256_int4_bs32_sym_f32", 1, 256, 256, 4, 32, F32, F32, F32,
             x_dist="uniform", scale_lo=0.005, scale_hi=0.02, zp=None, seed=SEED_BASE + 0),
    Workload("decode_m1_k4096_n11008_int4_bs32_asym_bf16", 1, 11008, 4096, 4, 32, BF16, BF16, F16,
             x_dist="normal", scale_lo=0.001, scale_hi=0.01, zp=(0, 15), seed=SEED_BASE + 1),
    Workload("decode_m1_k11008_n4096_int8_bs128_asym_f16", 1, 4096, 11008, 8, 128, F16, F16, F32,
             x_dist="normal", scale_lo=1e-4, scale_hi=1e-3, zp=(120, 136), seed=SEED_BASE + 2),
    Workload("batch_m8_k4096_n14336_int2_bs64_asym_bf16", 8, 14336, 4096, 2, 64, BF16, BF16, F16,
             x_dist="normal", scale_lo=0.01, scale_hi=0.05, zp=(0, 3), seed=SEED_BASE + 3),
    Workload("prefill_m512_k4096_n4096_int4_bs32_sym_bf16", 512, 4096, 4096, 4, 32, BF16, BF16, F16,
             x_dist="normal", scale_lo=0.001, scale_hi=0.01, zp=None, seed=SEED_BASE + 4),
]


def config(index: int) -> Workload:
    return CONFIGS[index]


def variant(w: Workload, **changes) -> Workload:
    return dataclasses.replace(w, **changes)


def generate(w: Workload, rng: Optional[np.random.Generator] = None) -> dict:
    """Draw one workload's inputs.

    Returns a dict with
      x      : [M, K] storage (float32 or uint16 bit patterns)
      b      : [N, KB, blob] uint8 packed codes (ORT layout)
      scales : [N, KB] storage
      zp     : [N, ceil(KB*bits/8)] uint8 or None
    Draw order is fixed (x, scales, b, zp) so a seed fully determines the data.
    """
    if rng is None:
        rng = np.random.default_rng(w.seed)
    if w.x_dist == "normal":
        x64 = rng.standard_normal((w.M, w.K))
    elif w.x_dist == "uniform":
        x64 = rng.uniform(-1.0, 1.0, (w.M, w.K))
    else:
        raise ValueError(w.x_dist)
    s64 = rng.uniform(w.scale_lo, w.scale_hi, (w.N, w.kblocks))
    b = rng.integers(0, 256, size=(w.N, w.kblocks, w.blob), dtype=np.uint8)
    zp = None
    if w.zp is not None:
        lo, hi = w.zp
        full = (lo == 0 and hi == (1 << w.bits) - 1)
        if full:
            zp = rng.integers(0, 256, size=(w.N, w.zp_row_bytes), dtype=np.uint8)
        elif w.bits == 8:
            zp = rng.integers(lo, hi + 1, size=(w.N, w.zp_row_bytes), dtype=np.uint8)
        else:
            raise ValueError("a partial zero-point range needs packing; draw it in the caller")
    return {
        "x": to_storage(x64, w.act_dtype),
        "b": b,
        "scales": to_storage(s64, w.scale_dtype),
        "zp": zp,
    }


@dataclasses.dataclass(frozen=True)
class MoeWorkload:
    """A grouped (mixture-of-experts) instance: T tokens, S expert slots per
    token, E experts that share one [N, K] weight shape.

    ids: "distinct" draws S different experts per token (top-S routing);
    "repeat" draws every slot independently (an expert may repeat within a
    token).  x_per_slot: X is [T, S, K] (one row per slot) instead of [T, K].
    """
    name: str
    T: int
    S: int
    E: int
    N: int
    K: int
    bits: int
    bs: int
    act_dtype: int
    out_dtype: int
    scale_dtype: int
    x_per_slot: bool = False
    ids: str = "distinct"
    scale_lo: float = 0.001
    scale_hi: float = 0.01
    zp: Optional[tuple] = None
    seed: int = SEED_BASE

    def expert(self) -> Workload:
        """One expert's dense shape (M = the most rows it can own)."""
        return Workload(self.name + "_expert", self.T * self.S, self.N, self.K, self.bits, self.bs,
                        self.act_dtype, self.out_dtype, self.scale_dtype, "normal", self.scale_lo,
                        self.scale_hi, self.zp, self.seed)

    def bytes(self, ids: np.ndarray) -> int:
        """Algorithmic bytes: the selected experts' codes, scales and zero points once each, X and Y."""
        w = self.expert()
        active = len(np.unique(ids))
        per_expert = (w.N * w.kblocks * w.blob + w.N * w.kblocks * DTYPE_BYTES[self.scale_dtype] +
                      (w.N * w.zp_row_bytes if self.zp is not None else 0))
        xrows = self.T * (self.S if self.x_per_slot else 1)
        return (active * per_expert + xrows * self.K * DTYPE_BYTES[self.act_dtype] +
                self.T * self.S * self.N * DTYPE_BYTES[self.out_dtype])


MOE_CONFIGS = [
    MoeWorkload("moe_t4_top2_e8_k4096_n14336_int4_bs32_asym_bf16", 4, 2, 8, 14336, 4096, 4, 32, BF16, BF16, F16,
                scale_lo=0.001, scale_hi=0.01, zp=(0, 15), seed=SEED_BASE + 10),
]


def generate_moe(w: MoeWorkload, rng: Optional[np.random.Generator] = None) -> dict:
    """Draw one grouped workload's inputs.

    Returns a dict with
      x      : [T, K] or [T, S, K] storage
      ids    : [T, S] int32 expert indices
      b      : [E, N, KB, blob] uint8 packed codes (ORT layout per expert)
      scales : [E, N, KB] storage
      zp     : [E, N, ceil(KB*bits/8)] uint8 or None
    Draw order is fixed (x, ids, scales, b, zp).
    """
    if rng is None:
        rng = np.random.default_rng(w.seed)
    ew = w.expert()
    x64 = rng.standard_normal((w.T, w.S, w.K) if w.x_per_slot else (w.T, w.K))
    if w.ids == "distinct":
        if w.S > w.E:
            raise ValueError("distinct routing needs S <= E")
        ids = np.stack([rng.permutation(w.E)[:w.S] for _ in range(w.T)]) if w.T else np.zeros((0, w.S))
    elif w.ids == "repeat":
        ids = rng.integers(0, w.E, size=(w.T, w.S))
    else:
        raise ValueError(w.ids)
    s64 = rng.uniform(w.scale_lo, w.scale_hi, (w.E, w.N, ew.kblocks))
    b = rng.integers(0, 256, size=(w.E, w.N, ew.kblocks, ew.blob), dtype=np.uint8)
    zp = None
    if w.zp is not None:
        lo, hi = w.zp
        if lo == 0 and hi == (1 << w.bits) - 1:
            zp = rng.integers(0, 256, size=(w.E, w.N, ew.zp_row_bytes), dtype=np.uint8)
        elif w.bits == 8:
            zp = rng.integers(lo, hi + 1, size=(w.E, w.N, ew.zp_row_bytes), dtype=np.uint8)
        else:
            raise ValueError("a partial zero-point range needs packing; draw it in the caller")
    return {
        "x": to_storage(x64, w.act_dtype),
        "ids": np.ascontiguousarray(ids, dtype=np.int32).reshape(w.T, w.S),
        "b": b,
        "scales": to_storage(s64, w.scale_dtype),
        "zp": zp,
    }
