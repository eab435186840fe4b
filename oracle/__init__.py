"""CPU oracle for block-quantized weight-only matmul (MatMulNBits).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product (the
CUDA library and its Python binding) never imports, links or loads it, and it
imports nothing from the product.

The arithmetic lives in ``mnb_oracle.c`` (plain C, element-by-element unpack,
f32 dequantisation exactly as defined by onnx-runtime-ep-cpu 0.1.0-dev.5,
src/kernels/matmul_nbits.rs, ``dequantize_nbits_value``; f64 accumulation).
This module only compiles it with gcc, loads it with ctypes and marshals
numpy arrays.  Inputs are taken as already-widened values: activations as
f64 and scales as f32 (every storage dtype of the operator widens exactly to
these).

Parity status of each function is recorded in its docstring; all are pinned
by ``tests/test_oracle_pins.py`` (``matmul_grouped`` by
``tests/test_oracle_grouped_pins.py``, the FP8 / NVFP4 functions by
``tests/test_oracle_fp_formats_pins.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mnb_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmnb_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        ci = ctypes.c_int
        lib.oracle_code.argtypes = [p, i64, i64, ci, ci, i64, i64]
        lib.oracle_code.restype = ci
        lib.oracle_zero_point.argtypes = [p, i64, i64, ci, ci, i64, i64]
        lib.oracle_zero_point.restype = ci
        lib.oracle_weight.argtypes = [p, p, p, p, i64, i64, ci, ci, i64, i64]
        lib.oracle_weight.restype = ctypes.c_float
        lib.oracle_dequantize.argtypes = [p, p, p, p, i64, i64, ci, ci, p]
        lib.oracle_dequantize.restype = None
        lib.oracle_matmul.argtypes = [p, p, p, p, p, p, i64, i64, i64, ci, ci, p, p]
        lib.oracle_matmul.restype = None
        lib.oracle_matmul_points.argtypes = [p, p, p, p, p, p, i64, i64, i64, ci, ci, p, p, i64, p, p]
        lib.oracle_matmul_points.restype = None
        lib.oracle_quantize_act.argtypes = [p, i64, i64, ci, p, p]
        lib.oracle_quantize_act.restype = None
        lib.oracle_matmul_a8.argtypes = [p, p, p, p, p, p, i64, i64, i64, ci, ci, p, p]
        lib.oracle_matmul_a8.restype = None
        for name in ("oracle_fp8_e4m3", "oracle_fp8_e5m2", "oracle_e4m3fn_scale", "oracle_e2m1"):
            getattr(lib, name).argtypes = [ci]
            getattr(lib, name).restype = ctypes.c_float
        lib.oracle_matmul_fp8.argtypes = [p, p, p, i64, i64, i64, ci, p, p]
        lib.oracle_matmul_fp8.restype = None
        lib.oracle_nvfp4_weight.argtypes = [p, p, ctypes.c_float, i64, i64, i64]
        lib.oracle_nvfp4_weight.restype = ctypes.c_float
        lib.oracle_matmul_nvfp4.argtypes = [p, p, p, ctypes.c_float, i64, i64, i64, p, p]
        lib.oracle_matmul_nvfp4.restype = None
        lib.oracle_threads.argtypes = []
        lib.oracle_threads.restype = ci
        lib.oracle_set_threads.argtypes = [ci]
        lib.oracle_set_threads.restype = None
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u8(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.uint8)


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def threads() -> int:
    return _load().oracle_threads()


def set_threads(t: int) -> None:
    _load().oracle_set_threads(int(t))


def code(b, N, K, bits, bs, n, k) -> int:
    """Code q[n, k] of B ([N, KB, bs*bits/8] bytes, LSB first).  Pinned."""
    b = _u8(b)
    return _load().oracle_code(_ptr(b), N, K, bits, bs, n, k)


def zero_point(zp, N, K, bits, bs, n, g) -> int:
    """Zero point of (n, group g), packed at ``bits`` width; None => 2^(bits-1).  Pinned."""
    zp = _u8(zp)
    return _load().oracle_zero_point(_ptr(zp), N, K, bits, bs, n, g)


def dequantize(b, scales_f32, zp, N, K, bits, bs, g_idx=None) -> np.ndarray:
    """w[N, K] f32 = fl32((q - zp) * scale).  Pinned (bit-exact closed form)."""
    b, s, zp, g = _u8(b), _f32(scales_f32), _u8(zp), _i32(g_idx)
    w = np.empty((N, K), dtype=np.float32)
    _load().oracle_dequantize(_ptr(b), _ptr(s), _ptr(zp), _ptr(g), N, K, bits, bs, _ptr(w))
    return w


def matmul(x_f64, b, scales_f32, zp, N, K, bits, bs, g_idx=None, bias_f64=None):
    """(y[M, N] f64, absdot[M, N] f64) with y = sum_k x*w (+ bias).  Pinned."""
    x = _f64(x_f64).reshape(-1, K)
    M = x.shape[0]
    b, s, zp, g, bias = _u8(b), _f32(scales_f32), _u8(zp), _i32(g_idx), _f64(bias_f64)
    y = np.empty((M, N), dtype=np.float64)
    mag = np.empty((M, N), dtype=np.float64)
    _load().oracle_matmul(_ptr(x), _ptr(b), _ptr(s), _ptr(zp), _ptr(g), _ptr(bias), M, N, K, bits, bs,
                          _ptr(y), _ptr(mag))
    return y, mag


def matmul_points(x_f64, b, scales_f32, zp, N, K, bits, bs, ms, ns, g_idx=None, bias_f64=None):
    """Selected outputs y[ms[i], ns[i]] and their absdot.  Same arithmetic as ``matmul``."""
    x = _f64(x_f64).reshape(-1, K)
    M = x.shape[0]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    P = ms.size
    b, s, zp, g, bias = _u8(b), _f32(scales_f32), _u8(zp), _i32(g_idx), _f64(bias_f64)
    y = np.empty(P, dtype=np.float64)
    mag = np.empty(P, dtype=np.float64)
    _load().oracle_matmul_points(_ptr(x), _ptr(b), _ptr(s), _ptr(zp), _ptr(g), _ptr(bias), M, N, K, bits,
                                 bs, _ptr(ms), _ptr(ns), P, _ptr(y), _ptr(mag))
    return y, mag


def quantize_act(x_f32, K, bs):
    """Per-(m, K-block) symmetric int8 activations: (qa[M, KB*bs] int8, sa[M, KB] f32).  Pinned."""
    x = _f32(x_f32).reshape(-1, K)
    M = x.shape[0]
    kb = -(-K // bs)
    qa = np.empty((M, kb * bs), dtype=np.int8)
    sa = np.empty((M, kb), dtype=np.float32)
    _load().oracle_quantize_act(_ptr(x), M, K, bs, _ptr(qa), _ptr(sa))
    return qa, sa


def matmul_a8(qa, sa, b, scales_f32, zp, N, K, bits, bs, bias_f64=None):
    """int8-activation product: (y[M, N] f64, absdot[M, N]).  Pinned (integer identities)."""
    qa = np.ascontiguousarray(qa, dtype=np.int8)
    sa = _f32(sa)
    M = qa.shape[0]
    b, s, zp, bias = _u8(b), _f32(scales_f32), _u8(zp), _f64(bias_f64)
    y = np.empty((M, N), dtype=np.float64)
    mag = np.empty((M, N), dtype=np.float64)
    _load().oracle_matmul_a8(_ptr(qa), _ptr(sa), _ptr(b), _ptr(s), _ptr(zp), _ptr(bias), M, N, K, bits, bs,
                             _ptr(y), _ptr(mag))
    return y, mag


def matmul_grouped(x_f64, ids, b, scales_f32, zp, E, N, K, bits, bs, x_per_slot=False):
    """Grouped (mixture-of-experts) product: (y[T, S, N] f64, absdot[T, S, N]).

    y[t, s, :] = x_row(t, s) . dequant(B_e)^T with e = ids[t, s], where x_row is
    x[t] (x: [T, K], one activation row shared by a token's slots) or x[t, s]
    (x: [T, S, K]).  The steps are those of ggml's MUL_MAT_ID as the SpacemiT
    backend computes it (toy 0.8.0, data/vendor/ggml/src/ggml-cpu/spacemit/
    ime.cpp, forward_mul_mat_id): group the (token, slot) rows by the expert
    they select, in ascending token-then-slot order, then multiply each group
    by its expert's matrix (here ``matmul``, the pinned plain product) and
    write each row back to its (token, slot).  With S = 1 it is rlx's grouped
    dequant matmul (rlx-cpu 0.2.13, src/thunk/ops/quant.rs,
    exec_dequant_grouped_mat_mul_gguf).  An expert id outside [0, E) is an
    error, as the page's assertion makes it.
    b: [E, N, KB, blob] uint8, scales_f32: [E, N, KB], zp: [E, N, zp_row] or None.
    Pinned by a one-hot expert-sum restatement, relabelling invariance and
    the E = 1 and equal-slot-rows reductions.
    """
    ids = np.asarray(ids)
    T, S = ids.shape
    x = np.asarray(x_f64, dtype=np.float64)
    if np.any(ids < 0) or np.any(ids >= E):
        raise ValueError("expert id out of range")
    y = np.zeros((T, S, N), dtype=np.float64)
    mag = np.zeros((T, S, N), dtype=np.float64)
    for e in range(E):
        rows = [(t, s) for t in range(T) for s in range(S) if ids[t, s] == e]
        if not rows:
            continue
        xe = np.stack([x[t, s] if x_per_slot else x[t] for (t, s) in rows])
        ye, me = matmul(xe, b[e], scales_f32[e], None if zp is None else zp[e], N, K, bits, bs)
        for r, (t, s) in enumerate(rows):
            y[t, s] = ye[r]
            mag[t, s] = me[r]
    return y, mag


# ---- other weight formats: FP8 and NVFP4 (rlx-cpu 0.2.13, src/thunk/ops/quant.rs) ----

def _decode_each(fn, codes):
    codes = np.asarray(codes)
    return np.array([fn(int(c)) for c in codes.ravel()], dtype=np.float32).reshape(codes.shape)


def fp8_decode(codes, e5m2=False) -> np.ndarray:
    """FP8 codes to f32 as the page's fp8_e4m3_to_f32 / fp8_e5m2_to_f32 define them
    (exponent all ones: infinity or NaN).  Pinned."""
    lib = _load()
    return _decode_each(lib.oracle_fp8_e5m2 if e5m2 else lib.oracle_fp8_e4m3, codes)


def e4m3fn_scale(codes) -> np.ndarray:
    """NVFP4 block-scale codes to f32 (OCP E4M3, no infinity; the page's
    fp8_e4m3_scale_to_f32 is not printed).  Pinned."""
    return _decode_each(_load().oracle_e4m3fn_scale, codes)


def e2m1(nibbles) -> np.ndarray:
    """FP4 E2M1 codes to f32 (OCP E2M1; the page's fp4_e2m1_to_f32 is not printed).  Pinned."""
    return _decode_each(_load().oracle_e2m1, nibbles)


def matmul_fp8(x_f64, w8, scales_f32, K, N, e5m2=False):
    """dequant_matmul_fp8: (y[M, N] f64, absdot) with y[i, j] = sum_p x[i, p] * fp8(w8[p, j]) * s[j];
    w8 is [K, N] uint8, scales [N] f32 or None (1.0).  Pinned."""
    x = _f64(x_f64).reshape(-1, K)
    M = x.shape[0]
    w8, s = _u8(w8), _f32(scales_f32)
    y = np.empty((M, N), dtype=np.float64)
    mag = np.empty((M, N), dtype=np.float64)
    _load().oracle_matmul_fp8(_ptr(x), _ptr(w8), _ptr(s), M, K, N, 1 if e5m2 else 0, _ptr(y), _ptr(mag))
    return y, mag


def nvfp4_weights(w4, scale8, global_scale, K, N) -> np.ndarray:
    """The dequantised NVFP4 weights [K, N] f32, each formed as the page forms it.  Pinned."""
    lib = _load()
    w4, s8 = _u8(w4), _u8(scale8)
    out = np.empty((K, N), dtype=np.float32)
    for p in range(K):
        for j in range(N):
            out[p, j] = lib.oracle_nvfp4_weight(_ptr(w4), _ptr(s8), float(global_scale), N, p, j)
    return out


def matmul_nvfp4(x_f64, w4, scale8, global_scale, K, N):
    """dequant_matmul_nvfp4: (y[M, N] f64, absdot); w4 holds K*N nibbles (flat index p*N + j, low nibble
    first), scale8 the [ceil(K/16), N] e4m3 block scales.  Pinned."""
    x = _f64(x_f64).reshape(-1, K)
    M = x.shape[0]
    w4, s8 = _u8(w4), _u8(scale8)
    y = np.empty((M, N), dtype=np.float64)
    mag = np.empty((M, N), dtype=np.float64)
    _load().oracle_matmul_nvfp4(_ptr(x), _ptr(w4), _ptr(s8), float(global_scale), M, K, N, _ptr(y), _ptr(mag))
    return y, mag
