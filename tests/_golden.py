"""Readers for the hand-worked fixtures in tests/golden/ and test-side helpers.

The helpers here pack codes for hand-built test cases and compute comparison
tolerances.  They belong to the tests: neither the oracle nor the CUDA path
imports them.
"""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                out.append(line.split())
    return out


def pack_codes_test(codes, bits):
    """Pack integer codes LSB-first into bytes (test-side packer, written from
    the storage rule: element i at bit i*bits)."""
    codes = [int(c) for c in codes]
    nbytes = -(-len(codes) * bits // 8)
    out = bytearray(nbytes)
    for i, c in enumerate(codes):
        bit = i * bits
        out[bit // 8] |= (c & ((1 << bits) - 1)) << (bit % 8)
    return np.frombuffer(bytes(out), dtype=np.uint8).copy()


def pack_matrix_test(q, bits, bs):
    """q: [N, K] integer codes -> ORT B [N, KB, bs*bits/8], tail codes zero."""
    q = np.asarray(q)
    N, K = q.shape
    kb = -(-K // bs)
    blob = bs * bits // 8
    out = np.zeros((N, kb, blob), dtype=np.uint8)
    for n in range(N):
        for b in range(kb):
            seg = list(q[n, b * bs:min(K, (b + 1) * bs)])
            seg += [0] * (bs - len(seg))
            out[n, b] = pack_codes_test(seg, bits)
    return out


def pack_zp_test(z, bits):
    """z: [N, KB] zero points -> [N, ceil(KB*bits/8)] bytes."""
    z = np.asarray(z)
    N, kb = z.shape
    rb = -(-kb * bits // 8)
    out = np.zeros((N, rb), dtype=np.uint8)
    for n in range(N):
        out[n] = pack_codes_test(list(z[n]), bits)[:rb] if rb else out[n]
    return out


def half_ulp(v, out_dtype):
    """Half a unit in the last place of |v| in the output dtype (0 for f32)."""
    v = np.abs(np.asarray(v, dtype=np.float64))
    if out_dtype == 0:
        return np.zeros_like(v)
    mant = 10 if out_dtype == 1 else 7
    min_exp = -14 if out_dtype == 1 else -126
    e = np.floor(np.log2(np.maximum(v, 1e-300)))
    e = np.maximum(e, min_exp)
    return 0.5 * np.exp2(e - mant)


def tolerance(y_ref, absdot, out_dtype):
    """|y - y_ref| <= 2e-3 * sum_k |x_k w_k| + 1e-6 (+ half an output ulp)."""
    return 2e-3 * np.asarray(absdot) + 1e-6 + half_ulp(y_ref, out_dtype)
