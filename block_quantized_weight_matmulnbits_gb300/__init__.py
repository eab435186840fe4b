"""Python binding of libmnb (block-quantized weight-only matmul for GB300, sm_103a).

Argument marshalling only: every function forwards to the C entry point of
the same name in ``include/mnb.h`` (loaded with ctypes from the in-tree build)
and raises ``MnbError`` on a non-OK status.  Tensors are passed by device
pointer; streams default to torch's current stream.  Nothing here computes
any part of the operation, and there is no fallback: if the CUDA library
cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import threading

from . import _build

MNB_OK, MNB_ERR_INVALID_ARG, MNB_ERR_UNSUPPORTED, MNB_ERR_CUDA, MNB_ERR_NO_MEM, MNB_ERR_TIMEOUT, \
    MNB_ERR_LAYOUT_MISMATCH = range(7)
MNB_F32, MNB_F16, MNB_BF16 = 0, 1, 2
MNB_FLAG_PDL = 1
MNB_FLAG_KPERM = 2
MNB_WF_E4M3, MNB_WF_E5M2, MNB_WF_NVFP4 = 1, 2, 3
KERNELS = {"auto": 0, "gemv": 1, "gemv_mma": 2, "gemm_tc": 3, "generic": 4, "gemv_i8": 5}
KERNEL_NAMES = {v: k for k, v in KERNELS.items()}

# Every symbol include/mnb.h declares.
EXPORTS = [
    "mnb_packed_size", "mnb_pack_weights", "mnb_unpack_codes", "mnb_dequantize", "mnb_matmul",
    "mnb_matmul_ex", "mnb_workspace_size", "mnb_quantize_activations", "mnb_select_kernel",
    "mnb_get_device_error", "mnb_status_string", "mnb_kernel_name", "mnb_abi_version", "mnb_matmul_a8_static",
    "mnb_matmul_host_io", "mnb_matmul_grouped", "mnb_fp_packed_size", "mnb_pack_fp_weights", "mnb_matmul_fp",
    "mnb_matmul_fp_ex", "mnb_packed_size_gidx", "mnb_pack_weights_gidx", "mnb_workspace_size_ex",
]
MNB_A8_STATIC_SCRATCH_BYTES = 1 << 20
MNB_HOST_IO_X_BYTES = 8 << 20


class MnbError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class MatmulArgs(ctypes.Structure):
    _fields_ = [
        ("x", ctypes.c_void_p), ("packed_b", ctypes.c_void_p), ("scales", ctypes.c_void_p),
        ("zero_points", ctypes.c_void_p), ("g_idx", ctypes.c_void_p), ("bias", ctypes.c_void_p),
        ("y", ctypes.c_void_p), ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
        ("bits", ctypes.c_int), ("block_size", ctypes.c_int), ("act_dtype", ctypes.c_int),
        ("out_dtype", ctypes.c_int), ("scale_dtype", ctypes.c_int), ("bias_dtype", ctypes.c_int),
        ("accuracy_level", ctypes.c_int), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("kernel", ctypes.c_int), ("stream", ctypes.c_void_p), ("flags", ctypes.c_int),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build: bool = True):
    """Build (if stale) and load libmnb.so; raises if that is impossible."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build() if build else _build.LIB
        lib = ctypes.CDLL(path)
        vp, i64, ci, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        sig = {
            "mnb_packed_size": (sz, [i64, i64, ci, ci]),
            "mnb_pack_weights": (ci, [vp, vp, sz, i64, i64, ci, ci, vp]),
            "mnb_packed_size_gidx": (sz, [i64, i64, ci, ci]),
            "mnb_workspace_size_ex": (sz, [i64, i64, i64, ci, ci, ci, ci]),
            "mnb_pack_weights_gidx": (ci, [vp, vp, vp, sz, i64, i64, ci, ci, vp]),
            "mnb_unpack_codes": (ci, [vp, vp, i64, i64, ci, ci, vp]),
            "mnb_dequantize": (ci, [vp, vp, vp, vp, i64, i64, ci, ci, ci, vp]),
            "mnb_matmul": (ci, [vp, vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, ci, ci, vp]),
            "mnb_matmul_ex": (ci, [ctypes.POINTER(MatmulArgs)]),
            "mnb_workspace_size": (sz, [i64, i64, i64, ci, ci, ci]),
            "mnb_quantize_activations": (ci, [vp, vp, vp, i64, i64, ci, ci, vp]),
            "mnb_select_kernel": (ci, [i64, i64, i64, ci, ci, ci, ci]),
            "mnb_get_device_error": (ci, [ctypes.POINTER(ci)]),
            "mnb_status_string": (ctypes.c_char_p, [ci]),
            "mnb_kernel_name": (ctypes.c_char_p, [ci]),
            "mnb_abi_version": (ci, []),
            "mnb_matmul_a8_static": (ci, [vp, vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, ci, ci, vp]),
            "mnb_matmul_host_io": (ci, [ctypes.POINTER(MatmulArgs)]),
            "mnb_matmul_grouped": (ci, [vp, vp, vp, vp, vp, vp, i64, i64, i64, ci, i64, i64, ci, ci, ci, ci, ci,
                                        vp]),
            "mnb_fp_packed_size": (sz, [i64, i64, ci]),
            "mnb_pack_fp_weights": (ci, [vp, vp, sz, i64, i64, ci, vp]),
            "mnb_matmul_fp": (ci, [vp, vp, vp, ctypes.c_float, vp, i64, i64, i64, ci, ci, ci, vp]),
            "mnb_matmul_fp_ex": (ci, [vp, vp, vp, ctypes.c_float, vp, i64, i64, i64, ci, ci, ci, vp, ci]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != MNB_OK:
        raise MnbError(status, what)


def status_string(status: int) -> str:
    try:
        return load().mnb_status_string(status).decode()
    except Exception:  # the library itself may be what failed to load
        return f"status {status}"


def mnb_abi_version() -> int:
    return load().mnb_abi_version()


def mnb_packed_size(N, K, bits, block_size) -> int:
    return load().mnb_packed_size(N, K, bits, block_size)


def mnb_pack_weights(b_ort, packed_b, N, K, bits, block_size, stream=None):
    _check(load().mnb_pack_weights(_ptr(b_ort), _ptr(packed_b), packed_b.numel() * packed_b.element_size(),
                                   N, K, bits, block_size, _stream(stream)), "mnb_pack_weights")


def mnb_packed_size_gidx(N, K, bits, block_size) -> int:
    return load().mnb_packed_size_gidx(N, K, bits, block_size)


def mnb_pack_weights_gidx(b_ort, g_idx, packed_b, N, K, bits, block_size, stream=None):
    """Act-order pack: depths sorted by their g_idx block, the permutation stored in the buffer
    (use it with flags=MNB_FLAG_KPERM and no g_idx)."""
    _check(load().mnb_pack_weights_gidx(_ptr(b_ort), _ptr(g_idx), _ptr(packed_b),
                                        packed_b.numel() * packed_b.element_size(), N, K, bits, block_size,
                                        _stream(stream)), "mnb_pack_weights_gidx")


def mnb_unpack_codes(packed_b, b_ort, N, K, bits, block_size, stream=None):
    _check(load().mnb_unpack_codes(_ptr(packed_b), _ptr(b_ort), N, K, bits, block_size, _stream(stream)),
           "mnb_unpack_codes")


def mnb_dequantize(packed_b, scales, zero_points, w_nk, N, K, bits, block_size, scale_dtype, stream=None):
    _check(load().mnb_dequantize(_ptr(packed_b), _ptr(scales), _ptr(zero_points), _ptr(w_nk), N, K, bits,
                                 block_size, scale_dtype, _stream(stream)), "mnb_dequantize")


def mnb_matmul(x, packed_b, scales, zero_points, y, M, N, K, bits, block_size, act_dtype, out_dtype,
               scale_dtype, stream=None):
    _check(load().mnb_matmul(_ptr(x), _ptr(packed_b), _ptr(scales), _ptr(zero_points), _ptr(y), M, N, K, bits,
                             block_size, act_dtype, out_dtype, scale_dtype, _stream(stream)), "mnb_matmul")


def _matmul_args(x, packed_b, scales, zero_points, y, M, N, K, bits, block_size, act_dtype, out_dtype,
                 scale_dtype, g_idx, bias, bias_dtype, accuracy_level, workspace, kernel, stream, flags):
    a = MatmulArgs()
    a.x, a.packed_b, a.scales, a.zero_points = _ptr(x), _ptr(packed_b), _ptr(scales), _ptr(zero_points)
    a.g_idx, a.bias, a.y = _ptr(g_idx), _ptr(bias), _ptr(y)
    a.M, a.N, a.K, a.bits, a.block_size = M, N, K, bits, block_size
    a.act_dtype, a.out_dtype, a.scale_dtype, a.bias_dtype = act_dtype, out_dtype, scale_dtype, bias_dtype
    a.accuracy_level = accuracy_level
    a.workspace = _ptr(workspace)
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    a.kernel = KERNELS[kernel] if isinstance(kernel, str) else int(kernel)
    a.stream = _stream(stream)
    a.flags = flags
    return a


def mnb_matmul_ex(x, packed_b, scales, zero_points, y, M, N, K, bits, block_size, act_dtype, out_dtype,
                  scale_dtype, g_idx=None, bias=None, bias_dtype=MNB_F32, accuracy_level=0, workspace=None,
                  kernel="auto", stream=None, flags=0):
    a = _matmul_args(x, packed_b, scales, zero_points, y, M, N, K, bits, block_size, act_dtype, out_dtype,
                     scale_dtype, g_idx, bias, bias_dtype, accuracy_level, workspace, kernel, stream, flags)
    _check(load().mnb_matmul_ex(ctypes.byref(a)), f"mnb_matmul_ex[{kernel}]")


def mnb_matmul_host_io(x, packed_b, scales, zero_points, y, M, N, K, bits, block_size, act_dtype, out_dtype,
                       scale_dtype, g_idx=None, bias=None, bias_dtype=MNB_F32, accuracy_level=0, workspace=None,
                       kernel="auto", stream=None, flags=0):
    """As mnb_matmul_ex, with x and y page-locked host tensors (e.g. .pin_memory())."""
    a = _matmul_args(x, packed_b, scales, zero_points, y, M, N, K, bits, block_size, act_dtype, out_dtype,
                     scale_dtype, g_idx, bias, bias_dtype, accuracy_level, workspace, kernel, stream, flags)
    _check(load().mnb_matmul_host_io(ctypes.byref(a)), f"mnb_matmul_host_io[{kernel}]")


def mnb_matmul_a8_static(x, packed_b, scales, zero_points, y, M, N, K, bits, block_size, act_dtype, out_dtype,
                         scale_dtype, stream=None):
    _check(load().mnb_matmul_a8_static(_ptr(x), _ptr(packed_b), _ptr(scales), _ptr(zero_points), _ptr(y), M, N, K,
                                       bits, block_size, act_dtype, out_dtype, scale_dtype, _stream(stream)),
           "mnb_matmul_a8_static")


def mnb_matmul_grouped(x, ids, packed_b, scales, zero_points, y, T, S, E, N, K, bits, block_size, act_dtype,
                       out_dtype, scale_dtype, x_per_slot=False, stream=None):
    """Grouped (mixture-of-experts) product: y[t, s] = x_row(t, s) . dequant(B[ids[t, s]])^T."""
    _check(load().mnb_matmul_grouped(_ptr(x), _ptr(ids), _ptr(packed_b), _ptr(scales), _ptr(zero_points), _ptr(y),
                                     T, S, E, 1 if x_per_slot else 0, N, K, bits, block_size, act_dtype, out_dtype,
                                     scale_dtype, _stream(stream)), "mnb_matmul_grouped")


def mnb_fp_packed_size(N, K, fmt) -> int:
    return load().mnb_fp_packed_size(N, K, fmt)


def mnb_pack_fp_weights(w_kn, packed, N, K, fmt, stream=None):
    """Re-tile a [K, N] FP8 / NVFP4 weight (device uint8) for mnb_matmul_fp."""
    _check(load().mnb_pack_fp_weights(_ptr(w_kn), _ptr(packed), packed.numel() * packed.element_size(), N, K, fmt,
                                      _stream(stream)), "mnb_pack_fp_weights")


def mnb_matmul_fp(x, packed, scales, global_scale, y, M, N, K, fmt, act_dtype, out_dtype, stream=None, flags=0):
    """Y = X . W for an FP8 (scales f32 [N] or None) or NVFP4 (e4m3 [ceil(K/16), N] scales) weight;
    flags (MNB_FLAG_*) go through mnb_matmul_fp_ex."""
    if flags:
        _check(load().mnb_matmul_fp_ex(_ptr(x), _ptr(packed), _ptr(scales), float(global_scale), _ptr(y), M, N, K,
                                       fmt, act_dtype, out_dtype, _stream(stream), int(flags)), "mnb_matmul_fp_ex")
        return
    _check(load().mnb_matmul_fp(_ptr(x), _ptr(packed), _ptr(scales), float(global_scale), _ptr(y), M, N, K, fmt,
                                act_dtype, out_dtype, _stream(stream)), "mnb_matmul_fp")


def mnb_workspace_size_ex(M, N, K, bits, block_size, accuracy_level, flags) -> int:
    return load().mnb_workspace_size_ex(M, N, K, bits, block_size, accuracy_level, flags)


def mnb_workspace_size(M, N, K, bits, block_size, accuracy_level) -> int:
    return load().mnb_workspace_size(M, N, K, bits, block_size, accuracy_level)


def mnb_quantize_activations(x, qa, sa, M, K, block_size, act_dtype, stream=None):
    _check(load().mnb_quantize_activations(_ptr(x), _ptr(qa), _ptr(sa), M, K, block_size, act_dtype,
                                           _stream(stream)), "mnb_quantize_activations")


def mnb_select_kernel(M, N, K, bits, block_size, act_dtype, accuracy_level=0) -> str:
    return KERNEL_NAMES[load().mnb_select_kernel(M, N, K, bits, block_size, act_dtype, accuracy_level)]


def mnb_get_device_error() -> int:
    code = ctypes.c_int(0)
    _check(load().mnb_get_device_error(ctypes.byref(code)), "mnb_get_device_error")
    return code.value


def mnb_status_string(status: int) -> str:
    return status_string(status)


def mnb_kernel_name(k: int) -> str:
    return load().mnb_kernel_name(k).decode()
