"""Thin ctypes binding of libq4lin.so, with the C ABI's names (include/q4lin.h).

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels.  If the library has not been built this module raises at import time; there
is no fallback of any kind.

``q4lin_run`` and friends take raw integers for pointers and the stream.  ``linear``
is a convenience that takes torch CUDA tensors, checks their dtypes/shapes/contiguity,
and passes their data pointers and the current stream to ``q4lin_run``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libq4lin.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"{_LIB_PATH} is missing: build it with `python -m bit_weight_quantized_int4_gb300.build` "
        "(the q4lin CUDA library is required; there is no fallback)")
_lib = ctypes.CDLL(_LIB_PATH)

# ---- constants (mirror include/q4lin.h) ----
Q4LIN_OK = 0
Q4LIN_ERR_INVALID_ARG = 1
Q4LIN_ERR_UNSUPPORTED = 2
Q4LIN_ERR_CUDA = 3
Q4LIN_ERR_TIMEOUT = 4
Q4LIN_ERR_NO_DEVICE = 5
Q4LIN_ERR_TOO_LARGE = 6

Q4LIN_SCALE_F32 = 0
Q4LIN_SCALE_F16 = 1

Q4LIN_PATH_AUTO = 0
Q4LIN_PATH_GEMV = 1
Q4LIN_PATH_FFMA = 2
Q4LIN_PATH_TC = 3
Q4LIN_PATH_TC_SMALL = 4
PATH_NAMES = {0: "auto", 1: "gemv", 2: "ffma", 3: "tc", 4: "tc_small"}

Q4LIN_KERNEL_NONE = 0
Q4LIN_KERNEL_GEMV_TMA = 1
Q4LIN_KERNEL_MULTIROW = 2
Q4LIN_KERNEL_ROWSTREAM = 3
Q4LIN_KERNEL_GENERIC = 4
Q4LIN_KERNEL_TC = 5
Q4LIN_KERNEL_TC_F16 = 6
Q4LIN_KERNEL_GEMV_TMA_FIXED = 7
Q4LIN_KERNEL_TC_SMALL = 8
Q4LIN_KERNEL_TC_SMALL_BF16 = 9
KERNEL_NAMES = {0: "none", 1: "gemv_tma", 2: "multirow", 3: "rowstream", 4: "generic",
                5: "tc", 6: "tc_f16", 7: "gemv_tma_fixed", 8: "tc_small", 9: "tc_small_bf16"}

Q4LIN_OPT_FORCE_PATH = 1
Q4LIN_OPT_NIBBLE_EVEN_HIGH = 2
Q4LIN_OPT_WAIT_LIMIT = 3
Q4LIN_OPT_PDL = 4
Q4LIN_OPT_TC_SKIP_FIRST_COPY = 5
Q4LIN_OPT_TC_F16 = 6
Q4LIN_OPT_TC_SMALL_OPERANDS = 7

_vp, _i64, _i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int

_lib.q4lin_create.argtypes = [ctypes.POINTER(_vp), _i32]
_lib.q4lin_create.restype = _i32
_lib.q4lin_destroy.argtypes = [_vp]
_lib.q4lin_destroy.restype = _i32
_lib.q4lin_run.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32, _vp]
_lib.q4lin_run.restype = _i32
class q4lin_problem_t(ctypes.Structure):
    _fields_ = [("x", _vp), ("qweight", _vp), ("scales", _vp), ("bias", _vp), ("out", _vp),
                ("M", _i64), ("N", _i64), ("K", _i64), ("group_size", _i64),
                ("scale_dtype", _i32)]


_lib.q4lin_run_grouped.argtypes = [_vp, ctypes.POINTER(q4lin_problem_t), _i32, _vp]
_lib.q4lin_run_grouped.restype = _i32
_lib.q4lin_run_static_scratch.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp]
_lib.q4lin_run_static_scratch.restype = _i32
_lib.q4lin_run_backward_dx.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32,
                                       _vp]
_lib.q4lin_run_backward_dx.restype = _i32
_lib.q4lin_run_requant.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp]
_lib.q4lin_run_requant.restype = _i32
_lib.q4lin_plan.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32,
                            ctypes.POINTER(_i32)]
_lib.q4lin_plan.restype = _i32
_lib.q4lin_plan_kernel.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32,
                                   ctypes.POINTER(_i32)]
_lib.q4lin_plan_kernel.restype = _i32
_lib.q4lin_set_option.argtypes = [_vp, _i32, _i64]
_lib.q4lin_set_option.restype = _i32
_lib.q4lin_get_option.argtypes = [_vp, _i32, ctypes.POINTER(_i64)]
_lib.q4lin_get_option.restype = _i32
_lib.q4lin_check_device_status.argtypes = [_vp, _vp, ctypes.POINTER(_i32)]
_lib.q4lin_check_device_status.restype = _i32
_lib.q4lin_status_string.argtypes = [_i32]
_lib.q4lin_status_string.restype = ctypes.c_char_p


class Q4LinError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {q4lin_status_string(status)} (status {status})")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def q4lin_status_string(status: int) -> str:
    return _lib.q4lin_status_string(int(status)).decode()


def q4lin_create(device: int = 0) -> int:
    h = _vp()
    st = _lib.q4lin_create(ctypes.byref(h), int(device))
    if st != Q4LIN_OK:
        raise Q4LinError(st, "q4lin_create")
    return h.value


def q4lin_destroy(handle: int) -> int:
    return _lib.q4lin_destroy(handle)


def q4lin_run(handle, x, qweight, scales, bias, out, M, N, K, group_size, scale_dtype,
              stream) -> int:
    """Raw call: pointers and the stream are integers (0 / None for NULL)."""
    return _lib.q4lin_run(handle, x, qweight, scales, bias, out, M, N, K, group_size,
                          scale_dtype, stream)


def q4lin_run_grouped(handle, problems, stream) -> int:
    """problems: a sequence of q4lin_problem_t (or of 10-tuples in its field order)."""
    arr = (q4lin_problem_t * max(1, len(problems)))()
    for i, p in enumerate(problems):
        arr[i] = p if isinstance(p, q4lin_problem_t) else q4lin_problem_t(*p)
    return _lib.q4lin_run_grouped(handle, arr, len(problems), stream)


def q4lin_run_grouped_array(handle, array, count, stream) -> int:
    """Raw call with a prebuilt ctypes array of q4lin_problem_t (no per-call marshalling)."""
    return _lib.q4lin_run_grouped(handle, array, int(count), stream)


def q4lin_run_static_scratch(x, qweight, scales, bias, out, N, K, group_size, scale_dtype,
                             stream) -> int:
    """Raw call of the allocation-free decode GEMV (pointers and stream as integers)."""
    return _lib.q4lin_run_static_scratch(x, qweight, scales, bias, out, N, K, group_size,
                                         scale_dtype, stream)


def q4lin_run_backward_dx(handle, d_out, qweight, scales, d_x, M, N, K, group_size,
                          scale_dtype, stream) -> int:
    """Raw call: d_x[M,K] = d_out[M,N] @ dequant(W)[N,K] (pointers and stream as integers)."""
    return _lib.q4lin_run_backward_dx(handle, d_out, qweight, scales, d_x, M, N, K,
                                      group_size, scale_dtype, stream)


def q4lin_run_requant(handle, latent, scales, qweight, N, K, group_size, scale_dtype,
                      stream) -> int:
    """Raw call: packed codes of fp32 latents [N,K] with frozen scales (integers as pointers)."""
    return _lib.q4lin_run_requant(handle, latent, scales, qweight, N, K, group_size,
                                  scale_dtype, stream)


def q4lin_plan(handle, x, qweight, scales, bias, out, M, N, K, group_size, scale_dtype):
    """Returns (status, path)."""
    path = _i32(0)
    st = _lib.q4lin_plan(handle, x, qweight, scales, bias, out, M, N, K, group_size,
                         scale_dtype, ctypes.byref(path))
    return st, path.value


def q4lin_plan_kernel(handle, x, qweight, scales, bias, out, M, N, K, group_size,
                      scale_dtype):
    """Returns (status, kernel)."""
    kernel = _i32(0)
    st = _lib.q4lin_plan_kernel(handle, x, qweight, scales, bias, out, M, N, K, group_size,
                                scale_dtype, ctypes.byref(kernel))
    return st, kernel.value


def q4lin_set_option(handle, option: int, value: int) -> int:
    return _lib.q4lin_set_option(handle, int(option), int(value))


def q4lin_get_option(handle, option: int):
    v = _i64(0)
    st = _lib.q4lin_get_option(handle, int(option), ctypes.byref(v))
    return st, v.value


def q4lin_check_device_status(handle, stream):
    code = _i32(0)
    st = _lib.q4lin_check_device_status(handle, stream, ctypes.byref(code))
    return st, code.value


# ---------------------------------------------------------------- torch convenience
class Handle:
    """Owns a q4lin handle for one CUDA device."""

    def __init__(self, device: int = 0):
        self.device = device
        self.ptr = q4lin_create(device)

    def close(self):
        if self.ptr:
            q4lin_destroy(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_option(self, option: int, value: int):
        st = q4lin_set_option(self.ptr, option, value)
        if st != Q4LIN_OK:
            raise Q4LinError(st, "q4lin_set_option")


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check_args(x, qweight, scales, bias, group_size):
    import torch
    if x.dtype != torch.float32 or not x.is_contiguous() or x.dim() != 2:
        raise ValueError("x must be a contiguous float32 [M, K] tensor")
    M, K = x.shape
    if qweight.dtype != torch.uint8 or not qweight.is_contiguous() or qweight.dim() != 2 \
            or qweight.shape[1] != (K + 1) // 2:
        raise ValueError("qweight must be a contiguous uint8 [N, ceil(K/2)] tensor")
    N = qweight.shape[0]
    if scales.dtype == torch.float16:
        sd = Q4LIN_SCALE_F16
    elif scales.dtype == torch.float32:
        sd = Q4LIN_SCALE_F32
    else:
        raise ValueError("scales must be float32 or float16")
    if not scales.is_contiguous() or scales.numel() != -(-K // group_size) * N:
        raise ValueError("scales must be a contiguous [ceil(K/group_size), N] tensor")
    if bias is not None and (bias.dtype != torch.float32 or not bias.is_contiguous()
                             or bias.numel() != N):
        raise ValueError("bias must be a contiguous float32 [N] tensor or None")
    return M, N, K, sd


def linear(handle: Handle, x, qweight, scales, bias, group_size: int, out=None,
           stream=None):
    """out[M,N] = x @ dequant(qweight)^T (+ bias) on the current (or given) stream."""
    import torch
    M, N, K, sd = _check_args(x, qweight, scales, bias, group_size)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    s = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
    st = q4lin_run(handle.ptr, _ptr(x), _ptr(qweight), _ptr(scales), _ptr(bias),
                   _ptr(out), M, N, K, group_size, sd, s)
    if st != Q4LIN_OK:
        raise Q4LinError(st, "q4lin_run")
    return out


def plan(handle: Handle, x, qweight, scales, bias, group_size: int, out) -> str:
    """Name of the kernel family q4lin_run would use for these tensors."""
    M, N, K, sd = _check_args(x, qweight, scales, bias, group_size)
    st, path = q4lin_plan(handle.ptr, _ptr(x), _ptr(qweight), _ptr(scales), _ptr(bias),
                          _ptr(out), M, N, K, group_size, sd)
    if st != Q4LIN_OK:
        raise Q4LinError(st, "q4lin_plan")
    return PATH_NAMES[path]


def plan_kernel(handle: Handle, x, qweight, scales, bias, group_size: int, out) -> str:
    """Name of the kernel q4lin_run would launch for these tensors."""
    M, N, K, sd = _check_args(x, qweight, scales, bias, group_size)
    st, kernel = q4lin_plan_kernel(handle.ptr, _ptr(x), _ptr(qweight), _ptr(scales),
                                   _ptr(bias), _ptr(out), M, N, K, group_size, sd)
    if st != Q4LIN_OK:
        raise Q4LinError(st, "q4lin_plan_kernel")
    return KERNEL_NAMES[kernel]
