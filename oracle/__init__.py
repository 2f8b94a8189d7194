"""TEST INFRASTRUCTURE ONLY: the fp64 CPU oracle of the 4-bit weight-quantized linear.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The product library never does, and this package imports nothing
from the product package: the two share no code.

The arithmetic lives in ``q4_oracle.c`` (plain C, IEEE double, k ascending); this module
compiles it with gcc and marshals numpy arrays through ctypes.  See the C file's header
for the passages each routine follows and the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_q4.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile q4_oracle.c into liboracle_q4.so (gcc -O2, no fast-math, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall",
               "-Werror", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, i32, vp, dp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
        lib.q4o_num_threads.argtypes = []
        lib.q4o_num_threads.restype = ctypes.c_int
        lib.q4o_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.q4o_f16_to_f64.restype = ctypes.c_double
        lib.q4o_linear.argtypes = [vp, vp, vp, i32, vp, i64, i64, i64, i64, i32, dp, dp]
        lib.q4o_linear.restype = i32
        lib.q4o_linear_at.argtypes = [vp, vp, vp, i32, vp, i64, i64, i64, i64, i32,
                                      vp, vp, i64, dp, dp]
        lib.q4o_linear_at.restype = i32
        lib.q4o_linear_qcs4w.argtypes = [vp, vp, vp, i32, vp, i64, i64, i64, dp, dp]
        lib.q4o_linear_qcs4w.restype = i32
        lib.q4o_backward_dx.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, i32, dp, dp]
        lib.q4o_backward_dx.restype = i32
        lib.q4o_requant.argtypes = [vp, vp, i32, i64, i64, i64, i32, vp]
        lib.q4o_requant.restype = i32
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _scales_kind(scales: np.ndarray) -> int:
    if scales.dtype == np.float16:
        return 1
    if scales.dtype == np.float32:
        return 0
    raise TypeError(f"scales must be float32 or float16, got {scales.dtype}")


def _prep(x, qweight, scales, bias, K):
    x = np.ascontiguousarray(x, dtype=np.float32)
    qweight = np.ascontiguousarray(qweight, dtype=np.uint8)
    scales = np.ascontiguousarray(scales)
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
    M = x.shape[0] if x.ndim == 2 else 1
    if x.size != M * K:
        raise ValueError("x must hold M*K values")
    N = qweight.shape[0]
    if qweight.shape[1] != (K + 1) // 2:
        raise ValueError("qweight must be [N, ceil(K/2)]")
    return x, qweight, scales, bias, M, N


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().q4o_num_threads())


def f16_to_f64(bits: int) -> float:
    """The oracle's own IEEE binary16 decode of one bit pattern."""
    return _load().q4o_f16_to_f64(int(bits))


def linear(x, qweight, scales, bias, K: int, group_size: int,
           even_high: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 out[M,N] (bias included) and mag[M,N] = sum_k |x*w| by the definition.

    x: float32 [M,K]; qweight: uint8 [N, ceil(K/2)]; scales: float32 or float16
    [ceil(K/group_size), N]; bias: float32 [N] or None.
    """
    x, qweight, scales, bias, M, N = _prep(x, qweight, scales, bias, K)
    G = -(-K // group_size)
    if scales.size != G * N:
        raise ValueError("scales must be [ceil(K/group_size), N]")
    out = np.empty((M, N), np.float64)
    mag = np.empty((M, N), np.float64)
    rc = _load().q4o_linear(_ptr(x), _ptr(qweight), _ptr(scales), _scales_kind(scales),
                            _ptr(bias), M, N, K, group_size, int(even_high),
                            _ptr(out), _ptr(mag))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out, mag


def linear_at(x, qweight, scales, bias, K: int, group_size: int, ms, ns,
              even_high: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """Like ``linear`` but only the elements (ms[i], ns[i]); returns 1-D arrays."""
    x, qweight, scales, bias, M, N = _prep(x, qweight, scales, bias, K)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    if ms.shape != ns.shape:
        raise ValueError("ms and ns must have the same length")
    out = np.empty(ms.size, np.float64)
    mag = np.empty(ms.size, np.float64)
    rc = _load().q4o_linear_at(_ptr(x), _ptr(qweight), _ptr(scales), _scales_kind(scales),
                               _ptr(bias), M, N, K, group_size, int(even_high),
                               _ptr(ms), _ptr(ns), ms.size, _ptr(out), _ptr(mag))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out, mag


def linear_qcs4w(x, qweight, scales_n, bias, K: int) -> Tuple[np.ndarray, np.ndarray]:
    """The separately written per-channel routine (scales_n: [N])."""
    x, qweight, scales_n, bias, M, N = _prep(x, qweight, scales_n, bias, K)
    if scales_n.size != N:
        raise ValueError("scales_n must be [N]")
    out = np.empty((M, N), np.float64)
    mag = np.empty((M, N), np.float64)
    rc = _load().q4o_linear_qcs4w(_ptr(x), _ptr(qweight), _ptr(scales_n),
                                  _scales_kind(scales_n), _ptr(bias), M, N, K,
                                  _ptr(out), _ptr(mag))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out, mag


def backward_dx(d_out, qweight, scales, K: int, group_size: int,
                even_high: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 d_x[M,K] = d_out[M,N] @ dequant(W)[N,K] and mag[M,K] = sum_n |d_out * w|.

    d_out: float32 [M,N]; qweight: uint8 [N, ceil(K/2)]; scales: float32 or float16
    [ceil(K/group_size), N].
    """
    qweight = np.ascontiguousarray(qweight, dtype=np.uint8)
    scales = np.ascontiguousarray(scales)
    N = qweight.shape[0]
    d_out = np.ascontiguousarray(d_out, dtype=np.float32).reshape(-1, N)
    M = d_out.shape[0]
    if qweight.shape[1] != (K + 1) // 2:
        raise ValueError("qweight must be [N, ceil(K/2)]")
    if scales.size != -(-K // group_size) * N:
        raise ValueError("scales must be [ceil(K/group_size), N]")
    d_x = np.empty((M, K), np.float64)
    mag = np.empty((M, K), np.float64)
    rc = _load().q4o_backward_dx(_ptr(d_out), _ptr(qweight), _ptr(scales),
                                 _scales_kind(scales), M, N, K, group_size, int(even_high),
                                 _ptr(d_x), _ptr(mag))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return d_x, mag


def requant(latent, scales, group_size: int, even_high: bool = False) -> np.ndarray:
    """Packed codes uint8 [N, ceil(K/2)] of fp32 latents [N,K] with frozen scales
    [ceil(K/group_size), N]: clamp(round(latent / scale), -8, 7) + 8, zero scale -> 8."""
    latent = np.ascontiguousarray(latent, dtype=np.float32)
    scales = np.ascontiguousarray(scales)
    N, K = latent.shape
    if scales.size != -(-K // group_size) * N:
        raise ValueError("scales must be [ceil(K/group_size), N]")
    out = np.empty((N, (K + 1) // 2), np.uint8)
    rc = _load().q4o_requant(_ptr(latent), _ptr(scales), _scales_kind(scales), N, K,
                             group_size, int(even_high), _ptr(out))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out
