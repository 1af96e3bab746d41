"""CPU baseline of the benchmark: a fused low-bit qGEMV on all host cores.

MEASUREMENT INFRASTRUCTURE (``qgemv_cpu.cc``): only ``bench.py`` and the
tests load it.  It is not the oracle (the plain fp64 definition in
``oracle/``) and not a fallback of the GPU library: it times the CPU method
of the "Mixed-width quantization" page (sections 4.1-4.2: unpack fused with
an fp32 multiply-accumulate, the group scale factored out of the inner sum)
over ``std::thread`` row blocks on every hardware thread.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qgemv_cpu.cc")
_LIB = os.path.join(_HERE, "libqgemv_cpu.so")
CXXFLAGS = ["-O3", "-std=c++17", "-fPIC", "-shared", "-pthread"]

_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", *CXXFLAGS, "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        L.cpuq_gemv.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32]
        L.cpuq_gemv.restype = i32
        L.cpuq_hardware_concurrency.argtypes = []
        L.cpuq_hardware_concurrency.restype = i32
        _lib = L
    return _lib


def cores() -> int:
    return int(lib().cpuq_hardware_concurrency())


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None and a.size else None


class HostWeight:
    """A quantized matrix as host numpy arrays (the library's planar layout)."""

    def __init__(self, N, K, bits, group, packed, scale, zp, cb, row_ptr, col, val):
        self.N, self.K, self.bits, self.group = N, K, bits, group
        c = lambda a, dt: None if a is None else np.ascontiguousarray(a).view(dt)
        self.packed = c(packed, np.uint8)
        self.scale = c(scale, np.uint16)
        self.zp = c(zp, np.uint8)
        self.cb = c(cb, np.uint16)
        self.row_ptr = c(row_ptr, np.int32)
        self.col = c(col, np.int32)
        self.val = c(val, np.uint16)
        self.nnz = 0 if self.col is None else int(self.col.size)

    @staticmethod
    def from_device(qw) -> "HostWeight":
        h = lambda t: None if t is None else t.cpu().numpy()
        return HostWeight(qw.N, qw.K, qw.bits, qw.group, h(qw.packed), h(qw.scale), h(qw.zp), h(qw.codebook),
                          h(qw.row_ptr), h(qw.col), h(qw.val))

    @staticmethod
    def from_oracle(q) -> "HostWeight":
        return HostWeight(q.N, q.K, q.bits, q.group, q.packed, q.scale, q.zp, q.cb, q.row_ptr, q.col, q.val)

    def nbytes_packed(self) -> int:
        return int(self.packed.nbytes)


def gemv(x_f32: np.ndarray, w: HostWeight, y: np.ndarray | None = None, threads: int = 0) -> np.ndarray:
    """y [N] fp32 for one token x [K] (fp32)."""
    x_f32 = np.ascontiguousarray(x_f32, dtype=np.float32).ravel()
    assert x_f32.size == w.K
    if y is None:
        y = np.empty(w.N, np.float32)
    t = lib().cpuq_gemv(_p(x_f32), w.N, w.K, w.bits, w.group, _p(w.packed), _p(w.scale), _p(w.zp), _p(w.cb),
                        _p(w.row_ptr), _p(w.col), _p(w.val), w.nnz, _p(y), threads)
    if t < 0:
        raise ValueError("cpuq_gemv rejected its arguments")
    return y
