"""Python face of the CPU oracle (``qoracle.c``).

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The product library
never calls it, and it never calls the product library.

Every function takes and returns numpy arrays (torch CPU tensors are accepted
as inputs).  fp16/bf16 data travel as their uint16 bit patterns.

What each function follows is cited in ``qoracle.c``; in short:
``quantize`` is the affine asymmetric quantizer ("Inference acceleration guide" page,
section 1.1) with per-group statistics after excluding the largest-magnitude
outliers, which are kept in FP16 ("70B on one GPU" page, section 2), a
4-entry k-means codebook at 2 bits ("Mixed-width quantization" page, sections 2.1 and 4.1) and
LSB-first packing ("Mixed-width quantization" page, sections 3.1-3.2); ``linear`` is
y = x . (x_hat + S)^T in fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qoracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile ``qoracle.c`` into ``liboracle.so`` with gcc (IEEE, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


class _QW(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("bits", ctypes.c_int32), ("group", ctypes.c_int32),
                ("packed", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("zp", ctypes.c_void_p), ("cb", ctypes.c_void_p),
                ("nnz", ctypes.c_int64), ("row_ptr", ctypes.c_void_p),
                ("col", ctypes.c_void_p), ("val", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
        L.orc_nnz.argtypes = [i64, i64, f32]
        L.orc_nnz.restype = i64
        L.orc_sizes.argtypes = [i64, i64, ctypes.c_int, ctypes.c_int, f32, vp]
        L.orc_sizes.restype = ctypes.c_int
        L.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_f16_to_f64.restype = ctypes.c_double
        L.orc_f32_to_f16_array.argtypes = [vp, i64, ctypes.c_int, vp]
        L.orc_f16_to_f32_array.argtypes = [vp, i64, vp]
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f64.restype = ctypes.c_double
        L.orc_pack.argtypes = [vp, i64, ctypes.c_int, vp]
        L.orc_unpack.argtypes = [vp, i64, ctypes.c_int, vp]
        L.orc_select_outliers.argtypes = [vp, i64, i64, f32, vp, vp]
        L.orc_select_outliers.restype = i64
        L.orc_quantize.argtypes = [vp, i64, i64, ctypes.c_int, ctypes.c_int, f32,
                                   vp, vp, vp, vp, vp, vp, vp]
        L.orc_quantize.restype = ctypes.c_int
        L.orc_quantize_mode.argtypes = [vp, i64, i64, ctypes.c_int, ctypes.c_int, f32, ctypes.c_int,
                                        vp, vp, vp, vp, vp, vp, vp]
        L.orc_quantize_mode.restype = ctypes.c_int
        L.orc_dequant_rows.argtypes = [ctypes.POINTER(_QW), i64, i64, vp]
        L.orc_dequant_rows.restype = ctypes.c_int
        L.orc_linear_rows.argtypes = [vp, i64, i64, ctypes.POINTER(_QW), i64, i64, vp]
        L.orc_linear_rows.restype = ctypes.c_int
        L.orc_quantize_act_int8.argtypes = [vp, i64, i64, i64, vp, vp]
        L.orc_quantize_act_int8.restype = ctypes.c_int
        L.orc_linear_w8a8.argtypes = [vp, i64, i64, i64, ctypes.POINTER(_QW), i64, i64, vp]
        L.orc_linear_w8a8.restype = ctypes.c_int
        L.orc_diagnostics.argtypes = [vp, ctypes.POINTER(_QW), ctypes.c_double, vp, vp]
        L.orc_diagnostics.restype = ctypes.c_int
        L.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_to_f64.restype = ctypes.c_double
        L.orc_e4m3_ceil_normal.argtypes = [ctypes.c_double]
        L.orc_e4m3_ceil_normal.restype = ctypes.c_int
        L.orc_fp8_matrix_exponent.argtypes = [vp, i64]
        L.orc_fp8_matrix_exponent.restype = ctypes.c_int
        L.orc_quantize_fp8.argtypes = [vp, i64, i64, ctypes.c_int, ctypes.c_int, f32, ctypes.c_int,
                                       vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64]
        L.orc_quantize_fp8.restype = i64
        L.orc_fp8_expand.argtypes = [vp, i32, i64, i64, vp, vp, vp, vp]
        L.orc_fp8_expand.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None and a.size else None


def as_u16(a) -> np.ndarray:
    """fp16 / bf16 data (numpy or torch, CPU) as a contiguous uint16 array."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous().view(torch.int16).numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    return a.view(np.uint16)


# ------------------------------------------------------------------ scalars
def nnz(N: int, K: int, frac: float) -> int:
    return int(lib().orc_nnz(N, K, float(np.float32(frac))))


def sizes(N, K, bits, group, frac):
    """Bytes of (packed, scale, zp, codebook, nnz, row_ptr, col, val)."""
    out = np.zeros(8, np.int64)
    rc = lib().orc_sizes(N, K, bits, group, float(np.float32(frac)), _p(out))
    if rc != 0:
        raise ValueError(f"orc_sizes rejected N={N} K={K} bits={bits} group={group} frac={frac}")
    keys = ("packed", "scale", "zp", "codebook", "nnz", "row_ptr", "col", "val")
    return dict(zip(keys, (int(v) for v in out)))


def f32_to_f16(a, mode: str = "rn") -> np.ndarray:
    """IEEE binary16 bit patterns of float32 values; mode 'rn' (ties to even) or 'ru' (toward +inf)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    lib().orc_f32_to_f16_array(_p(a), a.size, 0 if mode == "rn" else 1, _p(out))
    return out


def f16_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().orc_f16_to_f32_array(_p(h), h.size, _p(out))
    return out


def bf16_to_f64(b) -> np.ndarray:
    b = as_u16(b).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ------------------------------------------------------------------ packing
def pack(codes, bits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8).ravel()
    out = np.empty((codes.size * bits + 7) // 8, np.uint8)
    lib().orc_pack(_p(codes), codes.size, bits, _p(out))
    return out


def unpack(data, n: int, bits: int) -> np.ndarray:
    data = np.ascontiguousarray(data, dtype=np.uint8).ravel()
    out = np.empty(n, np.uint8)
    lib().orc_unpack(_p(data), n, bits, _p(out))
    return out


# ------------------------------------------------------------------ quantizer
@dataclass
class QWeight:
    """A quantized matrix in the canonical planar layout (numpy, host)."""
    N: int
    K: int
    bits: int
    group: int
    packed: np.ndarray            # uint8 [N, K*bits/8]
    scale: np.ndarray | None      # uint16 (fp16) [N, K/group]
    zp: np.ndarray | None         # uint8 [N, K/group]
    cb: np.ndarray | None         # uint16 (fp16) [N, K/group, 4]
    row_ptr: np.ndarray           # int32 [N+1]
    col: np.ndarray               # int32 [nnz]
    val: np.ndarray               # uint16 (fp16) [nnz]
    # E4M3 scales (``scale_fmt='fp8'``): ``scale`` then holds the fp16 value
    # each group stores, expanded from these by ``orc_fp8_expand``
    scale8: np.ndarray | None = None      # uint8 [N, K/group], 0x7F = fp16 fallback
    scale_exp: int = 0                    # the matrix exponent E
    fb_row_ptr: np.ndarray | None = None  # int32 [N+1]
    fb_col: np.ndarray | None = None      # int32 [nfb] group index within the row
    fb_val: np.ndarray | None = None      # uint16 (fp16) [nfb]

    @property
    def nnz(self) -> int:
        return int(self.col.size)

    def _struct(self) -> _QW:
        return _QW(self.N, self.K, self.bits, self.group, _p(self.packed),
                   _p(self.scale) if self.scale is not None else None,
                   _p(self.zp) if self.zp is not None else None,
                   _p(self.cb) if self.cb is not None else None,
                   self.nnz, _p(self.row_ptr), _p(self.col), _p(self.val))


def select_outliers(W, frac: float):
    """CSR (row_ptr, col) of the floor(frac*N*K) largest |w| (ties: lower index)."""
    W = as_u16(W)
    N, K = W.shape
    n = nnz(N, K, frac)
    row_ptr = np.empty(N + 1, np.int32)
    col = np.empty(max(n, 1), np.int32)
    got = lib().orc_select_outliers(_p(W), N, K, float(np.float32(frac)), _p(row_ptr), _p(col))
    if got < 0:
        raise RuntimeError(f"orc_select_outliers failed ({got})")
    return row_ptr, col[:n]


MODES = {"asymmetric": 0, "symmetric": 1, "linear2": 2}


def quantize(W, bits: int, group: int, frac: float = 0.0, mode: str = "asymmetric",
             scale_fmt: str = "fp16") -> QWeight:
    """Quantize and pack W [N, K] (fp16).  mode: 'asymmetric' (affine with a
    zero point at 3-8 bits, k-means codebook at 2), 'symmetric' (no zero
    point: the affine format with the zero point fixed at 2^(b-1); at 2
    bits the constants -s, 0, s, s) or 'linear2' (2 bits only: the affine
    grid's four constants).  scale_fmt 'fp8' (bits 3-8, asymmetric or
    symmetric): E4M3 group scales with an fp16 fallback (``orc_quantize_fp8``)."""
    W = as_u16(W)
    N, K = W.shape
    sz = sizes(N, K, bits, group, frac)
    ng = K // group
    n = sz["nnz"]
    packed = np.empty((N, K * bits // 8), np.uint8)
    row_ptr = np.empty(N + 1, np.int32)
    col = np.empty(max(n, 1), np.int32)
    val = np.empty(max(n, 1), np.uint16)
    if scale_fmt == "fp8":
        scale8 = np.empty((N, ng), np.uint8)
        zp = np.empty((N, ng), np.uint8)
        E = ctypes.c_int32(0)
        fb_row_ptr = np.empty(N + 1, np.int32)
        fb_col = np.empty(N * ng, np.int32)
        fb_val = np.empty(N * ng, np.uint16)
        nfb = lib().orc_quantize_fp8(_p(W), N, K, bits, group, float(np.float32(frac)), MODES[mode],
                                     _p(packed), _p(scale8), _p(zp), _p(row_ptr), _p(col), _p(val),
                                     ctypes.addressof(E), _p(fb_row_ptr), _p(fb_col), _p(fb_val), N * ng)
        if nfb < 0:
            raise ValueError(f"orc_quantize_fp8 failed ({nfb})")
        scale = np.empty((N, ng), np.uint16)
        rc = lib().orc_fp8_expand(_p(scale8), E.value, N, ng, _p(fb_row_ptr), _p(fb_col), _p(fb_val), _p(scale))
        if rc != 0:
            raise ValueError(f"orc_fp8_expand failed ({rc})")
        return QWeight(N, K, bits, group, packed, scale, zp, None, row_ptr, col[:n], val[:n],
                       scale8, E.value, fb_row_ptr, fb_col[:nfb].copy(), fb_val[:nfb].copy())
    assert scale_fmt == "fp16", scale_fmt
    scale = np.empty((N, ng), np.uint16) if bits != 2 else None
    zp = np.empty((N, ng), np.uint8) if bits != 2 else None
    cb = np.empty((N, ng, 4), np.uint16) if bits == 2 else None
    rc = lib().orc_quantize_mode(_p(W), N, K, bits, group, float(np.float32(frac)), MODES[mode], _p(packed),
                            _p(scale) if scale is not None else None,
                            _p(zp) if zp is not None else None,
                            _p(cb) if cb is not None else None,
                            _p(row_ptr), _p(col), _p(val))
    if rc != 0:
        raise ValueError(f"orc_quantize failed ({rc})")
    return QWeight(N, K, bits, group, packed, scale, zp, cb, row_ptr, col[:n], val[:n])


def e4m3_value(code: int) -> float:
    """Value of an E4M3 byte (``orc_e4m3_to_f64``)."""
    return lib().orc_e4m3_to_f64(code)


def e4m3_ceil_normal(t: float) -> int:
    """Least normal E4M3 code with value >= t, or -1 (``orc_e4m3_ceil_normal``)."""
    return lib().orc_e4m3_ceil_normal(float(t))


def fp8_matrix_exponent(s16) -> int:
    """Lower median of floor(log2 s) over fp16 scales (``orc_fp8_matrix_exponent``)."""
    s16 = np.ascontiguousarray(as_u16(s16)).ravel()
    return lib().orc_fp8_matrix_exponent(_p(s16), s16.size)


def dequant(q: QWeight, n0: int = 0, n1: int | None = None) -> np.ndarray:
    """x_hat + S for rows [n0, n1) as float64 [n1-n0, K]."""
    n1 = q.N if n1 is None else n1
    out = np.empty((n1 - n0, q.K), np.float64)
    s = q._struct()
    rc = lib().orc_dequant_rows(ctypes.byref(s), n0, n1, _p(out))
    if rc != 0:
        raise ValueError(f"orc_dequant_rows failed ({rc})")
    return out


def linear(x, q: QWeight, n0: int = 0, n1: int | None = None) -> np.ndarray:
    """y [M, n1-n0] = x . (x_hat + S)[n0:n1]^T in fp64; x bf16 [M, K]."""
    x = as_u16(x)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    assert K == q.K, (K, q.K)
    n1 = q.N if n1 is None else n1
    y = np.empty((M, n1 - n0), np.float64)
    s = q._struct()
    rc = lib().orc_linear_rows(_p(x), M, K, ctypes.byref(s), n0, n1, _p(y))
    if rc != 0:
        raise ValueError(f"orc_linear_rows failed ({rc})")
    return y


def quantize_act_int8(x):
    """(q int8 [M, K], s fp32 [M]): per-token symmetric INT8 quantization of bf16 x."""
    x = as_u16(x)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    q = np.empty((M, K), np.int8)
    s = np.empty(M, np.float32)
    lib().orc_quantize_act_int8(_p(np.ascontiguousarray(x)), M, K, K, _p(q), _p(s))
    return q, s


def linear_w8a8(x, q: QWeight, n0: int = 0, n1: int | None = None) -> np.ndarray:
    """y [M, n1-n0] = (int8-quantized x) . (x_hat + S)[n0:n1]^T in fp64."""
    x = as_u16(x)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    n1 = q.N if n1 is None else n1
    y = np.empty((M, n1 - n0), np.float64)
    s = q._struct()
    rc = lib().orc_linear_w8a8(_p(np.ascontiguousarray(x)), M, K, K, ctypes.byref(s), n0, n1, _p(y))
    if rc != 0:
        raise ValueError(f"orc_linear_w8a8 failed ({rc})")
    return y


def tile_param_bytes(bits: int, group: int) -> int:
    """Parameter bytes per row of one tile block: 4 (fp16 scale | zp << 16)
    or 8 (2-bit codebook) per group the 64-wide K block touches (two at
    group 32, else one)."""
    return (8 if bits == 2 else 4) * (2 if group == 32 else 1)


def tiles(q: QWeight) -> np.ndarray:
    """The tile-ordered copy of q, written out block by block from the planar
    arrays: for each 256-row tile and 64-wide K block, 512 * bits words (word
    i of thread t = 2r + h at i * 512 + t, the thread's chunk being the 32
    codes [64 kb + 32 h, 64 kb + 32 h + 32) of row r as 4 * bits bytes of the
    LSB-first stream), then per row the parameters of the groups the block
    touches in ascending order: the parameter word (fp16 scale | zp << 16)
    or, at 2 bits, the 4 fp16 codebook entries.  Rows past N stay 0."""
    b, K, N = q.bits, q.K, q.N
    KB, NT = K // 64, (N + 255) // 256
    pb = tile_param_bytes(b, q.group)
    blk = 2048 * b + 256 * pb
    out = np.zeros(NT * KB * blk, np.uint8)
    for nt in range(NT):
        for kb in range(KB):
            base = (nt * KB + kb) * blk
            words = out[base:base + 2048 * b].view(np.uint32).reshape(b, 512)
            prm = out[base + 2048 * b:base + blk]
            groups = sorted({(64 * kb + 32 * h) // q.group for h in range(2)})
            for r in range(256):
                n = nt * 256 + r
                if n >= N:
                    continue
                for h in range(2):
                    lo = (2 * kb + h) * 4 * b
                    words[:, 2 * r + h] = q.packed[n, lo:lo + 4 * b].view(np.uint32)
                for i, g in enumerate(groups):
                    at = pb * r + (pb // len(groups)) * i
                    if b == 2:
                        prm[at:at + 8] = q.cb[n, g].view(np.uint8)
                    else:
                        prm[at:at + 4] = np.array([int(q.scale[n, g]) | (int(q.zp[n, g]) << 16)],
                                                  np.uint32).view(np.uint8)
    return out


def diagnostics(W, q: QWeight, threshold: float = 8.0):
    """Per-layer diagnostics of q against the original fp16 W: dict with
    max_abs_err, rmse, cosine, max_range_ratio, groups_over (threshold) and
    the per-group ratio array [N, K/group] (see ``orc_diagnostics``)."""
    W = as_u16(W)
    assert W.shape == (q.N, q.K)
    out = np.zeros(5, np.float64)
    ratio = np.empty((q.N, q.K // q.group), np.float64)
    s = q._struct()
    rc = lib().orc_diagnostics(_p(np.ascontiguousarray(W)), ctypes.byref(s), float(threshold), _p(out), _p(ratio))
    if rc != 0:
        raise ValueError(f"orc_diagnostics failed ({rc})")
    return dict(max_abs_err=out[0], rmse=out[1], cosine=out[2], max_range_ratio=out[3], groups_over=int(out[4]),
                ratio=ratio)


def moe(x, topk, experts) -> np.ndarray:
    """y [T, k, N] with y[t, j] = x[t] . (x_hat + S)_{topk[t, j]}^T (no gate weights).

    Routing is plain selection: the rows routed to each expert are gathered,
    passed through ``linear`` with that expert's weights, and written back.
    """
    x = as_u16(x)
    topk = np.asarray(topk)
    T, k = topk.shape
    N = experts[0].N
    y = np.zeros((T, k, N), np.float64)
    for e, q in enumerate(experts):
        tt, jj = np.nonzero(topk == e)
        if tt.size == 0:
            continue
        y[tt, jj] = linear(x[tt], q)
    return y
