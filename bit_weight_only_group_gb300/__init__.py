"""Python binding of libqgemm: fused-dequantization linear layers over
weight-only, group-wise, asymmetric low-bit weights on GB300 (sm_103a).

This module only marshals arguments: PyTorch supplies device memory and the
current CUDA stream, and every step of the computation runs in the library's
own CUDA kernels, reached through the C ABI declared in ``include/qgemm.h``.
If ``libqgemm.so`` is missing the functions raise; there is no fallback.

Entry points (same names as the C ABI):

* ``qpack_query_sizes(N, K, bits, group, outlier_frac)`` -> dict of bytes
* ``qpack_quantize(W, bits, group, outlier_frac)`` -> :class:`QWeight`
* ``qgemm_forward(x, qw)`` -> y = x . (dequant(W) + outliers)^T
* ``qgemm_moe_grouped(x, topk_ids, experts)`` -> y [T, k, N]
* ``qgemm_moe_grouped_multi(x, topk_ids, [experts_0, experts_1])`` -> [y_0, y_1]
  (products sharing one routing, e.g. an MoE layer's gate and up)
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqgemm.so")

QG_OK = 0
STATUS_NAMES = {0: "QG_OK", -1: "QG_ERR_INVALID_ARG", -2: "QG_ERR_UNSUPPORTED", -3: "QG_ERR_ALIGNMENT",
                -4: "QG_ERR_WORKSPACE", -5: "QG_ERR_CUDA", -6: "QG_ERR_TIMEOUT", -7: "QG_ERR_DEVICE_STATUS"}
Y_F32, Y_BF16 = 0, 1

QUANT_MODES = {"asymmetric": 0, "symmetric": 1, "linear2": 2}

ABI_FUNCTIONS = ("qpack_query_sizes", "qpack_workspace_size", "qpack_quantize", "qpack_quantize_mode",
                 "qpack_quantize_noalloc",
                 "qgemm_workspace_size",
                 "qgemm_forward", "qgemm_forward_multi", "qgemm_moe_workspace_size", "qgemm_moe_grouped",
                 "qgemm_moe_grouped_multi",
                 "qgemm_device_status", "qgemm_selftest_bounded_wait", "qdiag_workspace_size", "qdiag_layer",
                 "qgemm_w8a8_workspace_size", "qgemm_forward_w8a8",
                 "qrepack_tiles_size", "qrepack_tiles", "qgemm_tiles_workspace_size", "qgemm_forward_tiles",
                 "qgemm_set_dependent_launch", "qgemm_last_error")


class QgError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class QgQWeight(ctypes.Structure):
    """Mirror of ``qg_qweight`` in include/qgemm.h."""
    _fields_ = [("N", ctypes.c_int32), ("K", ctypes.c_int32), ("bits", ctypes.c_int32),
                ("group", ctypes.c_int32), ("packed", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("zp", ctypes.c_void_p), ("codebook", ctypes.c_void_p), ("nnz", ctypes.c_int32),
                ("out_row_ptr", ctypes.c_void_p), ("out_col", ctypes.c_void_p),
                ("out_val", ctypes.c_void_p), ("scale8", ctypes.c_void_p), ("scale8_exp", ctypes.c_void_p),
                ("fb_row_ptr", ctypes.c_void_p), ("fb_col", ctypes.c_void_p), ("fb_val", ctypes.c_void_p),
                ("fb_cap", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m bit_weight_only_group_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        i32, f32, vp, sz = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
        psz, pi32 = ctypes.POINTER(sz), ctypes.POINTER(i32)
        pq = ctypes.POINTER(QgQWeight)
        L.qpack_query_sizes.argtypes = [i32, i32, i32, i32, f32, psz, psz, psz, psz, pi32]
        L.qpack_workspace_size.argtypes = [i32, i32, psz]
        L.qpack_quantize.argtypes = [vp, f32, pq, vp, sz, vp]
        L.qpack_quantize_mode.argtypes = [vp, f32, ctypes.c_int, pq, vp, sz, vp]
        L.qgemm_workspace_size.argtypes = [i32, pq, psz]
        L.qgemm_forward.argtypes = [vp, i32, i32, pq, vp, i32, ctypes.c_int, vp, sz, vp]
        L.qgemm_moe_workspace_size.argtypes = [i32, i32, i32, pq, psz]
        L.qgemm_moe_grouped.argtypes = [vp, i32, vp, i32, pq, i32, vp, ctypes.c_int, vp, sz, vp]
        L.qgemm_moe_grouped_multi.argtypes = [vp, i32, vp, i32, pq, i32, i32, ctypes.POINTER(vp), ctypes.c_int, vp,
                                              sz, vp]
        L.qgemm_device_status.argtypes = [pi32, i32]
        L.qgemm_selftest_bounded_wait.argtypes = [i32, vp]
        L.qdiag_workspace_size.argtypes = [i32, i32, i32, psz]
        L.qgemm_w8a8_workspace_size.argtypes = [i32, pq, psz]
        L.qrepack_tiles_size.argtypes = [pq, psz]
        L.qrepack_tiles.argtypes = [pq, vp, sz, vp]
        L.qgemm_tiles_workspace_size.argtypes = [i32, pq, psz]
        L.qgemm_forward_tiles.argtypes = [vp, i32, i32, pq, vp, vp, i32, ctypes.c_int, vp, sz, vp]
        L.qgemm_forward_w8a8.argtypes = [vp, i32, i32, pq, vp, i32, ctypes.c_int, vp, sz, vp]
        L.qdiag_layer.argtypes = [vp, pq, f32, vp, vp, vp, sz, vp]
        L.qgemm_forward_multi.argtypes = [vp, i32, i32, pq, i32, ctypes.POINTER(vp), pi32, ctypes.c_int, vp, sz, vp]
        for name in ABI_FUNCTIONS[:-1]:
            getattr(L, name).restype = ctypes.c_int
        L.qgemm_last_error.argtypes = []
        L.qgemm_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def last_error() -> str:
    return lib().qgemm_last_error().decode()


def _check(st: int, where: str):
    if st != QG_OK:
        raise QgError(st, where, last_error())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() else None


# --------------------------------------------------------------------- sizes
def qpack_query_sizes(N: int, K: int, bits: int, group: int, outlier_frac: float = 0.0) -> dict:
    p, s, z, c = (ctypes.c_size_t() for _ in range(4))
    n = ctypes.c_int32()
    _check(lib().qpack_query_sizes(N, K, bits, group, outlier_frac, ctypes.byref(p), ctypes.byref(s),
                                   ctypes.byref(z), ctypes.byref(c), ctypes.byref(n)), "qpack_query_sizes")
    return dict(packed=p.value, scale=s.value, zp=z.value, codebook=c.value, nnz=n.value)


def qpack_workspace_size(N: int, K: int) -> int:
    b = ctypes.c_size_t()
    _check(lib().qpack_workspace_size(N, K, ctypes.byref(b)), "qpack_workspace_size")
    return b.value


# --------------------------------------------------------------------- weights
@dataclass
class QWeight:
    """A quantized matrix in device memory (canonical planar layout)."""
    N: int
    K: int
    bits: int
    group: int
    packed: torch.Tensor                 # uint8 [N, K*bits/8]
    scale: torch.Tensor | None           # int16 (fp16 bits) [N, K/group]
    zp: torch.Tensor | None              # uint8 [N, K/group]
    codebook: torch.Tensor | None        # int16 (fp16 bits) [N, K/group, 4]
    row_ptr: torch.Tensor | None         # int32 [N+1]
    col: torch.Tensor | None             # int32 [nnz]
    val: torch.Tensor | None             # int16 (fp16 bits) [nnz]
    nnz: int = 0
    # 8-bit (E4M3) scales in place of ``scale``, with the fp16 fallback list
    scale8: torch.Tensor | None = None       # uint8 [N, K/group], 0x7F = fallback
    scale8_exp: torch.Tensor | None = None   # int32 [1]: the matrix exponent E
    fb_row_ptr: torch.Tensor | None = None   # int32 [N+1]
    fb_col: torch.Tensor | None = None       # int32 [fb_cap]
    fb_val: torch.Tensor | None = None       # int16 (fp16 bits) [fb_cap]

    @staticmethod
    def empty(N: int, K: int, bits: int, group: int, outlier_frac: float = 0.0, device="cuda",
              scale_fmt: str = "fp16", fb_cap: int | None = None) -> "QWeight":
        """Buffers for a quantized matrix.  scale_fmt 'fp8': 8-bit scales
        with a fallback list of fb_cap entries (default: 1 % of the groups,
        at least 64)."""
        sz = qpack_query_sizes(N, K, bits, group, outlier_frac)
        ng = K // group
        u8, i16, i32 = torch.uint8, torch.int16, torch.int32
        nnz = sz["nnz"]
        f8 = scale_fmt == "fp8"
        if f8 and fb_cap is None:
            fb_cap = max(64, N * ng // 100)
        return QWeight(
            N, K, bits, group,
            packed=torch.empty((N, K * bits // 8), dtype=u8, device=device),
            scale=torch.empty((N, ng), dtype=i16, device=device) if bits != 2 and not f8 else None,
            zp=torch.empty((N, ng), dtype=u8, device=device) if bits != 2 else None,
            codebook=torch.empty((N, ng, 4), dtype=i16, device=device) if bits == 2 else None,
            row_ptr=torch.empty(N + 1, dtype=i32, device=device),
            col=torch.empty(max(nnz, 1), dtype=i32, device=device)[:nnz],
            val=torch.empty(max(nnz, 1), dtype=i16, device=device)[:nnz],
            nnz=nnz,
            scale8=torch.empty((N, ng), dtype=u8, device=device) if f8 else None,
            scale8_exp=torch.zeros(1, dtype=i32, device=device) if f8 else None,
            fb_row_ptr=torch.zeros(N + 1, dtype=i32, device=device) if f8 else None,
            fb_col=torch.empty(max(fb_cap, 1), dtype=i32, device=device)[:fb_cap] if f8 else None,
            fb_val=torch.empty(max(fb_cap, 1), dtype=i16, device=device)[:fb_cap] if f8 else None)

    @property
    def fb_cap(self) -> int:
        return 0 if self.fb_col is None else int(self.fb_col.numel())

    def desc(self) -> QgQWeight:
        return QgQWeight(self.N, self.K, self.bits, self.group, _ptr(self.packed), _ptr(self.scale),
                         _ptr(self.zp), _ptr(self.codebook), self.nnz, _ptr(self.row_ptr),
                         _ptr(self.col), _ptr(self.val), _ptr(self.scale8), _ptr(self.scale8_exp),
                         _ptr(self.fb_row_ptr), _ptr(self.fb_col), _ptr(self.fb_val), self.fb_cap)

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in
                   (self.packed, self.scale, self.zp, self.codebook, self.row_ptr, self.col, self.val,
                    self.scale8, self.scale8_exp, self.fb_row_ptr, self.fb_col, self.fb_val)
                   if t is not None)


def qpack_quantize(W: torch.Tensor, bits: int, group: int, outlier_frac: float = 0.0,
                   out: QWeight | None = None, workspace: torch.Tensor | None = None, stream=None,
                   mode: str = "asymmetric", scale_fmt: str = "fp16", fb_cap: int | None = None) -> QWeight:
    """Quantize and pack W [N, K] (fp16, CUDA) on the device.  mode:
    'asymmetric' (qpack_quantize), 'symmetric' or 'linear2'
    (qpack_quantize_mode); scale_fmt 'fp8': 8-bit scales (bits 3..8)."""
    if W.dtype != torch.float16 or not W.is_cuda or W.dim() != 2:
        raise ValueError("W must be a 2-D float16 CUDA tensor")
    W = W.contiguous()
    N, K = W.shape
    qw = out if out is not None else QWeight.empty(N, K, bits, group, outlier_frac, W.device, scale_fmt, fb_cap)
    ws_bytes = qpack_workspace_size(N, K)
    ws = workspace if workspace is not None else torch.empty(ws_bytes, dtype=torch.uint8, device=W.device)
    d = qw.desc()
    if mode == "asymmetric":
        _check(lib().qpack_quantize(_ptr(W), outlier_frac, ctypes.byref(d), _ptr(ws), ws.numel(), _stream(stream)),
               "qpack_quantize")
    else:
        _check(lib().qpack_quantize_mode(_ptr(W), outlier_frac, QUANT_MODES[mode], ctypes.byref(d), _ptr(ws),
                                         ws.numel(), _stream(stream)), "qpack_quantize_mode")
    return qw


def qpack_quantize_noalloc(W: torch.Tensor, bits: int, group: int, outlier_frac: float = 0.0,
                           out: QWeight | None = None, stream=None, scale_fmt: str = "fp16") -> QWeight:
    """qpack_quantize for callers that cannot allocate device memory: the
    library uses its own fixed scratch array (see include/qgemm.h).  Pass
    ``out`` (allocated beforehand) to keep this call allocation-free."""
    if W.dtype != torch.float16 or not W.is_cuda or W.dim() != 2 or not W.is_contiguous():
        raise ValueError("W must be a contiguous 2-D float16 CUDA tensor")
    N, K = W.shape
    qw = out if out is not None else QWeight.empty(N, K, bits, group, outlier_frac, W.device, scale_fmt)
    f = lib().qpack_quantize_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_float, ctypes.POINTER(QgQWeight), ctypes.c_void_p]
    f.restype = ctypes.c_int
    d = qw.desc()
    _check(f(_ptr(W), outlier_frac, ctypes.byref(d), _stream(stream)), "qpack_quantize_noalloc")
    return qw


def qgemm_workspace_size(M: int, qw: QWeight) -> int:
    b = ctypes.c_size_t()
    d = qw.desc()
    _check(lib().qgemm_workspace_size(M, ctypes.byref(d), ctypes.byref(b)), "qgemm_workspace_size")
    return b.value


def qgemm_forward(x: torch.Tensor, qw: QWeight, out: torch.Tensor | None = None,
                  out_dtype: torch.dtype = torch.float32, workspace: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """y [M, N] = x [M, K] (bf16, CUDA) times (dequant(W) + outliers)^T."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D bfloat16 CUDA tensor with unit inner stride")
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, qw.N), dtype=out_dtype, device=x.device)
    yt = Y_BF16 if out.dtype == torch.bfloat16 else Y_F32
    if out.dtype not in (torch.float32, torch.bfloat16) or out.stride(1) != 1:
        raise ValueError("out must be float32 or bfloat16 with unit inner stride")
    need = qgemm_workspace_size(M, qw)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    d = qw.desc()
    _check(lib().qgemm_forward(_ptr(x), M, x.stride(0), ctypes.byref(d), _ptr(out), out.stride(0), yt,
                               _ptr(workspace) if need else None, workspace.numel() if need else 0,
                               _stream(stream)), "qgemm_forward")
    return out


def qgemm_forward_multi(x: torch.Tensor, qws, outs=None, out_dtype: torch.dtype = torch.float32,
                        workspace: torch.Tensor | None = None, stream=None):
    """[y_q [M, N_q] for each weight]: the products of x with up to four
    weights that share K, bits and group, in one call."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D bfloat16 CUDA tensor with unit inner stride")
    M = x.shape[0]
    if outs is None:
        outs = [torch.empty((M, q.N), dtype=out_dtype, device=x.device) for q in qws]
    if len(outs) != len(qws):
        raise ValueError("one output per weight")
    yt = Y_BF16 if outs[0].dtype == torch.bfloat16 else Y_F32
    for o in outs:
        if o.dtype != outs[0].dtype or o.dtype not in (torch.float32, torch.bfloat16) or o.stride(1) != 1:
            raise ValueError("outputs must share one dtype (float32 or bfloat16) with unit inner stride")
    need = max(qgemm_workspace_size(M, q) for q in qws)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    descs = _desc_array(qws)
    ys = (ctypes.c_void_p * len(outs))(*[o.data_ptr() for o in outs])
    ld = (ctypes.c_int32 * len(outs))(*[o.stride(0) for o in outs])
    _check(lib().qgemm_forward_multi(_ptr(x), M, x.stride(0), descs, len(qws), ys, ld, yt,
                                     _ptr(workspace) if need else None, workspace.numel() if need else 0,
                                     _stream(stream)), "qgemm_forward_multi")
    return outs


def _desc_array(experts):
    arr = (QgQWeight * len(experts))()
    for i, q in enumerate(experts):
        arr[i] = q.desc()
    return arr


def qgemm_moe_workspace_size(T: int, k: int, experts) -> int:
    b = ctypes.c_size_t()
    arr = _desc_array(experts)
    _check(lib().qgemm_moe_workspace_size(T, k, len(experts), arr, ctypes.byref(b)), "qgemm_moe_workspace_size")
    return b.value


def qgemm_moe_grouped(x: torch.Tensor, topk_ids: torch.Tensor, experts, out: torch.Tensor | None = None,
                      out_dtype: torch.dtype = torch.float32, workspace: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """y [T, k, N]: y[t, j] = x[t] . (dequant(W_e) + outliers_e)^T with e = topk_ids[t, j]."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous bfloat16 CUDA tensor [T, K]")
    if topk_ids.dtype != torch.int32 or not topk_ids.is_contiguous():
        raise ValueError("topk_ids must be a contiguous int32 tensor [T, k]")
    T, k = topk_ids.shape
    N = experts[0].N
    if out is None:
        out = torch.empty((T, k, N), dtype=out_dtype, device=x.device)
    yt = Y_BF16 if out.dtype == torch.bfloat16 else Y_F32
    arr = _desc_array(experts)
    need = qgemm_moe_workspace_size(T, k, experts)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    _check(lib().qgemm_moe_grouped(_ptr(x), T, _ptr(topk_ids), k, arr, len(experts), _ptr(out), yt,
                                   _ptr(workspace), workspace.numel(), _stream(stream)), "qgemm_moe_grouped")
    return out


def qgemm_moe_grouped_multi(x: torch.Tensor, topk_ids: torch.Tensor, experts_per_product, outs=None,
                            out_dtype: torch.dtype = torch.float32, workspace: torch.Tensor | None = None,
                            stream=None) -> list:
    """[y_p]: the grouped product of each expert list in experts_per_product
    (at most 2 lists of equal length, all matrices of one shape, width and
    group) over one routing of topk_ids."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous bfloat16 CUDA tensor [T, K]")
    if topk_ids.dtype != torch.int32 or not topk_ids.is_contiguous():
        raise ValueError("topk_ids must be a contiguous int32 tensor [T, k]")
    n = len(experts_per_product)
    E = len(experts_per_product[0])
    if any(len(ex) != E for ex in experts_per_product):
        raise ValueError("every product needs the same number of experts")
    T, k = topk_ids.shape
    N = experts_per_product[0][0].N
    if outs is None:
        outs = [torch.empty((T, k, N), dtype=out_dtype, device=x.device) for _ in range(n)]
    if len(outs) != n:
        raise ValueError("one output per product")
    yt = Y_BF16 if outs[0].dtype == torch.bfloat16 else Y_F32
    if any(o.dtype != outs[0].dtype for o in outs):
        raise ValueError("outputs must share one dtype")
    arr = _desc_array([w for ex in experts_per_product for w in ex])
    ys = (ctypes.c_void_p * n)(*[o.data_ptr() for o in outs])
    need = qgemm_moe_workspace_size(T, k, experts_per_product[0])
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    _check(lib().qgemm_moe_grouped_multi(_ptr(x), T, _ptr(topk_ids), k, arr, E, n, ys, yt, _ptr(workspace),
                                         workspace.numel(), _stream(stream)), "qgemm_moe_grouped_multi")
    return outs


def qgemm_set_dependent_launch(enable: bool) -> None:
    """Programmatic dependent launch of the dense products (decode and tensor-core kernels), process-wide."""
    lib().qgemm_set_dependent_launch.argtypes = [ctypes.c_int32]
    _check(lib().qgemm_set_dependent_launch(1 if enable else 0), "qgemm_set_dependent_launch")


def qgemm_device_status(reset: bool = False) -> int:
    """Status word of the decode kernels on the current device (0 = QG_OK,
    QG_ERR_TIMEOUT after a bounded wait gave up).  Synchronizes the device."""
    v = ctypes.c_int32(0)
    _check(lib().qgemm_device_status(ctypes.byref(v), 1 if reset else 0), "qgemm_device_status")
    return v.value


def qgemm_selftest_bounded_wait(poll_limit: int = 2, stream=None) -> None:
    """Launch the kernel whose bounded mbarrier wait must give up; afterwards
    qgemm_device_status() reads QG_ERR_TIMEOUT (-6)."""
    _check(lib().qgemm_selftest_bounded_wait(poll_limit, _stream(stream)), "qgemm_selftest_bounded_wait")


class QgDiag(ctypes.Structure):
    """Mirror of ``qg_diag`` in include/qgemm.h."""
    _fields_ = [("max_abs_err", ctypes.c_double), ("rmse", ctypes.c_double), ("cosine", ctypes.c_double),
                ("max_range_ratio", ctypes.c_double), ("groups_over", ctypes.c_int64)]


def qdiag_layer(W: torch.Tensor, qw: QWeight, threshold: float = 8.0, ratio: bool = False, stream=None):
    """Diagnostics of qw against the original fp16 W [N, K] (CUDA), computed
    on the device: dict of max_abs_err, rmse, cosine, max_range_ratio,
    groups_over (and the per-group ratio tensor [N, K/group] if asked).
    Reading the result synchronizes the stream."""
    if W.dtype != torch.float16 or not W.is_cuda or tuple(W.shape) != (qw.N, qw.K) or not W.is_contiguous():
        raise ValueError("W must be the contiguous fp16 CUDA [N, K] matrix of qw")
    b = ctypes.c_size_t()
    _check(lib().qdiag_workspace_size(qw.N, qw.K, qw.group, ctypes.byref(b)), "qdiag_workspace_size")
    ws = torch.empty(max(b.value, 1), dtype=torch.uint8, device=W.device)
    out = torch.zeros(5, dtype=torch.float64, device=W.device)   # one qg_diag (40 bytes)
    r = torch.empty((qw.N, qw.K // qw.group), dtype=torch.float32, device=W.device) if ratio else None
    d = qw.desc()
    _check(lib().qdiag_layer(_ptr(W), ctypes.byref(d), threshold, _ptr(r), _ptr(out), _ptr(ws), ws.numel(),
                             _stream(stream)), "qdiag_layer")
    raw = out.cpu().numpy().tobytes()
    res = QgDiag.from_buffer_copy(raw)
    o = dict(max_abs_err=res.max_abs_err, rmse=res.rmse, cosine=res.cosine, max_range_ratio=res.max_range_ratio,
             groups_over=int(res.groups_over))
    if ratio:
        o["ratio"] = r
    return o


def qgemm_forward_w8a8(x: torch.Tensor, qw: QWeight, out: torch.Tensor | None = None,
                       out_dtype: torch.dtype = torch.float32, workspace: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """W8A8 decode product (M <= 16): x [M, K] bf16 quantized to int8 per token
    inside the call, times the 8-bit weight qw."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D bfloat16 CUDA tensor with unit inner stride")
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, qw.N), dtype=out_dtype, device=x.device)
    yt = Y_BF16 if out.dtype == torch.bfloat16 else Y_F32
    b = ctypes.c_size_t()
    d = qw.desc()
    _check(lib().qgemm_w8a8_workspace_size(M, ctypes.byref(d), ctypes.byref(b)), "qgemm_w8a8_workspace_size")
    if b.value and (workspace is None or workspace.numel() < b.value):
        workspace = torch.empty(b.value, dtype=torch.uint8, device=x.device)
    _check(lib().qgemm_forward_w8a8(_ptr(x), M, x.stride(0), ctypes.byref(d), _ptr(out), out.stride(0), yt,
                                    _ptr(workspace) if b.value else None, workspace.numel() if b.value else 0,
                                    _stream(stream)), "qgemm_forward_w8a8")
    return out


def qrepack_tiles(qw: QWeight, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The tile-ordered copy of qw (uint8 CUDA tensor) for qgemm_forward_tiles."""
    b = ctypes.c_size_t()
    d = qw.desc()
    _check(lib().qrepack_tiles_size(ctypes.byref(d), ctypes.byref(b)), "qrepack_tiles_size")
    if out is None:
        out = torch.empty(b.value, dtype=torch.uint8, device=qw.packed.device)
    _check(lib().qrepack_tiles(ctypes.byref(d), _ptr(out), out.numel(), _stream(stream)), "qrepack_tiles")
    return out


def qgemm_forward_tiles(x: torch.Tensor, qw: QWeight, tiles: torch.Tensor, out: torch.Tensor | None = None,
                        out_dtype: torch.dtype = torch.float32, workspace: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """y = x . (dequant(W) + outliers)^T on the tensor cores from the tile-ordered copy."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D bfloat16 CUDA tensor with unit inner stride")
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, qw.N), dtype=out_dtype, device=x.device)
    yt = Y_BF16 if out.dtype == torch.bfloat16 else Y_F32
    d = qw.desc()
    b = ctypes.c_size_t()
    _check(lib().qgemm_tiles_workspace_size(M, ctypes.byref(d), ctypes.byref(b)), "qgemm_tiles_workspace_size")
    if b.value and (workspace is None or workspace.numel() < b.value):
        workspace = torch.empty(b.value, dtype=torch.uint8, device=x.device)
    _check(lib().qgemm_forward_tiles(_ptr(x), M, x.stride(0), ctypes.byref(d), _ptr(tiles), _ptr(out), out.stride(0),
                                     yt, _ptr(workspace) if b.value else None, workspace.numel() if b.value else 0,
                                     _stream(stream)), "qgemm_forward_tiles")
    return out
