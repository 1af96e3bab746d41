"""qpack_quantize_noalloc -- the quantizer entry point for callers that
cannot allocate device memory (code inside an application that owns the
allocator, or where cudaMalloc's implicit synchronization is not allowed) --
gives the same bytes as qpack_quantize with a caller workspace.

Both are called through the C ABI with ctypes.  Two noalloc calls in a row
(different shapes and widths) check that the shared scratch array, which
keeps the previous call's contents, does not leak into the next result.
This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _parity import assert_quantized_equal

pytestmark = pytest.mark.gpu


def _quantize_with_workspace(qg, W, bits, group, frac):
    qw = qg.QWeight.empty(W.shape[0], W.shape[1], bits, group, frac)
    ws = torch.empty(qg.qpack_workspace_size(*W.shape), dtype=torch.uint8, device="cuda")
    d = qw.desc()
    st = qg.lib().qpack_quantize(ctypes.c_void_p(W.data_ptr()), frac, ctypes.byref(d),
                                 ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, qg.last_error()
    return qw


def _quantize_noalloc(qg, W, bits, group, frac):
    qw = qg.QWeight.empty(W.shape[0], W.shape[1], bits, group, frac)
    f = qg.lib().qpack_quantize_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_float, ctypes.POINTER(qg.QgQWeight), ctypes.c_void_p]
    f.restype = ctypes.c_int
    d = qw.desc()
    st = f(ctypes.c_void_p(W.data_ptr()), frac, ctypes.byref(d),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, qg.last_error()
    return qw


def _same(a, b):
    for name in ("packed", "scale", "zp", "codebook", "row_ptr", "col", "val"):
        ta, tb = getattr(a, name), getattr(b, name)
        if ta is None:
            assert tb is None
            continue
        assert torch.equal(ta, tb), name


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    import bit_weight_only_group_gb300 as qg
    cases = [(256, 2048, 4, 128, 0.002, 11), (130, 1024, 2, 64, 0.01, 12)]
    for N, K, bits, group, frac, seed in cases:
        W = wl.gen_weight(N, K, seed=seed, outlier_frac=frac, outlier_seed=seed + 1).cuda()
        ref = _quantize_with_workspace(qg, W, bits, group, frac)
        got = _quantize_noalloc(qg, W, bits, group, frac)
        torch.cuda.synchronize()
        _same(got, ref)
        # and the bytes are the oracle's
        assert_quantized_equal(got, oracle.quantize(W.cpu(), bits, group, frac))


def test_noalloc_rejects_matrices_with_outliers_beyond_its_scratch():
    # with outliers the selection needs 12 bytes of scratch per row: 100,000
    # rows do not fit the fixed array and the call is refused before any launch
    import bit_weight_only_group_gb300 as qg
    N, K = 100_000, 64
    nnz = oracle.nnz(N, K, 0.001)
    d = qg.QgQWeight(N, K, 4, 64, 0x100000, 0x200000, 0x300000, None, nnz, 0x500000, 0x600000, 0x700000)
    f = qg.lib().qpack_quantize_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_float, ctypes.POINTER(qg.QgQWeight), ctypes.c_void_p]
    f.restype = ctypes.c_int
    st = f(ctypes.c_void_p(0x400000), 0.001, ctypes.byref(d), None)
    assert st == -4
    assert "scratch" in qg.last_error()


def test_noalloc_without_outliers_takes_any_row_count():
    # no outliers: no scratch is used, so a matrix far above the scratch's
    # row limit quantizes, with the same bytes as the workspace entry point
    import bit_weight_only_group_gb300 as qg
    N, K = 100_000, 128
    W = wl.gen_weight(N, K, seed=21).cuda()
    ref = _quantize_with_workspace(qg, W, 4, 128, 0.0)
    got = _quantize_noalloc(qg, W, 4, 128, 0.0)
    torch.cuda.synchronize()
    _same(got, ref)
