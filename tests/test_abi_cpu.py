"""The C-ABI library without a GPU: it builds, loads, exports every symbol
the header declares, answers the host-only size queries like the oracle, and
rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qg():
    from bit_weight_only_group_gb300 import build
    build.build()
    import bit_weight_only_group_gb300 as qg
    return qg


def _declared():
    src = open(os.path.join(ROOT, "include", "qgemm.h")).read()
    return re.findall(r"QG_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)


def test_every_declared_symbol_is_exported(qg):
    names = _declared()
    assert set(names) == set(qg.ABI_FUNCTIONS)
    L = qg.lib()
    for n in names:
        assert hasattr(L, n), n


@pytest.mark.parametrize("N,K,bits,group,frac", [
    (4096, 4096, 4, 128, 0.0), (4096, 4096, 2, 128, 0.001), (11008, 4096, 3, 64, 0.001),
    (4096, 11008, 5, 128, 0.001), (1024, 8192, 6, 64, 0.002), (7, 64, 2, 64, 0.5), (4096, 4096, 3, 32, 0.001),
    (96, 256, 2, 32, 0.0)])
def test_sizes_match_oracle(qg, N, K, bits, group, frac):
    got = qg.qpack_query_sizes(N, K, bits, group, frac)
    ref = oracle.sizes(N, K, bits, group, frac)
    for k in ("packed", "scale", "zp", "codebook", "nnz"):
        assert got[k] == ref[k], k


def test_sizes_reject_bad_shapes(qg):
    with pytest.raises(qg.QgError) as e:
        qg.qpack_query_sizes(64, 100, 4, 64)
    assert e.value.status == -1
    with pytest.raises(qg.QgError) as e:
        qg.qpack_query_sizes(64, 128, 7, 64)
    assert e.value.status == -2
    with pytest.raises(qg.QgError) as e:
        qg.qpack_query_sizes(64, 128, 4, 16)
    assert e.value.status == -2
    with pytest.raises(qg.QgError) as e:
        qg.qpack_query_sizes(64, 128, 4, 64, 1.0)
    assert e.value.status == -1
    with pytest.raises(qg.QgError):
        qg.qpack_query_sizes(0, 128, 4, 64)


def _fake_desc(qg, N=64, K=128, bits=4, group=64, nnz=0, base=0x100000):
    d = qg.QgQWeight(N, K, bits, group, base, base + 0x10000, base + 0x20000, 0, nnz, None, None, None)
    if bits == 2:
        d.scale = None
        d.zp = None
        d.codebook = base + 0x30000
    return d


def test_scale8_descriptor_checks_without_gpu(qg):
    # 8-bit scales: the products and the quantizers refuse a descriptor whose
    # 8-bit scale arrays are missing or misaligned, before any launch
    L = qg.lib()
    y = ctypes.c_void_p(0x200000)
    x = ctypes.c_void_p(0x300000)

    def d8(**kw):
        d = _fake_desc(qg)
        d.scale = None
        d.scale8, d.scale8_exp, d.fb_row_ptr = 0x140000, 0x150000, 0x160000
        d.fb_col, d.fb_val, d.fb_cap = 0x170000, 0x180000, 16
        for k, v in kw.items():
            setattr(d, k, v)
        return d

    cases = [(d8(scale8_exp=None), -1), (d8(fb_row_ptr=None), -1), (d8(fb_col=None), -1),
             (d8(fb_cap=-1), -1), (d8(scale8_exp=0x150002), -3), (d8(fb_val=0x180001), -3),
             (d8(zp=None), -1)]
    d2 = _fake_desc(qg, bits=2)
    d2.scale8 = 0x140000
    cases.append((d2, -1))
    for d, expect in cases:
        assert L.qgemm_forward(x, 1, 128, ctypes.byref(d), y, 64, 0, None, 0, None) == expect, qg.last_error()
        assert L.qpack_quantize(x, 0.0, ctypes.byref(d), None, 0, None) == expect
    # fb_cap = 0 needs no list arrays
    ok = d8(fb_col=None, fb_val=None, fb_cap=0)
    assert L.qpack_quantize(x, 0.0, ctypes.byref(ok), None, 0, None) == -4   # passes the checks, lacks workspace


def test_host_validation_without_gpu(qg):
    L = qg.lib()
    d = _fake_desc(qg)
    y = ctypes.c_void_p(0x200000)
    x = ctypes.c_void_p(0x300000)
    # null x
    assert L.qgemm_forward(None, 1, 128, ctypes.byref(d), y, 64, 0, None, 0, None) == -1
    assert "null" in qg.last_error()
    # ldx < K, ldy < N
    assert L.qgemm_forward(x, 1, 64, ctypes.byref(d), y, 64, 0, None, 0, None) == -1
    assert L.qgemm_forward(x, 1, 128, ctypes.byref(d), y, 32, 0, None, 0, None) == -1
    # M = 0 is a no-op
    assert L.qgemm_forward(None, 0, 128, ctypes.byref(d), None, 64, 0, None, 0, None) == 0
    # misaligned packed
    bad = _fake_desc(qg, base=0x100004)
    assert L.qgemm_forward(x, 1, 128, ctypes.byref(bad), y, 64, 0, None, 0, None) == -3
    # unsupported width and group
    for dd in (_fake_desc(qg, bits=7), _fake_desc(qg, group=16)):
        assert L.qgemm_forward(x, 1, 128, ctypes.byref(dd), y, 64, 0, None, 0, None) == -2
    # outliers declared but arrays missing
    assert L.qgemm_forward(x, 1, 128, ctypes.byref(_fake_desc(qg, nnz=3)), y, 64, 0, None, 0, None) == -1
    # 2-bit needs a codebook
    d2 = _fake_desc(qg, bits=2)
    d2.codebook = None
    assert L.qgemm_forward(x, 1, 128, ctypes.byref(d2), y, 64, 0, None, 0, None) == -1


def test_quantize_validation_without_gpu(qg):
    L = qg.lib()
    W = ctypes.c_void_p(0x400000)
    d = _fake_desc(qg, N=64, K=1024, nnz=oracle.nnz(64, 1024, 0.001))
    d.out_row_ptr, d.out_col, d.out_val = 0x500000, 0x510000, 0x520000
    ws_need = qg.qpack_workspace_size(64, 1024)
    ws = ctypes.c_void_p(0x600000)
    # nnz must equal floor(frac*N*K)
    assert L.qpack_quantize(W, 0.002, ctypes.byref(d), ws, ws_need, None) == -1
    # workspace too small / missing
    assert L.qpack_quantize(W, 0.001, ctypes.byref(d), ws, ws_need - 1, None) == -4
    assert L.qpack_quantize(W, 0.001, ctypes.byref(d), None, ws_need, None) == -4
    # misaligned W and workspace
    assert L.qpack_quantize(ctypes.c_void_p(0x400002), 0.001, ctypes.byref(d), ws, ws_need, None) == -3
    assert L.qpack_quantize(W, 0.001, ctypes.byref(d), ctypes.c_void_p(0x600010), ws_need, None) == -3


def test_both_quantizers_refuse_the_same_bad_descriptors(qg):
    # qpack_quantize and qpack_quantize_noalloc share their argument checks:
    # each bad descriptor gets the same status from both, before any launch
    L = qg.lib()
    f = L.qpack_quantize_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_float, ctypes.POINTER(qg.QgQWeight), ctypes.c_void_p]
    f.restype = ctypes.c_int
    W = ctypes.c_void_p(0x400000)
    ws = ctypes.c_void_p(0x600000)

    def good():
        d = _fake_desc(qg, N=64, K=1024, nnz=oracle.nnz(64, 1024, 0.001))
        d.out_row_ptr, d.out_col, d.out_val = 0x500000, 0x510000, 0x520000
        return d

    cases = []
    d = good(); d.out_col = 0x510002; cases.append(("misaligned out_col", d, 0.001, -3))
    d = good(); d.out_val = 0x520001; cases.append(("misaligned out_val", d, 0.001, -3))
    d = good(); d.out_row_ptr = 0x500002; cases.append(("misaligned row_ptr", d, 0.001, -3))
    d = good(); d.scale = 0x110001; cases.append(("misaligned scale", d, 0.001, -3))
    d = good(); d.bits, d.scale, d.zp, d.codebook = 2, None, None, 0x130004
    cases.append(("misaligned codebook", d, 0.001, -3))
    d = good(); d.packed = 0x100008; cases.append(("misaligned packed", d, 0.001, -3))
    d = good(); cases.append(("wrong nnz", d, 0.002, -1))
    d = good(); d.out_col = None; cases.append(("null outlier array", d, 0.001, -1))
    d = good(); d.N, d.K, d.nnz = 1 << 20, 1 << 15, 0; cases.append(("N*K above the product limit", d, 0.0, -1))
    d = good(); d.bits = 7; cases.append(("unsupported width", d, 0.001, -2))
    d = good(); d.group = 256; cases.append(("unsupported group", d, 0.001, -2))
    d = good(); cases.append(("outlier_frac out of range", d, 1.5, -1))
    for what, d, frac, expect in cases:
        a = L.qpack_quantize(W, frac, ctypes.byref(d), ws, 1 << 30, None)
        b = f(W, frac, ctypes.byref(d), None)
        assert a == b == expect, (what, a, b)
    assert f(ctypes.c_void_p(0x400002), 0.001, ctypes.byref(good()), None) == -3   # misaligned W
    assert f(None, 0.001, ctypes.byref(good()), None) == -1


def test_quantize_mode_validation_without_gpu(qg):
    L = qg.lib()
    W = ctypes.c_void_p(0x400000)
    ws = ctypes.c_void_p(0x600000)
    d = _fake_desc(qg, N=64, K=1024)
    need = qg.qpack_workspace_size(64, 1024)
    assert L.qpack_quantize_mode(W, 0.0, 7, ctypes.byref(d), ws, need, None) == -1      # unknown mode
    assert L.qpack_quantize_mode(W, 0.0, 2, ctypes.byref(d), ws, need, None) == -2      # linear2 needs 2 bits
    assert L.qpack_quantize_mode(W, 0.0, 1, ctypes.byref(d), ws, need - 1, None) == -4  # workspace
    assert L.qpack_quantize_mode(ctypes.c_void_p(0x400002), 0.0, 1, ctypes.byref(d), ws, need, None) == -3


def test_w8a8_validation_without_gpu(qg):
    L = qg.lib()
    x, y, ws = ctypes.c_void_p(0x300000), ctypes.c_void_p(0x200000), ctypes.c_void_p(0x600000)
    d4 = _fake_desc(qg, N=64, K=128)
    d8 = _fake_desc(qg, N=64, K=128, bits=8)
    need = ctypes.c_size_t()
    assert L.qgemm_w8a8_workspace_size(4, ctypes.byref(d8), ctypes.byref(need)) == 0 and need.value > 0
    assert L.qgemm_forward_w8a8(x, 4, 128, ctypes.byref(d4), y, 64, 0, ws, need.value, None) == -2   # not 8-bit
    assert L.qgemm_forward_w8a8(x, 17, 128, ctypes.byref(d8), y, 64, 0, ws, need.value, None) == -2  # M > 16
    assert L.qgemm_forward_w8a8(x, 4, 128, ctypes.byref(d8), y, 64, 0, ws, need.value - 1, None) == -4
    assert L.qgemm_forward_w8a8(x, 0, 128, ctypes.byref(d8), y, 64, 0, None, 0, None) == 0            # no-op


def test_diagnostics_validation_without_gpu(qg):
    L = qg.lib()
    d = _fake_desc(qg, N=64, K=1024)
    need = ctypes.c_size_t()
    assert L.qdiag_workspace_size(64, 1024, 64, ctypes.byref(need)) == 0 and need.value > 0
    W, out, ws = ctypes.c_void_p(0x400000), ctypes.c_void_p(0x700000), ctypes.c_void_p(0x600000)
    assert L.qdiag_layer(None, ctypes.byref(d), 8.0, None, out, ws, need.value, None) == -1
    assert L.qdiag_layer(W, ctypes.byref(d), 8.0, None, ctypes.c_void_p(0x700004), ws, need.value, None) == -3
    assert L.qdiag_layer(W, ctypes.byref(d), 8.0, None, out, ws, need.value - 1, None) == -4
    assert L.qdiag_layer(W, ctypes.byref(d), float("nan"), None, out, ws, need.value, None) == -1


def test_valid_call_without_a_device_reports_cuda_error(qg):
    # every argument passes host validation; the first CUDA call then fails
    # (no device here) and the status says so instead of crashing
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    L = qg.lib()
    d = _fake_desc(qg)
    st = L.qgemm_forward(ctypes.c_void_p(0x300000), 1, 128, ctypes.byref(d), ctypes.c_void_p(0x200000), 64, 0,
                         None, 0, None)
    assert st == -5
    assert qg.last_error()


def test_forward_multi_validation_without_gpu(qg):
    # bad counts, mismatched weights and null outputs are rejected on the host
    L = qg.lib()
    d = _fake_desc(qg)
    arr = (qg.QgQWeight * 2)(d, d)
    ys = (ctypes.c_void_p * 2)(0x200000, 0x300000)
    ld = (ctypes.c_int32 * 2)(d.N, d.N)
    x = ctypes.c_void_p(0x100000)
    assert L.qgemm_forward_multi(x, 1, d.K, arr, 0, ys, ld, 0, None, 0, None) == -1
    assert L.qgemm_forward_multi(x, 1, d.K, arr, 5, ys, ld, 0, None, 0, None) == -1
    bad = (qg.QgQWeight * 2)(d, d)
    bad[1].K = d.K * 2
    assert L.qgemm_forward_multi(x, 1, d.K, bad, 2, ys, ld, 0, None, 0, None) == -1
    ys0 = (ctypes.c_void_p * 2)(0x200000, None)
    assert L.qgemm_forward_multi(x, 1, d.K, arr, 2, ys0, ld, 0, None, 0, None) == -1
    short = (ctypes.c_int32 * 2)(d.N, d.N - 1)
    assert L.qgemm_forward_multi(x, 1, d.K, arr, 2, ys, short, 0, None, 0, None) == -1
    assert L.qgemm_forward_multi(x, 0, d.K, arr, 2, ys, ld, 0, None, 0, None) == 0   # M = 0: nothing to do


def test_device_status_query_without_gpu(qg):
    # a NULL output is rejected on the host; without a device the read fails
    # with a CUDA status instead of crashing
    import torch
    L = qg.lib()
    assert L.qgemm_device_status(None, 0) == -1
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    v = ctypes.c_int32(123)
    assert L.qgemm_device_status(ctypes.byref(v), 0) == -5
    assert v.value == 123


def test_moe_validation_without_gpu(qg):
    L = qg.lib()
    arr = (qg.QgQWeight * 2)(_fake_desc(qg), _fake_desc(qg, N=128))
    x, ids, y = ctypes.c_void_p(0x300000), ctypes.c_void_p(0x310000), ctypes.c_void_p(0x320000)
    assert L.qgemm_moe_grouped(x, 4, ids, 2, arr, 2, y, 0, None, 0, None) == -1   # N differs
    arr2 = (qg.QgQWeight * 1)(_fake_desc(qg))
    assert L.qgemm_moe_grouped(x, 4, ids, 2, arr2, 300, y, 0, None, 0, None) == -1  # E too large
    assert L.qgemm_moe_grouped(x, 0, ids, 2, arr2, 1, y, 0, None, 0, None) == 0     # T = 0
    b = ctypes.c_size_t()
    assert L.qgemm_moe_workspace_size(256, 2, 1, arr2, ctypes.byref(b)) == 0 and b.value > 0
    assert L.qgemm_moe_grouped(x, 4, ids, 2, arr2, 1, y, 0, None, 0, None) == -4    # no workspace


def test_moe_multi_validation_without_gpu(qg):
    # product counts outside 1..2, mismatched experts and null outputs are
    # rejected on the host; T = 0 is a no-op
    L = qg.lib()
    d = _fake_desc(qg)
    arr = (qg.QgQWeight * 4)(d, d, d, d)
    x, ids = ctypes.c_void_p(0x300000), ctypes.c_void_p(0x310000)
    ys = (ctypes.c_void_p * 2)(0x320000, 0x330000)
    assert L.qgemm_moe_grouped_multi(x, 4, ids, 2, arr, 2, 0, ys, 0, None, 0, None) == -1
    assert L.qgemm_moe_grouped_multi(x, 4, ids, 2, arr, 1, 3, ys, 0, None, 0, None) == -1
    bad = (qg.QgQWeight * 4)(d, d, d, d)
    bad[3].N = d.N * 2
    assert L.qgemm_moe_grouped_multi(x, 4, ids, 2, bad, 2, 2, ys, 0, None, 0, None) == -1
    ys0 = (ctypes.c_void_p * 2)(0x320000, None)
    assert L.qgemm_moe_grouped_multi(x, 4, ids, 2, arr, 2, 2, ys0, 0, None, 0, None) == -1
    assert L.qgemm_moe_grouped_multi(x, 0, ids, 2, arr, 2, 2, ys, 0, None, 0, None) == 0
    assert L.qgemm_moe_grouped_multi(x, 4, ids, 2, arr, 2, 2, ys, 0, None, 0, None) == -4   # no workspace
