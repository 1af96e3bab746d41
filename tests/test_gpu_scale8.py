"""8-bit (E4M3) group scales with the fp16 fallback list on the device: the
quantizer's bytes (codes, 8-bit scales, matrix exponent, fallback list)
equal to the oracle's, the capacity check, and every product entry point on
such weights against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _parity import assert_quantized_equal, check_product, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    import bit_weight_only_group_gb300 as qg
    qg.lib()
    return qg


def _wmax(q):
    return float(np.abs(oracle.dequant(q)).max())


@pytest.mark.parametrize("bits", [3, 4, 5, 6, 8])
@pytest.mark.parametrize("group", [32, 128])
@pytest.mark.parametrize("mode", ["asymmetric", "symmetric"])
@pytest.mark.parametrize("frac", [0.0, 0.002])
def test_scale8_quantize_bit_exact(qg, bits, group, mode, frac):
    W = wl.gen_weight(136, 1024, seed=bits + group, outlier_frac=frac, outlier_seed=3)
    qw = qg.qpack_quantize(W.cuda(), bits, group, frac, mode=mode, scale_fmt="fp8")
    torch.cuda.synchronize()
    assert_quantized_equal(qw, oracle.quantize(W, bits, group, frac, mode=mode, scale_fmt="fp8"))


@pytest.mark.parametrize("bits,group", [(3, 32), (5, 64), (4, 128)])
def test_scale8_fallback_groups_bit_exact(qg, bits, group):
    # groups spread over about twenty binades: several per row fall back
    W = wl.gen_spread_scale_weight(200, 1024, group, seed=bits)
    ref = oracle.quantize(W, bits, group, 0.001, scale_fmt="fp8")
    assert ref.fb_col.size > 50
    qg.qgemm_device_status(reset=True)
    qw = qg.qpack_quantize(W.cuda(), bits, group, 0.001, scale_fmt="fp8", fb_cap=ref.fb_col.size)
    torch.cuda.synchronize()
    assert qg.qgemm_device_status() == 0
    assert_quantized_equal(qw, ref)


def test_scale8_extreme_groups_bit_exact(qg):
    W = wl.gen_extreme_weight(136, 512, 128, seed=3)
    for frac in (0.0, 0.004):
        for mode in ("asymmetric", "symmetric"):
            ref = oracle.quantize(W, 4, 128, frac, mode=mode, scale_fmt="fp8")
            qw = qg.qpack_quantize(W.cuda(), 4, 128, frac, mode=mode, scale_fmt="fp8")
            torch.cuda.synchronize()
            assert_quantized_equal(qw, ref)


def test_scale8_capacity_overflow_is_reported(qg):
    W = wl.gen_spread_scale_weight(64, 512, 32, seed=9)
    ref = oracle.quantize(W, 4, 32, 0.0, scale_fmt="fp8")
    need = ref.fb_col.size
    assert need > 8
    qg.qgemm_device_status(reset=True)
    qw = qg.qpack_quantize(W.cuda(), 4, 32, 0.0, scale_fmt="fp8", fb_cap=need - 3)
    torch.cuda.synchronize()
    assert qg.qgemm_device_status(reset=True) == -4          # QG_ERR_WORKSPACE
    assert qg.qgemm_device_status() == 0
    # the row pointer still counts every fallback group; the listed ones are right
    assert np.array_equal(qw.fb_row_ptr.cpu().numpy(), ref.fb_row_ptr)
    assert np.array_equal(qw.fb_col.cpu().numpy(), ref.fb_col[:need - 3])


def test_scale8_noalloc_bit_exact(qg):
    W = wl.gen_spread_scale_weight(96, 512, 32, seed=4)
    ref = oracle.quantize(W, 3, 32, 0.002, scale_fmt="fp8")
    out = qg.QWeight.empty(96, 512, 3, 32, 0.002, scale_fmt="fp8", fb_cap=ref.fb_col.size + 5)
    qw = qg.qpack_quantize_noalloc(W.cuda(), 3, 32, 0.002, out=out)
    torch.cuda.synchronize()
    assert_quantized_equal(qw, ref)


@pytest.mark.parametrize("bits,group", [(3, 32), (4, 128), (5, 64), (6, 32), (8, 128)])
@pytest.mark.parametrize("M", [1, 8, 32, 300])
def test_scale8_products(qg, bits, group, M):
    N, K, frac = 200, 1024, 0.002
    W = wl.gen_spread_scale_weight(N, K, group, seed=11 * bits)
    q = oracle.quantize(W, bits, group, frac, scale_fmt="fp8")
    assert q.fb_col.size > 0
    qd = to_device(q)
    x = wl.gen_x(M, K, seed=M)
    y = qg.qgemm_forward(x.cuda(), qd)
    yt = qg.qgemm_forward_tiles(x.cuda(), qd, qg.qrepack_tiles(qd))
    torch.cuda.synchronize()
    ref = oracle.linear(x, q)
    check_product(y, ref, x, _wmax(q))
    check_product(yt, ref, x, _wmax(q))


def test_scale8_repack_equals_the_oracle_layout(qg):
    W = wl.gen_spread_scale_weight(300, 512, 32, seed=5)
    q = oracle.quantize(W, 5, 32, 0.003, scale_fmt="fp8")
    t = qg.qrepack_tiles(to_device(q))
    torch.cuda.synchronize()
    assert np.array_equal(t.cpu().numpy(), oracle.tiles(q))


def test_scale8_forward_multi_and_grouped(qg):
    K, E, T, k = 512, 4, 60, 2
    qs = [oracle.quantize(wl.gen_spread_scale_weight(136, K, 64, seed=20 + e), 4, 64, 0.002, scale_fmt="fp8")
          for e in range(E)]
    x = wl.gen_x(T, K, seed=21)
    ys = qg.qgemm_forward_multi(x[:5].cuda(), [to_device(q) for q in qs[:3]])
    topk = wl.gen_topk(T, k, E, seed=22)
    ym = qg.qgemm_moe_grouped(x.cuda(), topk.cuda(), [to_device(q) for q in qs])
    torch.cuda.synchronize()
    for q, y in zip(qs[:3], ys):
        check_product(y, oracle.linear(x[:5], q), x[:5], _wmax(q))
    wmax = max(_wmax(q) for q in qs)
    check_product(ym.reshape(T * k, -1), oracle.moe(x, topk.numpy(), qs).reshape(T * k, -1),
                  x.repeat_interleave(k, 0), wmax)


def test_scale8_diagnostics_and_w8a8(qg):
    W = wl.gen_spread_scale_weight(200, 1024, 32, seed=31)
    q = oracle.quantize(W, 8, 32, 0.002, scale_fmt="fp8")
    qd = to_device(q)
    got = qg.qdiag_layer(W.cuda(), qd, threshold=3.0)
    ref = oracle.diagnostics(W, q, threshold=3.0)
    assert got["max_abs_err"] == pytest.approx(ref["max_abs_err"], rel=1e-6, abs=1e-12)
    assert got["rmse"] == pytest.approx(ref["rmse"], rel=1e-5, abs=1e-12)
    assert got["cosine"] == pytest.approx(ref["cosine"], abs=2e-6)
    assert got["groups_over"] == ref["groups_over"]
    x = wl.gen_x(4, 1024, seed=32)
    y = qg.qgemm_forward_w8a8(x.cuda(), qd)
    torch.cuda.synchronize()
    check_product(y, oracle.linear_w8a8(x, q), x, _wmax(q))
