"""Quantizer variants (symmetric at every width, linear 2-bit constants) on
the device: bytes equal to the oracle's, and the products on them (decode
and tensor-core kernels, grouped kernel) within the stated tolerance."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _parity import assert_quantized_equal, check_product, to_device

pytestmark = pytest.mark.gpu

CASES = [(b, "symmetric") for b in (2, 3, 4, 5, 6, 8)] + [(2, "linear2")]


@pytest.fixture(scope="module")
def qg():
    import bit_weight_only_group_gb300 as qg
    qg.lib()
    return qg


@pytest.mark.parametrize("bits,mode", CASES)
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("frac", [0.0, 0.003])
def test_variant_quantize_bit_exact(qg, bits, mode, group, frac):
    W = wl.gen_weight(136, 1024, seed=bits + group, outlier_frac=frac, outlier_seed=5)
    qw = qg.qpack_quantize(W.cuda(), bits, group, frac, mode=mode)
    torch.cuda.synchronize()
    assert_quantized_equal(qw, oracle.quantize(W, bits, group, frac, mode=mode))


@pytest.mark.parametrize("bits,mode", CASES)
def test_variant_extreme_groups_bit_exact(qg, bits, mode):
    W = wl.gen_extreme_weight(136, 512, 128, seed=3)
    for frac in (0.0, 0.004):
        qw = qg.qpack_quantize(W.cuda(), bits, 128, frac, mode=mode)
        torch.cuda.synchronize()
        assert_quantized_equal(qw, oracle.quantize(W, bits, 128, frac, mode=mode))


@pytest.mark.parametrize("bits,mode", CASES)
@pytest.mark.parametrize("M", [1, 7, 300])
def test_variant_products(qg, bits, mode, M):
    N, K, frac = 200, 1024, 0.002
    W = wl.gen_weight(N, K, seed=40 + bits, outlier_frac=frac, outlier_seed=41)
    q = oracle.quantize(W, bits, 128, frac, mode=mode)
    x = wl.gen_x(M, K, seed=M)
    y = qg.qgemm_forward(x.cuda(), to_device(q))
    torch.cuda.synchronize()
    check_product(y, oracle.linear(x, q), x, float(np.abs(oracle.dequant(q)).max()))


def test_variant_grouped_product(qg):
    # symmetric 4-bit experts take the grouped tensor-core kernel
    N, K, E, T, k = 136, 512, 4, 60, 2
    qs = [oracle.quantize(wl.gen_weight(N, K, seed=60 + e, outlier_frac=0.002, outlier_seed=e), 4, 128, 0.002,
                          mode="symmetric") for e in range(E)]
    x = wl.gen_x(T, K, seed=61)
    topk = wl.gen_topk(T, k, E, seed=62)
    y = qg.qgemm_moe_grouped(x.cuda(), topk.cuda(), [to_device(q) for q in qs])
    torch.cuda.synchronize()
    wmax = max(float(np.abs(oracle.dequant(q)).max()) for q in qs)
    check_product(y.reshape(T * k, N), oracle.moe(x, topk.numpy(), qs).reshape(T * k, N), x.repeat_interleave(k, 0),
                  wmax)


def test_variant_rejections(qg):
    W = wl.gen_weight(64, 128).cuda()
    with pytest.raises(qg.QgError) as e:
        qg.qpack_quantize(W, 4, 64, 0.0, mode="linear2")
    assert e.value.status == -2
