"""GPU quantize-and-pack is bit-exact with the oracle: packed bytes, fp16
scales, zero-points, codebooks and the outlier CSR."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _parity import assert_quantized_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    import bit_weight_only_group_gb300 as qg
    qg.lib()
    return qg


def _run(qg, W, bits, group, frac):
    qw = qg.qpack_quantize(W.cuda(), bits, group, frac)
    torch.cuda.synchronize()
    return qw


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("N,K,frac", [(96, 512, 0.002), (33, 256, 0.0), (7, 1024, 0.01)])
def test_quantize_bit_exact_small(qg, bits, group, N, K, frac):
    W = wl.gen_weight(N, K, seed=1000 + N + bits, outlier_frac=frac, outlier_seed=2000 + group)
    qw = _run(qg, W, bits, group, frac)
    assert_quantized_equal(qw, oracle.quantize(W, bits, group, frac))


@pytest.mark.parametrize("bits", [2, 4, 5])
def test_quantize_threshold_ties(qg, bits):
    # few distinct magnitudes: the outlier count cuts through a block of ties
    rng = np.random.default_rng(bits)
    N, K = 40, 256
    mags = rng.choice([0.01, 0.02, 0.5, 1.0], size=(N, K), p=[0.6, 0.3, 0.07, 0.03])
    W = torch.from_numpy((mags * rng.choice([-1.0, 1.0], size=(N, K))).astype(np.float16))
    frac = 0.05
    qw = _run(qg, W, bits, 128, frac)
    assert_quantized_equal(qw, oracle.quantize(W, bits, 128, frac))


@pytest.mark.parametrize("bits", [2, 3, 6])
def test_quantize_degenerate_groups(qg, bits):
    N, K = 8, 256
    W = torch.zeros((N, K), dtype=torch.float16)
    W[1] = 0.75                          # one-signed rows
    W[2] = -0.125
    W[3, :128] = 5.0                     # a whole group of equal large values
    W[4, 7] = 2.0 ** -24                 # smallest subnormal
    W[5, ::2] = 65504.0                  # largest fp16
    W[5, 1::2] = -65504.0
    for frac in (0.0, 0.1):
        qw = _run(qg, W, bits, 128, frac)
        assert_quantized_equal(qw, oracle.quantize(W, bits, 128, frac))


@pytest.mark.parametrize("bits,group", [(4, 128), (2, 128), (3, 64), (5, 128), (6, 64), (2, 64)])
def test_quantize_bit_exact_4096(qg, bits, group):
    frac = 0.0 if (bits, group) == (4, 128) else 0.001
    W = wl.gen_weight(4096, 4096, outlier_frac=frac)
    qw = _run(qg, W, bits, group, frac)
    assert_quantized_equal(qw, oracle.quantize(W, bits, group, frac))


def test_quantize_bit_exact_11008x4096(qg):
    W = wl.gen_weight(11008, 4096, outlier_frac=0.001)
    qw = _run(qg, W, 2, 128, 0.001)
    assert_quantized_equal(qw, oracle.quantize(W, 2, 128, 0.001))
