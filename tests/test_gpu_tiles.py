"""The one-time device repack into the tile-ordered layout (bytes equal to
the oracle's layout) and the tensor-core product that streams it: against
the fp64 oracle, bit for bit against the planar tensor-core path (the same
arithmetic on the same operands) and across repeated calls."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _parity import check_product, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    import bit_weight_only_group_gb300 as qg
    qg.lib()
    return qg


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
@pytest.mark.parametrize("group", [32, 64, 128])
def test_repack_bytes_equal_the_oracle_layout(qg, bits, group):
    N, K = 300, 512
    q = oracle.quantize(wl.gen_weight(N, K, seed=bits + group, outlier_frac=0.003, outlier_seed=1), bits, group, 0.003)
    t = qg.qrepack_tiles(to_device(q))
    torch.cuda.synchronize()
    assert np.array_equal(t.cpu().numpy(), oracle.tiles(q))


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("M", [1, 100, 300])
def test_tiles_product(qg, bits, group, M):
    N, K, frac = 300, 1024, 0.003
    q = oracle.quantize(wl.gen_weight(N, K, seed=7 * bits + group, outlier_frac=frac, outlier_seed=2), bits, group,
                        frac)
    qd = to_device(q)
    t = qg.qrepack_tiles(qd)
    x = wl.gen_x(M, K, seed=M)
    y = qg.qgemm_forward_tiles(x.cuda(), qd, t)
    torch.cuda.synchronize()
    check_product(y, oracle.linear(x, q), x, float(np.abs(oracle.dequant(q)).max()))
    for _ in range(3):
        assert torch.equal(qg.qgemm_forward_tiles(x.cuda(), qd, t), y)
    if M > 32:   # the planar tensor-core path computes the same operands in the same order
        assert torch.equal(qg.qgemm_forward(x.cuda(), qd), y)


@pytest.mark.parametrize("bits", [3, 4, 8])
def test_tiles_product_extreme_groups(qg, bits):
    W = wl.gen_extreme_weight(136, 512, 128, seed=12)
    q = oracle.quantize(W, bits, 128, 0.004)
    qd = to_device(q)
    x = wl.gen_x(300, 512, seed=13)
    y = qg.qgemm_forward_tiles(x.cuda(), qd, qg.qrepack_tiles(qd))
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
    check_product(y, oracle.linear(x, q), x, float(np.abs(oracle.dequant(q)).max()))


def test_tiles_full_size_sampled(qg):
    # the 70B prefill shape (8192 x 8192, M = 2048, INT4 g128), device-quantized
    # without outliers; sampled tokens and rows against the oracle
    M, N, K = 2048, 8192, 8192
    W = wl.gen_weight(N, K, seed=21)
    qw = qg.qpack_quantize(W.cuda(), 4, 128, 0.0)
    x = wl.gen_x(M, K, seed=22)
    t = qg.qrepack_tiles(qw)
    y = qg.qgemm_forward_tiles(x.cuda(), qw, t)
    torch.cuda.synchronize()
    assert torch.equal(y, qg.qgemm_forward_tiles(x.cuda(), qw, t))
    assert torch.equal(y, qg.qgemm_forward(x.cuda(), qw))
    toks = torch.arange(0, M, 97)
    for n0 in (0, N - 64):
        q = oracle.quantize(W[n0:n0 + 64], 4, 128, 0.0)
        check_product(y[toks.cuda(), n0:n0 + 64], oracle.linear(x[toks], q), x[toks],
                      float(np.abs(oracle.dequant(q)).max()))
