"""W8A8 decode product (int8 weights, int8 activations quantized per token
inside the call) against the fp64 oracle's product of the same quantized
activations with the same weights."""
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


def _xhat(x):
    q, s = oracle.quantize_act_int8(x)
    import torch as t
    return t.from_numpy((q.astype(np.float64) * s[:, None]).astype(np.float32)).to(t.bfloat16)


@pytest.mark.parametrize("mode", ["asymmetric", "symmetric"])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("M", [1, 2, 3, 8, 16])
def test_w8a8_against_oracle(qg, mode, group, M):
    N, K, frac = 200, 1024, 0.003
    W = wl.gen_weight(N, K, seed=M + group, outlier_frac=frac, outlier_seed=3)
    q = oracle.quantize(W, 8, group, frac, mode=mode)
    x = wl.gen_x(M, K, seed=M)
    y = qg.qgemm_forward_w8a8(x.cuda(), to_device(q))
    torch.cuda.synchronize()
    # the bound of the stated tolerance, with the quantized activations as x
    check_product(y, oracle.linear_w8a8(x, q), x, float(np.abs(oracle.dequant(q)).max()))


def test_w8a8_full_size_rows(qg):
    # the 70B gate shape 28672 x 8192 at M = 1, device-quantized (no outliers,
    # so the oracle quantizes just the sampled rows)
    N, K = 28672, 8192
    W = wl.gen_weight(N, K, seed=8)
    qw = qg.qpack_quantize(W.cuda(), 8, 128, 0.0)
    x = wl.gen_x(1, K, seed=9)
    y = qg.qgemm_forward_w8a8(x.cuda(), qw, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    for n0 in (0, N // 2, N - 64):
        q = oracle.quantize(W[n0:n0 + 64], 8, 128, 0.0)
        ref = oracle.linear_w8a8(x, q)
        yb = y[:, n0:n0 + 64].float()
        # bf16 output: one more rounding (2^-9 relative)
        assert np.allclose(yb.cpu().numpy(), ref, rtol=2 ** -8, atol=1e-3 * np.abs(ref).max())


def test_w8a8_rejections(qg):
    W = wl.gen_weight(64, 128).cuda()
    q4 = qg.qpack_quantize(W, 4, 64, 0.0)
    with pytest.raises(qg.QgError) as e:
        qg.qgemm_forward_w8a8(wl.gen_x(1, 128).cuda(), q4)
    assert e.value.status == -2
    q8 = qg.qpack_quantize(W, 8, 64, 0.0)
    with pytest.raises(qg.QgError) as e:
        qg.qgemm_forward_w8a8(wl.gen_x(17, 128).cuda(), q8)
    assert e.value.status == -2
