"""The product on weights whose groups reach the edges of fp16's range
(ramps over [0, 65504] and [-65504, 65504], a range whose top grid point lies
past 65504, single 65504 entries), on degenerate groups (all zero, constant,
one-signed), and on large x, against the fp64 oracle -- through the decode
kernel (M <= 64), the tensor-core kernel (M > 64) and the grouped kernels.

The outliers of the "70B on one GPU" page (section 2) are kept exactly in
FP16; the dequantized weight (q - zp) * scale of such a group can lie above
65504 (up to about 67700 at 4 bits), which no fp16 value holds.  The
tensor-core kernels therefore build these rows at scale * 2^-e and multiply
their outputs by 2^e; an operand that overflowed to infinity, or saturated
at 65504, fails these checks."""
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


_cache = {}


def _extreme(N, K, bits, group, frac):
    key = (N, K, bits, group, frac)
    if key not in _cache:
        W = wl.gen_extreme_weight(N, K, group, seed=300 + bits)
        q = oracle.quantize(W, bits, group, frac)
        _cache[key] = (W, q, float(np.abs(oracle.dequant(q)).max()))
    return _cache[key]


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6])
@pytest.mark.parametrize("group", [64, 128])
@pytest.mark.parametrize("frac", [0.0, 0.004])
def test_extreme_groups_quantize_bit_exact(qg, bits, group, frac):
    W, q, _ = _extreme(136, 512, bits, group, frac)
    qw = qg.qpack_quantize(W.cuda(), bits, group, frac)
    torch.cuda.synchronize()
    assert_quantized_equal(qw, q)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6])
@pytest.mark.parametrize("group", [64, 128])
@pytest.mark.parametrize("frac", [0.0, 0.004])
@pytest.mark.parametrize("M", [1, 8, 300])
def test_extreme_groups_product(qg, bits, group, frac, M):
    W, q, wmax = _extreme(136, 512, bits, group, frac)
    x = wl.gen_x(M, 512, seed=M + bits)
    y = qg.qgemm_forward(x.cuda(), to_device(q))
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
    check_product(y, oracle.linear(x, q), x, wmax)


@pytest.mark.parametrize("bits", [3, 4, 5, 6])
@pytest.mark.parametrize("M", [1, 300])
def test_extreme_one_hot_reads_back_the_dequantized_value(qg, bits, M):
    # x = e_k at the column of each extreme value reads w_hat[n, k] back (one
    # fp16 rounding of (q - zp) * scale on the tensor-core path): an operand
    # held at 65504 instead of a grid point near 67700 misses by about 2200
    group = 128
    W, q, _ = _extreme(136, 512, bits, group, 0.0)
    xhat = oracle.dequant(q)
    qd = to_device(q)
    for c in [0, 1, group // 3, group - 1]:
        x = torch.zeros((M, 512), dtype=torch.bfloat16)
        x[:, c] = 1.0
        got = qg.qgemm_forward(x.cuda(), qd).double().cpu().numpy()[M - 1]
        ref = xhat[:, c]
        # one fp16 rounding of the operand at most (2^-11 relative), exact on the decode path
        assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -11 + 1e-6), (c, np.abs(got - ref).max())


@pytest.mark.parametrize("M", [1, 300])
def test_large_x_within_fp16_range(qg, M):
    # x is converted bf16 -> fp16 on every path: values up to 6e4 stay exact
    N, K = 136, 512
    W = wl.gen_weight(N, K, seed=5)
    q = oracle.quantize(W, 4, 128, 0.0)
    x = wl.gen_x(M, K, seed=6).float()
    x[:, ::7] *= 2.0e4
    x = x.clamp(-6.0e4, 6.0e4).to(torch.bfloat16)
    y = qg.qgemm_forward(x.cuda(), to_device(q))
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
    check_product(y, oracle.linear(x, q), x, float(np.abs(oracle.dequant(q)).max()))


@pytest.mark.parametrize("bits", [4, 3])
def test_extreme_groups_grouped_product(qg, bits):
    # 4 bits: the grouped tensor-core kernel; 3 bits: the grouped decode kernel
    N, K, E, T, k = 136, 512, 4, 90, 2
    qs = []
    for e in range(E):
        W = wl.gen_extreme_weight(N, K, 128, seed=400 + e) if e % 2 == 0 else wl.gen_weight(N, K, seed=400 + e)
        qs.append(oracle.quantize(W, bits, 128, 0.002))
    wmax = max(float(np.abs(oracle.dequant(q)).max()) for q in qs)
    x = wl.gen_x(T, K, seed=7)
    topk = wl.gen_topk(T, k, E, seed=8)
    y = qg.qgemm_moe_grouped(x.cuda(), topk.cuda(), [to_device(q) for q in qs])
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
    ref = oracle.moe(x, topk.numpy(), qs)
    check_product(y.reshape(T * k, N), ref.reshape(T * k, N), x.repeat_interleave(k, 0), wmax)
