"""The benchmark's CPU baseline (fused fp32 qGEMV on all host cores) against
the fp64 oracle, at every width, both groups, with outliers: the bench's CPU
figure is only meaningful if the CPU program computes the same product."""
import numpy as np
import pytest

import cpu_baseline
import oracle
import workloads as wl
from _parity import check_product


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
@pytest.mark.parametrize("group", [64, 128])
def test_cpu_baseline_matches_oracle(bits, group):
    N, K, frac = 136, 1024, 0.003
    W = wl.gen_weight(N, K, seed=bits * 10 + group, outlier_frac=frac, outlier_seed=bits)
    q = oracle.quantize(W, bits, group, frac)
    x = wl.gen_x(1, K, seed=bits)
    y = cpu_baseline.gemv(oracle.bf16_to_f64(x).astype(np.float32), cpu_baseline.HostWeight.from_oracle(q))
    import torch
    check_product(torch.from_numpy(y[None, :]), oracle.linear(x, q), x, float(np.abs(oracle.dequant(q)).max()))


def test_cpu_baseline_threads_and_edges():
    assert cpu_baseline.cores() >= 1
    N, K = 7, 256
    q = oracle.quantize(wl.gen_weight(N, K, seed=3), 4, 128, 0.0)
    x = wl.gen_x(1, K, seed=4)
    xf = oracle.bf16_to_f64(x).astype(np.float32)
    hw = cpu_baseline.HostWeight.from_oracle(q)
    one = cpu_baseline.gemv(xf, hw, threads=1)
    many = cpu_baseline.gemv(xf, hw, threads=64)     # more threads than rows
    assert np.array_equal(one, many)
    zero = cpu_baseline.gemv(np.zeros(K, np.float32), hw)
    assert (zero == 0).all()
