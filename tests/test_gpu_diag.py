"""Device layer diagnostics (max |error|, RMSE, cosine, per-group dynamic-
range ratio) against the fp64 oracle, every width and group, with outliers,
on Gaussian layers and on layers with extreme and degenerate groups."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _parity import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    import bit_weight_only_group_gb300 as qg
    qg.lib()
    return qg


def _check(got, ref):
    # the device sums in fp32 within a group and fp64 across groups; the
    # maximum and the ratios are exact up to one fp32 rounding
    assert got["max_abs_err"] == pytest.approx(ref["max_abs_err"], rel=1e-6, abs=1e-12)
    assert got["rmse"] == pytest.approx(ref["rmse"], rel=1e-5, abs=1e-12)
    assert got["cosine"] == pytest.approx(ref["cosine"], abs=2e-6)
    if np.isinf(ref["max_range_ratio"]):
        assert np.isinf(got["max_range_ratio"])
    else:
        assert got["max_range_ratio"] == pytest.approx(ref["max_range_ratio"], rel=1e-6)
    assert got["groups_over"] == ref["groups_over"]
    r = got["ratio"].double().cpu().numpy()
    fin = np.isfinite(ref["ratio"])
    assert (np.isinf(r) == ~fin).all()
    assert np.allclose(r[fin], ref["ratio"][fin], rtol=1e-6, atol=0)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
@pytest.mark.parametrize("group", [32, 64, 128])
def test_diagnostics_against_oracle(qg, bits, group):
    N, K, frac = 200, 1024, 0.002
    W = wl.gen_weight(N, K, seed=bits + group, outlier_frac=frac, outlier_seed=9)
    q = oracle.quantize(W, bits, group, frac)
    got = qg.qdiag_layer(W.cuda(), to_device(q), threshold=3.0, ratio=True)
    _check(got, oracle.diagnostics(W, q, threshold=3.0))


@pytest.mark.parametrize("bits", [2, 4, 5])
def test_diagnostics_extreme_groups(qg, bits):
    W = wl.gen_extreme_weight(136, 512, 128, seed=11)
    W[9, 200] = 0.0
    q = oracle.quantize(W, bits, 128, 0.004)
    got = qg.qdiag_layer(W.cuda(), to_device(q), threshold=50.0, ratio=True)
    _check(got, oracle.diagnostics(W, q, threshold=50.0))


def test_diagnostics_full_size_gate_matrix(qg):
    # a 28672 x 8192 INT4 layer (0.1 % outliers) quantized on the device: the
    # device figures against the oracle's on the same quantized bytes
    N, K = 28672, 8192
    W = wl.gen_weight(N, K, seed=5, outlier_frac=0.001, outlier_seed=6, distinct_positions=False)
    qw = qg.qpack_quantize(W.cuda(), 4, 128, 0.001)
    got = qg.qdiag_layer(W.cuda(), qw, threshold=10.0, ratio=True)
    h = lambda t: None if t is None else t.cpu().numpy()
    q = oracle.QWeight(N, K, 4, 128, h(qw.packed), h(qw.scale).view(np.uint16), h(qw.zp), None, h(qw.row_ptr),
                       h(qw.col), h(qw.val).view(np.uint16))
    _check(got, oracle.diagnostics(W, q, threshold=10.0))
