"""The fused product on the GPU against the fp64 oracle, for every width,
group size and M path, with outliers, ragged N, strided x / y."""
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


_cache = {}


def _weights(N, K, bits, group, frac, seed):
    key = (N, K, bits, group, frac, seed)
    if key not in _cache:
        W = wl.gen_weight(N, K, seed=seed, outlier_frac=frac, outlier_seed=seed + 1)
        q = oracle.quantize(W, bits, group, frac)
        _cache[key] = (q, np.abs(oracle.dequant(q)).max())
    return _cache[key]


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 16, 27, 64])
def test_product_small(qg, bits, group, M):
    N, K, frac = 200, 1024, 0.002            # N not a multiple of the 64-row tile
    q, wmax = _weights(N, K, bits, group, frac, seed=17 * bits + group)
    x = wl.gen_x(M, K, seed=M)
    y = qg.qgemm_forward(x.cuda(), to_device(q))
    torch.cuda.synchronize()
    check_product(y, oracle.linear(x, q), x, wmax)


@pytest.mark.parametrize("bits", [2, 4, 6])
@pytest.mark.parametrize("M", [33, 64, 65, 130])
def test_product_above_decode_range(qg, bits, M):
    N, K = 136, 512
    q, wmax = _weights(N, K, bits, 128, 0.002, seed=5)
    x = wl.gen_x(M, K, seed=M)
    y = qg.qgemm_forward(x.cuda(), to_device(q))
    torch.cuda.synchronize()
    check_product(y, oracle.linear(x, q), x, wmax)


def test_product_strided_and_bf16_output(qg):
    N, K, M = 192, 768, 9
    q, wmax = _weights(N, K, 5, 64, 0.003, seed=9)
    xbig = wl.gen_x(M, K + 40, seed=3).cuda()
    x = xbig[:, 16:16 + K]                     # row stride K + 40, unaligned start
    ybig = torch.full((M, N + 8), 7.0, device="cuda")
    y = ybig[:, :N]
    qd = to_device(q)
    qg.qgemm_forward(x, qd, out=y)
    yb = qg.qgemm_forward(x, qd, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    check_product(y, oracle.linear(x.cpu(), q), x.cpu(), wmax)
    assert (ybig[:, N:] == 7.0).all()          # nothing written past N
    assert torch.equal(yb, y.to(torch.bfloat16))


def test_zero_weights_and_zero_x_give_exact_zero(qg):
    N, K = 64, 256
    for bits in (2, 4, 5):
        q = oracle.quantize(np.zeros((N, K), np.float16), bits, 128, 0.0)
        y = qg.qgemm_forward(wl.gen_x(3, K).cuda(), to_device(q))
        assert (y == 0).all()
    q, _ = _weights(N, K, 3, 64, 0.0, seed=4)
    y = qg.qgemm_forward(torch.zeros((2, K), dtype=torch.bfloat16, device="cuda"), to_device(q))
    assert (y == 0).all()


def test_one_hot_x_reads_back_dequantized_columns(qg):
    N, K = 128, 512
    q, _ = _weights(N, K, 6, 128, 0.004, seed=21)
    D = oracle.dequant(q)
    ks = [0, 1, 63, 64, 127, 300, 511]
    x = torch.zeros((len(ks), K), dtype=torch.bfloat16)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y = qg.qgemm_forward(x.cuda(), to_device(q)).double().cpu().numpy()
    ref = D[:, ks].T
    assert np.allclose(y, ref, rtol=2 ** -10, atol=0), np.abs(y - ref).max()


@pytest.mark.parametrize("bits,group,M", [(4, 128, 1), (2, 128, 8), (3, 64, 32), (5, 128, 1), (6, 64, 8),
                                          (2, 64, 32)])
def test_product_4096(qg, bits, group, M):
    frac = 0.0 if bits == 4 else 0.001
    q, wmax = _weights(4096, 4096, bits, group, frac, seed=1234)
    x = wl.gen_x(M, 4096)
    y = qg.qgemm_forward(x.cuda(), to_device(q))
    torch.cuda.synchronize()
    check_product(y, oracle.linear(x, q), x, wmax)


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("M,N,K", [(300, 600, 1024), (129, 256, 384), (1000, 700, 512)])
def test_tensor_core_path_against_oracle(qg, group, M, N, K):
    # M above the decode range runs the tcgen05 kernel (128 x 256 tiles, K in
    # blocks of 64); ragged M and N exercise the zero-filled TMA edges
    q, wmax = _weights(N, K, 4, group, 0.003, seed=M + N)
    x = wl.gen_x(M, K, seed=M)
    qd = to_device(q)
    assert qg.qgemm_workspace_size(M, qd) > 0
    y = qg.qgemm_forward(x.cuda(), qd)
    yb = qg.qgemm_forward(x.cuda(), qd, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    check_product(y, oracle.linear(x, q), x, wmax)
    assert torch.equal(yb, y.to(torch.bfloat16))


@pytest.mark.parametrize("bits", [2, 3, 5, 6, 8])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("M,N,K", [(300, 600, 1024), (129, 200, 384)])
def test_tensor_core_path_every_width(qg, bits, group, M, N, K):
    # 2/3/5/6-bit weights above the decode range: the tcgen05 kernel with the
    # codes read by the dequantization threads and unpacked by the width's
    # pair plan (x permuted to match), FP16 outliers patched into the operand
    q, wmax = _weights(N, K, bits, group, 0.003, seed=M + N + bits)
    x = wl.gen_x(M, K, seed=M + bits)
    qd = to_device(q)
    y = qg.qgemm_forward(x.cuda(), qd)
    torch.cuda.synchronize()
    check_product(y, oracle.linear(x, q), x, wmax)
    for _ in range(3):   # fixed accumulation order: repeated calls agree bit for bit
        assert torch.equal(qg.qgemm_forward(x.cuda(), qd), y)


@pytest.mark.parametrize("bits", [2, 5])
def test_tensor_core_path_every_width_full_size_sampled(qg, bits):
    # 11008 x 4096 at M = 2048 (the mixed-width sweep's larger shape at the
    # prefill length); no outliers, so the oracle quantizes only the sampled
    # rows of the seeded W while the device quantizes all of it
    M, N, K = 2048, 11008, 4096
    W = wl.gen_weight(N, K, seed=77 + bits)
    qw = qg.qpack_quantize(W.cuda(), bits, 128, 0.0)
    x = wl.gen_x(M, K, seed=78)
    y = qg.qgemm_forward(x.cuda(), qw)
    torch.cuda.synchronize()
    toks = torch.arange(0, M, 89)
    for n0 in (0, 5504 - 32, N - 64):
        q = oracle.quantize(W[n0:n0 + 64], bits, 128, 0.0)
        wmax = float(np.abs(oracle.dequant(q)).max())
        check_product(y[toks.cuda(), n0:n0 + 64], oracle.linear(x[toks], q), x[toks], wmax)


def test_device_status_stays_clear(qg):
    # the tensor-core kernel's bounded waits never give up on valid inputs:
    # after products of both groups the status word is still QG_OK
    qg.qgemm_device_status(reset=True)
    for group in (64, 128):
        q, wmax = _weights(512, 1024, 4, group, 0.001, seed=group)
        x = wl.gen_x(300, 1024)
        y = qg.qgemm_forward(x.cuda(), to_device(q))
        torch.cuda.synchronize()
        check_product(y, oracle.linear(x, q), x, wmax)
    assert qg.qgemm_device_status() == 0


def test_bounded_wait_gives_up_and_reports_timeout(qg):
    # a kernel waits on an mbarrier that nothing arrives on, with a poll
    # limit of 2: the wait runs out, the status word reads QG_ERR_TIMEOUT,
    # reading it with reset clears it, and the context stays usable
    assert qg.qgemm_device_status(reset=True) in (0, -6)
    qg.qgemm_selftest_bounded_wait(2)
    torch.cuda.synchronize()
    assert qg.qgemm_device_status(reset=True) == -6
    assert qg.qgemm_device_status() == 0
    q, wmax = _weights(256, 512, 4, 128, 0.0, seed=3)
    x = wl.gen_x(300, 512)
    y = qg.qgemm_forward(x.cuda(), to_device(q))
    torch.cuda.synchronize()
    check_product(y, oracle.linear(x, q), x, wmax)
    assert qg.qgemm_device_status() == 0


@pytest.mark.parametrize("group", [32, 64, 128])
def test_tensor_core_path_repeatable(qg, group):
    # the accumulation order of the tensor-core kernel is fixed, so repeated
    # calls must agree bit for bit; a ring slot reused too early shows up here
    # as a few corrupted weight rows in some of the runs
    M, N, K = 300, 600, 1024
    q, _ = _weights(N, K, 4, group, 0.003, seed=M + N)
    x = wl.gen_x(M, K, seed=M).cuda()
    qd = to_device(q)
    y0 = qg.qgemm_forward(x, qd)
    for _ in range(30):
        assert torch.equal(qg.qgemm_forward(x, qd), y0)


def test_tensor_core_path_full_size_sampled(qg):
    # the prefill shape of the 70B-shaped stack (M = 2048, 8192 x 8192, INT4
    # group 128, 0.1 % outliers); the oracle checks sampled tokens and rows
    M, N, K = 2048, 8192, 8192
    W = wl.gen_weight(N, K, outlier_frac=0.001)
    q = oracle.quantize(W, 4, 128, 0.001)
    x = wl.gen_x(M, K)
    y = qg.qgemm_forward(x.cuda(), to_device(q))
    torch.cuda.synchronize()
    toks = torch.arange(0, M, 97)
    for n0 in (0, 4096 - 32, N - 64):
        n1 = n0 + 64
        wmax = float(np.abs(oracle.dequant(q, n0, n1)).max())
        check_product(y[toks.cuda(), n0:n1], oracle.linear(x[toks], q, n0, n1), x[toks], wmax)


@pytest.mark.parametrize("bits,group,M", [(4, 128, 1), (4, 128, 8), (3, 64, 16), (4, 128, 130), (5, 32, 4), (2, 32, 130),
                                          (4, 128, 64), (6, 64, 100), (3, 64, 300)])
def test_forward_multi_against_oracle(qg, bits, group, M):
    # a fused projection: three weights sharing x (different N, one ragged
    # tile) in one call; each output is the single product of its weight
    K = 1024
    shapes = [(512, 11), (128, 12), (200, 13)]
    qs = [_weights(N, K, bits, group, 0.002, seed=sd) for N, sd in shapes]
    x = wl.gen_x(M, K, seed=M + 5)
    qds = [to_device(q) for q, _ in qs]
    ys = qg.qgemm_forward_multi(x.cuda(), qds)
    torch.cuda.synchronize()
    for (q, wmax), y in zip(qs, ys):
        check_product(y, oracle.linear(x, q), x, wmax)
    if M > 16:
        # on the tensor cores the later products read the first one's
        # conversion of x and run the single call's kernels: equal bit for bit
        for qd, y in zip(qds, ys):
            assert torch.equal(y, qg.qgemm_forward(x.cuda(), qd))


def test_decode_full_size_sampled(qg):
    # the decode launches of the 70B-shaped stack at full size, M = 1, as the
    # bench step issues them: fused q/k/v, o alone, fused gate/up, down alone.
    # No outliers (a row's quantization then depends on that row only), so
    # the oracle quantizes just the sampled rows of each seeded W while the
    # device quantizes all of it.
    hid, ffn, kv = 8192, 28672, 1024
    shapes = {"q": (hid, hid), "k": (kv, hid), "v": (kv, hid), "o": (hid, hid),
              "gate": (ffn, hid), "up": (ffn, hid), "down": (hid, ffn)}
    Ws = {p: wl.gen_weight(N, K, seed=2000 + i) for i, (p, (N, K)) in enumerate(shapes.items())}
    qws = {p: qg.qpack_quantize(W.cuda(), 4, 128, 0.0) for p, W in Ws.items()}
    x_hid, x_ffn = wl.gen_x(1, hid, seed=41), wl.gen_x(1, ffn, seed=42)
    ys = {}
    ys.update(zip(("q", "k", "v"), qg.qgemm_forward_multi(x_hid.cuda(), [qws["q"], qws["k"], qws["v"]])))
    ys["o"] = qg.qgemm_forward(x_hid.cuda(), qws["o"])
    ys.update(zip(("gate", "up"), qg.qgemm_forward_multi(x_hid.cuda(), [qws["gate"], qws["up"]])))
    ys["down"] = qg.qgemm_forward(x_ffn.cuda(), qws["down"])
    torch.cuda.synchronize()
    for p, (N, K) in shapes.items():
        x = x_ffn if K == ffn else x_hid
        for n0 in sorted({0, (N // 2) // 64 * 64 - 32, N - 64}):
            q = oracle.quantize(Ws[p][n0:n0 + 64], 4, 128, 0.0)
            wmax = float(np.abs(oracle.dequant(q)).max())
            check_product(ys[p][:, n0:n0 + 64], oracle.linear(x, q), x, wmax)


@pytest.mark.parametrize("M", [1, 16, 64])
def test_decode_long_k_with_outliers(qg, M):
    # the down projection's K = 28672 with 0.1 % outliers, quantized whole by
    # the oracle: about 29 outliers per row, so the decode kernel's outlier
    # cursor refills many times across the cluster's ranks
    N, K, frac = 256, 28672, 0.001
    q, wmax = _weights(N, K, 4, 128, frac, seed=901)
    per_row = np.diff(q.row_ptr)
    assert per_row.mean() > 20 and per_row.max() > 40
    x = wl.gen_x(M, K, seed=902)
    y = qg.qgemm_forward(x.cuda(), to_device(q))
    torch.cuda.synchronize()
    check_product(y, oracle.linear(x, q), x, wmax)


def _forward_raw(qg, x, qd, ws):
    """qgemm_forward through the C ABI with an explicit workspace (None: none)."""
    import ctypes
    M, K = x.shape
    y = torch.empty((M, qd.N), dtype=torch.float32, device="cuda")
    d = qd.desc()
    st = qg.lib().qgemm_forward(x.data_ptr(), M, K, ctypes.byref(d), y.data_ptr(), qd.N, 0,
                                None if ws is None else ws.data_ptr(), 0 if ws is None else ws.numel(), None)
    assert st == 0, qg.last_error()
    return y


@pytest.mark.parametrize("bits,group", [(4, 128), (2, 128), (3, 64), (5, 32), (8, 128), (6, 32)])
@pytest.mark.parametrize("M", [8, 11, 13, 16])
def test_decode_converted_x_matches_per_cta_staging(qg, bits, group, M):
    # from M = 8 the call converts x once into fragment order in the workspace
    # and the CTAs bulk-copy it; without a workspace every CTA converts its own
    # x blocks: the operands, and so the results, are the same bit for bit
    N, K = 200, 2048
    q, wmax = _weights(N, K, bits, group, 0.002, seed=3 * bits + group)
    qd = to_device(q)
    x = wl.gen_x(M, K, seed=M + 100).cuda()
    need = qg.qgemm_workspace_size(M, qd)
    assert need >= 2 * K * M
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    y_conv = _forward_raw(qg, x, qd, ws)
    y_cta = _forward_raw(qg, x, qd, None)
    torch.cuda.synchronize()
    assert torch.equal(y_conv, y_cta)
    check_product(y_conv, oracle.linear(x.cpu(), q), x.cpu(), wmax)
    assert qg.qgemm_device_status() == 0


@pytest.mark.parametrize("bits,group,M,ytype", [(4, 128, 64, torch.float32), (5, 32, 40, torch.bfloat16),
                                                (2, 128, 128, torch.float32), (3, 64, 33, torch.float32),
                                                (4, 64, 17, torch.float32), (6, 128, 200, torch.float32),
                                                (8, 32, 256, torch.bfloat16)])
def test_tensor_core_split_k_against_oracle_and_repeatable(qg, bits, group, M, ytype):
    # up to 256 tokens the tensor-core kernel splits K over several CTAs per
    # tile; a second kernel sums the partial tiles in a fixed order, so the
    # result is repeatable bit for bit, and matches the oracle
    N, K = 600, 4096
    q, wmax = _weights(N, K, bits, group, 0.003, seed=M + bits)
    qd = to_device(q)
    x = wl.gen_x(M, K, seed=M).cuda()
    y0 = qg.qgemm_forward(x, qd, out_dtype=ytype)
    for _ in range(10):
        assert torch.equal(qg.qgemm_forward(x, qd, out_dtype=ytype), y0)
    torch.cuda.synchronize()
    if ytype == torch.float32:
        check_product(y0, oracle.linear(x.cpu(), q), x.cpu(), wmax)
    else:
        y32 = qg.qgemm_forward(x, qd)
        assert torch.equal(y0, y32.to(torch.bfloat16))
    assert qg.qgemm_device_status() == 0


def test_decode_without_dependent_launch_gives_the_same_result(qg):
    # with programmatic dependent launch off, the kernels of a product wait
    # for the previous kernel on the stream before they start; the products
    # are the same bit for bit (a device-side copy of the weights may precede
    # them).  M = 64 is the split-K tensor-core chain, M = 300 the unsplit one.
    N, K = 512, 2048
    q, wmax = _weights(N, K, 4, 128, 0.002, seed=77)
    qd = to_device(q)
    for M in (1, 16, 64, 300):
        x = wl.gen_x(M, K, seed=M + 7).cuda()
        y_on = qg.qgemm_forward(x, qd)
        try:
            qg.qgemm_set_dependent_launch(False)
            packed = qd.packed.clone()
            qd.packed.zero_()
            qd.packed.copy_(packed)          # a kernel writing the weights just before the product
            y_off = qg.qgemm_forward(x, qd)
        finally:
            qg.qgemm_set_dependent_launch(True)
        torch.cuda.synchronize()
        assert torch.equal(y_on, y_off)
        check_product(y_off, oracle.linear(x.cpu(), q), x.cpu(), wmax)
