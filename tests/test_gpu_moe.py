"""Grouped product over top-k routed experts against the oracle."""
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


def _experts(E, N, K, bits, group, frac, seed):
    qs = [oracle.quantize(wl.gen_weight(N, K, seed=seed + e, outlier_frac=frac, outlier_seed=seed + 100 + e),
                          bits, group, frac) for e in range(E)]
    wmax = max(np.abs(oracle.dequant(q)).max() for q in qs)
    return qs, wmax


@pytest.mark.parametrize("bits,group", [(4, 128), (2, 64), (5, 128), (8, 64), (4, 32), (3, 32)])
@pytest.mark.parametrize("T,k,E", [(37, 2, 4), (128, 2, 8), (3, 3, 5)])
def test_moe_small(qg, bits, group, T, k, E):
    N, K = 136, 512
    qs, wmax = _experts(E, N, K, bits, group, 0.002, seed=40)
    x = wl.gen_x(T, K, seed=T)
    topk = wl.gen_topk(T, k, E, seed=T + 1)
    y = qg.qgemm_moe_grouped(x.cuda(), topk.cuda(), [to_device(q) for q in qs])
    torch.cuda.synchronize()
    ref = oracle.moe(x, topk.numpy(), qs)
    check_product(y.reshape(T * k, N), ref.reshape(T * k, N), x.repeat_interleave(k, 0), wmax)


def test_moe_skips_invalid_ids_and_handles_empty_experts(qg):
    N, K, E, T, k = 64, 256, 6, 20, 2
    qs, wmax = _experts(E, N, K, 4, 128, 0.0, seed=70)
    x = wl.gen_x(T, K, seed=1)
    topk = torch.full((T, k), 1, dtype=torch.int32)
    topk[:, 1] = 3
    topk[5, 0] = -1                            # invalid ids are skipped
    topk[6, 1] = E
    y = torch.full((T, k, N), 9.0, device="cuda")
    qg.qgemm_moe_grouped(x.cuda(), topk.cuda(), [to_device(q) for q in qs], out=y)
    torch.cuda.synchronize()
    yc = y.double().cpu().numpy()
    assert (yc[5, 0] == 9.0).all() and (yc[6, 1] == 9.0).all()
    valid = np.ones((T, k), bool)
    valid[5, 0] = valid[6, 1] = False
    tk = topk.numpy().copy()
    tk[~valid] = 0
    ref = oracle.moe(x, tk, qs)
    check_product(torch.from_numpy(yc[valid]), ref[valid], x.repeat_interleave(k, 0)[valid.ravel()], wmax)


def test_moe_layer_4096_experts(qg):
    # the MoE workload: hidden 4096, 16 experts, 3072x4096 gate projection,
    # 256 tokens, top-2 from a Zipf(1.1) popularity; a sample of tokens is
    # checked against the oracle
    cfg = wl.MoE()
    qs, wmax = _experts(cfg.n_experts, cfg.ffn, cfg.hidden, 4, 128, 0.0, seed=500)
    x = wl.gen_x(cfg.tokens, cfg.hidden)
    topk = wl.gen_topk(cfg.tokens, cfg.top_k, cfg.n_experts)
    y = qg.qgemm_moe_grouped(x.cuda(), topk.cuda(), [to_device(q) for q in qs])
    torch.cuda.synchronize()
    sample = np.arange(0, cfg.tokens, 16)
    ref = oracle.moe(x[sample], topk.numpy()[sample], qs)
    got = y[torch.from_numpy(sample).cuda()]
    k = cfg.top_k
    check_product(got.reshape(-1, cfg.ffn), ref.reshape(-1, cfg.ffn), x[sample].repeat_interleave(k, 0), wmax)


@pytest.mark.parametrize("group,T,k,E,hot", [(64, 300, 2, 3, True), (128, 300, 2, 3, True), (128, 40, 2, 40, False)])
def test_moe_tensor_core_chunks_and_fallback(qg, group, T, k, E, hot):
    # 4-bit experts run on the tensor cores in chunks of up to 64 routed
    # pairs per expert: with `hot` routing, expert 0 receives every token's
    # first slot (300 pairs, five chunks); more than 32 experts take the
    # decode kernel instead
    N, K = 200, 640
    qs, wmax = _experts(E, N, K, 4, group, 0.002, seed=90)
    x = wl.gen_x(T, K, seed=T + 3)
    topk = wl.gen_topk(T, k, E, seed=T + 4)
    if hot:
        g = torch.Generator().manual_seed(T + 5)
        topk[:, 0] = 0
        topk[:, 1] = torch.randint(1, E, (T,), generator=g).to(topk.dtype)
    y = qg.qgemm_moe_grouped(x.cuda(), topk.cuda(), [to_device(q) for q in qs])
    torch.cuda.synchronize()
    ref = oracle.moe(x, topk.numpy(), qs)
    check_product(y.reshape(T * k, N), ref.reshape(T * k, N), x.repeat_interleave(k, 0), wmax)
    assert qg.qgemm_device_status() == 0


@pytest.mark.parametrize("bits,group,E,T", [(4, 128, 16, 300), (4, 64, 3, 90), (4, 128, 20, 60), (3, 128, 5, 40)])
def test_moe_multi_against_oracle(qg, bits, group, E, T):
    # two products over one routing (gate and up): 4-bit with 2 * E <= 32
    # experts takes the tensor cores (the 300-token case puts some experts
    # above one 64-token chunk), 2 * 20 experts and 3-bit take the decode
    # kernel, launched per product over the shared routing
    N, K, k = 200, 640, 2
    qa, wa = _experts(E, N, K, bits, group, 0.002, seed=110)
    qb, wb = _experts(E, N, K, bits, group, 0.002, seed=310)
    x = wl.gen_x(T, K, seed=T + 7)
    topk = wl.gen_topk(T, k, E, seed=T + 8)
    ya, yb = qg.qgemm_moe_grouped_multi(x.cuda(), topk.cuda(), [[to_device(q) for q in qa], [to_device(q) for q in qb]])
    torch.cuda.synchronize()
    for y, qs, wmax in ((ya, qa, wa), (yb, qb, wb)):
        ref = oracle.moe(x, topk.numpy(), qs)
        check_product(y.reshape(T * k, N), ref.reshape(T * k, N), x.repeat_interleave(k, 0), wmax)
    # where the single calls take the same kernel (not 4-bit with 16 < E <= 32,
    # which one product alone runs on the tensor cores), the fused call equals
    # two single calls bit for bit
    if not (bits == 4 and 16 < E <= 32):
        sa = qg.qgemm_moe_grouped(x.cuda(), topk.cuda(), [to_device(q) for q in qa])
        sb = qg.qgemm_moe_grouped(x.cuda(), topk.cuda(), [to_device(q) for q in qb])
        torch.cuda.synchronize()
        assert torch.equal(sa, ya) and torch.equal(sb, yb)
    assert qg.qgemm_device_status() == 0


def test_moe_layer_4096_experts_with_outliers(qg):
    # the MoE workload's gate projection (16 experts of 3072 x 4096, INT4
    # group 128) with 0.1 % FP16 outliers per expert, 256 tokens top-2 Zipf
    cfg = wl.MoE()
    qs, wmax = _experts(cfg.n_experts, cfg.ffn, cfg.hidden, 4, 128, 0.001, seed=600)
    x = wl.gen_x(cfg.tokens, cfg.hidden, seed=601)
    topk = wl.gen_topk(cfg.tokens, cfg.top_k, cfg.n_experts)
    y = qg.qgemm_moe_grouped(x.cuda(), topk.cuda(), [to_device(q) for q in qs])
    torch.cuda.synchronize()
    pairs = torch.arange(0, cfg.tokens * cfg.top_k, 7)
    tok, slot = pairs // cfg.top_k, pairs % cfg.top_k
    ref = oracle.moe(x[tok], topk[tok].numpy(), qs)          # [n, k, N]
    got = y[tok.cuda(), slot.cuda()]
    check_product(got, ref[np.arange(len(pairs)), slot.numpy()], x[tok], wmax)
