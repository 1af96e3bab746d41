"""Pins for the CPU oracle: facts from the pages and from mathematics that the
oracle must reproduce.  None of these re-states the oracle's own formulas;
each checks a property a plausible slip (dropped term, wrong sign, wrong
shift, transposed operand, wrong rounding mode) would break.
"""
import math
import os

import numpy as np
import pytest

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([s.strip() for s in line.split("|")])
    return rows


# ---------------------------------------------------------------- packing
PACK_ROWS = [(int(b), [int(c) for c in cs.split()], bytes.fromhex(h.replace(" ", "")))
             for b, cs, h in _golden_rows("pack_examples.txt")]


@pytest.mark.parametrize("bits,codes,expect", PACK_ROWS)
def test_pack_matches_hand_worked_units(bits, codes, expect):
    assert oracle.pack(codes, bits).tobytes() == expect
    got = oracle.unpack(np.frombuffer(expect, np.uint8), len(codes), bits)
    assert got.tolist() == codes


UNIT = {2: 4, 3: 8, 4: 2, 5: 8, 6: 4}   # values per packing unit ("Mixed-width quantization" page, section 3.1)
UNIT_BYTES = {2: 1, 3: 3, 4: 1, 5: 5, 6: 3}


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6])
def test_pack_every_code_at_every_lane(bits):
    qmax = (1 << bits) - 1
    for background in (0, qmax):
        for lane in range(UNIT[bits]):
            for c in range(qmax + 1):
                u = [background] * UNIT[bits]
                u[lane] = c
                p = oracle.pack(u, bits)
                assert p.size == UNIT_BYTES[bits]
                assert oracle.unpack(p, len(u), bits).tolist() == u


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6])
def test_pack_units_are_independent_and_roundtrip(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, size=UNIT[bits] * 97).astype(np.uint8)
    p = oracle.pack(codes, bits)
    assert p.size == codes.size * bits // 8
    assert (oracle.unpack(p, codes.size, bits) == codes).all()
    # the stream is the concatenation of its units
    ub, uv = UNIT_BYTES[bits], UNIT[bits]
    for i in range(0, codes.size // uv, 13):
        assert oracle.pack(codes[i * uv:(i + 1) * uv], bits).tobytes() == p[i * ub:(i + 1) * ub].tobytes()


# ---------------------------------------------------------------- fp16 rounding
def test_f16_round_nearest_even_matches_numpy():
    rng = np.random.default_rng(7)
    parts = [rng.standard_normal(100000) * s for s in (1e-7, 1e-5, 1e-3, 1.0, 300.0, 3e4)]
    # midpoints between neighbouring fp16 values exercise ties-to-even
    h = np.arange(0, 0x7BFF, 7, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mids = ((lo + hi) / 2).astype(np.float32)
    edges = np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, 65536.0, 1e9, 2.0 ** -24,
                      2.0 ** -25, 2.0 ** -26, 6.1e-5, -65520.0], np.float32)
    v = np.concatenate(parts + [mids, -mids, edges]).astype(np.float32)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert (oracle.f32_to_f16(v, "rn") == ref).all()


def test_f16_round_up_is_least_upper_bound():
    rng = np.random.default_rng(8)
    v = np.concatenate([np.abs(rng.standard_normal(100000)) * s for s in (1e-6, 1e-3, 0.02, 1.0, 500.0)])
    v = np.concatenate([v, -v]).astype(np.float32)
    h = oracle.f32_to_f16(v, "ru").view(np.float16)
    up = h.astype(np.float64)
    assert (up >= v.astype(np.float64)).all()
    below = np.nextafter(h, np.float16(-np.inf)).astype(np.float64)
    assert (below < v.astype(np.float64)).all()
    # values already in fp16 are unchanged
    exact = rng.standard_normal(1000).astype(np.float16)
    assert (oracle.f32_to_f16(exact.astype(np.float32), "ru") == exact.view(np.uint16)).all()


# ---------------------------------------------------------------- sizing
def _sizing():
    return {r[0]: (float(r[1]), float(r[2])) for r in _golden_rows("sizing.txt")}


def _bytes(layer):
    s = oracle.sizes(layer.N, layer.K, layer.bits, layer.group, layer.frac)
    return sum(v for k, v in s.items() if k != "nnz")


def test_sizing_4096_layer_at_2p5_bits():
    v, _ = _sizing()["layer_4096_2p5bit_bytes"]
    s = oracle.sizes(4096, 4096, 2, 128, 0.0)
    assert s["packed"] + s["codebook"] == v
    assert (s["packed"] + s["codebook"]) * 8 / (4096 * 4096) == 2.5


def test_sizing_scale_overhead_per_group():
    g = _sizing()
    # one fp16 per group: 16 bits spread over the group's weights
    for group, key in ((64, "scale_overhead_bits_g64"), (128, "scale_overhead_bits_g128")):
        s = oracle.sizes(4096, 4096, 4, group, 0.0)
        assert s["scale"] * 8 / (4096 * 4096) == g[key][0]


def test_sizing_70b_stack_is_36GB():
    v, tol = _sizing()["stack70b_int4_outliers_GB"]
    total = sum(_bytes(L) for L in wl.stack_70b())
    assert abs(total / 1e9 - v) <= tol, total


def test_sizing_7b_mixed_stack_is_a_bit_over_3GB():
    g = _sizing()
    total = sum(_bytes(L) for L in wl.stack_7b()) / 1e9
    assert g["stack7b_mixed_GB_min"][0] < total < g["stack7b_mixed_GB_max"][0], total
    # average payload width of the stack is about 3.5 bits ("Mixed-width quantization" page, section 2.2: 3.4-3.6)
    w = sum(L.N * L.K * L.bits for L in wl.stack_7b()) / sum(L.N * L.K for L in wl.stack_7b())
    assert 3.4 <= w <= 3.7, w


def test_nnz_is_floor_of_fraction():
    assert oracle.nnz(4096, 4096, 0.001) == 16777
    assert oracle.nnz(11008, 4096, 0.001) == 45088
    assert oracle.nnz(4096, 4096, 0.0) == 0
    assert oracle.nnz(10, 10, 0.001) == 0


# ---------------------------------------------------------------- outliers
def test_outliers_recover_the_planted_set():
    N, K = 96, 1024
    W = wl.gen_weight(N, K, seed=11, outlier_frac=0.001, outlier_seed=12)
    n = oracle.nnz(N, K, 0.001)
    assert n == wl.planted_count(N, K, 0.001) > 0
    w = W.float().numpy()
    planted = set(np.flatnonzero(np.abs(w) >= 3.0).tolist())
    assert len(planted) == n
    row_ptr, col = oracle.select_outliers(W, 0.001)
    got = set()
    for r in range(N):
        cs = col[row_ptr[r]:row_ptr[r + 1]]
        assert (np.diff(cs) > 0).all()
        got |= {r * K + int(c) for c in cs}
    assert got == planted


def test_outlier_ties_break_by_lower_index():
    rng = np.random.default_rng(3)
    N, K = 6, 64
    mags = rng.choice([0.5, 1.0, 2.0], size=(N, K), p=[0.5, 0.4, 0.1])
    w = (mags * rng.choice([-1.0, 1.0], size=(N, K))).astype(np.float16)
    frac = 0.2   # cuts inside the block of |w| == 1.0
    n = oracle.nnz(N, K, frac)
    flat = np.abs(w.astype(np.float64)).ravel()
    expect = sorted(range(N * K), key=lambda i: (-flat[i], i))[:n]
    row_ptr, col = oracle.select_outliers(w, frac)
    got = sorted(r * K + int(c) for r in range(N) for c in col[row_ptr[r]:row_ptr[r + 1]])
    assert got == sorted(expect)


# ---------------------------------------------------------------- affine quantizer
def _groups(q: oracle.QWeight):
    codes = np.stack([oracle.unpack(q.packed[r], q.K, q.bits) for r in range(q.N)])
    return codes.reshape(q.N, q.K // q.group, q.group)


def _outlier_mask(q):
    m = np.zeros((q.N, q.K), bool)
    for r in range(q.N):
        m[r, q.col[q.row_ptr[r]:q.row_ptr[r + 1]]] = True
    return m


@pytest.mark.parametrize("bits", [3, 4, 5, 6, 8])
@pytest.mark.parametrize("group", [32, 64, 128])
def test_affine_codes_are_nearest_grid_points(bits, group):
    N, K, frac = 24, 1024, 0.002
    W = wl.gen_weight(N, K, seed=100 + bits, outlier_frac=frac, outlier_seed=200 + group)
    q = oracle.quantize(W, bits, group, frac)
    qmax = (1 << bits) - 1
    w = W.double().numpy()
    xhat = oracle.dequant(q)
    out = _outlier_mask(q)
    assert out.sum() == oracle.nnz(N, K, frac)
    # outliers are reproduced exactly: the dense part is 0 and S holds fp16(w)
    assert (xhat[out] == w[out]).all()
    assert (q.val == W.numpy().view(np.uint16)[out]).all()
    s = oracle.f16_to_f32(q.scale).astype(np.float64)          # [N, ng]
    zp = q.zp.astype(np.float64)
    assert (q.zp <= qmax).all()
    sg = np.repeat(s, group, axis=1)
    zg = np.repeat(zp, group, axis=1)
    err = np.abs(w - xhat)
    # round-trip bound: half a step, plus an fp32 rounding slack of the quotient
    assert (err[~out] <= sg[~out] * (0.5 + 2.0 ** -20)).all()
    # brute force over all 2^b grid points: the chosen one is the nearest
    grid = (np.arange(qmax + 1)[None, None, :] - zg[..., None]) * sg[..., None]
    best = np.abs(w[..., None] - grid).min(axis=-1)
    assert (err[~out] <= best[~out] + sg[~out] * 2.0 ** -20).all()
    # the code at an outlier is the zero point
    codes = _groups(q).reshape(N, K)
    assert (codes[out] == zg[out]).all()


@pytest.mark.parametrize("bits", [4, 5, 6])
def test_affine_scale_is_least_fp16_step_covering_the_range(bits):
    N, K, group = 32, 1024, 128
    W = wl.gen_weight(N, K, seed=31 + bits)
    q = oracle.quantize(W, bits, group, 0.0)
    qmax = (1 << bits) - 1
    w = W.float().numpy().reshape(N, K // group, group)
    mn = np.minimum(w.min(-1), 0).astype(np.float32)
    mx = np.maximum(w.max(-1), 0).astype(np.float32)
    need = (mx - mn) / np.float32(qmax)                          # fp32 quotient
    s = q.scale.view(np.float16)
    assert (s.astype(np.float32) >= need).all()
    assert (np.nextafter(s, np.float16(0)).astype(np.float32) < need).all()


def test_affine_grid_aligned_ramp_is_exact():
    # values on a 0.25-spaced grid spanning 16 levels reproduce exactly at 4 bits
    ramp = (np.arange(16) - 5) * 0.25
    row = np.tile(ramp, 8)                                       # 128 values
    W = np.stack([row, row[::-1], np.roll(row, 3)]).astype(np.float16)
    q = oracle.quantize(W, 4, 128, 0.0)
    assert (oracle.dequant(q) == W.astype(np.float64)).all()
    assert (q.scale.view(np.float16) == np.float16(0.25)).all()
    assert (q.zp == 5).all()


def test_affine_exact_ties_round_half_to_even():
    # "round" in the quantizer formula (inference-acceleration guide page,
    # section 1.1) read as round half to even.  Two 4-bit groups whose range
    # is exactly 3.75 force scale = 3.75 / 15 = 0.25 (exact in fp32 and fp16),
    # and weights at odd multiples of 0.125 land exactly on k + 1/2.  The
    # codes below are worked out by hand; rounding half away from zero, or
    # half up, gives a different code for every tie.
    g = 64
    a = np.zeros(g, np.float16)             # min -1.25, max 2.5: zp = -round(-5) = 5 (no tie)
    a[:9] = [-1.25, 2.5, 0.125, 0.625, -0.125, -0.625, 1.125, 0.375, -0.375]
    b = np.zeros(g, np.float16)             # min -1.125, max 2.625: min/scale = -4.5 is a tie
    b[:3] = [-1.125, 2.625, 0.875]
    q = oracle.quantize(np.concatenate([a, b])[None, :], 4, g, 0.0)
    assert (q.scale.view(np.float16) == np.float16(0.25)).all()
    # zp = 0 - round(min / scale): round(-5) = -5 and round(-4.5) = -4 (even)
    assert q.zp.tolist() == [[5, 4]]
    codes = oracle.unpack(q.packed[0], 2 * g, 4)
    # group a, q = round(w / 0.25) + 5: -5 -> 0, 10 -> 15, 0.5 -> 0, 2.5 -> 2,
    # -0.5 -> 0, -2.5 -> -2, 4.5 -> 4, 1.5 -> 2, -1.5 -> -2; zeros -> 5
    assert codes[:9].tolist() == [0, 15, 5, 7, 5, 3, 9, 7, 3]
    assert (codes[9:g] == 5).all()
    # group b, q = round(w / 0.25) + 4: -4.5 -> -4, 10.5 -> 10, 3.5 -> 4; zeros -> 4
    assert codes[g:g + 3].tolist() == [0, 14, 8]
    assert (codes[g + 3:] == 4).all()


def test_affine_zero_and_one_signed_groups():
    W = np.zeros((2, 128), np.float16)
    W[1, :] = np.float16(0.75)                                   # all positive
    q = oracle.quantize(W, 4, 128, 0.0)
    xhat = oracle.dequant(q)
    assert (xhat[0] == 0).all()
    assert (q.zp[1] == 0).all()                                  # range widened to include 0
    assert (np.abs(xhat[1] - 0.75) <= q.scale.view(np.float16)[1, 0] / 2).all()


@pytest.mark.parametrize("bits", [4, 5, 6])
def test_affine_error_is_uniform_noise(bits):
    # rounding to a grid of step s leaves errors ~ U(-s/2, s/2): E[e^2] = s^2/12
    N, K, group = 512, 1024, 128
    W = wl.gen_weight(N, K, seed=55)
    q = oracle.quantize(W, bits, group, 0.0)
    e = (W.double().numpy() - oracle.dequant(q)).reshape(N, K // group, group)
    s = q.scale.view(np.float16).astype(np.float64)
    ratio = ((e ** 2).mean(-1) / s ** 2).mean()
    assert abs(ratio - 1 / 12) < 0.1 / 12, ratio


# ---------------------------------------------------------------- codebook (2 bit)
def test_codebook_codes_nearest_and_lloyd_not_worse_than_uniform():
    N, K, group, frac = 32, 1024, 64, 0.002
    W = wl.gen_weight(N, K, seed=91, outlier_frac=frac, outlier_seed=92)
    q = oracle.quantize(W, 2, group, frac)
    w = W.double().numpy()
    out = _outlier_mask(q)
    cb = q.cb.view(np.float16).astype(np.float64)                 # [N, ng, 4]
    assert (np.diff(cb, axis=-1) >= 0).all()                      # ascending
    codes = _groups(q)
    wg = w.reshape(N, -1, group)
    og = out.reshape(N, -1, group)
    for r in range(N):
        for j in range(K // group):
            keep = ~og[r, j]
            v = wg[r, j][keep]
            e = cb[r, j]
            d = np.abs(v[:, None] - e[None, :])
            chosen = d[np.arange(v.size), codes[r, j][keep]]
            assert (chosen <= d.min(1) + 1e-12).all()
            # Lloyd never increases distortion from its uniform start
            mn, mx = min(v.min(), 0.0), max(v.max(), 0.0)
            uni = mn + np.arange(4) * (mx - mn) / 3
            d_uni = (np.abs(v[:, None] - uni[None, :]).min(1) ** 2).sum()
            d_cb = (chosen ** 2).sum()
            assert d_cb <= d_uni * (1 + 1e-3) + 1e-12
            # outliers: code nearest to 0, residual restores w to fp16 precision
            for k in np.flatnonzero(og[r, j]):
                c = codes[r, j][k]
                assert c == int(np.argmin(np.abs(e)))
    xhat = oracle.dequant(q)
    assert (np.abs(xhat[out] - w[out]) <= np.abs(w[out]) * 2.0 ** -10).all()


def test_codebook_is_a_lloyd_fixed_point_near_the_gaussian_optimum():
    # A converged k-means codebook satisfies the centroid condition: each
    # entry is the mean of the values coded to it (up to fp16 rounding of the
    # entry).  Max (1960): the 4-level minimum-MSE quantizer of N(0,1) has
    # levels +-0.4528, +-1.5104 and distortion 0.1175.  Per-group k-means on
    # 128 samples fits its own sample: its in-sample distortion lies below
    # the population optimum and its outer levels sit further out.
    n_groups, group = 3000, 128
    w = wl.gen_group_values(n_groups, group, seed=5, std=1.0)
    q = oracle.quantize(w.reshape(1, -1), 2, group, 0.0)
    cb = q.cb.view(np.float16).astype(np.float64).reshape(n_groups, 4)
    codes = _groups(q).reshape(n_groups, group)
    v = w.astype(np.float64)
    dev = []
    for gi in range(n_groups):
        for j in range(4):
            sel = codes[gi] == j
            if sel.any():
                dev.append(abs(v[gi][sel].mean() - cb[gi, j]) / max(abs(cb[gi, j]), 1e-3))
    dev = np.array(dev)
    assert np.quantile(dev, 0.95) < 2.0 ** -10, np.quantile(dev, 0.95)
    xhat = oracle.dequant(q).reshape(n_groups, group)
    dist = ((v - xhat) ** 2).mean()
    assert 0.100 < dist < 0.1175, dist
    lv = cb.mean(0)
    assert abs(lv.sum()) < 0.05                                   # symmetric input
    assert 0.40 < -lv[1] < 0.55 and 0.40 < lv[2] < 0.55, lv
    assert 1.45 < -lv[0] < 1.80 and 1.45 < lv[3] < 1.80, lv


def test_codebook_tie_rules_on_a_closed_form_group():
    # Values -3, -1, 1, 3 (32 each) start Lloyd exactly on its fixed point
    # [-3, -1, 1, 3].  Two zeros sit exactly between -1 and 1: ties go to
    # the lower entry, so the -1 cell becomes {31 x -1, 2 x 0} with mean
    # -31/33, and stays so.  The two largest |w| (the first two 3.0 by
    # index) are outliers; the entry nearest to 0 is then -31/33.
    g = np.concatenate([np.full(32, -3.0), np.full(31, -1.0), [0.0, 0.0],
                        np.full(31, 1.0), np.full(32, 3.0)])
    W = g.astype(np.float16)[None, :]
    q = oracle.quantize(W, 2, 128, 0.0)
    e = q.cb.view(np.float16).astype(np.float64).ravel()
    assert e[0] == -3.0 and e[2] == 1.0 and e[3] == 3.0
    assert e[1] == float(np.float16(-31.0 / 33.0))
    codes = _groups(q).ravel()
    assert (codes[63:65] == 1).all()
    # outlier tie: a symmetric codebook has two entries nearest to 0
    g2 = np.concatenate([np.full(32, -3.0), np.full(32, -1.0), np.full(32, 1.0), np.full(32, 3.0)])
    W2 = g2.astype(np.float16)[None, :]
    q2 = oracle.quantize(W2, 2, 128, 2.0 / 128 + 1e-6)
    assert q2.nnz == 2
    codes2 = _groups(q2).ravel()
    assert (q2.col == [0, 1]).all()
    assert (codes2[q2.col] == 1).all()                            # entry -1, the lower of +-1
    assert (q2.val.view(np.float16) == np.float16(-2.0)).all()    # -3 - (-1)


# ---------------------------------------------------------------- the product
@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_linear_is_x_times_dequant_transposed(bits):
    N, K, M = 8, 128, 3
    W = wl.gen_weight(N, K, seed=71, outlier_frac=0.02, outlier_seed=72)
    q = oracle.quantize(W, bits, 64, 0.02)
    x = wl.gen_x(M, K, seed=73)
    y = oracle.linear(x, q)
    ref = oracle.bf16_to_f64(x) @ oracle.dequant(q).T
    assert y.shape == (M, N)
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-13)


def test_linear_one_hot_selects_a_column():
    N, K = 8, 256
    W = wl.gen_weight(N, K, seed=81, outlier_frac=0.01, outlier_seed=82)
    q = oracle.quantize(W, 5, 128, 0.01)
    D = oracle.dequant(q)
    for k in (0, 1, 127, 128, 255):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80                                          # bf16 1.0
        assert (oracle.linear(x, q)[0] == D[:, k]).all()


def test_linear_additive_over_disjoint_support_and_zero_weights():
    N, K = 16, 256
    W = wl.gen_weight(N, K, seed=83)
    q = oracle.quantize(W, 3, 64, 0.0)
    x = oracle.as_u16(wl.gen_x(2, K, seed=84)).copy()
    x1, x2 = x.copy(), x.copy()
    x1[:, K // 2:] = 0
    x2[:, :K // 2] = 0
    y, y1, y2 = (oracle.linear(a, q) for a in (x, x1, x2))
    assert np.allclose(y, y1 + y2, rtol=1e-13, atol=1e-13)
    qz = oracle.quantize(np.zeros((N, K), np.float16), 4, 128, 0.0)
    assert (oracle.linear(x, qz) == 0).all()


def test_linear_row_ranges_agree_with_full():
    N, K = 40, 128
    q = oracle.quantize(wl.gen_weight(N, K, seed=85), 6, 128, 0.0)
    x = wl.gen_x(4, K, seed=86)
    full = oracle.linear(x, q)
    assert (oracle.linear(x, q, 7, 23) == full[:, 7:23]).all()


def test_moe_routes_each_pair_to_its_expert():
    E, N, K, T, k = 4, 8, 128, 10, 2
    experts = [oracle.quantize(wl.gen_weight(N, K, seed=300 + e), 4, 128, 0.0) for e in range(E)]
    x = wl.gen_x(T, K, seed=310)
    topk = wl.gen_topk(T, k, E, seed=311).numpy()
    y = oracle.moe(x, topk, experts)
    xb = oracle.as_u16(x)
    for t in range(T):
        for j in range(k):
            assert (y[t, j] == oracle.linear(xb[t:t + 1], experts[topk[t, j]])[0]).all()
    assert all(len(set(r)) == k for r in topk.tolist())


# ---------------------------------------------------------------- layer diagnostics
def test_diagnostics_hand_worked_group():
    # "Mixed-width quantization" page, section 6.1 (max |error|, RMSE, cosine
    # of unpacked vs original weights) and 6.2 (block max over second max).
    # One 4-bit group of 64: w0 = 1.5, w1 = 0.75, zeros elsewhere.  By hand:
    # scale = fp16 rounded up of 1.5 / 15 = 0.10003662109375, zp = 0,
    # q0 = round(14.9945) = 15, q1 = round(7.4973) = 7, so
    # w_hat0 = 1.50054931640625 and w_hat1 = 0.70025634765625.
    W = np.zeros((1, 64), np.float16)
    W[0, 0], W[0, 1] = 1.5, 0.75
    q = oracle.quantize(W, 4, 64, 0.0)
    assert q.scale.view(np.float16)[0, 0] == np.float16(0.10003662109375)
    h0, h1 = 1.50054931640625, 0.70025634765625
    e0, e1 = 1.5 - h0, 0.75 - h1
    d = oracle.diagnostics(W, q, threshold=1.5)
    assert d["max_abs_err"] == abs(e1) == 0.04974365234375
    assert d["rmse"] == pytest.approx(math.sqrt((e0 ** 2 + e1 ** 2) / 64), rel=1e-15)
    cos = (1.5 * h0 + 0.75 * h1) / (math.hypot(1.5, 0.75) * math.hypot(h0, h1))
    assert d["cosine"] == pytest.approx(cos, rel=1e-15)
    assert d["ratio"].tolist() == [[2.0]] and d["max_range_ratio"] == 2.0 and d["groups_over"] == 1
    assert oracle.diagnostics(W, q, threshold=2.0)["groups_over"] == 0


def test_diagnostics_range_ratio_special_groups():
    W = np.zeros((1, 5 * 64), np.float16)
    W[0, 64:128][10] = 0.5                       # one nonzero: ratio +inf
    W[0, 128:192][[3, 40]] = [-0.25, 0.25]       # equal magnitudes: 1
    W[0, 192:256][[0, 1, 2]] = [3.0, -4.0, 1.0]  # 4 / 3 (magnitudes, either sign)
    W[0, 256:320][5] = -2.0                      # one nonzero, negative: +inf
    d = oracle.diagnostics(W, oracle.quantize(W, 5, 64, 0.0), threshold=1.2)
    r = d["ratio"][0]
    assert r[0] == 1.0 and np.isinf(r[1]) and r[2] == 1.0 and r[3] == pytest.approx(4 / 3) and np.isinf(r[4])
    assert d["groups_over"] == 3 and np.isinf(d["max_range_ratio"])


def test_diagnostics_exact_layer_and_outliers_count_as_exact():
    # weights on the 4-bit grid reproduce exactly: no error, cosine 1; an
    # outlier is stored in FP16 and added back, so it adds no error either
    ramp = np.tile((np.arange(16) - 5) * 0.25, 8)
    W = np.stack([ramp, ramp[::-1]]).astype(np.float16)
    d = oracle.diagnostics(W, oracle.quantize(W, 4, 128, 0.0))
    assert d["max_abs_err"] == 0.0 and d["rmse"] == 0.0 and d["cosine"] == 1.0
    W2 = W.copy()
    W2[1, 7] = np.float16(1000.0)
    q2 = oracle.quantize(W2, 4, 128, 1 / 256)    # exactly one outlier: the 1000
    assert q2.nnz == 1 and q2.col.tolist() == [7]
    d2 = oracle.diagnostics(W2, q2)
    assert d2["max_range_ratio"] == 1000.0 / 2.5


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6])
def test_diagnostics_invariants(bits):
    N, K, group = 48, 512, 64
    W = wl.gen_weight(N, K, seed=70 + bits, outlier_frac=0.002, outlier_seed=71)
    q = oracle.quantize(W, bits, group, 0.002)
    d = oracle.diagnostics(W, q)
    e = W.double().numpy() - oracle.dequant(q)
    assert d["max_abs_err"] == np.abs(e).max()
    assert d["rmse"] <= d["max_abs_err"]
    assert -1.0 <= d["cosine"] <= 1.0
    if bits != 2:   # affine: half a step per element at most
        s = oracle.f16_to_f32(q.scale).astype(np.float64).max()
        assert d["max_abs_err"] <= s * (0.5 + 2.0 ** -20)
    # wider codes fit better
    if bits >= 3:
        dq = oracle.diagnostics(W, oracle.quantize(W, bits - 1 if bits > 3 else 3, group, 0.002))
        assert dq["rmse"] >= d["rmse"] * (1 - 1e-12)


# ---------------------------------------------------------------- quantizer variants
def _codes(q):
    return oracle.unpack(q.packed[0], q.K, q.bits)


def test_symmetric_3bit_hand_worked():
    # no zero point ("Mixed-width quantization" page, section 2.3), integer
    # range [-3, 3] at 3 bits (the symmetric convention of the inference-
    # acceleration guide page, section 1.1): amax 1.5 -> scale 0.5, stored
    # codes q + 4; ties round to even (-2.5 -> -2, 1.5 -> 2, 0.5 -> 0)
    W = np.zeros((1, 64), np.float16)
    W[0, :6] = [1.5, -1.25, 0.75, -0.75, 0.25, 1.0]
    q = oracle.quantize(W, 3, 64, 0.0, mode="symmetric")
    assert q.scale.view(np.float16)[0, 0] == np.float16(0.5) and q.zp[0, 0] == 4
    c = _codes(q)
    assert c[:6].tolist() == [7, 2, 6, 2, 4, 6] and (c[6:] == 4).all()


def test_symmetric_2bit_constants_hand_worked():
    # 2 bits, symmetric: levels -s, 0, s with s = amax (the fourth constant repeats s)
    W = np.zeros((1, 64), np.float16)
    W[0, :5] = [0.75, -0.3, 0.4, -0.75, 0.2]
    q = oracle.quantize(W, 2, 64, 0.0, mode="symmetric")
    assert q.cb.view(np.float16)[0, 0].tolist() == [-0.75, 0.0, 0.75, 0.75]
    c = _codes(q)
    assert c[:5].tolist() == [2, 1, 2, 0, 1] and (c[5:] == 1).all()


def test_linear2_hand_worked():
    # the affine grid at 2 bits: range [-1.25, 2.5] -> scale 1.25, zp 1;
    # constants (i - 1) * 1.25; 0.5 -> 0 and 1.5 -> 2 (ties to even)
    W = np.zeros((1, 64), np.float16)
    W[0, :4] = [-1.25, 2.5, 0.625, 1.875]
    q = oracle.quantize(W, 2, 64, 0.0, mode="linear2")
    assert q.cb.view(np.float16)[0, 0].tolist() == [-1.25, 0.0, 1.25, 2.5]
    c = _codes(q)
    assert c[:4].tolist() == [0, 3, 1, 3] and (c[4:] == 1).all()


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6])
def test_symmetric_is_odd_and_within_half_a_step(bits):
    # round half to even and a clamp at +-qs are odd functions: quantizing -W
    # gives exactly -w_hat; every non-outlier is within half a step; the
    # outliers come back exactly
    N, K, group, frac = 24, 512, 64, 0.004
    W = wl.gen_weight(N, K, seed=80 + bits, outlier_frac=frac, outlier_seed=81)
    q = oracle.quantize(W, bits, group, frac, mode="symmetric")
    qn = oracle.quantize(-W, bits, group, frac, mode="symmetric")
    xh, xn = oracle.dequant(q), oracle.dequant(qn)
    assert np.array_equal(xn, -xh)
    w = W.double().numpy()
    out = _outlier_mask(q)
    assert (xh[out] == w[out]).all()
    if bits == 2:
        s = q.cb.view(np.float16)[..., 2].astype(np.float64)
    else:
        s = q.scale.view(np.float16).astype(np.float64)
        assert (q.zp == 1 << (bits - 1)).all() and (_groups(q) != 0).all()
    sg = np.repeat(s, group, axis=1)
    if bits > 2:
        assert (np.abs(w - xh)[~out] <= sg[~out] * (0.5 + 2.0 ** -20)).all()
    else:   # 3 levels: values beyond s/2 of every level can only be above 1.5 s, impossible by amax = s
        assert (np.abs(w - xh)[~out] <= sg[~out] * (0.5 + 2.0 ** -20)).all()


def test_linear2_constants_are_the_affine_grid():
    N, K, group, frac = 24, 512, 128, 0.004
    W = wl.gen_weight(N, K, seed=90, outlier_frac=frac, outlier_seed=91)
    q = oracle.quantize(W, 2, group, frac, mode="linear2")
    cb = q.cb.view(np.float16).astype(np.float64)             # [N, ng, 4]
    step = cb[..., 1:] - cb[..., :-1]
    # uniform: equal steps (each constant rounded to fp16 once)
    assert np.allclose(step, step[..., :1], rtol=2e-3)
    assert ((cb == 0).sum(-1) == 1).all()                       # the zero code's constant is exactly 0
    out = _outlier_mask(q)
    assert (oracle.dequant(q)[out] == W.double().numpy()[out]).all()


def test_int8_packing_is_one_byte_per_code():
    # 8 bits: the stream's bytes are the codes themselves
    codes = np.arange(256, dtype=np.uint8)
    assert oracle.pack(codes, 8).tolist() == codes.tolist()
    assert oracle.sizes(4096, 4096, 8, 128, 0.0)["packed"] == 4096 * 4096


# ---------------------------------------------------------------- W8A8
def _bf16(vals):
    import torch
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)[None, :]


def test_activation_int8_hand_worked():
    # per-token symmetric INT8 ("Inference acceleration guide" page, sections
    # 1.1-1.2): amax = 127/64 gives scale 1/64 exactly; 3/128 * 64 = 1.5 -> 2
    # and 1/128 * 64 = 0.5 -> 0 (ties to even)
    x = _bf16([1.984375, -1.0, 0.5, 0.0234375, 0.0078125, -1.984375, 0.0])
    q, s = oracle.quantize_act_int8(x)
    assert s.tolist() == [1 / 64]
    assert q[0].tolist() == [127, -64, 32, 2, 0, -127, 0]
    q0, s0 = oracle.quantize_act_int8(_bf16([0.0, 0.0]))
    assert s0.tolist() == [1.0] and q0.tolist() == [[0, 0]]


def test_w8a8_product_is_the_product_of_the_quantized_activations():
    N, K = 24, 256
    W = wl.gen_weight(N, K, seed=101, outlier_frac=0.004, outlier_seed=102)
    qw = oracle.quantize(W, 8, 128, 0.004)
    x = wl.gen_x(3, K, seed=103)
    q, s = oracle.quantize_act_int8(x)
    xhat = q.astype(np.float64) * s[:, None].astype(np.float64)
    # the same sum two ways: the oracle's W8A8 product, and dequantize-then-matmul
    assert np.allclose(oracle.linear_w8a8(x, qw), xhat @ oracle.dequant(qw).T, rtol=1e-12, atol=1e-12)
    # each activation within half a step of its value, the largest at +-127
    xf = oracle.bf16_to_f64(x)
    assert (np.abs(xhat - xf) <= s[:, None] * (0.5 + 2.0 ** -20)).all()
    assert (np.abs(q).max(1) == 127).all()


# ---------------------------------------------------------------- tile-ordered copy
@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
@pytest.mark.parametrize("group", [32, 128])
def test_tiles_layout_reads_back_every_code_and_parameter(bits, group):
    # read the layout back with the thread/word formula and compare with the
    # planar stream unpacked by the generic bit loop: every code of every row
    # (ragged last tile) and the group parameters land where stated
    N, K = 300, 256
    q = oracle.quantize(wl.gen_weight(N, K, seed=bits), bits, group, 0.0)
    t = oracle.tiles(q)
    npg = 2 if group == 32 else 1                  # groups one 64-wide K block touches
    per = 8 if bits == 2 else 4                    # parameter bytes per group
    blk = 2048 * bits + 256 * per * npg
    KB = K // 64
    assert t.size == ((N + 255) // 256) * KB * blk
    for n in (0, 1, 255, 256, 299):
        nt, r = divmod(n, 256)
        row = oracle.unpack(q.packed[n], K, bits)
        for kb in range(KB):
            base = (nt * KB + kb) * blk
            words = t[base:base + 2048 * bits].view(np.uint32).reshape(bits, 512)
            for h in range(2):
                chunk = words[:, 2 * r + h].astype(np.uint32).view(np.uint8)
                assert oracle.unpack(chunk, 32, bits).tolist() == row[64 * kb + 32 * h:64 * kb + 32 * h + 32].tolist()
            prm = t[base + 2048 * bits:base + blk]
            for i in range(npg):
                g = 64 * kb // group + i
                at = per * npg * r + per * i
                if bits == 2:
                    assert prm[at:at + 8].view(np.uint16).tolist() == q.cb[n, g].tolist()
                else:
                    w = int(prm[at:at + 4].view(np.uint32)[0])
                    assert (w & 0xFFFF, w >> 16) == (int(q.scale[n, g]), int(q.zp[n, g]))
    # rows past N are zero in the last tile
    base = (1 * KB + 0) * blk
    words = t[base:base + 2048 * bits].view(np.uint32).reshape(bits, 512)
    assert (words[:, 2 * 44:] == 0).all()


# ---------------------------------------------------------------- group 32 and E4M3 scales
def test_sizing_block32_effective_bits():
    # "Mixed-width quantization" page, section 2.3: one fp16 scale per block
    # of 32 gives 3.5 / 5.5 / 6.5 effective bits at 3 / 5 / 6 bits, and an
    # 8-bit scale costs 8 bits per 32 weights (0.25 bit)
    g = _sizing()
    for bits in (3, 5, 6):
        s = oracle.sizes(4096, 4096, bits, 32, 0.0)
        assert (s["packed"] + s["scale"]) * 8 / (4096 * 4096) == g[f"effective_bits_g32_fp16_b{bits}"][0]
    q = oracle.quantize(wl.gen_weight(64, 1024, seed=5), 3, 32, 0.0, scale_fmt="fp8")
    assert q.scale8.nbytes * 8 / (64 * 1024) == g["scale_overhead_bits_g32_fp8"][0]


def _torch_e4m3(codes):
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    t = torch.tensor(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def test_e4m3_decode_matches_the_library_format():
    # every one of the 256 codes decodes as torch's float8_e4m3fn does
    # (a library routine of the same format); 0x7F and 0xFF are its NaNs
    codes = np.arange(256)
    ref = _torch_e4m3(codes)
    mine = np.array([oracle.e4m3_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert nan.tolist() == np.isnan(mine).tolist() and nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert (mine[~nan] == ref[~nan]).all()
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x08) == 2.0 ** -6


def test_e4m3_round_up_is_least_normal_upper_bound():
    # hand-worked: 1 -> 0x38; 0.3 = 1.2 * 2^-2 rounds up to 1.25 * 2^-2 = 0x2A;
    # 448 -> 0x7E; just above 448, or below 2^-6, there is no normal code
    assert oracle.e4m3_ceil_normal(1.0) == 0x38
    assert oracle.e4m3_ceil_normal(0.3) == 0x2A
    assert oracle.e4m3_ceil_normal(448.0) == 0x7E
    assert oracle.e4m3_ceil_normal(448.0001) == -1
    assert oracle.e4m3_ceil_normal(2.0 ** -6) == 0x08
    assert oracle.e4m3_ceil_normal(2.0 ** -6 * 0.999) == -1
    # every t: the chosen value is >= t and the normal code below it is < t,
    # checked against the library's decode of the codes
    table = _torch_e4m3(np.arange(0x08, 0x7F))
    rng = np.random.default_rng(7)
    for t in np.concatenate([2.0 ** rng.uniform(-6, np.log2(448), 300), table]):
        c = oracle.e4m3_ceil_normal(float(t))
        assert table[c - 0x08] >= t
        assert c == 0x08 or table[c - 0x09] < t


def test_fp8_matrix_exponent_is_the_lower_median():
    h = lambda v: np.array(v, np.float16).view(np.uint16)
    # floor(log2) of 1, 0.25, 3, 0.5 = 0, -2, 1, -1: sorted -2, -1, 0, 1 -> -1
    assert oracle.fp8_matrix_exponent(h([1.0, 0.25, 3.0, 0.5])) == -1
    assert oracle.fp8_matrix_exponent(h([1.0, 0.25, 3.0, 0.5, 100.0])) == 0
    assert oracle.fp8_matrix_exponent(h([2.0 ** -24, 2.0 ** -20, 65504.0])) == -20   # fp16 subnormals count
    assert oracle.fp8_matrix_exponent(h([0.75])) == -1


def test_fp8_scales_hand_worked():
    # seven 4-bit groups of 32, asymmetric.  Fp16 scales (range / 15): 0.25,
    # 0.5, 1, fp16_up(0.3) = 0.30004883, 2^-12, 128, 2^-10; floor(log2) = -2,
    # -1, 0, -2, -12, 7, -10; sorted -12, -10, -2, -2, -1, 0, 7 -> E = -2.  In
    # the format's terms (x 4): 1, 2, 4 exact (0x38, 0x40, 0x48); 1.2002
    # rounds up to 1.25 (0x3A, stored scale 0.3125); 2^-10 is below every
    # E4M3 value, 512 above 448, and 2^-8 only a subnormal: all three keep fp16.
    g = 32
    W = np.zeros((1, 7 * g), np.float32)
    W[0, 0:2] = [-1.0, 2.75]
    W[0, g:g + 2] = [-2.5, 5.0]
    W[0, 2 * g:2 * g + 2] = [-5.0, 10.0]
    W[0, 3 * g:3 * g + 3] = [-1.5, 3.0, 0.5]
    W[0, 4 * g:4 * g + 2] = [-5 * 2.0 ** -12, 10 * 2.0 ** -12]
    W[0, 5 * g:5 * g + 2] = [-640.0, 1280.0]
    W[0, 6 * g:6 * g + 2] = [-5 * 2.0 ** -10, 10 * 2.0 ** -10]
    q = oracle.quantize(W.astype(np.float16), 4, g, 0.0, scale_fmt="fp8")
    assert q.scale_exp == -2
    assert q.scale8[0].tolist() == [0x38, 0x40, 0x48, 0x3A, 0x7F, 0x7F, 0x7F]
    assert q.fb_row_ptr.tolist() == [0, 3]
    assert q.fb_col.tolist() == [4, 5, 6]
    assert q.fb_val.view(np.float16).tolist() == [2.0 ** -12, 128.0, 2.0 ** -10]
    assert q.scale[0].view(np.float16).tolist() == [0.25, 0.5, 1.0, 0.3125, 2.0 ** -12, 128.0, 2.0 ** -10]
    # group 3 with scale 0.3125: zp = -round(-1.5 / 0.3125 = -4.8) = 5;
    # 3.0 / 0.3125 = 9.6 -> 10 + 5 = 15; 0.5 / 0.3125 = 1.6 -> 2 + 5 = 7
    codes = oracle.unpack(q.packed[0], 7 * g, 4)
    assert int(q.zp[0, 3]) == 5
    assert codes[3 * g:3 * g + 4].tolist() == [0, 15, 7, 5]


@pytest.mark.parametrize("mode", ["asymmetric", "symmetric"])
@pytest.mark.parametrize("bits,group", [(3, 32), (4, 128), (6, 64), (8, 128)])
def test_fp8_scales_round_up_and_keep_half_step_bound(mode, bits, group):
    N, K, frac = 48, 1024, 0.002
    W = wl.gen_weight(N, K, seed=60 + bits, outlier_frac=frac, outlier_seed=61)
    q16 = oracle.quantize(W, bits, group, frac, mode=mode)
    q8 = oracle.quantize(W, bits, group, frac, mode=mode, scale_fmt="fp8")
    s16 = q16.scale.view(np.float16).astype(np.float64)
    s8 = q8.scale.view(np.float16).astype(np.float64)
    fb = q8.scale8 == 0x7F
    # stored scale: the fp16 one where it falls back, else rounded up by less
    # than one E4M3 step (1/8 relative) from it
    assert (s8[fb] == s16[fb]).all()
    assert (s8[~fb] >= s16[~fb]).all() and (s8[~fb] < s16[~fb] * 1.125).all()
    assert (q8.scale8[~fb] >= 0x08).all() and (q8.scale8[~fb] <= 0x7E).all()
    # every non-outlier is within half a stored step of its dequantized value
    out = _outlier_mask(q8)
    err = np.abs(W.double().numpy() - oracle.dequant(q8))
    sg = np.repeat(s8, group, axis=1)
    assert (err[~out] <= sg[~out] * (0.5 + 2.0 ** -20)).all()
    assert (err[out] == 0).all()
    # Gaussian weights with their outliers taken out: no group falls back
    # (the page reports under 0.3 % on real layers)
    assert fb.mean() < 0.003


def test_fp8_fallback_rows_list_every_fallback_group_once():
    rng = np.random.default_rng(3)
    N, K, g = 40, 512, 32
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    # groups scaled far down or far up fall outside the window
    tiny = rng.random((N, K // g)) < 0.05
    huge = rng.random((N, K // g)) < 0.03
    f = np.where(tiny, 2.0 ** -11, np.where(huge, 2.0 ** 9, 1.0))
    W = (W.reshape(N, K // g, g) * f[..., None]).reshape(N, K).astype(np.float16)
    q = oracle.quantize(W, 5, g, 0.0, scale_fmt="fp8")
    fb = q.scale8 == 0x7F
    assert (fb >= (tiny | huge)).all() and fb.sum() == q.fb_col.size
    for n in range(N):
        cols = q.fb_col[q.fb_row_ptr[n]:q.fb_row_ptr[n + 1]]
        assert cols.tolist() == np.nonzero(fb[n])[0].tolist()
