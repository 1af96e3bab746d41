"""Helpers for GPU-vs-oracle parity tests: moving quantized weights between
the oracle (numpy) and the device, and the tolerance of the product."""
import numpy as np
import torch

import oracle

# Product tolerance (stated for the method's outputs against the fp64 oracle):
# per output row m, max_n |y - y_ref| <= 2e-3 * ||x_m||_2 * max |w_hat + S|,
# and relative L2 over the whole y <= 1e-3.
MAX_ABS_FACTOR = 2e-3
REL_L2 = 1e-3


def to_device(q: oracle.QWeight, device="cuda"):
    import bit_weight_only_group_gb300 as qg
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).view(dt)).to(device)
    return qg.QWeight(
        q.N, q.K, q.bits, q.group,
        packed=t(q.packed, np.uint8),
        scale=t(q.scale, np.int16) if q.scale is not None and q.scale8 is None else None,
        zp=t(q.zp, np.uint8) if q.zp is not None else None,
        codebook=t(q.cb, np.int16) if q.cb is not None else None,
        row_ptr=t(q.row_ptr, np.int32),
        col=t(q.col, np.int32) if q.nnz else torch.empty(0, dtype=torch.int32, device=device),
        val=t(q.val, np.int16) if q.nnz else torch.empty(0, dtype=torch.int16, device=device),
        nnz=q.nnz, **_fp8_fields(q, t, device))


def _fp8_fields(q, t, device):
    """The 8-bit scale arrays of an oracle weight (its fp16 ``scale`` then
    only expands them and is not sent)."""
    if q.scale8 is None:
        return {}
    nfb = int(q.fb_col.size)
    return dict(scale8=t(q.scale8, np.uint8),
                scale8_exp=torch.tensor([q.scale_exp], dtype=torch.int32, device=device),
                fb_row_ptr=t(q.fb_row_ptr, np.int32),
                fb_col=t(q.fb_col, np.int32) if nfb else torch.empty(0, dtype=torch.int32, device=device),
                fb_val=t(q.fb_val, np.int16) if nfb else torch.empty(0, dtype=torch.int16, device=device))


def to_host(qw) -> dict:
    c = lambda t: None if t is None else t.cpu().numpy()
    out = dict(packed=c(qw.packed), scale=c(qw.scale), zp=c(qw.zp), cb=c(qw.codebook))
    out["row_ptr"] = c(qw.row_ptr)
    out["col"] = c(qw.col)
    out["val"] = c(qw.val)
    for k in ("scale8", "scale8_exp", "fb_row_ptr", "fb_col", "fb_val"):
        out[k] = c(getattr(qw, k))
    return out


def assert_quantized_equal(qw, ref: oracle.QWeight):
    h = to_host(qw)
    assert np.array_equal(h["packed"], ref.packed), "packed bytes differ"
    if ref.bits == 2:
        assert np.array_equal(h["cb"].view(np.uint16), ref.cb), "codebooks differ"
    elif ref.scale8 is not None:
        assert int(h["scale8_exp"][0]) == ref.scale_exp, "matrix exponents differ"
        assert np.array_equal(h["scale8"], ref.scale8), "8-bit scales differ"
        assert np.array_equal(h["fb_row_ptr"], ref.fb_row_ptr), "fallback row pointers differ"
        nfb = ref.fb_col.size
        assert np.array_equal(h["fb_col"][:nfb], ref.fb_col), "fallback groups differ"
        assert np.array_equal(h["fb_val"][:nfb].view(np.uint16), ref.fb_val), "fallback scales differ"
        assert np.array_equal(h["zp"], ref.zp), "zero-points differ"
    else:
        assert np.array_equal(h["scale"].view(np.uint16), ref.scale), "scales differ"
        assert np.array_equal(h["zp"], ref.zp), "zero-points differ"
    assert qw.nnz == ref.nnz
    if ref.nnz:
        assert np.array_equal(h["row_ptr"], ref.row_ptr), "row_ptr differs"
        assert np.array_equal(h["col"], ref.col), "outlier columns differ"
        assert np.array_equal(h["val"].view(np.uint16), ref.val), "outlier values differ"


def check_product(y, y_ref: np.ndarray, x, wabs_max: float):
    """y (device, [M, n]) against the fp64 oracle y_ref under the stated bound."""
    y = y.double().cpu().numpy()
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    xf = oracle.bf16_to_f64(x)
    xn = np.sqrt((xf ** 2).sum(1))
    err = np.abs(y - y_ref).max(1)
    bound = MAX_ABS_FACTOR * xn * wabs_max
    assert (err <= bound).all(), f"max |dy| {err.max():.3e} above bound {bound[err.argmax()]:.3e}"
    den = np.linalg.norm(y_ref)
    rel = np.linalg.norm(y - y_ref) / den if den > 0 else np.linalg.norm(y)
    assert rel <= REL_L2, f"relative L2 {rel:.3e}"
    return rel
