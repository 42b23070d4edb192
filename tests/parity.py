"""Comparison rules shared by the parity tests.

Tolerances (written here, applied everywhere):

* float32 outputs: relative error at most ``FP32_REL_TOL`` = 2e-6 against the
  oracle, measured as |got - ref| / max(|ref|, 2^-126).  The kernels evaluate
  each output with Kahan's difference of products (error <= 2^-23 relative) and
  the oracle rounds the binary64 result once, so the expected gap is below
  2.4e-7; 2e-6 is the stated bar.
* float16 / bfloat16 outputs: at most ``HALF_ULP_TOL`` = 1 unit in the last place
  of the output type.  The binary32 result is within 2^-23 of the exact value
  (Kahan's form; the 16-bit cache kernels that use one FMA after a product that
  is exact in binary32 are correctly rounded), so narrowing it differs from
  narrowing the exact value by at most one ulp.
* columns the operator must not touch: bit-exact.
* NaN matches NaN (any payload); +0 matches -0; infinities must match exactly.
"""
import numpy as np
import torch

FP32_REL_TOL = 2e-6
HALF_ULP_TOL = 1


def same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    view = {8: torch.int64, 4: torch.int32, 2: torch.int16}[a.element_size()]
    return torch.equal(a.detach().cpu().contiguous().view(view), b.detach().cpu().contiguous().view(view))


def ulp_distance(a: torch.Tensor, b: torch.Tensor) -> np.ndarray:
    a = a.detach().cpu().contiguous()
    b = b.detach().cpu().contiguous()
    view = {4: torch.int32, 2: torch.int16}[a.element_size()]
    nbits = 8 * a.element_size()
    ia = a.view(view).numpy().astype(np.int64) & ((1 << nbits) - 1)
    ib = b.view(view).numpy().astype(np.int64) & ((1 << nbits) - 1)
    sign = 1 << (nbits - 1)
    oa = np.where(ia & sign, -(ia & (sign - 1)), ia)
    ob = np.where(ib & sign, -(ib & (sign - 1)), ib)
    d = np.abs(oa - ob)
    na = torch.isnan(a.float()).numpy()
    nb = torch.isnan(b.float()).numpy()
    d = np.where(na & nb, 0, d)
    return np.where(na ^ nb, 1 << 40, d)


def compare(got: torch.Tensor, ref: torch.Tensor) -> dict:
    """Error summary of ``got`` against the oracle's ``ref`` (same dtype)."""
    assert got.dtype == ref.dtype and got.shape == ref.shape, (got.dtype, ref.dtype, got.shape, ref.shape)
    g = got.detach().cpu()
    r = ref.detach().cpu()
    out = {"n": int(r.numel())}
    if r.dtype == torch.float32:
        gd = g.double().numpy()
        rd = r.double().numpy()
        both_nan = np.isnan(gd) & np.isnan(rd)
        inf_ok = np.isinf(rd) & (gd == rd)
        with np.errstate(invalid="ignore"):
            rel = np.abs(gd - rd) / np.maximum(np.abs(rd), 2.0 ** -126)
        rel = np.where(both_nan | inf_ok, 0.0, rel)
        rel = np.where(np.isnan(rel), np.inf, rel)
        out["max_rel"] = float(rel.max()) if rel.size else 0.0
        out["ok"] = out["max_rel"] <= FP32_REL_TOL
    else:
        d = ulp_distance(g, r)
        out["max_ulp"] = int(d.max()) if d.size else 0
        out["ok"] = out["max_ulp"] <= HALF_ULP_TOL
    return out


def assert_matches(got: torch.Tensor, ref: torch.Tensor, what: str = "") -> dict:
    res = compare(got, ref)
    assert res["ok"], "%s: %s" % (what, res)
    return res


def ulp_of(ref: torch.Tensor) -> np.ndarray:
    """One unit in the last place of each element of ``ref`` (its own dtype)."""
    r = ref.detach().cpu().float().abs().double().numpy()
    bits = {torch.float32: 24, torch.float16: 11, torch.bfloat16: 8}[ref.dtype]
    emin = {torch.float32: -126, torch.float16: -14, torch.bfloat16: -126}[ref.dtype]
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(r > 0, r, 1.0)))
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - (bits - 1)).astype(np.int64))


def assert_close_scaled(got: torch.Tensor, ref: torch.Tensor, scale: np.ndarray, rel: float, what: str = ""):
    """|got - ref| <= 1 ulp(ref) + rel * scale, elementwise (NaN matches NaN).

    For results computed from intermediates that already carry binary32
    rounding (e.g. a normalisation before a rotation), ``scale`` is the size of
    the terms that cancel, so the bound does not blow up under cancellation."""
    g = got.detach().cpu().double().numpy()
    r = ref.detach().cpu().double().numpy()
    both_nan = np.isnan(g) & np.isnan(r)
    with np.errstate(invalid="ignore"):
        err = np.abs(g - r)
    bound = ulp_of(ref) + rel * np.broadcast_to(scale, r.shape)
    bad = ~(both_nan | (err <= bound))
    assert not bad.any(), "%s: %d elements out of bound, worst excess %g" % (
        what, int(bad.sum()), float(np.nanmax(np.where(bad, err - bound, 0))))


def compare_terms(got: torch.Tensor, ref: torch.Tensor, terms: np.ndarray, rel: float = FP32_REL_TOL) -> dict:
    """Element-wise comparison relative to the terms that form each result.

    For an output o = a*c - b*s (or b*c + a*s) built from values a, b that
    are themselves computed (e.g. RMS-normalised), ``terms`` is |a*c| + |b*s|
    in float64; a binary32 evaluation is accurate to a small multiple of
    2^-24 of that sum, whatever cancellation happens in o.  Bound:
      float32:          |got - ref| <= rel * terms
      float16/bfloat16: |got - ref| <= 1 ulp(ref) + rel * terms
    NaN matches NaN.  Returns the largest |got - ref| / bound (at most 1 when
    ``ok``), the largest |got - ref| / terms, the largest ulp distance, the
    element count and ``ok``."""
    g = got.detach().cpu().double().numpy()
    r = ref.detach().cpu().double().numpy()
    t = np.broadcast_to(np.asarray(terms, dtype=np.float64), r.shape)
    both_nan = np.isnan(g) & np.isnan(r)
    with np.errstate(invalid="ignore"):
        err = np.where(both_nan, 0.0, np.abs(g - r))
    err = np.where(np.isnan(err), np.inf, err)
    bound = rel * t
    if ref.dtype != torch.float32:
        bound = bound + ulp_of(ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = np.where(err == 0, 0.0, err / t)
    with np.errstate(divide="ignore", invalid="ignore"):
        of_bound = np.where(err == 0, 0.0, err / bound)
    ulps = ulp_distance(got, ref)
    return {"n": int(r.size), "ok": bool((err <= bound).all()),
            "max_err_over_bound": float(of_bound.max()) if of_bound.size else 0.0,
            "max_err_over_terms": float(scaled.max()) if scaled.size else 0.0,
            "max_ulp": int(ulps.max()) if ulps.size else 0,
            "out_of_bound": int((err > bound).sum())}


def assert_matches_rows(got: torch.Tensor, ref: torch.Tensor, what: str = "", rows: int = 1 << 16) -> None:
    """assert_matches for large tensors: the same rules (float32: relative
    error <= FP32_REL_TOL; half types: <= HALF_ULP_TOL ulps; NaN matches NaN,
    +0 matches -0), evaluated with torch integer and float ops a block of rows
    (last dim) at a time."""
    assert got.shape == ref.shape and got.dtype == ref.dtype, (got.shape, ref.shape, got.dtype, ref.dtype)
    g = got.detach().cpu().reshape(-1, got.shape[-1])
    r = ref.detach().cpu().reshape(-1, ref.shape[-1])
    for i in range(0, g.shape[0], rows):
        gb, rb = g[i:i + rows], r[i:i + rows]
        both_nan = torch.isnan(gb) & torch.isnan(rb)
        one_nan = torch.isnan(gb) ^ torch.isnan(rb)
        assert not bool(one_nan.any()), "%s rows %d..: NaN against a number" % (what, i)
        if ref.dtype == torch.float32:
            gd, rd = gb.double(), rb.double()
            inf_ok = torch.isinf(rd) & (gd == rd)
            rel = (gd - rd).abs() / rd.abs().clamp_min(2.0 ** -126)
            rel = torch.where(both_nan | inf_ok, torch.zeros_like(rel), rel)
            worst = float(torch.nan_to_num(rel, nan=float("inf")).max())
            assert worst <= FP32_REL_TOL, "%s rows %d..: max relative error %g" % (what, i, worst)
        else:
            ia = gb.view(torch.int16).to(torch.int32)
            ib = rb.view(torch.int16).to(torch.int32)
            oa = torch.where(ia < 0, -(ia & 0x7FFF), ia)  # sign-magnitude -> ordered integers
            ob = torch.where(ib < 0, -(ib & 0x7FFF), ib)
            d = torch.where(both_nan, torch.zeros_like(oa), (oa - ob).abs())
            worst = int(d.max())
            assert worst <= HALF_ULP_TOL, "%s rows %d..: max %d ulp" % (what, i, worst)
