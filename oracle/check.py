"""Acceptance criterion for a computed Y against the oracle's double-precision Y.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages judge a fused kernel by the share of elements whose relative error
against a higher-precision reference exceeds 1 % (page "Riepilogo Tecnico ...
Inferenza Efficiente di LLM", section "Contributi Chiave", item 3: the fused
kernels show 0 % such elements).  The bar applied here makes that concrete so
that it is meaningful near zero, where a relative error is undefined:

  (1) every element: |y - ref| <= 1e-2 * |ref| + 1e-3 * max|ref|;
  (2) no element with |ref| > 1e-2 * rms(ref) has |y - ref| / |ref| > 1e-2.

Non-finite values anywhere in y fail (1).

For a result that passes through an intermediate BF16 rounding (the MLP block:
Y is rounded to BF16 before the down projection), the kernel rounds Y from an
FP32 value and the oracle from the exact value, so the two may pick
neighbouring BF16 numbers for a value near a rounding midpoint; both are
correct roundings.  Such results keep (1) unchanged and widen (2) per element
by ``sig_slack``: the most the result can move when every intermediate value
that lies within the kernel's FP32 error bound of a BF16 midpoint rounds the
other way (``bf16_rounding_slack``, propagated by the caller through the
next product).  No fraction of elements is exempt from either rule.
"""
from __future__ import annotations

import numpy as np

REL = 1e-2           # 1 % relative, the pages' mismatch threshold
ABS_OF_MAX = 1e-3    # absolute floor as a fraction of max|ref|
SIG_OF_RMS = 1e-2    # "significant" elements: |ref| above this fraction of rms(ref)


EPS_ACC = 2.0 ** -17  # modelled FP32 accumulation error of the gate and up sums (see below)


def bf16_rounding_slack(y, g, u, gabs, uabs, K: int) -> np.ndarray:
    """Per element of an exact Y = SiLU(G) * U: how far the kernel's BF16 value
    of y may lie from the oracle's (y rounded to nearest even) -- zero unless
    y is near a BF16 rounding midpoint.

    Error model of the kernel's FP32 value of y (all inputs exact BF16):
      * G and U are FP32 sums of K exact products on the tensor cores, in
        K/16 accumulation steps.  Their error is taken as at most
        EPS_ACC (|G| + Gabs/sqrt(K)), Gabs = sum_k |a_k w_k| (likewise U),
        with EPS_ACC = 2^-17: the running sum is of the order of
        |G| + Gabs/sqrt(K), and K/16 roundings of half an ulp each give a
        random-walk error near 2 u32 of it; 2^-17 = 128 u32 leaves a margin
        of about 30 for the tail over the ~10^8 elements a test run checks.
        This is a model with a margin, not a worst-case bound (the tensor
        cores' internal summation order and guard bits are not documented);
      * y = g u / (1 + e^-g): |dy/dg| <= 1.1 |u|, |dy/du| = |SiLU(g)|;
      * the epilogue's exponential carries at most (2 + 1.2 |g|) binary32
        ulps (2^-23 each) relative, the fast division 2 ulps, the sum and
        the product half an ulp each: (5 + 1.2 |g|) 2^-23 |y| in all.
    With dy the resulting bound, the kernel's BF16 value of y rounds as y
    does unless y lies within dy of a BF16 midpoint; there the two BF16
    values may differ by at most the spacing around that midpoint plus dy
    (the slack).  At y = 0 the kernel's value is within dy of 0 (slack 2 dy)."""
    y, g, u = (np.asarray(t, dtype=np.float64) for t in (y, g, u))
    gabs, uabs = np.asarray(gabs, dtype=np.float64), np.asarray(uabs, dtype=np.float64)
    dg = EPS_ACC * (np.abs(g) + gabs / np.sqrt(K))
    du = EPS_ACC * (np.abs(u) + uabs / np.sqrt(K))
    with np.errstate(over="ignore", invalid="ignore"):
        silu_g = g / (1.0 + np.exp(-g))
    silu_g = np.where(np.isfinite(silu_g), silu_g, np.where(g > 0, g, 0.0))
    dy = 1.1 * np.abs(u) * dg + np.abs(silu_g) * du + (5.0 + 1.2 * np.abs(g)) * 2.0 ** -23 * np.abs(y)
    ay = np.abs(y)
    m, e = np.frexp(ay)                    # ay = m 2^e, m in [0.5, 1)
    spacing = np.ldexp(1.0, e - 8)         # BF16: 8 significant bits
    t = np.where(ay > 0, m * 256.0, 0.0)   # in [128, 256)
    d_in = np.abs(t - np.floor(t) - 0.5) * spacing
    # just above a power of two the nearest midpoint may lie below it, where
    # the spacing is half as large
    d_below = np.where((t >= 128.0) & (t < 128.125), (t - 128.0 + 0.25) * spacing, np.inf)
    slack = np.where(d_in <= dy, spacing + dy, 0.0)
    slack = np.maximum(slack, np.where(d_below <= dy, spacing / 2 + dy, 0.0))
    return np.where(ay > 0, slack, 2.0 * dy)


def parity_report(y, ref, sig_slack=None) -> dict:
    """Compare y (any float array) with ref (float64) element by element.
    ``sig_slack`` (same shape as ref): per-element allowance added to rule (2)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if y.shape != ref.shape:
        raise ValueError(f"shape mismatch {y.shape} vs {ref.shape}")
    n = ref.size
    if n == 0:
        return {"n": 0, "ok": True, "n_over_bound": 0, "n_rel_mismatch_sig": 0,
                "mismatch_pct_all": 0.0, "max_abs_err": 0.0, "max_ref": 0.0,
                "rms_ref": 0.0, "max_rel_err_sig": 0.0}
    absref = np.abs(ref)
    max_ref = float(absref.max())
    rms_ref = float(np.sqrt(np.mean(ref * ref)))
    finite = np.isfinite(y)
    err = np.where(finite, np.abs(y - ref), np.inf)
    bound = REL * absref + ABS_OF_MAX * max_ref
    over = err > bound
    sig = absref > SIG_OF_RMS * rms_ref
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(absref > 0, err / absref, np.where(err > 0, np.inf, 0.0))
        if sig_slack is not None:
            e2 = np.maximum(err - np.asarray(sig_slack, dtype=np.float64), 0.0)
            rel2 = np.where(absref > 0, e2 / absref, np.where(e2 > 0, np.inf, 0.0))
        else:
            rel2 = rel
    rel_sig = rel2[sig]
    n_rel_sig = int(np.count_nonzero(rel_sig > REL))
    nonzero = absref > 0
    mismatch_all = float(np.count_nonzero(rel[nonzero] > REL)) / max(1, int(nonzero.sum()))
    rep = {
        "n": int(n),
        "n_over_bound": int(np.count_nonzero(over)),
        "n_rel_mismatch_sig": n_rel_sig,
        "n_significant": int(sig.sum()),
        "mismatch_pct_all": 100.0 * mismatch_all,
        "max_abs_err": float(err.max()),
        "max_ref": max_ref,
        "rms_ref": rms_ref,
        "max_rel_err_sig": float(rel_sig.max()) if rel_sig.size else 0.0,
    }
    rep["ok"] = rep["n_over_bound"] == 0 and n_rel_sig == 0
    if not rep["ok"]:
        idx = np.unravel_index(int(np.argmax(np.where(over, err - bound, -np.inf))), ref.shape)
        rep["worst_index"] = [int(i) for i in idx]
        rep["worst_y"] = float(y[idx])
        rep["worst_ref"] = float(ref[idx])
    return rep


def assert_parity(y, ref, what: str = "", sig_slack=None) -> dict:
    rep = parity_report(y, ref, sig_slack)
    if not rep["ok"]:
        raise AssertionError(f"parity failed {what}: {rep}")
    return rep
