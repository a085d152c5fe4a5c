"""Parity metric and tolerances.

Per output tensor, row-wise normwise relative error:
    err_i = max_f |g[i,f] - r[i,f]| / max_f |r[i,f]|
Rows whose reference is all zero use the absolute error (<= 1e-6).  A
per-element relative error is ill-conditioned under cancellation, hence the
row-wise form.

Tolerances (row-wise relative): fp32 sum, mean, SpMM and attention 1e-4;
bf16-input paths with fp32 accumulation 2e-2; max/argmax, indexing,
permutation and build outputs bit-exact.

Gradients whose terms cancel (the attention backward: the score gradients
of a row sum to zero) are compared per element against the magnitude of
the terms they sum, the scale a floating-point sum's error is bounded by:
    |g - r| <= tol * S,   S = sum over the terms of |term|
(assert_terms_close).  A row whose terms cancel can be far smaller than
its terms, so its row-wise relative error says nothing about the kernel.
"""
import numpy as np

TOL_F32 = 1e-4
TOL_BF16 = 2e-2
ABS_ZERO_ROW = 1e-6


def rowwise_rel_err(got, ref):
    got = np.asarray(got, np.float64).reshape(len(got), -1)
    ref = np.asarray(ref, np.float64).reshape(len(ref), -1)
    if got.shape != ref.shape:
        raise AssertionError(f"shape {got.shape} != {ref.shape}")
    if got.size == 0:
        return np.zeros(len(got)), np.zeros(len(got), bool)
    scale = np.max(np.abs(ref), axis=1)
    diff = np.abs(got - ref)
    diff = np.where(np.isnan(diff), np.inf, diff)
    err = np.max(diff, axis=1)
    zero = scale == 0
    rel = np.where(zero, err, err / np.where(zero, 1.0, scale))
    return rel, zero


def assert_rowwise_close(got, ref, tol, what=""):
    rel, zero = rowwise_rel_err(got, ref)
    bad_rel = (~zero) & (rel > tol)
    bad_abs = zero & (rel > ABS_ZERO_ROW)
    if np.any(bad_rel) or np.any(bad_abs):
        i = int(np.argmax(np.where(zero, rel / ABS_ZERO_ROW, rel / tol)))
        raise AssertionError(f"{what}: row {i} error {rel[i]:.3e} > tol "
                             f"({'abs' if zero[i] else 'rel'}); worst over "
                             f"{int(bad_rel.sum() + bad_abs.sum())} rows")
    return float(np.max(rel)) if len(rel) else 0.0


def assert_lse_close(got, ref, tol, what="lse"):
    """logsumexp: absolute error (a shift of L is a relative error of
    exp(L))."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(got - ref))
    d = np.where(np.isnan(d), np.inf, d)
    if np.max(d, initial=0.0) > tol:
        i = np.unravel_index(int(np.argmax(d)), d.shape)
        raise AssertionError(f"{what}: {i} got {got[i]} ref {ref[i]}")
    return float(np.max(d, initial=0.0))


def assert_terms_close(got, ref, scale, tol, what=""):
    """|got - ref| <= tol * scale element by element, scale the summed
    magnitude of each element's terms (an element without terms must match
    to 1e-12)."""
    got = np.asarray(got, np.float64).reshape(-1)
    ref = np.asarray(ref, np.float64).reshape(-1)
    scale = np.asarray(scale, np.float64).reshape(-1)
    if not (got.shape == ref.shape == scale.shape):
        raise AssertionError(f"{what}: shapes {got.shape} {ref.shape} {scale.shape}")
    diff = np.abs(got - ref)
    diff = np.where(np.isnan(diff), np.inf, diff)
    ratio = diff / (tol * scale + 1e-12)
    if ratio.size and np.max(ratio) > 1.0:
        k = int(np.argmax(ratio))
        raise AssertionError(f"{what}: element {k} error {diff[k]:.3e} > {tol:g} x terms "
                             f"{scale[k]:.3e} ({int(np.sum(ratio > 1))} elements)")
    return float(np.max(diff / np.maximum(scale, 1e-300), initial=0.0))
