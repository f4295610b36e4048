"""Shared test helpers: independent float64 brute force (numpy matmul on gathered
adapter matrices) and the parity metrics.  No kernel or oracle arithmetic here."""
from __future__ import annotations

import numpy as np

from workloads import bf16_bits_to_f32, to_bf16_bits


def f64(bits) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


def adapter_mats(case: dict, k: int):
    """(A_k [d_in, r], B_k [r, d_out]) in float64, gathered with numpy fancy indexing."""
    r = int(case["rank"][k])
    A = f64(case["a_pool"][case["a_pages"][k, :r], :case["d_in"]]).T
    B = f64(case["b_pool"][case["b_pages"][k, :r], :case["d_out"]])
    return A, B


def exact_delta(case: dict, x=None, ids=None) -> np.ndarray:
    """s_k (x_i A_k) B_k per row in float64 (0 for released rows)."""
    x = case["x"] if x is None else x
    ids = case["ids"] if ids is None else ids
    X = f64(x)
    out = np.zeros((X.shape[0], case["d_out"]), np.float64)
    for k in np.unique(ids[ids >= 0]):
        rows = np.flatnonzero(ids == k)
        A, B = adapter_mats(case, int(k))
        out[rows] = float(case["scale"][k]) * ((X[rows] @ A) @ B)
    return out


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (normal range), float64."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def assert_nearest_bf16(out_bits, exact, slack=1e-9):
    """out must be a nearest bf16 to the exact float64 value (ties either way only
    within float64 noise)."""
    out = f64(out_bits)
    err = np.abs(out - exact)
    half = 0.5 * np.maximum(bf16_ulp(out), bf16_ulp(exact))
    bad = err > half * (1 + slack) + 1e-300
    assert not bad.any(), (
        f"{bad.sum()} elements not nearest: e.g. out={out[bad][:4]} exact={exact[bad][:4]}")


def parity(got_bits, ref_bits):
    """(relative Frobenius error, max abs error / rms(ref)) of two bf16 arrays."""
    return parity_values(f64(got_bits), f64(ref_bits))


def parity_values(g, r):
    """The same two figures for float arrays."""
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    diff = g - r
    den = np.sqrt(np.sum(r * r))
    rms = np.sqrt(np.mean(r * r)) if r.size else 0.0
    rel = float(np.sqrt(np.sum(diff * diff)) / den) if den > 0 else float(np.abs(diff).max(initial=0))
    mx = float(np.abs(diff).max(initial=0.0) / rms) if rms > 0 else float(np.abs(diff).max(initial=0))
    return rel, mx


def assert_parity(got_bits, ref_bits, rel_tol=5e-3, max_tol=2e-2, what="",
                  step_frac=1e-3):
    """Relative Frobenius error <= rel_tol, and every element within
    max(max_tol * rms(ref), one bf16 step at |ref|): both sides round once to bf16,
    and where their fp32 / double sums straddle a rounding boundary they differ by
    one bf16 step, which above |y| ~ 2.6 rms is larger than 2e-2 rms.  The one-step
    allowance may cover at most step_frac of the elements (at least one): a rare
    straddle is expected, a systematic one-step bias is not.  Returns a dict of the
    figures (rel_frob, max_abs/rms, elements beyond max_tol*rms, their count limit)."""
    rel, mx = parity(got_bits, ref_bits)
    g, r = f64(got_bits), f64(ref_bits)
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    err = np.abs(g - r)
    bound = np.maximum(max_tol * rms, bf16_ulp(r))
    worst = float((err / bound).max(initial=0.0))
    n_step = int((err > max_tol * rms).sum())
    cap = max(1, int(step_frac * r.size))
    stats = {"what": what, "rel_frob": rel, "max_abs_over_rms": mx, "one_step": n_step,
             "one_step_cap": cap, "elements": int(r.size)}
    assert rel <= rel_tol and worst <= 1.0 and n_step <= cap, (
        f"{what}: rel_frob={rel:.3e} max_abs/rms={mx:.3e} worst/bound={worst:.3f} "
        f"one-step allowance used by {n_step} of {r.size} elements (cap {cap})")
    return stats


__all__ = ["f64", "adapter_mats", "exact_delta", "assert_nearest_bf16", "parity",
           "assert_parity", "parity_values", "to_bf16_bits", "bf16_ulp"]
