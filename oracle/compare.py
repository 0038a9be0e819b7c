"""Comparison of a bf16 result against the float64 reference.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

* ``within_tolerance``: the pass rule |y - ref| <= 1e-2 * |ref| + 1e-3, applied
  to every element.
* ``mismatch_rate``: share of elements that break that rule. This is how the
  pages' accuracy figure ("zero mismatches", the share of outputs with more than
  1% relative error against an FP32 reference; "Tile-Level Activation Overlap
  for Efficient LLM Inference", gist.science, section "Key Contributions") is
  read here: a pure 1% relative test is undefined at ref = 0, so the 1e-3
  absolute floor is added.
* ``relative_mismatch_rate``: the pure relative form, over |ref| >= 1e-3 only.
* ``bf16_ulp_distance``: distance in bf16 steps between y and bf16(ref),
  counting on the ordered integer line of bf16 values (+0 and -0 coincide).
"""
from __future__ import annotations

import numpy as np

from .swiglu_ref import bf16_bits_to_f64, f64_to_bf16_bits

RTOL = 1e-2
ATOL = 1e-3


def _excess(y: np.ndarray, ref: np.ndarray) -> np.ndarray:
    return np.abs(y - ref) - (RTOL * np.abs(ref) + ATOL)


def within_tolerance(y_bits, ref) -> np.ndarray:
    """Boolean mask: element passes |y - ref| <= 1e-2 |ref| + 1e-3."""
    y = bf16_bits_to_f64(y_bits)
    ref = np.asarray(ref, dtype=np.float64)
    return _excess(y, ref) <= 0.0


def mismatch_rate(y_bits, ref) -> float:
    ok = within_tolerance(y_bits, ref)
    return float(1.0 - ok.mean()) if ok.size else 0.0


def relative_mismatch_rate(y_bits, ref, floor: float = 1e-3) -> float:
    y = bf16_bits_to_f64(y_bits)
    ref = np.asarray(ref, dtype=np.float64)
    sel = np.abs(ref) >= floor
    if not sel.any():
        return 0.0
    rel = np.abs(y[sel] - ref[sel]) / np.abs(ref[sel])
    return float((rel > RTOL).mean())


def _ordered(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp_distance(y_bits, ref) -> np.ndarray:
    """Number of bf16 steps between y and the bf16 rounding of ref."""
    ref_bits = f64_to_bf16_bits(ref)
    return np.abs(_ordered(y_bits) - _ordered(ref_bits))


def report(y_bits, ref) -> dict:
    """Summary used by tests and by the bench's parity line."""
    y = bf16_bits_to_f64(y_bits)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(y - ref)
    ulp = bf16_ulp_distance(y_bits, ref)
    return {
        "n": int(ref.size),
        "max_abs_err": float(err.max()) if err.size else 0.0,
        "max_excess": float(_excess(y, ref).max()) if err.size else -1.0,
        "tolerance_pass": bool((_excess(y, ref) <= 0).all()),
        "mismatch_rate": mismatch_rate(y_bits, ref),
        "relative_mismatch_rate": relative_mismatch_rate(y_bits, ref),
        "bf16_ulp_gt1_rate": float((ulp > 1).mean()) if ulp.size else 0.0,
        "max_bf16_ulp": int(ulp.max()) if ulp.size else 0,
        "nonfinite": int((~np.isfinite(y)).sum()),
    }
