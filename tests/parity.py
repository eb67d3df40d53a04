"""Comparison rules between the CUDA path and the CPU oracle.

Tolerances (the operator's contract):
  * E4M3 codes: at least 99.99% equal in value (+0 and -0 count as equal:
    the sign of an exact zero is not fixed by the method), the rest at most
    one E4M3 step apart;
  * alpha and s: relative difference at most 1e-6;
  * bf16 reconstruction: relative RMS difference at most 1e-3.
Both sides hand an fp32 number to the E4M3 rounding, so the codes can only
differ where the two fp32 values straddle a rounding boundary.
"""

from __future__ import annotations

import numpy as np

CODE_EQUAL_FRACTION = 0.9999
SCALE_RTOL = 1e-6
RECON_REL_RMS = 1e-3


def e4m3_ordinal(codes: np.ndarray) -> np.ndarray:
    """Position of each code on the value line (both zeros at 0)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def compare_codes(got: np.ndarray, want: np.ndarray, what: str = "codes") -> dict:
    og, ow = e4m3_ordinal(got), e4m3_ordinal(want)
    assert og.shape == ow.shape, (what, og.shape, ow.shape)
    diff = np.abs(og - ow)
    frac = float(np.mean(diff == 0)) if diff.size else 1.0
    worst = int(diff.max()) if diff.size else 0
    assert frac >= CODE_EQUAL_FRACTION, f"{what}: only {frac:.6%} equal"
    assert worst <= 1, f"{what}: codes differ by {worst} E4M3 steps"
    return {"equal_fraction": frac, "max_steps": worst}


def compare_int8_codes(got: np.ndarray, want: np.ndarray, what: str = "int8 codes") -> dict:
    """INT8 fallback codes: the same bar, steps of one integer."""
    og = np.asarray(got, dtype=np.uint8).view(np.int8).astype(np.int64)
    ow = np.asarray(want, dtype=np.uint8).view(np.int8).astype(np.int64)
    assert og.shape == ow.shape, (what, og.shape, ow.shape)
    diff = np.abs(og - ow)
    frac = float(np.mean(diff == 0)) if diff.size else 1.0
    worst = int(diff.max()) if diff.size else 0
    assert frac >= CODE_EQUAL_FRACTION, f"{what}: only {frac:.6%} equal"
    assert worst <= 1, f"{what}: codes differ by {worst}"
    return {"equal_fraction": frac, "max_steps": worst}


def compare_scales(got: np.ndarray, want: np.ndarray, what: str) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    rel = np.abs(got - want) / np.abs(want)
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= SCALE_RTOL, f"{what}: relative difference {worst:.3e}"
    return worst


def rel_rms(got: np.ndarray, want: np.ndarray) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / den) if den > 0 else float(np.linalg.norm(got))


def compare_recon(got: np.ndarray, want: np.ndarray, what: str = "reconstruction") -> float:
    r = rel_rms(got, want)
    assert r <= RECON_REL_RMS, f"{what}: relative RMS {r:.3e}"
    return r
