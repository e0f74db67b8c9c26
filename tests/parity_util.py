"""Shared pieces of the GPU parity tests: error metrics and the tolerances.

Tolerances (element by element against the double-precision oracle):
* bf16 attention: max-abs <= 1e-2 and relative L2 <= 2e-3 (the stated bar).
* fp32 attention: max-abs <= 1e-5 and relative L2 <= 2e-6. Derivation: the
  kernel accumulates in fp32 (unit roundoff 6e-8); a score carries about
  sqrt(d) * 6e-8 relative error and exp2f at most 2 ulp, so each softmax
  weight is off by ~1e-6 relative at worst, and outputs (weighted means of
  N(0,1) values, |out| < 4) by a few 1e-7 typically and ~1e-6 at worst.
* Scatter, block tables, slot mappings and block copies: bit-exact.
"""
import numpy as np

from workloads import bf16_bits_to_f32

TOL = {"bf16": (1e-2, 2e-3), "f32": (1e-5, 2e-6)}


def as_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    return a.astype(np.float64) if dtype == "f32" else bf16_bits_to_f32(a).astype(np.float64)


def errors(got: np.ndarray, want: np.ndarray):
    d = got - want
    return float(np.max(np.abs(d))), float(np.linalg.norm(d) / max(np.linalg.norm(want), 1e-300))


def assert_close(got_bits: np.ndarray, want: np.ndarray, dtype: str, what: str = ""):
    got = as_f64(got_bits, dtype)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    mx, rl = errors(got, want)
    tmax, trel = TOL[dtype]
    assert mx <= tmax and rl <= trel, f"{what}: max-abs {mx:.3g} (<= {tmax}), rel-L2 {rl:.3g} (<= {trel})"
    return mx, rl
