"""Comparison helpers for GPU-vs-oracle parity (test infrastructure).

Tolerances (floating point): max relative error per element, over elements
whose oracle magnitude exceeds 1e-3,
  * <= 5e-3 for one block's output residual stream,
  * <= 2e-2 for the final actions / latents after all steps.
bf16 values written to a cache are compared in units in the last place: the
GPU rounds an fp32 value, the oracle a float64 one, so a value next to a
rounding boundary may land one ulp apart; nothing above the 1e-3 magnitude
floor may differ by more.  Below the floor (where a bf16 ulp is smaller than
the fp32 accumulation error of the value) the difference must stay within one
ulp of a value at the floor.
Integer maps (slots, positions) must match exactly.
"""
import os

import numpy as np

REPORT = []   # (what, measured, bound) of every comparison made in this session

BLOCK_TOL = 5e-3
FINAL_TOL = 2e-2
FLOOR = 1e-3


def max_rel_err(got, ref, floor=FLOOR):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in GPU output"
    m = np.abs(ref) > floor
    if not np.any(m):
        return 0.0
    return float(np.max(np.abs(got[m] - ref[m]) / np.abs(ref[m])))


def assert_rel(got, ref, tol, what=""):
    e = max_rel_err(got, ref)
    REPORT.append((what, e, tol))
    assert e <= tol, f"{what}: max relative error {e:.3e} > {tol:.1e}"
    return e


def assert_scale_rel(got, ref, tol, what=""):
    """max |got - ref| / rms(ref) <= tol (for bf16 chain outputs)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got))
    e = float(np.max(np.abs(got - ref)) / np.sqrt(np.mean(ref * ref)))
    REPORT.append((what + " (scale-relative)", e, tol))
    assert e <= tol, f"{what}: max error / rms {e:.3e} > {tol:.1e}"
    return e


def bf16_ulp_distance(a_bits, b_bits):
    """Distance in representable bf16 steps between two arrays of bit patterns."""
    def ordered(bits):
        b = np.asarray(bits, dtype=np.uint16).astype(np.int32)
        return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + b)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def _decode(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def assert_bf16_close(got_bits, ref_bits, what="", max_ulp=1, min_exact=0.99):
    d = bf16_ulp_distance(got_bits, ref_bits)
    g, r = _decode(got_bits), _decode(ref_bits)
    big = np.abs(r) > FLOOR
    bad = big & (d > max_ulp)
    assert not bad.any(), f"{what}: {int(bad.sum())} values above the floor differ by more than {max_ulp} ulp"
    small_tol = max_ulp * 2.0 ** (np.floor(np.log2(FLOOR)) - 7)
    bad_small = (~big) & (np.abs(g - r) > small_tol)
    assert not bad_small.any(), f"{what}: {int(bad_small.sum())} values below the floor off by > {small_tol:.1e}"
    frac = float(np.mean(d == 0))
    REPORT.append((what + " (bit-exact fraction)", frac, min_exact))
    assert frac >= min_exact, f"{what}: only {frac:.4f} of values bit-exact"
    return frac
