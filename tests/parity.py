"""Shared helpers of the parity tests: tolerance checks and conversions.

Tolerance for floating-point results (stated for the routed-expert path):
  relative Frobenius error  ||gpu - ref|| / ||ref||  <= 5e-3      (bf16 path)
  max abs error             max |gpu - ref|          <= 2e-2 * rms(ref)
For outputs stored in bf16, two implementations that differ only in fp32
summation order can round to neighbouring bf16 values at every rounding point.
y and dx are rounded sums of k bf16-rounded terms (R3/R5, then R6), so an
element whose difference is within one bf16 spacing of the reference value
plus one spacing of each of its k terms (`flip` below, from the oracle's own
terms) also passes the max-abs test; other bf16 outputs get one spacing.
Weight gradients are compared as increments (after - before).
MXFP8 outputs: relative Frobenius error <= 1e-2.
Intermediates (a, h, ys, dA, hs) are diagnostics, not outputs: one bf16 flip
at an earlier rounding point (say of gate or up) can move a later intermediate
by several of its own bf16 steps, so there a small fraction of elements
(max_bad_frac) may exceed the max-abs limit; the Frobenius bound still holds.

Every compare also counts the elements whose difference exceeds the literal
max-abs bound 2e-2 * rms(ref), whatever the bf16 allowance, and the largest such
difference in bf16 steps of the reference value.  For bf16 results that count
must stay at or below LITERAL_FRAC of the elements.  With MOE_PARITY_STATS set
to a file path, each compare appends its figures there as one JSON line.
"""

import json
import os

import numpy as np

# at most this fraction of a bf16 result's elements may exceed the literal
# max-abs bound (they pass only through the bf16 rounding allowance)
LITERAL_FRAC = 1e-3
# fp32 weight gradients sum products of bf16 per-row operands (hs, dA): at most
# this fraction of their elements may exceed the literal max-abs bound, through
# bf16 flips of those operands (measured at the full workloads: up to 3.3e-5)
WGRAD_FLIP_FRAC = 1e-4

REL_FRO = 5e-3
MAX_ABS_RMS = 2e-2
REL_FRO_MXFP8 = 1e-2


def f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_spacing(v):
    """Distance from |v| to the next larger bf16 value (v given as float32)."""
    a = np.abs(np.asarray(v, np.float32))
    e = np.floor(np.log2(np.maximum(a, np.float32(2.0 ** -126))))
    return (2.0 ** (e - 7)).astype(np.float64)


def compare(got, ref, bf16_out=True, rel_fro=REL_FRO, what="", max_bad_frac=0.0, flip=None):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), what + ": non-finite values"
    diff = np.abs(got - ref)
    nref = np.linalg.norm(ref)
    rf = np.linalg.norm(got - ref) / max(nref, 1e-30)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    lim = MAX_ABS_RMS * rms
    bad = diff > lim
    if bf16_out:
        allow = bf16_spacing(ref) if flip is None else bf16_spacing(ref) + flip
        bad &= diff > allow * 1.0000001
    over = diff > lim                      # beyond the literal max-abs bound
    n_over = int(over.sum())
    steps = float((diff[over] / bf16_spacing(ref[over])).max()) if n_over else 0.0
    info = "%s: rel_fro=%.3e max_abs=%.3e (limit %.3e) n_bad=%d n_over_literal=%d/%d (max %.2f bf16 steps)" % (
        what, rf, diff.max() if diff.size else 0.0, lim, int(bad.sum()), n_over, diff.size, steps)
    path = os.environ.get("MOE_PARITY_STATS")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"what": what, "n": int(diff.size), "rel_fro": rf,
                                "max_abs": float(diff.max() if diff.size else 0.0),
                                "literal_limit": float(lim), "n_over_literal": n_over,
                                "frac_over_literal": n_over / max(diff.size, 1),
                                "max_over_bf16_steps": steps, "n_bad": int(bad.sum()),
                                "bf16_out": bool(bf16_out)}) + "\n")
    assert rf <= rel_fro, info
    assert bad.sum() <= max_bad_frac * bad.size, info
    if bf16_out and max_bad_frac < 1.0:
        assert n_over <= LITERAL_FRAC * diff.size, info
    return rf, float(diff.max() if diff.size else 0.0)


def term_flips(terms):
    """Sum over the k terms [..., k, d] (bf16 bits) of one bf16 spacing each."""
    v = f32(terms)
    sp = np.where(v != 0, bf16_spacing(v), 0.0)
    return sp.sum(axis=-2)
