"""Comparison rules between the CUDA path and the oracle.

Tolerances (stated once, used by every parity test):
* BF16 outputs (attention out, compressed cmp_kv): max |err| <= 2e-2 and
  mean |err| <= 2e-3 against the float64 oracle, plus the per-row bounds of
  "DeepSeek V4.1 Flash" (tests/golden/row_tolerances.txt).
* Indexer scores: |err| <= 1e-4 * |s|, or, where heads cancel,
  |err| <= 1e-5 * scale_c * sum_h |w_h| * sum_d |q_hd * k_cd|.
* Top-k: the selected set equals the oracle's wherever the oracle's k-th and
  (k+1)-th scores are separated by more than their tolerances; otherwise
  every selected entry must score within tolerance of every unselected one
  (the Top-K acceptance rule of "DeepSeek V4.1 Flash": eligibility,
  uniqueness, ascending positions, trailing -1, cutoff score quality).
* INT8 codes: within +-1 of the oracle's, and different on at most 1e-3 of
  the codes.  The GPU computes the pooled value in FP32, the oracle in
  float64; where an intermediate BF16 rounding (after pooling, after RMSNorm)
  or the final round-half-even sits on a tie, the two can round apart by one
  BF16 ulp or one code.  Scales within 1e-6 relative.
* lse: within 2e-3 absolute.  The tensor-core path feeds the query to the
  MMA in BF16; its 448 unrotated channels are BF16 inputs already, the 64
  rotated channels are rounded (relative error <= 2^-9).  A logit then moves
  by about softmax_scale * 2^-9 * sqrt(64) * E|q| * E|k| ~ 4e-4 for N(0,1)
  data; 2e-3 is five times that.  Denominators are summed in FP32.
"""

import numpy as np

from golden.load import constants

ROW = constants("row_tolerances.txt")
BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
SCORE_REL = 1e-4
SCORE_FLOOR = 1e-5
LSE_ABS = 2e-3
INT8_FLIP_RATE = 1e-3


def check_bf16(got, ref, what="output", magnitude=1.0):
    """``magnitude`` scales the absolute bounds for outputs whose values are
    larger than the O(1) outputs of the workloads (BF16 error is relative)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    assert err.max() <= BF16_MAX_ABS * magnitude, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= BF16_MEAN_ABS * magnitude, f"{what}: mean abs err {err.mean():.3e}"
    # per-row bounds (rows = all but the last axis)
    g2 = got.reshape(-1, got.shape[-1])
    r2 = ref.reshape(-1, ref.shape[-1])
    rms_ref = np.sqrt(np.mean(r2 ** 2, axis=1))
    rms_err = np.sqrt(np.mean((g2 - r2) ** 2, axis=1))
    max_err = np.max(np.abs(g2 - r2), axis=1)
    bad = rms_err > ROW["rms_abs"] + ROW["rms_rel"] * rms_ref
    assert not bad.any(), f"{what}: {bad.sum()} rows over the RMS bound"
    bad = max_err > ROW["max_abs"] + ROW["max_rel"] * rms_ref
    assert not bad.any(), f"{what}: {bad.sum()} rows over the peak bound"
    return float(err.max()), float(err.mean())


def score_tolerance(q_rot, w, keys, scales):
    """Per-entry score tolerance (see module docstring).  q_rot [H, Di] float64
    (already rotated), w [H], keys [n, Di] float64, scales [n]."""
    mag = np.abs(keys) @ np.abs(q_rot).T  # [n, H]: sum_d |q_hd k_cd|
    floor = SCORE_FLOOR * scales * (mag @ np.abs(w))
    return floor


def check_scores(got, ref, floor):
    got = np.asarray(got, np.float64)
    tol = np.maximum(SCORE_REL * np.abs(ref), floor)
    err = np.abs(got - ref)
    bad = err > tol
    assert not bad.any(), (f"{bad.sum()} scores out of tolerance; worst "
                           f"{(err / np.maximum(tol, 1e-300)).max():.2f}x tol")
    return tol


def check_topk(sel, ref_scores, tol, k):
    """GPU selection `sel` (length k, ascending, -1 padded) against the oracle's
    float64 scores of the visible entries."""
    sel = np.asarray(sel, np.int64)
    V = len(ref_scores)
    n = min(k, V)
    chosen = sel[:n]
    assert np.all(sel[n:] == -1), "padding must be -1"
    assert np.all(chosen >= 0) and np.all(chosen < V), "eligibility"
    assert np.all(np.diff(chosen) > 0), "ascending and unique"
    if V <= k:
        assert np.array_equal(chosen, np.arange(V))
        return True
    mask = np.zeros(V, bool)
    mask[chosen] = True
    lo_in = np.min(ref_scores[mask] + tol[mask])
    hi_out = np.max(ref_scores[~mask] - tol[~mask])
    assert lo_in >= hi_out, "cutoff score quality: an unselected entry clearly beats a selected one"
    # exact set where the oracle's boundary is clear
    order = np.argsort(-ref_scores, kind="stable")
    kth, k1 = order[k - 1], order[k]
    clear = (ref_scores[kth] - tol[kth]) > (ref_scores[k1] + tol[k1])
    if clear:
        assert np.array_equal(np.sort(order[:k]), chosen), "set differs at a clear boundary"
    return clear


def check_int8(codes, scale, ref_codes, ref_scale):
    codes = np.asarray(codes, np.int64)
    ref_codes = np.asarray(ref_codes, np.int64)
    assert abs(float(scale) - float(ref_scale)) <= 1e-6 * abs(float(ref_scale)), "scale"
    diff = np.abs(codes - ref_codes)
    assert diff.max() <= 1, "code off by more than one"
    return int((diff > 0).sum())


def check_fp4(codes, sbytes, ref_codes, ref_sbytes, group, scale_fmt):
    """A packed E2M1 row and its scale bytes from the GPU against the
    oracle's.  Scale bytes may differ by one (an amax at a rounding boundary
    of the scale); in groups whose scales agree, a code may differ only to a
    neighbouring magnitude of the same sign (a quotient at a tie of the E2M1
    grid).  Returns (differing scale groups, differing codes)."""
    import oracle as O

    sb = np.asarray(sbytes, np.int64)
    rsb = np.asarray(ref_sbytes, np.int64)
    assert np.all(np.abs(sb - rsb) <= 1), "scale bytes differ by more than one"
    same = np.repeat(sb == rsb, group)
    c = O.unpack_nibbles(codes).astype(np.int64)[same]
    rc = O.unpack_nibbles(ref_codes).astype(np.int64)[same]
    diff = c != rc
    mag, rmag = c & 7, rc & 7
    ok = (np.abs(mag - rmag) <= 1) & (((c ^ rc) & 8 == 0) | (mag == 0) | (rmag == 0))
    assert np.all(ok[diff]), "a code differs by more than one grid step"
    return int((sb != rsb).sum()), int(diff.sum())


def check_mxfp8(codes, sbytes, ref_codes, ref_sbytes, group=32):
    """MXFP8 codes (E4M3, one byte a channel) and E8M0 scale bytes from the
    GPU against the oracle's, with the same allowances as check_fp4: a scale
    byte may differ by one, a code (where the scales agree) only to the
    neighbouring E4M3 value of the same sign.  Returns (differing scale
    groups, differing codes)."""
    sb = np.asarray(sbytes, np.int64)
    rsb = np.asarray(ref_sbytes, np.int64)
    assert np.all(np.abs(sb - rsb) <= 1), "scale bytes differ by more than one"
    same = np.repeat(sb == rsb, group)
    c = np.asarray(codes, np.int64)[same]
    rc = np.asarray(ref_codes, np.int64)[same]
    diff = c != rc
    mag, rmag = c & 0x7F, rc & 0x7F
    ok = (np.abs(mag - rmag) <= 1) & (((c ^ rc) & 0x80 == 0) | (mag == 0) | (rmag == 0))
    assert np.all(ok[diff]), "a code differs by more than one step"
    return int((sb != rsb).sum()), int(diff.sum())

