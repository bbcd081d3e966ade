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
* Published codes (INT8, FP4, MXFP8): every code equals the oracle's except
  where a rounding decision sits on a tie, and each differing code must be
  shown to sit there.  The GPU pools in FP32, the oracle in float64, so the
  pooled value's BF16 rounding can go the other way when the oracle's pooled
  value lies within the FP32 error bound of a BF16 tie (``pooled_error_bound``:
  4 sigma of the K-term FP32 logit sums, carried through the softmax; a
  rotated channel shares its RoPE partner's flag); and the final rounding
  (round-half-even of y/s for INT8, the nearest E2M1 or E4M3 value) can go
  the other way where the quotient lies within 1e-3 (relative for the
  low-bit grids) of a tie.  INT8 scales within 1e-6 relative, unless the
  row's largest element is itself at a BF16 tie (then the row's codes may
  move by one); a low-bit scale byte may differ by one only where the
  group's largest element is at a BF16 tie or amax / top sits within 1e-3
  of the scale rule's boundary (that group's codes are then not compared).
* lse: within 2e-3 absolute.  The tensor-core path feeds the query to the
  MMA in BF16; its 448 unrotated channels are BF16 inputs already, the 64
  rotated channels are rounded (relative error <= 2^-9).  A logit then moves
  by about softmax_scale * 2^-9 * sqrt(64) * E|q| * E|k| ~ 4e-4 for N(0,1)
  data; 2e-3 is five times that.  Denominators are summed in FP32.
"""

import numpy as np

from golden.load import constants

ROW = constants("row_tolerances.txt")
U32 = 2.0 ** -24  # FP32 unit roundoff
TIE_SIGMAS = 4.0
HALF_BAND = 1e-3  # quotient distance from a rounding tie that may round either way
BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
SCORE_REL = 1e-4
SCORE_FLOOR = 1e-5
LSE_ABS = 2e-3
INT8_FLIP_RATE = 1e-3

E2M1_TIES = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


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


# ------------------------------------------------------------------ rounding ties


def bf16_tie_distance(v):
    """Distance of each value from the nearest BF16 rounding tie (the
    midpoint of two neighbouring BF16 values)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    ulp = np.exp2(e - 7)  # BF16 spacing in [2^e, 2^(e+1))
    r = a / ulp - 0.5
    d = np.abs(r - np.rint(r)) * ulp
    # the tie just below 2^e, where the spacing halves
    below = a - (np.exp2(e) - np.exp2(e - 9))
    return np.where(a > 0, np.minimum(d, np.abs(below)), np.inf)


def pooled_error_bound(rec, dx):
    """FP32 error bound of the GPU's pooled value of one published group
    (per channel), from the oracle's trace record: each logit is a dx-term
    FP32 dot product plus the APE, whose rounding errors add up like a
    random walk: about u * sqrt(dx) times the partial sums' size, which
    stays within a few times the root sum of squares of the terms (``mag``);
    taken as TIE_SIGMAS * 4 * u * sqrt(dx) * mag.  A logit error d_j moves
    the softmax weights by w_j (d_j - mean d), hence the pooled value by at
    most 2 max d * sum_j w_j |kv_j - y|; exp, sum and division add a few u."""
    lg, kv, mag, y = rec["logits"], rec["kvs"], rec["mag"], rec["pooled"]
    dl = TIE_SIGMAS * 4 * np.sqrt(dx) * U32 * mag + 4 * U32 * np.abs(lg)
    w = np.exp(lg - lg.max(axis=0))
    w /= w.sum(axis=0)
    return (2 * dl.max(axis=0) * (w * np.abs(kv - y)).sum(axis=0) +
            8 * U32 * (w * np.abs(kv)).sum(axis=0))


def tie_flags(rec, dx, rope_dim=64):
    """Channels whose published value may legitimately differ from the
    oracle's by a BF16 rounding of the pooled value: the pooled value within
    its FP32 bound of a BF16 tie (after RMSNorm, also the normalised value
    within a few u of one).  On rotated rows a flag covers both channels of
    its RoPE pair (the rotation mixes them)."""
    f = bf16_tie_distance(rec["pooled"]) <= pooled_error_bound(rec, dx)
    if rec.get("normed") is not None:
        # RMSNorm: its own FP32 rounding, and a pooled flip moves the row's
        # norm by at most one BF16 ulp of the largest square's share
        v = np.asarray(rec["normed"], np.float64)
        yb = np.asarray(rec["ybf16"], np.float64)
        share = float(np.max(yb * yb) / max(np.sum(yb * yb), 1e-300))
        band = 16 * U32 * np.abs(v) + (np.abs(v) * 2.0 ** -7 * share if f.any() else 0.0)
        f = f | (bf16_tie_distance(v) <= band)
    if rec["rotated"]:
        d = len(f)
        pr = f[d - rope_dim:].reshape(-1, 2).any(axis=1)
        f = f.copy()
        f[d - rope_dim:] = np.repeat(pr, 2)
    return f


def check_int8_tied(codes, scale, ref_codes, ref_scale, rec, dx):
    """One INT8 row against the oracle's under the tie rule (module
    docstring).  Returns the number of differing codes."""
    codes = np.asarray(codes, np.int64)
    ref_codes = np.asarray(ref_codes, np.int64)
    diff = codes != ref_codes
    assert np.all(np.abs(codes - ref_codes) <= 1), "code off by more than one"
    ties = tie_flags(rec, dx)
    y = np.asarray(rec["y"], np.float64)
    if abs(float(scale) - float(ref_scale)) > 1e-6 * abs(float(ref_scale)):
        amax_ch = int(np.argmax(np.abs(y)))
        assert ties[amax_ch], "scale differs but the row's largest element is not at a BF16 tie"
        return int(diff.sum())
    q = np.abs(y / float(ref_scale))
    half = np.abs(q - np.floor(q) - 0.5) <= HALF_BAND
    bad = diff & ~(ties | half)
    assert not bad.any(), (f"{int(bad.sum())} INT8 codes differ away from any rounding tie "
                           f"(channels {np.nonzero(bad)[0][:8].tolist()})")
    return int(diff.sum())


def _e4m3_mids():
    import oracle as O

    v = np.sort(O.e4m3_decode(np.arange(0, 127)))
    return (v[1:] + v[:-1]) / 2


def _group_scale_tied(ties, y32, sb, rsb, group, scale_fmt):
    """Groups whose scale byte may differ by one: the group's largest element
    at a BF16 tie, or amax / top within HALF_BAND of the scale rule's
    boundary (a power of two for E8M0, an E4M3 rounding tie for E4M3)."""
    a = np.abs(y32).reshape(-1, group)
    amax = a.max(axis=1)
    arg = a.argmax(axis=1)
    tg = ties.reshape(-1, group)[np.arange(len(arg)), arg]
    top = 448.0 if scale_fmt == "mxfp8" else 6.0
    r = amax / top
    if scale_fmt == "e4m3":
        mids = _e4m3_mids()
        near = np.array([np.min(np.abs(x - mids)) <= HALF_BAND * x for x in r])
    else:
        lg = np.log2(np.where(r > 0, r, 1.0))
        near = np.abs(lg - np.rint(lg)) <= HALF_BAND
    return tg | near


def check_lowbit_tied(codes, sbytes, ref_codes, ref_sbytes, rec, dx, group, scale_fmt):
    """One low-bit row (packed E2M1 with E4M3 or E8M0 scales, or MXFP8 codes
    with ``scale_fmt="mxfp8"``) against the oracle's under the tie rule.
    Returns (differing scale groups, differing codes)."""
    import oracle as O

    sb = np.asarray(sbytes, np.int64)
    rsb = np.asarray(ref_sbytes, np.int64)
    assert np.all(np.abs(sb - rsb) <= 1), "scale bytes differ by more than one"
    y32 = np.asarray(rec["y"], np.float64).astype(np.float32).astype(np.float64)
    ties = tie_flags(rec, dx)
    gdiff = sb != rsb
    if gdiff.any():
        ok = _group_scale_tied(ties, y32, sb, rsb, group, scale_fmt)
        assert np.all(ok[gdiff]), "a scale byte differs away from a rounding tie"
    same = np.repeat(~gdiff, group)
    if scale_fmt == "mxfp8":
        c = np.asarray(codes, np.int64)
        rc = np.asarray(ref_codes, np.int64)
        scale = O.e8m0_decode(rsb)
        q = np.abs(y32 / np.repeat(scale, group))
        mids = _e4m3_mids()
        idx = np.clip(np.searchsorted(mids, q), 1, len(mids) - 1)
        dist = np.minimum(np.abs(q - mids[idx - 1]), np.abs(q - mids[np.minimum(idx, len(mids) - 1)]))
        grid_tie = dist <= HALF_BAND * np.maximum(q, 1e-30)
        step = np.abs((c & 0x7F) - (rc & 0x7F))
    else:
        c = O.unpack_nibbles(codes).astype(np.int64)
        rc = O.unpack_nibbles(ref_codes).astype(np.int64)
        dec = O.e8m0_decode if scale_fmt == "e8m0" else O.e4m3_decode
        scale = dec(rsb)
        q = np.abs(y32 / np.where(np.repeat(scale, group) > 0, np.repeat(scale, group), np.inf))
        grid_tie = np.min(np.abs(q[:, None] - E2M1_TIES[None, :]) /
                          E2M1_TIES[None, :], axis=1) <= HALF_BAND
        step = np.abs((c & 7) - (rc & 7))
    diff = (c != rc) & same
    assert np.all(step[diff] <= 1), "a code differs by more than one grid step"
    sbit = 0x80 if scale_fmt == "mxfp8" else 8
    mag_c, mag_r = c & (sbit - 1), rc & (sbit - 1)
    assert np.all(((c ^ rc) & sbit == 0) | (mag_c == 0) | (mag_r == 0)), "a code's sign differs"
    bad = diff & ~(ties | grid_tie)
    assert not bad.any(), (f"{int(bad.sum())} low-bit codes differ away from any rounding tie "
                           f"(channels {np.nonzero(bad)[0][:8].tolist()})")
    return int(gdiff.sum()), int(diff.sum())
