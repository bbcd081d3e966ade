"""Plain CPU oracle for compressed sparse attention (CSA).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import or call
this module: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library; both
sides only share the seeded input generator in ``workloads``.

Everything is computed in float64 with numpy, one definition at a time,
straight from the pages:

* "DeepSeek V4.1 Flash" (pypto-lib), sections "Serving-owned full RoPE
  tables" (FP32 half-width tables, adjacent-pair rotation, negative position =
  identity), "Compressor state ownership" (pooling softmax, BF16 rounding
  before RMSNorm, the recurrent state ring of kv rows and gate scores across
  calls, Top-K acceptance rules, per-row tolerances).
* "Hyper-Parallel ... DeepSeek V4 CP" (gitcode issue #2), sections
  "二阶段 CP 总体算法" (shared-KV sparse attention with sinks, softmax_scale,
  ori_win_left = 127), "7. Window KV Halo" (window includes self),
  "8.2 ratio=128" and "10.3 Causal mask" (slot c visible to position p iff
  c < (p + 1) // ratio).
* "DeepSeek V4-Flash, MTP point", sections "What is quantized" (INT8 per-row
  amax floored at 1e-4, scaled to 127, FP32 per-row scale) and "Attention
  paths" (main compressor rotate=False, index-key compressor rotate=True).
* "DeepSeek V4.1 Flash", the production cache ABI (window KV MXFP8 E4M3 with
  E8M0 group-of-32 scales, compressed KV packed E2M1 with E4M3 group-of-16
  scales, index keys packed E2M1 with E8M0 group-of-32 scales; quantised on
  publication, dequantised on reads).  The rounding rules of the two FP4
  publications are readings (the pages give only the formats).

Readings taken where the pages are silent: ReLU per index head; the
index-key scale applied after the head sum; the gate input x of the
compressor is a separate [rows, Dx] operand (the workloads pass the raw KV
rows); the sink is already a logit; lse includes the sink; RMSNorm
optional; RoPE uses the last ``rope_dim`` dims; the overlapping ratio-4
compressor ("Hyper-Parallel ... DeepSeek V4 CP", "6.1 ratio4 CSA:
compressor halo") pools groups g - 1 and g into entry g, token q's logit
taking ape[q % ratio].

Parity pins live in ``tests/test_oracle_pins.py``.  Functions without an
independent pin: none (every function below has at least one).
"""

from __future__ import annotations

import numpy as np

BLOCK = 128  # rows per page

# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------


def bf16_round(x):
    """Round float64 values to the nearest BF16 value, ties to even.

    BF16 keeps 8 significant bits.  Written from the definition: x = m * 2**e
    with m in [0.5, 1); keep round-half-even(m * 2**8) / 2**8.  Normal range
    only (the workloads never approach BF16's overflow or subnormal range).
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def quantize_int8(y):
    """Per-row INT8 quantisation on write ("DeepSeek V4-Flash, MTP point",
    "What is quantized"): the row's amax, floored at 1e-4, is scaled to 127.

    Returns (codes int8, scale float64) with scale = max(amax, 1e-4) / 127 and
    code = clamp(round-half-even(y / scale), -127, 127).
    """
    y = np.asarray(y, dtype=np.float64)
    amax = np.max(np.abs(y)) if y.size else 0.0
    scale = max(amax, 1e-4) / 127.0
    codes = np.clip(np.rint(y / scale), -127, 127).astype(np.int8)
    return codes, scale


# --------------------------------------------------------------------------
# Low-bit cache formats ("DeepSeek V4.1 Flash", production cache ABI: window
# KV MXFP8 E4M3 with E8M0 group-of-32 scales; compressed KV packed MXFP4 E2M1
# with E4M3 group-of-16 scales; index keys packed E2M1 with E8M0 group-of-32
# scales; quantised on cache publication, dequantised on cache reads)
# --------------------------------------------------------------------------


def e2m1_decode(codes):
    """Value of 4-bit E2M1 codes (sign, 2 exponent bits with bias 1, 1
    mantissa bit; exponent 0 is subnormal): float64, same shape."""
    c = np.asarray(codes, dtype=np.int64)
    e, m = (c >> 1) & 3, c & 1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e - 1))
    return np.where(c & 8, -mag, mag)


def e4m3_decode(b):
    """Value of E4M3 bytes (sign, 4 exponent bits with bias 7, 3 mantissa
    bits; exponent 0 is subnormal; no infinities, S.1111.111 is NaN)."""
    b = np.asarray(b, dtype=np.int64)
    e, m = (b >> 3) & 15, b & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((b & 0x7F) == 0x7F, np.nan, mag)
    return np.where(b & 0x80, -mag, mag)


def e8m0_decode(b):
    """Value of E8M0 scale bytes: 2^(b - 127); 255 is NaN."""
    b = np.asarray(b, dtype=np.int64)
    return np.where(b == 255, np.nan, np.ldexp(1.0, b - 127))


def round_e2m1(x):
    """E2M1 code of the representable value nearest to each x (ties: the
    code with mantissa bit 0), magnitudes above 6 saturating to 6; the sign
    bit is set for x < 0 (also when the magnitude rounds to 0)."""
    x = np.asarray(x, dtype=np.float64)
    grid = e2m1_decode(np.arange(8))                      # the 8 magnitudes
    mag = _nearest_even(np.minimum(np.abs(x), 6.0), grid)
    return (mag | np.where(x < 0, 8, 0)).astype(np.uint8)


def _nearest_even(x, grid):
    """Index of the grid value nearest to each x; of two equally near ones
    (always neighbours) the even index."""
    d = np.abs(x[..., None] - grid)
    near = d == d.min(axis=-1, keepdims=True)
    return np.argmax(near * (2 - (np.arange(len(grid)) & 1)), axis=-1)


def round_e4m3(x):
    """E4M3 byte of the representable value nearest to each x >= 0 (ties:
    the even byte, i.e. mantissa ending in 0), saturating at 448."""
    x = np.asarray(x, dtype=np.float64)
    assert np.all(x >= 0)
    grid = e4m3_decode(np.arange(127))                    # 0 .. 448, ascending
    return _nearest_even(np.minimum(x, 448.0), grid).astype(np.uint8)


def pack_nibbles(codes):
    """Two E2M1 codes per byte: element 2i in the low nibble, 2i+1 in the high."""
    c = np.asarray(codes, dtype=np.uint8).reshape(-1, 2)
    return (c[:, 0] | (c[:, 1] << 4)).astype(np.uint8)


def unpack_nibbles(packed):
    p = np.asarray(packed, dtype=np.uint8).reshape(-1)
    return np.stack([p & 15, p >> 4], axis=-1).reshape(-1)


def _e8m0_exponent(amax):
    """Smallest e with 6 * 2^e >= amax, clamped to [-127, 127] (amax = 0:
    -127): with amax = M * 2^K, M in [1, 2), e = K - 2 + (M > 1.5)."""
    if amax == 0.0:
        return -127
    m, k = np.frexp(amax)  # amax = m * 2^k, m in [0.5, 1)
    e = (k - 1) - 2 + (1 if 2.0 * m > 1.5 else 0)
    return int(min(127, max(-127, e)))


def quantize_fp4_e8m0(y, group=32):
    """Index-key publication as packed E2M1 with one E8M0 scale per 32 dims.
    Reading (the pages give the format, not the rounding rule): a group's
    scale is the smallest power of two 2^e with 6 * 2^e >= its amax, so no
    element clips; codes are the nearest E2M1 of y / 2^e, the quotient taken
    in FP32 as the device takes it.  Returns (packed uint8 [n/2], scale
    bytes uint8 [n/group])."""
    y = np.asarray(y, dtype=np.float64).astype(np.float32)
    codes, sbytes = [], []
    for grp in y.reshape(-1, group):
        e = _e8m0_exponent(float(np.max(np.abs(grp))))
        q = grp / np.float32(np.ldexp(1.0, e))           # FP32 quotient
        codes.append(round_e2m1(q))
        sbytes.append(e + 127)
    return pack_nibbles(np.concatenate(codes)), np.array(sbytes, dtype=np.uint8)


def quantize_fp4_e4m3(y, group=16):
    """Compressed-KV publication as packed E2M1 with one E4M3 scale per 16
    channels.  Reading: the scale is the E4M3 value nearest to amax / 6 (so
    the largest element lands near the top code), codes the nearest E2M1 of
    y / scale (saturating at 6); both quotients taken in FP32 as the device
    takes them; a scale that rounds to 0 gives zero codes."""
    y = np.asarray(y, dtype=np.float64).astype(np.float32)
    codes, sbytes = [], []
    for grp in y.reshape(-1, group):
        amax = np.float32(np.max(np.abs(grp)))
        sb = int(round_e4m3(float(amax / np.float32(6.0))))
        s = np.float32(e4m3_decode(sb))
        codes.append(round_e2m1(grp / s) if s > 0 else np.zeros(group, np.uint8))
        sbytes.append(sb)
    return pack_nibbles(np.concatenate(codes)), np.array(sbytes, dtype=np.uint8)


def _e8m0_exponent_for(amax, top):
    """Smallest e with top * 2^e >= amax, clamped to [-127, 127] (amax = 0:
    -127), for a top code of the form 1.f * 2^t."""
    if amax == 0.0:
        return -127
    e = int(np.ceil(np.log2(amax / top)))
    # exact correction of the logarithm's rounding near powers of two
    while top * np.ldexp(1.0, e - 1) >= amax:
        e -= 1
    while top * np.ldexp(1.0, e) < amax:
        e += 1
    return int(min(127, max(-127, e)))


def quantize_mxfp8(y, group=32):
    """Index-key publication in the FP8 index plane.  Reading (the pages name
    an FP8 index plane but give no layout; this takes the MXFP8 layout they
    give for the window KV): E4M3 codes with one E8M0 scale per 32 dims; a
    group's scale is the smallest power of two 2^e with 448 * 2^e >= its
    amax (no element clips), codes the nearest E4M3 of y / 2^e (ties to the
    even code), the quotient taken in FP32.  Returns (codes uint8 [n], scale
    bytes uint8 [n/group])."""
    y = np.asarray(y, dtype=np.float64).astype(np.float32)
    codes, sbytes = [], []
    for grp in y.reshape(-1, group):
        e = _e8m0_exponent_for(float(np.max(np.abs(grp))), 448.0)
        q = (grp / np.float32(np.ldexp(1.0, e))).astype(np.float64)
        mag = round_e4m3(np.abs(q))
        codes.append((mag | np.where(q < 0, 0x80, 0)).astype(np.uint8))
        sbytes.append(e + 127)
    return np.concatenate(codes), np.array(sbytes, dtype=np.uint8)


def dequant_fp4(packed, sbytes, group, scale_fmt):
    """Values of one packed E2M1 row with its scale bytes (``scale_fmt``
    "e8m0" or "e4m3")."""
    v = e2m1_decode(unpack_nibbles(packed))
    dec = e8m0_decode if scale_fmt == "e8m0" else e4m3_decode
    return v * np.repeat(dec(np.asarray(sbytes)), group)


def dequant_mxfp8(codes, sbytes, group=32):
    """Values of one MXFP8 row: E4M3 bytes times their group's E8M0 scale."""
    return e4m3_decode(codes) * np.repeat(e8m0_decode(np.asarray(sbytes)), group)


class LowBitPool:
    """A paged cache pool held in a low-bit format: ``codes`` uint8 [pages,
    128, bytes per row] and ``scales`` uint8 [pages, 128, groups per row];
    ``fmt`` is "fp4_e4m3" (packed E2M1, E4M3 per 16: compressed KV),
    "fp4_e8m0" (packed E2M1, E8M0 per 32: index keys) or "mxfp8" (E4M3, E8M0
    per 32: window KV)."""

    def __init__(self, codes, scales, fmt):
        assert fmt in ("fp4_e4m3", "fp4_e8m0", "mxfp8")
        self.codes, self.scales, self.fmt = codes, scales, fmt

    def dequant_row(self, codes, sbytes):
        if self.fmt == "mxfp8":
            return dequant_mxfp8(codes, sbytes)
        if self.fmt == "fp4_e4m3":
            return dequant_fp4(codes, sbytes, 16, "e4m3")
        return dequant_fp4(codes, sbytes, 32, "e8m0")

    def dequant_rows(self, codes, sbytes):
        """``dequant_row`` of every row of codes [n, bytes] / sbytes [n, groups]."""
        codes = np.asarray(codes, dtype=np.int64)
        sbytes = np.asarray(sbytes, dtype=np.int64)
        if self.fmt == "mxfp8":
            vals, scl, group = e4m3_decode(codes), e8m0_decode(sbytes), 32
        else:
            nib = np.stack([codes & 15, codes >> 4], axis=-1).reshape(len(codes),
                                                                      2 * codes.shape[1])
            vals = e2m1_decode(nib)
            if self.fmt == "fp4_e4m3":
                scl, group = e4m3_decode(sbytes), 16
            else:
                scl, group = e8m0_decode(sbytes), 32
        return vals * np.repeat(scl, group, axis=1)


# --------------------------------------------------------------------------
# RoPE (DeepSeek V4.1 Flash, "Serving-owned full RoPE tables")
# --------------------------------------------------------------------------


def rope_rotate(vec, pos, cos_tab, sin_tab, rope_dim=64, inverse=False):
    """Rotate the last ``rope_dim`` entries of ``vec`` (shape [..., D]) at
    position ``pos`` by adjacent pairs (x[2i], x[2i+1]) using table row
    ``pos``: (a, b) -> (a*c - b*s, a*s + b*c).  A negative position, or one
    at or beyond the table capacity, leaves the vector unrotated (capacity
    overflow is an error the device reports; the oracle mirrors its identity
    fallback).  ``inverse`` rotates by the opposite angle.
    """
    v = as_f64(vec).copy()
    if pos < 0 or pos >= cos_tab.shape[0]:
        return v
    c = as_f64(cos_tab[pos])
    s = as_f64(sin_tab[pos])
    if inverse:
        s = -s
    D = v.shape[-1]
    a = v[..., D - rope_dim::2].copy()
    b = v[..., D - rope_dim + 1::2].copy()
    v[..., D - rope_dim::2] = a * c - b * s
    v[..., D - rope_dim + 1::2] = a * s + b * c
    return v


# --------------------------------------------------------------------------
# visibility and paging
# --------------------------------------------------------------------------


def visible_count(p, ratio, n_cmp):
    """Compressed slot c is visible to query position p iff c < (p + 1) // ratio
    ("Hyper-Parallel ... DeepSeek V4 CP", "10.3 Causal mask"), and only
    published slots exist (c < n_cmp)."""
    if p < 0:
        return 0
    return max(0, min(int(n_cmp), (int(p) + 1) // int(ratio)))


def window_positions(p, window=128):
    """Raw window of a query at position p: [max(0, p - window + 1), p],
    self included (ori_win_left = window - 1, ori_win_right = 0;
    "Hyper-Parallel ... DeepSeek V4 CP", "7. Window KV Halo")."""
    if p < 0:
        return []
    return list(range(max(0, p - window + 1), p + 1))


def as_f64(a):
    """float64 numpy copy of a numpy array or a (CPU) torch tensor of any dtype."""
    if hasattr(a, "detach"):
        import torch
        return a.detach().to(torch.float64).cpu().numpy()
    return np.asarray(a, dtype=np.float64)


def cache_rows(pool, table_row, logical):
    """``page_rows`` of a cache pool in any format: a ``LowBitPool`` is
    dequantised row by row (cache reads dequantise), anything else is read
    as it is."""
    if not isinstance(pool, LowBitPool):
        return page_rows(pool, table_row, logical)
    logical = list(logical)
    codes = page_rows(pool.codes, table_row, logical).astype(np.int64)
    scales = page_rows(pool.scales, table_row, logical).astype(np.int64)
    return pool.dequant_rows(codes, scales)


def page_rows(pool, table_row, logical):
    """Rows ``logical`` (iterable of request-local positions) of a paged pool
    [pages, 128, ...] through one request's block table row, as float64."""
    logical = np.asarray(list(logical), dtype=np.int64)
    phys = np.asarray(table_row, dtype=np.int64)[logical // BLOCK]
    assert np.all(phys >= 0), "read through an unmapped page"
    if hasattr(pool, "detach"):
        import torch
        return as_f64(pool[torch.from_numpy(phys), torch.from_numpy(logical % BLOCK)])
    return np.asarray(pool[phys, logical % BLOCK], dtype=np.float64)


# --------------------------------------------------------------------------
# a1: gated compressor
# --------------------------------------------------------------------------


def compress(x, kv, w_gate, ape, ratio, positions, row_req, gamma=None, rms_eps=1e-6,
             rotate=False, rope_cos=None, rope_sin=None, rope_dim=64, out="bf16", overlap=False,
             trace=None):
    """Gated compression of every complete group of ``ratio`` rows.

    ``overlap`` (the ratio-4 overlapping compressor, "Hyper-Parallel ...
    DeepSeek V4 CP", "6.1 ratio4 CSA: compressor halo": a group needs the
    ratio tokens before it, a shard's first slot is invalid; reading: entry
    g pools the tokens of group g - 1 and group g, those at positions >= 0,
    each token's logit taking ape[position % ratio]) widens every group's
    window to 2 * ratio tokens.

    A group g of request b is the positions g*r .. g*r + r - 1; it is complete
    in this chunk when rows t-r+1 .. t all belong to b at those consecutive
    positions, with p_t % r == r - 1.  Per channel d (512-channel KV plus a
    512-channel gate score per token: "DeepSeek V4.1 Flash", "Compressor state
    ownership", the recurrent-state row layout):

        logit[j, d] = (x_j @ w_gate)[d] + ape[j, d]
        w[:, d]     = softmax over j of logit[:, d]
        y[d]        = sum_j w[j, d] * kv_j[d]

    then y is rounded to BF16 ("BF16 rounding before RMSNorm"), optionally
    RMS-normalised with ``gamma`` (rounded to BF16 again), optionally rotated
    at the group start position g*r ("compression-group start positions";
    rotate=True for the index-key compressor, "DeepSeek V4-Flash, MTP point",
    "Attention paths"), and published as BF16 (``out="bf16"``), as INT8
    codes with an FP32 per-row scale (``out="int8"``), or in a low-bit cache
    format (``out="fp4_e4m3"``: packed E2M1 with E4M3 scales per 16;
    ``out="fp4_e8m0"``: packed E2M1 with E8M0 scales per 32; ``out="mxfp8"``:
    E4M3 with E8M0 scales per 32; "DeepSeek V4.1 Flash", production cache ABI
    and the FP8 index plane, quantised on publication).

    Returns a list of (request, g, values) for bf16, (request, g, codes,
    scale) for int8, or (request, g, packed codes, scale bytes) for the
    low-bit formats, in row order.

    ``trace`` (a list, or None) receives one record per published group with
    the intermediate values a comparison needs to tell a rounding tie from an
    error (see ``_publish_group``); the arithmetic is the same either way.
    """
    x, kv, w_gate, ape = as_f64(x), as_f64(kv), as_f64(w_gate), as_f64(ape)
    positions = as_f64(positions).astype(np.int64)
    row_req = as_f64(row_req).astype(np.int64)
    r = int(ratio)
    results = []
    for t in range(len(positions)):
        b, p = int(row_req[t]), int(positions[t])
        if b < 0 or p < 0 or p % r != r - 1:
            continue
        n = min(p + 1, 2 * r) if overlap else r  # the group's window of tokens
        if t < n - 1:
            continue
        rows = [t - n + 1 + j for j in range(n)]
        if any(int(row_req[s]) != b or int(positions[s]) != p - n + 1 + j
               for j, s in enumerate(rows)):
            continue
        pos = np.array([p - n + 1 + j for j in range(n)])
        logits = x[rows] @ w_gate + ape[pos % r]  # [n, D]
        mag = None
        if trace is not None:  # sqrt(sum_i (x_i w_id)^2 + ape_d^2) per token and channel
            mag = np.sqrt((x[rows] ** 2) @ (w_gate ** 2) + ape[pos % r] ** 2)
        results.append(_publish_group(b, p // r, r, logits, kv[rows], gamma, rms_eps, rotate,
                                      rope_cos, rope_sin, rope_dim, out, trace, mag))
    return results


def _publish_group(b, g, r, logits, kvs, gamma, rms_eps, rotate, rope_cos, rope_sin, rope_dim,
                   out, trace=None, mag=None):
    """Pool one group from its r gate scores and kv rows ([r, D] each) and
    publish it: the per-channel softmax over the r tokens, BF16 rounding,
    optional RMSNorm, optional rotation at the group start, BF16 or INT8.

    With ``trace`` (a list) a record is appended: b, g, the logits and kv
    rows, ``mag`` (per token and channel, the root sum of squares of the
    terms of its logit),
    ``pooled`` (the pooled value before its BF16 rounding), ``ybf16`` (after
    it), ``normed`` (the RMSNorm output before its rounding, or None) and
    ``y`` (the value handed to the publication format)."""
    mx = logits.max(axis=0, keepdims=True)
    e = np.exp(logits - mx)
    w = e / e.sum(axis=0, keepdims=True)
    y = (w * kvs).sum(axis=0)
    pooled = y
    y = bf16_round(y)
    ybf16, normed = y, None
    if gamma is not None:
        g_ = as_f64(gamma)
        normed = y / np.sqrt(np.mean(y * y) + rms_eps) * g_
        y = bf16_round(normed)
    if rotate:
        y = rope_rotate(y, g * r, rope_cos, rope_sin, rope_dim)
    if trace is not None:
        trace.append(dict(b=b, g=g, logits=logits, kvs=kvs, mag=mag, pooled=pooled, y=y,
                          ybf16=ybf16, normed=normed, rotated=bool(rotate)))
    if out == "bf16":
        return (b, g, bf16_round(y))
    if out == "fp4_e4m3":
        return (b, g) + quantize_fp4_e4m3(y)
    if out == "fp4_e8m0":
        return (b, g) + quantize_fp4_e8m0(y)
    if out == "mxfp8":
        return (b, g) + quantize_mxfp8(y)
    codes, scale = quantize_int8(y)
    return (b, g, codes, scale)


def compress_stateful(x, kv, w_gate, ape, ratio, positions, row_req, state, state_table,
                      gamma=None, rms_eps=1e-6, rotate=False, rope_cos=None, rope_sin=None,
                      rope_dim=64, out="bf16", overlap=False, trace=None):
    """One chunk of the compressor with its recurrent state ring ("DeepSeek
    V4.1 Flash", "Compressor state ownership").

    ``state`` (float64 [n_blocks, cap, 2 D], updated in place) is the ring:
    slot p % cap of request b's block ``state_table[b]`` holds the kv row of
    position p followed by its gate score x_p @ w_gate + ape[p % r].  A token
    that closes a group (p % r == r - 1) pools its r tokens as compress()
    does, taking each predecessor from the chunk when it is a preceding row of
    the same request and otherwise (a position before the chunk start) from
    the ring.  Every read happens before any write; then the last
    min(chunk length, cap) tokens of each request's chunk write their slots.
    ``state_table[b] < 0`` disables request b (nothing published or written);
    negative positions neither publish nor write.  Returns the published
    groups as compress() does; ``overlap`` widens the windows as there (the
    ring then needs at least 2 * ratio slots); ``trace`` as in compress()
    (a token taken from the ring has |its stored score| as its ``mag``).
    """
    x, kv, w_gate, ape = as_f64(x), as_f64(kv), as_f64(w_gate), as_f64(ape)
    positions = as_f64(positions).astype(np.int64)
    row_req = as_f64(row_req).astype(np.int64)
    table = as_f64(state_table).astype(np.int64)
    assert not overlap or state.shape[1] >= 2 * int(ratio)
    r, D, cap = int(ratio), kv.shape[1], state.shape[1]
    T = len(positions)

    def live(t):
        b, p = int(row_req[t]), int(positions[t])
        return b >= 0 and p >= 0 and int(table[b]) >= 0

    score = {t: x[t] @ w_gate + ape[int(positions[t]) % r] for t in range(T) if live(t)}
    results = []
    for t in range(T):
        if not live(t):
            continue
        b, p = int(row_req[t]), int(positions[t])
        if p % r != r - 1:
            continue
        blk = int(table[b])
        logits, kvs, mags = [], [], []
        n = min(p + 1, 2 * r) if overlap else r
        for j in range(n - 1, -1, -1):  # positions p - j, oldest first
            s_ = t - j
            if s_ >= 0 and int(row_req[s_]) == b and int(positions[s_]) == p - j:
                logits.append(score[s_])
                kvs.append(kv[s_])
                if trace is not None:
                    mags.append(np.sqrt((x[s_] ** 2) @ (w_gate ** 2) + ape[(p - j) % r] ** 2))
            else:
                slot = state[blk, (p - j) % cap]
                kvs.append(slot[:D].copy())
                logits.append(slot[D:].copy())
                if trace is not None:
                    mags.append(np.abs(slot[D:]))
        results.append(_publish_group(b, p // r, r, np.stack(logits), np.stack(kvs), gamma,
                                      rms_eps, rotate, rope_cos, rope_sin, rope_dim, out, trace,
                                      np.stack(mags) if trace is not None else None))
    # writes: the last min(chunk length, cap) rows of each request's chunk
    last_row = {}
    for t in range(T):
        if live(t):
            last_row[int(row_req[t])] = t
    for t in range(T):
        if not live(t):
            continue
        b, p = int(row_req[t]), int(positions[t])
        if t > last_row[b] - cap:
            state[int(table[b]), p % cap, :D] = kv[t]
            state[int(table[b]), p % cap, D:] = score[t]
    return results


# --------------------------------------------------------------------------
# a3: lightning-indexer scores
# --------------------------------------------------------------------------


def index_scores(q_idx_row, w_row, p, n_cmp_b, ratio, idx_pool, idx_scale_pool, table_row,
                 relu=True, rope_cos=None, rope_sin=None, rope_dim=64):
    """Scores of one query row against every visible compressed entry:

        score[c] = scale_c * sum_h w[h] * ReLU(q_h . k_c),   c < visible_count

    with q_h the row's index query of head h rotated at the row position p
    (when tables are given) and k_c the INT8 index key of entry c
    ("Hyper-Parallel ... DeepSeek V4 CP", "10. ratio=4 Global Top-k"; INT8
    keys with an FP32 per-row scale: "DeepSeek V4-Flash, MTP point", "What is
    quantized").  Since scale_c > 0, ReLU(scale * x) = scale * ReLU(x), so the
    scale is applied after the head sum.  With ``idx_pool`` a ``LowBitPool``
    (packed E2M1 keys with E8M0 group scales, "DeepSeek V4.1 Flash",
    production cache ABI) k_c is the dequantised key and scale_c = 1
    (``idx_scale_pool`` unused).  Returns float64 [visible].
    """
    nv = visible_count(p, ratio, n_cmp_b)
    q = as_f64(q_idx_row)  # [H, Di]
    if rope_cos is not None:
        q = rope_rotate(q, p, rope_cos, rope_sin, rope_dim)
    keys = cache_rows(idx_pool, table_row, range(nv))  # [nv, Di]
    scales = (np.ones(nv) if isinstance(idx_pool, LowBitPool) else
              page_rows(idx_scale_pool, table_row, range(nv)))
    dots = keys @ q.T  # [nv, H]
    if relu:
        dots = np.maximum(dots, 0.0)
    return scales * (dots @ as_f64(w_row))


# --------------------------------------------------------------------------
# a4: top-k
# --------------------------------------------------------------------------


def topk_select(scores, k):
    """The k best entries by (score descending, index ascending), emitted as
    logical positions in ascending order with trailing -1 padding
    ("DeepSeek V4.1 Flash": logical-position ordering and trailing -1
    padding in the Top-K acceptance rule; indexer workspaces padded with -1).
    """
    scores = np.asarray(scores, dtype=np.float64)
    order = np.argsort(-scores, kind="stable")  # stable: equal scores keep ascending index
    chosen = np.sort(order[:k])
    out = np.full(k, -1, dtype=np.int64)
    out[:len(chosen)] = chosen
    return out


def select_blocks(scores, n_blocks, block=8):
    """Level one of the hierarchical indexer ("DeepSeek V4.1 Flash": the
    first selection takes 2,048 blocks of eight compressed positions, which
    later reindex layers search).  A block's score is the largest score of
    its visible positions (a reading: the page does not say how blocks are
    ranked); the n_blocks best blocks by (score descending, block ascending)
    are emitted ascending with trailing -1 padding, as topk_select does."""
    scores = np.asarray(scores, dtype=np.float64)
    nb = (len(scores) + block - 1) // block
    best = np.array([scores[i * block:(i + 1) * block].max() for i in range(nb)])
    return topk_select(best, n_blocks)


def topk_in_blocks(scores, blocks, k, block=8):
    """Level two (reindex): the k best visible positions inside the given
    candidate blocks (-1 entries ignored), by (score descending, position
    ascending), emitted ascending with trailing -1 padding."""
    scores = np.asarray(scores, dtype=np.float64)
    V = len(scores)
    pos = sorted({b * block + i for b in np.asarray(blocks).tolist() if b >= 0
                  for i in range(block) if b * block + i < V})
    pos = np.array(pos, dtype=np.int64)
    sel = topk_select(scores[pos], k) if len(pos) else np.full(k, -1, dtype=np.int64)
    return np.where(sel >= 0, pos[np.maximum(sel, 0)] if len(pos) else -1, -1)


# --------------------------------------------------------------------------
# a5 / a6: shared-KV sparse attention with sink
# --------------------------------------------------------------------------


def sparse_attention(q_row, p, topk_row, kv_pool, kv_table_row, cmp_pool, cmp_table_row,
                     sink, scale, window=128, rope_cos=None, rope_sin=None, rope_dim=64,
                     inv_rope_out=False):
    """One query row of shared-KV sparse attention
    ("Hyper-Parallel ... DeepSeek V4 CP", "二阶段 CP 总体算法", Stage-2 with
    cmp_sparse_indices, sinks, softmax_scale and ori_win_left = 127; the
    candidate list is the selected compressed entries plus the raw window,
    "9.1 Small-op fallback 路径": kv_full = [window kv, compressed kv]).

    Each candidate row is both key and value.  Per head h:
        l_i  = scale * q_h . k_i      (q rotated at p when tables are given)
        o_h  = sum_i e^{l_i} k_i / (sum_i e^{l_i} + e^{sink_h})
        lse_h = log(sum_i e^{l_i} + e^{sink_h})
    A sink of None means -inf (plain softmax).  Two passes: max, then sums.
    Either pool may be a ``LowBitPool`` (rows dequantised as they are read).
    Returns (out [H, D] float64, lse [H] float64).
    """
    q = as_f64(q_row)
    H, D = q.shape
    if rope_cos is not None:
        q = rope_rotate(q, p, rope_cos, rope_sin, rope_dim)
    sel = [int(c) for c in np.asarray(topk_row).ravel() if int(c) >= 0]
    parts = []
    if sel:
        parts.append(cache_rows(cmp_pool, cmp_table_row, sel))
    win = window_positions(p, window)
    if win:
        parts.append(cache_rows(kv_pool, kv_table_row, win))
    K = np.concatenate(parts, axis=0) if parts else np.zeros((0, D))
    logits = scale * (q @ K.T)  # [H, n]
    snk = np.full(H, -np.inf) if sink is None else as_f64(sink)
    m = np.maximum(logits.max(axis=1) if K.shape[0] else np.full(H, -np.inf), snk)
    out = np.zeros((H, D))
    lse = np.full(H, -np.inf)
    for h in range(H):
        if not np.isfinite(m[h]):
            continue
        e = np.exp(logits[h] - m[h])
        s = e.sum() + np.exp(snk[h] - m[h])
        out[h] = (e @ K) / s
        lse[h] = m[h] + np.log(s)
    if inv_rope_out and rope_cos is not None:
        out = rope_rotate(out, p, rope_cos, rope_sin, rope_dim, inverse=True)
    return out, lse
