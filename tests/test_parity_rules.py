"""The comparison rules of ``parity.py`` on the CPU: a code that differs at a
rounding tie is accepted, a code that differs anywhere else is caught.
Mistakes are planted on the oracle's own output (no GPU involved)."""

import numpy as np
import pytest
import torch

import oracle as O
from parity import bf16_tie_distance, check_int8_tied, check_lowbit_tied, tie_flags


def _groups(out, d=128, dx=128, n=64, rotate=True, seed=3):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.standard_normal((n, dx)).astype(np.float32)).bfloat16()
    w = torch.from_numpy((rng.standard_normal((dx, d)) / np.sqrt(dx)).astype(np.float32)).bfloat16()
    ape = torch.from_numpy(rng.standard_normal((4, d)).astype(np.float32))
    from workloads import rope_tables
    cos, sin = rope_tables(4096)
    trace = []
    res = O.compress(x, x if d == dx else torch.from_numpy(
        rng.standard_normal((n, d)).astype(np.float32)).bfloat16(), w, ape, 4,
        np.arange(n), np.zeros(n, int), rotate=rotate, rope_cos=cos, rope_sin=sin, out=out,
        trace=trace)
    return res, trace, dx


def test_bf16_tie_distance_values():
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 2 ** -9, 0.75, -(3.0 + 3 * 2 ** -7)])
    assert np.allclose(bf16_tie_distance(v), [2 ** -9, 0.0, 2 ** -9, 2 ** -9, 0.0])


def test_int8_rule_accepts_the_oracle_and_catches_a_planted_shift():
    res, trace, dx = _groups("int8")
    for (_, _, codes, scale), rec in zip(res, trace):
        assert check_int8_tied(codes, np.float32(scale), codes, np.float32(scale), rec, dx) == 0
    # +1 on a code far from any tie must fail
    (_, _, codes, scale), rec = res[0], trace[0]
    q = np.abs(rec["y"] / scale)
    far = np.nonzero((np.abs(q - np.floor(q) - 0.5) > 0.1) & ~tie_flags(rec, dx) &
                     (np.abs(codes.astype(int)) < 127))[0]
    assert len(far)
    bad = codes.astype(np.int64).copy()
    bad[far[0]] += 1
    with pytest.raises(AssertionError):
        check_int8_tied(bad, np.float32(scale), codes, np.float32(scale), rec, dx)


def test_int8_rule_accepts_a_flip_at_a_half_tie():
    res, trace, dx = _groups("int8")
    (_, _, codes, scale), rec = res[1], trace[1]
    # make one quotient sit on a .5 tie: the code may then round either way
    rec = dict(rec)
    y = rec["y"].copy()
    i = int(np.argsort(np.abs(y))[len(y) // 2])
    k = np.floor(abs(y[i]) / scale)
    y[i] = np.sign(y[i]) * (k + 0.5) * scale
    rec["y"] = y
    ref = codes.astype(np.int64).copy()
    ref[i] = int(np.sign(y[i]) * k)
    got = ref.copy()
    got[i] = int(np.sign(y[i]) * (k + 1))
    assert check_int8_tied(got, np.float32(scale), ref, np.float32(scale), rec, dx) == 1


def test_fp4_rule_accepts_the_oracle_and_catches_a_planted_step():
    res, trace, dx = _groups("fp4_e8m0")
    for (_, _, codes, sb), rec in zip(res, trace):
        assert check_lowbit_tied(codes, sb, codes, sb, rec, dx, 32, "e8m0") == (0, 0)
    (_, _, codes, sb), rec = res[2], trace[2]
    c = O.unpack_nibbles(codes).astype(np.int64)
    ok = ~tie_flags(rec, dx)
    i = int(np.nonzero(ok & ((c & 7) > 0) & ((c & 7) < 7))[0][0])
    c2 = c.copy()
    c2[i] = (c[i] & 8) | ((c[i] & 7) + 1)
    y32 = rec["y"].astype(np.float32).astype(np.float64)
    q = abs(y32[i]) / 2.0 ** (int(sb[i // 32]) - 127)
    if np.min(np.abs(q - np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]))) > 1e-2:
        with pytest.raises(AssertionError):
            check_lowbit_tied(O.pack_nibbles(c2.astype(np.uint8)), sb, codes, sb, rec, dx, 32,
                              "e8m0")


def test_mxfp8_rule_catches_a_sign_flip():
    res, trace, dx = _groups("mxfp8")
    (_, _, codes, sb), rec = res[0], trace[0]
    c = codes.astype(np.int64).copy()
    i = int(np.nonzero((c & 0x7F) > 8)[0][0])
    c[i] ^= 0x80
    with pytest.raises(AssertionError):
        check_lowbit_tied(c.astype(np.uint8), sb, codes, sb, rec, dx, 32, "mxfp8")
