"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks the oracle against something it does not compute itself:
a worked example printed on the pages (``tests/golden``), a hand-computed
value, a closed form, a library routine (torch's BF16 cast, numpy complex
multiplication, scipy's softmax/logsumexp, numpy's lexsort), or an
invariant that a dropped term, a wrong sign or index, or a transposed
operand would break.
"""

import numpy as np
import pytest
import torch
from scipy.special import expit, logsumexp, softmax

import oracle as O
from golden.load import constants, rows
from workloads import BLOCK, rope_tables

COS, SIN = rope_tables(4096, 64, 10000.0)


def _cplx_rotate(v, pos, rope_dim=64):
    """Rotation of adjacent pairs written as complex multiplication by e^{i*angle}."""
    v = np.asarray(v, dtype=np.float64).copy()
    D = v.shape[-1]
    z = v[..., D - rope_dim::2] + 1j * v[..., D - rope_dim + 1::2]
    rot = np.asarray(COS[pos], np.float64) + 1j * np.asarray(SIN[pos], np.float64)
    z = z * rot
    v[..., D - rope_dim::2] = z.real
    v[..., D - rope_dim + 1::2] = z.imag
    return v


# ---------------------------------------------------------------- formats


def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    # add exact ties (low 16 bits == 0x8000, normal range): must round half to even
    expo = rng.integers(100, 150, 2000, dtype=np.uint32) << np.uint32(23)
    mant = rng.integers(0, 128, 2000, dtype=np.uint32) << np.uint32(16)
    ties = (expo | mant | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties, -ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_round(x.astype(np.float64)), ref)


def test_int8_quant_constants_and_worked_example():
    c = constants("int8_quant_constants.txt")
    codes, s = O.quantize_int8(np.zeros(128))
    assert s == pytest.approx(c["amax_eps"] / c["scale_max"], rel=1e-15)
    assert np.all(codes == 0)
    # hand-computed: amax 1 -> scale 1/127; 0.5*127 = 63.5 -> 64 (half to even),
    # 0.25*127 = 31.75 -> 32, -1 -> -127
    codes, s = O.quantize_int8(np.array([0.5, -1.0, 0.25, 0.0]))
    assert s == pytest.approx(1.0 / 127.0, rel=1e-15)
    assert codes.tolist() == [64, -127, 32, 0]
    # 1.5/127 -> rounds to 2 (even), 2.5/127 -> 2 (even)
    codes, s = O.quantize_int8(np.array([1.0, 1.5 / 127, 2.5 / 127]))
    assert codes.tolist() == [127, 2, 2]


def test_int8_quant_error_bound_and_amax_code():
    rng = np.random.default_rng(3)
    for _ in range(50):
        y = rng.standard_normal(128) * rng.uniform(0.01, 10)
        codes, s = O.quantize_int8(y)
        assert np.max(np.abs(codes.astype(np.float64) * s - y)) <= s / 2 * (1 + 1e-12)
        i = np.argmax(np.abs(y))
        assert abs(int(codes[i])) == 127 and np.sign(codes[i]) == np.sign(y[i])


# ---------------------------------------------------------------- RoPE


def test_rope_identity_at_zero_and_negative_positions():
    rng = np.random.default_rng(0)
    v = rng.standard_normal((3, 512))
    assert np.array_equal(O.rope_rotate(v, 0, COS, SIN), v)
    assert np.array_equal(O.rope_rotate(v, -1, COS, SIN), v)
    assert np.array_equal(O.rope_rotate(v, -77, COS, SIN), v)
    # beyond capacity: identity (the device flags it)
    assert np.array_equal(O.rope_rotate(v, 4096, COS, SIN), v)


def test_rope_is_complex_multiplication_of_adjacent_pairs():
    rng = np.random.default_rng(1)
    for D in (512, 128):
        v = rng.standard_normal((5, D))
        for pos in (1, 7, 300, 4095):
            got = O.rope_rotate(v, pos, COS, SIN)
            assert np.allclose(got, _cplx_rotate(v, pos), rtol=0, atol=1e-12)
            assert np.array_equal(got[:, :D - 64], v[:, :D - 64])


def test_rope_relative_position_norm_and_inverse():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    base = O.rope_rotate(q, 40, COS, SIN) @ O.rope_rotate(k, 10, COS, SIN)
    for shift in (1, 100, 2000):
        other = O.rope_rotate(q, 40 + shift, COS, SIN) @ O.rope_rotate(k, 10 + shift, COS, SIN)
        assert other == pytest.approx(base, rel=1e-5, abs=1e-5)
    r = O.rope_rotate(q, 1234, COS, SIN)
    pair = lambda x: x[64::2] ** 2 + x[65::2] ** 2  # noqa: E731
    assert np.allclose(pair(r), pair(q), rtol=1e-6)
    back = O.rope_rotate(r, 1234, COS, SIN, inverse=True)
    assert np.allclose(back, q, atol=1e-6)


# ---------------------------------------------------------------- visibility / window


def test_causal_visibility_worked_example_and_brute_force():
    for p, r, vis in rows("causal_visibility.txt"):
        p, r = int(p), int(r)
        want = [int(c) for c in vis.split(",")]
        assert list(range(O.visible_count(p, r, 10**9))) == want
    # brute force: slot c pools positions c*r .. c*r+r-1; it is visible iff all
    # of them are at or before p
    for r in (1, 2, 4, 128):
        for p in range(0, 600, 7):
            brute = sum(1 for c in range(1000) if c * r + r - 1 <= p)
            assert O.visible_count(p, r, 10**9) == brute
            assert O.visible_count(p, r, 3) == min(3, brute)
    assert O.visible_count(-1, 2, 100) == 0


def test_window_worked_example():
    for p, w, vis in rows("window_example.txt"):
        assert O.window_positions(int(p), int(w)) == [int(x) for x in vis.split(",")]
    assert O.window_positions(0, 128) == [0]
    assert O.window_positions(300, 128) == list(range(173, 301))


# ---------------------------------------------------------------- compressor


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)


def _chunk(rng, n, D=64, Dx=64):
    kv = _bf16(rng.standard_normal((n, D)))
    x = _bf16(rng.standard_normal((n, Dx)))
    return x, kv


def test_compress_ratio1_is_identity():
    rng = np.random.default_rng(4)
    x, kv = _chunk(rng, 6)
    w = _bf16(rng.standard_normal((64, 64)))
    ape = rng.standard_normal((1, 64))
    res = O.compress(x, kv, w, ape, 1, np.arange(10, 16), np.zeros(6, int))
    assert [g for _, g, _ in res] == list(range(10, 16))
    for i, (_, _, y) in enumerate(res):
        assert np.array_equal(y, kv[i].double().numpy())


def test_compress_equal_logits_give_the_mean():
    rng = np.random.default_rng(5)
    x, kv = _chunk(rng, 8)
    w = torch.zeros((64, 64), dtype=torch.bfloat16)
    res = O.compress(x, kv, w, np.zeros((4, 64)), 4, np.arange(8), np.zeros(8, int))
    assert len(res) == 2
    for b, g, y in res:
        mean = kv[4 * g:4 * g + 4].double().numpy().mean(axis=0)
        # the only difference from the plain mean is the final BF16 rounding
        assert np.all(np.abs(y - mean) <= 2.0 ** -8 * np.abs(mean) * (1 + 1e-12))


def test_compress_ratio128_groups():
    """HCA's ratio 128 ("Hyper-Parallel ... DeepSeek V4 CP", "ratio=128":
    non-overlapping compression): equal logits pool each 128-token group to
    its mean, only complete groups publish, and a one-hot APE row picks that
    token of every group."""
    rng = np.random.default_rng(6)
    x, kv = _chunk(rng, 300, D=32, Dx=16)
    w = torch.zeros((16, 32), dtype=torch.bfloat16)
    res = O.compress(x, kv, w, np.zeros((128, 32)), 128, np.arange(300), np.zeros(300, int))
    assert [g for _, g, _ in res] == [0, 1]  # tokens 256..299 do not close a group
    for _, g, y in res:
        mean = kv[128 * g:128 * g + 128].double().numpy().mean(axis=0)
        assert np.all(np.abs(y - mean) <= 2.0 ** -8 * np.abs(mean) * (1 + 1e-12) + 1e-12)
    ape = np.zeros((128, 32))
    ape[77] = 80.0  # token 77 of each group dominates every channel's softmax
    for _, g, y in O.compress(x, kv, w, ape, 128, np.arange(300), np.zeros(300, int)):
        assert np.array_equal(y, kv[128 * g + 77].double().numpy())


def test_compress_one_hot_ape_selects_a_row():
    rng = np.random.default_rng(6)
    x, kv = _chunk(rng, 4)
    w = _bf16(rng.standard_normal((64, 64)) * 0.01)
    ape = np.zeros((4, 64))
    ape[2] = 1e4
    (_, _, y), = O.compress(x, kv, w, ape, 4, np.arange(4), np.zeros(4, int))
    assert np.array_equal(y, kv[2].double().numpy())


def test_compress_gate_orientation_is_x_times_w():
    # x_j0 has a single 1 at input channel k0; w_gate[k0, d0] is huge.
    # Output channel d0 must select row j0; every other channel is the mean.
    kv = _bf16(np.random.default_rng(8).standard_normal((4, 64)))
    x = torch.zeros((4, 64), dtype=torch.bfloat16)
    j0, k0, d0 = 1, 5, 40
    x[j0, k0] = 1.0
    w = torch.zeros((64, 64), dtype=torch.bfloat16)
    w[k0, d0] = 1e4
    (_, _, y), = O.compress(x, kv, w, np.zeros((4, 64)), 4, np.arange(4), np.zeros(4, int))
    kvd = kv.double().numpy()
    assert y[d0] == kvd[j0, d0]
    others = [d for d in range(64) if d != d0]
    assert np.allclose(y[others], kvd[:, others].mean(axis=0), rtol=2 ** -7, atol=1e-6)
    assert not np.isclose(y[k0], kvd[j0, k0]) or np.isclose(kvd[:, k0].mean(), kvd[j0, k0])


def test_compress_weights_sum_to_one_and_order_of_ape_rows():
    rng = np.random.default_rng(9)
    v = rng.standard_normal(64)
    kv = _bf16(np.tile(v, (4, 1)))
    x = _bf16(rng.standard_normal((4, 64)))
    w = _bf16(rng.standard_normal((64, 64)))
    ape = rng.standard_normal((4, 64)) * 3
    (_, _, y), = O.compress(x, kv, w, ape, 4, np.arange(4), np.zeros(4, int))
    assert np.array_equal(y, kv[0].double().numpy())  # any convex combination of equal rows
    # APE row j applies to the j-th token of the group (position % ratio == j)
    kv2 = _bf16(rng.standard_normal((4, 64)))
    for j in range(4):
        ape_hot = np.zeros((4, 64))
        ape_hot[j] = 1e4
        (_, _, yb), = O.compress(x, kv2, w, ape_hot, 4, np.arange(8, 12), np.zeros(4, int))
        assert np.array_equal(yb, kv2[j].double().numpy())


def test_compress_softmax_matches_scipy():
    rng = np.random.default_rng(10)
    x, kv = _chunk(rng, 4)
    w = _bf16(rng.standard_normal((64, 64)) / 8)
    ape = rng.standard_normal((4, 64))
    (_, _, y), = O.compress(x, kv, w, ape, 4, np.arange(4), np.zeros(4, int))
    logits = x.double().numpy() @ w.double().numpy() + ape
    ref = (softmax(logits, axis=0) * kv.double().numpy()).sum(axis=0)
    assert np.allclose(y, ref, rtol=2 ** -8, atol=1e-12)


def test_compress_only_complete_groups_and_requests():
    rng = np.random.default_rng(11)
    x, kv = _chunk(rng, 9)
    w = _bf16(rng.standard_normal((64, 64)))
    ape = rng.standard_normal((2, 64))
    # request 0: positions 5..8 (groups (6,7) complete; 5 and 8 are halves)
    # request 1: positions 0..2 (group (0,1)); one padding row
    pos = np.array([5, 6, 7, 8, 0, 1, 2, -1, 3])
    req = np.array([0, 0, 0, 0, 1, 1, 1, -1, 1])
    got = [(b, g) for b, g, _ in O.compress(x, kv, w, ape, 2, pos, req)]
    assert got == [(0, 3), (1, 0)]  # row 8 (pos 3) follows a padding row: incomplete


def test_compress_rotate_uses_group_start_and_int8_path():
    rng = np.random.default_rng(12)
    x, kv = _chunk(rng, 8, D=128, Dx=128)
    w = _bf16(rng.standard_normal((128, 128)) / 11)
    ape = rng.standard_normal((4, 128))
    pos = np.arange(100, 108)
    plain = O.compress(x, kv, w, ape, 4, pos, np.zeros(8, int))
    rot = O.compress(x, kv, w, ape, 4, pos, np.zeros(8, int), rotate=True, rope_cos=COS,
                     rope_sin=SIN)
    q8 = O.compress(x, kv, w, ape, 4, pos, np.zeros(8, int), rotate=True, rope_cos=COS,
                    rope_sin=SIN, out="int8")
    for (_, g, yp), (_, g2, yr), (_, g3, codes, s) in zip(plain, rot, q8):
        assert g == g2 == g3
        want = _cplx_rotate(yp, g * 4)
        assert np.allclose(yr, want, rtol=2 ** -8, atol=1e-6)
        assert np.max(np.abs(codes * s - want)) <= s / 2 + 1e-9


def _stateful_run(x, kv, w, ape, r, reqs, splits, cap=4, **kw):
    """Feed requests' token streams chunk by chunk (``splits``: per call, the
    number of tokens of each request), carrying one ring per request."""
    D = kv.shape[1]
    n_req = len(reqs)
    state = np.full((n_req + 2, cap, 2 * D), np.nan)  # blocks 1.. hold the requests
    table = np.arange(1, n_req + 1)
    done = [0] * n_req
    out = []
    for call in splits:
        rows, pos, req = [], [], []
        for b, n in enumerate(call):
            for i in range(n):
                rows.append(reqs[b][done[b] + i])
                pos.append(done[b] + i)
                req.append(b)
            done[b] += n
        if not rows:
            continue
        idx = np.array(rows)
        out += O.compress_stateful(x[idx], kv[idx], w, ape, r, np.array(pos), np.array(req),
                                   state, table, **kw)
    return out, state, table


@pytest.mark.parametrize("r,splits", [
    (2, [[1, 1]] * 9),                         # one token per call (decode)
    (2, [[3, 2], [1, 4], [5, 1], [2, 2]]),     # odd chunk starts: a pair closes across calls
    (4, [[1, 1]] * 11),
    (4, [[2, 3], [7, 1], [1, 6], [3, 2]]),     # chunks longer than the ring
    (4, [[6, 0], [0, 5], [5, 6]]),             # idle requests in some calls
])
def test_stateful_compress_equals_one_shot(r, splits):
    """Chunked calls with the state ring publish exactly the groups the
    one-shot compressor publishes over each request's whole stream."""
    rng = np.random.default_rng(40 + r)
    lens = [sum(c[b] for c in splits) for b in range(2)]
    n = sum(lens)
    x, kv = _chunk(rng, n, D=64, Dx=32)
    w = _bf16(rng.standard_normal((32, 64)) / 6)
    ape = rng.standard_normal((r, 64))
    reqs = [list(range(0, lens[0])), list(range(lens[0], n))]
    got, _, _ = _stateful_run(x, kv, w, ape, r, reqs, splits)
    want = []
    for b in range(2):
        idx = np.array(reqs[b])
        for _, g, y in O.compress(x[idx], kv[idx], w, ape, r, np.arange(len(idx)),
                                  np.zeros(len(idx), int)):
            want.append((b, g, y))
    assert sorted((b, g) for b, g, _ in got) == sorted((b, g) for b, g, _ in want)
    ref = {(b, g): y for b, g, y in want}
    for b, g, y in got:
        assert np.array_equal(y, ref[(b, g)]), (b, g)


def test_stateful_compress_int8_rotated_equals_one_shot():
    rng = np.random.default_rng(47)
    x, kv = _chunk(rng, 13, D=128, Dx=64)
    w = _bf16(rng.standard_normal((64, 128)) / 8)
    ape = rng.standard_normal((4, 128))
    kw = dict(rotate=True, rope_cos=COS, rope_sin=SIN, out="int8")
    got, _, _ = _stateful_run(x, kv, w, ape, 4, [list(range(13))], [[3], [1], [6], [3]], **kw)
    want = O.compress(x, kv, w, ape, 4, np.arange(13), np.zeros(13, int), **kw)
    assert [(g, c.tolist(), sc) for _, g, c, sc in got] == [(g, c.tolist(), sc) for _, g, c, sc in want]


# Overlapping ratio-4 compression ("Hyper-Parallel ... DeepSeek V4 CP",
# "6.1 ratio4 CSA: compressor halo": a group needs the ratio tokens before
# it; reading: entry g
# pools groups g - 1 and g, each token's logit taking ape[position % ratio]).


def test_overlap_equal_logits_give_the_two_group_mean():
    rng = np.random.default_rng(48)
    x, kv = _chunk(rng, 12)
    w = torch.zeros((64, 64), dtype=torch.bfloat16)
    res = O.compress(x, kv, w, np.zeros((4, 64)), 4, np.arange(12), np.zeros(12, int),
                     overlap=True)
    assert [g for _, g, _ in res] == [0, 1, 2]
    for _, g, y in res:
        lo = max(0, 4 * g - 4)  # entry 0 has no previous group
        mean = kv[lo:4 * g + 4].double().numpy().mean(axis=0)
        assert np.all(np.abs(y - mean) <= 2.0 ** -8 * np.abs(mean) * (1 + 1e-12))


def test_overlap_one_hot_ape_picks_that_token_of_both_groups():
    rng = np.random.default_rng(49)
    x, kv = _chunk(rng, 12)
    w = torch.zeros((64, 64), dtype=torch.bfloat16)
    ape = np.zeros((4, 64))
    ape[1] = 1e4  # positions 1, 5, 9: one in each group, equal logits
    res = O.compress(x, kv, w, ape, 4, np.arange(12), np.zeros(12, int), overlap=True)
    k = kv.double().numpy()
    (_, _, y0), (_, _, y1), (_, _, y2) = res
    assert np.array_equal(y0, k[1])
    for y, (a, b) in ((y1, (1, 5)), (y2, (5, 9))):
        two = _bf16(0.5 * (k[a] + k[b])).double().numpy()
        assert np.array_equal(y, two)


def test_overlap_odd_entries_are_the_double_ratio_groups():
    """Entry 2k + 1 of the overlapping ratio-r compressor pools positions
    2rk .. 2rk + 2r - 1, the k-th group of the plain ratio-2r compressor
    whose APE repeats the ratio-r rows twice."""
    rng = np.random.default_rng(50)
    x, kv = _chunk(rng, 27, D=64, Dx=32)
    w = _bf16(rng.standard_normal((32, 64)) / 6)
    ape = rng.standard_normal((4, 64))
    ov = O.compress(x, kv, w, ape, 4, np.arange(27), np.zeros(27, int), overlap=True)
    assert [g for _, g, _ in ov] == list(range(6))
    wide = O.compress(x, kv, w, np.concatenate([ape, ape]), 8, np.arange(27), np.zeros(27, int))
    assert [g for _, g, _ in wide] == [0, 1, 2]
    for _, k, y in wide:
        assert np.array_equal(ov[2 * k + 1][2], y)


def test_overlap_needs_the_whole_window_in_the_chunk():
    """One-shot calls publish an entry only when its whole window (the
    previous group too) is in the chunk as the same request's rows."""
    rng = np.random.default_rng(51)
    x, kv = _chunk(rng, 10)
    w = torch.zeros((64, 64), dtype=torch.bfloat16)
    got = O.compress(x, kv, w, np.zeros((2, 64)), 2, np.arange(8, 18), np.zeros(10, int),
                     overlap=True)
    assert [g for _, g, _ in got] == [5, 6, 7, 8]  # entry 4 lacks positions 6, 7


@pytest.mark.parametrize("r,splits", [
    (4, [[1, 1]] * 13),                        # decode: every window reaches back one group
    (4, [[2, 3], [7, 1], [1, 6], [3, 2]]),     # chunk starts inside groups
    (2, [[3, 2], [1, 4], [5, 1], [2, 2]]),
    (4, [[6, 0], [0, 5], [5, 6]]),             # idle requests in some calls
])
def test_stateful_overlap_equals_one_shot(r, splits):
    rng = np.random.default_rng(52 + r)
    lens = [sum(c[b] for c in splits) for b in range(2)]
    n = sum(lens)
    x, kv = _chunk(rng, n, D=64, Dx=32)
    w = _bf16(rng.standard_normal((32, 64)) / 6)
    ape = rng.standard_normal((r, 64))
    reqs = [list(range(0, lens[0])), list(range(lens[0], n))]
    got, _, _ = _stateful_run(x, kv, w, ape, r, reqs, splits, cap=2 * r, overlap=True)
    want = []
    for b in range(2):
        idx = np.array(reqs[b])
        for _, g, y in O.compress(x[idx], kv[idx], w, ape, r, np.arange(len(idx)),
                                  np.zeros(len(idx), int), overlap=True):
            want.append((b, g, y))
    assert sorted((b, g) for b, g, _ in got) == sorted((b, g) for b, g, _ in want)
    ref = {(b, g): y for b, g, y in want}
    for b, g, y in got:
        assert np.array_equal(y, ref[(b, g)]), (b, g)


def test_state_ring_holds_the_last_tokens():
    """After a call, slot p % cap of the request's block holds the kv row and
    the gate score of the last min(chunk length, cap) positions; older slots
    keep what they had."""
    rng = np.random.default_rng(48)
    x, kv = _chunk(rng, 12, D=16, Dx=8)
    w = _bf16(rng.standard_normal((8, 16)))
    ape = rng.standard_normal((2, 16))
    cap = 4
    state = np.full((3, cap, 32), -7.0)
    table = np.array([2])
    # call 1: positions 0..1 (two slots written); call 2: positions 2..8 (last four written)
    O.compress_stateful(x[:2], kv[:2], w, ape, 2, np.arange(2), np.zeros(2, int), state, table)
    assert np.all(state[2, 2:] == -7.0) and np.all(state[:2] == -7.0)
    O.compress_stateful(x[2:9], kv[2:9], w, ape, 2, np.arange(2, 9), np.zeros(7, int), state,
                        table)
    xf, kvf, wf = O.as_f64(x), O.as_f64(kv), O.as_f64(w)
    for p in range(5, 9):
        slot = state[2, p % cap]
        assert np.array_equal(slot[:16], kvf[p])
        assert np.allclose(slot[16:], xf[p] @ wf + ape[p % 2], rtol=1e-12, atol=1e-12)


def test_stateful_disabled_requests_and_negative_positions():
    rng = np.random.default_rng(49)
    x, kv = _chunk(rng, 6, D=16, Dx=8)
    w = _bf16(rng.standard_normal((8, 16)))
    ape = rng.standard_normal((2, 16))
    state = np.zeros((2, 4, 32))
    # request 0 disabled (-1), request 1 with a negative position row
    req = np.array([0, 0, 1, 1, 1, 1])
    pos = np.array([0, 1, -1, 1, 2, 3])
    out = O.compress_stateful(x, kv, w, ape, 2, pos, req, state, np.array([-1, 1]))
    assert [(b, g) for b, g, _ in out] == [(1, 0), (1, 1)]  # (1, 0) takes position 0 from the ring
    assert np.all(state[0] == 0.0)
    assert np.all(state[1, 0] == 0.0)  # the negative-position row wrote nothing


def test_compress_rmsnorm_unit_gamma():
    rng = np.random.default_rng(13)
    x, kv = _chunk(rng, 4)
    w = _bf16(rng.standard_normal((64, 64)) / 8)
    (_, _, y), = O.compress(x, kv, w, np.zeros((4, 64)), 4, np.arange(4), np.zeros(4, int),
                            gamma=torch.ones(64, dtype=torch.bfloat16))
    assert np.sqrt(np.mean(y * y)) == pytest.approx(1.0, rel=1e-2)


# ---------------------------------------------------------------- indexer


def _one_page_pool(keys, scales):
    n, Di = keys.shape
    pool = np.zeros((2, BLOCK, Di), np.int8)
    sp = np.zeros((2, BLOCK), np.float32)
    pool[1, :n] = keys
    sp[1, :n] = scales
    return pool, sp, np.array([1, 0])


def test_index_scores_hand_example():
    # one head, dim 4 (no rotation): q = [1, 2, 0, -1]
    # key a = [3, -1, 5, 2]: dot = 3 - 2 + 0 - 2 = -1 -> ReLU 0
    # key b = [1, 1, 1, 1]:  dot = 2 -> 0.5 * 2.0 * 2 = 2
    pool, sp, table = _one_page_pool(np.array([[3, -1, 5, 2], [1, 1, 1, 1]], np.int8),
                                     np.array([0.5, 0.5], np.float32))
    q = np.array([[1.0, 2.0, 0.0, -1.0]])
    s = O.index_scores(q, [2.0], p=1, n_cmp_b=2, ratio=1, idx_pool=pool, idx_scale_pool=sp,
                       table_row=table)
    assert s.tolist() == [0.0, 2.0]
    s = O.index_scores(q, [2.0], p=1, n_cmp_b=2, ratio=1, idx_pool=pool, idx_scale_pool=sp,
                       table_row=table, relu=False)
    assert s.tolist() == [-1.0, 2.0]
    # visibility: at p = 0 with ratio 1 only entry 0 is visible
    s = O.index_scores(q, [2.0], p=0, n_cmp_b=2, ratio=1, idx_pool=pool, idx_scale_pool=sp,
                       table_row=table)
    assert s.tolist() == [0.0]


def test_index_scores_heads_weights_and_scale():
    rng = np.random.default_rng(14)
    keys = rng.integers(-127, 128, (20, 8), dtype=np.int8)
    scales = rng.uniform(1e-3, 1e-2, 20).astype(np.float32)
    pool, sp, table = _one_page_pool(keys, scales)
    q = rng.standard_normal((3, 8))
    w = rng.standard_normal(3)
    kw = dict(p=100, n_cmp_b=20, ratio=1, idx_pool=pool, idx_scale_pool=sp, table_row=table)
    s = O.index_scores(q, w, **kw)
    # one head at a time: contributions add, and a head with a negative dot adds nothing
    per = [O.index_scores(q[h:h + 1], w[h:h + 1], **kw) for h in range(3)]
    assert np.allclose(s, sum(per), rtol=1e-12, atol=1e-12)
    for h in range(3):
        dots = keys.astype(np.float64) @ q[h]
        assert np.all(per[h][dots < 0] == 0)
        assert np.allclose(per[h][dots > 0], scales.astype(np.float64)[dots > 0] * w[h] * dots[dots > 0])
    # doubling every scale doubles every score
    pool2, sp2, _ = _one_page_pool(keys, scales * 2)
    s2 = O.index_scores(q, w, **{**kw, "idx_pool": pool2, "idx_scale_pool": sp2})
    assert np.allclose(s2, 2 * s, rtol=1e-6)


def test_index_scores_rotate_query_at_row_position_and_paging():
    rng = np.random.default_rng(15)
    nkeys = 300
    keys = rng.integers(-127, 128, (nkeys, 128), dtype=np.int8)
    scales = rng.uniform(1e-3, 1e-2, nkeys).astype(np.float32)
    pool = np.zeros((5, BLOCK, 128), np.int8)
    sp = np.zeros((5, BLOCK), np.float32)
    table = np.array([3, 0, 4])
    for c in range(nkeys):
        pool[table[c // BLOCK], c % BLOCK] = keys[c]
        sp[table[c // BLOCK], c % BLOCK] = scales[c]
    q = rng.standard_normal((4, 128))
    w = rng.standard_normal(4)
    p = 700
    s = O.index_scores(q, w, p, nkeys, 2, pool, sp, table, rope_cos=COS, rope_sin=SIN)
    assert len(s) == min(nkeys, (p + 1) // 2)
    qr = _cplx_rotate(q, p)
    dots = np.maximum(keys[:len(s)].astype(np.float64) @ qr.T, 0)
    assert np.allclose(s, scales[:len(s)] * (dots @ w), rtol=1e-9, atol=1e-9)
    # a different physical placement of the same logical pages changes nothing
    pool_b = np.zeros_like(pool)
    sp_b = np.zeros_like(sp)
    table_b = np.array([1, 2, 0])
    for j in range(3):
        pool_b[table_b[j]] = pool[table[j]]
        sp_b[table_b[j]] = sp[table[j]]
    s_b = O.index_scores(q, w, p, nkeys, 2, pool_b, sp_b, table_b, rope_cos=COS, rope_sin=SIN)
    assert np.array_equal(s, s_b)


# ---------------------------------------------------------------- top-k


def test_topk_matches_lexsort_with_ties():
    rng = np.random.default_rng(16)
    for n, k in [(50, 10), (300, 128), (1000, 999), (64, 64), (20, 64)]:
        s = rng.integers(-5, 6, n).astype(np.float64)  # many ties
        got = O.topk_select(s, k)
        order = np.lexsort((np.arange(n), -s))  # primary -score, then index
        want = np.sort(order[:k])
        assert np.array_equal(got[:len(want)], want)
        assert np.all(got[len(want):] == -1)
        assert np.all(np.diff(got[:len(want)]) > 0)


def test_select_blocks_hand_examples():
    # block 4: maxima 5, 9, 8 -> the two best blocks are 1 and 2
    s = [1, 5, 2, 3, 9, 0, 4, 4, 8]
    assert O.select_blocks(s, 2, block=4).tolist() == [1, 2]
    # the largest entry ranks a block, not its sum or mean: block 0 sums to 20, block 1 to 9
    s = [5, 5, 5, 5, 9, 0, 0, 0]
    assert O.select_blocks(s, 1, block=4).tolist() == [1]
    # equal maxima: the lower block wins
    s = [7, 0, 0, 0, 1, 7, 1, 1, 7, 7, 7, 7]
    assert O.select_blocks(s, 2, block=4).tolist() == [0, 1]
    # a ragged last block competes with its visible entries only; padding past the blocks
    s = [0, 0, 0, 0, 0, 0, 0, 0, 3]
    assert O.select_blocks(s, 4, block=8).tolist() == [0, 1, -1, -1]
    assert O.select_blocks(s, 1, block=8).tolist() == [1]


def test_topk_in_blocks_hand_examples():
    s = [1, 5, 2, 3, 9, 0, 4, 4, 8]
    # blocks 0 and 2 of four: positions 0..3 and 8; the 9 at position 4 is outside
    assert O.topk_in_blocks(s, [0, 2], 3, block=4).tolist() == [1, 3, 8]
    # -1 entries are ignored; too few eligible positions pad with -1
    assert O.topk_in_blocks(s, [2, -1], 3, block=4).tolist() == [8, -1, -1]
    assert O.topk_in_blocks(s, [-1, -1], 2, block=4).tolist() == [-1, -1]
    # ties inside the candidates: the lower position wins
    s = [4, 4, 0, 0, 4, 4, 4, 4]
    assert O.topk_in_blocks(s, [1, 0], 3, block=4).tolist() == [0, 1, 4]


def _dominates(s, a, b):
    return s[a] > s[b] or (s[a] == s[b] and a < b)


def test_topk_in_blocks_by_pairwise_dominance():
    """Brute force: every emitted position is eligible and beats every
    eligible position left out, and exactly min(k, eligible) are emitted."""
    rng = np.random.default_rng(48)
    for V, nb, k in [(37, 2, 5), (64, 3, 24), (65, 9, 30), (8, 1, 8), (100, 4, 7)]:
        s = rng.integers(-3, 4, V).astype(np.float64)
        n_all = (V + 7) // 8
        blocks = rng.choice(n_all, size=min(nb, n_all), replace=False)
        got = O.topk_in_blocks(s, blocks, k)
        elig = [p for p in range(V) if p // 8 in set(blocks.tolist())]
        chosen = [int(p) for p in got if p >= 0]
        assert len(chosen) == min(k, len(elig))
        assert chosen == sorted(chosen) and np.all(got[len(chosen):] == -1)
        assert set(chosen) <= set(elig)
        for a in chosen:
            for b in elig:
                if b not in chosen:
                    assert _dominates(s, a, b)


def test_select_blocks_by_pairwise_dominance():
    rng = np.random.default_rng(49)
    for V, nb in [(37, 2), (64, 5), (129, 16), (7, 1)]:
        s = rng.integers(-3, 4, V).astype(np.float64)
        n_all = (V + 7) // 8
        m = [max(s[8 * b:8 * b + 8]) for b in range(n_all)]
        got = [int(b) for b in O.select_blocks(s, nb) if b >= 0]
        assert len(got) == min(nb, n_all) and got == sorted(got)
        for a in got:
            for b in range(n_all):
                if b not in got:
                    assert _dominates(m, a, b)


@pytest.mark.parametrize("V,k,extra", [(64, 8, 0), (1000, 64, 0), (1000, 64, 5), (9, 2, 0),
                                       (4096, 512, 0)])
def test_two_level_selection_equals_flat_when_k_fits(V, k, extra):
    """With as many candidate blocks as selected positions (or more), ranking
    the same scores in two levels loses nothing: a position among the overall
    k best lies in a block whose maximum outranks every block without one."""
    rng = np.random.default_rng(V + k + extra)
    s = rng.integers(-4, 5, V).astype(np.float64)  # ties across blocks
    blocks = O.select_blocks(s, k + extra)
    assert np.array_equal(O.topk_in_blocks(s, blocks, k), O.topk_select(s, k))
    # with every block a candidate the second level is the flat top-k
    assert np.array_equal(O.topk_in_blocks(s, np.arange((V + 7) // 8), k), O.topk_select(s, k))


# ---------------------------------------------------------------- attention


def _attn_fixture(rng, n_cmp=40, kv_len=50, D=512, H=4):
    P = 4
    kv_pool = _bf16(rng.standard_normal((P, BLOCK, D)))
    cmp_pool = _bf16(rng.standard_normal((P, BLOCK, D)))
    kv_table = np.array([2, -1, -1, -1])
    cmp_table = np.array([3, -1, -1, -1])
    q = _bf16(rng.standard_normal((H, D)))
    sink = rng.standard_normal(H)
    return kv_pool, cmp_pool, kv_table, cmp_table, q, sink


def _dense_candidates(kv_pool, cmp_pool, kv_table, cmp_table, sel, win):
    rows_ = [cmp_pool[cmp_table[c // BLOCK], c % BLOCK].double().numpy() for c in sel]
    rows_ += [kv_pool[kv_table[p // BLOCK], p % BLOCK].double().numpy() for p in win]
    return np.stack(rows_)


def test_attention_without_sink_is_textbook_softmax_attention():
    rng = np.random.default_rng(17)
    kv_pool, cmp_pool, kv_table, cmp_table, q, _ = _attn_fixture(rng)
    sel = [3, 7, 11, -1, -1]
    p, scale = 45, 1 / np.sqrt(512)
    out, lse = O.sparse_attention(q, p, sel, kv_pool, kv_table, cmp_pool, cmp_table, None, scale,
                                  window=8)
    K = _dense_candidates(kv_pool, cmp_pool, kv_table, cmp_table, [3, 7, 11], range(38, 46))
    logits = scale * q.double().numpy() @ K.T
    assert np.allclose(out, softmax(logits, axis=1) @ K, rtol=1e-10, atol=1e-12)
    assert np.allclose(lse, logsumexp(logits, axis=1), rtol=1e-12)


def test_attention_sink_sits_in_the_denominator():
    rng = np.random.default_rng(18)
    kv_pool, cmp_pool, kv_table, cmp_table, q, sink = _attn_fixture(rng)
    sel = [0, 5, 9]
    p, scale = 20, 1 / np.sqrt(512)
    out, lse = O.sparse_attention(q, p, sel, kv_pool, kv_table, cmp_pool, cmp_table, sink, scale,
                                  window=16)
    K = _dense_candidates(kv_pool, cmp_pool, kv_table, cmp_table, sel, range(5, 21))
    logits = scale * q.double().numpy() @ K.T
    ext = np.concatenate([logits, sink[:, None]], axis=1)
    wts = softmax(ext, axis=1)[:, :-1]
    assert np.allclose(out, wts @ K, rtol=1e-10, atol=1e-12)
    assert np.allclose(lse, logsumexp(ext, axis=1), rtol=1e-12)


def test_attention_single_candidate_closed_form():
    rng = np.random.default_rng(19)
    kv_pool, cmp_pool, kv_table, cmp_table, q, sink = _attn_fixture(rng)
    scale = 0.05
    out, lse = O.sparse_attention(q, 0, [-1, -1], kv_pool, kv_table, cmp_pool, cmp_table, sink,
                                  scale)
    v = kv_pool[kv_table[0], 0].double().numpy()
    ell = scale * q.double().numpy() @ v
    assert np.allclose(out, expit(ell - sink)[:, None] * v[None, :], rtol=1e-12, atol=1e-14)
    assert np.allclose(lse, np.logaddexp(ell, sink), rtol=1e-12)


def test_attention_full_selection_equals_dense_and_paging_invariance():
    rng = np.random.default_rng(20)
    kv_pool, cmp_pool, kv_table, cmp_table, q, sink = _attn_fixture(rng)
    p, r, n_cmp = 37, 2, 19
    nv = O.visible_count(p, r, n_cmp)
    sel = O.topk_select(rng.standard_normal(nv), 64)  # k >= visible: everything, then -1
    assert np.array_equal(sel[:nv], np.arange(nv)) and np.all(sel[nv:] == -1)
    scale = 1 / np.sqrt(512)
    out, lse = O.sparse_attention(q, p, sel, kv_pool, kv_table, cmp_pool, cmp_table, sink, scale)
    K = _dense_candidates(kv_pool, cmp_pool, kv_table, cmp_table, range(nv), range(0, p + 1))
    ext = np.concatenate([scale * q.double().numpy() @ K.T, sink[:, None]], axis=1)
    assert np.allclose(out, softmax(ext, axis=1)[:, :-1] @ K, rtol=1e-10, atol=1e-12)
    # move the pages elsewhere
    kv2, cmp2 = kv_pool.clone(), cmp_pool.clone()
    kv2[0], cmp2[1] = kv_pool[kv_table[0]], cmp_pool[cmp_table[0]]
    out2, lse2 = O.sparse_attention(q, p, sel, kv2, np.array([0, -1, -1, -1]), cmp2,
                                    np.array([1, -1, -1, -1]), sink, scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_attention_rotates_query_at_row_position_and_inverse_output():
    rng = np.random.default_rng(21)
    kv_pool, cmp_pool, kv_table, cmp_table, q, sink = _attn_fixture(rng)
    p, scale = 60, 1 / np.sqrt(512)
    sel = [1, 2]
    out, _ = O.sparse_attention(q, p, sel, kv_pool, kv_table, cmp_pool, cmp_table, sink, scale,
                                rope_cos=COS, rope_sin=SIN)
    K = _dense_candidates(kv_pool, cmp_pool, kv_table, cmp_table, sel, range(0, p + 1))
    qr = _cplx_rotate(q.double().numpy(), p)
    ext = np.concatenate([scale * qr @ K.T, sink[:, None]], axis=1)
    want = softmax(ext, axis=1)[:, :-1] @ K
    assert np.allclose(out, want, rtol=1e-9, atol=1e-12)
    out_inv, _ = O.sparse_attention(q, p, sel, kv_pool, kv_table, cmp_pool, cmp_table, sink,
                                    scale, rope_cos=COS, rope_sin=SIN, inv_rope_out=True)
    assert np.allclose(_cplx_rotate(out_inv, p), want, atol=1e-9)


# ---------------------------------------------------------------- low-bit cache formats


def test_e2m1_values_match_the_format_table():
    # the E2M1 value table of the OCP microscaling format: magnitudes of codes 0..7
    want = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert O.e2m1_decode(np.arange(8)).tolist() == want
    assert O.e2m1_decode(np.arange(8, 16)).tolist() == [-v for v in want]


def test_e4m3_and_e8m0_decoders_match_torch():
    b = torch.arange(256, dtype=torch.uint8)
    want = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_decode(np.arange(256))
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(got[~np.isnan(got)], want[~np.isnan(want)])
    if hasattr(torch, "float8_e8m0fnu"):
        want = b.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        got = O.e8m0_decode(np.arange(256))
        assert np.array_equal(np.isnan(got), np.isnan(want))
        assert np.array_equal(got[~np.isnan(got)], want[~np.isnan(want)])
    assert O.e8m0_decode([127, 0, 254]).tolist() == [1.0, 2.0 ** -127, 2.0 ** 127]


def test_round_e4m3_matches_torch_cast():
    rng = np.random.default_rng(50)
    grid = O.e4m3_decode(np.arange(127))
    mids = (grid[1:] + grid[:-1]) / 2  # every tie
    x = np.concatenate([grid, mids, rng.uniform(0, 448, 2000), rng.uniform(0, 2 ** -5, 500)])
    x = x.astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.round_e4m3(x.astype(np.float64)), want)
    assert O.round_e4m3([1e6]).tolist() == [0x7E]  # saturates at 448


def test_round_e2m1_ties_and_saturation():
    x = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.26, 0.74, 5.5, 7.0, 100.0]
    # ties go to the code with mantissa bit 0: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0,
    # 1.75 -> 2.0, 2.5 -> 2.0, 3.5 -> 4.0, 5.0 -> 4.0
    assert O.round_e2m1(x).tolist() == [0, 2, 2, 4, 4, 6, 6, 1, 1, 7, 7, 7]
    assert O.round_e2m1([-0.3, -0.1, -6.0, 0.0]).tolist() == [9, 8, 15, 0]


def test_round_e2m1_is_nearest_by_brute_force():
    rng = np.random.default_rng(51)
    x = rng.uniform(-7, 7, 5000)
    got = O.e2m1_decode(O.round_e2m1(x))
    grid = np.array([-6, -4, -3, -2, -1.5, -1, -0.5, 0, 0.5, 1, 1.5, 2, 3, 4, 6])
    best = np.min(np.abs(np.clip(x, -6, 6)[:, None] - grid), axis=1)
    assert np.allclose(np.abs(np.clip(x, -6, 6) - got), best)


def test_nibble_packing_order():
    assert O.pack_nibbles([1, 2, 15, 0]).tolist() == [0x21, 0x0F]
    assert O.unpack_nibbles([0x21, 0x0F]).tolist() == [1, 2, 15, 0]


def test_fp4_e8m0_quantiser_scale_rule_and_error_bound():
    rng = np.random.default_rng(52)
    for _ in range(200):
        y = rng.standard_normal(128) * np.exp(rng.uniform(-8, 8))
        packed, sb = O.quantize_fp4_e8m0(y)
        back = O.dequant_fp4(packed, sb, 32, "e8m0")
        for gi in range(4):
            grp = y[32 * gi:32 * gi + 32]
            amax = np.max(np.abs(grp))
            e = int(sb[gi]) - 127
            # the smallest power of two that keeps every element inside the E2M1 range
            assert 6 * 2.0 ** e >= amax > 6 * 2.0 ** (e - 1)
            # no clipping; the error is at most half a step of the E2M1 grid (steps
            # 0.5 below 2, 1 below 4, 2 above) times the scale
            err = np.abs(back[32 * gi:32 * gi + 32] - grp)
            step = np.where(np.abs(grp) / 2.0 ** e < 2, 0.5, np.where(np.abs(grp) / 2.0 ** e < 4,
                                                                       1.0, 2.0))
            assert np.all(err <= step / 2 * 2.0 ** e * (1 + 1e-6))
    # exactly representable groups come back exactly; zero groups get scale byte 0
    y = np.concatenate([np.array([0.5, -3, 6, 1.5] * 8) * 4.0, np.zeros(32),
                        np.array([1.0] * 32), np.array([-6.0] + [0.0] * 31) * 2 ** -20])
    packed, sb = O.quantize_fp4_e8m0(y)
    assert sb.tolist() == [129, 0, 125, 107]  # amax 1: 6 * 2^-2 >= 1 > 6 * 2^-3
    assert np.array_equal(O.dequant_fp4(packed, sb, 32, "e8m0"), y)


def test_fp4_e4m3_quantiser_hand_example_and_bound():
    # amax 15 -> scale E4M3(15 / 6 = 2.5) = 2.5 exactly; 15 / 2.5 = 6 -> code 7,
    # 7 / 2.5 = 2.8 -> 3.0 (code 5), -1 / 2.5 = -0.4 -> -0.5 (code 9)
    y = np.zeros(16)
    y[:3] = [15.0, 7.0, -1.0]
    packed, sb = O.quantize_fp4_e4m3(y)
    assert sb.tolist() == [0x42]  # 0.1000.010 = 1.25 * 2^1
    assert O.unpack_nibbles(packed)[:4].tolist() == [7, 5, 9, 0]
    rng = np.random.default_rng(53)
    for _ in range(200):
        y = rng.standard_normal(512) * np.exp(rng.uniform(-4, 4))
        packed, sb = O.quantize_fp4_e4m3(y)
        back = O.dequant_fp4(packed, sb, 16, "e4m3")
        s = np.repeat(O.e4m3_decode(sb), 16)
        # the scale is the E4M3 rounding of amax/6 (torch's cast as the reference)
        amax6 = (np.abs(y.reshape(32, 16)).max(axis=1).astype(np.float32) / np.float32(6))
        assert np.array_equal(sb, torch.from_numpy(amax6).to(torch.float8_e4m3fn)
                              .view(torch.uint8).numpy())
        # error: half a grid step times the scale, or the clipping at 6 * scale
        q = np.abs(y) / s
        step = np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
        bound = np.maximum(step / 2 * s, np.abs(y) - 6 * s) * (1 + 1e-6)
        assert np.all(np.abs(back - y) <= bound)


def test_mxfp8_dequant_hand_example():
    # 0x38 = 1.0, 0xB8 = -1.0, 0x7E = 448, 0x01 = 2^-9; scales 2^1 and 2^-3
    codes = np.array([0x38, 0xB8, 0x7E, 0x01] + [0] * 28 + [0x38] + [0] * 31)
    got = O.dequant_mxfp8(codes, [128, 124])
    assert got[:4].tolist() == [2.0, -2.0, 896.0, 2.0 ** -8]
    assert got[32] == 2.0 ** -3


def test_compress_fp4_publication_quantises_the_bf16_row():
    rng = np.random.default_rng(54)
    x, kv = _chunk(rng, 8, D=128, Dx=64)
    w = _bf16(rng.standard_normal((64, 128)) / 8)
    ape = rng.standard_normal((4, 128))
    pos, req = np.arange(8), np.zeros(8, int)
    plain = O.compress(x, kv, w, ape, 4, pos, req)
    for fmt, fn in (("fp4_e4m3", O.quantize_fp4_e4m3), ("fp4_e8m0", O.quantize_fp4_e8m0)):
        got = O.compress(x, kv, w, ape, 4, pos, req, out=fmt)
        assert [(b, g) for b, g, *_ in got] == [(b, g) for b, g, _ in plain]
        for (_, _, codes, sb), (_, _, y) in zip(got, plain):
            c2, s2 = fn(y)
            assert np.array_equal(codes, c2) and np.array_equal(sb, s2)


def _lowbit_pool(rng, pages, fmt, D):
    nbytes = D if fmt == "mxfp8" else D // 2
    groups = D // (16 if fmt == "fp4_e4m3" else 32)
    codes = rng.integers(0, 256, size=(pages, BLOCK, nbytes), dtype=np.uint8)
    if fmt == "mxfp8":  # no NaN codes
        codes[(codes & 0x7F) == 0x7F] = 0
    if fmt == "fp4_e4m3":
        scales = rng.integers(0x20, 0x50, size=(pages, BLOCK, groups), dtype=np.uint8)
    else:
        scales = rng.integers(120, 132, size=(pages, BLOCK, groups), dtype=np.uint8)
    return O.LowBitPool(codes, scales, fmt)


def _dequant_pool(pool):
    P, R = pool.codes.shape[:2]
    D = pool.codes.shape[2] * (1 if pool.fmt == "mxfp8" else 2)
    out = np.zeros((P, R, D))
    for i in range(P):
        for j in range(R):
            out[i, j] = pool.dequant_row(pool.codes[i, j], pool.scales[i, j])
    return out


def test_lowbit_pools_read_as_their_dequantised_values():
    """Index scores and attention over low-bit pools equal the same calls over
    float pools holding the dequantised values (cache reads dequantise), and
    dequantised FP4 / MXFP8 values are exactly BF16-representable."""
    rng = np.random.default_rng(55)
    idx = _lowbit_pool(rng, 3, "fp4_e8m0", 128)
    cmp = _lowbit_pool(rng, 3, "fp4_e4m3", 512)
    kvp = _lowbit_pool(rng, 3, "mxfp8", 512)
    idx_f, cmp_f, kv_f = _dequant_pool(idx), _dequant_pool(cmp), _dequant_pool(kvp)
    for f in (idx_f, cmp_f, kv_f):
        assert np.array_equal(O.bf16_round(f), f)
    table = np.array([2, 0, 1])
    q_idx = rng.standard_normal((64, 128))
    w = rng.standard_normal(64)
    s1 = O.index_scores(q_idx, w, 700, 300, 2, idx, None, table, rope_cos=COS, rope_sin=SIN)
    s2 = O.index_scores(q_idx, w, 700, 300, 2, idx_f, np.ones((3, BLOCK)), table, rope_cos=COS,
                        rope_sin=SIN)
    assert np.array_equal(s1, s2)
    # brute force on a few entries: the plain weighted ReLU sum over dequantised keys
    qr = O.rope_rotate(q_idx, 700, COS, SIN)
    for c in (0, 131, 299):
        k = O.dequant_fp4(idx.codes[table[c // BLOCK], c % BLOCK],
                          idx.scales[table[c // BLOCK], c % BLOCK], 32, "e8m0")
        want = sum(w[h] * max(0.0, float(qr[h] @ k)) for h in range(64))
        assert np.isclose(s1[c], want, rtol=1e-12, atol=1e-12)
    q = _bf16(rng.standard_normal((4, 512)))
    sel = np.array([3, 17, 200, -1])
    a1 = O.sparse_attention(q, 300, sel, kvp, table, cmp, table, np.zeros(4), 0.05,
                            rope_cos=COS, rope_sin=SIN)
    a2 = O.sparse_attention(q, 300, sel, kv_f, table, cmp_f, table, np.zeros(4), 0.05,
                            rope_cos=COS, rope_sin=SIN)
    assert np.array_equal(a1[0], a2[0]) and np.array_equal(a1[1], a2[1])


def test_lowbit_row_decoders_agree():
    """The vectorised pool reader equals the one-row definitions."""
    rng = np.random.default_rng(56)
    for fmt, D in (("fp4_e4m3", 512), ("fp4_e8m0", 128), ("mxfp8", 512)):
        pool = _lowbit_pool(rng, 1, fmt, D)
        rows = pool.dequant_rows(pool.codes[0], pool.scales[0])
        for j in (0, 5, 127):
            assert np.array_equal(rows[j], pool.dequant_row(pool.codes[0, j], pool.scales[0, j]))
        # no rows (a query that sees no compressed entry)
        assert pool.dequant_rows(pool.codes[0, :0], pool.scales[0, :0]).shape == (0, D)


def test_mxfp8_quantiser_scale_rule_and_torch_codes():
    """FP8 index plane (MXFP8 reading): the scale is the smallest power of two
    keeping every element within 448, the codes torch's E4M3 cast of the FP32
    quotient, and E4M3-representable groups come back exactly."""
    rng = np.random.default_rng(57)
    for _ in range(100):
        y = rng.standard_normal(128) * np.exp(rng.uniform(-10, 10))
        codes, sb = O.quantize_mxfp8(y)
        for gi in range(4):
            grp = y[32 * gi:32 * gi + 32]
            amax = np.max(np.abs(grp))
            e = int(sb[gi]) - 127
            assert 448 * 2.0 ** e >= amax > 448 * 2.0 ** (e - 1)
            q = torch.from_numpy(grp.astype(np.float32) / np.float32(2.0 ** e))
            want = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(codes[32 * gi:32 * gi + 32], want)
        back = O.dequant_mxfp8(codes, sb)
        # relative error of E4M3 rounding: at most 2^-4 of the value, or half
        # the subnormal step 2^-10 times the scale
        scl = np.repeat(2.0 ** (sb.astype(np.int64) - 127), 32)
        assert np.all(np.abs(back - y) <= np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10 * scl))
    y = np.array([1.0, -448.0 / 256, 0.5, 3.0] * 8 + [0.0] * 32)
    codes, sb = O.quantize_mxfp8(y)
    assert sb.tolist() == [120, 0]  # amax 3: 448 * 2^-7 = 3.5 >= 3 > 448 * 2^-8
    assert np.array_equal(O.dequant_mxfp8(codes, sb)[:32], y[:32])
    assert not codes[32:].any()
