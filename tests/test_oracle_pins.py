"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin is a value the pages print, a closed form, a library routine that a
special case reduces to, an invariant, or brute force on tiny inputs.  The
planted-mistake tests at the end compile altered copies of the oracle and show
that each plausible mistake fails at least one of these pins.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import qsa_inputs as qi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def widen(h):
    return qi.bf16_bits_to_f32(np.asarray(h, np.uint16))


# --------------------------------------------------------------------------
# bf16 narrowing: reduces to torch's round-to-nearest-even cast
# --------------------------------------------------------------------------

def test_bf16_narrowing_matches_torch_cast(orc):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    # exact ties: low half exactly 0x8000 with both parities of the kept lsb
    ties = (np.arange(2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    specials = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.4028235e38, 1e-40, -1e-45],
                        np.float32)
    for v in np.concatenate([vals[:5000], ties, specials]):
        want = torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16)
        assert orc.f32_to_bf16(v) == (int(want.item()) & 0xFFFF), v


def test_bf16_narrowing_keeps_nan(orc):
    h = orc.f32_to_bf16(float("nan"))
    assert (h & 0x7F80) == 0x7F80 and (h & 0x007F) != 0


# --------------------------------------------------------------------------
# RoPE tables
# --------------------------------------------------------------------------

def test_rope_position_zero_is_identity(orc):
    c, s = orc.rope_table(4)
    assert np.all(c[0] == 0x3F80) and np.all(s[0] == 0)


def test_rope_closed_form_angles(orc):
    theta = 10000.0
    c, s = orc.rope_table(300, theta)
    for p in (1, 2, 3, 7, 100, 299):
        for j in (0, 1, 5, 16, 31):
            ang = p * theta ** (-(2 * j) / 64.0)
            for tab, fn in ((c, math.cos), (s, math.sin)):
                got = float(widen(tab[p, j]))
                # bf16 keeps 8 significant bits: half an ulp is <= 2^-9 relative
                assert abs(got - fn(ang)) <= 2.0**-8 * max(abs(fn(ang)), 2.0**-8) + 1e-6, (p, j)
                assert tab[p, j] == tab[p, j + 32]


def test_rope_unit_circle(orc):
    c, s = orc.rope_table(4096, 10000.0)
    cf, sf = widen(c).astype(np.float64), widen(s).astype(np.float64)
    assert np.max(np.abs(cf**2 + sf**2 - 1.0)) < 2 * 2.0**-8


def test_rope_theta_matters(orc):
    c1, _ = orc.rope_table(64, 10000.0)
    c2, _ = orc.rope_table(64, 1e7)
    assert np.array_equal(c1[:, 0], c2[:, 0])        # inv_freq[0] = 1 for every theta
    assert not np.array_equal(c1[:, 16], c2[:, 16])


# --------------------------------------------------------------------------
# Pooling
# --------------------------------------------------------------------------

def const_keys(n_blocks, value, stride=128):
    k = np.zeros((4 * n_blocks, stride), np.uint16)
    k[:, :128] = qi.to_bf16_bits(np.full((4 * n_blocks, 128), value, np.float32))
    return k


def test_pool_constant_vector_closed_form(orc):
    """All four tokens = all-ones vector, w = 0, eps = 0: the normed key is all
    ones; block 0 is unrotated and block b is rotated at its first token 4b:
    out_i = bf16(c_i - s_i), out_{i+32} = bf16(c_i + s_i), out_{64..} = 1."""
    nb = 40
    c, s = orc.rope_table(4 * nb)
    w = np.zeros(128, np.uint16)
    out = orc.pool_blocks(const_keys(nb, 1.0), 128, 0, nb, w, c, s, 0.0)
    assert np.all(out[0] == 0x3F80)
    for b in range(nb):
        cf = widen(c[4 * b, :32]).astype(np.float32)
        sf = widen(s[4 * b, :32]).astype(np.float32)
        assert np.array_equal(out[b, :32], qi.to_bf16_bits(cf - sf)), b
        assert np.array_equal(out[b, 32:64], qi.to_bf16_bits(cf + sf)), b
        assert np.all(out[b, 64:] == 0x3F80)


def test_pool_weight_enters_as_one_plus_w(orc):
    rng = np.random.default_rng(3)
    w = qi.normal_bf16(rng, (128,), 0.1)
    c, s = orc.rope_table(4)
    out = orc.pool_blocks(const_keys(1, 1.0), 128, 0, 1, w, c, s, 0.0)
    want = qi.to_bf16_bits(np.float32(1.0) + widen(w))
    assert np.array_equal(out[0], want)


def test_pool_eps_and_mean_closed_form(orc):
    """Tiny keys make eps visible: constant 2^-10 keys, eps = 1e-6.
    mean = 2^-10, ms = 2^-20, y = 2^-10 / sqrt(2^-20 + 1e-6)."""
    c, s = orc.rope_table(4)
    w = np.zeros(128, np.uint16)
    out = orc.pool_blocks(const_keys(1, 2.0**-10), 128, 0, 1, w, c, s, 1e-6)
    y = 2.0**-10 / math.sqrt(2.0**-20 + 1e-6)
    want = qi.to_bf16_bits(np.array([y], np.float32))[0]
    assert np.all(out[0] == want), (hex(out[0, 0]), hex(want))


def test_pool_mean_of_distinct_tokens(orc):
    """Tokens 3, 1, 0, 0 average to 1 on dims 64..127 (unrotated) and tokens
    2, 2, 2, 2 give 2 on dims 0..63: with eps = 0, w = 0 the rms is
    sqrt((64*1 + 64*4)/128) = sqrt(2.5)."""
    k = np.zeros((4, 128), np.float32)
    k[:, :64] = 2.0
    k[0, 64:], k[1, 64:] = 3.0, 1.0
    c, s = orc.rope_table(4)
    out = orc.pool_blocks(qi.to_bf16_bits(k), 128, 0, 1, np.zeros(128, np.uint16), c, s, 0.0)
    r = 1.0 / math.sqrt(2.5)
    assert np.all(out[0, 64:] == qi.to_bf16_bits(np.array([r], np.float32))[0])
    assert np.all(out[0, :64] == qi.to_bf16_bits(np.array([2 * r], np.float32))[0])


def test_pool_power_of_two_scale_invariance(orc):
    rng = np.random.default_rng(11)
    keys = qi.raw_keys(rng, 4 * 64)
    w = qi.normal_bf16(rng, (128,), 0.1)
    c, s = orc.rope_table(4 * 64)
    a = orc.pool_blocks(keys, 128, 0, 64, w, c, s, 0.0)
    for k in (-6, 3):
        scaled = qi.to_bf16_bits(widen(keys) * np.float32(2.0**k))
        b = orc.pool_blocks(scaled, 128, 0, 64, w, c, s, 0.0)
        assert np.array_equal(a, b)


def test_pool_unit_rms_and_rotation_preserves_pair_norms(orc):
    rng = np.random.default_rng(12)
    nb = 256
    keys = qi.raw_keys(rng, 4 * nb, token_scale=True)
    c, s = orc.rope_table(4 * nb)
    out = widen(orc.pool_blocks(keys, 128, 0, nb, np.zeros(128, np.uint16), c, s, 1e-6))
    out = out.astype(np.float64)
    rms = np.sqrt(np.mean(out**2, axis=1))
    assert np.all(np.abs(rms - 1.0) < 0.02)
    # unrotated copy: block 0 of each key group pooled at position 0 has no rotation
    pair_rot = out[:, :32] ** 2 + out[:, 32:64] ** 2
    un = np.zeros_like(out)
    for b in range(nb):
        kb = keys[4 * b:4 * b + 4]
        un[b] = widen(orc.pool_blocks(kb, 128, 0, 1, np.zeros(128, np.uint16), c, s, 1e-6)[0])
    pair_un = un[:, :32] ** 2 + un[:, 32:64] ** 2
    assert np.allclose(pair_rot, pair_un, rtol=0.03, atol=1e-3)
    assert np.array_equal(out[:, 64:], un[:, 64:])


def test_pool_stride_and_offset_indexing(orc):
    """The fused q|k layout (stride 640, key at column 512) and a compact copy give
    the same keys; pooling [f, f+n) from token 4f equals that slice of a full pool."""
    rng = np.random.default_rng(13)
    T = 4 * 48
    fq = qi.fused_qk(rng, T)
    kw = qi.normal_bf16(rng, (128,), 0.1)
    c, s = orc.rope_table(T)
    compact = np.ascontiguousarray(fq[:, 512:640])
    full = orc.pool_blocks(compact, 128, 0, 48, kw, c, s, 1e-6)
    fused = orc.pool_blocks(fq.reshape(-1)[512:], 640, 0, 48, kw, c, s, 1e-6)
    assert np.array_equal(full, fused)
    part = orc.pool_blocks(compact[4 * 17:], 128, 17, 9, kw, c, s, 1e-6, total_blocks=48)
    assert np.array_equal(part[17:26], full[17:26])
    assert np.all(part[:17] == 0) and np.all(part[26:] == 0)


def mean_cast_case():
    """Raw keys of one block whose f32 mean must be rounded to bf16 to give the
    expected block key (see test_pool_mean_is_cast_to_bf16_before_the_norm)."""
    k = np.zeros((4, 128), np.float32)
    k[0, :126] = 2.0**-8
    k[1, :126] = 3 * 2.0**-17
    k[:, 126:] = 64.0
    w = np.zeros(128, np.float32)
    w[:] = 0.5
    return qi.to_bf16_bits(k), qi.to_bf16_bits(w)


def test_pool_mean_is_cast_to_bf16_before_the_norm(orc):
    """PR #1160 description: the four raw keys are averaged in float32 and the
    mean is cast back to bf16 before the norm.  These inputs make that cast
    decide the output bits.
      dims 0..125: tokens 2^-8, 3*2^-17, 0, 0.  The f32 mean is 2^-10 (1 + 3*2^-9),
                   which bf16 rounds up to 2^-10 (1 + 2^-7).
      dims 126, 127: four tokens of 64, so the mean is 64.
    With eps = 0 the mean square is 2*64^2/128 = 64 plus the small dims' share
    (below 2^-20, under half an f32 ulp of 64), so r = 1/sqrt(64) = 1/8 exactly.
    w = 0.5 gives a gain of 1.5, and block 0 sits at position 0 (no rotation).
      small dims: 2^-13 (1 + 2^-7) * 1.5 = 2^-13 * 1.51171875, halfway between the
                  bf16 values 2^-13 * 1.5078125 and 2^-13 * 1.515625; the tie goes
                  to the even one, 1.515625.  (Kept in f32, the mean would give
                  2^-13 * 1.5087890625, which rounds to 1.5078125.)
      large dims: 64 / 8 * 1.5 = 12."""
    k, w = mean_cast_case()
    c, s = orc.rope_table(4)
    out = orc.pool_blocks(k, 128, 0, 1, w, c, s, 0.0)
    small = qi.to_bf16_bits(np.array([2.0**-13 * 1.515625], np.float32))[0]
    assert widen(small) == np.float32(2.0**-13 * 1.515625)      # a bf16 value
    assert np.all(out[0, :126] == small), hex(out[0, 0])
    assert np.all(out[0, 126:] == qi.to_bf16_bits(np.array([12.0], np.float32))[0])


def test_pool_depends_on_the_bf16_mean_only(orc):
    """PR #1160 description (mean in float32, cast back to bf16): a block's key
    is a function of the bf16 mean of its four tokens.  Replacing the four
    tokens by four copies of that mean (its exact sum rounded once to f32, then
    torch's bf16 cast) must give the same key bits, at every block position."""
    rng = np.random.default_rng(14)
    nb = 96
    keys = qi.raw_keys(rng, 4 * nb, token_scale=True)
    kw = qi.normal_bf16(rng, (128,), 0.1)
    c, s = orc.rope_table(4 * nb)
    kf = widen(keys).astype(np.float64).reshape(nb, 4, 128)
    mean = (kf.sum(axis=1).astype(np.float32) * np.float32(0.25))
    mean_bf16 = qi.to_bf16_bits(mean)
    # the f32 means are rarely bf16 values, so this case tests the cast
    assert np.mean(widen(mean_bf16) != mean) > 0.5
    replicated = np.repeat(mean_bf16, 4, axis=0)
    a = orc.pool_blocks(keys, 128, 0, nb, kw, c, s, 1e-6)
    b = orc.pool_blocks(replicated, 128, 0, nb, kw, c, s, 1e-6)
    assert np.array_equal(a, b)


# --------------------------------------------------------------------------
# Scoring
# --------------------------------------------------------------------------

def onehot_q(dims, signs=(1, 1, 1, 1)):
    q = np.zeros((4, 128), np.float32)
    for h, (d, sg) in enumerate(zip(dims, signs)):
        q[h, d] = sg
    return qi.to_bf16_bits(q)


def test_score_onehot_closed_form(orc):
    rng = np.random.default_rng(21)
    keys = qi.normal_bf16(rng, (50, 128))
    kf = widen(keys).astype(np.float64)
    dims = (3, 77, 0, 127)
    got = orc.score_row(onehot_q(dims), keys, 50)
    want = sum(np.maximum(kf[:, d], 0.0) for d in dims) / math.sqrt(128.0)
    assert np.allclose(got, want, rtol=1e-6, atol=0)


def test_score_relu_is_per_head(orc):
    """Head 1 is the negation of head 0: per-head relu gives |k_d|, a relu after
    the head sum would give 0."""
    rng = np.random.default_rng(22)
    keys = qi.normal_bf16(rng, (64, 128))
    kf = widen(keys).astype(np.float64)
    q = onehot_q((5, 5, 9, 9), (1, -1, 1, -1))
    got = orc.score_row(q, keys, 64)
    want = (np.abs(kf[:, 5]) + np.abs(kf[:, 9])) / math.sqrt(128.0)
    assert np.allclose(got, want, rtol=1e-6)
    assert np.all(got > 0)


def test_score_zero_query_and_power_of_two_linearity(orc):
    rng = np.random.default_rng(23)
    keys = qi.normal_bf16(rng, (80, 128))
    q = qi.normal_bf16(rng, (4, 128))
    assert np.all(orc.score_row(np.zeros((4, 128), np.uint16), keys, 80) == 0)
    a = orc.score_row(q, keys, 80)
    b = orc.score_row(qi.to_bf16_bits(widen(q) * 2), keys, 80)
    assert np.array_equal(b, a * 2)


def test_score_all_negative_heads_give_zero(orc):
    rng = np.random.default_rng(24)
    keys = np.abs(widen(qi.normal_bf16(rng, (30, 128)))) + 0.01
    q = -np.abs(widen(qi.normal_bf16(rng, (4, 128)))) - 0.01
    got = orc.score_row(qi.to_bf16_bits(q), qi.to_bf16_bits(keys), 30)
    assert np.all(got == 0)


def test_score_nan_propagates(orc):
    rng = np.random.default_rng(25)
    keys = qi.normal_bf16(rng, (10, 128))
    keys[4, 17] = 0x7FC0
    got = orc.score_row(qi.normal_bf16(rng, (4, 128)), keys, 10)
    assert np.isnan(got[4]) and np.all(np.isfinite(np.delete(got, 4)))


def test_score_rows_prefix_sentinel_and_key_base(orc):
    rng = np.random.default_rng(26)
    T = 64
    fq = qi.fused_qk(rng, T)
    qw, kw = qi.norm_weights(rng)
    c, s = orc.rope_table(T)
    keys = orc.pool_blocks(np.ascontiguousarray(fq[:, 512:]), 128, 0, T // 4, kw, c, s, 1e-6)
    cols = 20
    pos = np.array([0, 3, 4, 40, 63, 62], np.int32)
    vis = np.array([1, 4, 2, 41, 60, 0], np.int32)
    sc = np.full((len(pos), cols), -7.0, np.float32)
    rc, _ = orc.score_rows(fq, 640, pos, len(pos), T, qw, c, s, 1e-6, keys, sc, cols,
                           visible_len=vis)
    assert rc == 0
    for i, (p, v) in enumerate(zip(pos, vis)):
        n = v // 4
        assert np.all(sc[i, n:] == -7.0)
        qp = orc.qprep(fq[i, :512], p, qw, c, s, 1e-6)
        assert np.array_equal(sc[i, :n], orc.score_row(qp, keys, n))
    # key_base: row i reads its own key set
    keys2 = np.concatenate([np.zeros((5, 128), np.uint16), keys])
    sc2 = np.full((len(pos), cols), -7.0, np.float32)
    rc, _ = orc.score_rows(fq, 640, pos, len(pos), T, qw, c, s, 1e-6, keys2, sc2, cols,
                           visible_len=vis, key_base=np.full(len(pos), 5, np.int64))
    assert rc == 0 and np.array_equal(sc, sc2)


def test_score_rows_range_errors(orc):
    T = 16
    c, s = orc.rope_table(T)
    z = np.zeros(128, np.uint16)
    fq = np.zeros((3, 640), np.uint16)
    keys = np.zeros((4, 128), np.uint16)
    sc = np.zeros((3, 4), np.float32)
    for pos, vis, bad in (([0, 16, 1], None, 1), ([0, -1, 1], None, 1), ([0, 5, 1], [1, 7, 1], 1)):
        rc, row = orc.score_rows(fq, 640, np.array(pos, np.int32), 3, T, z, c, s, 1e-6, keys, sc, 4,
                                 visible_len=None if vis is None else np.array(vis, np.int32))
        assert rc == 3 and row == bad


def test_query_rotates_at_the_row_position(orc):
    """PR #1160 description: each query head is normed and then rotated at the
    row's own position p.  All four heads are one-hot on dim i < 32 (w = 0,
    eps = 0): the norm gives bf16(sqrt(128)) = 11.3125 on dim i, and RoPE at p
    moves it to bf16(11.3125 c) on dim i and bf16(11.3125 s) on dim i + 32
    (c, s: the table's bf16 cos/sin at row p, column i; the product of two
    8-bit significands is exact in f32).  Block 0's key is e_i, block 1's is
    e_{i+32}; with the head sum of four equal relus the scores are
    4 relu(bf16(11.3125 c)) / sqrt(128) and 4 relu(bf16(11.3125 s)) / sqrt(128)."""
    T = 400
    c, s = orc.rope_table(T)
    cf, sf = widen(c).astype(np.float32), widen(s).astype(np.float32)
    n = np.float32(11.3125)
    cases = [(p, i) for p in (9, 14, 37, 101, 250, 399) for i in (0, 1, 7, 31)]
    fq = np.zeros((len(cases), 640), np.float32)
    for r, (p, i) in enumerate(cases):
        fq[r, [i, 128 + i, 256 + i, 384 + i]] = 1.0
    pos = np.array([p for p, _ in cases], np.int32)
    sc = np.full((len(cases), 4), -7.0, np.float32)
    for i in sorted({i for _, i in cases}):
        rows = [r for r, (_, ii) in enumerate(cases) if ii == i]
        keys = np.zeros((T // 4, 128), np.float32)
        keys[0, i], keys[1, i + 32] = 1.0, 1.0
        sub = np.full((len(rows), 4), -7.0, np.float32)
        rc, _ = orc.score_rows(qi.to_bf16_bits(fq[rows]), 640, pos[rows], len(rows), T,
                               np.zeros(128, np.uint16), c, s, 0.0, qi.to_bf16_bits(keys), sub, 4,
                               visible_len=np.full(len(rows), 8, np.int32))
        assert rc == 0
        sc[rows] = sub
    for r, (p, i) in enumerate(cases):
        rot = qi.to_bf16_bits(np.array([n * cf[p, i], n * sf[p, i]], np.float32))
        want = 4.0 * np.maximum(widen(rot).astype(np.float64), 0.0) / math.sqrt(128.0)
        assert np.allclose(sc[r, :2], want.astype(np.float32), rtol=1e-6, atol=0), (p, i)
        assert np.all(sc[r, 2:] == -7.0)
    # the cases span both signs of cos and sin, so a missing or wrong rotation shows
    assert np.any(sc[:, 0] == 0) and np.any(sc[:, 1] == 0)
    assert np.mean(sc[:, 0] > 0) > 0.3 and np.mean(sc[:, 1] > 0) > 0.3


# --------------------------------------------------------------------------
# Selection: brute force, an independent radix select, closed forms, invariants
# --------------------------------------------------------------------------

def brute_force_mask(scores, p, tokens, budget):
    """O(n^2): block b is kept iff fewer than K blocks precede it in the
    canonical order (higher score, or equal score and lower index)."""
    n, tail = (p + 1) // 4, (p + 1) % 4
    K = min(budget // 4, n)
    v = [0.0 if x == 0 else float(x) for x in scores[:n]]
    m = np.zeros(tokens, np.uint8)
    for b in range(n):
        rank = sum(1 for c in range(n) if v[c] > v[b] or (v[c] == v[b] and c < b))
        if rank < K:
            m[4 * b:4 * b + 4] = 1
    m[4 * n:p + 1] = 1
    return m


def radix_mask(scores, p, tokens, budget):
    """Independent algorithm: 8-bit MSD radix select over order-preserving u32 keys."""
    n = (p + 1) // 4
    K = min(budget // 4, n)
    s = np.asarray(scores[:n], np.float32).copy()
    s[s == 0] = 0.0
    u = s.view(np.uint32).astype(np.uint64)
    key = np.where(u >> 31 == 1, (~u) & 0xFFFFFFFF, u | 0x80000000).astype(np.uint64)
    prefix, need = 0, K
    for shift in (24, 16, 8, 0):
        hi = key >> (shift + 8)
        cand = (hi == prefix) if shift < 24 else np.ones(n, bool)
        digit = (key >> shift) & 0xFF
        cnt = np.bincount(digit[cand].astype(np.int64), minlength=256)
        above = 0
        for d in range(255, -1, -1):
            if above + cnt[d] >= need:
                break
            above += cnt[d]
        need -= above
        prefix = (prefix << 8) | d
    kept = key > prefix
    eq = np.nonzero(key == prefix)[0][:need]
    kept[eq] = True
    m = np.zeros(tokens, np.uint8)
    for b in np.nonzero(kept)[0]:
        m[4 * b:4 * b + 4] = 1
    m[4 * n:p + 1] = 1
    return m


def test_select_exhaustive_tiny_rows(orc):
    alphabet = [-0.0, 0.0, 1.0, 2.0, -1.0]
    for n in range(1, 6):
        for combo in itertools.product(alphabet, repeat=n):
            s = np.array(combo, np.float32)
            for tail in (0, 3):
                p = 4 * n - 1 + tail
                if tail == 3:
                    p = 4 * n + 2
                for budget in (4, 8, 12):
                    got, rc = orc.select_row(s, p, p + 3, budget)
                    assert rc == 0
                    assert np.array_equal(got, brute_force_mask(s, p, p + 3, budget)), (combo, p, budget)


def test_select_random_small_rows_vs_brute_force_and_radix(orc):
    rng = np.random.default_rng(31)
    for trial in range(300):
        n = int(rng.integers(1, 13))
        p = 4 * n - 1 + int(rng.integers(0, 4))
        tokens = p + 1 + int(rng.integers(0, 9))
        s = rng.choice(np.array([-0.0, 0.0, 0.5, 1.0, 1.0, 2.0, 3.5], np.float32), size=n)
        s = s + (rng.random(n) < 0.3) * rng.standard_normal(n).astype(np.float32)
        s = s.astype(np.float32)
        budget = 4 * int(rng.integers(1, 15))
        got, rc = orc.select_row(s, p, tokens, budget)
        assert rc == 0
        assert np.array_equal(got, brute_force_mask(s, p, tokens, budget))
        if n > budget // 4:
            assert np.array_equal(got, radix_mask(s, p, tokens, budget))


def test_select_long_rows_vs_independent_radix(orc):
    rng = np.random.default_rng(32)
    for n, budget in ((513, 2048), (2048, 2048), (5000, 2044), (4000, 4), (3000, 512)):
        s = qi.stress_scores(rng, 1, n)[0]
        p = 4 * n - 1 + int(rng.integers(0, 4))
        got, rc = orc.select_row(s, p, p + 1, budget)
        assert rc == 0
        assert np.array_equal(got, radix_mask(s, p, p + 1, budget))


def test_select_invariants(orc):
    rng = np.random.default_rng(33)
    tokens = 9000
    for trial in range(40):
        p = int(rng.integers(0, tokens))
        budget = 4 * int(rng.integers(1, 513))
        n, tail = (p + 1) // 4, (p + 1) % 4
        s = qi.stress_scores(rng, 1, max(n, 1), zero_frac=0.4, levels=16)[0]
        m, rc = orc.select_row(s, p, tokens, budget)
        assert rc == 0
        K = min(budget // 4, n)
        assert int(m.sum()) == 4 * K + tail                      # closed form
        assert np.all(m[p + 1:] == 0)                             # causality
        assert np.all(m[4 * n:p + 1] == 1)                        # the tail
        blk = m[:4 * n].reshape(n, 4) if n else np.zeros((0, 4))
        assert np.all((blk.min(1) == blk.max(1)))                  # whole blocks only
        kept = blk[:, 0] == 1 if n else np.zeros(0, bool)
        if n > budget // 4:
            sv = np.where(s[:n] == 0, 0.0, s[:n])
            assert sv[kept].min() >= sv[~kept].max()              # kept >= dropped
            cut = sv[kept].min()
            eqi = np.nonzero(sv == cut)[0]
            k_eq = kept[eqi]
            assert np.all(k_eq[:k_eq.sum()]) and not np.any(k_eq[k_eq.sum():])  # tie prefix
        else:
            assert np.all(m[:p + 1] == 1)                         # all-kept prefix


def test_select_signed_zero_ties(orc):
    # blocks: 5, -0, +0, -0, +0 ; keep 3 -> 5 and the two lowest-index zeros (1, 2)
    s = np.array([5.0, -0.0, 0.0, -0.0, 0.0], np.float32)
    m, rc = orc.select_row(s, 19, 20, 12)
    assert rc == 0
    assert list(m.reshape(5, 4)[:, 0]) == [1, 1, 1, 0, 0]
    s = np.array([0.0, -0.0, 5.0, 0.0, -0.0], np.float32)
    m, _ = orc.select_row(s, 19, 20, 12)
    assert list(m.reshape(5, 4)[:, 0]) == [1, 1, 1, 0, 0]


def test_select_nonfinite_and_range(orc):
    s = np.array([1.0, np.nan, 2.0, 3.0], np.float32)
    m, rc = orc.select_row(s, 15, 16, 4)
    assert rc == 4 and np.all(m == 0xAB)                      # row untouched
    m, rc = orc.select_row(s, 15, 16, 16)                     # all-kept: reads no score
    assert rc == 0 and np.all(m == 1)
    s = np.array([1.0, np.inf, 2.0, 3.0], np.float32)
    assert orc.select_row(s, 15, 16, 8)[1] == 4
    assert orc.select_row(s, 16, 16, 8)[1] == 3
    assert orc.select_row(s, -1, 16, 8)[1] == 3
    for bad in (0, -4, 6, 2052):
        assert orc.select_row(s, 3, 16, bad)[1] == 1


def test_select_golden_geometry(orc):
    """Block counts, keep and mask length that the pages print (see the fixture)."""
    rows = []
    with open(os.path.join(GOLDEN, "select_geometry.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(x) for x in line.split()[:6]])
    assert len(rows) == 7
    rng = np.random.default_rng(34)
    for p, budget, blocks, tail, keep, ones in rows:
        s = rng.standard_normal(blocks).astype(np.float32)
        m, rc = orc.select_row(s, p, p + 1, budget)
        assert rc == 0
        assert (p + 1) // 4 == blocks and (p + 1) % 4 == tail
        assert int(m.sum()) == ones == 4 * keep + tail
        if blocks > keep:
            kept = np.nonzero(m[:4 * blocks:4])[0]
            top = np.argsort(-s, kind="stable")[:keep]
            assert np.array_equal(np.sort(top), kept)


# --------------------------------------------------------------------------
# Planted mistakes: each altered copy of the oracle must fail a pin above
# --------------------------------------------------------------------------

SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "qsa_oracle.c")


# ---- token list and paged gather (metrale layers/qsa.rs decode_select)

def test_mask_tokens_equals_nonzero(orc):
    """The token list is every set mask byte, ascending: numpy's nonzero on random
    masks; the count is reported even when the list is capped."""
    rng = np.random.default_rng(11)
    for tokens in (1, 7, 64, 1000):
        m = (rng.random(tokens) < 0.3).astype(np.uint8)
        got, n = orc.mask_tokens(m)
        assert n == int(m.sum()) and np.array_equal(got, np.nonzero(m)[0])
        cap = max(1, n // 2)
        got_c, n_c = orc.mask_tokens(m, cap)
        assert n_c == n and np.array_equal(got_c, np.nonzero(m)[0][:cap])


def test_mask_tokens_of_a_selection_is_the_pages_list(orc):
    """decode_select's list: the kept blocks (top keep by (-score, index), then
    sorted ascending) expanded to their 4 tokens each, then the tail tokens --
    built here from a numpy sort, compared with the oracle's select + list."""
    rng = np.random.default_rng(12)
    for p, budget in ((2052, 2048), (4099, 64), (30001, 2048), (9, 4)):
        n = (p + 1) // 4
        sc = (rng.integers(0, 40, size=n) / 8.0).astype(np.float32)   # ties at the cut
        mask, rc = orc.select_row(sc, p, p + 7, budget)
        assert rc == 0
        keep = min(budget // 4, n)
        order = np.lexsort((np.arange(n), -sc.astype(np.float64)))[:keep]
        blocks = np.sort(order)
        want = np.concatenate([(4 * blocks[:, None] + np.arange(4)).reshape(-1),
                               np.arange(4 * n, p + 1)]).astype(np.int32)
        got, cnt = orc.mask_tokens(mask)
        assert cnt == 4 * keep + (p + 1) % 4
        assert np.array_equal(got, want)


def test_gather_equals_fancy_indexing(orc):
    """Output row i is the pool row of token sel[i]: page table[t // page_size],
    slot t % page_size -- numpy fancy indexing on a shuffled page table."""
    rng = np.random.default_rng(13)
    page_size, width, pages = 16, 96, 40
    pool = rng.integers(0, 65535, size=(pages * page_size, width)).astype(np.uint16)
    table = rng.permutation(pages).astype(np.int32)[:30]
    sel = np.sort(rng.choice(30 * page_size, size=100, replace=False)).astype(np.int32)
    got, rc = orc.gather(pool, table, page_size, width, sel)
    assert rc == 0
    want = pool.reshape(pages, page_size, width)[table[sel // page_size], sel % page_size]
    assert np.array_equal(got, want)


def test_gather_refuses_tokens_past_the_table(orc):
    pool = np.zeros((32, 8), np.uint16)
    table = np.array([1, 0], np.int32)
    assert orc.gather(pool, table, 16, 8, np.array([31], np.int32))[1] == 0
    assert orc.gather(pool, table, 16, 8, np.array([32], np.int32))[1] == 1
    assert orc.gather(pool, table, 16, 8, np.array([-1], np.int32))[1] == 1

# --------------------------------------------------------------------------
# sparse attention over the selected tokens (atlas qsa_select.rs prefill_select)
# --------------------------------------------------------------------------

def bf16_ulp_close(got, want, ulps=1):
    """bf16 bit patterns within `ulps` units in the last place (same sign)."""
    g = np.asarray(got, np.uint16).astype(np.int32)
    w = np.asarray(want, np.uint16).astype(np.int32)
    return bool(np.all(np.abs(g - w) <= ulps))


def attn_case(rng, nq=4, nkv=2, hd=16, page_size=4, pages=12, table_len=10):
    k = qi.normal_bf16(rng, (pages * page_size, nkv * hd))
    v = qi.normal_bf16(rng, (pages * page_size, nkv * hd))
    table = rng.permutation(pages)[:table_len].astype(np.int32)
    q = qi.normal_bf16(rng, (nq * hd,))
    return q, k, v, table


def test_sparse_attn_one_token_is_its_value_row(orc):
    """One selected token: every head's output is that token's V row of the
    head's KV group (heads 0..G-1 read KV head 0, the next G KV head 1...)."""
    rng = np.random.default_rng(21)
    for nq, nkv in ((4, 2), (6, 3), (4, 1), (2, 2)):
        hd = 16
        q, k, v, table = attn_case(rng, nq, nkv, hd)
        t = 17
        out, rc = orc.sparse_attn(q, nq, nkv, hd, k, v, table, 4, np.array([t], np.int32), 0.25)
        assert rc == 0
        slot = table[t // 4] * 4 + t % 4
        vrow = v[slot].reshape(nkv, hd)
        for h in range(nq):
            assert np.array_equal(out.reshape(nq, hd)[h], vrow[h // (nq // nkv)]), (nq, nkv, h)


def test_sparse_attn_equal_logits_give_the_mean(orc):
    """q = 0 makes every logit equal: the output is the plain mean of the
    selected V rows (rounded to f32, then bf16)."""
    rng = np.random.default_rng(22)
    nq, nkv, hd, ps = 4, 2, 16, 4
    _, k, v, table = attn_case(rng, nq, nkv, hd, ps)
    q = np.zeros(nq * hd, np.uint16)
    sel = np.array([0, 3, 9, 21, 30, 39], np.int32)
    out, rc = orc.sparse_attn(q, nq, nkv, hd, k, v, table, ps, sel, 0.7)
    assert rc == 0
    slots = table[sel // ps] * ps + sel % ps
    vv = widen(v[slots]).astype(np.float64).reshape(len(sel), nkv, hd)
    for h in range(nq):
        mean = vv[:, h // 2, :].mean(axis=0).astype(np.float32)
        want = qi.to_bf16_bits(mean)
        assert bf16_ulp_close(out.reshape(nq, hd)[h], want), h


def test_sparse_attn_two_tokens_logistic_weights(orc):
    """Two tokens whose logits differ by D: weights sigmoid(D) and 1 - sigmoid(D)
    (the closed form of a two-way softmax), with D = scale * (q . (k1 - k2))."""
    nq, nkv, hd, ps = 2, 1, 8, 4
    table = np.arange(4, dtype=np.int32)
    k = np.zeros((16, hd), np.float32)
    v = np.zeros((16, hd), np.float32)
    k[5, 0], k[9, 0] = 1.5, -0.5
    v[5] = np.linspace(-1, 1, hd)
    v[9] = np.linspace(2, -3, hd)
    q = np.zeros((nq, hd), np.float32)
    q[0, 0], q[1, 0] = 2.0, -1.0
    scale = 0.375
    out, rc = orc.sparse_attn(qi.to_bf16_bits(q.ravel()), nq, nkv, hd, qi.to_bf16_bits(k),
                              qi.to_bf16_bits(v), table, ps, np.array([5, 9], np.int32), scale)
    assert rc == 0
    for h in range(nq):
        d = scale * q[h, 0] * (k[5, 0] - k[9, 0])
        w = 1.0 / (1.0 + math.exp(-d))
        want = qi.to_bf16_bits((w * v[5] + (1 - w) * v[9]).astype(np.float32))
        assert bf16_ulp_close(out.reshape(nq, hd)[h], want), h


def test_sparse_attn_scale_multiplies_the_logits(orc):
    """scale s with q equals scale 1 with s*q when s is a power of two (s*q is
    exact in bf16)."""
    rng = np.random.default_rng(23)
    nq, nkv, hd, ps = 4, 2, 16, 4
    q, k, v, table = attn_case(rng, nq, nkv, hd, ps)
    sel = np.array([1, 2, 6, 11, 25, 38], np.int32)
    a, _ = orc.sparse_attn(q, nq, nkv, hd, k, v, table, ps, sel, 0.25)
    q4 = qi.to_bf16_bits(widen(q) * np.float32(0.25))
    b, _ = orc.sparse_attn(q4, nq, nkv, hd, k, v, table, ps, sel, 1.0)
    assert np.array_equal(a, b)
    c, _ = orc.sparse_attn(q, nq, nkv, hd, k, v, table, ps, sel, 1.0)
    assert not np.array_equal(a, c)


def test_sparse_attn_reads_through_the_page_table(orc):
    """The same row through a shuffled page table and through the identity
    table over a pool whose pages numpy rearranged: identical outputs; and a
    permuted token list gives the same output up to summation order."""
    rng = np.random.default_rng(24)
    nq, nkv, hd, ps = 4, 2, 16, 4
    q, k, v, table = attn_case(rng, nq, nkv, hd, ps)
    sel = np.array([0, 5, 6, 7, 13, 22, 31, 39], np.int32)
    a, rc = orc.sparse_attn(q, nq, nkv, hd, k, v, table, ps, sel, 0.3)
    assert rc == 0
    kc = k.reshape(-1, ps, nkv * hd)[table].reshape(-1, nkv * hd)
    vc = v.reshape(-1, ps, nkv * hd)[table].reshape(-1, nkv * hd)
    b, _ = orc.sparse_attn(q, nq, nkv, hd, kc, vc, np.arange(len(table), dtype=np.int32), ps, sel,
                           0.3)
    assert np.array_equal(a, b)
    c, _ = orc.sparse_attn(q, nq, nkv, hd, k, v, table, ps, sel[::-1].copy(), 0.3)
    assert bf16_ulp_close(a, c)


def test_sparse_attn_refuses_tokens_past_the_table(orc):
    rng = np.random.default_rng(25)
    q, k, v, table = attn_case(rng)
    assert orc.sparse_attn(q, 4, 2, 16, k, v, table, 4, np.array([39], np.int32), 1.0)[1] == 0
    assert orc.sparse_attn(q, 4, 2, 16, k, v, table, 4, np.array([40], np.int32), 1.0)[1] == 1
    assert orc.sparse_attn(q, 4, 2, 16, k, v, table, 4, np.array([-2], np.int32), 1.0)[1] == 1
    out, rc = orc.sparse_attn(q, 4, 2, 16, k, v, table, 4, np.zeros(0, np.int32), 1.0)
    assert rc == 0 and not out.any()          # no selected token: zeros

# --------------------------------------------------------------------------
# the index_qk_proj projection y = x W^T (a dense bf16 linear layer)
# --------------------------------------------------------------------------

def test_proj_selecting_weights_copy_columns(orc):
    """W whose row n is the unit vector e_{perm(n)}: y[:, n] = x[:, perm(n)]
    exactly (a single exact product per output)."""
    rng = np.random.default_rng(31)
    hidden, out = 48, 16
    x = qi.normal_bf16(rng, (7, hidden))
    perm = rng.permutation(hidden)[:out]
    w = np.zeros((out, hidden), np.float32)
    w[np.arange(out), perm] = 1.0
    y, rc = orc.proj(x, qi.to_bf16_bits(w))
    assert rc == 0
    assert np.array_equal(y, x[:, perm])


def test_proj_matches_numpy_matmul(orc):
    """Against numpy's float64 matmul of the widened operands, rounded to f32
    then bf16 (equal up to the double summation order: at most one bf16 step)."""
    rng = np.random.default_rng(32)
    x = qi.normal_bf16(rng, (9, 200))
    w = qi.normal_bf16(rng, (24, 200), std=0.05)
    y, rc = orc.proj(x, w)
    assert rc == 0
    ref = (widen(x).astype(np.float64) @ widen(w).astype(np.float64).T).astype(np.float32)
    want = qi.to_bf16_bits(ref)
    assert np.all(np.abs(y.astype(np.int32) - want.astype(np.int32)) <= 1)
    assert np.mean(y == want) > 0.99


def test_proj_is_linear_in_powers_of_two(orc):
    """y(2x) = 2 y(x) and y(x, -W) = -y(x, W), bit for bit."""
    rng = np.random.default_rng(33)
    x = qi.normal_bf16(rng, (4, 64))
    w = qi.normal_bf16(rng, (8, 64))
    y, _ = orc.proj(x, w)
    y2, _ = orc.proj(qi.to_bf16_bits(widen(x) * 2), w)
    assert np.array_equal(widen(y2), widen(y) * 2)
    yn, _ = orc.proj(x, w ^ np.uint16(0x8000))
    assert np.array_equal(widen(yn), -widen(y))

MUTANTS = {
    "tokens_count_capped": ("    return n;\n}\n\n/*\n * [LAYER] metrale layers/qsa.rs decode_select's gather",
                            "    return n < cap ? n : cap;\n}\n\n/*\n * [LAYER] metrale layers/qsa.rs decode_select's gather"),
    "gather_page_not_scaled": ("(int64_t)table[t / page_size] * page_size + t % page_size",
                               "(int64_t)table[t / page_size] + t % page_size"),
    "gather_ignores_table": ("(int64_t)table[t / page_size] * page_size", "(int64_t)(t / page_size) * page_size"),
    "attn_heads_interleaved": ("const int32_t g = h / group;", "const int32_t g = h % nkv;"),
    "attn_no_scale": ("w[j] = d * scale;", "w[j] = d;"),
    "attn_slot_ignores_table": ("return (int64_t)table[page] * page_size + (t - page * page_size);",
                                "return (int64_t)page * page_size + (t - page * page_size);"),
    "attn_drops_last_token": ("for (int32_t j = 0; j < n_sel; ++j) {\n            const int32_t t = sel[j];\n            const uint16_t *v",
                              "for (int32_t j = 0; j + 1 < n_sel; ++j) {\n            const int32_t t = sel[j];\n            const uint16_t *v"),
    "attn_values_from_keys": ("const uint16_t *v = v_pool + (", "const uint16_t *v = k_pool + ("),
    "attn_no_normalisation": ("orc_narrow((float)(acc[e] / den))", "orc_narrow((float)acc[e])"),
    "proj_weight_transposed": ("const uint16_t *wn = w + (int64_t)n * hidden;",
                               "const uint16_t *wn = w + n;"),
    "proj_drops_last_k": ("for (int32_t k = 0; k < hidden; ++k)\n                acc +=",
                          "for (int32_t k = 0; k + 1 < hidden; ++k)\n                acc +="),
    "proj_rounds_through_bf16_early": ("acc += (double)orc_widen(xr[k]) * (double)orc_widen(wn[k]);",
                                       "acc = orc_round_bf16((float)(acc + (double)orc_widen(xr[k]) * (double)orc_widen(wn[k])));"),
    "drop_tail": ("mask_row[t] = 1;", "(void)t;"),
    "keep_one_fewer": ("for (int32_t i = 0; i < keep; ++i)", "for (int32_t i = 0; i < keep - 1; ++i)"),
    "keep_one_more": ("for (int32_t i = 0; i < keep; ++i)", "for (int32_t i = 0; i <= keep && i < blocks; ++i)"),
    "invert_order": ("if (a->v > b->v)\n        return -1;", "if (a->v < b->v)\n        return -2;"),
    "ties_descending_index": ("return (a->b < b->b) ? -1 : (a->b > b->b);", "return (a->b > b->b) ? -1 : (a->b < b->b);"),
    "ignore_causality": ("memset(mask_row, 1, (size_t)p + 1);", "memset(mask_row, 1, (size_t)tokens);"),
    "relu_after_sum": [("float s = ((rl[0] + rl[1]) + rl[2]) + rl[3];",
                        "float s = orc_relu(((rl[0] + rl[1]) + rl[2]) + rl[3]);"),
                       ("rl[h] = orc_relu((float)acc);", "rl[h] = (float)acc;")],
    "no_relu": ("rl[h] = orc_relu((float)acc);", "rl[h] = (float)acc;"),
    "rope_at_block_end": ("(int64_t)ORC_RATIO * b, cos_t", "(int64_t)ORC_RATIO * b + 3, cos_t"),
    "rope_sign_flip": ("out[i] = orc_narrow(a - b);", "out[i] = orc_narrow(a + b);"),
    "rope_pairs_wrong": ("float x2 = n[i + ORC_HALF];", "float x2 = n[i + 64];"),
    "weight_w_not_1pw": ("float gain = 1.0f + orc_widen(w[d]);", "float gain = orc_widen(w[d]);"),
    "pool_by_sum": ("float mean = (float)acc * 0.25f;", "float mean = (float)acc;"),
    "drop_eps": ("float r = 1.0f / sqrtf(ms + eps);", "float r = 1.0f / sqrtf(ms);"),
    "no_scale": ("out[b] = (float)((double)s / root);", "out[b] = s;"),
    "wrong_head_offset": ("orc_widen(q_prepped[h * ORC_HD + d])", "orc_widen(q_prepped[d])"),
    "transposed_key": ("* (double)orc_widen(k[d]);", "* (double)orc_widen(block_keys[(int64_t)d * ORC_HD + b]);"),
    "stride_ignored": ("acc += (double)orc_widen(k0[(int64_t)t * key_stride + d]);",
                       "acc += (double)orc_widen(k0[(int64_t)t * ORC_HD + d]);"),
    "cos_sin_swapped": ("float c = orc_widen(crow[i]);", "float c = orc_widen(srow[i]);"),
    "mean_kept_f32": ("m[d] = orc_round_bf16(mean);", "m[d] = mean;"),
    "qprep_unrotated": ("orc_norm_rope(x, q_norm_w, pos, cos_t, sin_t, eps, q_out + h * ORC_HD);",
                        "orc_norm_rope(x, q_norm_w, 0, cos_t, sin_t, eps, q_out + h * ORC_HD);"),
    "qprep_at_block_start": ("orc_qprep(q + (int64_t)i * q_stride, p, q_norm_w",
                             "orc_qprep(q + (int64_t)i * q_stride, p - p % ORC_RATIO, q_norm_w"),
}

# the pins that must catch the mistakes (each mutant must fail at least one)
PIN_TESTS = [
    test_select_exhaustive_tiny_rows, test_select_invariants, test_select_signed_zero_ties,
    test_select_golden_geometry, test_pool_constant_vector_closed_form,
    test_pool_weight_enters_as_one_plus_w, test_pool_eps_and_mean_closed_form,
    test_pool_mean_of_distinct_tokens, test_pool_stride_and_offset_indexing,
    test_pool_mean_is_cast_to_bf16_before_the_norm, test_pool_depends_on_the_bf16_mean_only,
    test_score_onehot_closed_form, test_score_relu_is_per_head,
    test_query_rotates_at_the_row_position,
    test_mask_tokens_equals_nonzero, test_mask_tokens_of_a_selection_is_the_pages_list,
    test_gather_equals_fancy_indexing, test_gather_refuses_tokens_past_the_table,
    test_sparse_attn_one_token_is_its_value_row, test_sparse_attn_equal_logits_give_the_mean,
    test_sparse_attn_two_tokens_logistic_weights, test_sparse_attn_scale_multiplies_the_logits,
    test_sparse_attn_reads_through_the_page_table, test_sparse_attn_refuses_tokens_past_the_table,
    test_proj_selecting_weights_copy_columns, test_proj_matches_numpy_matmul,
    test_proj_is_linear_in_powers_of_two,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    import oracle

    edits = MUTANTS[name]
    if isinstance(edits, tuple):
        edits = [edits]
    src = open(SRC).read()
    for before, after in edits:
        assert src.count(before) == 1, f"mutation anchor for {name} not unique"
        src = src.replace(before, after)
    path = tmp_path / f"mut_{name}.c"
    path.write_text(src)
    lib = oracle.load_from(oracle.compile_shared(str(path), str(tmp_path / f"mut_{name}.so")))
    mutant = oracle.Oracle(lib)
    caught = []
    for pin in PIN_TESTS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every pin"
