"""GPU parity of qsa_pool_blocks and qsa_score_rows against the oracle.

Pooled keys and scores must match within 5e-3 absolute + 1e-3 relative; the
pooling is built to reproduce the oracle's rounding points, so the tests also
report (and bound) how many pooled bf16 values differ at all.
"""
import numpy as np
import pytest
import torch

import qsa_inputs as qi
from qsa_cases import (EPS, THETA, assert_close, bf16_close, long_keys_case, oracle_scores,
                       prefill_case)

pytestmark = pytest.mark.gpu


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def host16(t):
    return t.cpu().numpy().view(np.uint16)


@pytest.fixture(scope="module")
def qsa():
    import sparse_attention_token_qsa_gb300 as m

    return m


@pytest.fixture(scope="module")
def tables(qsa):
    c, s = qsa.qsa_rope_tables(262144 + 8, THETA)
    return c, s, dev(c), dev(s)


def gpu_pool(qsa, tables, keys_flat_dev, key_stride, first, n, k_norm_w, total_blocks):
    c, s, cd, sd = tables
    out = torch.full((total_blocks, 128), 0x7FAB, dtype=torch.int16, device="cuda")
    qsa.qsa_pool_blocks(keys_flat_dev, key_stride, first, n, dev(k_norm_w), cd, sd, c.shape[0],
                        EPS, out)
    torch.cuda.synchronize()
    return host16(out)


def test_pool_fused_layout_prefill(qsa, orc, tables):
    case = prefill_case()
    T = case["T"]
    c, s, _, _ = tables
    nb = T // 4
    fq_dev = dev(case["fq"])
    got = gpu_pool(qsa, tables, fq_dev.view(-1)[512:], 640, 0, nb, case["k_norm_w"], nb)
    want = orc.pool_blocks(case["fq"].reshape(-1)[512:], 640, 0, nb, case["k_norm_w"], c, s, EPS)
    exact = bf16_close(got, want, "pooled keys (fused layout)")
    assert exact == got.size, f"{got.size - exact} pooled values differ from the oracle"


def test_pool_long_context_token_scaled(qsa, orc, tables):
    case = long_keys_case()
    keys = case["keys"]
    nb = keys.shape[0] // 4
    c, s, _, _ = tables
    got = gpu_pool(qsa, tables, dev(keys).view(-1), 128, 0, nb, case["k_norm_w"], nb)
    want = orc.pool_blocks(keys, 128, 0, nb, case["k_norm_w"], c, s, EPS)
    exact = bf16_close(got, want, "pooled keys (64k, per-token scales)")
    assert exact >= got.size - 2, f"{got.size - exact} pooled values differ from the oracle"


@pytest.mark.parametrize("first,n", [(0, 1), (5, 17), (1000, 333), (16383, 1)])
def test_pool_ranges_only_touch_their_blocks(qsa, orc, tables, first, n):
    case = long_keys_case()
    keys = case["keys"]
    c, s, _, _ = tables
    total = keys.shape[0] // 4
    kd = dev(keys)
    got = gpu_pool(qsa, tables, kd.view(-1)[4 * first * 128:], 128, first, n, case["k_norm_w"], total)
    want = orc.pool_blocks(keys[4 * first:], 128, first, n, case["k_norm_w"], c, s, EPS,
                           total_blocks=total)
    assert np.array_equal(got[first:first + n], want[first:first + n])
    untouched = np.ones(total, bool)
    untouched[first:first + n] = False
    assert np.all(got[untouched] == 0x7FAB)


def pooled_prefill(orc, case, c, s):
    nb = case["T"] // 4
    return orc.pool_blocks(case["fq"].reshape(-1)[512:], 640, 0, nb, case["k_norm_w"], c, s, EPS)


@pytest.mark.parametrize("path", [1, 2, 3])
def test_score_prefill_all_rows(qsa, orc, tables, path):
    """Every row of the 2304-token prefill, scored against the oracle's pooled keys;
    entries past each row's prefix keep their sentinel."""
    case = prefill_case()
    T = case["T"]
    c, s, cd, sd = tables
    keys = pooled_prefill(orc, case, c, s)
    cols = T // 4 + 4
    sc = torch.full((T, cols), -7.0, dtype=torch.float32, device="cuda")
    st = qsa.new_status()
    qsa.qsa_score_rows_with(dev(case["fq"]), 640, dev(case["pos"]), None, T, T,
                            dev(case["q_norm_w"]), cd, sd, c.shape[0], EPS, dev(keys), None, sc,
                            cols, st, path=path, workspace=qsa.new_workspace(T))
    assert qsa.qsa_read_status(st) == (0, 0)
    got = sc.cpu().numpy()
    want, res = oracle_scores(orc, case["fq"], 640, case["pos"], T, case["q_norm_w"], c, s, keys,
                              cols)
    assert all(rc == 0 for rc, _ in res)
    worst = assert_close(got, want, "prefill scores")
    assert worst < 5e-3


@pytest.mark.parametrize("path", [1, 3])
def test_score_decode_rows_long_context(qsa, orc, tables, path):
    """Decode rows at 64k (16384 blocks each), visible_len and key_base variants,
    on the SIMT and the streaming tcgen05 scorer."""
    case = long_keys_case()
    keys_raw = case["keys"]
    c, s, cd, sd = tables
    nb = keys_raw.shape[0] // 4
    keys = orc.pool_blocks(keys_raw, 128, 0, nb, case["k_norm_w"], c, s, EPS)
    rows = 8
    q = case["q"][:rows]
    pos = np.array([65535, 65534, 65280, 40000, 4, 3, 70, 65535], np.int32)
    vis = np.array([65536, 65533, 65281, 100, 5, 0, 71, 65532], np.int32)
    base = np.array([0, 0, 0, 0, 0, 0, 0, 0], np.int64)
    cols = 16384 + 12
    for use_vis, use_base in ((False, False), (True, False), (True, True)):
        sc = torch.full((rows, cols), -7.0, dtype=torch.float32, device="cuda")
        st = qsa.new_status()
        qsa.qsa_score_rows_with(dev(q), 512, dev(pos), dev(vis) if use_vis else None, rows,
                                65536, dev(case["q_norm_w"]), cd, sd, c.shape[0], EPS, dev(keys),
                                dev(base) if use_base else None, sc, cols, st, path=path)
        assert qsa.qsa_read_status(st) == (0, 0)
        got = sc.cpu().numpy()
        want, _ = oracle_scores(orc, q, 512, pos, 65536, case["q_norm_w"], c, s, keys, cols,
                                visible_len=vis if use_vis else None,
                                key_base=base if use_base else None)
        assert_close(got, want, f"decode scores vis={use_vis} base={use_base}")


@pytest.mark.parametrize("path", [0, 1, 3])
def test_score_key_base_per_sequence(qsa, orc, tables, path):
    """Rows of different sequences in one call: key_base selects each row's key set
    (the last row's blocks end the key buffer, so a scorer that read past them
    would read past the allocation)."""
    rng = qi.rng_for(3, salt=1)
    c, s, cd, sd = tables
    lens = [4000, 9000, 6001]
    kw = qi.normal_bf16(rng, (128,), 0.1)
    qw = qi.normal_bf16(rng, (128,), 0.1)
    pooled, base = [], []
    off = 0
    for L in lens:
        raw = qi.raw_keys(rng, L)
        pooled.append(orc.pool_blocks(raw, 128, 0, L // 4, kw, c, s, EPS))
        base.append(off)
        off += L // 4
    keys = np.concatenate(pooled)
    base = np.array(base, np.int64)
    pos = np.array([L - 1 for L in lens], np.int32)
    q = qi.fused_qk(rng, 3)[:, :512].copy()
    cols = 2252
    sc = torch.full((3, cols), -7.0, dtype=torch.float32, device="cuda")
    st = qsa.new_status()
    qsa.qsa_score_rows_with(dev(q), 512, dev(pos), None, 3, 9000, dev(qw), cd, sd, c.shape[0],
                            EPS, dev(keys), dev(base), sc, cols, st, path=path)
    assert qsa.qsa_read_status(st) == (0, 0)
    want, _ = oracle_scores(orc, q, 512, pos, 9000, qw, c, s, keys, cols, key_base=base)
    assert_close(sc.cpu().numpy(), want, "per-sequence scores")


@pytest.mark.parametrize("path", [1, 2, 3])
def test_score_nan_key_propagates(qsa, orc, tables, path):
    case = prefill_case(T=512)
    c, s, cd, sd = tables
    keys = pooled_prefill(orc, case, c, s)
    keys[37, 5] = 0x7FC0
    T = 512
    cols = 128
    sc = torch.full((T, cols), -7.0, dtype=torch.float32, device="cuda")
    st = qsa.new_status()
    qsa.qsa_score_rows_with(dev(case["fq"]), 640, dev(case["pos"]), None, T, T,
                            dev(case["q_norm_w"]), cd, sd, c.shape[0], EPS, dev(keys), None, sc,
                            cols, st, path=path, workspace=qsa.new_workspace(T))
    assert qsa.qsa_read_status(st) == (0, 0)
    got = sc.cpu().numpy()
    rows_seeing = np.arange(T)[(np.arange(T) + 1) // 4 > 37]
    assert np.all(np.isnan(got[rows_seeing, 37]))
    want, _ = oracle_scores(orc, case["fq"], 640, case["pos"], T, case["q_norm_w"], c, s, keys, cols)
    assert_close(got, want, "scores with a NaN key")


@pytest.mark.parametrize("path", [1, 3])
def test_score_row_range_errors(qsa, tables, path):
    c, s, cd, sd = tables
    q = torch.zeros((3, 640), dtype=torch.int16, device="cuda")
    keys = torch.zeros((64, 128), dtype=torch.int16, device="cuda")
    w = torch.zeros(128, dtype=torch.int16, device="cuda")
    for pos, vis, bad in (([0, 256, 1], None, 1), ([0, -1, 1], None, 1),
                          ([9, 9, 9], [10, 11, 4], 1)):
        sc = torch.full((3, 64), -7.0, dtype=torch.float32, device="cuda")
        st = qsa.new_status()
        qsa.qsa_score_rows_with(q, 640, dev(np.array(pos, np.int32)),
                                None if vis is None else dev(np.array(vis, np.int32)), 3, 256, w,
                                cd, sd, c.shape[0], EPS, keys, None, sc, 64, st, path=path)
        code, row = qsa.qsa_read_status(st)
        assert (code, row) == (3, bad)
        assert np.all(sc.cpu().numpy()[bad] == -7.0)


def test_score_stream_negative_key_base_is_a_row_error(qsa, orc, tables):
    """The streaming tcgen05 scorer reads only a row's own blocks and addresses
    them from key_base: a negative key_base is recorded as a row-range error for
    that row, which it leaves unwritten, and the other rows are scored."""
    c, s, cd, sd = tables
    rng = qi.rng_for(3, salt=77)
    keys = qi.normal_bf16(rng, (3 * 600, 128))
    q = qi.fused_qk(rng, 3)[:, :512].copy()
    qw = qi.normal_bf16(rng, (128,), 0.1)
    pos = np.array([2399, 1999, 2100], np.int32)
    base = np.array([0, -5, 1200], np.int64)
    cols = 604
    sc = torch.full((3, cols), -7.0, dtype=torch.float32, device="cuda")
    st = qsa.new_status()
    qsa.qsa_score_rows_with(dev(q), 512, dev(pos), None, 3, 2400, dev(qw), cd, sd, c.shape[0], EPS,
                            dev(keys), dev(base), sc, cols, st, path=qsa.QSA_SCORE_STREAM)
    assert qsa.qsa_read_status(st) == (3, 1)
    got = sc.cpu().numpy()
    assert np.all(got[1] == -7.0)
    ok_rows = np.array([0, 2])
    want, _ = oracle_scores(orc, q[ok_rows], 512, pos[ok_rows], 2400, qw, c, s, keys, cols,
                            key_base=base[ok_rows])
    assert_close(got[ok_rows], want, "rows beside the bad key_base")


@pytest.mark.parametrize("n_rows,tokens,seed", [(100, 3000, 1), (64, 520, 2), (1, 9000, 3),
                                                (257, 4100, 4)])
def test_score_tc_ragged_tiles(qsa, orc, tables, n_rows, tokens, seed):
    """Tensor-core scorer on ragged shapes: rows not a multiple of the 64-row tile,
    block counts not a multiple of the 128-block tile, arbitrary positions and
    visible lengths (including empty prefixes), one invalid row."""
    rng = qi.rng_for(2, salt=seed)
    c, s, cd, sd = tables
    raw = qi.raw_keys(rng, tokens)
    qw, kw = qi.norm_weights(rng)
    nb = tokens // 4
    keys = orc.pool_blocks(raw, 128, 0, nb, kw, c, s, EPS)
    q = qi.fused_qk(rng, n_rows)
    pos = rng.integers(0, tokens, size=n_rows).astype(np.int32)
    pos[: min(4, n_rows)] = np.arange(min(4, n_rows))
    vis = (pos + 1).astype(np.int32)
    cut = rng.random(n_rows) < 0.3
    vis[cut] = rng.integers(0, pos[cut] + 2).astype(np.int32)
    cols = nb + 4 - nb % 4 + 4
    sc = torch.full((n_rows, cols), -7.0, dtype=torch.float32, device="cuda")
    st = qsa.new_status()
    ws = qsa.new_workspace(n_rows)
    qsa.qsa_score_rows_with(dev(q), 640, dev(pos), dev(vis), n_rows, tokens, dev(qw), cd, sd,
                            c.shape[0], EPS, dev(keys), None, sc, cols, st, path=2, workspace=ws)
    assert qsa.qsa_read_status(st) == (0, 0)
    want, _ = oracle_scores(orc, q, 640, pos, tokens, qw, c, s, keys, cols, visible_len=vis)
    assert_close(sc.cpu().numpy(), want, f"tcgen05 scores {n_rows}x{tokens}")
    if n_rows >= 3:   # an out-of-range row is reported and left untouched
        pos_bad = pos.copy()
        pos_bad[2] = tokens
        sc.fill_(-7.0)
        st = qsa.new_status()
        qsa.qsa_score_rows_with(dev(q), 640, dev(pos_bad), None, n_rows, tokens, dev(qw), cd, sd,
                                c.shape[0], EPS, dev(keys), None, sc, cols, st, path=2,
                                workspace=ws)
        assert qsa.qsa_read_status(st) == (3, 2)
        got = sc.cpu().numpy()
        assert np.all(got[2] == -7.0)
        want2, _ = oracle_scores(orc, q, 640, pos, tokens, qw, c, s, keys, cols)
        keep = np.ones(n_rows, bool)
        keep[2] = False
        assert_close(got[keep], want2[keep], "tcgen05 scores beside a bad row")


def test_score_tc_chunk_64k_sampled(qsa, orc, tables):
    """Chunked prefill: 4096 rows at positions 61440..65535 of a 64k sequence,
    the [16384, 128] x [128, 16384] contraction; sampled rows against the oracle,
    the sentinel on every row past its prefix."""
    rng = qi.rng_for(2)
    c, s, cd, sd = tables
    tokens, first, rows = 65536, 61440, 4096
    raw = qi.raw_keys(rng, tokens)
    qw, kw = qi.norm_weights(rng)
    keys_d = torch.zeros((tokens // 4, 128), dtype=torch.int16, device="cuda")
    qsa.qsa_pool_blocks(dev(raw).view(-1), 128, 0, tokens // 4, dev(kw), cd, sd, c.shape[0], EPS,
                        keys_d)
    keys = keys_d.cpu().numpy().view(np.uint16)
    q = qi.fused_qk(rng, rows)
    pos = np.arange(first, first + rows, dtype=np.int32)
    cols = tokens // 4
    sc = torch.full((rows, cols), -7.0, dtype=torch.float32, device="cuda")
    st = qsa.new_status()
    qsa.qsa_score_rows(dev(q), 640, dev(pos), None, rows, tokens, dev(qw), cd, sd, c.shape[0], EPS,
                       keys_d, None, sc, cols, st, workspace=qsa.new_workspace(rows))
    assert qsa.qsa_read_status(st) == (0, 0)
    got = sc.cpu().numpy()
    n = (pos + 1) // 4
    for i in range(rows):
        assert np.all(got[i, n[i]:] == -7.0)
    sample = np.unique(np.concatenate([np.arange(0, 4), np.arange(60, 68), np.arange(rows - 4, rows),
                                       rng.choice(rows, 40, replace=False)]))
    want, _ = oracle_scores(orc, q[sample], 640, pos[sample], tokens, qw, c, s, keys, cols)
    assert_close(got[sample], want, "64k chunk scores (sampled rows)")


def test_score_tc_rows_past_one_slab(qsa, orc, tables):
    """More rows than one launch of the tensor-core scorer balances (65536):
    the rows go in two slabs, the second launched behind the first; rows on
    both sides of the slab edge against the oracle, an invalid row in the
    second slab reported with its global index."""
    rng = qi.rng_for(2, salt=66)
    c, s, cd, sd = tables
    tokens, rows = 1024, 65536 + 200
    raw = qi.raw_keys(rng, tokens)
    qw, kw = qi.norm_weights(rng)
    nb = tokens // 4
    keys = orc.pool_blocks(raw, 128, 0, nb, kw, c, s, EPS)
    q = qi.fused_qk(rng, rows)
    pos = rng.integers(0, tokens, size=rows).astype(np.int32)
    bad = 65536 + 17
    pos[bad] = tokens                       # out of range, in the second slab
    cols = nb
    sc = torch.full((rows, cols), -7.0, dtype=torch.float32, device="cuda")
    st = qsa.new_status()
    qsa.qsa_score_rows_with(dev(q), 640, dev(pos), None, rows, tokens, dev(qw), cd, sd,
                            c.shape[0], EPS, dev(keys), None, sc, cols, st, path=2,
                            workspace=qsa.new_workspace(rows))
    assert qsa.qsa_read_status(st) == (3, bad)
    got = sc.cpu().numpy()
    assert np.all(got[bad] == -7.0)
    sample = np.array([0, 1, 65470, 65535, 65536, 65537, 65560, rows - 1])
    want, _ = oracle_scores(orc, q[sample], 640, pos[sample], tokens, qw, c, s, keys, cols)
    assert_close(got[sample], want, "scores on both sides of the slab edge")


def test_pool_rounds_the_mean_to_bf16_like_the_oracle(qsa, orc, tables):
    """The closed-form case where the bf16 cast of the f32 mean decides the key
    bits (a tie after the gain): the GPU must give the oracle's bits, at block 0
    (no rotation) and at later blocks (rotated at 4b)."""
    import test_oracle_pins as pins

    k, w = pins.mean_cast_case()
    nb = 9
    keys = np.tile(k, (nb, 1))
    c, s, cd, sd = tables
    out = torch.full((nb, 128), 0x7FAB, dtype=torch.int16, device="cuda")
    qsa.qsa_pool_blocks(dev(keys).view(-1), 128, 0, nb, dev(w), cd, sd, c.shape[0], 0.0, out)
    got = host16(out)
    want = orc.pool_blocks(keys, 128, 0, nb, w, c, s, 0.0)
    small = qi.to_bf16_bits(np.array([2.0**-13 * 1.515625], np.float32))[0]
    assert np.all(got[0, :126] == small)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("path", [1, 2, 3])
def test_score_one_hot_queries_rotate_at_their_positions(qsa, orc, tables, path):
    """One-hot query heads on dim i against one-hot keys e_i and e_{i+32}: the
    two scores are the rotated query's cos and sin components, so they pin the
    query's RoPE position on both scorers (oracle closed form in the pins)."""
    c, s, cd, sd = tables
    T = 4096
    cases = [(p, i) for p in (9, 14, 37, 101, 250, 399, 2050, 4095) for i in (0, 1, 7, 31)]
    n = len(cases)
    # 64 rows or more keep the tensor-core path on its own shape; pad with copies
    reps = -(-64 // n)
    cases = (cases * reps)[:max(64, n)]
    n = len(cases)
    fq = np.zeros((n, 640), np.float32)
    for r, (p, i) in enumerate(cases):
        fq[r, [i, 128 + i, 256 + i, 384 + i]] = 1.0
    fqb = qi.to_bf16_bits(fq)
    pos = np.array([p for p, _ in cases], np.int32)
    zero_w = np.zeros(128, np.uint16)
    cols = T // 4
    for i in sorted({i for _, i in cases}):
        keys = np.zeros((T // 4, 128), np.float32)
        keys[0, i], keys[1, i + 32] = 1.0, 1.0
        keys = qi.to_bf16_bits(keys)
        rows = np.array([r for r, (_, ii) in enumerate(cases) if ii == i])
        vis = np.full(n, 8, np.int32)
        sc = torch.full((n, cols), -7.0, dtype=torch.float32, device="cuda")
        st = qsa.new_status()
        qsa.qsa_score_rows_with(dev(fqb), 640, dev(pos), dev(vis), n, T, dev(zero_w), cd, sd,
                                c.shape[0], 0.0, dev(keys), None, sc, cols, st, path=path,
                                workspace=qsa.new_workspace(n))
        assert qsa.qsa_read_status(st) == (0, 0)
        got = sc.cpu().numpy()[rows]
        want = np.full((len(rows), cols), -7.0, np.float32)
        rc, _ = orc.score_rows(fqb[rows], 640, pos[rows], len(rows), T, zero_w, c, s, 0.0, keys,
                               want, cols, visible_len=vis[rows])
        assert rc == 0
        assert_close(got, want, f"one-hot query scores, dim {i}", atol=0, rtol=1e-6)
        assert np.all(got[:, 2:] == -7.0)


def _bf16_bits(x):
    """bf16 bits of float32 values that bf16 represents exactly."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32)
    assert np.all(b & 0xFFFF == 0), "value not representable in bf16"
    return (b >> 16).astype(np.uint16)


def special_sum_keys(n_blocks=4096, seed=11):
    """Raw keys whose 4-token sums exercise both ways the pool kernel forms the
    exact sum: plain f32 adds when a dim's four magnitudes lie within 2^14 of
    each other and below 2^125, the TwoSum cascade otherwise.  Block kinds
    cycle with the block index, so a warp (two blocks) mixes kinds; per-dim
    draws make some warps take the plain adds and others not."""
    rng = np.random.default_rng(seed)
    q = lambda v: (np.asarray(v, np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)
    out = np.empty((n_blocks * 4, 128), np.float32)
    for b in range(n_blocks):
        kind = b % 8      # a warp pools blocks 2w and 2w + 1: kinds (0,1) (2,3) (4,5) (6,7)
        if kind in (0, 5):  # ordinary values
            v = rng.standard_normal((4, 128))
        elif kind == 1:    # magnitudes exactly 2^14 apart: the plain adds' edge, still exact
            e = rng.integers(-20, 20, (1, 128))
            v = np.ldexp(1.0, e) * np.array([[1.0], [2.0 ** -14], [-1.0], [2.0 ** -7]])
        elif kind == 2:    # signed zeros only (the sum is +0)
            v = np.where(rng.random((4, 128)) < 0.5, -0.0, 0.0)
        elif kind == 3:    # bf16 subnormals next to small normals
            v = np.ldexp(rng.integers(1, 128, (4, 128)).astype(np.float64), -133)
            v[0] *= np.where(rng.random(128) < 0.5, 1, 2 ** 6)
        elif kind == 4:    # large (squares still finite in f32), cancelling
            v = np.ldexp(rng.choice([1.0, -1.0, 1.5, -1.25], (4, 128)), rng.integers(50, 60, (4, 128)))
        elif kind == 6:    # 2^23 apart: TwoSum, where plain f32 adds would round
            e = rng.integers(-20, 20, (1, 128))
            v = np.ldexp(1.0, e) * np.array([[1.0], [2.0 ** -23 * 1.0078125], [1.0], [2.0 ** -31]])
        else:              # wide random exponents, one zero
            v = np.ldexp(rng.standard_normal((4, 128)), rng.integers(-30, 30, (4, 128)))
            v[rng.integers(0, 4)] = 0.0
        out[4 * b:4 * b + 4] = q(v)
    return _bf16_bits(out)


def test_pool_sum_paths_bit_exact(qsa, orc, tables):
    keys = special_sum_keys()
    nb = keys.shape[0] // 4
    c, s, _, _ = tables
    kw = qi.norm_weights(qi.rng_for(3))[1]
    got = gpu_pool(qsa, tables, dev(keys).view(-1), 128, 0, nb, kw, nb)
    want = orc.pool_blocks(keys, 128, 0, nb, kw, c, s, EPS)
    assert np.array_equal(got, want), f"{int(np.sum(got != want))} pooled values differ"


def test_tile_and_streaming_tcgen05_scorers_agree_bit_for_bit(qsa, tables):
    """The tile scorer (M128 N256: 64 rows x 4 heads) and the streaming scorer
    (M128 N16: one row's 4 heads) run the same per-(block, head) MMA over K and
    the same epilogue, so their scores are identical, bit for bit, on every
    row shape (full tiles, a partial last tile, short and empty prefixes)."""
    c, s, cd, sd = tables
    rng = qi.rng_for(3, salt=99)
    T = 65536
    nb = T // 4
    keys = qi.torch_normal_bf16(torch, (nb, 128), qi.seed_for(3, 98), "cuda")
    rows = 70
    q = qi.fused_qk(rng, rows)
    qw = qi.normal_bf16(rng, (128,), 0.1)
    pos = rng.integers(0, T, size=rows).astype(np.int32)
    pos[:4] = [T - 1, 0, 3, 511]
    out = []
    for path in (qsa.QSA_SCORE_TCGEN05, qsa.QSA_SCORE_STREAM):
        sc = torch.full((rows, nb), -7.0, dtype=torch.float32, device="cuda")
        st = qsa.new_status()
        qsa.qsa_score_rows_with(dev(q), 640, dev(pos), None, rows, T, dev(qw), cd, sd, c.shape[0],
                                EPS, keys, None, sc, nb, st, path=path,
                                workspace=qsa.new_workspace(rows))
        assert qsa.qsa_read_status(st) == (0, 0)
        out.append(sc.cpu().numpy())
    assert np.array_equal(out[0].view(np.uint32), out[1].view(np.uint32))
