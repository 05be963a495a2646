"""GPU parity of qsa_select_mask against the oracle: bit-exact masks.

The selection is integer work over the oracle's own f32 scores, so every case
compares whole mask rows byte for byte.
"""
import numpy as np
import pytest
import torch

import qsa_inputs as qi
from qsa_cases import check_mask_structure, oracle_masks

pytestmark = pytest.mark.gpu


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


@pytest.fixture(scope="module")
def qsa():
    import sparse_attention_token_qsa_gb300 as m

    return m


def gpu_select(qsa, scores, score_cols, pos, tokens, budget, mask_offset=0, expect=0):
    n_rows = len(pos)
    s = dev(scores)
    p = dev(np.asarray(pos, np.int32))
    buf = torch.full((n_rows * tokens + mask_offset + 16,), 0xAB, dtype=torch.uint8, device="cuda")
    mask = buf[mask_offset:mask_offset + n_rows * tokens]
    st = qsa.new_status()
    qsa.qsa_select_mask(s, score_cols, p, n_rows, tokens, budget, mask, st)
    code, row = qsa.qsa_read_status(st)
    assert code == expect, (code, row)
    out = mask.view(n_rows, tokens).cpu().numpy()
    # guard bytes around the mask are untouched
    g = buf.cpu().numpy()
    assert np.all(g[:mask_offset] == 0xAB) and np.all(g[mask_offset + n_rows * tokens:] == 0xAB)
    return out, row


def test_select_stress_ties_all_budgets(qsa, orc):
    """Selection-only stress at 256k: relu-sum-like scores, 70% exact zeros (half
    -0.0), the rest on 64 levels; every budget the stress names.  96 rows split
    over clusters of 4 are enough CTAs for the many-row block shape."""
    rng = qi.rng_for(4)
    rows, tokens = 96, 262144
    cols = tokens // 4
    scores = qi.stress_scores(rng, rows, cols)
    pos = np.full(rows, tokens - 1, np.int32)
    pos[1::3] = tokens - 2          # 65535 blocks, tail 3
    pos[2::3] = tokens - 7          # 65534 blocks, tail 2
    for budget in (4, 512, 2048, 2044):
        got, _ = gpu_select(qsa, scores, cols, pos, tokens, budget)
        want, codes = oracle_masks(orc, scores, cols, pos, tokens, budget)
        assert all(c == 0 for c in codes)
        for r in range(rows):
            assert np.array_equal(got[r], want[r]), (budget, r)


def test_select_many_long_rows_one_cta_each(qsa, orc):
    """More rows than two waves of CTAs at 256k: each 65536-block row runs on one
    CTA of the shape without a key cache (no cluster), stress scores with massive
    ties, and rows of every tail."""
    rng = qi.rng_for(4, salt=320)
    rows, tokens = 320, 262144
    cols = tokens // 4
    scores = qi.stress_scores(rng, rows, cols, zero_frac=0.5, levels=256)
    pos = np.full(rows, tokens - 1, np.int32)
    pos[1::4] = tokens - 2
    pos[2::4] = tokens - 3
    pos[3::4] = rng.integers(2051, tokens, size=len(pos[3::4]))
    for budget in (2048, 4):
        got, _ = gpu_select(qsa, scores, cols, pos, tokens, budget)
        want, codes = oracle_masks(orc, scores, cols, pos, tokens, budget)
        assert all(c == 0 for c in codes)
        bad = [r for r in range(rows) if not np.array_equal(got[r], want[r])]
        assert not bad, (budget, bad[:8])


@pytest.mark.parametrize("k", [16, 17, 40])
def test_select_many_rows_candidates_crowding_one_thread(qsa, orc, k):
    """Many 16384-block rows (one CTA each, no key cache): the threshold bin's
    keys sit in the positions one thread of the compaction pass reads (block
    1024 j + e), k of them; 16 fit that thread's candidate slots, more send
    the row to the rounds over every key.  Every fourth row is plain random;
    tails of 0, 3 and 2 tokens."""
    rng = qi.rng_for(4, salt=900 + k)
    rows, tokens = 320, 65536
    cols = tokens // 4
    scores = rng.random((rows, cols), dtype=np.float32)
    pos = (tokens - 1 - (np.arange(rows) % 3)).astype(np.int32)
    crowd = (1024 * np.arange(16)[:, None] + np.arange(4)[None, :]).ravel()   # one thread's keys
    for r in range(rows):
        if r % 4 == 3:
            continue
        n = (int(pos[r]) + 1) // 4
        top = rng.choice(np.setdiff1d(np.arange(n), crowd), size=500, replace=False)
        scores[r, top] = rng.uniform(4.0, 8.0, size=500).astype(np.float32)
        at = rng.choice(crowd[crowd < n], size=k, replace=False)
        scores[r, at] = (2.0 + np.arange(k) * 2.0 ** -10).astype(np.float32)   # one 12-bit bin
    got, _ = gpu_select(qsa, scores, cols, pos, tokens, 2048)
    want, codes = oracle_masks(orc, scores, cols, pos, tokens, 2048)
    assert all(c == 0 for c in codes)
    bad = [r for r in range(rows) if not np.array_equal(got[r], want[r])]
    assert not bad, bad[:8]


def test_select_prefill_rows_with_injected_ties(qsa, orc):
    """Single-sequence prefill geometry (T=2304): every row, all-kept rows below
    the inert bound and truncating rows above it; 32 truncating rows get exact
    ties at their cut and ~30% +-0.0 scores."""
    rng = qi.rng_for(0, salt=7)
    T = 2304
    cols = T // 4
    scores = rng.standard_normal((T, cols)).astype(np.float32) * 2.0
    scores = np.maximum(scores, 0).astype(np.float32)
    pos = np.arange(T, dtype=np.int32)
    trunc = np.arange(2051, T)
    for r in rng.choice(trunc, size=32, replace=False):
        n = (r + 1) // 4
        qi.sprinkle_signed_zeros(scores[r], rng, 0.3, n)
        cut = np.sort(np.where(scores[r, :n] == 0, 0, scores[r, :n]))[::-1][511]
        qi.set_blocks_to(scores[r], rng, np.float32(cut), int(rng.integers(8, 41)), n)
    got, _ = gpu_select(qsa, scores, cols, pos, T, 2048)
    want, codes = oracle_masks(orc, scores, cols, pos, T, 2048)
    assert all(c == 0 for c in codes)
    bad = [r for r in range(T) if not np.array_equal(got[r], want[r])]
    assert not bad, bad[:10]
    for r in (0, 1, 2, 3, 2046, 2047, 2050, 2051, 2054, T - 1):
        check_mask_structure(got[r], r, T, 2048)


def test_select_all_zero_rows_fill_in_index_order(qsa, orc):
    tokens = 8192
    cols = tokens // 4
    scores = np.zeros((6, cols), np.float32)
    scores[1, ::2] = -0.0
    pos = np.array([8191, 8191, 4096, 2051, 3000, 8190], np.int32)
    got, _ = gpu_select(qsa, scores, cols, pos, tokens, 2048)
    want, _ = oracle_masks(orc, scores, cols, pos, tokens, 2048)
    assert np.array_equal(got, want)
    assert np.all(got[0, :2048] == 1) and np.all(got[0, 2048:] == 0)


@pytest.mark.parametrize("tokens,offset", [(1000, 0), (1003, 1), (4099, 3), (65536, 5), (70001, 2)])
def test_select_ragged_rows_and_unaligned_masks(qsa, orc, tokens, offset):
    """Rows of every length in one launch, tokens not a multiple of 16, mask rows
    at odd byte offsets, score_cols with spare capacity."""
    rng = qi.rng_for(4, salt=tokens)
    rows = 64
    cols = ((tokens // 4 + 3) // 4) * 4 + 8
    scores = qi.stress_scores(rng, rows, cols, zero_frac=0.3, levels=16)
    pos = rng.integers(0, tokens, size=rows).astype(np.int32)
    pos[:6] = [0, 1, 2, 3, tokens - 1, min(tokens - 1, 2050)]
    for budget in (4, 64, 2048):
        got, _ = gpu_select(qsa, scores, cols, pos, tokens, budget, mask_offset=offset)
        want, codes = oracle_masks(orc, scores, cols, pos, tokens, budget)
        assert all(c == 0 for c in codes)
        for r in range(rows):
            assert np.array_equal(got[r], want[r]), (budget, r, pos[r])


@pytest.mark.parametrize("rows", [1, 2, 8, 40])
def test_select_cluster_split_rows(qsa, orc, rows):
    """Few long rows split over clusters of CTAs (decode shapes at 64k and 256k)."""
    rng = qi.rng_for(3, salt=rows)
    tokens = 262144 if rows <= 8 else 65536
    cols = tokens // 4
    scores = np.maximum(rng.standard_normal((rows, cols)).astype(np.float32), 0)
    scores[:, rng.choice(cols, 50, replace=False)] = scores[0, 7]        # ties across slices
    pos = rng.integers(tokens // 2, tokens, size=rows).astype(np.int32)
    pos[0] = tokens - 1
    got, _ = gpu_select(qsa, scores, cols, pos, tokens, 2048)
    want, _ = oracle_masks(orc, scores, cols, pos, tokens, 2048)
    for r in range(rows):
        assert np.array_equal(got[r], want[r]), r


@pytest.mark.parametrize("rows", [3, 32])
@pytest.mark.parametrize("kind", ["plateau", "plateau_one_slice", "low_bits", "stress", "nonfinite",
                                  "skewed", "sparse_top"])
def test_select_cluster_rows_rounds_and_ties(qsa, orc, kind, rows):
    """Few long rows on clusters of the key-caching shape (3 rows: 8 CTAs each,
    32 rows: 4 each), where every CTA runs the candidate rounds on its own list.
    A plateau of equal keys straddling the cut, spread over every rank's slice
    or inside one slice (the cut placed by the ranks' tie counts); keys that
    differ only in their last four bits (every round, then the final one-key
    check); stress scores; a non-finite score in a middle rank's slice; one
    slice holding every large score, so the other CTAs' first window over the
    round-0 bins misses the row's highest bin; and 300 huge scores over tiny
    ones, so the window holds too few keys for budgets above 1200."""
    rng = qi.rng_for(4, salt=1000 + rows)
    tokens = 262144
    cols = tokens // 4
    pos = np.full(rows, tokens - 1, np.int32)
    pos[1::3] = tokens - 2
    pos[2::3] = tokens - 7 - 4 * rng.integers(0, 30000, size=len(pos[2::3]))
    if kind == "stress":
        scores = qi.stress_scores(rng, rows, cols)
    elif kind == "skewed":
        scores = rng.random((rows, cols), dtype=np.float32)
        for r in range(rows):
            n = (int(pos[r]) + 1) // 4
            scores[r, 3 * n // 4:n] *= np.float32(2.0 ** 40)
    elif kind == "sparse_top":
        scores = rng.random((rows, cols), dtype=np.float32) * np.float32(2.0 ** -100)
        for r in range(rows):
            n = (int(pos[r]) + 1) // 4
            hi = rng.choice(n, 300, replace=False)
            scores[r, hi] = (np.float32(1.0) + rng.random(300, dtype=np.float32)) * np.float32(2.0 ** 100)
    else:
        scores = rng.random((rows, cols), dtype=np.float32)
        for r in range(rows):
            n = (int(pos[r]) + 1) // 4
            hi = rng.choice(n, 300, replace=False)            # kept outright
            scores[r, hi] = np.float32(2.0) + rng.random(300, dtype=np.float32)
            if kind == "plateau_one_slice":                    # 600 blocks inside one slice
                start = int(rng.integers(n // 3, n // 3 + 2000))
                mid = np.setdiff1d(np.arange(start, start + 1200, 2), hi)[:600]
            else:
                mid = np.setdiff1d(rng.choice(n, 900, replace=False), hi)[:600]
            if kind == "low_bits":
                bits = np.float32(1.5).view(np.uint32) + rng.integers(0, 16, size=len(mid)).astype(np.uint32)
                scores[r, mid] = bits.astype(np.uint32).view(np.float32)
            else:
                scores[r, mid] = np.float32(1.5)
    expect_row = None
    if kind == "nonfinite":
        scores[1, 40000] = np.nan
        expect_row = 1
    for budget in (512, 2044, 2048):
        got, row = gpu_select(qsa, scores, cols, pos, tokens, budget, expect=4 if expect_row else 0)
        want, codes = oracle_masks(orc, scores, cols, pos, tokens, budget)
        for r in range(rows):
            if r == expect_row:
                assert row == r and codes[r] == 4
                assert np.all((got[r] == 0xAB) | (got[r] <= 1))   # unspecified, within the row
            else:
                assert np.array_equal(got[r], want[r]), (kind, budget, r, pos[r])


def test_select_low_byte_differences_and_deep_truncation(qsa, orc):
    """Keys that differ only in their lowest byte, and budget 4 at 256k."""
    rng = qi.rng_for(4, salt=99)
    tokens = 262144
    cols = tokens // 4
    base = np.float32(1.5).view(np.uint32)
    bits = (base + rng.integers(0, 256, size=(2, cols)).astype(np.uint32)).astype(np.uint32)
    scores = bits.view(np.float32)
    pos = np.array([tokens - 1, tokens - 3], np.int32)
    for budget in (4, 2048, 1028):
        got, _ = gpu_select(qsa, scores, cols, pos, tokens, budget)
        want, _ = oracle_masks(orc, scores, cols, pos, tokens, budget)
        assert np.array_equal(got, want), budget


def test_select_nonfinite_row_reported_and_untouched(qsa, orc):
    tokens = 16384
    cols = tokens // 4
    rng = qi.rng_for(4, salt=5)
    scores = rng.random((4, cols)).astype(np.float32)
    scores[2, 1000] = np.nan
    scores[0, 3] = np.inf     # row 0 is all-kept: its scores are not read
    pos = np.array([1000, 16383, 16383, 9000], np.int32)
    got, row = gpu_select(qsa, scores, cols, pos, tokens, 2048, expect=4)
    assert row == 2
    assert np.all((got[2] == 0xAB) | (got[2] <= 1))   # unspecified, within the row
    want, codes = oracle_masks(orc, scores, cols, pos, tokens, 2048)
    assert codes == [0, 0, 4, 0]
    for r in (0, 1, 3):
        assert np.array_equal(got[r], want[r])


@pytest.mark.parametrize("bits", [0x7F800000, 0xFF800000, 0x7FC00001, 0xFFC00000, 0xFF800001])
def test_select_each_nonfinite_kind_reported(qsa, orc, bits):
    """+inf, -inf, a positive and two negative NaNs: each one, anywhere in a
    truncating row's prefix, is an error for that row alone; the same value
    past the row's prefix, or in an all-kept row, is never read."""
    tokens = 65536
    cols = tokens // 4
    rng = qi.rng_for(4, salt=bits & 0xFFFF)
    scores = rng.random((4, cols)).astype(np.float32)
    bad = np.array([bits], np.uint32).view(np.float32)[0]
    scores[1, 12345] = bad     # inside row 1's prefix
    scores[2, 15000] = bad     # past row 2's prefix (pos 40000 -> 10000 blocks)
    scores[3, 100] = bad       # row 3 keeps every block: its scores are not read
    pos = np.array([65535, 65535, 40000, 2000], np.int32)
    got, row = gpu_select(qsa, scores, cols, pos, tokens, 2048, expect=4)
    assert row == 1
    assert np.all((got[1] == 0xAB) | (got[1] <= 1))   # unspecified, within the row
    want, codes = oracle_masks(orc, scores, cols, pos, tokens, 2048)
    assert codes == [0, 4, 0, 0]
    for r in (0, 2, 3):
        assert np.array_equal(got[r], want[r])


def test_select_row_out_of_range_reported(qsa):
    tokens = 4096
    cols = tokens // 4
    scores = np.ones((3, cols), np.float32)
    pos = np.array([5, 4096, 7], np.int32)
    got, row = gpu_select(qsa, scores, cols, pos, tokens, 2048, expect=3)
    assert row == 1 and np.all(got[1] == 0xAB)
    assert np.all(got[0, :6] == 1) and np.all(got[0, 6:] == 0)


# ---- rows built to defeat the sampled band (the kernel then selects the row
# again from its full histogram): the sample is 8 * NT scores in runs of 8
# starting at ((t * (n - 8)) // (NT - 1)) & ~7 for t < NT, NT = 256 or 512


def sampled_blocks(n):
    """Every block a sampled-band pass could read: runs of `run` scores starting
    at (t * (n - run)) // (nt - 1), rounded down to 4 (or 8), for each thread t
    of either block shape and each run length the kernel may use."""
    hit = np.zeros(n, bool)
    for nt in (256, 512):
        t = np.arange(nt, dtype=np.int64)
        for run in (8, 16, 32):
            for align in (3, 7):
                at = ((t * (n - run)) // (nt - 1)) & ~align
                hit[(at[:, None] + np.arange(run)[None, :]).ravel()] = True
    return hit


def band_rows(rng, rows, n, kind):
    s = rng.random((rows, n)).astype(np.float32)          # U(0, 1)
    free = np.flatnonzero(~sampled_blocks(n))
    for r in range(rows):
        if kind == "unsampled_top":      # 2000 tied top scores, none in the sample
            s[r, rng.choice(free, 2000, replace=False)] = 10.0
        elif kind == "exact_upper_edge":  # 512 top scores unseen, 2000 below them seen
            s[r, rng.choice(n, 2000, replace=False)] = 5.0
            s[r, rng.choice(free, 512, replace=False)] = 10.0
        elif kind == "band_overflow":     # the keep-th score in a bin of 6000 ties
            s[r, rng.choice(n, 6000, replace=False)] = 5.0
            s[r, rng.choice(n, 100, replace=False)] = 10.0
    return s


@pytest.mark.parametrize("kind", ["unsampled_top", "exact_upper_edge", "band_overflow"])
def test_select_rows_that_mislead_the_sample(qsa, orc, kind):
    """320 rows at 256k (the many-row shape, where long rows are sampled): a
    sample that misses every top score, a keep-th score exactly at the band's
    upper edge, and a band holding more ties than the candidate list."""
    rows, tokens = 320, 262144
    rng = qi.rng_for(4, salt=len(kind) * 1000 + rows)
    n = tokens // 4
    scores = band_rows(rng, rows, n, kind)
    pos = np.full(rows, tokens - 1, np.int32)
    got, _ = gpu_select(qsa, scores, n, pos, tokens, 2048)
    want, codes = oracle_masks(orc, scores, n, pos, tokens, 2048)
    assert all(c == 0 for c in codes)
    for r in range(rows):
        assert np.array_equal(got[r], want[r]), r
