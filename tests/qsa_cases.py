"""Workload builders and comparison helpers shared by the GPU parity tests.

Inputs come from ``qsa_inputs`` (seeded, synthetic); expected values come only
from the oracle.  The oracle runs row-parallel on host threads (its C calls
release the GIL), never forked after CUDA initialisation.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import qsa_inputs as qi

TOL_ABS = 5e-3
TOL_REL = 1e-3
EPS = 1e-6
THETA = 10000.0
BUDGET = 2048


def n_threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def parallel_rows(fn, n_rows: int, chunk: int = 16):
    """Run fn(lo, hi) over row chunks on host threads; returns the results in order."""
    spans = [(lo, min(n_rows, lo + chunk)) for lo in range(0, n_rows, chunk)]
    with cf.ThreadPoolExecutor(max_workers=n_threads()) as ex:
        return list(ex.map(lambda s: fn(*s), spans))


def oracle_scores(orc, q, q_stride, pos, tokens, q_norm_w, cos_t, sin_t, block_keys, score_cols,
                  visible_len=None, key_base=None, fill=-7.0):
    """Oracle scores for every row (row-parallel).  q: [rows, >=512] uint16."""
    n = len(pos)
    out = np.full((n, score_cols), fill, np.float32)

    def run(lo, hi):
        sub = np.ascontiguousarray(out[lo:hi])
        rc, row = orc.score_rows(q[lo:hi], q_stride, pos[lo:hi], hi - lo, tokens, q_norm_w, cos_t,
                                 sin_t, EPS, block_keys, sub, score_cols,
                                 visible_len=None if visible_len is None else visible_len[lo:hi],
                                 key_base=None if key_base is None else key_base[lo:hi])
        out[lo:hi] = sub
        return rc, row + lo

    res = parallel_rows(run, n)
    return out, res


def oracle_masks(orc, scores, score_cols, pos, tokens, budget, rows=None):
    rows = np.arange(len(pos)) if rows is None else np.asarray(rows)
    out = np.full((len(rows), tokens), 0xAB, np.uint8)

    def run(lo, hi):
        codes = []
        for j in range(lo, hi):
            r = rows[j]
            m, rc = orc.select_row(scores[r, :max(1, (pos[r] + 1) // 4)], int(pos[r]), tokens, budget)
            out[j] = m
            codes.append(rc)
        return codes

    codes = sum(parallel_rows(run, len(rows), chunk=4), [])
    return out, codes


def assert_close(got, want, what, atol=TOL_ABS, rtol=TOL_REL):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    nan_g, nan_w = np.isnan(got), np.isnan(want)
    assert np.array_equal(nan_g, nan_w), f"{what}: NaN pattern differs"
    g, w = got[~nan_w], want[~nan_w]
    err = np.abs(g - w)
    bound = atol + rtol * np.abs(w)
    if err.size and not np.all(err <= bound):
        i = int(np.argmax(err / bound))
        raise AssertionError(f"{what}: worst |diff| {err[i]:.3e} vs bound {bound[i]:.3e} "
                             f"(got {g[i]!r}, want {w[i]!r}, flat index {i})")
    return float(err.max()) if err.size else 0.0


def bf16_close(got_bits, want_bits, what, atol=TOL_ABS, rtol=TOL_REL):
    """Compare bf16 arrays (uint16 bits) within the float tolerance; returns #bit-exact."""
    g = qi.bf16_bits_to_f32(got_bits)
    w = qi.bf16_bits_to_f32(want_bits)
    assert_close(g, w, what, atol, rtol)
    return int(np.sum(np.asarray(got_bits) == np.asarray(want_bits)))


def kth_score(row_scores, n, K):
    v = np.where(row_scores[:n] == 0, 0.0, row_scores[:n]).astype(np.float64)
    return np.sort(v)[::-1][K - 1]


def check_mask_structure(mask_row, p, tokens, budget):
    """Structural validity of one mask row (PR #1178 tie criteria)."""
    n, tail = (p + 1) // 4, (p + 1) % 4
    K = min(budget // 4, n)
    assert mask_row.shape == (tokens,)
    assert set(np.unique(mask_row)).issubset({0, 1})
    assert int(mask_row.sum()) == 4 * K + tail
    assert np.all(mask_row[p + 1:] == 0)
    assert np.all(mask_row[4 * n:p + 1] == 1)
    if n:
        blk = mask_row[:4 * n].reshape(n, 4)
        assert np.all(blk.min(1) == blk.max(1))


def assert_masks_agree_up_to_tolerance(got, want, oracle_row_scores, p, budget, what):
    """End-to-end gate: masks may differ only on blocks whose oracle score is within
    tolerance of the row's keep-th score."""
    if np.array_equal(got, want):
        return 0
    n = (p + 1) // 4
    K = min(budget // 4, n)
    T = kth_score(oracle_row_scores, n, K)
    diff_blocks = np.nonzero(got[:4 * n:4] != want[:4 * n:4])[0]
    assert np.array_equal(got[4 * n:], want[4 * n:]), f"{what}: tail/zero region differs"
    s = np.where(oracle_row_scores[diff_blocks] == 0, 0.0, oracle_row_scores[diff_blocks])
    bad = np.abs(s - T) > TOL_ABS + TOL_REL * abs(T)
    assert not np.any(bad), f"{what}: blocks {diff_blocks[bad][:8]} differ away from the cut {T}"
    return len(diff_blocks)


# ---------------------------------------------------------------- workloads

def prefill_case(T=2304, seed_index=0):
    """Single-sequence prefill (T tokens, every row queried)."""
    rng = qi.rng_for(seed_index)
    fq = qi.fused_qk(rng, T)
    qw, kw = qi.norm_weights(rng)
    return dict(fq=fq, q_norm_w=qw, k_norm_w=kw, T=T, pos=np.arange(T, dtype=np.int32))


def long_keys_case(tokens=65536, seed_index=1, token_scale=True):
    rng = qi.rng_for(seed_index)
    keys = qi.raw_keys(rng, tokens, token_scale=token_scale)
    qw, kw = qi.norm_weights(rng)
    q = qi.fused_qk(rng, 256)[:, :512]
    return dict(keys=keys, q_norm_w=qw, k_norm_w=kw, q=np.ascontiguousarray(q), tokens=tokens)


def index_select_tc(qsa, keys, key_stride, first, count, k_norm_w, q, q_stride, pos, n_rows,
                    tokens, q_norm_w, cos_t, sin_t, table_rows, eps, budget, block_keys, scores,
                    score_cols, mask, status):
    """qsa_index_select's three stages with the tensor-core scorer forced: the
    same MMA per (block, head) as the fused decode kernel, so its scores must
    equal that kernel's bit for bit."""
    if count:
        qsa.qsa_pool_blocks(keys, key_stride, first, count, k_norm_w, cos_t, sin_t, table_rows, eps,
                            block_keys)
    qsa.qsa_score_rows_with(q, q_stride, pos, None, n_rows, tokens, q_norm_w, cos_t, sin_t,
                            table_rows, eps, block_keys, None, scores, score_cols, status,
                            path=qsa.QSA_SCORE_TCGEN05, workspace=qsa.new_workspace(n_rows))
    qsa.qsa_select_mask(scores, score_cols, pos, n_rows, tokens, budget, mask, status)
