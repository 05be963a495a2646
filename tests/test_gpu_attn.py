"""qsa_sparse_attn against the oracle.

Tolerance, from the arithmetic: the kernel rounds each softmax weight to bf16
before the weighted sum of V (and normalises by the sum of the same rounded
weights), so the output is a convex combination of the selected V rows whose
weights are each within 2^-8 (relative) of the exact ones: the error is at
most 2^-8 * max |v| over the selected rows of the head's KV group.  Both sides
then round to bf16, which may land one bf16 step apart (2^-7 |out|).  Dots and
sums in f32 add ~1e-6 relative.  Every element is held to
    |got - want| <= 2^-8 * max|v| + 2^-7 * |want| + 1e-6.
Wrong tokens, heads, pages or scales move outputs by O(|v|); the peaked cases
(one dominant token per row) make such mistakes O(1).
"""
import numpy as np
import pytest
import torch

import qsa_inputs as qi
from qsa_cases import BUDGET

pytestmark = pytest.mark.gpu

SENT = 0x7FAB


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


@pytest.fixture(scope="module")
def qsa():
    import sparse_attention_token_qsa_gb300 as m

    return m


def f32(bits):
    return qi.bf16_bits_to_f32(bits)


def run_attn(qsa, q_np, nq, nkv, hd, k_np, v_np, page_size, tables, sel_np, n_sel_np, max_sel,
             scale, q_pad=0, out_pad=0, pool_pages=None):
    """One call; tables [rows, len] or [len] (shared).  Returns out [rows, nq*hd]
    bits (padding columns checked untouched) and the status."""
    rows = q_np.shape[0]
    row_len = nq * hd
    qs = row_len + q_pad
    qbuf = np.zeros((rows, qs), np.uint16)
    qbuf[:, :row_len] = q_np
    os_ = row_len + out_pad
    out = torch.full((rows, os_), SENT, dtype=torch.int16, device="cuda")
    st = qsa.new_status()
    shared = tables.ndim == 1
    pages = k_np.shape[0] // page_size if pool_pages is None else pool_pages
    qsa.qsa_sparse_attn(dev(qbuf), qs, nq, nkv, hd, dev(k_np), dev(v_np), pages, page_size,
                        dev(tables), tables.shape[-1], 0 if shared else tables.shape[-1],
                        dev(sel_np), sel_np.shape[1], dev(n_sel_np), rows, max_sel, scale, out, os_,
                        st)
    torch.cuda.synchronize()
    o = out.cpu().numpy().view(np.uint16)
    assert np.all(o[:, row_len:] == SENT), "wrote past a row"
    return o[:, :row_len], qsa.qsa_read_status(st)


def check_rows(orc, got, q_np, nq, nkv, hd, k_np, v_np, page_size, tables, sel_np, n_sel_np,
               max_sel, scale, rows=None):
    group = nq // nkv
    for r in (range(q_np.shape[0]) if rows is None else rows):
        n = max(0, min(int(n_sel_np[r]), max_sel))
        table = tables if tables.ndim == 1 else tables[r]
        sel = sel_np[r, :n]
        want, rc = orc.sparse_attn(q_np[r], nq, nkv, hd, k_np, v_np, table, page_size, sel, scale)
        assert rc == 0
        g = f32(got[r]).reshape(nq, hd)
        w = f32(want).reshape(nq, hd)
        if n == 0:
            assert np.all(got[r] == 0), f"row {r}: an empty list gives zeros"
            continue
        slots = table[sel // page_size] * page_size + sel % page_size
        vsel = np.abs(f32(v_np[slots]).reshape(n, nkv, hd))
        for h in range(nq):
            vmax = float(vsel[:, h // group, :].max())
            tol = 2.0 ** -8 * vmax + 2.0 ** -7 * np.abs(w[h]) + 1e-6
            err = np.abs(g[h] - w[h])
            assert np.all(err <= tol), (f"row {r} head {h}: max err {err.max():.3g} "
                                        f"(tol {tol[np.argmax(err - tol)]:.3g})")


def make_case(rng, rows, nq, nkv, hd, page_size, table_len, counts, q_std=2.0, extra_pages=8):
    pages = table_len + extra_pages
    k_np = qi.normal_bf16(rng, (pages * page_size, nkv * hd))
    v_np = qi.normal_bf16(rng, (pages * page_size, nkv * hd))
    tables = qi.page_tables(rng, rows, table_len, pages)
    q_np = qi.normal_bf16(rng, (rows, nq * hd), std=q_std)
    sel_cols = max(max(counts), 1) + 3
    sel_np = np.full((rows, sel_cols), -1, np.int32)
    n_sel = np.zeros(rows, np.int32)
    for r, c in enumerate(counts):
        toks = np.sort(rng.choice(table_len * page_size, size=c, replace=False)).astype(np.int32)
        sel_np[r, :c] = toks
        n_sel[r] = c
    return q_np, k_np, v_np, tables, sel_np, n_sel


@pytest.mark.parametrize("nq,nkv,hd", [(16, 2, 256), (8, 1, 128), (6, 2, 128), (24, 2, 256),
                                       (4, 4, 256)])
def test_attn_matches_oracle(qsa, orc, nq, nkv, hd):
    """Ragged lists (empty, one token, a partial tile, exactly one tile, one
    more, many tiles over every warp), groups of 8, 1, 3 and 12 query heads per
    KV head (12: two head chunks)."""
    rng = qi.rng_for(6, salt=nq * 1000 + nkv * 10 + hd)
    counts = [0, 1, 7, 16, 17, 300, 64, 129]
    page_size, table_len = 16, 40
    q_np, k_np, v_np, tables, sel_np, n_sel = make_case(rng, len(counts), nq, nkv, hd, page_size,
                                                        table_len, counts)
    scale = 1.0 / np.sqrt(hd)
    got, st = run_attn(qsa, q_np, nq, nkv, hd, k_np, v_np, page_size, tables, sel_np, n_sel,
                       sel_np.shape[1], scale, q_pad=8, out_pad=16)
    assert st == (0, 0)
    check_rows(orc, got, q_np, nq, nkv, hd, k_np, v_np, page_size, tables, sel_np, n_sel,
               sel_np.shape[1], scale)


def test_attn_one_dominant_token_per_row(qsa, orc):
    """Each row's list holds one token whose key is its query heads' direction
    scaled up (a tail token for some rows): the output is that token's V row,
    so a wrong token, head group or page shows up as an O(1) error."""
    rng = qi.rng_for(6, salt=77)
    nq, nkv, hd, page_size, table_len = 16, 2, 256, 16, 160
    counts = [40, 200, 2051, 3, 16]
    q_np, k_np, v_np, tables, sel_np, n_sel = make_case(rng, len(counts), nq, nkv, hd, page_size,
                                                        table_len, counts, q_std=1.0)
    group = nq // nkv
    for r, c in enumerate(counts):
        j = c - 1 if r % 2 == 0 else int(rng.integers(0, c))   # the tail token, or any
        t = sel_np[r, j]
        slot = tables[r][t // page_size] * page_size + t % page_size
        for g in range(nkv):
            qg = f32(q_np[r]).reshape(nq, hd)[g * group:(g + 1) * group].sum(axis=0)
            k_np[slot, g * hd:(g + 1) * hd] = qi.to_bf16_bits(qg / np.abs(qg).max() * 4.0)
    scale = 1.0 / np.sqrt(hd) * 4.0
    got, st = run_attn(qsa, q_np, nq, nkv, hd, k_np, v_np, page_size, tables, sel_np, n_sel,
                       sel_np.shape[1], scale)
    assert st == (0, 0)
    check_rows(orc, got, q_np, nq, nkv, hd, k_np, v_np, page_size, tables, sel_np, n_sel,
               sel_np.shape[1], scale)


def test_attn_shared_table_cut_lists_and_bad_tokens(qsa, orc):
    """One shared page table; max_sel cuts the lists; a token past the table
    (row 2) and a table entry outside the pool (row 4, through a per-row table
    copy) are reported as QSA_ERR_TOKEN_RANGE and the other rows are exact."""
    rng = qi.rng_for(6, salt=5)
    nq, nkv, hd, page_size, table_len = 8, 2, 128, 8, 50
    counts = [100, 60, 80, 5, 90]
    q_np, k_np, v_np, tables, sel_np, n_sel = make_case(rng, len(counts), nq, nkv, hd, page_size,
                                                        table_len, counts)
    shared = tables[0].copy()
    max_sel = 70
    got, st = run_attn(qsa, q_np, nq, nkv, hd, k_np, v_np, page_size, shared, sel_np, n_sel,
                       max_sel, 0.09)
    assert st == (0, 0)
    check_rows(orc, got, q_np, nq, nkv, hd, k_np, v_np, page_size, shared, sel_np, n_sel, max_sel,
               0.09)
    bad_sel = sel_np.copy()
    bad_sel[2, 10] = table_len * page_size          # past the table
    got, st = run_attn(qsa, q_np, nq, nkv, hd, k_np, v_np, page_size, shared, bad_sel, n_sel,
                       max_sel, 0.09)
    assert st == (qsa.QSA_ERR_TOKEN_RANGE, 2)
    check_rows(orc, got, q_np, nq, nkv, hd, k_np, v_np, page_size, shared, bad_sel, n_sel, max_sel,
               0.09, rows=[0, 1, 3, 4])
    per_row = np.stack([shared] * len(counts))
    per_row[4, sel_np[4, 3] // page_size] = k_np.shape[0] // page_size   # outside the pool
    got, st = run_attn(qsa, q_np, nq, nkv, hd, k_np, v_np, page_size, per_row, sel_np, n_sel,
                       max_sel, 0.09)
    assert st == (qsa.QSA_ERR_TOKEN_RANGE, 4)
    check_rows(orc, got, q_np, nq, nkv, hd, k_np, v_np, page_size, per_row, sel_np, n_sel,
               max_sel, 0.09, rows=[0, 1, 2, 3])


def prefill_lists(rng, positions, budget=BUDGET):
    """Each row's selected tokens as the selection defines them: budget/4
    blocks of the row's complete ones (drawn at random here) and the tail,
    ascending."""
    keep = budget // 4
    out = []
    for p in positions:
        n = (p + 1) // 4
        blocks = np.sort(rng.choice(n, size=min(keep, n), replace=False))
        toks = (4 * blocks[:, None] + np.arange(4)[None, :]).ravel()
        out.append(np.concatenate([toks, np.arange(4 * n, p + 1)]).astype(np.int32))
    return out


def test_attn_prefill_chunk_64k_sampled_rows(qsa, orc):
    """The benchmarked shape: 4096 rows at positions 61440..65535 of one 64k
    sequence, 16 query heads over 2 KV heads of 256, pages of 16 shuffled over
    the pool, 2048 + tail selected tokens per row; 8 rows checked."""
    rng = qi.rng_for(6, salt=64)
    tokens, first, rows = 65536, 61440, 4096
    nq, nkv, hd, page_size = 16, 2, 256, 16
    table_len = tokens // page_size
    pages = table_len + 32
    k_np = qi.normal_bf16(rng, (pages * page_size, nkv * hd))
    v_np = qi.normal_bf16(rng, (pages * page_size, nkv * hd))
    table = rng.permutation(pages)[:table_len].astype(np.int32)
    q_np = qi.normal_bf16(rng, (rows, nq * hd), std=2.0)
    lists = prefill_lists(rng, range(first, tokens))
    sel_cols = BUDGET + 3
    sel_np = np.full((rows, sel_cols), -1, np.int32)
    n_sel = np.zeros(rows, np.int32)
    for r, l in enumerate(lists):
        sel_np[r, :len(l)] = l
        n_sel[r] = len(l)
    scale = 1.0 / 16.0
    got, st = run_attn(qsa, q_np, nq, nkv, hd, k_np, v_np, page_size, table, sel_np, n_sel,
                       sel_cols, scale)
    assert st == (0, 0)
    check_rows(orc, got, q_np, nq, nkv, hd, k_np, v_np, page_size, table, sel_np, n_sel, sel_cols,
               scale, rows=[0, 1, 2, 3, 1000, 2047, 4094, 4095])


@pytest.mark.parametrize("page_size", [1, 5, 12, 1000])
def test_attn_page_sizes(qsa, orc, page_size):
    """Page sizes of one token, odd and not a power of two, and larger than a
    row's whole list: the token -> page division (a multiply-high and a shift
    for every size but one) finds each token's slot."""
    rng = qi.rng_for(6, salt=300 + page_size)
    nq, nkv, hd = 8, 2, 128
    counts = [1, 33, 64, 97]
    table_len = max(4, (3000 + page_size - 1) // page_size)
    q_np, k_np, v_np, tables, sel_np, n_sel = make_case(rng, len(counts), nq, nkv, hd, page_size,
                                                        table_len, counts, extra_pages=3)
    scale = 1.0 / np.sqrt(hd)
    got, st = run_attn(qsa, q_np, nq, nkv, hd, k_np, v_np, page_size, tables, sel_np, n_sel,
                       sel_np.shape[1], scale)
    assert st == (0, 0)
    check_rows(orc, got, q_np, nq, nkv, hd, k_np, v_np, page_size, tables, sel_np, n_sel,
               sel_np.shape[1], scale)
