"""qsa_mask_tokens and qsa_gather_kv against the oracle.

Both are integer and byte work, so the bar is bit-exact: every listed token,
every count and every gathered bf16 bit pattern equals the oracle's, and every
output element the call must not touch keeps its sentinel.
"""
import numpy as np
import pytest
import torch

import qsa_inputs as qi
from qsa_cases import BUDGET, oracle_masks

pytestmark = pytest.mark.gpu

SENT_SEL = -5
SENT_KV = 0x7FAB


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def host_u16(t):
    return t.cpu().numpy().view(np.uint16)


@pytest.fixture(scope="module")
def qsa():
    import sparse_attention_token_qsa_gb300 as m

    return m


def run_mask_tokens(qsa, mask_np, sel_cols, offset=0):
    """One call over mask_np [n_rows, tokens] placed at a byte offset; returns
    (sel, n_sel) as host arrays."""
    n_rows, tokens = mask_np.shape
    buf = torch.zeros(n_rows * tokens + offset + 16, dtype=torch.uint8, device="cuda")
    buf[offset:offset + n_rows * tokens] = dev(mask_np.reshape(-1))
    mask = buf[offset:offset + n_rows * tokens]
    sel = torch.full((max(n_rows * sel_cols, 1),), SENT_SEL, dtype=torch.int32, device="cuda")
    n_sel = torch.full((n_rows,), -1, dtype=torch.int32, device="cuda")
    qsa.qsa_mask_tokens(mask, n_rows, tokens, sel, sel_cols, n_sel)
    torch.cuda.synchronize()
    return sel.cpu().numpy()[:n_rows * sel_cols].reshape(n_rows, sel_cols), n_sel.cpu().numpy()


def check_mask_tokens(orc, mask_np, sel, n_sel, sel_cols):
    for r in range(mask_np.shape[0]):
        want, n = orc.mask_tokens(mask_np[r], sel_cols)
        assert n_sel[r] == n, f"row {r}: count {n_sel[r]} != {n}"
        k = min(n, sel_cols)
        assert np.array_equal(sel[r, :k], want), f"row {r}: token list differs"
        assert np.all(sel[r, k:] == SENT_SEL), f"row {r}: wrote past its count"


def random_mask(rng, n_rows, tokens, density):
    """Random bytes, each non-zero with probability `density` (any non-zero
    value marks a token)."""
    keep = rng.random((n_rows, tokens)) < density
    vals = rng.integers(1, 256, size=(n_rows, tokens)).astype(np.uint8)
    return np.where(keep, vals, 0).astype(np.uint8)


@pytest.mark.parametrize("tokens,offset", [(65536, 0), (30001, 3), (8192, 0), (8193, 5), (7, 1),
                                           (16, 0), (1, 0)])
def test_mask_tokens_random_masks(qsa, orc, tokens, offset):
    """Ragged token counts (rows then start at every alignment), masks at odd
    byte offsets, densities from empty to full."""
    rng = qi.rng_for(2, salt=tokens + offset)
    rows = [random_mask(rng, 1, tokens, d)[0] for d in (0.0, 0.003, 0.05, 0.5, 0.97, 1.0)]
    mask_np = np.stack(rows)
    sel, n_sel = run_mask_tokens(qsa, mask_np, tokens + 3, offset)
    check_mask_tokens(orc, mask_np, sel, n_sel, tokens + 3)


def test_mask_tokens_of_selection_masks(qsa, orc):
    """The lists of masks the selection writes (kept blocks' tokens, then the
    tail) fit in budget + 3 columns and equal the oracle's."""
    rng = qi.rng_for(2, salt=91)
    tokens = 65536
    nb = tokens // 4
    pos = np.array([tokens - 1, tokens - 2, 2050, 3, 0, 40001, 2047], np.int32)
    scores = rng.standard_normal((len(pos), nb)).astype(np.float32)
    masks, codes = oracle_masks(orc, scores, nb, pos, tokens, BUDGET)
    assert all(c == 0 for c in codes)
    sel, n_sel = run_mask_tokens(qsa, masks, BUDGET + 3)
    check_mask_tokens(orc, masks, sel, n_sel, BUDGET + 3)
    assert np.all(n_sel <= BUDGET + 3)


@pytest.mark.parametrize("sel_cols", [0, 1, 100, 4095])
def test_mask_tokens_cut_at_sel_cols(qsa, orc, sel_cols):
    """A list longer than sel_cols is cut; the count is still the whole count."""
    rng = qi.rng_for(2, salt=500 + sel_cols)
    mask_np = random_mask(rng, 3, 20011, 0.4)
    sel, n_sel = run_mask_tokens(qsa, mask_np, sel_cols)
    check_mask_tokens(orc, mask_np, sel, n_sel, sel_cols)


def test_mask_tokens_empty_and_many_rows(qsa, orc):
    """tokens = 0 gives empty lists; 70000 rows of 16 tokens (more rows than a
    grid's y extent)."""
    n_sel = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    sel = torch.full((8,), SENT_SEL, dtype=torch.int32, device="cuda")
    mask = torch.zeros(16, dtype=torch.uint8, device="cuda")
    qsa.qsa_mask_tokens(mask, 4, 0, sel, 2, n_sel)
    torch.cuda.synchronize()
    assert np.all(n_sel.cpu().numpy() == 0) and np.all(sel.cpu().numpy() == SENT_SEL)
    rng = qi.rng_for(2, salt=7)
    mask_np = random_mask(rng, 70000, 16, 0.3)
    sel, n_sel = run_mask_tokens(qsa, mask_np, 16)
    want_n = (mask_np != 0).sum(axis=1)
    assert np.array_equal(n_sel, want_n)
    for r in rng.choice(70000, 64, replace=False):
        want, n = orc.mask_tokens(mask_np[r], 16)
        assert n == n_sel[r] and np.array_equal(sel[r, :n], want)


# ---- qsa_gather_kv


def run_gather(qsa, k_np, v_np, width, table_np, page_size, sel_np, n_sel_np, max_sel, out_rows,
               pool_pages=None):
    """One call; table_np is [n_rows, table_len] (per-row tables) or
    [table_len] (one table shared by every row).  Returns k_out, v_out as
    [n_rows, out_rows, width] host arrays and the status."""
    n_rows, sel_cols = sel_np.shape
    shared = table_np.ndim == 1
    table_len = table_np.shape[-1]
    pages = k_np.shape[0] // page_size if pool_pages is None else pool_pages
    k_out = torch.full((n_rows * out_rows, width), SENT_KV, dtype=torch.int16, device="cuda")
    v_out = torch.full((n_rows * out_rows, width), SENT_KV, dtype=torch.int16, device="cuda")
    st = qsa.new_status()
    qsa.qsa_gather_kv(dev(k_np), dev(v_np), width, pages, dev(table_np), table_len,
                      0 if shared else table_len, page_size, dev(sel_np), sel_cols, dev(n_sel_np),
                      n_rows, max_sel, k_out, v_out, out_rows, st)
    torch.cuda.synchronize()
    shape = (n_rows, out_rows, width)
    return host_u16(k_out).reshape(shape), host_u16(v_out).reshape(shape), qsa.qsa_read_status(st)


def check_gather(orc, k_np, v_np, width, table_np, page_size, sel_np, n_sel_np, max_sel, k_out,
                 v_out, skip_rows=()):
    for r in range(sel_np.shape[0]):
        if r in skip_rows:
            continue
        n = max(0, min(int(n_sel_np[r]), max_sel))
        table = table_np if table_np.ndim == 1 else table_np[r]
        for pool, out, what in ((k_np, k_out, "K"), (v_np, v_out, "V")):
            want, rc = orc.gather(pool, table, page_size, width, sel_np[r, :n])
            assert rc == 0
            assert np.array_equal(out[r, :n], want), f"row {r}: {what} rows differ"
            assert np.all(out[r, n:] == SENT_KV), f"row {r}: {what} written past its count"


def sorted_tokens(rng, limit, count):
    return np.sort(rng.choice(limit, size=min(count, limit), replace=False)).astype(np.int32)


@pytest.mark.parametrize("width,page_size", [(512, 16), (8, 16), (520, 1), (1024, 64), (256, 7)])
def test_gather_matches_oracle_per_row_tables(qsa, orc, width, page_size):
    """Per-row shuffled page tables; counts from empty to the whole column
    count, and one row cut by max_sel; widths that end inside the copy loop."""
    rng = qi.rng_for(2, salt=width * 131 + page_size)
    table_len = max(40, -(-300 // page_size))  # room for 300 distinct tokens
    pages = table_len + 56
    k_np = qi.paged_kv_pool(rng, pages, page_size, width)
    v_np = qi.paged_kv_pool(rng, pages, page_size, width)
    n_rows, sel_cols = 6, 300
    tables = qi.page_tables(rng, n_rows, table_len, pages)
    limit = table_len * page_size
    sel_np = np.full((n_rows, sel_cols), -9, np.int32)
    n_sel = np.array([0, 1, 37, 260, 300, 300], np.int32)
    for r in range(n_rows):
        toks = sorted_tokens(rng, limit, int(n_sel[r]))
        n_sel[r] = len(toks)
        sel_np[r, :len(toks)] = toks
    n_sel[5] = 10 ** 6  # a count above max_sel: cut at max_sel
    max_sel = 280
    k_out, v_out, st = run_gather(qsa, k_np, v_np, width, tables, page_size, sel_np, n_sel, max_sel,
                                  max_sel + 5)
    assert st == (0, 0)
    check_gather(orc, k_np, v_np, width, tables, page_size, sel_np, n_sel, max_sel, k_out, v_out)


def test_gather_shared_table_and_unsorted_tokens(qsa, orc):
    """One table for all rows (table_cols = 0); tokens in any order, repeats
    allowed (each listed token is copied where it is listed)."""
    rng = qi.rng_for(2, salt=17)
    width, page_size, pages, table_len = 512, 16, 64, 64
    k_np = qi.paged_kv_pool(rng, pages, page_size, width)
    v_np = qi.paged_kv_pool(rng, pages, page_size, width)
    table = rng.permutation(pages).astype(np.int32)
    n_rows, sel_cols = 4, 129
    sel_np = rng.integers(0, table_len * page_size, size=(n_rows, sel_cols)).astype(np.int32)
    sel_np[1, 5:9] = sel_np[1, 0]
    n_sel = np.array([129, 128, 3, 64], np.int32)
    k_out, v_out, st = run_gather(qsa, k_np, v_np, width, table, page_size, sel_np, n_sel, 129, 129)
    assert st == (0, 0)
    check_gather(orc, k_np, v_np, width, table, page_size, sel_np, n_sel, 129, k_out, v_out)


@pytest.mark.parametrize("case,bad", list(enumerate(["past_table", "negative", "page_past_pool",
                                                     "negative_page"])))
def test_gather_out_of_range_reports_and_reads_nothing(qsa, orc, case, bad):
    """A token past the table, a negative token, or a table entry outside the
    pool: QSA_ERR_TOKEN_RANGE with the row, that token's output rows left
    alone, every other token still gathered."""
    rng = qi.rng_for(2, salt=900 + case)
    width, page_size, pages, table_len = 64, 16, 32, 20
    k_np = qi.paged_kv_pool(rng, pages, page_size, width)
    v_np = qi.paged_kv_pool(rng, pages, page_size, width)
    tables = qi.page_tables(rng, 3, table_len, pages)
    sel_np = np.stack([sorted_tokens(rng, table_len * page_size, 50) for _ in range(3)])
    n_sel = np.full(3, 50, np.int32)
    j = 17  # row 1's bad entry
    if bad == "past_table":
        sel_np[1, j] = table_len * page_size
    elif bad == "negative":
        sel_np[1, j] = -3
    else:
        tables[1, sel_np[1, j] // page_size] = pages if bad == "page_past_pool" else -1
    k_out, v_out, st = run_gather(qsa, k_np, v_np, width, tables, page_size, sel_np, n_sel, 50, 50)
    assert st == (qsa.QSA_ERR_TOKEN_RANGE, 1)
    check_gather(orc, k_np, v_np, width, tables, page_size, sel_np, n_sel, 50, k_out, v_out,
                 skip_rows=(1,))
    good = [i for i in range(50) if i != j and tables[1, sel_np[1, i] // page_size] in range(pages)]
    for pool, out in ((k_np, k_out), (v_np, v_out)):
        want, rc = orc.gather(pool, tables[1], page_size, width, sel_np[1, good])
        assert rc == 0 and np.array_equal(out[1, good], want)
        assert np.all(out[1, j] == SENT_KV)


def test_gather_many_rows(qsa, orc):
    """70000 rows (more than a grid's y extent), two tokens each, shared table."""
    rng = qi.rng_for(2, salt=70000)
    width, page_size, pages = 8, 4, 16
    k_np = qi.paged_kv_pool(rng, pages, page_size, width)
    v_np = qi.paged_kv_pool(rng, pages, page_size, width)
    table = rng.permutation(pages).astype(np.int32)
    n_rows = 70000
    sel_np = rng.integers(0, pages * page_size, size=(n_rows, 2)).astype(np.int32)
    n_sel = rng.integers(0, 3, size=n_rows).astype(np.int32)
    k_out, v_out, st = run_gather(qsa, k_np, v_np, width, table, page_size, sel_np, n_sel, 2, 2)
    assert st == (0, 0)
    # the whole output follows from numpy indexing of the pool (pinned to the
    # oracle's gather on a sample of rows below)
    slot = table[sel_np // page_size] * page_size + sel_np % page_size
    live = np.arange(2)[None, :] < n_sel[:, None]
    assert np.array_equal(k_out[live], k_np[slot[live]])
    assert np.array_equal(v_out[live], v_np[slot[live]])
    assert np.all(k_out[~live] == SENT_KV) and np.all(v_out[~live] == SENT_KV)
    rows = rng.choice(n_rows, 32, replace=False)
    check_gather(orc, k_np, v_np, width, table, page_size, sel_np[rows], n_sel[rows], 2,
                 k_out[rows], v_out[rows])


def test_decode_mask_to_gathered_kv(qsa, orc):
    """The decode chain at 64k: selection masks -> token lists -> K/V rows of a
    paged cache (2 KV heads x 256, pages of 16 tokens), both device calls
    chained on the stream, against the oracle's list and gather."""
    rng = qi.rng_for(1, salt=4242)
    tokens = 65536
    nb = tokens // 4
    pos = np.array([tokens - 1, 50001, 2050, 9], np.int32)
    n_rows = len(pos)
    scores = rng.standard_normal((n_rows, nb)).astype(np.float32)
    masks, _ = oracle_masks(orc, scores, nb, pos, tokens, BUDGET)
    width, page_size = 512, 16
    table_len = tokens // page_size
    pages = table_len + 64
    k_np = qi.paged_kv_pool(rng, pages, page_size, width)
    v_np = qi.paged_kv_pool(rng, pages, page_size, width)
    tables = qi.page_tables(rng, n_rows, table_len, pages)
    sel_cols = BUDGET + 3
    sel = torch.full((n_rows, sel_cols), SENT_SEL, dtype=torch.int32, device="cuda")
    n_sel = torch.zeros(n_rows, dtype=torch.int32, device="cuda")
    k_out = torch.full((n_rows * sel_cols, width), SENT_KV, dtype=torch.int16, device="cuda")
    v_out = torch.full((n_rows * sel_cols, width), SENT_KV, dtype=torch.int16, device="cuda")
    st = qsa.new_status()
    qsa.qsa_mask_tokens(dev(masks), n_rows, tokens, sel, sel_cols, n_sel)
    qsa.qsa_gather_kv(dev(k_np), dev(v_np), width, pages, dev(tables), table_len, table_len,
                      page_size, sel, sel_cols, n_sel, n_rows, sel_cols, k_out, v_out, sel_cols, st)
    torch.cuda.synchronize()
    assert qsa.qsa_read_status(st) == (0, 0)
    k_o = host_u16(k_out).reshape(n_rows, sel_cols, width)
    v_o = host_u16(v_out).reshape(n_rows, sel_cols, width)
    for r in range(n_rows):
        toks, n = orc.mask_tokens(masks[r], sel_cols)
        assert n == int(n_sel[r]) == min(BUDGET, 4 * ((pos[r] + 1) // 4)) + (pos[r] + 1) % 4
        for pool, out in ((k_np, k_o), (v_np, v_o)):
            want, rc = orc.gather(pool, tables[r], page_size, width, toks)
            assert rc == 0 and np.array_equal(out[r, :n], want)
            assert np.all(out[r, n:] == SENT_KV)
