"""End-to-end parity of qsa_index_select (pool -> score -> select) against the oracle.

Masks may differ from the oracle's only on blocks whose oracle score lies within
the score tolerance of the row's keep-th score; everything else is bit-exact.
"""
import numpy as np
import pytest
import torch

import qsa_inputs as qi
from qsa_cases import (BUDGET, EPS, THETA, assert_close, assert_masks_agree_up_to_tolerance,
                       check_mask_structure, long_keys_case, oracle_masks, oracle_scores,
                       prefill_case)

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


@pytest.fixture(scope="module")
def tables(qsa):
    c, s = qsa.qsa_rope_tables(65536 + 8, THETA)
    return c, s, dev(c), dev(s)


def test_prefill_end_to_end(qsa, orc, tables):
    """Single-sequence prefill, T = 2304, every row; four rows have q = 0 (all-zero
    score rows: ties at 0.0 everywhere)."""
    case = prefill_case()
    T = case["T"]
    fq = case["fq"].copy()
    zero_rows = [2100, 2200, 2301, 2303]
    fq[zero_rows, :512] = 0
    c, s, cd, sd = tables
    nb = T // 4
    cols = nb
    fq_d = dev(fq)
    bk = torch.zeros((nb, 128), dtype=torch.int16, device="cuda")
    sc = torch.full((T, cols), -7.0, dtype=torch.float32, device="cuda")
    mask = torch.full((T, T), 0xAB, dtype=torch.uint8, device="cuda")
    st = qsa.new_status()
    qsa.qsa_index_select(fq_d.view(-1)[512:], 640, 0, nb, dev(case["k_norm_w"]), fq_d, 640,
                         dev(case["pos"]), T, T, dev(case["q_norm_w"]), cd, sd, c.shape[0], EPS,
                         BUDGET, bk, sc, cols, mask, st, workspace=qsa.new_workspace(T))
    assert qsa.qsa_read_status(st) == (0, 0)
    keys_o = orc.pool_blocks(fq.reshape(-1)[512:], 640, 0, nb, case["k_norm_w"], c, s, EPS)
    assert np.array_equal(bk.cpu().numpy().view(np.uint16), keys_o)
    sc_o, _ = oracle_scores(orc, fq, 640, case["pos"], T, case["q_norm_w"], c, s, keys_o, cols)
    got_sc = sc.cpu().numpy()
    assert_close(got_sc, sc_o, "end-to-end scores")
    mask_o, codes = oracle_masks(orc, sc_o, cols, case["pos"], T, BUDGET)
    assert all(c_ == 0 for c_ in codes)
    got = mask.cpu().numpy()
    tied = 0
    for r in range(T):
        check_mask_structure(got[r], r, T, BUDGET)
        tied += assert_masks_agree_up_to_tolerance(got[r], mask_o[r], sc_o[r], r, BUDGET, f"row {r}")
    for r in zero_rows:
        assert np.array_equal(got[r], mask_o[r])
    assert tied <= 16


def test_decode_steps_end_to_end(qsa, orc, tables):
    """Decode at 64k: the block cache holds every earlier block, each step pools the
    block its token completes, scores one row and selects."""
    case = long_keys_case()
    keys = case["keys"]
    c, s, cd, sd = tables
    tokens = 65536
    nb = tokens // 4
    first_step = 65528
    keys_o = orc.pool_blocks(keys, 128, 0, nb, case["k_norm_w"], c, s, EPS)
    cache = dev(keys_o.copy())
    cache[(first_step + 1) // 4:] = 0x7FAB        # blocks not yet pooled
    keys_d = dev(keys)
    cols = nb
    kw = dev(case["k_norm_w"])
    qw = dev(case["q_norm_w"])
    for k, p in enumerate(range(first_step, tokens)):
        completes = (p + 1) % 4 == 0
        b_new = (p + 1) // 4 - 1
        pos = dev(np.array([p], np.int32))
        q = dev(case["q"][k:k + 1])
        sc = torch.full((1, cols), -7.0, dtype=torch.float32, device="cuda")
        mask = torch.full((1, tokens), 0xAB, dtype=torch.uint8, device="cuda")
        st = qsa.new_status()
        qsa.qsa_index_select(keys_d.view(-1)[4 * b_new * 128:] if completes else keys_d, 128,
                             b_new if completes else 0, 1 if completes else 0, kw, q, 512, pos, 1,
                             tokens, qw, cd, sd, c.shape[0], EPS, BUDGET, cache, sc, cols, mask, st)
        assert qsa.qsa_read_status(st) == (0, 0)
        n = (p + 1) // 4
        assert np.array_equal(cache[:n].cpu().numpy().view(np.uint16), keys_o[:n])
        sc_o, _ = oracle_scores(orc, case["q"][k:k + 1], 512, np.array([p], np.int32), tokens,
                                case["q_norm_w"], c, s, keys_o, cols)
        assert_close(sc.cpu().numpy(), sc_o, f"decode step {p}")
        mask_o, _ = oracle_masks(orc, sc_o, cols, np.array([p], np.int32), tokens, BUDGET)
        got = mask.cpu().numpy()[0]
        check_mask_structure(got, p, tokens, BUDGET)
        assert_masks_agree_up_to_tolerance(got, mask_o[0], sc_o[0], p, BUDGET, f"step {p}")


def test_index_select_matches_the_single_stage_entries(qsa, orc, tables):
    """1600 rows at 64k: qsa_index_select's scores and masks must equal, bit for
    bit, those of qsa_score_rows + qsa_select_mask, and an out-of-range row near
    the end is reported by its index."""
    rng = qi.rng_for(3, salt=1600)
    tokens, rows = 65536, 1600
    nb = tokens // 4
    c, s, cd, sd = tables
    keys = qi.normal_bf16(rng, (nb, 128))
    q = qi.normal_bf16(rng, (rows, 512))
    qw, kw = qi.norm_weights(rng)
    pos = rng.integers(2000, tokens, size=rows).astype(np.int32)
    pos[1599] = tokens + 5                     # out of range
    ws = qsa.new_workspace(rows)
    outs = []
    for fused in (True, False):
        bk = dev(keys)
        sc = torch.full((rows, nb), -7.0, dtype=torch.float32, device="cuda")
        mask = torch.full((rows, tokens), 0xAB, dtype=torch.uint8, device="cuda")
        st = qsa.new_status()
        if fused:
            qsa.qsa_index_select(bk, 128, 0, 0, dev(kw), dev(q), 512, dev(pos), rows, tokens,
                                 dev(qw), cd, sd, c.shape[0], EPS, BUDGET, bk, sc, nb, mask, st,
                                 workspace=ws)
        else:
            qsa.qsa_score_rows(dev(q), 512, dev(pos), None, rows, tokens, dev(qw), cd, sd,
                               c.shape[0], EPS, bk, None, sc, nb, st, workspace=ws)
            qsa.qsa_select_mask(sc, nb, dev(pos), rows, tokens, BUDGET, mask, st)
        torch.cuda.synchronize()
        outs.append((sc.cpu().numpy(), mask.cpu().numpy(), qsa.qsa_read_status(st)))
    (fsc, fmask, fst), (psc, pmask, pst) = outs
    assert fst == (qsa.QSA_ERR_ROW_RANGE, 1599) and pst == (qsa.QSA_ERR_ROW_RANGE, 1599)
    assert np.array_equal(fsc, psc)
    assert np.array_equal(fmask, pmask)
    # and a few rows against the oracle's selection of these scores
    check = [0, 767, 768, 1535, 1536, 1598]
    want, codes = oracle_masks(orc, fsc, nb, pos, tokens, BUDGET, rows=check)
    assert all(cd_ == 0 for cd_ in codes)
    for k, r in enumerate(check):
        assert np.array_equal(fmask[r], want[k]), r
