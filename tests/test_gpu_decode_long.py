"""The long-context decode case at its full size, in the launch configuration the
bench times: 32 sequences of 131072..262144 tokens, one row each, per-sequence
block keys addressed through key_base (1.5M blocks, 400 MB), scored by
qsa_score_rows (the streaming tcgen05 scorer, one wave of CTAs) and selected
by qsa_select_mask (clusters of 4 CTAs a row).  Sampled rows' scores against
the oracle's, every row's mask against the oracle's selection over the GPU's
own scores (bit for bit), and the SIMT scorer on the same sampled rows."""
import numpy as np
import pytest
import torch

import qsa_inputs as qi
from qsa_cases import BUDGET, EPS, THETA, assert_close, check_mask_structure, oracle_masks, oracle_scores

pytestmark = pytest.mark.gpu


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def test_long_decode_full_size_scores_and_masks(orc):
    import sparse_attention_token_qsa_gb300 as qsa

    n_seq, tokens = 32, 262144
    rng = qi.rng_for(3, salt=4242)
    lens = qi.long_context_lengths(rng, n_seq)
    nbs = lens // 4
    blk_off = np.concatenate([[0], np.cumsum(nbs)]).astype(np.int64)
    keys = qi.torch_normal_bf16(torch, (int(blk_off[-1]), 128), qi.seed_for(3, 77), "cuda")
    c, s = qsa.qsa_rope_tables(tokens, THETA)
    qw, _ = qi.norm_weights(rng)
    q = qi.normal_bf16(rng, (n_seq, 512))
    pos = (lens - 1).astype(np.int32)
    base = blk_off[:-1].copy()
    cols = tokens // 4
    head = (dev(q), 512, dev(pos), None, n_seq, tokens, dev(qw), dev(c), dev(s), tokens, EPS, keys,
            dev(base))

    sc = torch.full((n_seq, cols), -7.0, dtype=torch.float32, device="cuda")
    st = qsa.new_status()
    qsa.qsa_score_rows(*head, sc, cols, st)
    assert qsa.qsa_read_status(st) == (0, 0)
    mask = torch.full((n_seq, tokens), 0xAB, dtype=torch.uint8, device="cuda")
    qsa.qsa_select_mask(sc, cols, dev(pos), n_seq, tokens, BUDGET, mask, st)
    assert qsa.qsa_read_status(st) == (0, 0)
    got = sc.cpu().numpy()

    # sampled rows: the scores against the oracle's, and the SIMT scorer's within tolerance
    sc2 = torch.full((n_seq, cols), -7.0, dtype=torch.float32, device="cuda")
    qsa.qsa_score_rows_with(*head, sc2, cols, st, path=qsa.QSA_SCORE_SIMT)
    assert qsa.qsa_read_status(st) == (0, 0)
    simt = sc2.cpu().numpy()
    for i in (0, 13, 31):
        lo, hi = int(blk_off[i]), int(blk_off[i + 1])
        kh = keys[lo:hi].cpu().numpy().view(np.uint16)
        want, res = oracle_scores(orc, q[i:i + 1], 512, pos[i:i + 1], tokens, qw, c, s, kh, cols)
        assert res[0][0] == 0
        assert_close(got[i:i + 1], want, f"row {i} scores")
        assert np.all(got[i, nbs[i]:] == -7.0)  # past the row's blocks: untouched
        assert_close(simt[i:i + 1], want, f"row {i} SIMT scores")

    # every row's mask: the oracle's selection over the GPU's own scores
    m = mask.cpu().numpy()
    want_m, codes = oracle_masks(orc, got, cols, pos, tokens, BUDGET)
    assert all(cd == 0 for cd in codes)
    for i in range(n_seq):
        check_mask_structure(m[i], int(pos[i]), tokens, BUDGET)
        assert np.array_equal(m[i], want_m[i]), f"row {i}"
