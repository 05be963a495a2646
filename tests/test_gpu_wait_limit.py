"""A bounded device wait made to run out, on purpose and without a fault.

PR #1178's review note on environment side effects: a deliberate trap left
the GPU unusable, so every wait in this library is bounded and reports
QSA_ERR_TIMEOUT in the status word instead of trapping.  Here the limit is cut
to one SM cycle with qsa_set_wait_limit_cycles, so the fused decode step's
waits for its key copies, its MMAs and its grid barrier give up (the first
test of each finds the copy, the MMA or the other CTAs still in flight).  The
call must return, the status must be QSA_ERR_TIMEOUT for one of the rows, and
once the limit is restored and the workspace zeroed the next call must give
the exact selection again.
"""
import numpy as np
import pytest
import torch

from qsa_cases import BUDGET, EPS, THETA, check_mask_structure, long_keys_case, oracle_masks

pytestmark = pytest.mark.gpu


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def test_decode_barrier_runs_out_then_the_next_call_is_exact(orc):
    import sparse_attention_token_qsa_gb300 as qsa

    case = long_keys_case()
    tokens = 65536
    nb = tokens // 4
    c, s = qsa.qsa_rope_tables(tokens, THETA)
    cd, sd = dev(c), dev(s)
    keys = orc.pool_blocks(case["keys"], 128, 0, nb, case["k_norm_w"], c, s, EPS)
    cache = dev(keys)
    pos_np = np.array([65534, 40001], np.int32)     # two rows of many CTAs each
    n_rows = len(pos_np)
    args_head = (cache, 128, 0, 0, dev(case["k_norm_w"]), dev(case["q"][:n_rows]), 512,
                 dev(pos_np), n_rows, tokens, dev(case["q_norm_w"]), cd, sd, tokens, EPS, BUDGET,
                 cache)
    ws = qsa.new_decode_workspace(n_rows, tokens)

    default = qsa.qsa_wait_limit_cycles()
    sc = torch.full((n_rows, nb), -7.0, dtype=torch.float32, device="cuda")
    mask = torch.full((n_rows, tokens), 0xAB, dtype=torch.uint8, device="cuda")
    st = qsa.new_status()
    qsa.qsa_set_wait_limit_cycles(1)
    try:
        qsa.qsa_decode_index_select(*args_head, sc, nb, mask, st, ws)
        code, row = qsa.qsa_read_status(st)       # synchronises: the call has returned
    finally:
        qsa.qsa_set_wait_limit_cycles(default)
    assert qsa.qsa_wait_limit_cycles() == default == 4000000000
    assert code == qsa.QSA_ERR_TIMEOUT, (code, row)
    assert row in (0, 1)

    # the workspace may be dirty after an error: zero it; the next call, at the
    # default limit, is exact
    ws.zero_()
    sc = torch.full((n_rows, nb), -7.0, dtype=torch.float32, device="cuda")
    mask = torch.full((n_rows, tokens), 0xAB, dtype=torch.uint8, device="cuda")
    st = qsa.new_status()
    qsa.qsa_decode_index_select(*args_head, sc, nb, mask, st, ws)
    assert qsa.qsa_read_status(st) == (0, 0)
    assert int(ws.count_nonzero()) == 0
    got_sc, got = sc.cpu().numpy(), mask.cpu().numpy()
    want, codes = oracle_masks(orc, got_sc, nb, pos_np, tokens, BUDGET)
    assert codes == [0, 0]
    for i, p in enumerate(pos_np):
        check_mask_structure(got[i], int(p), tokens, BUDGET)
        assert np.array_equal(got[i], want[i]), f"row {i}"
