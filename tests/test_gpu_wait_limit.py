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

from qsa_cases import (BUDGET, EPS, THETA, assert_close, check_mask_structure, long_keys_case,
                       oracle_masks, oracle_scores)

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


@pytest.mark.parametrize("path", ["simt", "stream"])
def test_streaming_scorer_ring_wait_runs_out_then_the_next_call_is_exact(orc, path):
    """The streaming scorers' waits for each landed stage of their key ring (and,
    on the tcgen05 one, for the query operand and each accumulator) take the
    same limit.  64 rows of 64k, each over its own 4 MiB of block keys
    (256 MiB in all, twice L2), keep the kernel bound by its copies, so its
    consumers find stages still in flight; cut to one cycle, such a wait gives
    up, the CTA drains its own copies and records QSA_ERR_TIMEOUT.  Restored,
    the same call writes the same scores as before the cut."""
    import sparse_attention_token_qsa_gb300 as qsa
    import qsa_inputs as qi

    tokens = 65536
    nb = tokens // 4
    n_rows = 64
    case = long_keys_case()
    c, s = qsa.qsa_rope_tables(tokens, THETA)
    keys = qi.torch_normal_bf16(torch, (n_rows * nb, 128), 21, "cuda")
    base_np = (np.arange(n_rows, dtype=np.int64) * nb)
    pos_np = (65535 - 97 * np.arange(n_rows)).astype(np.int32)
    head = (dev(case["q"][:n_rows]), 512, dev(pos_np), None, n_rows, tokens,
            dev(case["q_norm_w"]), dev(c), dev(s), tokens, EPS, keys, dev(base_np))

    def run():
        sc = torch.full((n_rows, nb), -7.0, dtype=torch.float32, device="cuda")
        st = qsa.new_status()
        qsa.qsa_score_rows_with(*head, sc, nb, st, path=qsa.QSA_SCORE_SIMT if path == "simt"
                                else qsa.QSA_SCORE_STREAM)
        return sc, qsa.qsa_read_status(st)

    before, status = run()
    assert status == (0, 0)

    default = qsa.qsa_wait_limit_cycles()
    qsa.qsa_set_wait_limit_cycles(1)
    try:
        _, (code, row) = run()
    finally:
        qsa.qsa_set_wait_limit_cycles(default)
    assert qsa.qsa_wait_limit_cycles() == default
    assert code == qsa.QSA_ERR_TIMEOUT, (code, row)
    assert 0 <= row < n_rows

    after, status = run()
    assert status == (0, 0)
    assert torch.equal(after, before)
    # and the restored call's scores are the oracle's, within the score tolerance
    got = after.cpu().numpy()
    for i in (0, 31, 63):
        kh = keys[i * nb:(i + 1) * nb].cpu().numpy().view(np.uint16)
        want, res = oracle_scores(orc, np.ascontiguousarray(case["q"][i:i + 1]), 512,
                                  pos_np[i:i + 1], tokens, case["q_norm_w"], c, s, kh, nb)
        assert all(rc == 0 for rc, _ in res)
        nv = (int(pos_np[i]) + 1) // 4
        assert np.all(got[i, nv:] == -7.0)
        assert_close(got[i, :nv], want[0, :nv], f"row {i}")
