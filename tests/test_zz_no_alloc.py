"""qsa_score_rows_noalloc: tensor-core scoring for callers that cannot allocate.

Some callers cannot allocate device memory when they score (an engine that
reserves all free HBM for its KV cache up front, code that may not call the
CUDA allocator, a real-time loop that cannot afford an allocation mid-step).
For them the library keeps its own query-prep workspace in a file-scope device
array.  These tests call that entry point through the C ABI twice in a row,
with different inputs, and check each result against the regular entry point
given a caller-owned workspace (and, at the row limit, a sample of rows with
the oracle).  The file sorts last so that a run stopping at
the first failure has already run every other test; it also passes alone in a
fresh process, where the first call does the per-device set-up.
"""
import numpy as np
import pytest
import torch

import qsa_inputs as qi
from qsa_cases import EPS, THETA, assert_close

pytestmark = pytest.mark.gpu


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def make_case(seed, n_rows, tokens):
    rng = qi.rng_for(2, salt=seed)
    fq = qi.fused_qk(rng, n_rows)
    qw, _ = qi.norm_weights(rng)
    keys = qi.normal_bf16(rng, (tokens // 4, 128))
    pos = rng.integers(0, tokens, size=n_rows).astype(np.int32)
    pos[:3] = [0, 3, tokens - 1]
    return fq, qw, keys, pos


def test_noalloc_matches_workspace_entry_on_two_calls():
    import sparse_attention_token_qsa_gb300 as qsa

    tokens = 6000
    c, s = qsa.qsa_rope_tables(tokens, THETA)
    cd, sd = dev(c), dev(s)
    cols = tokens // 4 + 4 - (tokens // 4) % 4
    for seed, n_rows in ((1, 300), (2, 137)):   # two calls in a row, different inputs
        fq, qw, keys, pos = make_case(seed, n_rows, tokens)
        args = (dev(fq), 640, dev(pos), None, n_rows, tokens, dev(qw), cd, sd, tokens, EPS,
                dev(keys))
        want = torch.full((n_rows, cols), -7.0, dtype=torch.float32, device="cuda")
        st = qsa.new_status()
        qsa.qsa_score_rows_with(*args, None, want, cols, st, path=qsa.QSA_SCORE_TCGEN05,
                                workspace=qsa.new_workspace(n_rows))
        assert qsa.qsa_read_status(st) == (0, 0)
        got = torch.full((n_rows, cols), -7.0, dtype=torch.float32, device="cuda")
        st = qsa.new_status()
        qsa.qsa_score_rows_noalloc(*args, got, cols, st)
        assert qsa.qsa_read_status(st) == (0, 0)
        g, w = got.cpu().numpy(), want.cpu().numpy()
        assert np.array_equal(g == -7.0, w == -7.0)      # the same entries written
        assert_close(g, w, f"no-alloc scores, call with {n_rows} rows")


def test_noalloc_refuses_more_rows_than_its_array_holds():
    import sparse_attention_token_qsa_gb300 as qsa

    lib = qsa.library()
    # refused on the host before any pointer is used: the pointers are never read
    fake = 0x10000
    P = lambda x: __import__("ctypes").c_void_p(x)
    rc = lib.qsa_score_rows_noalloc(P(fake), 640, P(fake), None, qsa.QSA_NOALLOC_MAX_ROWS + 1,
                                    4096, P(fake), P(fake), P(fake), 4096, 1e-6, P(fake), P(fake),
                                    1024, P(fake), None)
    assert rc == qsa.QSA_ERR_INVALID_VALUE
    assert lib.qsa_score_rows_noalloc(None, 640, None, None, 0, 4096, None, None, None, 4096, 1e-6,
                                      None, None, 1024, None, None) == qsa.QSA_OK


def test_noalloc_at_its_row_limit_matches_workspace_entry_and_oracle(orc):
    """Exactly QSA_NOALLOC_MAX_ROWS rows: the whole array is in use and the last
    query box of the tensor-core scorer ends at the array's end.  Compared with
    the regular entry point given a caller workspace of the same size, and a
    sample of rows with the oracle."""
    import sparse_attention_token_qsa_gb300 as qsa

    n_rows, tokens = qsa.QSA_NOALLOC_MAX_ROWS, 2048
    c, s = qsa.qsa_rope_tables(tokens, THETA)
    cd, sd = dev(c), dev(s)
    cols = tokens // 4
    fq, qw, keys, pos = make_case(3, n_rows, tokens)
    args = (dev(fq), 640, dev(pos), None, n_rows, tokens, dev(qw), cd, sd, tokens, EPS, dev(keys))
    want = torch.full((n_rows, cols), -7.0, dtype=torch.float32, device="cuda")
    st = qsa.new_status()
    ws = torch.empty(qsa.qsa_score_workspace_bytes(n_rows), dtype=torch.uint8, device="cuda")
    qsa.qsa_score_rows_with(*args, None, want, cols, st, path=qsa.QSA_SCORE_TCGEN05, workspace=ws)
    assert qsa.qsa_read_status(st) == (0, 0)
    got = torch.full((n_rows, cols), -7.0, dtype=torch.float32, device="cuda")
    st = qsa.new_status()
    qsa.qsa_score_rows_noalloc(*args, got, cols, st)
    assert qsa.qsa_read_status(st) == (0, 0)
    g, w = got.cpu().numpy(), want.cpu().numpy()
    assert np.array_equal(g == -7.0, w == -7.0)
    assert_close(g, w, "no-alloc scores at the row limit")
    rows = np.r_[0:8, n_rows - 56:n_rows]           # the first rows and the array's last rows
    o = np.full((len(rows), cols), -7.0, np.float32)
    rc, _ = orc.score_rows(fq[rows], 640, pos[rows], len(rows), tokens, qw, c, s, EPS, keys, o,
                           cols)
    assert rc == 0
    assert_close(g[rows], o, "no-alloc scores at the row limit vs the oracle")
