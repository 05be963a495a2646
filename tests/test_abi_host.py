"""Host-only checks of the C ABI: no GPU, no launch.

Every call here is refused (or is an empty launch) before the library forms a
launch, so the dangling pointers below are never dereferenced.  Each refusal
test first makes the same call with valid arguments and a zero extent, which
must return QSA_OK: that positive control keeps the refusals from passing
vacuously (the pattern of the refusal test in PR #1160's review).
"""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qsa.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    import sparse_attention_token_qsa_gb300 as qsa

    return qsa.library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    import sparse_attention_token_qsa_gb300 as qsa

    names = header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(qsa.EXPORTED) == names


def test_version_and_status_strings(lib):
    assert lib.qsa_version() >= 100
    for code in range(7):
        assert lib.qsa_status_string(code)
    assert b"unknown" in lib.qsa_status_string(99)


A = 0x10000          # 16-byte aligned dangling pointer
B = 0x20000
U = 0x10002          # misaligned


def P(x):
    return ctypes.c_void_p(x)


def select(lib, scores=A, score_cols=64, pos=B, n_rows=1, tokens=256, budget=2048, mask=A,
           status=B):
    return lib.qsa_select_mask(P(scores), score_cols, P(pos), n_rows, tokens, budget, P(mask),
                               P(status), None)


def test_select_refusals(lib):
    assert select(lib, n_rows=0) == 0 and select(lib, tokens=0) == 0        # empty: no-op
    for kw in (dict(budget=0), dict(budget=-4), dict(budget=6), dict(budget=2052),
               dict(n_rows=-1), dict(tokens=-1), dict(score_cols=-4),
               dict(score_cols=60), dict(score_cols=66), dict(scores=0), dict(pos=0),
               dict(mask=0), dict(scores=U)):
        assert select(lib, **kw) == 1, kw
        assert select(lib, **{**kw, "n_rows": 0}) in (0, 1)
    # budget and negative extents are refused even on an empty launch
    assert select(lib, n_rows=0, budget=6) == 1
    assert select(lib, n_rows=-1, tokens=0) == 1


def pool(lib, keys=A, key_stride=640, first=0, n=0, w=A, cos=A, sin=A, rows=1 << 16, eps=1e-6,
         out=A):
    return lib.qsa_pool_blocks(P(keys), key_stride, first, n, P(w), P(cos), P(sin), rows, eps,
                               P(out), None)


def test_pool_refusals(lib):
    assert pool(lib) == 0                                  # zero blocks: no-op
    for kw in (dict(key_stride=120), dict(key_stride=644), dict(keys=U), dict(out=U), dict(w=U),
               dict(cos=0), dict(sin=0), dict(keys=0), dict(out=0), dict(eps=-1.0),
               dict(eps=float("nan")), dict(rows=4 * 9), dict(first=-1)):
        assert pool(lib, n=10, **kw) == 1, kw
    assert pool(lib, n=-1) == 1


def score(lib, q=A, q_stride=640, pos=B, vis=None, n_rows=0, tokens=4096, w=A, cos=A, sin=A,
          rows=4096, eps=1e-6, keys=A, base=None, scores=A, cols=1024, status=B, path=0, ws=None,
          wsb=0):
    return lib.qsa_score_rows_with(P(q), q_stride, P(pos), P(vis or 0), n_rows, tokens, P(w),
                                   P(cos), P(sin), rows, eps, P(keys), P(base or 0), P(scores),
                                   cols, P(status), path, P(ws or 0), wsb, None)


def test_score_refusals(lib):
    assert score(lib) == 0                                 # zero rows: no-op
    for kw in (dict(q_stride=504), dict(q_stride=644), dict(q=U), dict(keys=U), dict(scores=U),
               dict(cols=1020), dict(cols=1022), dict(rows=4095), dict(eps=-1e-6),
               dict(q=0), dict(pos=0), dict(keys=0), dict(scores=0), dict(w=0), dict(cos=0),
               dict(path=4), dict(path=-1), dict(path=2, base=B, ws=A, wsb=1 << 20), dict(path=2),
               dict(path=2, ws=A, wsb=3 * 1024 - 1), dict(path=2, ws=U, wsb=1 << 20),
               dict(wsb=-1)):
        assert score(lib, n_rows=3, **kw) == 1, kw
    assert score(lib, n_rows=-3) == 1
    assert lib.qsa_score_workspace_bytes(3) == 3 * 1024
    assert lib.qsa_score_workspace_bytes(0) == 0 and lib.qsa_score_workspace_bytes(-1) == -1


def test_index_select_refusals(lib):
    def call(**kw):
        a = dict(keys=A, ks=640, f=0, nb=0, kw=A, q=A, qs=640, pos=B, n=0, tokens=4096, qw=A,
                 cos=A, sin=A, rows=4096, eps=1e-6, budget=2048, bk=A, sc=A, cols=1024, mask=A,
                 st=B, ws=0, wsb=0)
        a.update(kw)
        return lib.qsa_index_select(P(a["keys"]), a["ks"], a["f"], a["nb"], P(a["kw"]), P(a["q"]),
                                    a["qs"], P(a["pos"]), a["n"], a["tokens"], P(a["qw"]),
                                    P(a["cos"]), P(a["sin"]), a["rows"], a["eps"], a["budget"],
                                    P(a["bk"]), P(a["sc"]), a["cols"], P(a["mask"]), P(a["st"]),
                                    P(a["ws"]), a["wsb"], None)
    assert call() == 0
    assert call(budget=2047) == 1
    assert call(nb=4, ks=100) == 1
    assert call(n=2, qs=100) == 1
    assert call(n=2, cols=100) == 1
    assert call(wsb=-5) == 1


def test_decode_workspace_bytes(lib):
    row = 262400 + 8 * (65536 // 4)         # histogram + counters, then the candidates
    assert lib.qsa_decode_workspace_bytes(1, 65536) == (row + 255) // 256 * 256
    assert lib.qsa_decode_workspace_bytes(3, 65536) == 3 * ((row + 255) // 256 * 256)
    assert lib.qsa_decode_workspace_bytes(2, 4099) % 256 == 0
    assert lib.qsa_decode_workspace_bytes(0, 65536) == 0
    assert lib.qsa_decode_workspace_bytes(-1, 65536) == -1


def test_decode_index_select_refusals(lib):
    """Decided on the host before any launch: the pointers are never read."""
    def call(**kw):
        a = dict(keys=A, ks=640, f=0, nb=0, kw=A, q=A, qs=640, pos=B, n=2, tokens=4096, qw=A,
                 cos=A, sin=A, rows=4096, eps=1e-6, budget=2048, bk=A, sc=A, cols=1024, mask=A,
                 st=B, ws=0, wsb=0)
        a.update(kw)
        return lib.qsa_decode_index_select(P(a["keys"]), a["ks"], a["f"], a["nb"], P(a["kw"]),
                                           P(a["q"]), a["qs"], P(a["pos"]), a["n"], a["tokens"],
                                           P(a["qw"]), P(a["cos"]), P(a["sin"]), a["rows"],
                                           a["eps"], a["budget"], P(a["bk"]), P(a["sc"]),
                                           a["cols"], P(a["mask"]), P(a["st"]), P(a["ws"]),
                                           a["wsb"], None)
    need = lib.qsa_decode_workspace_bytes(2, 4096)
    assert call() == 1                               # no workspace
    assert call(ws=A, wsb=need - 1) == 1             # too small
    assert call(ws=A + 8, wsb=need) == 1             # not 16-byte aligned
    assert call(ws=A, wsb=need, budget=2047) == 1    # what qsa_index_select refuses
    assert call(ws=A, wsb=need, n=2, cols=100) == 1
    assert call(n=0) == 0                            # nothing to do: no workspace needed


def test_mask_tokens_refusals(lib):
    def call(mask=A, n=2, tokens=4096, sel=A, cols=2051, n_sel=B):
        return lib.qsa_mask_tokens(P(mask), n, tokens, P(sel), cols, P(n_sel), None)
    assert call(n=0) == 0                            # nothing to do
    assert call(n=-1) == 1 and call(tokens=-1) == 1 and call(cols=-1) == 1
    assert call(n_sel=0) == 1 and call(mask=0) == 1 and call(sel=0) == 1
    assert call(n=1 << 30, tokens=1 << 20) == 1      # extent past the library's bound


def test_gather_kv_refusals(lib):
    def call(**kw):
        a = dict(k=A, v=B, width=512, pages=4096, table=A, tlen=4096, tcols=4096, psz=16, sel=A,
                 scols=2051, n_sel=B, n=2, max_sel=2051, ko=A, vo=B, orows=2051, st=B)
        a.update(kw)
        return lib.qsa_gather_kv(P(a["k"]), P(a["v"]), a["width"], a["pages"], P(a["table"]),
                                 a["tlen"], a["tcols"], a["psz"], P(a["sel"]), a["scols"],
                                 P(a["n_sel"]), a["n"], a["max_sel"], P(a["ko"]), P(a["vo"]),
                                 a["orows"], P(a["st"]), None)
    assert call(n=0) == 0 and call(max_sel=0) == 0 and call(width=0) == 0   # nothing to do
    for kw in (dict(width=12), dict(width=-8), dict(psz=0), dict(max_sel=2052),
               dict(orows=2050), dict(tcols=4095), dict(pages=-1), dict(k=U), dict(vo=U),
               dict(table=0), dict(st=0), dict(n_sel=0), dict(tlen=1 << 28, tcols=0)):
        assert call(**kw) == 1, kw


def test_sparse_attn_refusals(lib):
    def call(**kw):
        a = dict(q=A, qs=4096, nq=16, nkv=2, hd=256, k=A, v=B, pages=64, psz=16, table=A, tlen=64,
                 tcols=64, sel=A, scols=2051, n_sel=B, n=2, max_sel=2051, scale=0.0625, out=B,
                 os=4096, st=B)
        a.update(kw)
        return lib.qsa_sparse_attn(P(a["q"]), a["qs"], a["nq"], a["nkv"], a["hd"], P(a["k"]),
                                   P(a["v"]), a["pages"], a["psz"], P(a["table"]), a["tlen"],
                                   a["tcols"], P(a["sel"]), a["scols"], P(a["n_sel"]), a["n"],
                                   a["max_sel"], a["scale"], P(a["out"]), a["os"], P(a["st"]), None)
    assert call(n=0) == 0                             # nothing to do
    for kw in (dict(nq=15), dict(nkv=0), dict(hd=64), dict(psz=0), dict(psz=-3), dict(max_sel=2052),
               dict(tcols=63), dict(qs=4095), dict(qs=4100), dict(os=4000), dict(q=U),
               dict(out=U), dict(k=0), dict(sel=0), dict(table=0), dict(n_sel=0),
               dict(scale=float("nan")), dict(scale=float("inf")), dict(n=-1)):
        assert call(**kw) == 1, kw


def test_qk_proj_refusals(lib):
    def call(**kw):
        a = dict(x=A, xs=2560, w=B, n=2048, hid=2560, out=640, y=A, ys=640, st=B)
        a.update(kw)
        return lib.qsa_qk_proj(P(a["x"]), a["xs"], P(a["w"]), a["n"], a["hid"], a["out"],
                               P(a["y"]), a["ys"], P(a["st"]), None)
    assert call(n=0) == 0                             # nothing to do
    for kw in (dict(hid=0), dict(hid=2564), dict(out=648), dict(out=0), dict(xs=2552),
               dict(xs=2561), dict(ys=636), dict(x=U), dict(y=U), dict(w=0), dict(st=0),
               dict(n=-1), dict(n=65535 * 128 + 1)):
        assert call(**kw) == 1, kw


def test_status_calls_refuse_null(lib):
    assert lib.qsa_reset_status(None, None) == 1
    assert lib.qsa_read_status(None, None, None, None) == 1


def test_rope_tables_match_oracle(lib, orc):
    import sparse_attention_token_qsa_gb300 as qsa

    for theta in (10000.0, 1e7):
        c1, s1 = qsa.qsa_rope_tables(70000, theta)
        c2, s2 = orc.rope_table(70000, theta)
        assert np.array_equal(c1, c2) and np.array_equal(s1, s2)
    assert lib.qsa_rope_tables(-1, 1e4, None, None) == 1
    assert lib.qsa_rope_tables(4, 0.0, P(A), P(A)) == 1
    assert lib.qsa_rope_tables(0, 1e4, None, None) == 0


def test_wait_limit_is_settable_and_refuses_non_positive(lib):
    import sparse_attention_token_qsa_gb300 as qsa

    default = lib.qsa_wait_limit_cycles()
    assert default == 4000000000
    assert lib.qsa_set_wait_limit_cycles(0) == qsa.QSA_ERR_INVALID_VALUE
    assert lib.qsa_set_wait_limit_cycles(-7) == qsa.QSA_ERR_INVALID_VALUE
    assert lib.qsa_wait_limit_cycles() == default
    try:
        assert lib.qsa_set_wait_limit_cycles(12345) == qsa.QSA_OK
        assert lib.qsa_wait_limit_cycles() == 12345
    finally:
        assert lib.qsa_set_wait_limit_cycles(default) == qsa.QSA_OK
    assert lib.qsa_wait_limit_cycles() == default
