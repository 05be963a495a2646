"""Seeded random parity cases: shapes, budgets and score distributions drawn
at random (fixed seeds), each compared with the oracle bit for bit.

Selection: few long rows (clusters, key cache), many 64k-sized rows (two
passes, keys re-read), many 256k-sized rows (sampled band), small rows; scores
uniform, relu-like, quantised with masses of zeros, integer ties, signed and
extreme, or differing only in their lowest mantissa bits; signed zeros
sprinkled in; masks at odd byte offsets.

Fused decode: random row counts, contexts and positions, new blocks pooled in
the launch; scores equal to a two-kernel path's (the tensor-core scorer's, or
the streaming scorer's when the call falls back), masks to the oracle's
selection over them, and one workspace reused by every call left zero.
"""
import numpy as np
import pytest
import torch

import qsa_inputs as qi
from qsa_cases import EPS, THETA, index_select_tc, oracle_masks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qsa():
    import sparse_attention_token_qsa_gb300 as m

    return m


def d16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def random_scores(rng, kind, rows, cols):
    if kind == "uniform":
        sc = rng.random((rows, cols), dtype=np.float32)
    elif kind == "relu":
        sc = np.maximum(rng.standard_normal((rows, cols)).astype(np.float32), 0) * np.float32(3)
    elif kind == "stress":
        sc = qi.stress_scores(rng, rows, cols, zero_frac=float(rng.random()),
                              levels=int(rng.integers(1, 200)))
    elif kind == "ties":
        sc = np.round(rng.random((rows, cols)) * rng.integers(1, 50)).astype(np.float32)
    elif kind == "signed":
        scale = np.float32(rng.choice([1e-30, 1.0, 1e30]))
        sc = rng.standard_normal((rows, cols)).astype(np.float32) * scale
    else:  # low mantissa bits only
        sc = (np.float32(1.5) + rng.integers(0, 64, size=(rows, cols)).astype(np.float32)
              * np.float32(2.0 ** -22)).astype(np.float32)
    if rng.random() < 0.3:
        z = rng.random((rows, cols)) < 0.3
        sc[z] = np.where(rng.random(int(z.sum())) < 0.5, np.float32(0.0), np.float32(-0.0))
    return sc


@pytest.mark.parametrize("seed", range(6))
def test_select_random_cases(qsa, orc, seed):
    rng = qi.rng_for(9, salt=seed)
    kinds = ["uniform", "relu", "stress", "ties", "signed", "lowbits"]
    for _ in range(5):
        kind = kinds[int(rng.integers(len(kinds)))]
        shape = int(rng.integers(4))
        if shape == 0:
            rows, tokens = int(rng.integers(1, 9)), int(rng.integers(65536, 300000))
        elif shape == 1:
            rows, tokens = int(rng.integers(305, 340)), int(rng.integers(30000, 70000))
        elif shape == 2:
            rows, tokens = 305, int(rng.integers(131073, 262145))
        else:
            rows, tokens = int(rng.integers(1, 40)), int(rng.integers(1, 9000))
        cols = ((tokens // 4 + 3) // 4) * 4 + 4 * int(rng.integers(0, 3))
        budget = int(rng.choice([4, 512, 2044, 2048])) if rng.random() < 0.4 \
            else int(4 * rng.integers(1, 513))
        sc = random_scores(rng, kind, rows, cols)
        pos = rng.integers(0, tokens, size=rows).astype(np.int32)
        if rng.random() < 0.5:
            pos[:] = tokens - 1 - rng.integers(0, 4, size=rows)
        off = int(rng.integers(0, 4))
        buf = torch.full((rows * tokens + off + 16,), 0xAB, dtype=torch.uint8, device="cuda")
        mask = buf[off:off + rows * tokens]
        st = qsa.new_status()
        qsa.qsa_select_mask(torch.from_numpy(sc).cuda(), cols, torch.from_numpy(pos).cuda(), rows,
                            tokens, budget, mask, st)
        what = (kind, rows, tokens, cols, budget, off)
        assert qsa.qsa_read_status(st) == (0, 0), what
        g = buf.cpu().numpy()
        assert np.all(g[:off] == 0xAB) and np.all(g[off + rows * tokens:] == 0xAB), what
        got = g[off:off + rows * tokens].reshape(rows, tokens)
        want, codes = oracle_masks(orc, sc, cols, pos, tokens, budget)
        bad = [r for r in range(rows) if not np.array_equal(got[r], want[r])]
        assert not bad, (what, bad[:5])


def test_decode_random_cases(qsa, orc):
    rng = qi.rng_for(9, salt=100)
    max_t = 90000
    c, s = qsa.qsa_rope_tables(max_t + 8, THETA)
    cd, sd = d16(c), d16(s)
    ws = qsa.new_decode_workspace(8, max_t)
    for _ in range(20):
        rows = int(rng.integers(1, 9))
        tokens = int(rng.integers(4, max_t))
        nb = tokens // 4
        raw = qi.normal_bf16(rng, (tokens, 128))
        qw, kw = qi.norm_weights(rng)
        q = qi.normal_bf16(rng, (rows, 512))
        pos = rng.integers(0, tokens, size=rows).astype(np.int32)
        pos[0] = tokens - 1
        budget = int(4 * rng.integers(1, 513)) if rng.random() < 0.5 else 2048
        cols = ((nb + 3) // 4) * 4 + 4 * int(rng.integers(0, 2))
        first = int(rng.integers(0, max(1, nb)))
        cnt = int(rng.integers(0, min(200, nb - first) + 1)) if nb > first else 0
        outs = []
        for entry in ("decode", "tc", "stream"):
            cache = torch.zeros((max(nb, 1), 128), dtype=torch.int16, device="cuda")
            if nb:
                qsa.qsa_pool_blocks(d16(raw).view(-1), 128, 0, nb, d16(kw), cd, sd, c.shape[0], EPS,
                                    cache)
            if cnt:
                cache[first:first + cnt] = 0x7FAB          # pooled by the call itself
            sc = torch.full((rows, cols), -7.0, dtype=torch.float32, device="cuda")
            mask = torch.full((rows, tokens), 0xAB, dtype=torch.uint8, device="cuda")
            st = qsa.new_status()
            keys = d16(raw).view(-1)[4 * first * 128:] if cnt else d16(raw)
            args = (keys, 128, first if cnt else 0, cnt, d16(kw), d16(q), 512,
                    torch.from_numpy(pos).cuda(), rows, tokens, d16(qw), cd, sd, c.shape[0], EPS,
                    budget, cache, sc, cols, mask, st)
            if entry == "decode":
                qsa.qsa_decode_index_select(*args, ws)
            elif entry == "tc":
                index_select_tc(qsa, *args)
            else:
                qsa.qsa_index_select(*args)
            outs.append((qsa.qsa_read_status(st), sc.cpu().numpy(), mask.cpu().numpy(),
                         cache.cpu().numpy()))
        same = [o for o in outs[1:] if np.array_equal(o[1], outs[0][1])]
        (dc, dsc, dm, dk), (pc, psc, pm, pk) = outs[0], (same[0] if same else outs[1])
        what = (rows, tokens, budget, first, cnt)
        assert dc == (0, 0) and pc == (0, 0), what
        assert np.array_equal(dk, pk), what
        wrote = dsc != -7.0
        assert np.array_equal(wrote, psc != -7.0) and np.array_equal(dsc[wrote], psc[wrote]), what
        want, _ = oracle_masks(orc, dsc, cols, pos, tokens, budget)
        assert np.array_equal(dm, want) and np.array_equal(pm, want), what
        assert int(ws.count_nonzero()) == 0, what
