"""qsa_decode_index_select: pooling, scoring and selection with the fused
decode launch (one cooperative launch, each row over many CTAs), against the
oracle and against the single-stage entry points.

Its scores come from the same tcgen05 MMA per (block, head) as the tensor-core
scorer of qsa_score_rows_with, so they must equal that path's bit for bit (or,
when the rows' CTAs cannot all be co-resident and the call falls back to the
streaming scorer, that scorer's) and lie within tolerance of the oracle's; its
masks must equal, byte for byte, the oracle's selection over the GPU's own
scores (selection is exact integer work on given scores).  The zeroed
workspace must be zero again after every call that completes.
"""
import numpy as np
import pytest
import torch

import qsa_inputs as qi
from qsa_cases import (BUDGET, EPS, THETA, assert_close, assert_masks_agree_up_to_tolerance,
                       check_mask_structure, index_select_tc, long_keys_case, oracle_masks,
                       oracle_scores)

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


def run_both(qsa, tables, cache_np, q_np, pos_np, tokens, cols, qw, budget=BUDGET, mask_offset=0,
             keys=None, pool=(0, 0), ws=None):
    """One call of the decode entry and of the two-kernel path with each scorer
    on identical inputs; returns the decode outputs, the outputs of the
    two-kernel path whose scores equal the decode call's (the tensor-core one
    if neither does), and the workspace."""
    c, s, cd, sd = tables
    n_rows = len(pos_np)
    out = []
    for entry in ("decode", "tc", "stream"):
        cache = dev(cache_np.copy())
        sc = torch.full((n_rows, cols), -7.0, dtype=torch.float32, device="cuda")
        buf = torch.full((n_rows * tokens + mask_offset + 16,), 0xAB, dtype=torch.uint8,
                         device="cuda")
        mask = buf[mask_offset:mask_offset + n_rows * tokens]
        st = qsa.new_status()
        kd = keys if keys is not None else cache
        args = (kd, 128, pool[0], pool[1], dev(np.zeros(128, np.uint16)), dev(q_np), 512,
                dev(pos_np), n_rows, tokens, dev(qw), cd, sd, c.shape[0], EPS, budget, cache, sc,
                cols, mask, st)
        if entry == "decode":
            if ws is None:
                ws = qsa.new_decode_workspace(n_rows, tokens)
            qsa.qsa_decode_index_select(*args, ws)
        elif entry == "tc":
            index_select_tc(qsa, *args)
        else:
            qsa.qsa_index_select(*args)
        torch.cuda.synchronize()
        g = buf.cpu().numpy()
        assert np.all(g[:mask_offset] == 0xAB) and np.all(g[mask_offset + n_rows * tokens:] == 0xAB)
        out.append((sc.cpu().numpy(), mask.view(n_rows, tokens).cpu().numpy(),
                    qsa.qsa_read_status(st), cache.cpu().numpy().view(np.uint16)))
    same = [o for o in out[1:] if np.array_equal(o[0], out[0][0])]
    return out[0], (same[0] if same else out[1]), ws


def test_decode_steps_match_oracle_and_two_kernel_path(qsa, orc, tables):
    """Decode at 64k, eight consecutive steps: each pools the block its token
    completes, then one fused launch scores and selects."""
    case = long_keys_case()
    keys = case["keys"]
    c, s, cd, sd = tables
    tokens = 65536
    nb = tokens // 4
    first = 65528
    keys_o = orc.pool_blocks(keys, 128, 0, nb, case["k_norm_w"], c, s, EPS)
    cache = dev(keys_o.copy())
    cache[(first + 1) // 4:] = 0x7FAB              # blocks not yet pooled
    keys_d = dev(keys)
    kw, qw = dev(case["k_norm_w"]), dev(case["q_norm_w"])
    ws = qsa.new_decode_workspace(1, tokens)
    for k, p in enumerate(range(first, tokens)):
        completes = (p + 1) % 4 == 0
        b_new = (p + 1) // 4 - 1
        pos = np.array([p], np.int32)
        sc = torch.full((1, nb), -7.0, dtype=torch.float32, device="cuda")
        mask = torch.full((1, tokens), 0xAB, dtype=torch.uint8, device="cuda")
        st = qsa.new_status()
        qsa.qsa_decode_index_select(keys_d.view(-1)[4 * b_new * 128:] if completes else keys_d, 128,
                                    b_new if completes else 0, 1 if completes else 0, kw,
                                    dev(case["q"][k:k + 1]), 512, dev(pos), 1, tokens, qw, cd, sd,
                                    c.shape[0], EPS, BUDGET, cache, sc, nb, mask, st, ws)
        assert qsa.qsa_read_status(st) == (0, 0)
        assert int(ws.count_nonzero()) == 0, "workspace not left zero"
        n = (p + 1) // 4
        assert np.array_equal(cache[:n].cpu().numpy().view(np.uint16), keys_o[:n])
        got_sc = sc.cpu().numpy()
        sc_o, _ = oracle_scores(orc, case["q"][k:k + 1], 512, pos, tokens, case["q_norm_w"], c, s,
                                keys_o, nb)
        assert_close(got_sc, sc_o, f"decode step {p}")
        got = mask.cpu().numpy()[0]
        check_mask_structure(got, p, tokens, BUDGET)
        # selection: bit-exact against the oracle on the GPU's own scores
        want, codes = oracle_masks(orc, got_sc, nb, pos, tokens, BUDGET)
        assert codes == [0] and np.array_equal(got, want[0]), f"step {p}"
        mask_o, _ = oracle_masks(orc, sc_o, nb, pos, tokens, BUDGET)
        assert_masks_agree_up_to_tolerance(got, mask_o[0], sc_o[0], p, BUDGET, f"step {p}")


@pytest.mark.parametrize("tokens,mask_offset", [(65536, 0), (30001, 3), (4099, 1)])
def test_decode_rows_of_every_kind(qsa, orc, tables, tokens, mask_offset):
    """Several rows in one launch: under the budget (the whole prefix), at the
    inert bound, truncating, the very first tokens; ragged token counts, mask
    rows at odd byte offsets, score_cols with spare capacity."""
    rng = qi.rng_for(1, salt=tokens)
    nb = tokens // 4
    cols = ((nb + 3) // 4) * 4 + 8
    cache_np = qi.normal_bf16(rng, (nb, 128))
    pos = np.array([tokens - 1, min(2050, tokens - 1), 3, tokens - 2, 0, min(2051, tokens - 1),
                    tokens // 2], np.int32)
    q_np = qi.normal_bf16(rng, (len(pos), 512))
    qw, _ = qi.norm_weights(rng)
    (dsc, dmask, dst, _), (psc, pmask, pst, _), ws = run_both(
        qsa, tables, cache_np, q_np, pos, tokens, cols, qw, mask_offset=mask_offset)
    assert dst == (0, 0) and pst == (0, 0)
    assert int(ws.count_nonzero()) == 0
    wrote = dsc != -7.0
    assert np.array_equal(wrote, psc != -7.0)
    assert np.array_equal(dsc[wrote], psc[wrote]), "scores differ from the two-kernel path"
    assert np.array_equal(dmask, pmask), "masks differ from the two-kernel path"
    want, codes = oracle_masks(orc, dsc, cols, pos, tokens, BUDGET)
    assert all(c_ == 0 for c_ in codes)
    assert np.array_equal(dmask, want)
    c, s, _, _ = tables
    sc_o, _ = oracle_scores(orc, q_np, 512, pos, tokens, qw, c, s, cache_np, cols)
    for r in range(len(pos)):
        n = (pos[r] + 1) // 4
        assert_close(dsc[r, :n], sc_o[r, :n], f"row {r}")


def test_decode_exact_ties_cut_by_block_index(qsa, orc, tables):
    """Many blocks share one key, so their scores tie exactly; the ties straddle
    the keep-th place and are cut in ascending block order."""
    rng = qi.rng_for(1, salt=77)
    tokens = 65536
    nb = tokens // 4
    cache_np = qi.normal_bf16(rng, (nb, 128))
    q_np = qi.normal_bf16(rng, (3, 512))
    qw, _ = qi.norm_weights(rng)
    pos = np.array([tokens - 1, tokens - 3, 40003], np.int32)
    # one key repeated over 2000 blocks; a second, repeated over 600 blocks
    cache_np[rng.choice(nb, 2000, replace=False)] = cache_np[5]
    cache_np[rng.choice(nb, 600, replace=False)] = cache_np[9]
    (dsc, dmask, dst, _), (psc, pmask, pst, _), ws = run_both(qsa, tables, cache_np, q_np, pos,
                                                            tokens, nb, qw)
    assert dst == (0, 0) and int(ws.count_nonzero()) == 0
    assert np.array_equal(dmask, pmask)
    want, _ = oracle_masks(orc, dsc, nb, pos, tokens, BUDGET)
    assert np.array_equal(dmask, want)


def test_decode_all_zero_scores(qsa, orc, tables):
    """q = 0: every score is +0.0, the whole row ties; the first keep blocks win."""
    rng = qi.rng_for(1, salt=78)
    tokens = 16384
    nb = tokens // 4
    cache_np = qi.normal_bf16(rng, (nb, 128))
    q_np = np.zeros((2, 512), np.uint16)
    qw, _ = qi.norm_weights(rng)
    pos = np.array([tokens - 1, 9000], np.int32)
    (dsc, dmask, dst, _), (_, pmask, _, _), ws = run_both(qsa, tables, cache_np, q_np, pos, tokens,
                                                         nb, qw)
    assert dst == (0, 0) and int(ws.count_nonzero()) == 0
    assert np.all(dsc[0] == 0)
    assert np.array_equal(dmask, pmask)
    assert np.all(dmask[0, :2048] == 1) and np.all(dmask[0, 2048:] == 0)


def test_decode_nonfinite_and_out_of_range_rows(qsa, orc, tables):
    """A NaN key makes row 1's scores non-finite: the row is reported and its mask
    left alone; an out-of-range position is reported too; the other rows are
    correct and the workspace is left zero."""
    rng = qi.rng_for(1, salt=79)
    tokens = 65536
    nb = tokens // 4
    cache_np = qi.normal_bf16(rng, (nb, 128))
    q_np = qi.normal_bf16(rng, (3, 512))
    qw, _ = qi.norm_weights(rng)
    c, s, cd, sd = tables
    for bad_row, pos, code in ((1, np.array([65535, 65535, 30000], np.int32), 4),
                               (2, np.array([65535, 40000, 65536], np.int32), 3)):
        cache = cache_np.copy()
        if code == 4:
            cache[12345, 7] = 0x7FC0                 # NaN, read by rows 0 and 1 ...
            pos[0] = 40000                           # ... but row 0 stops before it
        ws = qsa.new_decode_workspace(3, tokens)
        sc = torch.full((3, nb), -7.0, dtype=torch.float32, device="cuda")
        mask = torch.full((3, tokens), 0xAB, dtype=torch.uint8, device="cuda")
        st = qsa.new_status()
        cache_d = dev(cache)
        qsa.qsa_decode_index_select(cache_d, 128, 0, 0, dev(np.zeros(128, np.uint16)), dev(q_np),
                                    512, dev(pos), 3, tokens, dev(qw), cd, sd, c.shape[0], EPS,
                                    BUDGET, cache_d, sc, nb, mask, st, ws)
        assert qsa.qsa_read_status(st) == (code, bad_row)
        assert int(ws.count_nonzero()) == 0
        got = mask.cpu().numpy()
        assert np.all(got[bad_row] == 0xAB)
        got_sc = sc.cpu().numpy()
        for r in range(3):
            if r == bad_row:
                continue
            want, _ = oracle_masks(orc, got_sc, nb, pos, tokens, BUDGET, rows=[r])
            assert np.array_equal(got[r], want[0]), r


def test_decode_many_rows_take_the_two_kernel_path(qsa, orc, tables):
    """More rows than can be co-resident: the call falls back to the scorer and
    the selector (same results, the workspace untouched)."""
    rng = qi.rng_for(1, salt=80)
    tokens = 65536
    nb = tokens // 4
    cache_np = qi.normal_bf16(rng, (nb, 128))
    n_rows = 40
    pos = rng.integers(tokens // 2, tokens, size=n_rows).astype(np.int32)
    q_np = qi.normal_bf16(rng, (n_rows, 512))
    qw, _ = qi.norm_weights(rng)
    (dsc, dmask, dst, _), (psc, pmask, _, _), ws = run_both(qsa, tables, cache_np, q_np, pos,
                                                           tokens, nb, qw)
    assert dst == (0, 0) and int(ws.count_nonzero()) == 0
    assert np.array_equal(dmask, pmask)
    assert np.array_equal(dsc[dsc != -7.0], psc[psc != -7.0])


def test_decode_workspace_reused_across_shapes(qsa, orc, tables):
    """One workspace, sized for the largest call, serves calls of 1, 4 and 2 rows
    at different context lengths in turn."""
    rng = qi.rng_for(1, salt=81)
    ws = qsa.new_decode_workspace(4, 65536)
    for n_rows, tokens in ((1, 65536), (4, 20000), (2, 65536), (1, 8192)):
        nb = tokens // 4
        cache_np = qi.normal_bf16(rng, (nb, 128))
        pos = rng.integers(tokens - 5000 if tokens > 5000 else 0, tokens, size=n_rows).astype(np.int32)
        q_np = qi.normal_bf16(rng, (n_rows, 512))
        qw, _ = qi.norm_weights(rng)
        (dsc, dmask, dst, _), (_, pmask, _, _), _ = run_both(qsa, tables, cache_np, q_np, pos,
                                                            tokens, nb, qw, ws=ws)
        assert dst == (0, 0) and int(ws.count_nonzero()) == 0
        assert np.array_equal(dmask, pmask), (n_rows, tokens)


def test_decode_with_inputs_and_mask_in_pinned_host_memory(qsa, orc, tables):
    """A decode step whose query rows, positions, raw keys (pooled this call) and
    mask live in pinned host memory, read and written in place by the kernels,
    gives exactly the results of the same call on device buffers."""
    rng = qi.rng_for(1, salt=82)
    c, s, cd, sd = tables
    tokens = 65536
    nb = tokens // 4
    raw = qi.normal_bf16(rng, (tokens, 128))
    qw_h, kw_h = qi.norm_weights(rng)
    cache_np = orc.pool_blocks(raw, 128, 0, nb - 1, kw_h, c, s, EPS, total_blocks=nb)
    q_np = qi.normal_bf16(rng, (2, 512))
    pos_np = np.array([tokens - 1, 50001], np.int32)     # row 0 completes block nb - 1
    outs = []
    for where in ("device", "host"):
        cache = dev(cache_np.copy())
        sc = torch.full((2, nb), -7.0, dtype=torch.float32, device="cuda")
        st = qsa.new_status()
        ws = qsa.new_decode_workspace(2, tokens)
        if where == "device":
            keys, q, pos = dev(raw), dev(q_np), dev(pos_np)
            mask = torch.full((2, tokens), 0xAB, dtype=torch.uint8, device="cuda")
        else:
            keys = torch.from_numpy(raw.view(np.int16)).pin_memory()
            q = torch.from_numpy(q_np.view(np.int16)).pin_memory()
            pos = torch.from_numpy(pos_np).pin_memory()
            mask = torch.full((2, tokens), 0xAB, dtype=torch.uint8).pin_memory()
        qsa.qsa_decode_index_select(keys.view(-1)[4 * (nb - 1) * 128:], 128, nb - 1, 1, dev(kw_h), q,
                                    512, pos, 2, tokens, dev(qw_h), cd, sd, c.shape[0], EPS, BUDGET,
                                    cache, sc, nb, mask, st, ws)
        assert qsa.qsa_read_status(st) == (0, 0)
        torch.cuda.synchronize()
        outs.append((cache.cpu().numpy(), sc.cpu().numpy(), mask.cpu().numpy().copy()))
        assert int(ws.count_nonzero()) == 0
    assert np.array_equal(outs[0][0], outs[1][0]), "pooled keys differ"
    assert np.array_equal(outs[0][1], outs[1][1]), "scores differ"
    assert np.array_equal(outs[0][2], outs[1][2]), "masks differ"
    want, _ = oracle_masks(orc, outs[1][1], nb, pos_np, tokens, BUDGET)
    assert np.array_equal(outs[1][2], want)


@pytest.mark.parametrize("first,count", [(16255, 2), (16300, 84), (16383, 1)])
def test_decode_pools_new_blocks_in_the_same_launch(qsa, orc, tables, first, count):
    """The fused launch pools the new blocks itself: a range straddling two CTAs'
    shares (each pools its own before its keys are copied), a long range, rows
    that see none of the new blocks; the cache, scores and masks equal those of
    the separate pool kernel and the oracle."""
    rng = qi.rng_for(1, salt=first)
    c, s, cd, sd = tables
    tokens = 65536
    nb = tokens // 4
    raw = qi.normal_bf16(rng, (tokens, 128))
    qw_h, kw_h = qi.norm_weights(rng)
    keys_o = orc.pool_blocks(raw, 128, 0, nb, kw_h, c, s, EPS)
    cache_np = keys_o.copy()
    cache_np[first:] = 0x7FAB                          # not pooled yet (NaN pattern)
    # the newest token completes block first + count - 1: no row sees further
    last = 4 * (first + count) - 1
    pos = np.array([last, 4 * first + 2, last - 1], np.int32)
    q_np = qi.normal_bf16(rng, (3, 512))
    outs = []
    for entry in ("decode", "tc", "stream"):
        cache = dev(cache_np)
        sc = torch.full((3, nb), -7.0, dtype=torch.float32, device="cuda")
        mask = torch.full((3, tokens), 0xAB, dtype=torch.uint8, device="cuda")
        st = qsa.new_status()
        args = (dev(raw).view(-1)[4 * first * 128:], 128, first, count, dev(kw_h), dev(q_np), 512,
                dev(pos), 3, tokens, dev(qw_h), cd, sd, c.shape[0], EPS, BUDGET, cache, sc, nb, mask,
                st)
        if entry == "decode":
            ws = qsa.new_decode_workspace(3, tokens)
            qsa.qsa_decode_index_select(*args, ws)
            torch.cuda.synchronize()
            assert int(ws.count_nonzero()) == 0
        elif entry == "tc":
            index_select_tc(qsa, *args)
        else:
            qsa.qsa_index_select(*args)
        assert qsa.qsa_read_status(st) == (0, 0)
        outs.append((cache.cpu().numpy().view(np.uint16), sc.cpu().numpy(), mask.cpu().numpy()))
    same = [o for o in outs[1:] if np.array_equal(o[1], outs[0][1])]
    outs = [outs[0], same[0] if same else outs[1]]
    top = first + count
    assert np.array_equal(outs[0][0][:top], keys_o[:top]), "pooled cache differs from the oracle"
    assert np.all(outs[0][0][top:] == 0x7FAB), "blocks past the new range were written"
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1]), "scores differ"
    assert np.array_equal(outs[0][2], outs[1][2]), "masks differ"
    want, _ = oracle_masks(orc, outs[0][1], nb, pos, tokens, BUDGET)
    assert np.array_equal(outs[0][2], want)


def test_decode_keep_th_key_far_below_the_top(qsa, orc, tables):
    """A few block keys scaled by 2^70 make a handful of scores ~2^70 times the
    rest: the keep-th score then lies thousands of 16-bit bins below the row's
    highest, outside the first window each CTA reads, so the bins below it are
    read a chunk at a time; the masks must still equal the two-kernel path and
    the oracle."""
    rng = qi.rng_for(1, salt=4097)
    tokens = 65536
    nb = tokens // 4
    cache_np = qi.normal_bf16(rng, (nb, 128))
    huge = rng.choice(nb - 100, 40, replace=False)
    cache_np[huge] = qi.to_bf16_bits(qi.bf16_bits_to_f32(cache_np[huge]) * np.float32(2.0 ** 70))
    q_np = qi.normal_bf16(rng, (3, 512))
    qw, _ = qi.norm_weights(rng)
    pos = np.array([tokens - 1, tokens - 3, 50001], np.int32)
    (dsc, dmask, dst, _), (psc, pmask, pst, _), ws = run_both(qsa, tables, cache_np, q_np, pos,
                                                            tokens, nb, qw)
    assert dst == (0, 0) and pst == (0, 0)
    assert int(ws.count_nonzero()) == 0
    assert np.isfinite(dsc[dsc != -7.0]).all()
    assert np.nanmax(dsc) > 2.0 ** 60            # the giant scores are there
    assert np.array_equal(dmask, pmask)
    want, codes = oracle_masks(orc, dsc, nb, pos, tokens, BUDGET)
    assert all(c == 0 for c in codes)
    assert np.array_equal(dmask, want)


def test_decode_long_rows_past_64k(qsa, orc):
    """Two rows of a 270000-token context (67500 blocks): the fused launch, or
    the two-kernel path when its CTAs do not fit, gives the results of one of
    the library's two-kernel paths and the oracle's selection over its scores."""
    tokens = 270000
    nb = tokens // 4
    c, s = qsa.qsa_rope_tables(tokens, THETA)
    cd, sd = dev(c), dev(s)
    rng = qi.rng_for(1, salt=270000)
    cache_np = qi.normal_bf16(rng, (nb, 128))
    q_np = qi.normal_bf16(rng, (2, 512))
    qw, _ = qi.norm_weights(rng)
    pos = np.array([tokens - 1, 100001], np.int32)
    outs = []
    for entry in ("decode", "tc", "stream"):
        cache = dev(cache_np)
        sc = torch.full((2, nb), -7.0, dtype=torch.float32, device="cuda")
        mask = torch.full((2, tokens), 0xAB, dtype=torch.uint8, device="cuda")
        st = qsa.new_status()
        args = (cache, 128, 0, 0, dev(np.zeros(128, np.uint16)), dev(q_np), 512, dev(pos), 2,
                tokens, dev(qw), cd, sd, tokens, EPS, BUDGET, cache, sc, nb, mask, st)
        if entry == "decode":
            qsa.qsa_decode_index_select(*args, qsa.new_decode_workspace(2, tokens))
        elif entry == "tc":
            index_select_tc(qsa, *args)
        else:
            qsa.qsa_index_select(*args)
        assert qsa.qsa_read_status(st) == (0, 0)
        outs.append((sc.cpu().numpy(), mask.cpu().numpy()))
    same = [o for o in outs[1:] if np.array_equal(o[0], outs[0][0])]
    assert same, "decode scores equal neither two-kernel path"
    assert np.array_equal(outs[0][1], same[0][1])
    want, codes = oracle_masks(orc, outs[0][0], nb, pos, tokens, BUDGET)
    assert codes == [0, 0] and np.array_equal(outs[0][1], want)
