"""Every entry point called from two host threads at once, on one device.

The launchers keep per-device set-up (kernel attributes, SM counts, the
fused decode step's co-residency) in caches that host threads share; two
threads that reach them together must both launch correctly.  Each thread runs
the whole chain on its own stream with its own inputs; the results must equal,
bit for bit, the same calls made afterwards from one thread (the kernels are
deterministic).
"""
import threading

import numpy as np
import pytest
import torch

import qsa_inputs as qi

pytestmark = pytest.mark.gpu

EPS, THETA, BUDGET = 1e-6, 10000.0, 2048


def chain(qsa, seed, stream):
    """The whole library on one stream; returns host copies of every output."""
    dev_ = torch.device("cuda")
    rng = qi.rng_for(11, salt=seed)
    T, R = 8192, 96
    nb = T // 4

    def d(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev_)

    with torch.cuda.stream(stream):
        c, s = qsa.qsa_rope_tables(T, THETA)
        cd, sd = d(c), d(s)
        qw, kw = (d(x) for x in qi.norm_weights(rng))
        raw = d(qi.raw_keys(rng, T))
        fq = d(qi.fused_qk(rng, R))
        pos = d(np.sort(rng.integers(0, T, size=R)).astype(np.int32))
        out = {}
        st = qsa.new_status()
        cache = torch.zeros((nb, 128), dtype=torch.int16, device=dev_)
        qsa.qsa_pool_blocks(raw, 128, 0, nb, kw, cd, sd, T, EPS, cache, stream=stream)
        for path in (qsa.QSA_SCORE_SIMT, qsa.QSA_SCORE_TCGEN05, qsa.QSA_SCORE_STREAM):
            sc = torch.full((R, nb), -7.0, dtype=torch.float32, device=dev_)
            qsa.qsa_score_rows_with(fq, 640, pos, None, R, T, qw, cd, sd, T, EPS, cache, None, sc,
                                    nb, st, path=path, workspace=qsa.new_workspace(R, dev_),
                                    stream=stream)
            out[f"score{path}"] = sc
        mask = torch.empty((R, T), dtype=torch.uint8, device=dev_)
        qsa.qsa_select_mask(out["score2"], nb, pos, R, T, BUDGET, mask, st, stream=stream)
        out["mask"] = mask
        cache2 = torch.zeros_like(cache)
        sc3 = torch.empty((R, nb), dtype=torch.float32, device=dev_)
        mask3 = torch.empty((R, T), dtype=torch.uint8, device=dev_)
        qsa.qsa_index_select(raw, 128, 0, nb, kw, fq, 640, pos, R, T, qw, cd, sd, T, EPS, BUDGET,
                             cache2, sc3, nb, mask3, st, workspace=qsa.new_workspace(R, dev_),
                             stream=stream)
        out.update(cache2=cache2, sc3=sc3, mask3=mask3)
        dpos = torch.tensor([T - 1, T - 2], dtype=torch.int32, device=dev_)
        sc4 = torch.empty((2, nb), dtype=torch.float32, device=dev_)
        mask4 = torch.empty((2, T), dtype=torch.uint8, device=dev_)
        ws = qsa.new_decode_workspace(2, T, dev_)
        qsa.qsa_decode_index_select(raw, 128, 0, 0, kw, fq[:2, :512].contiguous(), 512, dpos, 2,
                                    T, qw, cd, sd, T, EPS, BUDGET, cache2, sc4, nb, mask4, st, ws,
                                    stream=stream)
        out.update(sc4=sc4, mask4=mask4)
        sel_cols = BUDGET + 3
        sel = torch.full((R, sel_cols), -1, dtype=torch.int32, device=dev_)
        n_sel = torch.zeros(R, dtype=torch.int32, device=dev_)
        qsa.qsa_mask_tokens(mask, R, T, sel, sel_cols, n_sel, stream=stream)
        out.update(sel=sel, n_sel=n_sel)
        page, width = 16, 256                     # 2 KV heads x 128
        pages = T // page
        table = d(rng.permutation(pages).astype(np.int32))
        k_pool = d(qi.normal_bf16(rng, (pages * page, width)))
        v_pool = d(qi.normal_bf16(rng, (pages * page, width)))
        k_out = torch.zeros((R * sel_cols, width), dtype=torch.int16, device=dev_)
        v_out = torch.zeros_like(k_out)
        qsa.qsa_gather_kv(k_pool, v_pool, width, pages, table, pages, 0, page, sel, sel_cols,
                          n_sel, R, sel_cols, k_out, v_out, sel_cols, st, stream=stream)
        out.update(k_out=k_out, v_out=v_out)
        nq, nkv, hd = 8, 2, 128
        q = d(qi.normal_bf16(rng, (R, nq * hd)))
        att = torch.zeros((R, nq * hd), dtype=torch.int16, device=dev_)
        qsa.qsa_sparse_attn(q, nq * hd, nq, nkv, hd, k_pool, v_pool, pages, page, table, pages, 0,
                            sel, sel_cols, n_sel, R, sel_cols, hd ** -0.5, att, nq * hd, st,
                            stream=stream)
        out["att"] = att
        x = d(qi.normal_bf16(rng, (R, 2560)))
        w = d(qi.normal_bf16(rng, (640, 2560), 0.02))
        y = torch.zeros((R, 640), dtype=torch.int16, device=dev_)
        qsa.qsa_qk_proj(x, 2560, w, R, 2560, 640, y, 640, st, stream=stream)
        out["y"] = y
        out["status"] = st
    stream.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def test_two_host_threads_call_every_entry_point():
    import sparse_attention_token_qsa_gb300 as qsa

    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    results, errors = [None, None], []
    start = threading.Barrier(2)

    def worker(i):
        try:
            torch.cuda.set_device(0)
            start.wait()
            results[i] = chain(qsa, i, streams[i])
        except Exception as e:  # reported on the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(2):
        assert tuple(results[i]["status"]) == (0, 0)
        alone = chain(qsa, i, torch.cuda.Stream())
        for k in alone:
            assert np.array_equal(results[i][k], alone[k]), f"thread {i}: {k} differs"
