"""qsa_qk_proj against the oracle.

The kernel accumulates the exact bf16 x bf16 products in f32 in the tensor
core's order; the oracle sums them exactly and rounds once.  The f32 sum is
within hidden * 2^-24 * sum_k |x_k w_k| of the exact one, and each side then
rounds to bf16 (at most one bf16 step apart when the two straddle a rounding
boundary; a step is up to 2^-7 of the value, at the bottom of a binade), so
every element is held to
    |got - want| <= 2^-7 |want| + hidden * 2^-23 * sum_k |x_k w_k|,
and nearly all elements must match bit for bit.
"""
import numpy as np
import pytest
import torch

import qsa_inputs as qi

pytestmark = pytest.mark.gpu

SENT = 0x7FAB


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


@pytest.fixture(scope="module")
def qsa():
    import sparse_attention_token_qsa_gb300 as m

    return m


def run_proj(qsa, x_np, w_np, x_pad=0, y_pad=0):
    rows, hidden = x_np.shape
    out_cols = w_np.shape[0]
    xs = hidden + x_pad
    xb = np.zeros((max(rows, 1), xs), np.uint16)
    xb[:rows, :hidden] = x_np
    ys = out_cols + y_pad
    y = torch.full((max(rows, 1), ys), SENT, dtype=torch.int16, device="cuda")
    st = qsa.new_status()
    qsa.qsa_qk_proj(dev(xb), xs, dev(w_np), rows, hidden, out_cols, y, ys, st)
    torch.cuda.synchronize()
    yb = y.cpu().numpy().view(np.uint16)
    assert np.all(yb[:, out_cols:] == SENT), "wrote past a row"
    return yb[:rows, :out_cols], qsa.qsa_read_status(st)


def check(orc, got, x_np, w_np, rows=None):
    idx = np.arange(x_np.shape[0]) if rows is None else np.asarray(rows)
    want, rc = orc.proj(x_np[idx], w_np)
    assert rc == 0
    g = qi.bf16_bits_to_f32(got[idx]).astype(np.float64)
    w = qi.bf16_bits_to_f32(want).astype(np.float64)
    xa = np.abs(qi.bf16_bits_to_f32(x_np[idx]).astype(np.float64))
    wa = np.abs(qi.bf16_bits_to_f32(w_np).astype(np.float64))
    bound = 2.0 ** -7 * np.abs(w) + x_np.shape[1] * 2.0 ** -23 * (xa @ wa.T) + 1e-30
    err = np.abs(g - w)
    assert np.all(err <= bound), f"max err {err.max():.3g}"
    assert np.mean(got[idx] == want) > 0.98


@pytest.mark.parametrize("rows,hidden,out_cols", [(1, 64, 16), (127, 200, 80), (128, 64, 96),
                                                  (129, 512, 160), (300, 2560, 640),
                                                  (37, 8, 32)])
def test_proj_matches_oracle(qsa, orc, rows, hidden, out_cols):
    """Ragged row tiles, K slices past the edge (zero fill), a partial column
    tile, padded row strides on both sides."""
    rng = qi.rng_for(8, salt=rows * 7 + hidden * 13 + out_cols)
    x = qi.normal_bf16(rng, (rows, hidden))
    w = qi.normal_bf16(rng, (out_cols, hidden), std=1.0 / np.sqrt(hidden))
    got, st = run_proj(qsa, x, w, x_pad=8, y_pad=16)
    assert st == (0, 0)
    check(orc, got, x, w)


@pytest.mark.parametrize("n_rows", [2048, 4096, 4000])
def test_proj_slabs_sampled_rows(qsa, orc, n_rows):
    """The pages' slab (2048 rows, 80-column tiles) and longer launches that take
    160-column tiles (4096 rows; 4000: a ragged last row tile); hidden 2560, 640
    outputs; rows from every row tile's edges and middle checked."""
    rng = qi.rng_for(8, salt=n_rows)
    x = qi.normal_bf16(rng, (n_rows, 2560))
    w = qi.normal_bf16(rng, (640, 2560), std=0.02)
    got, st = run_proj(qsa, x, w)
    assert st == (0, 0)
    rows = sorted({min(r, n_rows - 1) for t in range((n_rows + 127) // 128)
                   for r in (128 * t, 128 * t + 61, 128 * t + 127)})
    check(orc, got, x, w, rows=rows)


def test_proj_exact_cases(qsa):
    """Unit-vector weights copy columns of x bit for bit; a zero weight gives
    zeros; an empty launch writes nothing."""
    rng = qi.rng_for(8, salt=1)
    x = qi.normal_bf16(rng, (200, 128))
    perm = rng.permutation(128)[:48]
    w = np.zeros((48, 128), np.float32)
    w[np.arange(48), perm] = 1.0
    got, st = run_proj(qsa, x, qi.to_bf16_bits(w))
    assert st == (0, 0) and np.array_equal(got, x[:, perm])
    got, _ = run_proj(qsa, x, np.zeros((16, 128), np.uint16))
    assert not got.any()
    y = torch.full((4, 16), SENT, dtype=torch.int16, device="cuda")
    st = qsa.new_status()
    qsa.qsa_qk_proj(dev(x), 128, dev(np.zeros((16, 128), np.uint16)), 0, 128, 16, y, 16, st)
    torch.cuda.synchronize()
    assert np.all(y.cpu().numpy().view(np.uint16) == SENT)
