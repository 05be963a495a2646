"""Seeded synthetic inputs for the QSA token indexer (pool -> score -> select).

This module only draws random numbers and lays them out.  It holds none of the
indexer's arithmetic (no pooling, norm, rotary embedding, scoring or
selection), so that the CPU oracle under ``oracle/`` and the CUDA path can both
be fed from it without sharing any of the method's code.

Every array is a plain numpy array:
  * bf16 data is carried as ``uint16`` bit patterns (the upper half of an
    IEEE float32), converted from float32 draws by torch's round-to-nearest
    cast;
  * positions and per-row offsets are ``int32`` / ``int64``;
  * selection-stress scores are ``float32``.

Geometry (fixed by the indexer on the pages: 4 query heads, head dim 128,
ratio 4, a fused q|k row of 640 columns, rotary dim 64).
"""
from __future__ import annotations

import numpy as np
import torch

N_HEADS = 4
HEAD_DIM = 128
RATIO = 4
FUSED_WIDTH = (N_HEADS + 1) * HEAD_DIM  # 640: four q heads, then the raw key
ROT_DIM = 64
BASE_SEED = 0x51A5EED


def seed_for(config_index: int, salt: int = 0) -> int:
    return BASE_SEED + config_index + 1000003 * salt


def rng_for(config_index: int, salt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed_for(config_index, salt)))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 bf16 bit patterns (torch's nearest-even cast)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 (exact widening)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def norm_weights(rng: np.random.Generator) -> tuple[np.ndarray, np.ndarray]:
    """q_norm_w, k_norm_w ~ N(0, 0.1) as bf16 (the weight enters as 1 + w)."""
    return normal_bf16(rng, (HEAD_DIM,), 0.1), normal_bf16(rng, (HEAD_DIM,), 0.1)


def fused_qk(rng: np.random.Generator, rows: int, token_scale: bool = False) -> np.ndarray:
    """[rows, 640] bf16: 4x128 query head columns then 128 raw key columns, N(0,1).

    With ``token_scale`` every row is multiplied by exp(U[ln 1/4, ln 4]), the
    per-token scale of the long-context decode workload."""
    x = rng.standard_normal((rows, FUSED_WIDTH), dtype=np.float32)
    if token_scale:
        s = np.exp(rng.uniform(np.log(0.25), np.log(4.0), size=(rows, 1))).astype(np.float32)
        x = x * s
    return to_bf16_bits(x)


def raw_keys(rng: np.random.Generator, tokens: int, token_scale: bool = False) -> np.ndarray:
    """[tokens, 128] bf16 raw indexer keys, N(0,1) (optionally per-token scaled)."""
    x = rng.standard_normal((tokens, HEAD_DIM), dtype=np.float32)
    if token_scale:
        s = np.exp(rng.uniform(np.log(0.25), np.log(4.0), size=(tokens, 1))).astype(np.float32)
        x = x * s
    return to_bf16_bits(x)


def stress_scores(rng: np.random.Generator, rows: int, cols: int, zero_frac: float = 0.7,
                  levels: int = 64, top: float = 4.0) -> np.ndarray:
    """Relu-sum-like f32 scores with massive ties.

    ``zero_frac`` of the entries are exactly zero, half of those written as
    -0.0; the rest are quantised to ``levels`` levels k/levels*top, k=1..levels.
    """
    u = rng.random((rows, cols))
    k = rng.integers(1, levels + 1, size=(rows, cols))
    vals = (k.astype(np.float32) / np.float32(levels)) * np.float32(top)
    zero = u < zero_frac
    neg = u < (zero_frac / 2.0)
    out = np.where(zero, np.float32(0.0), vals).astype(np.float32)
    out[neg] = np.float32(-0.0)
    return out


def set_blocks_to(row: np.ndarray, rng: np.random.Generator, value: np.float32, count: int,
                  limit: int) -> np.ndarray:
    """Overwrite ``count`` random entries of ``row[:limit]`` with ``value`` (tie injection)."""
    idx = rng.choice(limit, size=min(count, limit), replace=False)
    row[idx] = value
    return idx


def sprinkle_signed_zeros(row: np.ndarray, rng: np.random.Generator, frac: float, limit: int) -> None:
    """Set ~``frac`` of ``row[:limit]`` to +0.0 / -0.0 alternately."""
    n = int(frac * limit)
    idx = rng.choice(limit, size=n, replace=False)
    row[idx[0::2]] = np.float32(0.0)
    row[idx[1::2]] = np.float32(-0.0)


def long_context_lengths(rng: np.random.Generator, n_seq: int, lo: int = 131072,
                         hi: int = 262144) -> np.ndarray:
    """Sequence lengths drawn uniformly from [lo, hi] (inclusive)."""
    return rng.integers(lo, hi + 1, size=n_seq).astype(np.int64)


def torch_normal_bf16(torch, shape, seed: int, device, std: float = 1.0, token_scale: bool = False):
    """Large N(0,1) bf16 draws made on the device by torch's seeded generator
    (for benchmark-sized buffers; the oracle never sees these)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
    if token_scale:
        u = torch.rand((shape[0], 1), generator=g, device=device, dtype=torch.float32)
        x = x * torch.exp(np.log(0.25) + u * (np.log(4.0) - np.log(0.25)))
    return x.to(torch.bfloat16).view(torch.int16)


def paged_kv_pool(rng: np.random.Generator, pages: int, page_size: int, width: int) -> np.ndarray:
    """[pages * page_size, width] bf16 bit patterns, every 16-bit pattern
    possible (NaNs and infinities included: a gather copies bits)."""
    return rng.integers(0, 1 << 16, size=(pages * page_size, width), dtype=np.uint16)


def page_tables(rng: np.random.Generator, n_rows: int, table_len: int, pages: int) -> np.ndarray:
    """[n_rows, table_len] int32: each row's pages drawn without repeats from
    [0, pages), in shuffled order."""
    return np.stack([rng.permutation(pages)[:table_len] for _ in range(n_rows)]).astype(np.int32)
