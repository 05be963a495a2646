"""CPU oracle for the QSA token indexer -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``qsa_oracle.c`` (plain C11, single-threaded, no
fast-math, no FMA contraction); this module compiles it with gcc on first use
and wraps it with numpy.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library never loads it and shares no code with it.

Every wrapper returns ``(result, status, err_row)`` where ``status`` follows
the C oracle's codes: 0 ok, 1 invalid value, 3 row out of range, 4 non-finite
score in a truncating row.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle_qsa.so")

OK, ERR_INVALID_VALUE, ERR_ROW_RANGE, ERR_NONFINITE = 0, 1, 3, 4
HEADS, HEAD_DIM, RATIO, ROT = 4, 128, 4, 64

CFLAGS = ["-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()
_lib = None


def compile_shared(src: str, out: str, extra: list[str] | None = None) -> str:
    """Compile an oracle C source into a shared library with the oracle's flags."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", *CFLAGS, *(extra or []), "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def build(force: bool = False) -> str:
    """Compile liboracle_qsa.so if it is missing or older than its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        compile_shared(_SRC, tmp)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    i32, i64, f32, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
    lib.orc_f32_to_bf16.argtypes = [f32]
    lib.orc_f32_to_bf16.restype = ctypes.c_uint16
    lib.orc_rope_table.argtypes = [i32, f64, P, P]
    lib.orc_rope_table.restype = ctypes.c_int
    lib.orc_pool_blocks.argtypes = [P, i64, i32, i32, P, P, P, f32, P]
    lib.orc_pool_blocks.restype = ctypes.c_int
    lib.orc_qprep.argtypes = [P, i32, P, P, P, f32, P]
    lib.orc_qprep.restype = ctypes.c_int
    lib.orc_score_row.argtypes = [P, P, i32, P]
    lib.orc_score_row.restype = None
    lib.orc_score_rows.argtypes = [P, i64, P, P, i32, i32, P, P, P, f32, P, P, P, i64, P]
    lib.orc_score_rows.restype = ctypes.c_int
    lib.orc_select_row.argtypes = [P, i32, i32, i32, P]
    lib.orc_select_row.restype = ctypes.c_int
    lib.orc_select_rows.argtypes = [P, i64, P, i32, i32, i32, P, P]
    lib.orc_select_rows.restype = ctypes.c_int
    lib.orc_mask_tokens.argtypes = [P, i32, P, i32]
    lib.orc_mask_tokens.restype = i32
    lib.orc_gather.argtypes = [P, P, i32, i32, i32, P, i32, P]
    lib.orc_gather.restype = i32
    lib.orc_sparse_attn.argtypes = [P, i32, i32, i32, P, P, P, i32, i32, P, i32, f64, P]
    lib.orc_sparse_attn.restype = ctypes.c_int
    lib.orc_proj.argtypes = [P, i64, P, i32, i32, i32, P, i64]
    lib.orc_proj.restype = ctypes.c_int
    return lib


def load_from(path: str) -> ctypes.CDLL:
    """Load an oracle build from ``path`` (the tests load planted-mistake builds this way)."""
    return _bind(ctypes.CDLL(path))


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_from(build())
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """numpy-facing wrappers over one oracle build (the real one by default)."""

    def __init__(self, handle: ctypes.CDLL | None = None):
        self.L = handle if handle is not None else lib()

    def f32_to_bf16(self, x: float) -> int:
        return int(self.L.orc_f32_to_bf16(float(x)))

    def rope_table(self, max_pos: int, theta: float = 10000.0):
        cos_t = np.zeros((max_pos, ROT), np.uint16)
        sin_t = np.zeros((max_pos, ROT), np.uint16)
        rc = self.L.orc_rope_table(int(max_pos), float(theta), _p(cos_t), _p(sin_t))
        if rc != OK:
            raise ValueError(f"oracle rope_table status {rc}")
        return cos_t, sin_t

    def pool_blocks(self, keys: np.ndarray, key_stride: int, first_block: int, n_blocks: int,
                    k_norm_w, cos_t, sin_t, eps: float, block_keys: np.ndarray | None = None,
                    total_blocks: int | None = None) -> np.ndarray:
        """keys: flat uint16 view starting at token 4*first_block (row stride key_stride)."""
        keys = np.ascontiguousarray(keys, np.uint16)
        if block_keys is None:
            total = total_blocks if total_blocks is not None else first_block + n_blocks
            block_keys = np.zeros((total, HEAD_DIM), np.uint16)
        assert block_keys.flags.c_contiguous and block_keys.dtype == np.uint16
        need = (4 * n_blocks - 1) * key_stride + HEAD_DIM if n_blocks > 0 else 0
        assert keys.size >= need, "keys buffer too short"
        rc = self.L.orc_pool_blocks(_p(keys), int(key_stride), int(first_block), int(n_blocks),
                                    _p(_c(k_norm_w, np.uint16)), _p(_c(cos_t, np.uint16)),
                                    _p(_c(sin_t, np.uint16)), float(eps), _p(block_keys))
        if rc != OK:
            raise ValueError(f"oracle pool status {rc}")
        return block_keys

    def qprep(self, q_row, pos: int, q_norm_w, cos_t, sin_t, eps: float) -> np.ndarray:
        out = np.zeros((HEADS, HEAD_DIM), np.uint16)
        rc = self.L.orc_qprep(_p(_c(q_row, np.uint16)), int(pos), _p(_c(q_norm_w, np.uint16)),
                              _p(_c(cos_t, np.uint16)), _p(_c(sin_t, np.uint16)), float(eps),
                              _p(out))
        if rc != OK:
            raise ValueError(f"oracle qprep status {rc}")
        return out

    def score_row(self, q_prepped, block_keys, n_blocks: int) -> np.ndarray:
        out = np.zeros(n_blocks, np.float32)
        self.L.orc_score_row(_p(_c(q_prepped, np.uint16)), _p(_c(block_keys, np.uint16)),
                             int(n_blocks), _p(out))
        return out

    def score_rows(self, q, q_stride: int, pos, n_rows: int, tokens: int, q_norm_w, cos_t, sin_t,
                   eps: float, block_keys, scores: np.ndarray, score_cols: int,
                   visible_len=None, key_base=None):
        """Fills ``scores`` (float32, row stride score_cols) in place; returns (status, err_row)."""
        assert scores.dtype == np.float32 and scores.flags.c_contiguous
        err = np.zeros(1, np.int32)
        rc = self.L.orc_score_rows(_p(_c(q, np.uint16)), int(q_stride), _p(_c(pos, np.int32)),
                                   _p(_c(visible_len, np.int32)), int(n_rows), int(tokens),
                                   _p(_c(q_norm_w, np.uint16)), _p(_c(cos_t, np.uint16)),
                                   _p(_c(sin_t, np.uint16)), float(eps),
                                   _p(_c(block_keys, np.uint16)), _p(_c(key_base, np.int64)),
                                   _p(scores), int(score_cols), _p(err))
        return rc, int(err[0])

    def select_row(self, scores_row, pos: int, tokens: int, budget: int):
        mask = np.full(tokens, 0xAB, np.uint8)
        rc = self.L.orc_select_row(_p(_c(scores_row, np.float32)), int(pos), int(tokens),
                                   int(budget), _p(mask))
        return mask, rc

    def select_rows(self, scores, score_cols: int, pos, n_rows: int, tokens: int, budget: int,
                    mask: np.ndarray | None = None):
        if mask is None:
            mask = np.full((n_rows, tokens), 0xAB, np.uint8)
        err = np.zeros(1, np.int32)
        rc = self.L.orc_select_rows(_p(_c(scores, np.float32)), int(score_cols),
                                    _p(_c(pos, np.int32)), int(n_rows), int(tokens), int(budget),
                                    _p(mask), _p(err))
        return mask, rc, int(err[0])

    def mask_tokens(self, mask_row, cap: int | None = None) -> np.ndarray:
        """The tokens whose mask byte is set, ascending (all of them if cap is None)."""
        m = _c(mask_row, np.uint8)
        cap = int(m.size) if cap is None else int(cap)
        out = np.zeros(max(cap, 1), np.int32)
        n = int(self.L.orc_mask_tokens(_p(m), int(m.size), _p(out), cap))
        return out[:min(n, cap)].copy(), n

    def gather(self, pool, table, page_size: int, width: int, sel) -> tuple[np.ndarray, int]:
        """Rows of a paged pool [pages * page_size, width] for the tokens in sel."""
        pool = _c(pool, np.uint16)
        table = _c(table, np.int32)
        sel = _c(sel, np.int32)
        out = np.zeros((max(len(sel), 1), width), np.uint16)
        rc = self.L.orc_gather(_p(pool), _p(table), int(table.size), int(page_size), int(width),
                               _p(sel), int(sel.size), _p(out))
        return out[:len(sel)], int(rc)

    def sparse_attn(self, q_row, nq: int, nkv: int, hd: int, k_pool, v_pool, table,
                    page_size: int, sel, scale: float) -> tuple[np.ndarray, int]:
        """One row's attention over its selected tokens: bf16 [nq * hd] and the
        return code.  Pools are [slots, nkv, hd] bf16 bit patterns."""
        q = _c(q_row, np.uint16)
        kp, vp = _c(k_pool, np.uint16), _c(v_pool, np.uint16)
        table = _c(table, np.int32)
        sel = _c(sel, np.int32)
        out = np.zeros(nq * hd, np.uint16)
        rc = self.L.orc_sparse_attn(_p(q), int(nq), int(nkv), int(hd), _p(kp), _p(vp), _p(table),
                                    int(table.size), int(page_size), _p(sel), int(sel.size),
                                    float(scale), _p(out))
        return out, int(rc)

    def proj(self, x, w) -> tuple[np.ndarray, int]:
        """y = x W^T for bf16 x [rows, hidden] and W [out, hidden]: bf16 [rows, out]."""
        x = _c(x, np.uint16)
        w = _c(w, np.uint16)
        rows, hidden = x.shape
        out_cols = w.shape[0]
        y = np.zeros((max(rows, 1), out_cols), np.uint16)
        rc = self.L.orc_proj(_p(x), int(hidden), _p(w), int(rows), int(hidden), int(out_cols),
                             _p(y), int(out_cols))
        return y[:rows], int(rc)

