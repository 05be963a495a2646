"""GB300-native QSA token indexer: pool -> score -> select, behind libqsa.so.

This package is a thin ctypes binding over the C ABI declared in
``include/qsa.h``.  Every function has the C entry point's name and argument
order; device buffers are passed as CUDA torch tensors (their data pointers),
``stream`` is a torch CUDA stream (default: the current stream).  The binding
only marshals arguments: all work runs in the library's CUDA kernels.  There is
no CPU fallback: importing the package fails loudly when libqsa.so is missing
(build it with ``python sparse_attention_token_qsa_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqsa.so")

QSA_OK = 0
QSA_ERR_INVALID_VALUE = 1
QSA_ERR_LAUNCH = 2
QSA_ERR_ROW_RANGE = 3
QSA_ERR_NONFINITE = 4
QSA_ERR_TIMEOUT = 5
QSA_ERR_TOKEN_RANGE = 6

QSA_SCORE_AUTO = 0
QSA_SCORE_SIMT = 1
QSA_SCORE_TCGEN05 = 2
QSA_SCORE_STREAM = 3

HEADS, HEAD_DIM, RATIO, ROT_DIM, FUSED_WIDTH = 4, 128, 4, 64, 640

EXPORTED = ("qsa_version", "qsa_status_string", "qsa_rope_tables", "qsa_pool_blocks",
            "qsa_score_rows", "qsa_score_rows_with", "qsa_score_workspace_bytes",
            "qsa_score_rows_noalloc", "qsa_select_mask", "qsa_index_select",
            "qsa_decode_workspace_bytes", "qsa_decode_index_select", "qsa_mask_tokens",
            "qsa_gather_kv", "qsa_sparse_attn", "qsa_qk_proj", "qsa_reset_status",
            "qsa_read_status", "qsa_set_wait_limit_cycles", "qsa_wait_limit_cycles")


class QsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: status {code} ({status_string(code)})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libqsa.so is not built ({LIB_PATH}); run "
                          "`python sparse_attention_token_qsa_gb300/build.py` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, f64 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_double)
    sig = {
        "qsa_version": ([], i32),
        "qsa_status_string": ([i32], ctypes.c_char_p),
        "qsa_rope_tables": ([i32, f64, P, P], i32),
        "qsa_pool_blocks": ([P, i64, i32, i32, P, P, P, i32, f32, P, P], i32),
        "qsa_score_rows": ([P, i64, P, P, i32, i32, P, P, P, i32, f32, P, P, P, i64, P, P, i64, P],
                           i32),
        "qsa_score_rows_with": ([P, i64, P, P, i32, i32, P, P, P, i32, f32, P, P, P, i64, P, i32, P,
                                 i64, P], i32),
        "qsa_score_workspace_bytes": ([i32], i64),
        "qsa_score_rows_noalloc": ([P, i64, P, P, i32, i32, P, P, P, i32, f32, P, P, i64, P, P], i32),
        "qsa_select_mask": ([P, i64, P, i32, i32, i32, P, P, P], i32),
        "qsa_index_select": ([P, i64, i32, i32, P, P, i64, P, i32, i32, P, P, P, i32, f32, i32, P, P,
                              i64, P, P, P, i64, P], i32),
        "qsa_decode_workspace_bytes": ([i32, i32], i64),
        "qsa_decode_index_select": ([P, i64, i32, i32, P, P, i64, P, i32, i32, P, P, P, i32, f32, i32,
                                     P, P, i64, P, P, P, i64, P], i32),
        "qsa_mask_tokens": ([P, i32, i32, P, i64, P, P], i32),
        "qsa_gather_kv": ([P, P, i32, i32, P, i32, i64, i32, P, i64, P, i32, i32, P, P, i64, P, P],
                          i32),
        "qsa_sparse_attn": ([P, i64, i32, i32, i32, P, P, i32, i32, P, i32, i64, P, i64, P, i32,
                             i32, f32, P, i64, P, P], i32),
        "qsa_qk_proj": ([P, i64, P, i32, i32, i32, P, i64, P, P], i32),
        "qsa_reset_status": ([P, P], i32),
        "qsa_read_status": ([P, P, P, P], i32),
        "qsa_set_wait_limit_cycles": ([i64], i32),
        "qsa_wait_limit_cycles": ([], i64),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    return _lib


def status_string(code: int) -> str:
    return _lib.qsa_status_string(int(code)).decode()


def _dev(t: torch.Tensor | None, name: str):
    """The device-addressable pointer of a CUDA tensor, or of a pinned host tensor
    (page-locked host memory is mapped into the unified address space, so the
    kernels read and write it directly over the CPU-GPU link).  Anything else is
    refused: every computation runs in the library's kernels."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory: libqsa has no "
                         "CPU path")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, where: str) -> None:
    if rc != QSA_OK:
        raise QsaError(rc, where)


def qsa_version() -> int:
    return int(_lib.qsa_version())


def qsa_set_wait_limit_cycles(cycles: int) -> None:
    """The limit, in SM clock cycles, of the waits a caller may shorten (the
    streaming scorers' key-copy, operand and accumulator waits, the fused decode
    step's waits and barrier)."""
    _check(_lib.qsa_set_wait_limit_cycles(int(cycles)), "qsa_set_wait_limit_cycles")


def qsa_wait_limit_cycles() -> int:
    return int(_lib.qsa_wait_limit_cycles())


def qsa_rope_tables(max_pos: int, theta: float = 10000.0) -> tuple[np.ndarray, np.ndarray]:
    """Host cos/sin tables [max_pos, 64] as uint16 bf16 bit patterns."""
    cos_t = np.zeros((max_pos, ROT_DIM), np.uint16)
    sin_t = np.zeros((max_pos, ROT_DIM), np.uint16)
    _check(_lib.qsa_rope_tables(int(max_pos), float(theta),
                                cos_t.ctypes.data_as(ctypes.c_void_p),
                                sin_t.ctypes.data_as(ctypes.c_void_p)), "qsa_rope_tables")
    return cos_t, sin_t


def qsa_pool_blocks(keys, key_stride, first_block, n_blocks, k_norm_w, cos_t, sin_t, table_rows,
                    eps, block_keys, stream=None) -> None:
    _check(_lib.qsa_pool_blocks(_dev(keys, "keys"), int(key_stride), int(first_block),
                                int(n_blocks), _dev(k_norm_w, "k_norm_w"), _dev(cos_t, "cos_t"),
                                _dev(sin_t, "sin_t"), int(table_rows), float(eps),
                                _dev(block_keys, "block_keys"), _stream(stream)),
           "qsa_pool_blocks")


def _ws(workspace):
    if workspace is None:
        return None, 0
    return _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()


def qsa_score_workspace_bytes(n_rows: int) -> int:
    return int(_lib.qsa_score_workspace_bytes(int(n_rows)))


def new_workspace(n_rows: int, device="cuda") -> torch.Tensor:
    """A device workspace large enough for the tensor-core scorer."""
    return torch.empty(max(1, qsa_score_workspace_bytes(n_rows)), dtype=torch.uint8, device=device)


def qsa_score_rows_with(q, q_stride, pos, visible_len, n_rows, tokens, q_norm_w, cos_t, sin_t,
                        table_rows, eps, block_keys, key_base, scores, score_cols, dev_status,
                        path=QSA_SCORE_AUTO, workspace=None, stream=None) -> None:
    ws, wsb = _ws(workspace)
    _check(_lib.qsa_score_rows_with(_dev(q, "q"), int(q_stride), _dev(pos, "pos"),
                                    _dev(visible_len, "visible_len"), int(n_rows), int(tokens),
                                    _dev(q_norm_w, "q_norm_w"), _dev(cos_t, "cos_t"),
                                    _dev(sin_t, "sin_t"), int(table_rows), float(eps),
                                    _dev(block_keys, "block_keys"), _dev(key_base, "key_base"),
                                    _dev(scores, "scores"), int(score_cols),
                                    _dev(dev_status, "dev_status"), int(path), ws, int(wsb),
                                    _stream(stream)),
           "qsa_score_rows_with")


def qsa_score_rows(q, q_stride, pos, visible_len, n_rows, tokens, q_norm_w, cos_t, sin_t,
                   table_rows, eps, block_keys, key_base, scores, score_cols, dev_status,
                   workspace=None, stream=None) -> None:
    ws, wsb = _ws(workspace)
    _check(_lib.qsa_score_rows(_dev(q, "q"), int(q_stride), _dev(pos, "pos"),
                               _dev(visible_len, "visible_len"), int(n_rows), int(tokens),
                               _dev(q_norm_w, "q_norm_w"), _dev(cos_t, "cos_t"),
                               _dev(sin_t, "sin_t"), int(table_rows), float(eps),
                               _dev(block_keys, "block_keys"), _dev(key_base, "key_base"),
                               _dev(scores, "scores"), int(score_cols),
                               _dev(dev_status, "dev_status"), ws, int(wsb), _stream(stream)),
           "qsa_score_rows")


QSA_NOALLOC_MAX_ROWS = 8192


def qsa_score_rows_noalloc(q, q_stride, pos, visible_len, n_rows, tokens, q_norm_w, cos_t, sin_t,
                           table_rows, eps, block_keys, scores, score_cols, dev_status,
                           stream=None) -> None:
    """Tensor-core scoring with the library's built-in workspace (no allocation
    by anyone); at most QSA_NOALLOC_MAX_ROWS rows, calls must not overlap."""
    _check(_lib.qsa_score_rows_noalloc(_dev(q, "q"), int(q_stride), _dev(pos, "pos"),
                                       _dev(visible_len, "visible_len"), int(n_rows), int(tokens),
                                       _dev(q_norm_w, "q_norm_w"), _dev(cos_t, "cos_t"),
                                       _dev(sin_t, "sin_t"), int(table_rows), float(eps),
                                       _dev(block_keys, "block_keys"), _dev(scores, "scores"),
                                       int(score_cols), _dev(dev_status, "dev_status"),
                                       _stream(stream)),
           "qsa_score_rows_noalloc")


def qsa_select_mask(scores, score_cols, pos, n_rows, tokens, budget, mask, dev_status,
                    stream=None) -> None:
    _check(_lib.qsa_select_mask(_dev(scores, "scores"), int(score_cols), _dev(pos, "pos"),
                                int(n_rows), int(tokens), int(budget), _dev(mask, "mask"),
                                _dev(dev_status, "dev_status"), _stream(stream)),
           "qsa_select_mask")


def qsa_index_select(keys, key_stride, pool_first_block, pool_n_blocks, k_norm_w, q, q_stride, pos,
                     n_rows, tokens, q_norm_w, cos_t, sin_t, table_rows, eps, budget, block_keys,
                     scores, score_cols, mask, dev_status, workspace=None, stream=None) -> None:
    ws, wsb = _ws(workspace)
    _check(_lib.qsa_index_select(_dev(keys, "keys"), int(key_stride), int(pool_first_block),
                                 int(pool_n_blocks), _dev(k_norm_w, "k_norm_w"), _dev(q, "q"),
                                 int(q_stride), _dev(pos, "pos"), int(n_rows), int(tokens),
                                 _dev(q_norm_w, "q_norm_w"), _dev(cos_t, "cos_t"),
                                 _dev(sin_t, "sin_t"), int(table_rows), float(eps), int(budget),
                                 _dev(block_keys, "block_keys"), _dev(scores, "scores"),
                                 int(score_cols), _dev(mask, "mask"),
                                 _dev(dev_status, "dev_status"), ws, int(wsb), _stream(stream)),
           "qsa_index_select")


def qsa_decode_workspace_bytes(n_rows: int, tokens: int) -> int:
    return int(_lib.qsa_decode_workspace_bytes(int(n_rows), int(tokens)))


def new_decode_workspace(n_rows: int, tokens: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace for qsa_decode_index_select (each completed call
    leaves it zero again)."""
    n = max(16, qsa_decode_workspace_bytes(n_rows, tokens))
    return torch.zeros(n, dtype=torch.uint8, device=device)


def qsa_decode_index_select(keys, key_stride, pool_first_block, pool_n_blocks, k_norm_w, q, q_stride,
                            pos, n_rows, tokens, q_norm_w, cos_t, sin_t, table_rows, eps, budget,
                            block_keys, scores, score_cols, mask, dev_status, decode_ws,
                            stream=None) -> None:
    ws, wsb = _ws(decode_ws)
    _check(_lib.qsa_decode_index_select(_dev(keys, "keys"), int(key_stride), int(pool_first_block),
                                        int(pool_n_blocks), _dev(k_norm_w, "k_norm_w"),
                                        _dev(q, "q"), int(q_stride), _dev(pos, "pos"), int(n_rows),
                                        int(tokens), _dev(q_norm_w, "q_norm_w"),
                                        _dev(cos_t, "cos_t"), _dev(sin_t, "sin_t"),
                                        int(table_rows), float(eps), int(budget),
                                        _dev(block_keys, "block_keys"), _dev(scores, "scores"),
                                        int(score_cols), _dev(mask, "mask"),
                                        _dev(dev_status, "dev_status"), ws, int(wsb),
                                        _stream(stream)),
           "qsa_decode_index_select")


def qsa_mask_tokens(mask, n_rows, tokens, sel, sel_cols, n_sel, stream=None) -> None:
    _check(_lib.qsa_mask_tokens(_dev(mask, "mask"), int(n_rows), int(tokens), _dev(sel, "sel"),
                                int(sel_cols), _dev(n_sel, "n_sel"), _stream(stream)),
           "qsa_mask_tokens")


def qsa_gather_kv(k_pool, v_pool, width, pool_pages, table, table_len, table_cols, page_size, sel,
                  sel_cols, n_sel, n_rows, max_sel, k_out, v_out, out_rows, dev_status,
                  stream=None) -> None:
    _check(_lib.qsa_gather_kv(_dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), int(width),
                              int(pool_pages), _dev(table, "table"), int(table_len),
                              int(table_cols), int(page_size), _dev(sel, "sel"), int(sel_cols),
                              _dev(n_sel, "n_sel"), int(n_rows), int(max_sel),
                              _dev(k_out, "k_out"), _dev(v_out, "v_out"), int(out_rows),
                              _dev(dev_status, "dev_status"), _stream(stream)),
           "qsa_gather_kv")


def qsa_sparse_attn(q, q_stride, nq, nkv, head_dim, k_pool, v_pool, pool_pages, page_size, table,
                    table_len, table_cols, sel, sel_cols, n_sel, n_rows, max_sel, scale, out,
                    out_stride, dev_status, stream=None) -> None:
    _check(_lib.qsa_sparse_attn(_dev(q, "q"), int(q_stride), int(nq), int(nkv), int(head_dim),
                                _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), int(pool_pages),
                                int(page_size), _dev(table, "table"), int(table_len),
                                int(table_cols), _dev(sel, "sel"), int(sel_cols),
                                _dev(n_sel, "n_sel"), int(n_rows), int(max_sel), float(scale),
                                _dev(out, "out"), int(out_stride), _dev(dev_status, "dev_status"),
                                _stream(stream)),
           "qsa_sparse_attn")


def qsa_qk_proj(x, x_stride, w, n_rows, hidden, out_cols, y, y_stride, dev_status,
                stream=None) -> None:
    _check(_lib.qsa_qk_proj(_dev(x, "x"), int(x_stride), _dev(w, "w"), int(n_rows), int(hidden),
                            int(out_cols), _dev(y, "y"), int(y_stride),
                            _dev(dev_status, "dev_status"), _stream(stream)),
           "qsa_qk_proj")


def qsa_reset_status(dev_status, stream=None) -> None:
    _check(_lib.qsa_reset_status(_dev(dev_status, "dev_status"), _stream(stream)),
           "qsa_reset_status")


def qsa_read_status(dev_status, stream=None) -> tuple[int, int]:
    code, row = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(_lib.qsa_read_status(_dev(dev_status, "dev_status"), _stream(stream),
                                ctypes.byref(code), ctypes.byref(row)), "qsa_read_status")
    return int(code.value), int(row.value)


def new_status(device="cuda") -> torch.Tensor:
    """A zeroed device status word (int32[2])."""
    return torch.zeros(2, dtype=torch.int32, device=device)
