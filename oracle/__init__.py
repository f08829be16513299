"""MSA CPU oracle -- TEST INFRASTRUCTURE ONLY.

Python access to the plain C implementation in ``msa_oracle.c`` (compiled with gcc into
``_build/libmsa_oracle.so`` beside this file). Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this package; the CUDA library and its Python
binding never do.

Every function takes and returns numpy arrays. bf16 tensors travel as ``np.uint16`` bit
patterns. Attention results come back in fp64 (``o``) together with the bf16 rounding of
that fp64 value (``o_bf16``) -- the output dtype of the layer.

The method, its passages and the readings held fixed are documented at the top of
``msa_oracle.c``.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py`` against
brute force, closed forms, a textbook/library routine or an invariant; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmsa_oracle.so")
_lock = threading.Lock()
_lib = None

BLOCK = 128


def gcc_command(src: str, out: str) -> list:
    """The gcc line that builds a shared library from an oracle source file (portable C, no
    target-specific flags, no contraction of multiply-adds)."""
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
            src, "-o", out, "-lm", "-lpthread"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(gcc_command(_SRC, tmp), check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.oracle_round_bf16_array.restype = None
            lib.oracle_round_bf16_array.argtypes = [P, i64, P]
            lib.oracle_block_scores.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, i64, P, i32]
            lib.oracle_topk.argtypes = [P, P, i64, i32, i32, i32, P, P]
            lib.oracle_build_sparse_page_table.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P]
            lib.oracle_sparse_decode.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                                 i32, P, i64, P, P, i32]
            lib.oracle_paged_decode_flat.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i32, P,
                                                     i64, P, P, i32]
            lib.oracle_sparse_prefill.argtypes = [P, P, P, P, i64, i64, i32, i32, i32, i32, P,
                                                  i64, P, P, i32]
            lib.oracle_prefill_block_partial.argtypes = [P, P, P, i64, i64, i32, i32, i32, i64,
                                                         i32, i32, P, P]
            lib.oracle_lse_merge.argtypes = [P, P, i32, i32, P, P]
            lib.oracle_prefill_buckets.argtypes = [P, i64, i32, i32, i32, P, P]
            for name in ("oracle_block_scores", "oracle_topk", "oracle_build_sparse_page_table",
                         "oracle_sparse_decode", "oracle_paged_decode_flat",
                         "oracle_sparse_prefill", "oracle_prefill_block_partial",
                         "oracle_lse_merge", "oracle_prefill_buckets"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, name: str):
    if rc != 0:
        raise ValueError(f"{name}: invalid arguments (rc={rc})")


# ------------------------------------------------------------------------------ bf16

def bf16_to_f32(x: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    return (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_bf16(x) -> np.ndarray:
    """Round fp64 values to bf16 bit patterns, ties to even (one rounding)."""
    x = _c(np.asarray(x, dtype=np.float64), np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_round_bf16_array(_p(x), x.size, _p(out))
    return out


# ------------------------------------------------------------------------------ stage 1

def block_scores(q_idx, k_idx_pages, page_table, seq_lens, N: int, rows=None, nthreads=None):
    """Block scores [nrows, Hkv, max_blocks] (fp32); -inf where a block has no valid token.

    q_idx [B*N, Hkv, Di] u16, k_idx_pages [P, 128, Hkv, Di] u16, page_table [B, max_blocks]
    i32, seq_lens [B] i32. Row r = b*N + i is the query at position seq_lens[b] - N + i.
    """
    q_idx = _c(q_idx, np.uint16)
    k_idx_pages = _c(k_idx_pages, np.uint16)
    page_table = _c(page_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    B, max_blocks = page_table.shape
    Hkv, Di = q_idx.shape[1], q_idx.shape[2]
    assert q_idx.shape[0] == B * N and k_idx_pages.shape[1:] == (BLOCK, Hkv, Di)
    if rows is None:
        rows_a, nrows = None, B * N
    else:
        rows_a = _c(rows, np.int64)
        nrows = rows_a.size
    out = np.empty((nrows, Hkv, max_blocks), dtype=np.float32)
    rc = _load().oracle_block_scores(_p(q_idx), _p(k_idx_pages), _p(page_table), _p(seq_lens),
                                     B, N, Hkv, Di, max_blocks, _p(rows_a), nrows, _p(out),
                                     nthreads or default_threads())
    _check(rc, "block_scores")
    return out


def topk(scores, q_pos, k: int):
    """Top-k block selection per (row, group). Returns (block_ids i32, sel_scores f32)."""
    scores = _c(scores, np.float32)
    q_pos = _c(q_pos, np.int64)
    nrows, Hkv, max_blocks = scores.shape
    assert q_pos.shape == (nrows,)
    ids = np.empty((nrows, Hkv, k), dtype=np.int32)
    sel = np.empty((nrows, Hkv, k), dtype=np.float32)
    rc = _load().oracle_topk(_p(scores), _p(q_pos), nrows, Hkv, max_blocks, k, _p(ids), _p(sel))
    _check(rc, "topk")
    return ids, sel


def query_positions(seq_lens, N: int) -> np.ndarray:
    """Positions of the N query rows of each request: seq_lens[b] - N + i."""
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    return (seq_lens[:, None] - N + np.arange(N, dtype=np.int64)[None, :]).reshape(-1)


# ------------------------------------------------------------------------------ page table

def build_sparse_page_table(block_ids, page_table, seq_lens, N: int):
    block_ids = _c(block_ids, np.int32)
    page_table = _c(page_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    R, Hkv, k = block_ids.shape
    B, max_blocks = page_table.shape
    assert R == B * N
    fpt = np.empty((R * Hkv, k), dtype=np.int32)
    lens = np.empty((R * Hkv,), dtype=np.int32)
    rc = _load().oracle_build_sparse_page_table(_p(block_ids), _p(page_table), _p(seq_lens), B, N,
                                                Hkv, k, max_blocks, _p(fpt), _p(lens))
    _check(rc, "build_sparse_page_table")
    return fpt, lens


# ------------------------------------------------------------------------------ attention

def _finish(o, lse):
    return {"o": o, "lse": lse, "o_bf16": round_bf16(o)}


def sparse_decode(q, k_cache, v_cache, page_table, seq_lens, block_ids, N: int, units=None,
                  nthreads=None):
    """Plain-definition sparse decode attention. q [B*N, Hq, D]; caches [P,128,Hkv,D]."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    page_table = _c(page_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    block_ids = _c(block_ids, np.int32)
    R, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    B, max_blocks = page_table.shape
    k = block_ids.shape[2]
    units_a = None if units is None else _c(units, np.int64)
    n = R * Hq if units_a is None else units_a.size
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = _load().oracle_sparse_decode(_p(q), _p(k_cache), _p(v_cache), _p(page_table),
                                      _p(seq_lens), _p(block_ids), B, N, Hq, Hkv, D, k, max_blocks,
                                      _p(units_a), n, _p(o), _p(lse), nthreads or default_threads())
    _check(rc, "sparse_decode")
    return _finish(o, lse)


def paged_decode_flat(q, k_cache, v_cache, flat_page_table, flat_kv_lens, units=None,
                      nthreads=None):
    """Decode attention read through the strided per-head view and a flat page table."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    fpt = _c(flat_page_table, np.int32)
    lens = _c(flat_kv_lens, np.int32)
    R, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    k = fpt.shape[1]
    units_a = None if units is None else _c(units, np.int64)
    n = R * Hq if units_a is None else units_a.size
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = _load().oracle_paged_decode_flat(_p(q), _p(k_cache), _p(v_cache), _p(fpt), _p(lens), R, Hq,
                                          Hkv, D, k, _p(units_a), n, _p(o), _p(lse),
                                          nthreads or default_threads())
    _check(rc, "paged_decode_flat")
    return _finish(o, lse)


def sparse_prefill(q, k, v, block_ids, units=None, nthreads=None):
    """Plain-definition sparse prefill attention. q [T,Hq,D]; k, v [S_kv,Hkv,D]."""
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    block_ids = _c(block_ids, np.int32)
    T, Hq, D = q.shape
    S, Hkv, _ = k.shape
    topk_ = block_ids.shape[2]
    units_a = None if units is None else _c(units, np.int64)
    n = T * Hq if units_a is None else units_a.size
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = _load().oracle_sparse_prefill(_p(q), _p(k), _p(v), _p(block_ids), T, S, Hq, Hkv, D, topk_,
                                       _p(units_a), n, _p(o), _p(lse), nthreads or default_threads())
    _check(rc, "sparse_prefill")
    return _finish(o, lse)


def prefill_block_partial(q, k, v, t: int, h: int, block: int):
    """One block-major partial (o_j [D] fp64, lse_j) for query t, head h, block j."""
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    T, Hq, D = q.shape
    S, Hkv, _ = k.shape
    o = np.empty((D,), dtype=np.float64)
    lse = np.empty((1,), dtype=np.float64)
    rc = _load().oracle_prefill_block_partial(_p(q), _p(k), _p(v), T, S, Hq, Hkv, D, t, h, block,
                                              _p(o), _p(lse))
    _check(rc, "prefill_block_partial")
    return o, float(lse[0])


def lse_merge(o_parts, lse_parts):
    """Merge partials o_parts [n, D] (float32), lse_parts [n] -> (o [D] fp64, lse)."""
    o_parts = _c(o_parts, np.float32)
    lse_parts = _c(lse_parts, np.float32)
    n, D = o_parts.shape
    o = np.empty((D,), dtype=np.float64)
    lse = np.empty((1,), dtype=np.float64)
    rc = _load().oracle_lse_merge(_p(o_parts), _p(lse_parts), n, D, _p(o), _p(lse))
    _check(rc, "lse_merge")
    return o, float(lse[0])


def prefill_buckets(block_ids, nblk: int):
    """Invert block_ids [T, Hkv, k] into per-(group, block) lists of t*k + slot."""
    block_ids = _c(block_ids, np.int32)
    T, Hkv, k = block_ids.shape
    offsets = np.empty((Hkv, nblk + 1), dtype=np.int32)
    n_valid = int(np.count_nonzero((block_ids >= 0) & (block_ids < nblk)))
    entries = np.empty((max(n_valid, 1),), dtype=np.int32)
    rc = _load().oracle_prefill_buckets(_p(block_ids), T, Hkv, k, nblk, _p(offsets), _p(entries))
    _check(rc, "prefill_buckets")
    return offsets, entries[:n_valid]
