"""GB300-native MiniMax Sparse Attention (MSA) layer: Python binding of libmsa_gb300.so.

Each function marshals torch CUDA tensors into the C ABI of ``include/msa.h`` (pointers,
sizes, the current CUDA stream) and calls it; every step of the computation runs in the
library's CUDA kernels. There is no CPU or PyTorch fallback: a missing library raises.

Stage 1  ``index_score_topk``        block scores + top-k selection per (query row, KV group)
         ``build_sparse_page_table`` flattened per-(row, group) page tables over the
                                     strided per-head KV view
Stage 2  ``paged_sparse_decode``     paged decode attention over the selected pages
         ``sparse_prefill``          KV-block-major prefill attention + LSE merge
Pieces   ``prefill_bucket``, ``lse_merge``, ``device_error``
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import MSAError, library_path, load

__all__ = ["index_score_topk", "index_score_topk_noalloc", "build_sparse_page_table", "paged_sparse_decode", "sparse_prefill",
           "prefill_bucket", "lse_merge", "device_error", "Workspace", "MSAError", "load",
           "library_path", "BLOCK"]

BLOCK = 128


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, ndim: int | None = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got {tuple(t.shape)}")
    return t


class Workspace:
    """Caller-owned scratch memory for the C ABI, grown on demand and reused.

    One Workspace serves every call made on one stream; calls that may overlap on the
    GPU need separate Workspace objects.
    """

    def __init__(self):
        self._bufs: dict = {}

    def get(self, key: str, nbytes: int, device, zero: bool = False) -> torch.Tensor:
        nbytes = max(int(nbytes), 256)
        cur = self._bufs.get(key)
        if cur is None or cur.numel() < nbytes or cur.device != torch.device(device):
            alloc = torch.zeros if zero else torch.empty
            cur = alloc(nbytes, dtype=torch.uint8, device=device)
            self._bufs[key] = cur
        return cur


_default_ws: dict = {}


def _ws(ws: Workspace | None, device) -> Workspace:
    if ws is not None:
        return ws
    key = (torch.device(device), torch.cuda.current_stream(device).cuda_stream)
    if key not in _default_ws:
        _default_ws[key] = Workspace()
    return _default_ws[key]


# ------------------------------------------------------------------------------ stage 1

def index_score_topk(q_idx, k_idx_pages, page_table, seq_lens, N: int, topk: int,
                     with_scores: bool = True, workspace: Workspace | None = None,
                     out=None):
    """Block scores and top-k selection (``msa_index_score_topk``).

    q_idx [B*N, Hkv, Di] bf16, k_idx_pages [P, 128, Hkv, Di] bf16, page_table [B, max_blocks]
    int32, seq_lens [B] int32. Returns (block_ids [B*N, Hkv, topk] int32,
    scores [B*N, Hkv, topk] fp32 or None).
    """
    _need(q_idx, "q_idx", torch.bfloat16, 3)
    _need(k_idx_pages, "k_idx_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, max_blocks = page_table.shape
    R, Hkv, Di = q_idx.shape
    if R != B * N or k_idx_pages.shape[1:] != (BLOCK, Hkv, Di) or seq_lens.numel() != B:
        raise ValueError("index_score_topk: inconsistent shapes")
    dev = q_idx.device
    if out is None:
        ids = torch.empty((R, Hkv, topk), dtype=torch.int32, device=dev)
        sc = torch.empty((R, Hkv, topk), dtype=torch.float32, device=dev) if with_scores else None
    else:
        ids, sc = out
    lib = load()
    nbytes = lib.msa_index_score_topk_workspace_size(B, N, Hkv, max_blocks)
    buf = _ws(workspace, dev).get("score", nbytes, dev)
    rc = lib.msa_index_score_topk(_ptr(q_idx), _ptr(k_idx_pages), _ptr(page_table), _ptr(seq_lens),
                                  B, N, Hkv, Di, max_blocks, k_idx_pages.shape[0], topk, _ptr(ids),
                                  _ptr(sc), _ptr(buf), buf.numel(), _stream(dev))
    _lib.check("msa_index_score_topk", rc)
    return ids, sc


def index_score_topk_page_table(q_idx, k_idx_pages, page_table, seq_lens, N: int, topk: int,
                                with_scores: bool = True, workspace: Workspace | None = None):
    """Selection and its sparse page table in one call (``msa_index_score_topk_page_table``).

    Arguments as ``index_score_topk``. Returns (block_ids [B*N, Hkv, topk] int32, scores or None,
    flat_page_table [B*N*Hkv, topk] int32, flat_kv_lens [B*N*Hkv] int32).
    """
    _need(q_idx, "q_idx", torch.bfloat16, 3)
    _need(k_idx_pages, "k_idx_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, max_blocks = page_table.shape
    R, Hkv, Di = q_idx.shape
    if R != B * N or k_idx_pages.shape[1:] != (BLOCK, Hkv, Di) or seq_lens.numel() != B:
        raise ValueError("index_score_topk_page_table: inconsistent shapes")
    dev = q_idx.device
    ids = torch.empty((R, Hkv, topk), dtype=torch.int32, device=dev)
    sc = torch.empty((R, Hkv, topk), dtype=torch.float32, device=dev) if with_scores else None
    fpt = torch.empty((R * Hkv, topk), dtype=torch.int32, device=dev)
    lens = torch.empty((R * Hkv,), dtype=torch.int32, device=dev)
    lib = load()
    nbytes = lib.msa_index_score_topk_workspace_size(B, N, Hkv, max_blocks)
    buf = _ws(workspace, dev).get("score", nbytes, dev)
    rc = lib.msa_index_score_topk_page_table(
        _ptr(q_idx), _ptr(k_idx_pages), _ptr(page_table), _ptr(seq_lens), B, N, Hkv, Di,
        max_blocks, k_idx_pages.shape[0], topk, _ptr(ids), _ptr(sc), _ptr(fpt), _ptr(lens),
        _ptr(buf), buf.numel(), _stream(dev))
    _lib.check("msa_index_score_topk_page_table", rc)
    return ids, sc, fpt, lens


def index_score_topk_noalloc(q_idx, k_idx_pages, page_table, seq_lens, N: int, topk: int,
                             with_scores: bool = True, out=None):
    """``index_score_topk`` without a workspace (``msa_index_score_topk_noalloc``).

    For callers that cannot hand the library device scratch memory: the library uses a
    fixed 8 MiB array of its own on each device instead. Calls on one device share that
    array, so calls that may overlap on the GPU must not use this function. The first
    call on a device resolves the array's address; make it before any stream capture.
    Raises MSAError (MSA_ERR_UNSUPPORTED) when B*N*Hkv*max_blocks needs more scratch.
    """
    _need(q_idx, "q_idx", torch.bfloat16, 3)
    _need(k_idx_pages, "k_idx_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, max_blocks = page_table.shape
    R, Hkv, Di = q_idx.shape
    if R != B * N or k_idx_pages.shape[1:] != (BLOCK, Hkv, Di) or seq_lens.numel() != B:
        raise ValueError("index_score_topk_noalloc: inconsistent shapes")
    dev = q_idx.device
    if out is None:
        ids = torch.empty((R, Hkv, topk), dtype=torch.int32, device=dev)
        sc = torch.empty((R, Hkv, topk), dtype=torch.float32, device=dev) if with_scores else None
    else:
        ids, sc = out
    rc = load().msa_index_score_topk_noalloc(_ptr(q_idx), _ptr(k_idx_pages), _ptr(page_table),
                                             _ptr(seq_lens), B, N, Hkv, Di, max_blocks,
                                             k_idx_pages.shape[0], topk, _ptr(ids), _ptr(sc),
                                             _stream(dev))
    _lib.check("msa_index_score_topk_noalloc", rc)
    return ids, sc


def build_sparse_page_table(block_ids, page_table, seq_lens, N: int, num_pages: int, out=None):
    """Flattened sparse page tables (``msa_build_sparse_page_table``).

    Returns (flat_page_table [B*N*Hkv, topk] int32, flat_kv_lens [B*N*Hkv] int32).
    """
    _need(block_ids, "block_ids", torch.int32, 3)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    R, Hkv, topk = block_ids.shape
    B, max_blocks = page_table.shape
    if R != B * N:
        raise ValueError("build_sparse_page_table: block_ids rows != B*N")
    dev = block_ids.device
    if out is None:
        fpt = torch.empty((R * Hkv, topk), dtype=torch.int32, device=dev)
        lens = torch.empty((R * Hkv,), dtype=torch.int32, device=dev)
    else:
        fpt, lens = out
    rc = load().msa_build_sparse_page_table(_ptr(block_ids), _ptr(page_table), _ptr(seq_lens), B, N,
                                            Hkv, topk, max_blocks, num_pages, _ptr(fpt), _ptr(lens),
                                            _stream(dev))
    _lib.check("msa_build_sparse_page_table", rc)
    return fpt, lens


# ------------------------------------------------------------------------------ stage 2

def stage_selected_kv(k_cache, v_cache, flat_page_table, out=None):
    """Copy the selected blocks' K/V to a device staging cache (``msa_stage_selected_kv``).

    k_cache, v_cache [P, 128, Hkv, D] bf16: CUDA tensors or pinned host tensors (read by the
    device directly); flat_page_table [R*Hkv, topk] int32 (CUDA). Returns (k_stage, v_stage
    [R*topk, 128, Hkv, D] bf16, stage_page_table [R*Hkv, topk] int32) for ``paged_sparse_decode``,
    written into ``out`` when given.
    """
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        if not isinstance(t, torch.Tensor) or not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{name}: must be a CUDA tensor or pinned host memory")
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous bf16 [P, 128, Hkv, D] tensor")
    _need(flat_page_table, "flat_page_table", torch.int32, 2)
    P, _, Hkv, D = k_cache.shape
    RH, topk = flat_page_table.shape
    if v_cache.shape != k_cache.shape or RH % Hkv:
        raise ValueError("stage_selected_kv: inconsistent shapes")
    R = RH // Hkv
    dev = flat_page_table.device
    if out is None:
        k_stage = torch.empty((R * topk, BLOCK, Hkv, D), dtype=torch.bfloat16, device=dev)
        v_stage = torch.empty_like(k_stage)
        spt = torch.empty_like(flat_page_table)
    else:
        k_stage, v_stage, spt = out
        _need(k_stage, "k_stage", torch.bfloat16, 4)
        _need(v_stage, "v_stage", torch.bfloat16, 4)
        _need(spt, "stage_page_table", torch.int32, 2)
        if (k_stage.shape != (R * topk, BLOCK, Hkv, D) or v_stage.shape != k_stage.shape
                or spt.shape != flat_page_table.shape):
            raise ValueError("stage_selected_kv: output shapes do not match")
    rc = load().msa_stage_selected_kv(k_cache.data_ptr(), v_cache.data_ptr(), P,
                                      _ptr(flat_page_table), R, Hkv, D, topk, _ptr(k_stage),
                                      _ptr(v_stage), _ptr(spt), _stream(dev))
    _lib.check("msa_stage_selected_kv", rc)
    return k_stage, v_stage, spt


def paged_sparse_decode(q, k_cache, v_cache, flat_page_table, flat_kv_lens,
                        with_lse: bool = True, workspace: Workspace | None = None, out=None):
    """Paged sparse decode attention (``msa_paged_sparse_decode``).

    q [R, Hq, D] bf16; caches [P, 128, Hkv, D] bf16; flat tables from
    ``build_sparse_page_table``. Returns (o [R, Hq, D] bf16, lse [R, Hq] fp32 or None).
    """
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(flat_page_table, "flat_page_table", torch.int32, 2)
    _need(flat_kv_lens, "flat_kv_lens", torch.int32, 1)
    R, Hq, D = q.shape
    P, _, Hkv, _ = k_cache.shape
    topk = flat_page_table.shape[1]
    if v_cache.shape != k_cache.shape or flat_page_table.shape[0] != R * Hkv:
        raise ValueError("paged_sparse_decode: inconsistent shapes")
    dev = q.device
    if out is None:
        o = torch.empty((R, Hq, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((R, Hq), dtype=torch.float32, device=dev) if with_lse else None
    else:
        o, lse = out
    lib = load()
    nbytes = lib.msa_paged_sparse_decode_workspace_size(R, Hq, Hkv, topk)
    buf = _ws(workspace, dev).get("decode", nbytes, dev)
    rc = lib.msa_paged_sparse_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(flat_page_table),
                                     _ptr(flat_kv_lens), R, Hq, Hkv, D, topk, P, _ptr(o), _ptr(lse),
                                     _ptr(buf), buf.numel(), _stream(dev))
    _lib.check("msa_paged_sparse_decode", rc)
    return o, lse


def sparse_prefill(q, k, v, block_ids, with_lse: bool = True,
                   workspace: Workspace | None = None, out=None):
    """KV-block-major sparse prefill with LSE merge (``msa_sparse_prefill``).

    q [T, Hq, D] bf16 at positions S_kv-T..S_kv-1; k, v [S_kv, Hkv, D] bf16;
    block_ids [T, Hkv, topk] int32. Returns (o [T, Hq, D] bf16, lse [T, Hq] fp32 or None).
    """
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(block_ids, "block_ids", torch.int32, 3)
    T, Hq, D = q.shape
    S_kv, Hkv, _ = k.shape
    topk = block_ids.shape[2]
    if v.shape != k.shape or block_ids.shape[:2] != (T, Hkv):
        raise ValueError("sparse_prefill: inconsistent shapes")
    dev = q.device
    if out is None:
        o = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((T, Hq), dtype=torch.float32, device=dev) if with_lse else None
    else:
        o, lse = out
    lib = load()
    nbytes = lib.msa_sparse_prefill_workspace_size(T, S_kv, Hq, Hkv, topk)
    buf = _ws(workspace, dev).get("prefill", nbytes, dev)
    rc = lib.msa_sparse_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(block_ids), T, S_kv, Hq, Hkv, D, topk,
                                _ptr(o), _ptr(lse), _ptr(buf), buf.numel(), _stream(dev))
    _lib.check("msa_sparse_prefill", rc)
    return o, lse


def sparse_prefill_paged(q, k_cache, v_cache, page_table, block_ids, S_kv: int,
                         with_lse: bool = True, workspace: Workspace | None = None, out=None):
    """Sparse prefill over a paged K/V cache (``msa_sparse_prefill_paged``).

    q [T, Hq, D] bf16 at positions S_kv-T..S_kv-1; k_cache, v_cache [P, 128, Hkv, D] bf16;
    page_table [ceil(S_kv/128)] int32 (page of each 128-token block); block_ids
    [T, Hkv, topk] int32. Returns (o [T, Hq, D] bf16, lse [T, Hq] fp32 or None).
    """
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 1)
    _need(block_ids, "block_ids", torch.int32, 3)
    T, Hq, D = q.shape
    P, _, Hkv, _ = k_cache.shape
    topk = block_ids.shape[2]
    if v_cache.shape != k_cache.shape or block_ids.shape[:2] != (T, Hkv) \
            or page_table.numel() < (S_kv + 127) // 128:
        raise ValueError("sparse_prefill_paged: inconsistent shapes")
    dev = q.device
    if out is None:
        o = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((T, Hq), dtype=torch.float32, device=dev) if with_lse else None
    else:
        o, lse = out
    lib = load()
    nbytes = lib.msa_sparse_prefill_workspace_size(T, S_kv, Hq, Hkv, topk)
    buf = _ws(workspace, dev).get("prefill", nbytes, dev)
    rc = lib.msa_sparse_prefill_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), P,
                                      _ptr(block_ids), T, S_kv, Hq, Hkv, D, topk, _ptr(o),
                                      _ptr(lse), _ptr(buf), buf.numel(), _stream(dev))
    _lib.check("msa_sparse_prefill_paged", rc)
    return o, lse


def prefill_bucket(block_ids, nblk: int, workspace: Workspace | None = None):
    """Invert selections into per-(group, block) lists (``msa_prefill_bucket``).

    Returns (offsets [Hkv, nblk+1] int32, entries [T*Hkv*topk] int32; only the first
    sum over groups of offsets[g, nblk] entries are meaningful).
    """
    _need(block_ids, "block_ids", torch.int32, 3)
    T, Hkv, topk = block_ids.shape
    dev = block_ids.device
    offsets = torch.empty((Hkv, nblk + 1), dtype=torch.int32, device=dev)
    entries = torch.empty((max(T * Hkv * topk, 1),), dtype=torch.int32, device=dev)
    lib = load()
    nbytes = lib.msa_prefill_bucket_workspace_size(T, Hkv, topk, nblk)
    buf = _ws(workspace, dev).get("bucket", nbytes, dev)
    rc = lib.msa_prefill_bucket(_ptr(block_ids), T, Hkv, topk, nblk, _ptr(offsets), _ptr(entries),
                                _ptr(buf), buf.numel(), _stream(dev))
    _lib.check("msa_prefill_bucket", rc)
    return offsets, entries


def lse_merge(o_parts, lse_parts, with_lse: bool = True):
    """Merge partials o_parts [U, S, G, D] (bf16 or fp32) with lse_parts [U, S, G] fp32."""
    if o_parts.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("lse_merge: o_parts must be bf16 or fp32")
    _need(o_parts, "o_parts", o_parts.dtype, 4)
    _need(lse_parts, "lse_parts", torch.float32, 3)
    U, S, G, D = o_parts.shape
    if lse_parts.shape != (U, S, G):
        raise ValueError("lse_merge: lse_parts shape")
    dev = o_parts.device
    o = torch.empty((U, G, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((U, G), dtype=torch.float32, device=dev) if with_lse else None
    rc = load().msa_lse_merge(_ptr(o_parts), 1 if o_parts.dtype == torch.bfloat16 else 0,
                              _ptr(lse_parts), U, S, G, D, _ptr(o), _ptr(lse), _stream(dev))
    _lib.check("msa_lse_merge", rc)
    return o, lse


def device_error() -> int:
    """Synchronise and return (then clear) the kernels' device error word (0 = none)."""
    w = ctypes.c_uint32(0)
    rc = load().msa_device_error(ctypes.byref(w))
    if rc not in (0, -6):
        _lib.check("msa_device_error", rc)
    return int(w.value)
