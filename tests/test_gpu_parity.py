"""GPU parity: every C-ABI call against the CPU oracle on the same seeded inputs.

Sizes span several tiles and ragged tails (sequence lengths not multiples of 128, fewer
causal blocks than k, a query inside block 0) and finish in seconds on the oracle.
Tolerances (tests/_compare.py): block ids bit-exact up to near-tie swaps (1e-3 relative
on the oracle's scores), scores 1e-3 relative, attention o 2e-2 max-abs / 5e-3 mean-abs,
LSE 1e-3; page tables and bucket lists bit-exact.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_msa_gb300 as msa
import oracle
import workloads
from _compare import (check_attention, check_selected_scores, check_selection, f32, u16)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_sparse_attention_msa_gb300 import build
    build.build()
    msa.load()
    yield
    assert msa.device_error() == 0


def _score_case(seq_lens, N, Hkv, Di, topk, seed, n_planted=0):
    w = workloads.index_workload(seq_lens, N, Hkv, Di, seed=seed, device="cpu", n_planted=n_planted)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in w.items()}
    ids, sc = msa.index_score_topk(d["q_idx"], d["k_idx_pages"], d["page_table"], d["seq_lens"], N,
                                   topk)
    torch.cuda.synchronize()
    s_ref = oracle.block_scores(u16(w["q_idx"]), u16(w["k_idx_pages"]), w["page_table"].numpy(),
                                w["seq_lens"].numpy(), N)
    ids_ref, _ = oracle.topk(s_ref, oracle.query_positions(w["seq_lens"].numpy(), N), topk)
    ids_np = ids.cpu().numpy()
    check_selection(ids_np, ids_ref, s_ref)
    check_selected_scores(ids_np, sc.cpu().numpy(), s_ref)
    return w, ids_np, ids_ref


@pytest.mark.parametrize("seq_lens,N,Hkv,Di,topk", [
    ([517, 300, 1000, 128, 60], 1, 8, 128, 4),      # ragged, fewer blocks than k, one block
    ([5000, 129, 3000], 1, 2, 64, 16),              # Di 64, Hkv 2
    ([2000, 2049], 1, 16, 128, 6),                  # Hkv 16 (16 tokens per stage)
    ([1500, 700], 1, 1, 64, 3),                     # Hkv 1 (128-row stages)
    ([4096, 3000, 999, 12000], 4, 8, 128, 8),       # multi-token decode N = 4
    ([7000, 6100], 8, 4, 64, 16),                   # N = 8
])
def test_score_topk_streaming_path(seq_lens, N, Hkv, Di, topk):
    _score_case(seq_lens, N, Hkv, Di, topk, seed=hash((tuple(seq_lens), N, Hkv)) % 1000)


@pytest.mark.parametrize("seq_lens,N,Hkv,Di,topk", [
    ([517, 3000, 129, 7000], 2, 8, 128, 16),        # two rows per request, ragged, one short request
    ([2000, 4100, 260], 3, 2, 64, 6),               # odd row count, Di 64
    ([6000, 5000, 999, 12000], 8, 16, 128, 8),      # Hkv 16 (the largest): 4 ring stages
    ([3000, 16, 4097], 16, 1, 128, 5),              # 16 rows (a full MMA N), a request of 16 tokens
    ([9000, 1500], 12, 4, 64, 32),                  # k 32, rows straddling a block boundary
])
def test_score_topk_multi_token_tensor_core_path(seq_lens, N, Hkv, Di, topk):
    """2 <= N <= 16 query rows per request: the tensor-core scorer (128-token block as M, rows
    padded to 16 as N) with the top-k fused into its last CTA per request."""
    _score_case(seq_lens, N, Hkv, Di, topk, seed=hash((tuple(seq_lens), N, Di)) % 1000 + 3)


@pytest.mark.parametrize("seq_lens,N,Hkv,Di,topk", [
    ([700], 300, 2, 64, 4),                         # prefill chunk, ragged row tile
    ([2048, 1500], 33, 4, 128, 5),                  # two requests, N above the decode scorers' cap
    ([5000, 3000], 600, 2, 128, 8),                 # chunks after a prefix, several row tiles
    ([1300], 1300, 4, 128, 16),                     # whole sequence is the chunk, ragged tiles
    ([9000, 129, 4000], 129, 2, 64, 6),             # one request with seq == N, 4-block chunks
])
def test_score_topk_row_path(seq_lens, N, Hkv, Di, topk):
    _score_case(seq_lens, N, Hkv, Di, topk, seed=7)


def test_score_topk_planted_blocks_found():
    w, ids, _ = _score_case([60 * 128, 45 * 128 + 3, 70 * 128], 1, 8, 128, 16, seed=3, n_planted=8)
    planted = w["planted"].numpy()
    for b in range(3):
        for g in range(8):
            assert set(planted[b, g].tolist()) <= set(ids[b, g].tolist())


def test_score_topk_workspace_reuse_and_ties():
    # identical keys in every block -> all scores tie; the lower ids must win every time,
    # on repeated calls with the same (kept-zero) workspace
    seq_lens, N, Hkv, Di, k = [640, 1280], 1, 2, 64, 4
    w = workloads.index_workload(seq_lens, N, Hkv, Di, seed=1, device="cpu")
    w["k_idx_pages"][:] = w["k_idx_pages"][0:1, 0:1]
    ws = msa.Workspace()
    for _ in range(3):
        ids, _ = msa.index_score_topk(w["q_idx"].to(DEV), w["k_idx_pages"].to(DEV),
                                      w["page_table"].to(DEV), w["seq_lens"].to(DEV), N, k,
                                      workspace=ws)
        s_ref = oracle.block_scores(u16(w["q_idx"]), u16(w["k_idx_pages"]), w["page_table"].numpy(),
                                    w["seq_lens"].numpy(), N)
        ids_ref, _ = oracle.topk(s_ref, oracle.query_positions(w["seq_lens"].numpy(), N), k)
        assert np.array_equal(ids.cpu().numpy(), ids_ref)


@pytest.mark.parametrize("seq_lens,N,Hkv,Di,topk", [
    ([5000, 129, 3000, 777], 1, 8, 128, 16),     # decode: page table built in the scorer's tail
    ([2500, 1400], 4, 4, 64, 8),                  # multi-token rows, still the fused tail
    ([2048, 1500], 33, 2, 128, 5),                # long rows: scorer, top-k, page-table kernels
])
def test_index_score_topk_page_table_equals_the_two_calls(seq_lens, N, Hkv, Di, topk):
    w = workloads.index_workload(seq_lens, N, Hkv, Di, seed=31, device="cpu")
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in w.items()}
    args = (d["q_idx"], d["k_idx_pages"], d["page_table"], d["seq_lens"], N, topk)
    ids_f, sc_f, fpt_f, lens_f = msa.index_score_topk_page_table(*args)
    ids, sc = msa.index_score_topk(*args)
    fpt, lens = msa.build_sparse_page_table(ids, d["page_table"], d["seq_lens"], N,
                                            d["k_idx_pages"].shape[0])
    torch.cuda.synchronize()
    assert torch.equal(ids_f, ids) and torch.equal(sc_f, sc)
    assert torch.equal(fpt_f, fpt) and torch.equal(lens_f, lens)
    fpt_ref, lens_ref = oracle.build_sparse_page_table(ids.cpu().numpy(), w["page_table"].numpy(),
                                                       w["seq_lens"].numpy(), N)
    assert np.array_equal(fpt_f.cpu().numpy(), fpt_ref) and np.array_equal(lens_f.cpu().numpy(), lens_ref)
    assert msa.device_error() == 0


@pytest.mark.parametrize("N", [1, 3])
def test_sparse_page_table_bit_exact(N):
    w = workloads.decode_workload([517, 1500, 129, 9000], N, 16, 8, 128, 7, seed=2, device="cpu")
    fpt, lens = msa.build_sparse_page_table(w["block_ids"].to(DEV), w["page_table"].to(DEV),
                                            w["seq_lens"].to(DEV), N, w["num_pages"])
    fpt_ref, lens_ref = oracle.build_sparse_page_table(w["block_ids"].numpy(), w["page_table"].numpy(),
                                                       w["seq_lens"].numpy(), N)
    assert np.array_equal(fpt.cpu().numpy(), fpt_ref)
    assert np.array_equal(lens.cpu().numpy(), lens_ref)


@pytest.mark.parametrize("seq_lens,N,Hq,Hkv,topk", [
    ([517, 1500, 129, 9000, 40], 1, 64, 8, 16),      # G 8, ragged, 1-block request
    ([3000, 700], 1, 16, 4, 5),                       # G 4
    ([2500, 2600, 2700], 2, 32, 2, 9),                # G 16, N 2
    ([20000], 1, 8, 8, 32),                           # G 1, k 32
    ([3000, 5000, 700], 1, 32, 16, 8),                # Hkv 16 (the largest), G 2
])
def test_paged_sparse_decode(seq_lens, N, Hq, Hkv, topk):
    w = workloads.decode_workload(seq_lens, N, Hq, Hkv, 128, topk, seed=5, device="cpu")
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in w.items()}
    fpt, lens = msa.build_sparse_page_table(d["block_ids"], d["page_table"], d["seq_lens"], N,
                                            w["num_pages"])
    o, lse = msa.paged_sparse_decode(d["q"], d["k_cache"], d["v_cache"], fpt, lens)
    torch.cuda.synchronize()
    ref = oracle.sparse_decode(u16(w["q"]), u16(w["k_cache"]), u16(w["v_cache"]), w["page_table"].numpy(),
                               w["seq_lens"].numpy(), w["block_ids"].numpy(), N)
    check_attention(o, lse, ref, what="decode")


def test_paged_sparse_decode_few_rows_cluster_merge():
    """Few flattened rows (4 requests x 8 groups, the 1M-context batch shape at shorter
    contexts): each row is owned by a cluster whose 32 warps take a page range each and merge
    in distributed shared memory. Short requests leave some warps without a visible page."""
    seq_lens = [40000, 9000, 700, 128]
    N, Hq, Hkv, topk = 1, 64, 8, 32
    w = workloads.decode_workload(seq_lens, N, Hq, Hkv, 128, topk, seed=9, device="cpu")
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in w.items()}
    fpt, lens = msa.build_sparse_page_table(d["block_ids"], d["page_table"], d["seq_lens"], N,
                                            w["num_pages"])
    o, lse = msa.paged_sparse_decode(d["q"], d["k_cache"], d["v_cache"], fpt, lens)
    o2, lse2 = msa.paged_sparse_decode(d["q"], d["k_cache"], d["v_cache"], fpt, lens)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    ref = oracle.sparse_decode(u16(w["q"]), u16(w["k_cache"]), u16(w["v_cache"]), w["page_table"].numpy(),
                               w["seq_lens"].numpy(), w["block_ids"].numpy(), N)
    check_attention(o, lse, ref, what="decode")
    assert msa.device_error() == 0


def test_paged_sparse_decode_ranges_cross_rows():
    """More (row, page) units than the grid has warps: each warp's range covers several pages
    and crosses row boundaries, so rows are split into segments merged through their slots;
    ragged lengths leave some pages of a row unselected."""
    seq_lens = [int(x) for x in np.random.default_rng(3).integers(1, 4000, 150)]
    N, Hq, Hkv, topk = 2, 16, 4, 6
    w = workloads.decode_workload(seq_lens, N, Hq, Hkv, 128, topk, seed=6, device="cpu")
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in w.items()}
    fpt, lens = msa.build_sparse_page_table(d["block_ids"], d["page_table"], d["seq_lens"], N,
                                            w["num_pages"])
    assert fpt.numel() > 8 * 152  # units per launch exceed the warps of a full grid
    o, lse = msa.paged_sparse_decode(d["q"], d["k_cache"], d["v_cache"], fpt, lens)
    o2, lse2 = msa.paged_sparse_decode(d["q"], d["k_cache"], d["v_cache"], fpt, lens)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)  # no dependence on warp timing
    ref = oracle.sparse_decode(u16(w["q"]), u16(w["k_cache"]), u16(w["v_cache"]), w["page_table"].numpy(),
                               w["seq_lens"].numpy(), w["block_ids"].numpy(), N)
    check_attention(o, lse, ref, what="decode")
    assert msa.device_error() == 0


@pytest.mark.parametrize("T,S,Hq,Hkv,topk,n_shared", [
    (300, 700, 16, 2, 4, 2),        # chunk after a prefix, ragged
    (1000, 1000, 64, 8, 16, 12),    # causal, causal_prefill structure at small T
    (200, 200, 8, 8, 3, 0),         # G 1
    (129, 5000, 32, 2, 8, 4),       # G 16, long prefix
    (257, 800, 8, 4, 5, 3),         # G 2: block-major only
    (1, 4000, 64, 8, 16, 12),       # one query after a prefix: a pair with one valid query
    (300, 900, 32, 16, 4, 2),       # Hkv 16 (the largest), G 2
])
def test_sparse_prefill(T, S, Hq, Hkv, topk, n_shared):
    w = workloads.prefill_workload(T, S, Hq, Hkv, 128, topk, seed=11, device="cpu", n_shared=n_shared)
    o, lse = msa.sparse_prefill(w["q"].to(DEV), w["k"].to(DEV), w["v"].to(DEV), w["block_ids"].to(DEV))
    torch.cuda.synchronize()
    ref = oracle.sparse_prefill(u16(w["q"]), u16(w["k"]), u16(w["v"]), w["block_ids"].numpy())
    check_attention(o, lse, ref, what="prefill")


def test_sparse_prefill_shared_blocks_beyond_the_dense_cap():
    """k 64 with two query halves per 32-query pair choosing disjoint 62-block sets: 126 blocks
    are shared by at least half of the pair, more than the query-major pass takes, so the blocks
    past its cap must reach the output through the block-major pass."""
    T, prefix, Hq, Hkv, D, k = 64, 16384, 16, 2, 128, 64
    S = prefix + T
    gen = torch.Generator().manual_seed(77)
    q = workloads.randn_bf16((T, Hq, D), gen, "cpu", scale=D ** -0.5)
    kk = workloads.randn_bf16((S, Hkv, D), gen, "cpu")
    vv = workloads.randn_bf16((S, Hkv, D), gen, "cpu")
    local = (prefix + torch.arange(T)) // 128            # block 128 for every query
    ids = torch.empty((T, Hkv, k), dtype=torch.int32)
    for t in range(T):
        half = (t % 32) // 16
        body = torch.arange(1 + 62 * half, 63 + 62 * half)  # 62 blocks, disjoint per half
        row = torch.cat([torch.tensor([0]), body, local[t:t + 1]]).to(torch.int32)
        ids[t, :, :] = torch.sort(row).values
    o, lse = msa.sparse_prefill(q.to(DEV), kk.to(DEV), vv.to(DEV), ids.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.sparse_prefill(u16(q), u16(kk), u16(vv), ids.numpy())
    check_attention(o, lse, ref, what="prefill beyond the dense cap")


def test_sparse_prefill_beyond_two_million_tokens():
    """A 64-token chunk after a 2,098,152-token prefix (16392 blocks): the blocks a query pair
    shares lie on both sides of the 16384-block windows the shared-block selection counts in."""
    T, prefix, Hq, Hkv, D, k = 64, 16391 * 128 + 104, 8, 1, 128, 16
    S = prefix + T
    gen = torch.Generator().manual_seed(78)
    q = workloads.randn_bf16((T, Hq, D), gen, "cpu", scale=D ** -0.5)
    kk = workloads.randn_bf16((S, Hkv, D), gen, "cpu")
    vv = workloads.randn_bf16((S, Hkv, D), gen, "cpu")
    shared = [0, 100, 5000, 16383, 16384, 16385, 16390]
    ids = torch.empty((T, Hkv, k), dtype=torch.int32)
    for t in range(T):
        local = (prefix + t) // 128
        pool = torch.tensor([b for b in range(1, local) if b not in shared])
        extra = pool[torch.randperm(pool.numel(), generator=gen)[:k - len(shared) - 1]]
        row = torch.cat([torch.tensor(shared), extra, torch.tensor([local])]).to(torch.int32)
        ids[t, 0, :] = torch.sort(row).values
    o, lse = msa.sparse_prefill(q.to(DEV), kk.to(DEV), vv.to(DEV), ids.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.sparse_prefill(u16(q), u16(kk), u16(vv), ids.numpy())
    check_attention(o, lse, ref, what="prefill past 16384 blocks")


@pytest.mark.parametrize("T,prefix,Hq,Hkv,topk,n_shared", [
    (300, 1000, 64, 8, 8, 6),       # G 8: query-major pass + block-major remainder
    (200, 333, 16, 4, 4, 0),        # G 4: block-major only; partial last page
])
def test_sparse_prefill_paged_equals_contiguous(T, prefix, Hq, Hkv, topk, n_shared):
    """The paged form reads the same K/V through a shuffled page table: bit-identical to the
    contiguous form, and within tolerance of the oracle."""
    S = prefix + T
    w = workloads.prefill_workload(T, S, Hq, Hkv, 128, topk, seed=13, device="cpu", n_shared=n_shared)
    nblk = (S + 127) // 128
    P = nblk + 3                                   # a few unused pages
    gen = torch.Generator().manual_seed(14)
    perm = torch.randperm(P, generator=gen)[:nblk].to(torch.int32)
    pad = nblk * 128 - S
    def paged(x):
        xp = torch.cat([x, torch.zeros((pad,) + x.shape[1:], dtype=x.dtype)]).view(nblk, 128, Hkv, 128)
        cache = workloads.randn_bf16((P, 128, Hkv, 128), gen, "cpu")   # garbage in unused pages
        cache[perm.long()] = xp
        return cache
    kc, vc = paged(w["k"]), paged(w["v"])
    o_p, lse_p = msa.sparse_prefill_paged(w["q"].to(DEV), kc.to(DEV), vc.to(DEV), perm.to(DEV),
                                          w["block_ids"].to(DEV), S)
    o_c, lse_c = msa.sparse_prefill(w["q"].to(DEV), w["k"].to(DEV), w["v"].to(DEV),
                                    w["block_ids"].to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(o_p, o_c)
    assert torch.equal(lse_p, lse_c)
    ref = oracle.sparse_prefill(u16(w["q"]), u16(w["k"]), u16(w["v"]), w["block_ids"].numpy())
    check_attention(o_p, lse_p, ref, what="paged prefill")
    assert msa.device_error() == 0


@pytest.mark.parametrize("host", [True, False])
def test_staged_kv_decode_equals_decode_on_the_full_cache(host):
    """Selected blocks' K/V copied from the paged caches (pinned host memory or device) to a
    staging cache: the paged decode on it equals the decode on the full caches bit for bit (the
    same values in the same order, and the decode's sums do not depend on warp timing), and
    the oracle's sparse decode within the attention tolerances."""
    w = workloads.decode_workload([517, 1500, 129, 9000], 2, 32, 8, 128, 7, seed=9, device="cpu")
    kc = w["k_cache"].pin_memory() if host else w["k_cache"].to(DEV)
    vc = w["v_cache"].pin_memory() if host else w["v_cache"].to(DEV)
    fpt, lens = msa.build_sparse_page_table(w["block_ids"].to(DEV), w["page_table"].to(DEV),
                                            w["seq_lens"].to(DEV), 2, w["num_pages"])
    ks, vs, spt = msa.stage_selected_kv(kc, vc, fpt)
    q = w["q"].to(DEV)
    o_s, lse_s = msa.paged_sparse_decode(q, ks, vs, spt, lens)
    o_f, lse_f = msa.paged_sparse_decode(q, w["k_cache"].to(DEV), w["v_cache"].to(DEV), fpt, lens)
    torch.cuda.synchronize()
    assert torch.equal(lse_s, lse_f)
    assert torch.equal(o_s, o_f)
    assert torch.equal(spt < 0, fpt < 0)
    # and both equal the oracle's sparse decode on the same inputs
    ref = oracle.sparse_decode(u16(w["q"]), u16(w["k_cache"]), u16(w["v_cache"]), w["page_table"].numpy(),
                               w["seq_lens"].numpy(), w["block_ids"].numpy(), 2)
    check_attention(o_s, lse_s, ref, what=f"staged decode (host={host})")
    assert msa.device_error() == 0


def test_prefill_bucket_lists():
    w = workloads.prefill_workload(900, 1500, 16, 4, 128, 6, seed=4, device="cpu", n_shared=3)
    nblk = (1500 + 127) // 128
    off, ent = msa.prefill_bucket(w["block_ids"].to(DEV), nblk)
    off_ref, ent_ref = oracle.prefill_buckets(w["block_ids"].numpy(), nblk)
    off = off.cpu().numpy()
    ent = ent.cpu().numpy()
    assert np.array_equal(off, off_ref)
    base = 0
    for g in range(off.shape[0]):
        for j in range(nblk):
            a, b = base + off[g, j], base + off[g, j + 1]
            assert np.array_equal(np.sort(ent[a:b]), ent_ref[a:b])  # order inside a list is free
        base += off[g, nblk]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_lse_merge(dtype):
    g = torch.Generator().manual_seed(0)
    U, S, G, D = 37, 9, 4, 128
    o_parts = torch.randn(U, S, G, D, generator=g).to(dtype)
    lse_parts = torch.randn(U, S, G, generator=g) * 3
    lse_parts[0, :, :] = -float("inf")              # unit with no partial
    lse_parts[1, 1:, :] = -float("inf")             # single partial
    lse_parts[2, ::2, 1] = -float("inf")
    o, lse = msa.lse_merge(o_parts.to(DEV), lse_parts.to(DEV))
    torch.cuda.synchronize()
    o_np, lse_np = f32(o), lse.cpu().numpy()
    op = o_parts.float().numpy()
    lp = lse_parts.numpy()
    for u in range(U):
        for e in range(G):
            ref_o, ref_l = oracle.lse_merge(op[u, :, e], lp[u, :, e])
            assert np.abs(o_np[u, e] - ref_o).max() <= 1e-2
            if np.isfinite(ref_l):
                assert abs(lse_np[u, e] - ref_l) <= 1e-4
            else:
                assert lse_np[u, e] == -np.inf


def test_pr1_layer_end_to_end():
    """PR1: 2048-token layer (Hq 8, Hkv 2, Di 64, k 4): prefill then 16 decode steps."""
    w = workloads.tiny_layer("cpu", seed=0)
    T, Hq, Hkv, D, Di, k, P = w["T"], w["Hq"], w["Hkv"], w["D"], w["Di"], w["topk"], w["P"]
    kidx = w["k_idx"].view(P, 128, Hkv, Di)
    kc, vc = w["k"].view(P, 128, Hkv, D), w["v"].view(P, 128, Hkv, D)
    pt = w["page_table"]
    g_kidx, g_kc, g_vc, g_pt = kidx.to(DEV), kc.to(DEV), vc.to(DEV), pt.to(DEV)
    # prefill: score + top-k for all 2048 rows, then block-major attention on the GPU's selection
    sl = torch.tensor([T], dtype=torch.int32)
    ids, sc = msa.index_score_topk(w["q_idx"][:T].to(DEV), g_kidx, g_pt, sl.to(DEV), T, k)
    s_ref = oracle.block_scores(u16(w["q_idx"][:T]), u16(kidx), pt.numpy(), sl.numpy(), T)
    ids_ref, _ = oracle.topk(s_ref, oracle.query_positions(sl.numpy(), T), k)
    check_selection(ids.cpu().numpy(), ids_ref, s_ref)
    check_selected_scores(ids.cpu().numpy(), sc.cpu().numpy(), s_ref)
    o, lse = msa.sparse_prefill(w["q"][:T].to(DEV), w["k"][:T].to(DEV), w["v"][:T].to(DEV), ids)
    ref = oracle.sparse_prefill(u16(w["q"][:T]), u16(w["k"][:T]), u16(w["v"][:T]), ids.cpu().numpy())
    check_attention(o, lse, ref, what="pr1 prefill")
    # 16 decode steps: the cache already holds every token; step s sees seq_len T+s+1
    for s in range(16):
        pos = T + s
        sl = torch.tensor([pos + 1], dtype=torch.int32)
        q_idx = w["q_idx"][pos:pos + 1]
        ids, _ = msa.index_score_topk(q_idx.to(DEV), g_kidx, g_pt, sl.to(DEV), 1, k)
        s_ref = oracle.block_scores(u16(q_idx), u16(kidx), pt.numpy(), sl.numpy(), 1)
        ids_ref, _ = oracle.topk(s_ref, oracle.query_positions(sl.numpy(), 1), k)
        check_selection(ids.cpu().numpy(), ids_ref, s_ref)
        fpt, lens = msa.build_sparse_page_table(ids, g_pt, sl.to(DEV), 1, P)
        o, lse = msa.paged_sparse_decode(w["q"][pos:pos + 1].to(DEV), g_kc, g_vc, fpt, lens)
        ref = oracle.sparse_decode(u16(w["q"][pos:pos + 1]), u16(kc), u16(vc), pt.numpy(), sl.numpy(),
                                   ids.cpu().numpy(), 1)
        check_attention(o, lse, ref, what=f"pr1 decode step {s}")


def test_full_selection_equals_dense_causal_attention():
    """k >= number of causal blocks: MSA prefill is dense causal attention (oracle-checked)."""
    T = 600
    w = workloads.prefill_workload(T, T, 16, 2, 128, 5, seed=9, device="cpu", n_shared=0)
    assert (w["block_ids"][-1] >= 0).all()  # the last query keeps all 5 blocks
    o, lse = msa.sparse_prefill(w["q"].to(DEV), w["k"].to(DEV), w["v"].to(DEV), w["block_ids"].to(DEV))
    torch.cuda.synchronize()
    ref = oracle.sparse_prefill(u16(w["q"]), u16(w["k"]), u16(w["v"]), w["block_ids"].numpy())
    check_attention(o, lse, ref, what="dense-equivalent prefill")
