"""GPU parity at the full workload sizes, in the launch configuration bench.py times.

Where the oracle can compute every output in seconds it does (all rows of the decode scorers,
every flattened page table); otherwise outputs are compared on a seeded sample of units that
the oracle computes one by one. Tolerances are those of the other parity tests
(tests/_compare.py).
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_msa_gb300 as msa
import oracle
import workloads
from _compare import check_attention, check_selected_scores, check_selection, u16

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_sparse_attention_msa_gb300 import build
    build.build()
    msa.load()
    yield
    assert msa.device_error() == 0


def _sample(n_total: int, n: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = rng.choice(n_total, size=min(n, n_total), replace=False)
    return np.sort(np.concatenate([pick, [0, n_total - 1]])).astype(np.int64)


def test_decode_scoring_8x60032_full():
    """8 requests x 60032 tokens, Hkv 8, Di 128, k 16: every row, every group."""
    w = workloads.decode_scoring(DEV, seed=2)
    ids, sc = msa.index_score_topk(w["q_idx"], w["k_idx_pages"], w["page_table"], w["seq_lens"], 1,
                                   w["topk"])
    torch.cuda.synchronize()
    sl = w["seq_lens"].cpu().numpy()
    s_ref = oracle.block_scores(u16(w["q_idx"]), u16(w["k_idx_pages"]), w["page_table"].cpu().numpy(),
                                sl, 1)
    ids_ref, _ = oracle.topk(s_ref, oracle.query_positions(sl, 1), w["topk"])
    ids_np = ids.cpu().numpy()
    check_selection(ids_np, ids_ref, s_ref)
    check_selected_scores(ids_np, sc.cpu().numpy(), s_ref)
    planted = w["planted"].cpu().numpy()
    for b in range(w["B"]):
        for g in range(w["Hkv"]):
            assert set(planted[b, g].tolist()) <= set(ids_np[b, g].tolist())


def test_causal_prefill_32768_full():
    """32768-token causal chunk, Hq 64, Hkv 8, D 128, k 16: sampled (query, head) units."""
    w = workloads.causal_prefill(DEV, seed=3)
    o, lse = msa.sparse_prefill(w["q"], w["k"], w["v"], w["block_ids"])
    torch.cuda.synchronize()
    units = _sample(w["T"] * w["Hq"], 1024, seed=30)
    ref = oracle.sparse_prefill(u16(w["q"]), u16(w["k"]), u16(w["v"]), w["block_ids"].cpu().numpy(),
                                units=units)
    check_attention(o, lse, ref, units=units, what="causal_prefill prefill")


def test_paged_decode_64_requests_full():
    """64 requests, context ~U[8K,128K], Hq 64, Hkv 8, D 128, k 16: all page tables, sampled heads."""
    w = workloads.paged_decode(DEV, seed=4)
    fpt, lens = msa.build_sparse_page_table(w["block_ids"], w["page_table"], w["seq_lens"], 1,
                                            w["num_pages"])
    o, lse = msa.paged_sparse_decode(w["q"], w["k_cache"], w["v_cache"], fpt, lens)
    torch.cuda.synchronize()
    pt, sl, ids = (w[k].cpu().numpy() for k in ("page_table", "seq_lens", "block_ids"))
    fpt_ref, lens_ref = oracle.build_sparse_page_table(ids, pt, sl, 1)
    assert np.array_equal(fpt.cpu().numpy(), fpt_ref)
    assert np.array_equal(lens.cpu().numpy(), lens_ref)
    units = _sample(w["B"] * w["Hq"], 768, seed=40)
    ref = oracle.sparse_decode(u16(w["q"]), u16(w["k_cache"]), u16(w["v_cache"]), pt, sl, ids, 1,
                               units=units)
    check_attention(o, lse, ref, units=units, what="paged_decode decode")


def test_long_context_decode_pipeline_1m():
    """4 requests x 1,048,576 tokens, k 32: score -> top-k -> sparse page table -> paged decode."""
    w = workloads.long_context_decode(DEV, seed=5)
    ids, sc = msa.index_score_topk(w["q_idx"], w["k_idx_pages"], w["page_table"], w["seq_lens"], 1,
                                   w["topk"])
    fpt, lens = msa.build_sparse_page_table(ids, w["page_table"], w["seq_lens"], 1, w["num_pages"])
    o, lse = msa.paged_sparse_decode(w["q"], w["k_cache"], w["v_cache"], fpt, lens)
    torch.cuda.synchronize()
    pt, sl = w["page_table"].cpu().numpy(), w["seq_lens"].cpu().numpy()
    s_ref = oracle.block_scores(u16(w["q_idx"]), u16(w["k_idx_pages"]), pt, sl, 1)
    ids_ref, _ = oracle.topk(s_ref, oracle.query_positions(sl, 1), w["topk"])
    ids_np = ids.cpu().numpy()
    check_selection(ids_np, ids_ref, s_ref)
    check_selected_scores(ids_np, sc.cpu().numpy(), s_ref)
    fpt_ref, lens_ref = oracle.build_sparse_page_table(ids_np, pt, sl, 1)
    assert np.array_equal(fpt.cpu().numpy(), fpt_ref)
    assert np.array_equal(lens.cpu().numpy(), lens_ref)
    ref = oracle.sparse_decode(u16(w["q"]), u16(w["k_cache"]), u16(w["v_cache"]), pt, sl, ids_np, 1)
    check_attention(o, lse, ref, what="1M-token decode")


def test_long_context_prefill_chunk_on_1m_prefix():
    """32768-token chunk after a 1,048,576-token prefix, k 32: scoring of every row on the GPU
    (sampled rows against the oracle), then block-major attention on sampled units."""
    w = workloads.long_context_prefill(DEV, seed=6)
    T, S, Hkv, Di, P = w["T"], w["S"], w["Hkv"], w["Di"], w["P"]
    kidx_pages = w["k_idx"].view(P, 128, Hkv, Di)
    sl = torch.tensor([S], dtype=torch.int32, device=DEV)
    ids, sc = msa.index_score_topk(w["q_idx"], kidx_pages, w["page_table"], sl, T, w["topk"])
    torch.cuda.synchronize()
    rows = _sample(T, 96, seed=50)
    s_ref = oracle.block_scores(u16(w["q_idx"]), u16(kidx_pages), w["page_table"].cpu().numpy(),
                                sl.cpu().numpy(), T, rows=rows)
    q_pos = oracle.query_positions(sl.cpu().numpy(), T)[rows]
    ids_ref, _ = oracle.topk(s_ref, q_pos, w["topk"])
    ids_np = ids.cpu().numpy()
    check_selection(ids_np[rows], ids_ref, s_ref)
    check_selected_scores(ids_np[rows], sc.cpu().numpy()[rows], s_ref)
    k = w["k"][:S]
    v = w["v"][:S]
    o, lse = msa.sparse_prefill(w["q"], k, v, ids)
    torch.cuda.synchronize()
    units = _sample(T * w["Hq"], 768, seed=51)
    ref = oracle.sparse_prefill(u16(w["q"]), u16(k), u16(v), ids_np, units=units)
    check_attention(o, lse, ref, units=units, what="prefill chunk on a 1M prefix")
