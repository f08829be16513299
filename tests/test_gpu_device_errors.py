"""GPU tests of the device error word: inputs made bad on the host, of the kinds the kernels
check before they form any address from them, must set the matching bit of msa_device_error()
while every output still follows its documented rule.

  * an out-of-range page id in the scorer's page table is read as page 0 (bit 0);
  * a sequence length above max_blocks*128 is clamped to max_blocks*128 (bit 1);
  * the sparse page-table build writes -1 for a block id past the query's local block (bit 1)
    or whose page is out of range (bit 0);
  * the paged decode reads an out-of-range virtual page as page 0 of group 0 (bit 0).
The expected outputs are the oracle's on the inputs with the documented replacement applied.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_msa_gb300 as msa
import oracle
import workloads
from _compare import check_attention, check_selected_scores, check_selection, u16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
BAD_PAGE, BAD_BLOCK = 1, 2


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_sparse_attention_msa_gb300 import build
    build.build()
    msa.load()
    assert msa.device_error() == 0  # nothing left over from earlier tests
    yield
    assert msa.device_error() == 0


def _score_and_check(w, pt_gpu, sl_gpu, pt_ref, sl_ref, N, topk):
    ids, sc = msa.index_score_topk(w["q_idx"].to(DEV), w["k_idx_pages"].to(DEV), pt_gpu.to(DEV),
                                   sl_gpu.to(DEV), N, topk)
    word = msa.device_error()  # synchronises, reads and clears
    s_ref = oracle.block_scores(u16(w["q_idx"]), u16(w["k_idx_pages"]), pt_ref.numpy(),
                                sl_ref.numpy(), N)
    ids_ref, _ = oracle.topk(s_ref, oracle.query_positions(sl_ref.numpy(), N), topk)
    check_selection(ids.cpu().numpy(), ids_ref, s_ref)
    check_selected_scores(ids.cpu().numpy(), sc.cpu().numpy(), s_ref)
    return word


@pytest.mark.parametrize("seq_lens,N,Hkv,Di,topk", [
    ([3000, 2000, 1000, 5000], 1, 4, 64, 8),   # streaming scorer (N <= 8)
    ([2048, 1500], 40, 2, 128, 6),              # multi-row tensor-core scorer (N > 8)
])
def test_scorer_reads_an_out_of_range_page_as_page_zero(seq_lens, N, Hkv, Di, topk):
    w = workloads.index_workload(seq_lens, N, Hkv, Di, seed=41, device="cpu")
    pt_bad = w["page_table"].clone()
    pt_bad[1, 5] = w["num_pages"] + 7          # block 5 of request 1 is inside its length
    pt_ref = pt_bad.clone()
    pt_ref[1, 5] = 0
    word = _score_and_check(w, pt_bad, w["seq_lens"], pt_ref, w["seq_lens"], N, topk)
    assert word & BAD_PAGE, f"device error word {word:#x}"


def test_scorer_clamps_a_length_past_the_page_table():
    seq_lens, N, Hkv, Di, topk = [3000, 2000, 1000, 5000], 1, 4, 64, 8
    w = workloads.index_workload(seq_lens, N, Hkv, Di, seed=42, device="cpu")
    max_blocks = w["page_table"].shape[1]
    sl_bad = w["seq_lens"].clone()
    sl_bad[2] = max_blocks * 128 + 500         # request 2 claims more tokens than its table holds
    sl_ref = sl_bad.clone()
    sl_ref[2] = max_blocks * 128               # unused table entries are page 0: in range
    word = _score_and_check(w, w["page_table"], sl_bad, w["page_table"], sl_ref, N, topk)
    assert word & BAD_BLOCK, f"device error word {word:#x}"


def test_page_table_build_drops_bad_ids():
    seq_lens, N, Hq, Hkv, topk = [517, 1500, 129, 9000], 1, 16, 4, 5
    w = workloads.decode_workload(seq_lens, N, Hq, Hkv, 128, topk, seed=43, device="cpu")
    ids = w["block_ids"].clone()
    pt = w["page_table"].clone()
    ids[1, 2, 0] = 40                          # past request 1's local block (1499 // 128 = 11)
    pt[3, int(ids[3, 0, 1])] = w["num_pages"] + 3   # a kept block of request 3 on a bad page
    fpt, lens = msa.build_sparse_page_table(ids.to(DEV), pt.to(DEV), w["seq_lens"].to(DEV), N,
                                            w["num_pages"])
    word = msa.device_error()
    assert word & BAD_PAGE and word & BAD_BLOCK, f"device error word {word:#x}"
    ids_ref = ids.clone()
    ids_ref[1, 2, 0] = -1
    bad_blk = int(ids[3, 0, 1])
    ids_ref[3][ids_ref[3] == bad_blk] = -1     # every group of request 3 that kept that block
    fpt_ref, lens_ref = oracle.build_sparse_page_table(ids_ref.numpy(), pt.numpy(),
                                                       w["seq_lens"].numpy(), N)
    assert np.array_equal(fpt.cpu().numpy(), fpt_ref)
    assert np.array_equal(lens.cpu().numpy(), lens_ref)


def test_paged_decode_reads_a_bad_virtual_page_as_page_zero():
    seq_lens, N, Hq, Hkv, topk = [517, 1500, 129, 9000], 1, 32, 4, 5
    w = workloads.decode_workload(seq_lens, N, Hq, Hkv, 128, topk, seed=44, device="cpu")
    fpt, lens = oracle.build_sparse_page_table(w["block_ids"].numpy(), w["page_table"].numpy(),
                                               w["seq_lens"].numpy(), N)
    fpt_bad = fpt.copy()
    assert fpt_bad[6, 0] >= 0
    fpt_bad[6, 0] = w["num_pages"] * 128 * Hkv + 9   # past the last virtual page
    fpt_ref = fpt_bad.copy()
    fpt_ref[6, 0] = 0                                  # page 0, group 0
    o, lse = msa.paged_sparse_decode(w["q"].to(DEV), w["k_cache"].to(DEV), w["v_cache"].to(DEV),
                                     torch.from_numpy(fpt_bad).to(DEV), torch.from_numpy(lens).to(DEV))
    word = msa.device_error()
    assert word & BAD_PAGE, f"device error word {word:#x}"
    ref = oracle.paged_decode_flat(u16(w["q"]), u16(w["k_cache"]), u16(w["v_cache"]), fpt_ref, lens)
    check_attention(o, lse, ref, what="decode with a bad virtual page")
