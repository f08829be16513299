"""msa_index_score_topk_noalloc: index scoring + top-k for callers that cannot provide device
scratch memory (for example a plugin whose host framework owns all device memory, or a decode
loop that must not let a cudaMalloc synchronise the device). The library then uses its own
fixed scratch array, shared by every call on the device.

Checked through the C ABI against the workspace entry point msa_index_score_topk on the same
inputs, on two calls in a row with different shapes (the second call reuses the array the
first one left behind), with the tolerances of the other parity tests; once more against the
oracle on a prefill chunk (N > 8: the multi-row scorer and top-k, which use the same scratch);
and that a call allocates no device memory. The file is named to be collected last; it also
passes when run on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_msa_gb300 as msa
import oracle
import workloads
from _compare import SCORE_REL, check_selected_scores, check_selection, u16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_sparse_attention_msa_gb300 import build
    build.build()
    msa.load()


def _inputs(seq_lens, N, Hkv, Di, seed):
    w = workloads.index_workload(seq_lens, N, Hkv, Di, seed=seed, device="cpu", n_planted=0)
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in w.items()}


def _same(a, b):
    ids_a, sc_a = (x.cpu().numpy() for x in a)
    ids_b, sc_b = (x.cpu().numpy() for x in b)
    # both entry points run the same kernels on the same inputs: the ids must agree exactly
    assert np.array_equal(ids_a, ids_b)
    np.testing.assert_allclose(sc_a, sc_b, rtol=SCORE_REL, atol=1e-4)


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    cases = [([5000, 129, 3000, 777], 1, 8, 128, 16, 21),    # decode, ragged
             ([7000, 6100, 300], 4, 4, 64, 8, 22)]            # multi-token rows, other shape
    for seq_lens, N, Hkv, Di, k, seed in cases:
        d = _inputs(seq_lens, N, Hkv, Di, seed)
        args = (d["q_idx"], d["k_idx_pages"], d["page_table"], d["seq_lens"], N, k)
        got = msa.index_score_topk_noalloc(*args)
        ref = msa.index_score_topk(*args, workspace=msa.Workspace())
        torch.cuda.synchronize()
        _same(got, ref)
    assert msa.device_error() == 0


def test_noalloc_rejects_calls_beyond_its_scratch():
    # 64 requests x 8 groups x 8192 blocks of scores exceed the 8 MiB scratch
    B, Hkv, Di, mb = 64, 8, 128, 8192
    q_idx = torch.zeros((B, Hkv, Di), dtype=torch.bfloat16, device=DEV)
    k_idx = torch.zeros((1, 128, Hkv, Di), dtype=torch.bfloat16, device=DEV)
    pt = torch.zeros((B, mb), dtype=torch.int32, device=DEV)
    sl = torch.full((B,), 128, dtype=torch.int32, device=DEV)
    with pytest.raises(msa.MSAError, match="scratch"):
        msa.index_score_topk_noalloc(q_idx, k_idx, pt, sl, 1, 16)


def test_noalloc_multi_row_chunk_matches_oracle():
    # N > 8: the tensor-core scorer writes every block score into the scratch, then the top-k
    seq_lens, N, Hkv, Di, k = [2048, 1500], 300, 2, 128, 6
    w = workloads.index_workload(seq_lens, N, Hkv, Di, seed=23, device="cpu")
    d = {k_: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k_, v in w.items()}
    args = (d["q_idx"], d["k_idx_pages"], d["page_table"], d["seq_lens"], N, k)
    for _ in range(2):  # two calls in a row on the shared array
        ids, sc = msa.index_score_topk_noalloc(*args)
        torch.cuda.synchronize()
        s_ref = oracle.block_scores(u16(w["q_idx"]), u16(w["k_idx_pages"]), w["page_table"].numpy(),
                                    w["seq_lens"].numpy(), N)
        ids_ref, _ = oracle.topk(s_ref, oracle.query_positions(w["seq_lens"].numpy(), N), k)
        check_selection(ids.cpu().numpy(), ids_ref, s_ref)
        check_selected_scores(ids.cpu().numpy(), sc.cpu().numpy(), s_ref)
    _same((ids, sc), msa.index_score_topk(*args, workspace=msa.Workspace()))
    assert msa.device_error() == 0


def test_noalloc_call_allocates_no_device_memory():
    seq_lens, N, Hkv, Di, k = [5000, 129, 3000, 777], 1, 8, 128, 16
    d = _inputs(seq_lens, N, Hkv, Di, 24)
    args = (d["q_idx"], d["k_idx_pages"], d["page_table"], d["seq_lens"], N, k)
    R = len(seq_lens) * N
    out = (torch.empty((R, Hkv, k), dtype=torch.int32, device=DEV),
           torch.empty((R, Hkv, k), dtype=torch.float32, device=DEV))
    for _ in range(2):  # the first call on a device resolves the array; modules are loaded
        msa.index_score_topk_noalloc(*args, out=out)
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0 = torch.cuda.mem_get_info()[0]
    msa.index_score_topk_noalloc(*args, out=out)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
