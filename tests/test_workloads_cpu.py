"""The seeded selection generator (CPU): what it draws has the structure of MSA's top-k.

``workloads.sample_selection`` draws block selections without computing a block score. Its
draws must still be outcomes of the top-k rule: for every (row, group), the oracle's top-k
over scores that put 1 on the drawn non-forced blocks and 0 on the other candidates must
return exactly the drawn list (sink and local block forced, ids ascending, -1 padding only
when the query has fewer causal blocks than k). Boosted rows must keep their shared blocks,
and the free picks must be uniform over the candidates.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads


def _indicator_scores(ids: np.ndarray, q_pos: np.ndarray) -> np.ndarray:
    R, H, _ = ids.shape
    nblk = int(q_pos.max()) // 128 + 1
    s = np.zeros((R, H, nblk), dtype=np.float32)
    for r in range(R):
        for g in range(H):
            for j in ids[r, g]:
                if j >= 0:
                    s[r, g, j] = 1.0
    return s


@pytest.mark.parametrize("topk", [2, 3, 5, 16])
def test_draws_are_top_k_outcomes(topk):
    # positions in the first block, on block edges and ragged, up to 40 blocks
    q_pos = torch.tensor([0, 5, 127, 128, 255, 256, 300, 1000, 2047, 2048, 4000, 5119],
                         dtype=torch.int64)
    gen = workloads._gen(17 + topk, "cpu")
    ids = workloads.sample_selection(q_pos, 3, topk, gen).numpy()
    assert ids.shape == (q_pos.numel(), 3, topk) and ids.dtype == np.int32
    qp = q_pos.numpy()
    ref, _ = oracle.topk(_indicator_scores(ids, qp), qp, topk)
    assert np.array_equal(ids, ref)
    # the number of kept blocks: every causal block when there are at most k of them
    kept = (ids >= 0).sum(axis=2)
    assert np.array_equal(kept, np.minimum(topk, qp // 128 + 1)[:, None].repeat(3, axis=1))


def test_boosted_rows_keep_their_shared_blocks():
    R, H, topk = 64, 2, 8
    q_pos = torch.full((R,), 40 * 128 + 3, dtype=torch.int64)      # local block 40
    gen = workloads._gen(5, "cpu")
    shared = torch.full((R, H, 4), -1, dtype=torch.int64)
    shared[:, 0, :3] = torch.tensor([7, 19, 33])                     # group 0: three blocks
    shared[:, 1, :4] = torch.tensor([2, 3, 38, 39])                  # group 1: four blocks
    boosted = torch.zeros((R, H), dtype=torch.bool)
    boosted[::2] = True
    ids = workloads.sample_selection(q_pos, H, topk, gen, shared=shared, boosted=boosted).numpy()
    for r in range(R):
        for g in range(H):
            want = set(int(x) for x in shared[r, g] if x >= 0)
            if boosted[r, g]:
                assert want <= set(ids[r, g].tolist()), (r, g, ids[r, g])
    # unboosted rows are free draws: they miss at least one shared block somewhere
    free = [set(int(x) for x in shared[r, 0] if x >= 0) <= set(ids[r, 0].tolist())
            for r in range(1, R, 2)]
    assert not all(free)


def test_free_picks_are_uniform_over_the_candidates():
    # local block 11: candidates 1..10, k 5 keeps sink + local + 3 of the 10
    R = 20000
    q_pos = torch.full((R,), 11 * 128 + 64, dtype=torch.int64)
    ids = workloads.sample_selection(q_pos, 1, 5, workloads._gen(9, "cpu")).numpy()[:, 0]
    counts = np.bincount(ids[(ids > 0) & (ids < 11)], minlength=11)[1:11]
    expect = R * 3 / 10
    # binomial sd = sqrt(R * 0.3 * 0.7) ~ 65; allow 5 sd
    assert np.all(np.abs(counts - expect) < 5 * np.sqrt(R * 0.3 * 0.7)), counts
