"""Comparison helpers for parity tests: tolerances, near-tie rule, tensor conversions."""
import numpy as np
import torch

# Attention outputs in bf16: max-abs / mean-abs against the oracle; LSE absolute.
O_MAX_ABS = 2e-2
O_MEAN_ABS = 5e-3
LSE_ABS = 1e-3
# Block scores: relative; a selection swap is a match when the oracle scores of the
# swapped blocks differ by less than this (relative).
SCORE_REL = 1e-3


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float32).numpy()


def check_attention(o_gpu: torch.Tensor, lse_gpu, ref: dict, units=None, what=""):
    """o_gpu [..., D] bf16 vs ref['o'] (fp64 rows, one per unit); lse likewise."""
    D = o_gpu.shape[-1]
    o = f32(o_gpu).reshape(-1, D)
    if units is not None:
        o = o[units]
    err = np.abs(o - ref["o"])
    assert err.max() <= O_MAX_ABS, f"{what}: o max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: o mean-abs {err.mean():.3e}"
    if lse_gpu is not None:
        lse = f32(lse_gpu).reshape(-1)
        if units is not None:
            lse = lse[units]
        fin = np.isfinite(ref["lse"])
        assert np.array_equal(np.isfinite(lse), fin), f"{what}: lse finiteness differs"
        d = np.abs(lse[fin] - ref["lse"][fin])
        assert d.size == 0 or d.max() <= LSE_ABS, f"{what}: lse abs {d.max():.3e}"
    return err.max(), err.mean()


def check_selection(ids_gpu: np.ndarray, ids_ref: np.ndarray, scores_ref: np.ndarray):
    """Bit-exact block ids, except near-tie swaps decided on the oracle's block scores.

    ids_* [R, Hkv, k]; scores_ref [R, Hkv, max_blocks] (oracle block scores).
    Returns the number of (row, group) lists that differ only by near-tie swaps.
    """
    assert ids_gpu.shape == ids_ref.shape
    # The sink block 0 and the query's local block are always kept. The local block is the
    # last block with a finite oracle score: blocks past the query's position score -inf, and
    # the local block holds at least the query's own token. A dropped forced block must fail
    # here, before the near-tie rule below could excuse it.
    fin = np.isfinite(scores_ref)
    R, H = ids_gpu.shape[:2]
    local = fin.shape[2] - 1 - np.argmax(fin[:, :, ::-1], axis=2)      # [R, Hkv]
    has_any = fin.any(axis=2)
    for forced, what in ((np.zeros((R, H), dtype=np.int64), "sink block 0"), (local, "local block")):
        kept = (ids_gpu == forced[:, :, None]).any(axis=2)
        bad = np.nonzero(has_any & ~kept)
        assert bad[0].size == 0, (
            f"{what} missing in row {bad[0][0]} group {bad[1][0]}: {ids_gpu[bad[0][0], bad[1][0]]}")
    swaps = 0
    diff = np.nonzero((ids_gpu != ids_ref).any(axis=2))
    for r, g in zip(*diff):
        a = set(int(x) for x in ids_gpu[r, g] if x >= 0)
        b = set(int(x) for x in ids_ref[r, g] if x >= 0)
        assert len(a) == len(b), f"row {r} group {g}: {sorted(a)} vs {sorted(b)}"
        # distinct ids ascending, then -1 padding: the layout of every selection list
        row = [int(x) for x in ids_gpu[r, g]]
        assert row == sorted(a) + [-1] * (len(row) - len(a)), (
            f"row {r} group {g}: {row} is not distinct ascending ids followed by -1 padding")
        s = scores_ref[r, g]
        for x in a - b:
            for y in b - a:
                tol = SCORE_REL * max(abs(s[x]), abs(s[y]), 1e-30)
                assert s[y] - s[x] <= tol, (
                    f"row {r} group {g}: chose block {x} ({s[x]}) over {y} ({s[y]})")
        swaps += 1
    return swaps


def check_selected_scores(ids_gpu: np.ndarray, sc_gpu: np.ndarray, scores_ref: np.ndarray):
    """GPU scores of the kept blocks vs the oracle's score of the same block (relative)."""
    R, H, k = ids_gpu.shape
    valid = ids_gpu >= 0
    rr, gg, ii = np.nonzero(valid)
    ref = scores_ref[rr, gg, ids_gpu[rr, gg, ii]]
    got = sc_gpu[rr, gg, ii]
    np.testing.assert_allclose(got, ref, rtol=SCORE_REL, atol=1e-4)
    assert np.all(np.isneginf(sc_gpu[~valid]))
