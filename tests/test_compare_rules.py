"""The parity comparators themselves (CPU): the selection rule must reject a GPU selection
that drops a forced block (sink block 0, the query's local block) even when the block kept in
its place scores higher, or that breaks the list layout (ids ascending, then -1 padding), and
accept a near-tie swap of two non-forced blocks; the attention tolerances must pass the exact
result rounded to bf16 and reject a slip confined to one (query, head) unit."""
import numpy as np
import pytest
import torch

from _compare import check_attention, check_selection


def _case():
    # one row, one group, 6 blocks: 4 causal (local block 3), k 3
    s = np.full((1, 1, 6), -np.inf)
    s[0, 0, :4] = [1.0, 5.0, 5.0, 0.5]
    ids_ref = np.array([[[0, 1, 3]]], dtype=np.int32)
    return s, ids_ref


def test_same_selection_passes():
    s, ids_ref = _case()
    assert check_selection(ids_ref.copy(), ids_ref, s) == 0


def test_near_tie_swap_passes():
    s, ids_ref = _case()
    # blocks 1 and 2 tie exactly: keeping 2 instead of 1 is a near-tie swap
    assert check_selection(np.array([[[0, 2, 3]]], dtype=np.int32), ids_ref, s) == 1


@pytest.mark.parametrize("gpu,what", [([0, 1, 2], "local block"), ([1, 2, 3], "sink block 0")])
def test_dropped_forced_block_fails(gpu, what):
    s, ids_ref = _case()
    with pytest.raises(AssertionError, match=what):
        check_selection(np.array([gpu], dtype=np.int32)[None], ids_ref, s)


def test_clear_loss_fails():
    s, ids_ref = _case()
    s[0, 0, 2] = 4.0  # block 2 now clearly below block 1
    with pytest.raises(AssertionError, match="chose block 2"):
        check_selection(np.array([[[0, 2, 3]]], dtype=np.int32), ids_ref, s)


def _padded_case():
    # one row, one group, 3 causal blocks (local block 2) and k 4: one slot of padding
    s = np.full((1, 1, 6), -np.inf)
    s[0, 0, :3] = [1.0, 2.0, 0.5]
    return s, np.array([[[0, 1, 2, -1]]], dtype=np.int32)


@pytest.mark.parametrize("gpu", [[0, -1, 1, 2],    # padding inside the list
                                 [0, 1, 2, -2],    # padding other than -1
                                 [0, 2, 1, -1],    # ids not ascending
                                 [0, 1, 1, 2]])    # a repeated id in place of the padding
def test_broken_list_layout_fails(gpu):
    s, ids_ref = _padded_case()
    with pytest.raises(AssertionError):
        check_selection(np.array([gpu], dtype=np.int32)[None], ids_ref, s)


# --------------------------------------------------------------------------- attention tolerance

def _attention_case():
    import oracle
    import workloads
    T, S, Hq, Hkv, D, k = 64, 300, 4, 2, 128, 2
    w = workloads.prefill_workload(T, S, Hq, Hkv, D, k, seed=12, device="cpu", n_shared=1)
    u16 = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    q, kk, vv = u16(w["q"]), u16(w["k"]), u16(w["v"])
    ids = w["block_ids"].numpy()
    ref = oracle.sparse_prefill(q, kk, vv, ids)
    f = lambda x: oracle.bf16_to_f32(x).astype(np.float64)
    return dict(T=T, S=S, Hq=Hq, Hkv=Hkv, D=D, ids=ids, ref=ref, q=f(q), k=f(kk), v=f(vv))


def _attend(c, t, h, keep):
    """Attention of unit (t, h) over the key positions where keep[pos] holds, fp64."""
    g = h // (c["Hq"] // c["Hkv"])
    s = np.where(keep, c["k"][:, g] @ c["q"][t, h], -np.inf)
    lse = np.logaddexp.reduce(s)
    return np.exp(s - lse) @ c["v"][:, g], lse


def _visible(c, t, g, ids=None):
    pos = np.arange(c["S"])
    q_pos = c["S"] - c["T"] + t
    row = c["ids"][t, g] if ids is None else ids
    return np.isin(pos // 128, row[row >= 0]) & (pos <= q_pos)


def _gpu_like(c, o_rows, lse_rows):
    T, Hq, D = c["T"], c["Hq"], c["D"]
    o = torch.from_numpy(o_rows.reshape(T, Hq, D).astype(np.float32)).to(torch.bfloat16)
    return o, torch.from_numpy(lse_rows.reshape(T, Hq).astype(np.float32))


def test_exact_result_in_bf16_passes():
    c = _attention_case()
    check_attention(*_gpu_like(c, c["ref"]["o"], c["ref"]["lse"]), c["ref"])


@pytest.mark.parametrize("slip", ["dropped block", "one future key", "other group's keys",
                                  "unnormalised row"])
def test_single_unit_slips_fail(slip):
    from _compare import check_attention as check
    c = _attention_case()
    t, h = c["T"] - 10, 1                      # a query inside the last block, head 1 (group 0)
    g = h // (c["Hq"] // c["Hkv"])
    q_pos = c["S"] - c["T"] + t
    keep = _visible(c, t, g)
    if slip == "dropped block":                # the unit loses its non-local block
        row = c["ids"][t, g]
        keep = _visible(c, t, g, ids=row[row == q_pos // 128])
        o, lse = _attend(c, t, h, keep)
    elif slip == "one future key":             # causal mask off by one in the local block
        keep = keep.copy()
        keep[q_pos + 1] = True
        o, lse = _attend(c, t, h, keep)
    elif slip == "other group's keys":         # K/V of group 1 for a head of group 0
        o, lse = _attend(c, t, h + c["Hq"] // c["Hkv"], keep)
    else:                                      # o left as sum p v (no division by l)
        o, lse = _attend(c, t, h, keep)
        o = o * np.exp(lse - np.max(np.where(keep, c["k"][:, g] @ c["q"][t, h], -np.inf)))
    o_rows, lse_rows = c["ref"]["o"].copy(), c["ref"]["lse"].copy()
    u = t * c["Hq"] + h
    o_rows[u], lse_rows[u] = o, lse
    with pytest.raises(AssertionError):
        check(*_gpu_like(c, o_rows, lse_rows), c["ref"])
