"""Pins of the CPU oracle against facts fixed outside it (CPU only).

Each test checks one oracle routine against something other than itself: hand-derived
values, brute force on tiny inputs, a textbook/library routine (numpy/scipy dense
attention, numpy sorting) or an invariant of the method. The cases are chosen so that a
plausible slip (wrong group or page index, off-by-one mask, dropped tie rule, transposed
operand, wrong merge weight) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float32).numpy()


def bf16_bits(x) -> np.ndarray:
    return u16(torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


# --------------------------------------------------------------------------- bf16 rounding

def test_round_bf16_matches_torch_on_float_values():
    rng = np.random.default_rng(0)
    f32max = float(np.finfo(np.float32).max)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 8, 20000),
                        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-40, -2.5e-39,
                                  # overflow to infinity, the largest finite bf16, specials
                                  f32max, -f32max, 3.3895e38, np.inf, -np.inf])])
    x32 = x.astype(np.float32)
    ref = u16(torch.from_numpy(x32).to(torch.bfloat16))
    got = oracle.round_bf16(x32.astype(np.float64))
    assert np.array_equal(ref, got)
    # NaN stays NaN (all exponent bits, a nonzero fraction); its payload is not fixed
    nan = int(oracle.round_bf16([np.nan])[0])
    assert nan & 0x7F80 == 0x7F80 and nan & 0x007F != 0


def test_round_bf16_single_rounding_and_ties():
    # exact ties round to even
    assert oracle.round_bf16([1.0 + 2.0 ** -8])[0] == 0x3F80          # 1.0 (even)
    assert oracle.round_bf16([1.0 + 3 * 2.0 ** -8])[0] == 0x3F82      # 1 + 2^-6 (even)
    # just above a tie: must round up; a float-first path would land on the tie and go even
    assert oracle.round_bf16([1.0 + 2.0 ** -8 + 2.0 ** -40])[0] == 0x3F81
    assert oracle.round_bf16([-(1.0 + 2.0 ** -8 + 2.0 ** -40)])[0] == 0xBF81


# --------------------------------------------------------------------------- block scores

def _load_hand_scores():
    with open(os.path.join(GOLDEN, "hand_scores.json")) as f:
        fx = json.load(f)
    B, Hkv, Di = fx["B"], fx["Hkv"], fx["Di"]
    pt = np.array(fx["page_table"], dtype=np.int32)
    k_idx = np.zeros((fx["num_pages"], 128, Hkv, Di), dtype=np.float32)
    for b, s, e, g, vec in fx["k_idx_ranges"]:
        for pos in range(s, e):
            k_idx[pt[b, pos // 128], pos % 128, g] = vec
    return fx, bf16_bits(np.array(fx["q_idx"], dtype=np.float32)), bf16_bits(k_idx), pt


def test_block_scores_hand_fixture():
    fx, q_idx, k_idx, pt = _load_hand_scores()
    sl = np.array(fx["seq_lens"], dtype=np.int32)
    s = oracle.block_scores(q_idx, k_idx, pt, sl, N=1)
    assert np.array_equal(s, np.array(fx["expected_scores"], dtype=np.float32))


@pytest.mark.parametrize("k", ["2", "3", "4", "6"])
def test_topk_hand_fixture(k):
    fx, q_idx, k_idx, pt = _load_hand_scores()
    sl = np.array(fx["seq_lens"], dtype=np.int32)
    s = oracle.block_scores(q_idx, k_idx, pt, sl, N=1)
    ids, sel = oracle.topk(s, oracle.query_positions(sl, 1), int(k))
    exp = fx["expected_topk"][k]
    assert np.array_equal(ids, np.array(exp["ids"], dtype=np.int32))
    exp_s = np.array([[[float(v) for v in row] for row in r] for r in exp["scores"]], dtype=np.float32)
    assert np.array_equal(sel, exp_s)


def _dense_block_scores_bruteforce(q_idx, k_idx, pt, seq_lens, N):
    """Brute force: logical K per request, dense Q.K^T in float64, masked max-pool."""
    qf = oracle.bf16_to_f32(q_idx).astype(np.float64)
    kf = oracle.bf16_to_f32(k_idx).astype(np.float64)
    B, max_blocks = pt.shape
    R, Hkv, Di = qf.shape
    out = np.full((R, Hkv, max_blocks), -np.inf)
    for b in range(B):
        keys = kf[pt[b]].reshape(max_blocks * 128, Hkv, Di)  # logical order
        for i in range(N):
            r = b * N + i
            q_pos = seq_lens[b] - N + i
            for g in range(Hkv):
                s = keys[:, g, :] @ qf[r, g]
                s[q_pos + 1:] = -np.inf
                out[r, g] = s.reshape(max_blocks, 128).max(axis=1)
    return out


@pytest.mark.parametrize("seq_lens,N,Hkv,Di", [([517, 300, 128], 1, 2, 64),
                                               ([1000, 777], 3, 4, 128),
                                               ([129, 5], 2, 1, 64)])
def test_block_scores_bruteforce(seq_lens, N, Hkv, Di):
    w = workloads.index_workload(seq_lens, N, Hkv, Di, seed=11, device="cpu")
    q_idx, k_idx = u16(w["q_idx"]), u16(w["k_idx_pages"])
    pt, sl = w["page_table"].numpy(), w["seq_lens"].numpy()
    got = oracle.block_scores(q_idx, k_idx, pt, sl, N=N)
    ref = _dense_block_scores_bruteforce(q_idx, k_idx, pt, sl, N)
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    fin = np.isfinite(ref)
    np.testing.assert_allclose(got[fin], ref[fin], rtol=1e-5, atol=1e-4)
    # row subset returns the same rows
    rows = np.array([N * len(seq_lens) - 1, 0], dtype=np.int64)
    sub = oracle.block_scores(q_idx, k_idx, pt, sl, N=N, rows=rows)
    assert np.array_equal(sub, got[rows])


def test_planted_blocks_are_selected():
    # decode_scoring structure at reduced size: planted blocks gain ~2|q|^2 ~ 256 over noise ~ 11
    w = workloads.index_workload([60 * 128, 50 * 128 + 17], 1, 2, 128, seed=5, device="cpu",
                                 n_planted=8)
    sl = w["seq_lens"].numpy()
    s = oracle.block_scores(u16(w["q_idx"]), u16(w["k_idx_pages"]), w["page_table"].numpy(), sl, 1)
    ids, _ = oracle.topk(s, oracle.query_positions(sl, 1), 16)
    planted = w["planted"].numpy()
    for b in range(2):
        for g in range(2):
            assert set(planted[b, g].tolist()) <= set(ids[b, g].tolist())


# --------------------------------------------------------------------------- top-k

def _topk_bruteforce(scores_row, q_pos, k):
    """Enumerate every subset of the non-forced causal blocks; keep the max-sum ones and
    break ties by the lexicographically smallest sorted id tuple."""
    local = q_pos // 128
    forced = [0] if local == 0 else [0, local]
    cands = list(range(1, local))
    m = min(k - len(forced), len(cands))
    best = None
    for sub in itertools.combinations(cands, m):
        key = (-sum(scores_row[j] for j in sub), sub)
        if best is None or key < best:
            best = key
    kept = sorted(forced + list(best[1] if best else ()))
    return kept + [-1] * (k - len(kept))


def test_topk_bruteforce_with_ties():
    rng = np.random.default_rng(3)
    for trial in range(60):
        nblk = int(rng.integers(1, 11))
        q_pos = int(rng.integers((nblk - 1) * 128, nblk * 128))
        scores = rng.integers(-3, 4, size=(1, 1, nblk)).astype(np.float32)  # many ties
        for k in range(2, nblk + 3):
            ids, sel = oracle.topk(scores, np.array([q_pos]), k)
            exp = _topk_bruteforce(scores[0, 0], q_pos, k)
            assert ids[0, 0].tolist() == exp, (scores, q_pos, k)
            for i, j in enumerate(exp):
                assert sel[0, 0, i] == (scores[0, 0, j] if j >= 0 else -np.inf)


def test_topk_dominance_property_random():
    rng = np.random.default_rng(4)
    R, Hkv, nb, k = 40, 3, 200, 16
    scores = rng.standard_normal((R, Hkv, nb)).astype(np.float32)
    q_pos = rng.integers(0, nb * 128, size=R)
    ids, _ = oracle.topk(scores, q_pos, k)
    for r in range(R):
        local = q_pos[r] // 128
        for g in range(Hkv):
            row = ids[r, g]
            kept = [int(j) for j in row if j >= 0]
            assert kept == sorted(kept) and len(kept) == min(k, local + 1)
            assert 0 in kept and local in kept
            assert all(j == -1 for j in row[len(kept):])
            rest = [j for j in range(1, local) if j not in kept]
            chosen = [j for j in kept if 0 < j < local]
            if chosen and rest:
                assert min(scores[r, g, chosen]) >= max(scores[r, g, rest])


# --------------------------------------------------------------------------- page tables

def test_page_table_hand_fixtures():
    with open(os.path.join(GOLDEN, "hand_page_table.json")) as f:
        fx = json.load(f)
    fpt, lens = oracle.build_sparse_page_table(np.array(fx["block_ids"]), np.array(fx["page_table"]),
                                               np.array(fx["seq_lens"]), fx["N"])
    assert fpt.tolist() == fx["expected_flat_page_table"]
    assert lens.tolist() == fx["expected_flat_kv_lens"]
    hs = json.load(open(os.path.join(GOLDEN, "hand_scores.json")))
    ids = np.array(hs["expected_topk"]["3"]["ids"])
    fpt, lens = oracle.build_sparse_page_table(ids, np.array(hs["page_table"]), np.array(hs["seq_lens"]), 1)
    assert fpt.tolist() == hs["expected_page_table_k3"]["flat_page_table"]
    assert lens.tolist() == hs["expected_page_table_k3"]["flat_kv_lens"]


@pytest.mark.parametrize("N", [1, 3])
def test_strided_view_reproduces_logical_kv(N):
    w = workloads.decode_workload([517, 1500, 129], N, Hq=8, Hkv=4, D=16, topk=5, seed=7,
                                  device="cpu")
    k_cache = u16(w["k_cache"])
    pt, sl, ids = w["page_table"].numpy(), w["seq_lens"].numpy(), w["block_ids"].numpy()
    fpt, lens = oracle.build_sparse_page_table(ids, pt, sl, N)
    Hkv, D = 4, 16
    flat = k_cache.reshape(-1)
    for r in range(ids.shape[0]):
        b = r // N
        q_pos = sl[b] - N + r % N
        for g in range(Hkv):
            f = r * Hkv + g
            logical = []  # (page, tau) of every visible key, ascending position
            for j in ids[r, g]:
                if j < 0:
                    continue
                for tau in range(128):
                    if j * 128 + tau > q_pos:
                        break
                    logical.append(k_cache[pt[b, j], tau, g])
            assert lens[f] == len(logical)
            seen_pages = set()
            for n in range(lens[f]):
                v = int(fpt[f, n // 128])
                seen_pages.add(v)
                off = v * D + (n % 128) * Hkv * D
                assert np.array_equal(flat[off:off + D], logical[n])
            assert len(seen_pages) == int(np.count_nonzero(ids[r, g] >= 0))


# --------------------------------------------------------------------------- attention

def _dense_attention(qv, keys, vals):
    s = keys @ qv
    lse = logsumexp(s)
    return np.exp(s - lse) @ vals, lse


@pytest.mark.parametrize("N", [1, 2])
def test_decode_full_selection_equals_dense_causal(N):
    # k >= number of causal blocks: MSA decode is dense causal attention
    seq_lens = [300, 513, 40]
    Hq, Hkv, D = 8, 2, 32
    w = workloads.decode_workload(seq_lens, N, Hq, Hkv, D, topk=6, seed=9, device="cpu")
    q, kc, vc = u16(w["q"]), u16(w["k_cache"]), u16(w["v_cache"])
    pt, sl, ids = w["page_table"].numpy(), w["seq_lens"].numpy(), w["block_ids"].numpy()
    res = oracle.sparse_decode(q, kc, vc, pt, sl, ids, N)
    fpt, lens = oracle.build_sparse_page_table(ids, pt, sl, N)
    res_flat = oracle.paged_decode_flat(q, kc, vc, fpt, lens)
    assert np.array_equal(res["o"], res_flat["o"]) and np.array_equal(res["lse"], res_flat["lse"])
    qf, kf, vf = (oracle.bf16_to_f32(x).astype(np.float64) for x in (q, kc, vc))
    G = Hq // Hkv
    for r in range(len(seq_lens) * N):
        b = r // N
        q_pos = sl[b] - N + r % N
        for h in range(Hq):
            g = h // G
            keys = kf[pt[b]].reshape(-1, Hkv, D)[: q_pos + 1, g]
            vals = vf[pt[b]].reshape(-1, Hkv, D)[: q_pos + 1, g]
            o, lse = _dense_attention(qf[r, h], keys, vals)
            u = r * Hq + h
            np.testing.assert_allclose(res["o"][u], o, rtol=1e-10, atol=1e-12)
            assert abs(res["lse"][u] - lse) < 1e-10


@pytest.mark.parametrize("N", [1, 2])
def test_decode_sparse_equals_masked_dense(N):
    # k below the causal block count, selections drawn per KV group: each head attends to
    # the causal keys of its own group's kept blocks only (masked dense attention, scipy)
    seq_lens = [700, 1030, 129]
    Hq, Hkv, D, k = 8, 4, 32, 3
    w = workloads.decode_workload(seq_lens, N, Hq, Hkv, D, topk=k, seed=13, device="cpu")
    q, kc, vc = u16(w["q"]), u16(w["k_cache"]), u16(w["v_cache"])
    pt, sl, ids = w["page_table"].numpy(), w["seq_lens"].numpy(), w["block_ids"].numpy()
    # the groups of one row keep different blocks (else a group mix-up goes unseen)
    assert any(not np.array_equal(ids[r, 0], ids[r, g]) for r in range(ids.shape[0])
               for g in range(1, Hkv))
    qf, kf, vf = (oracle.bf16_to_f32(x).astype(np.float64) for x in (q, kc, vc))
    G = Hq // Hkv
    R = len(seq_lens) * N

    def masked_dense(u):
        r, h = divmod(int(u), Hq)
        b, g = r // N, h // G
        q_pos = sl[b] - N + r % N
        pos = np.arange(sl[b])
        keys = kf[pt[b]].reshape(-1, Hkv, D)[: sl[b], g]
        vals = vf[pt[b]].reshape(-1, Hkv, D)[: sl[b], g]
        sel = np.isin(pos // 128, ids[r, g][ids[r, g] >= 0]) & (pos <= q_pos)
        s = np.where(sel, keys @ qf[r, h], -np.inf)
        lse = logsumexp(s)
        return np.exp(s - lse) @ vals, lse

    res = oracle.sparse_decode(q, kc, vc, pt, sl, ids, N)
    for u in range(R * Hq):
        o, lse = masked_dense(u)
        np.testing.assert_allclose(res["o"][u], o, rtol=1e-10, atol=1e-12)
        assert abs(res["lse"][u] - lse) < 1e-10
    # a shuffled list of units (the sampled form the full-size tests use), logical and through
    # the strided view: slot i holds unit units[i]
    units = np.random.default_rng(N).permutation(R * Hq)[: R * Hq // 3].astype(np.int64)
    fpt, lens = oracle.build_sparse_page_table(ids, pt, sl, N)
    for sub in (oracle.sparse_decode(q, kc, vc, pt, sl, ids, N, units=units),
                oracle.paged_decode_flat(q, kc, vc, fpt, lens, units=units)):
        for i, u in enumerate(units):
            o, lse = masked_dense(u)
            np.testing.assert_allclose(sub["o"][i], o, rtol=1e-10, atol=1e-12)
            assert abs(sub["lse"][i] - lse) < 1e-10


def test_prefill_sparse_equals_masked_dense():
    T, S, Hq, Hkv, D, k = 300, 700, 4, 2, 32, 4
    w = workloads.prefill_workload(T, S, Hq, Hkv, D, k, seed=1, device="cpu", n_shared=2)
    q, kk, vv, ids = u16(w["q"]), u16(w["k"]), u16(w["v"]), w["block_ids"].numpy()
    res = oracle.sparse_prefill(q, kk, vv, ids)
    qf, kf, vf = (oracle.bf16_to_f32(x).astype(np.float64) for x in (q, kk, vv))
    pos = np.arange(S)
    for t in range(T):
        q_pos = S - T + t
        for h in range(Hq):
            g = h // (Hq // Hkv)
            sel = np.isin(pos // 128, ids[t, g][ids[t, g] >= 0]) & (pos <= q_pos)
            s = np.where(sel, kf[:, g] @ qf[t, h], -np.inf)
            lse = logsumexp(s)
            o = np.exp(s - lse) @ vf[:, g]
            u = t * Hq + h
            np.testing.assert_allclose(res["o"][u], o, rtol=1e-10, atol=1e-12)
            assert abs(res["lse"][u] - lse) < 1e-10
    # bf16 output is the single rounding of the fp64 result
    assert np.array_equal(res["o_bf16"], oracle.round_bf16(res["o"]))


def test_prefill_full_selection_equals_dense_causal_and_units():
    T, Hq, Hkv, D = 260, 4, 2, 16
    w = workloads.prefill_workload(T, T, Hq, Hkv, D, topk=3, seed=2, device="cpu", n_shared=0)
    q, kk, vv, ids = u16(w["q"]), u16(w["k"]), u16(w["v"]), w["block_ids"].numpy()
    res = oracle.sparse_prefill(q, kk, vv, ids)
    qf, kf, vf = (oracle.bf16_to_f32(x).astype(np.float64) for x in (q, kk, vv))
    for t in (0, 1, 127, 128, 200, 259):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            o, lse = _dense_attention(qf[t, h], kf[: t + 1, g], vf[: t + 1, g])
            np.testing.assert_allclose(res["o"][t * Hq + h], o, rtol=1e-10, atol=1e-12)
    units = np.array([5, T * Hq - 1, 0], dtype=np.int64)
    sub = oracle.sparse_prefill(q, kk, vv, ids, units=units)
    assert np.array_equal(sub["o"], res["o"][units])


def test_attention_closed_form_uniform_block():
    # identical keys -> uniform weights: o = mean(v), lse = s + log(n)
    T, S, D = 1, 200, 8
    q = np.zeros((T, 1, D), dtype=np.float32); q[0, 0, 0] = 0.5
    k = np.zeros((S, 1, D), dtype=np.float32); k[:, 0, 0] = 2.0
    v = np.arange(S * D, dtype=np.float32).reshape(S, 1, D) / 64.0
    ids = np.array([[[0, 1]]], dtype=np.int32)
    res = oracle.sparse_prefill(bf16_bits(q), bf16_bits(k), bf16_bits(v), ids)
    vv = oracle.bf16_to_f32(bf16_bits(v)).astype(np.float64)[:, 0]
    np.testing.assert_allclose(res["o"][0], vv.mean(axis=0), rtol=1e-12)
    assert abs(res["lse"][0] - (1.0 + math.log(S))) < 1e-12


# --------------------------------------------------------------------------- LSE merge

def test_lse_merge_of_block_partials_equals_single_softmax():
    T, S, Hq, Hkv, D = 200, 600, 4, 2, 32
    w = workloads.prefill_workload(T, S, Hq, Hkv, D, topk=4, seed=8, device="cpu", n_shared=2)
    q, kk, vv, ids = u16(w["q"]), u16(w["k"]), u16(w["v"]), w["block_ids"].numpy()
    full = oracle.sparse_prefill(q, kk, vv, ids)
    for t, h in [(0, 0), (57, 3), (199, 1), (130, 2)]:
        g = h // (Hq // Hkv)
        parts = [oracle.prefill_block_partial(q, kk, vv, t, h, int(j)) for j in ids[t, g] if j >= 0]
        o_p = np.stack([p[0] for p in parts]).astype(np.float32)
        l_p = np.array([p[1] for p in parts], dtype=np.float32)
        o, lse = oracle.lse_merge(o_p, l_p)
        u = t * Hq + h
        np.testing.assert_allclose(o, full["o"][u], rtol=1e-5, atol=1e-6)
        assert abs(lse - full["lse"][u]) < 1e-5


def test_lse_merge_closed_forms():
    o1 = np.array([[1.0, -2.0, 0.5]], dtype=np.float32)
    o, lse = oracle.lse_merge(o1, np.array([0.75], dtype=np.float32))
    assert np.array_equal(o, o1[0].astype(np.float64)) and lse == 0.75
    o2 = np.array([[1.0, 0.0], [0.0, 1.0]], dtype=np.float32)
    o, lse = oracle.lse_merge(o2, np.array([0.0, math.log(3.0)], dtype=np.float32))
    np.testing.assert_allclose(o, [0.25, 0.75], rtol=1e-7)
    assert abs(lse - np.logaddexp(0.0, np.float32(math.log(3.0)))) < 1e-12
    o, lse = oracle.lse_merge(o2, np.array([-np.inf, 2.0], dtype=np.float32))
    np.testing.assert_array_equal(o, [0.0, 1.0])
    o, lse = oracle.lse_merge(o2[:0], np.zeros(0, dtype=np.float32))
    assert lse == -np.inf and not o.any()
    # no partial with a visible key: a unit that sees nothing gives o = 0, lse = -inf
    o, lse = oracle.lse_merge(o2, np.array([-np.inf, -np.inf], dtype=np.float32))
    assert lse == -np.inf and not o.any()


def test_block_partial_of_a_block_after_the_query_is_empty():
    # a block whose first key lies after the query has no visible key: weight 0 (lse -inf),
    # o = 0, and merging it in changes nothing
    T, S, Hq, Hkv, D = 130, 400, 2, 1, 8
    w = workloads.prefill_workload(T, S, Hq, Hkv, D, topk=2, seed=3, device="cpu", n_shared=0)
    q, kk, vv = u16(w["q"]), u16(w["k"]), u16(w["v"])
    t = 0                                   # position S - T = 270: local block 2
    o3, lse3 = oracle.prefill_block_partial(q, kk, vv, t, 1, 3)
    assert lse3 == -np.inf and not np.any(o3)
    o2, lse2 = oracle.prefill_block_partial(q, kk, vv, t, 1, 2)
    o0, lse0 = oracle.prefill_block_partial(q, kk, vv, t, 1, 0)
    parts = np.stack([o0, o2]).astype(np.float32)
    with_empty = np.stack([o0, o2, o3]).astype(np.float32)
    a = oracle.lse_merge(parts, np.array([lse0, lse2], dtype=np.float32))
    b = oracle.lse_merge(with_empty, np.array([lse0, lse2, lse3], dtype=np.float32))
    assert np.array_equal(a[0], b[0]) and a[1] == b[1]


# --------------------------------------------------------------------------- bucketing

def test_prefill_buckets_invert_selection():
    w = workloads.prefill_workload(500, 900, 2, 2, 8, topk=5, seed=6, device="cpu", n_shared=2)
    ids = w["block_ids"].numpy()
    nblk = (900 + 127) // 128
    offsets, entries = oracle.prefill_buckets(ids, nblk)
    T, Hkv, k = ids.shape
    base = 0
    for g in range(Hkv):
        flat = ids[:, g, :].reshape(-1)  # index t*k + i
        valid = np.nonzero(flat >= 0)[0]
        order = valid[np.lexsort((valid, flat[valid]))]  # by block, then by (t, i)
        counts = np.bincount(flat[valid], minlength=nblk)
        assert np.array_equal(offsets[g], np.concatenate([[0], np.cumsum(counts)]))
        assert np.array_equal(entries[base:base + offsets[g, -1]], order)
        base += offsets[g, -1]
    assert base == entries.size
