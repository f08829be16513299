"""Host logic of bench.py (no GPU): the prefill FLOP split it reports, the traffic records it
reads, the clock-sample summary and the whole-job throughput."""
import json
import os

import numpy as np
import torch

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _selection(T, prefix, Hkv, k, seed):
    """Seeded causal selections: each (query, group) keeps its local block, block 0 and k-2
    other causal blocks, the span's first few blocks chosen far more often (so that pairs
    share blocks); -1 pads rows with fewer causal blocks than k."""
    rng = np.random.default_rng(seed)
    ids = np.full((T, Hkv, k), -1, dtype=np.int32)
    for t in range(T):
        local = (prefix + t) // 128
        for g in range(Hkv):
            cand = list(range(1, local))
            chosen = {0, local}
            common = [b for b in cand if b % 3 == 0][: k]
            rng.shuffle(common)
            for b in common + list(rng.permutation(cand)):
                if len(chosen) >= k:
                    break
                chosen.add(int(b))
            row = sorted(chosen)[:k]
            ids[t, g, : len(row)] = row
    return ids


def _split_by_loops(ids, S_kv, G, D):
    """The query-major selection rule written out with plain loops."""
    T, Hkv, k = ids.shape
    q0 = S_kv - T
    nq = 2 * (128 // G)
    thr = max(2, (nq + 1) // 2)

    def vis(t, j):
        local = (q0 + t) // 128
        if j < 0 or j > local:
            return 0
        return 128 if j < local else (q0 + t) % 128 + 1

    total = sum(4 * D * G * vis(t, int(j)) for t in range(T) for g in range(Hkv) for j in ids[t, g])
    qm = 0
    for g in range(Hkv):
        for s0 in range(0, T, 128):
            qs = list(range(s0, min(T, s0 + 128)))
            cnt = {}
            for t in qs:
                for j in ids[t, g]:
                    if j >= 0:
                        cnt[int(j)] = cnt.get(int(j), 0) + 1
            popular = {j for j, c in cnt.items() if 2 * c >= len(qs)}
            score = {t: sum(1 for j in ids[t, g] if j >= 0 and int(j) in popular) for t in qs}
            order = sorted(qs, key=lambda t: (-score[t], t))          # stable, descending
            for p0 in range(0, len(order), nq):
                pair = order[p0:p0 + nq]
                pc = {}
                for t in pair:
                    for j in ids[t, g]:
                        if j >= 0:
                            pc[int(j)] = pc.get(int(j), 0) + 1
                dense = sorted(j for j, c in pc.items() if c >= thr)[:64]
                for t in pair:
                    for j in ids[t, g]:
                        if int(j) in dense:
                            qm += 4 * D * G * vis(t, int(j))
    return total, qm


def test_prefill_split_matches_the_rule_written_out():
    T, prefix, Hkv, k, G, D = 300, 2048, 2, 8, 8, 128
    ids = _selection(T, prefix, Hkv, k, seed=4)
    got = bench.prefill_split(torch.from_numpy(ids), prefix + T, G, D)
    total, qm = _split_by_loops(ids, prefix + T, G, D)
    assert got["flops_total"] == total
    assert got["flops_query_major"] == qm
    assert got["flops_block_major"] == total - qm
    assert 0 < qm < total  # the seeded spans share blocks, and keep private ones
    # each (pair, block) item runs S and O for both 128-row tiles
    assert got["flops_query_major_executed"] == got["query_major_items"] * 8 * 128 ** 3


def test_prefill_split_without_the_query_major_pass():
    ids = _selection(130, 0, 2, 4, seed=5)
    got = bench.prefill_split(torch.from_numpy(ids), 130, 4, 128)  # G 4: block-major only
    assert got["flops_query_major"] == 0 and got["query_major_items"] == 0
    assert got["flops_block_major"] == got["flops_total"] == _split_by_loops(ids, 130, 4, 128)[0]


def test_recorded_traffic_needs_the_profiled_source():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    assert rec, "no traffic records"
    for kernel, r in rec.items():
        assert bench.recorded_traffic(kernel, r["source_hash"]) == r["bytes_per_launch"]
        assert bench.recorded_traffic(kernel, "0" * 16) is None
    assert bench.recorded_traffic("no_such_kernel", "0" * 16) is None


def test_prefill_traffic_is_the_sum_over_the_calls_kernels():
    got = bench.prefill_traffic()
    parts = [bench.recorded_traffic(k, bench.src_hash(*srcs)) for k, srcs in bench.PREFILL_KERNELS]
    if any(p is None for p in parts):
        assert got is None
    else:
        assert got == sum(parts)


def test_clock_summary():
    c = bench.ClockSampler(0)
    c.out = ("0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n"
             "0, 1965, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active\n"
             "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
             "garbage line\n")
    s = c.summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    empty = bench.ClockSampler(0)
    assert empty.summary()["reasons"] == ["unsampled"]


def test_job_throughput_counts_every_rank():
    assert bench.job_throughput(1e9, 2.0, 1) == 5e11
    assert bench.job_throughput(1e9, 2.0, 4) == 2e12


def test_visible_keys_equal_the_oracle_page_table_lengths():
    # the oracle's sparse page table counts, per flattened row, the tokens its query sees in
    # the kept blocks: the same quantity the bench turns into bytes and FLOPs
    import oracle
    import workloads
    N = 2
    w = workloads.decode_workload([517, 1500, 129, 128, 2], N, Hq=8, Hkv=4, D=16, topk=5,
                                  seed=3, device="cpu")
    sl = w["seq_lens"].numpy()
    q_pos = torch.from_numpy(oracle.query_positions(sl, N))
    got = bench.visible_keys(w["block_ids"], q_pos)                       # [R, Hkv]
    _, lens = oracle.build_sparse_page_table(w["block_ids"].numpy(), w["page_table"].numpy(), sl, N)
    assert np.array_equal(got.numpy().reshape(-1), np.asarray(lens).reshape(-1))


def test_headline_flops_equal_the_split_total():
    T, prefix, Hkv, k, G, D = 300, 2048, 2, 8, 8, 128
    ids = torch.from_numpy(_selection(T, prefix, Hkv, k, seed=6))
    q_pos = torch.arange(prefix, prefix + T, dtype=torch.int64)
    flops = 4 * D * G * int(bench.visible_keys(ids, q_pos).sum())
    assert flops == bench.prefill_split(ids, prefix + T, G, D)["flops_total"]

