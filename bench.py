"""Benchmark of the GB300 MSA layer hot path.

One step = one pass of every hot-path stage over its synthetic workload, inputs resident in
HBM (all larger than the 129 MB L2, so no flush is needed between steps):
  * index score + top-k     decode scoring: 8 requests x 60032 tokens, Hkv 8, Di 128, k 16
                            (8 planted high-affinity blocks per request and group)
  * sparse page table + paged sparse decode: 64 requests, context ~U[8K, 128K], Hq 64,
                            Hkv 8, D 128, k 16 (KV groups flattened into 512 rows)
  * sparse prefill (query ordering and shared-block selection, bucketing, query-major and
                            block-major attention partials, LSE merge): 32768-token causal
                            chunk, Hq 64, Hkv 8, D 128, k 16, clustered selections
The headline `value` is the index-score + top-k HBM throughput (GB/s of K-index scanned);
`stages` carries every stage's throughput and roofline fraction.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs its own replica of the workload (the layer shards by
request and KV group with no exchange): value = all ranks' bytes / max-over-ranks time.
`--impl reference` times the CPU oracle instead (rank 0 only) on the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import threading
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "index-score+topk & sparse-decode HBM GB/s; prefill sparse-attn TFLOP/s (%peak)"
# the workload the headline value is measured on, the same string in both arms
HEADLINE_WORKLOAD = ("decode index score + top-k: 8 requests x 60032 tokens (469 blocks), "
                     "Hkv 8, Di 128, k 16")
BLOCK = 128


# --------------------------------------------------------------------------- environment

def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(vals, ws: int, device):
    """Each value's maximum over all ranks (identity on one rank): the job's time is the slowest
    rank's."""
    if ws <= 1:
        return [float(v) for v in vals]
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def job_throughput(units_per_rank: float, ms: float, ws: int) -> float:
    """Whole-job throughput: every rank processes its own replica of `units_per_rank`, the job
    takes `ms` (the max over ranks)."""
    return units_per_rank * ws / (ms * 1e-3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms; only the lines that arrive
    between entering and leaving the `with` block (the timed region) are kept. Entering waits
    for nvidia-smi's first line so that sampling is running when the region starts."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.out = ""

    def _reader(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line))

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()
        t0 = time.monotonic()
        while not self.lines and time.monotonic() - t0 < 5.0:
            time.sleep(0.01)
        self.t_start = time.monotonic()
        return self

    def __exit__(self, *exc):
        t_end = time.monotonic()
        if self.proc is None:
            return
        time.sleep(0.15)  # a sample taken just before the end may still be in flight
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.thread.join(timeout=5)
        self.out = "".join(l for t, l in list(self.lines) if self.t_start <= t <= t_end + 0.1)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- workloads

def visible_keys(block_ids: torch.Tensor, q_pos: torch.Tensor) -> torch.Tensor:
    """Visible keys per (row, group) for kept blocks: 128 below the local block, q_pos%128+1 in it."""
    local = (q_pos // BLOCK)[:, None, None]
    ids = block_ids.to(torch.int64)
    n = torch.where(ids < local, torch.full_like(ids, BLOCK),
                    torch.where(ids == local, (q_pos % BLOCK + 1)[:, None, None].expand_as(ids),
                                torch.zeros_like(ids)))
    n = torch.where(ids >= 0, n, torch.zeros_like(n))
    return n.sum(dim=2)


def prefill_split(block_ids: torch.Tensor, S_kv: int, G: int, D: int) -> dict:
    """FLOPs of the two attention passes of msa_sparse_prefill, for reporting.

    Restates the selection rule of the query-major pass (G 8 / 16, key range <= 16384 blocks):
    the queries of each 128-query span are ranked by how many of their blocks at least half of
    the span chose (stable, descending); 2*128/G consecutive ranks form a pair; a block at
    least half of the pair's slots chose (at most 64 per pair, ascending) is computed
    query-major for the whole pair, every other selection block-major. Returns algorithmic
    FLOPs of each pass and the FLOPs the query-major pass executes (masked rows included)."""
    T, Hkv, k = block_ids.shape
    dev = block_ids.device
    pos = torch.arange(S_kv - T, S_kv, device=dev)
    ids = block_ids.long()
    valid = ids >= 0
    local = (pos // BLOCK)[:, None, None]
    vis = torch.where(ids < local, torch.full_like(ids, BLOCK), (pos % BLOCK + 1)[:, None, None].expand_as(ids))
    vis = torch.where(valid & (ids <= local), vis, torch.zeros_like(vis))
    flops_sel = 4 * D * G * vis                                  # per (t, g, slot)
    total = int(flops_sel.sum())
    nb = (S_kv + BLOCK - 1) // BLOCK
    if G not in (8, 16) or nb > 16384:
        return {"flops_total": total, "flops_block_major": total, "flops_query_major": 0,
                "flops_query_major_executed": 0, "query_major_items": 0}
    qpt = 128 // G
    nq = 2 * qpt
    nspan = (T + 127) // 128
    Tp = nspan * 128
    idp = torch.full((Tp, Hkv, k), -1, dtype=torch.long, device=dev)
    idp[:T] = ids
    vp = idp >= 0
    span = torch.arange(Tp, device=dev) // 128
    g_idx = torch.arange(Hkv, device=dev)[None, :, None].expand(Tp, Hkv, k)
    s_idx = span[:, None, None].expand(Tp, Hkv, k)
    col = torch.where(vp, idp, torch.full_like(idp, nb))        # invalid -> trash column nb
    key = (g_idx * nspan + s_idx) * (nb + 1) + col
    cnt = torch.zeros(Hkv * nspan * (nb + 1), dtype=torch.long, device=dev)
    cnt.scatter_add_(0, key.reshape(-1), vp.reshape(-1).long())
    nvalid = torch.clamp(T - torch.arange(nspan, device=dev) * 128, max=128)
    cnt3 = cnt.view(Hkv, nspan, nb + 1)
    pop = 2 * cnt3 >= nvalid[None, :, None]
    pop[:, :, nb] = False
    sel_pop = pop.view(-1)[key.reshape(-1)].view(Tp, Hkv, k) & vp
    score = sel_pop.sum(dim=2)                                   # [Tp, Hkv]
    score = torch.where(torch.arange(Tp, device=dev)[:, None] < T, score, torch.full_like(score, -1))
    sc = score.view(nspan, 128, Hkv).permute(2, 0, 1)            # [Hkv, nspan, 128]
    order = torch.sort(-sc, dim=2, stable=True).indices          # slot -> query within span
    rank = torch.empty_like(order)
    rank.scatter_(2, order, torch.arange(128, device=dev).expand_as(order))
    pair = (rank // nq).permute(1, 2, 0).reshape(Tp, Hkv)        # pair within span per (t, g)
    npp = 128 // nq
    pkey = ((g_idx * nspan + s_idx) * npp + pair[:, :, None]) * (nb + 1) + col
    pc = torch.zeros(Hkv * nspan * npp * (nb + 1), dtype=torch.long, device=dev)
    pc.scatter_add_(0, pkey.reshape(-1), vp.reshape(-1).long())
    pc = pc.view(-1, nb + 1)
    pc[:, nb] = 0
    thr = max(2, (nq + 1) // 2)
    dense = pc >= thr
    dense &= torch.cumsum(dense.long(), dim=1) <= 64             # kMaxDense per pair
    items = int(dense.sum())
    in_qm = dense.view(-1)[pkey.reshape(-1)].view(Tp, Hkv, k) & vp
    qm = int(flops_sel[in_qm[:T]].sum())
    return {"flops_total": total, "flops_query_major": qm, "flops_block_major": total - qm,
            "flops_query_major_executed": items * 2 * 2 * 2 * 128 * 128 * 128,
            "query_major_items": items}


def build_workloads(dev, seed_offset: int, small: bool = False):
    # --small (profiling captures only): 8 decode requests and an 8192-token prefill chunk
    wsc = workloads.decode_scoring(dev, seed=2 + seed_offset)
    wdc = workloads.paged_decode(dev, seed=4 + seed_offset, B=8 if small else None)
    wpf = workloads.causal_prefill(dev, seed=3 + seed_offset, T=8192 if small else None)
    # algorithmic work per stage
    B, Hkv, Di = wsc["B"], wsc["Hkv"], wsc["Di"]
    sl2 = wsc["seq_lens"].to(torch.int64)
    wsc["bytes"] = int(sl2.sum().item()) * Hkv * Di * 2 + wsc["q_idx"].numel() * 2 \
        + wsc["page_table"].numel() * 4 + B * Hkv * wsc["topk"] * 8
    q_pos4 = wdc["seq_lens"].to(torch.int64) - 1
    keys4 = visible_keys(wdc["block_ids"], q_pos4)                 # [B, Hkv]
    Gdc = wdc["Hq"] // wdc["Hkv"]
    wdc["bytes"] = int(keys4.sum().item()) * wdc["D"] * 2 * 2 + wdc["q"].numel() * 2 * 2 \
        + wdc["B"] * wdc["Hq"] * 4
    wdc["kv_bytes"] = int(keys4.sum().item()) * wdc["D"] * 2 * 2
    q_pos3 = torch.arange(wpf["S_kv"] - wpf["T"], wpf["S_kv"], device=dev, dtype=torch.int64)
    keys3 = visible_keys(wpf["block_ids"], q_pos3)                 # [T, Hkv]
    Gpf = wpf["Hq"] // wpf["Hkv"]
    wpf["flops"] = 4 * wpf["D"] * Gpf * int(keys3.sum().item())
    # bf16 partial rows (G per selection, D channels) written once and read once, + fp32 LSE
    nsel3 = int((wpf["block_ids"] >= 0).sum().item())
    wpf["partial_bytes"] = nsel3 * Gpf * (2 * wpf["D"] * 2 + 4 * 2)
    # bytes a perfect prefill must move: q read, each K/V row of the sequence read once, o
    # written, lse written
    wpf["algorithmic_bytes"] = (wpf["q"].numel() * 2 + wpf["k"].numel() * 2 * 2
                                + wpf["T"] * wpf["Hq"] * (wpf["D"] * 2 + 4))
    wpf["split"] = prefill_split(wpf["block_ids"], wpf["S_kv"], Gpf, wpf["D"])
    del Gdc
    return wsc, wdc, wpf


def prefill_sustained(msa, wpf, wsp, o3, lse3, pre_ms, pk, local, seconds=2.0):
    """The prefill call back to back for about `seconds`, the regime of the sustained bf16
    peak (cuBLAS looped for seconds under the power cap): TFLOP/s against that peak, with the
    clocks sampled over the loop."""
    n = max(10, int(seconds * 1e3 / max(pre_ms, 1e-3)))
    call = lambda: msa.sparse_prefill(wpf["q"], wpf["k"], wpf["v"], wpf["block_ids"], workspace=wsp,
                                      out=(o3, lse3))
    call()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        a.record()
        for _ in range(n):
            call()
        b.record()
        torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    tfl = wpf["flops"] / (ms * 1e-3) / 1e12
    return {"calls": n, "seconds": round(ms * n / 1e3, 2), "ms": round(ms, 4),
            "TFLOP/s": round(tfl, 1), "peak": pk["bf16_tflops_sustained"],
            "peak_kind": "sustained (measured, seconds-long loop)",
            "frac_bf16_sustained": round(tfl / pk["bf16_tflops_sustained"], 4),
            "clocks": clk.summary()}


def prefill_stage(wpf, pre_ms, pk):
    """The prefill call's line: end-to-end TFLOP/s against the burst bf16 peak (the call is timed
    alone per step, a few ms, not a seconds-long loop), its FLOP split between the query-major and
    block-major passes, and its DRAM traffic against the bytes a perfect call must move."""
    eps = 1e-9
    tfl = wpf["flops"] / (max(pre_ms, eps) * 1e-3) / 1e12
    sp = wpf["split"]
    traffic = prefill_traffic()
    return {"config": f"T {wpf['T']} causal, Hq {wpf['Hq']}, Hkv {wpf['Hkv']}, D {wpf['D']}, "
                      f"k {wpf['topk']}", "ms": round(pre_ms, 4),
            "TFLOP/s": round(tfl, 1),
            "frac_bf16": round(tfl / pk["bf16_tflops"], 4),
            "peak": pk["bf16_tflops"], "peak_kind": "burst (measured)",
            "frac_bf16_sustained": round(tfl / pk["bf16_tflops_sustained"], 4),
            "kernels": "selection + counting; list offsets + pair deal; placement; block-major attention "
                       "for the scattered selections; query-major attention for blocks shared "
                       "by a query pair; LSE merge "
                       "(per-kernel times: profiles/launches_bench_default.md)",
            "flops": wpf["flops"],
            # algorithmic FLOPs per pass, and what the query-major pass executes (its pairs'
            # rows that did not choose a block ride through the MMAs masked)
            "flops_query_major": sp["flops_query_major"],
            "flops_block_major": sp["flops_block_major"],
            "flops_query_major_executed": sp["flops_query_major_executed"],
            "query_major_items": sp["query_major_items"],
            # a purely block-major prefill writes one bf16 partial of G rows per (query, block)
            # selection and reads it back: that traffic alone takes block_major_floor_ms at the
            # measured HBM bandwidth
            "block_major_partials_bytes": wpf["partial_bytes"],
            "block_major_floor_ms": round(wpf["partial_bytes"] / pk["hbm_gbs"] / 1e6, 4),
            # q in, each K/V row once, o and lse out
            "algorithmic_bytes": wpf["algorithmic_bytes"],
            # DRAM bytes of every kernel of the call, from per-kernel captures (null when any
            # kernel's source changed since it was captured)
            "traffic_total": traffic,
            "traffic_over_algorithmic": (round(traffic / wpf["algorithmic_bytes"], 3)
                                         if traffic else None)}


def src_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "block_sparse_attention_msa_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, source_hash: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_hash") != source_hash:
        return None
    return rec.get("bytes_per_launch")


# Every kernel of one msa_sparse_prefill call and the source files its code comes from (the
# .cu file, and a kernel-specific header where it has one).
PREFILL_KERNELS = (("select_count_kernel", ("prefill_dense.cu",)),
                   ("bucket_lists_kernel", ("prefill.cu", "pair_deal.cuh")),
                   ("bucket_place_kernel", ("prefill.cu",)),
                   ("prefill_block_tc_kernel", ("prefill.cu",)),
                   ("prefill_dense_tc_kernel", ("prefill_dense.cu",)),
                   ("lse_merge_chunked_kernel", ("page_table_merge.cu",)))


def prefill_traffic():
    """DRAM bytes of one prefill call: the sum over its kernels' recorded captures (null while
    any of them is missing or its source changed since it was captured)."""
    tot = 0
    for name, srcs in PREFILL_KERNELS:
        b = recorded_traffic(name, src_hash(*srcs))
        if b is None:
            return None
        tot += b
    return tot


# --------------------------------------------------------------------------- our arm

def run_ours(args, ws, rank, local):
    import block_sparse_attention_msa_gb300 as msa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    msa.load(build_if_missing=True)
    pk = peaks()
    wsc, wdc, wpf = build_workloads(dev, seed_offset=1000 * rank, small=args.small)
    run = set(args.stages.split(","))
    wsp = msa.Workspace()
    # preallocated outputs
    Rsc = wsc["B"]
    ids_sc = torch.empty((Rsc, wsc["Hkv"], wsc["topk"]), dtype=torch.int32, device=dev)
    scores_sc = torch.empty((Rsc, wsc["Hkv"], wsc["topk"]), dtype=torch.float32, device=dev)
    Rdc = wdc["B"]
    fpt_dc = torch.empty((Rdc * wdc["Hkv"], wdc["topk"]), dtype=torch.int32, device=dev)
    len4 = torch.empty((Rdc * wdc["Hkv"],), dtype=torch.int32, device=dev)
    o4 = torch.empty((Rdc, wdc["Hq"], wdc["D"]), dtype=torch.bfloat16, device=dev)
    lse4 = torch.empty((Rdc, wdc["Hq"]), dtype=torch.float32, device=dev)
    o3 = torch.empty((wpf["T"], wpf["Hq"], wpf["D"]), dtype=torch.bfloat16, device=dev)
    lse3 = torch.empty((wpf["T"], wpf["Hq"]), dtype=torch.float32, device=dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record()
        if "score" in run:
            msa.index_score_topk(wsc["q_idx"], wsc["k_idx_pages"], wsc["page_table"], wsc["seq_lens"], 1,
                                 wsc["topk"], workspace=wsp, out=(ids_sc, scores_sc))
        if ev is not None:
            ev[1].record()
        if "decode" in run:
            msa.build_sparse_page_table(wdc["block_ids"], wdc["page_table"], wdc["seq_lens"], 1,
                                        wdc["num_pages"], out=(fpt_dc, len4))
        if ev is not None:
            ev[2].record()
        if "decode" in run:
            msa.paged_sparse_decode(wdc["q"], wdc["k_cache"], wdc["v_cache"], fpt_dc, len4, workspace=wsp,
                                    out=(o4, lse4))
        if ev is not None:
            ev[3].record()
        if "prefill" in run:
            msa.sparse_prefill(wpf["q"], wpf["k"], wpf["v"], wpf["block_ids"], workspace=wsp,
                               out=(o3, lse3))
        if ev is not None:
            ev[4].record()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        start.record()
        for k in range(args.steps):
            step(evs[k])
        stop.record()
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    total_ms = start.elapsed_time(stop)
    stage_ms = [sum(e[i].elapsed_time(e[i + 1]) for e in evs) / args.steps for i in range(4)]
    # the slowest rank sets the job's time
    total_ms, *stage_ms = max_over_ranks([total_ms] + stage_ms, ws, dev)
    ms_per_step = total_ms / args.steps
    score_ms, pt_ms, dec_ms, pre_ms = stage_ms
    # device error word: none expected
    err = msa.device_error()

    eps = 1e-9
    score_gbs = wsc["bytes"] / (max(score_ms, eps) * 1e-3) / 1e9
    dec_gbs = wdc["bytes"] / (max(pt_ms + dec_ms, eps) * 1e-3) / 1e9
    pre_tflops = wpf["flops"] / (max(pre_ms, eps) * 1e-3) / 1e12
    value = job_throughput(wsc["bytes"], max(score_ms, eps), ws) / 1e9

    # e2e through host buffers for the headline stage, and for the decode stage
    def rest_of_step():
        if "decode" in run:
            msa.build_sparse_page_table(wdc["block_ids"], wdc["page_table"], wdc["seq_lens"], 1,
                                        wdc["num_pages"], out=(fpt_dc, len4))
            msa.paged_sparse_decode(wdc["q"], wdc["k_cache"], wdc["v_cache"], fpt_dc, len4,
                                    workspace=wsp, out=(o4, lse4))
        if "prefill" in run:
            msa.sparse_prefill(wpf["q"], wpf["k"], wpf["v"], wpf["block_ids"], workspace=wsp,
                               out=(o3, lse3))

    e2e = e2e_score(msa, wsc, wsp, dev, args.steps, ws, between=rest_of_step) if "score" in run else None
    e2e_dec = e2e_decode(msa, wdc, wsp, dev, args.steps, ws) if "decode" in run else None
    # multi-token decode / verify rows, and decode from host-resident K/V caches (outside the
    # timed step: each is its own configuration)
    extra = {}
    if not args.no_extra and "prefill" in run and not args.small:
        extra["sparse_prefill_sustained"] = prefill_sustained(msa, wpf, wsp, o3, lse3, pre_ms, pk,
                                                              local)
    if not args.no_extra and {"score", "decode"} <= run:
        extra.update(multi_token_stages(msa, wsc, wdc, wsp, dev, max(10, args.steps), pk))
        if not args.no_host_stage:
            extra["sparse_decode_host_kv"] = staged_host_decode(msa, wdc, fpt_dc, len4, wsp, dev,
                                                                max(10, args.steps), pk)

    h_score = src_hash("score_topk.cu")
    roofline = {"kernel": "score_decode_kernel (msa_index_score_topk)", "bound": "hbm",
                "achieved": round(score_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(score_gbs / pk["hbm_gbs"], 4),
                "traffic": recorded_traffic("score_decode_kernel", h_score),
                "algorithmic_bytes": wsc["bytes"], "peak_source": pk["source"]}
    stages = {
        "index_score_topk": {"config": f"{wsc['B']} x {wsc['max_seq_len']} tokens, Hkv {wsc['Hkv']}, "
                                       f"Di {wsc['Di']}, k {wsc['topk']}", "ms": round(score_ms, 4),
                             "GB/s": round(score_gbs, 1), "frac_hbm": round(score_gbs / pk["hbm_gbs"], 4),
                             "bytes": wsc["bytes"]},
        "sparse_decode": {"config": f"{wdc['B']} req, ctx U[8K,128K], Hq {wdc['Hq']}, Hkv {wdc['Hkv']}, "
                                    f"D {wdc['D']}, k {wdc['topk']}",
                          "ms_page_table": round(pt_ms, 4), "ms_decode": round(dec_ms, 4),
                          "GB/s": round(dec_gbs, 1), "frac_hbm": round(dec_gbs / pk["hbm_gbs"], 4),
                          "bytes": wdc["bytes"], "kv_bytes": wdc["kv_bytes"],
                          "traffic": recorded_traffic("paged_decode_kernel", src_hash("decode.cu")),
                          "e2e": e2e_dec},
        "sparse_prefill": prefill_stage(wpf, pre_ms, pk),
    }
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded, device-generated)",
        "config": {"workload": HEADLINE_WORKLOAD,
                   "step": "the step also runs paged sparse decode (64 requests) and the sparse "
                           "prefill (32768 tokens); value is the scorer stage's GB/s",
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{ws}"},
        "roofline": roofline, "stages": stages, "e2e": e2e,
        # kernels of this library per step: scorer with its top-k (1); page table, decode,
        # merge (3); selection with counting, list offsets with the query-major pairs' deal,
        # placement, block-major attention, query-major attention, merge (6). Memsets not counted.
        "gpu_launches": args.steps * (("score" in run) * 1 + ("decode" in run) * 3
                                      + ("prefill" in run) * 6),
        "clocks": clk.summary(), "device_error_word": err,
    }
    for key, name in (("score", "index_score_topk"), ("decode", "sparse_decode"), ("prefill", "sparse_prefill")):
        if key not in run:
            stages[name] = None
    stages.update(extra)
    if "score" not in run:  # the headline is the scorer's: nothing to report without it
        line["value"] = None
        line["roofline"] = None
    if args.long_context:
        line["long_context"] = run_long_context(args, local)
    if args.small or run != {"score", "decode", "prefill"}:
        line["config"]["partial_run"] = f"stages={sorted(run)} small={args.small} (profiling only)"
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        if "score" in run:
            line["cpu_baseline"] = cpu_baseline(wsc, args.cpu_seconds)
            stages["index_score_topk"]["cpu_baseline"] = line["cpu_baseline"]
        if "decode" in run:
            stages["sparse_decode"]["cpu_baseline"] = cpu_baseline_decode(wdc)
        if "prefill" in run:
            stages["sparse_prefill"]["cpu_baseline"] = cpu_baseline_prefill(wpf)
    if rank == 0:
        print(json.dumps(line), flush=True)


def e2e_score(msa, wsc, wsp, dev, steps: int, ws: int, between=None):
    """Headline stage through the public API with pinned host buffers: per step the query
    index rows, page table and lengths go host->device and the selection comes back; the
    paged K-index cache is resident state (it is written once per token, not per step).
    `between` (untimed) runs the rest of the bench step before each timed call, so that the
    call meets the memory system in the state the in-step headline does."""
    h_q = wsc["q_idx"].cpu().pin_memory()
    h_pt = wsc["page_table"].cpu().pin_memory()
    h_sl = wsc["seq_lens"].cpu().pin_memory()
    R, Hkv, k = wsc["B"], wsc["Hkv"], wsc["topk"]
    h_ids = torch.empty((R, Hkv, k), dtype=torch.int32).pin_memory()
    h_sc = torch.empty((R, Hkv, k), dtype=torch.float32).pin_memory()
    d_q = torch.empty_like(wsc["q_idx"])
    d_pt = torch.empty_like(wsc["page_table"])
    d_sl = torch.empty_like(wsc["seq_lens"])
    ids = torch.empty((R, Hkv, k), dtype=torch.int32, device=dev)
    sc = torch.empty((R, Hkv, k), dtype=torch.float32, device=dev)

    def one():
        d_q.copy_(h_q, non_blocking=True)
        d_pt.copy_(h_pt, non_blocking=True)
        d_sl.copy_(h_sl, non_blocking=True)
        msa.index_score_topk(d_q, wsc["k_idx_pages"], d_pt, d_sl, 1, k, workspace=wsp, out=(ids, sc))
        h_ids.copy_(ids, non_blocking=True)
        h_sc.copy_(sc, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for s, e in evs:
        if between is not None:
            between()
        s.record()
        one()
        e.record()
    torch.cuda.synchronize()
    ms = max_over_ranks([sum(s.elapsed_time(e) for s, e in evs) / steps], ws, dev)[0]
    h2d = h_q.numel() * 2 + h_pt.numel() * 4 + h_sl.numel() * 4
    d2h = h_ids.numel() * 4 + h_sc.numel() * 4
    return {"value": round(job_throughput(wsc["bytes"], ms, ws) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "note": "per-step inputs copied from pinned host memory; paged K-index resident; "
                    "each timed call follows the step's other stages, as in the timed step"}


# --------------------------------------------------------------------------- extra stages

def _timed(fn, reps: int) -> float:
    """Mean ms per call of fn on the current stream, after 3 untimed calls."""
    for _ in range(3):
        fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def multi_token_stages(msa, wsc, wdc, wsp, dev, reps: int, pk) -> dict:
    """Multi-token decode / speculative verify: N query rows per request.

    * index score + top-k for N = 2, 4, 8 rows per request on the decode-scoring K-index (8
      requests x 60032 tokens): the streaming scorer reads the K-index once for all N rows;
    * sparse page table + paged decode for N = 2, 4 rows per request on the paged-decode caches
      (64 requests): each row reads its own selection (rows are not deduplicated)."""
    out = {}
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242)
    B, Hkv, Di, k = wsc["B"], wsc["Hkv"], wsc["Di"], wsc["topk"]
    kidx_bytes = int(wsc["seq_lens"].to(torch.int64).sum()) * Hkv * Di * 2 + wsc["page_table"].numel() * 4
    for N in (2, 4, 8):
        q_idx = workloads.randn_bf16((B * N, Hkv, Di), gen, dev)
        ids = torch.empty((B * N, Hkv, k), dtype=torch.int32, device=dev)
        sc = torch.empty((B * N, Hkv, k), dtype=torch.float32, device=dev)
        ms = _timed(lambda: msa.index_score_topk(q_idx, wsc["k_idx_pages"], wsc["page_table"],
                                                 wsc["seq_lens"], N, k, workspace=wsp,
                                                 out=(ids, sc)), reps)
        nbytes = kidx_bytes + q_idx.numel() * 2 + ids.numel() * 8
        gbs = nbytes / ms / 1e6
        out[f"index_score_topk_N{N}"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                         "frac_hbm": round(gbs / pk["hbm_gbs"], 4), "bytes": nbytes}
    Bd, Hq, Hkvd, D, kd = wdc["B"], wdc["Hq"], wdc["Hkv"], wdc["D"], wdc["topk"]
    sl = wdc["seq_lens"].to(torch.int64)
    for N in (2, 4):
        q = workloads.randn_bf16((Bd * N, Hq, D), gen, dev, scale=D ** -0.5)
        q_pos = (sl[:, None] - N + torch.arange(N, device=dev)[None, :]).reshape(-1)
        ids = workloads.sample_selection(q_pos, Hkvd, kd, gen)
        fpt = torch.empty((Bd * N * Hkvd, kd), dtype=torch.int32, device=dev)
        lens = torch.empty((Bd * N * Hkvd,), dtype=torch.int32, device=dev)
        o = torch.empty((Bd * N, Hq, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((Bd * N, Hq), dtype=torch.float32, device=dev)

        def f():
            msa.build_sparse_page_table(ids, wdc["page_table"], wdc["seq_lens"], N, wdc["num_pages"],
                                        out=(fpt, lens))
            msa.paged_sparse_decode(q, wdc["k_cache"], wdc["v_cache"], fpt, lens, workspace=wsp,
                                    out=(o, lse))
        ms = _timed(f, reps)
        kv = int(visible_keys(ids, q_pos).sum()) * D * 2 * 2
        nbytes = kv + q.numel() * 2 * 2 + lse.numel() * 4
        gbs = nbytes / ms / 1e6
        out[f"sparse_decode_N{N}"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                      "frac_hbm": round(gbs / pk["hbm_gbs"], 4), "bytes": nbytes,
                                      "kv_bytes": kv}
    return out


def staged_host_decode(msa, wdc, fpt_dc, len4, wsp, dev, reps: int, pk) -> dict:
    """KV residency split at the paged-decode workload: the K/V caches live in pinned host
    memory; per step the selected blocks' K/V rows are staged onto the device (read by the
    kernel over the host link) and the paged decode runs on the staging cache."""
    t0 = time.perf_counter()
    hk = torch.empty(wdc["k_cache"].shape, dtype=torch.bfloat16, pin_memory=True)
    hv = torch.empty(wdc["v_cache"].shape, dtype=torch.bfloat16, pin_memory=True)
    hk.copy_(wdc["k_cache"])
    hv.copy_(wdc["v_cache"])
    torch.cuda.synchronize()
    setup_s = time.perf_counter() - t0
    R, Hkv, D, k = wdc["B"], wdc["Hkv"], wdc["D"], wdc["topk"]
    ks = torch.empty((R * k, BLOCK, Hkv, D), dtype=torch.bfloat16, device=dev)
    vs = torch.empty_like(ks)
    spt = torch.empty_like(fpt_dc)
    o = torch.empty((R, wdc["Hq"], D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((R, wdc["Hq"]), dtype=torch.float32, device=dev)
    ms_stage = _timed(lambda: msa.stage_selected_kv(hk, hv, fpt_dc, out=(ks, vs, spt)), reps)

    def f():
        msa.stage_selected_kv(hk, hv, fpt_dc, out=(ks, vs, spt))
        msa.paged_sparse_decode(wdc["q"], ks, vs, spt, len4, workspace=wsp, out=(o, lse))
    ms = _timed(f, reps)
    staged = int((fpt_dc >= 0).sum()) * BLOCK * D * 2 * 2       # whole pages of one group, K + V
    del hk, hv
    return {"config": "paged-decode workload with K/V caches in pinned host memory",
            "ms_stage": round(ms_stage, 4), "ms_stage_and_decode": round(ms, 4),
            "staged_bytes": staged, "GB/s_staging": round(staged / ms_stage / 1e6, 1),
            "host_cache_bytes": 2 * wdc["k_cache"].numel() * 2, "setup_s": round(setup_s, 1)}


def e2e_decode(msa, wdc, wsp, dev, steps: int, ws: int) -> dict:
    """Sparse page table + paged decode through the public API from pinned host buffers: per
    step the queries, selections, lengths and page table go host->device and the output and
    LSE come back; the K/V caches are resident state."""
    R, Hq, D, Hkv, k = wdc["B"], wdc["Hq"], wdc["D"], wdc["Hkv"], wdc["topk"]
    hq = wdc["q"].cpu().pin_memory()
    hids = wdc["block_ids"].cpu().pin_memory()
    hsl = wdc["seq_lens"].cpu().pin_memory()
    hpt = wdc["page_table"].cpu().pin_memory()
    ho = torch.empty((R, Hq, D), dtype=torch.bfloat16).pin_memory()
    hlse = torch.empty((R, Hq), dtype=torch.float32).pin_memory()
    dq, dids, dsl, dpt = (torch.empty_like(x, device=dev) for x in (hq, hids, hsl, hpt))
    fpt = torch.empty((R * Hkv, k), dtype=torch.int32, device=dev)
    lens = torch.empty((R * Hkv,), dtype=torch.int32, device=dev)
    o = torch.empty((R, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((R, Hq), dtype=torch.float32, device=dev)

    def one():
        for d, h in ((dq, hq), (dids, hids), (dsl, hsl), (dpt, hpt)):
            d.copy_(h, non_blocking=True)
        msa.build_sparse_page_table(dids, dpt, dsl, 1, wdc["num_pages"], out=(fpt, lens))
        msa.paged_sparse_decode(dq, wdc["k_cache"], wdc["v_cache"], fpt, lens, workspace=wsp,
                                out=(o, lse))
        ho.copy_(o, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    ms = max_over_ranks([_timed(one, steps)], ws, dev)[0]
    h2d = sum(x.numel() * x.element_size() for x in (hq, hids, hsl, hpt))
    d2h = ho.numel() * 2 + hlse.numel() * 4
    return {"value": round(job_throughput(wdc["bytes"], ms, ws) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "note": "per-step inputs copied from pinned host memory; K/V caches resident"}


# --------------------------------------------------------------------------- CPU oracle, per stage

def cpu_baseline_decode(wdc, n_req: int = 16) -> dict:
    """The oracle's sparse decode on the first n_req requests of the paged-decode workload (all
    their rows and heads), GB/s over their selected K/V bytes."""
    import numpy as np
    import oracle
    u16 = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    ids = wdc["block_ids"][:n_req]
    pt = wdc["page_table"][:n_req]
    sel_pages = torch.gather(pt, 1, ids.clamp(min=0).long().reshape(n_req, -1))[ids.reshape(n_req, -1) >= 0]
    pages = torch.unique(sel_pages).long()
    remap = torch.zeros(wdc["num_pages"], dtype=torch.int32, device=pt.device)
    remap[pages] = torch.arange(pages.numel(), dtype=torch.int32, device=pt.device)
    pt_small = remap[pt.long()]                      # pages never selected map to 0, never read
    kc, vc = u16(wdc["k_cache"][pages]), u16(wdc["v_cache"][pages])
    q = u16(wdc["q"][:n_req])
    sl = wdc["seq_lens"][:n_req].cpu().numpy()
    ids_np = ids.cpu().numpy()
    kv = int(visible_keys(ids, (wdc["seq_lens"][:n_req].to(torch.int64) - 1)).sum()) * wdc["D"] * 4
    t0 = time.perf_counter()
    oracle.sparse_decode(q, kc, vc, pt_small.cpu().numpy(), sl, ids_np, 1)
    dt = time.perf_counter() - t0
    return {"value": round(kv / dt / 1e9, 3), "unit": "GB/s", "cores": oracle.default_threads(),
            "kind": "oracle", "sample": f"{n_req} of {wdc['B']} requests, all heads, in {dt:.2f} s"}


def cpu_baseline_prefill(wpf, n_rows: int = 128) -> dict:
    """The oracle's sparse prefill on n_rows query rows spread over the chunk (all heads),
    TFLOP/s over their algorithmic FLOPs."""
    import numpy as np
    import oracle
    u16 = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    T, Hq, D = wpf["T"], wpf["Hq"], wpf["D"]
    G = Hq // wpf["Hkv"]
    rows = torch.linspace(0, T - 1, n_rows).round().long().unique()
    units = (rows[:, None] * Hq + torch.arange(Hq)[None, :]).reshape(-1).numpy()
    q_pos = (wpf["S_kv"] - T + rows).to(wpf["block_ids"].device)
    flops = 4 * D * G * int(visible_keys(wpf["block_ids"][rows.to(q_pos.device)], q_pos).sum())
    q, k, v = u16(wpf["q"]), u16(wpf["k"]), u16(wpf["v"])
    ids = wpf["block_ids"].cpu().numpy()
    t0 = time.perf_counter()
    oracle.sparse_prefill(q, k, v, ids, units=units)
    dt = time.perf_counter() - t0
    return {"value": round(flops / dt / 1e12, 5), "unit": "TFLOP/s", "cores": oracle.default_threads(),
            "kind": "oracle", "sample": f"{rows.numel()} of {T} query rows (all {Hq} heads) in {dt:.2f} s"}


# --------------------------------------------------------------------------- CPU oracle

def _oracle_score_step(oracle, h):
    s = oracle.block_scores(h["q_idx"], h["k_idx"], h["pt"], h["sl"], 1, rows=h["rows"])
    ids, _ = oracle.topk(s, h["q_pos"][h["rows"]], h["topk"])
    return ids


def _host_scoring(wsc, rows):
    import numpy as np
    u16 = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    sl = wsc["seq_lens"].cpu().numpy()
    return {"q_idx": u16(wsc["q_idx"]), "k_idx": u16(wsc["k_idx_pages"]),
            "pt": wsc["page_table"].cpu().numpy(), "sl": sl, "topk": wsc["topk"],
            "q_pos": (sl.astype("int64") - 1), "rows": np.asarray(rows, dtype=np.int64)}


def cpu_baseline(wsc, seconds: float):
    """The oracle as it stands, timed on this host's cores on the headline workload."""
    import oracle
    B = wsc["B"]
    h = _host_scoring(wsc, list(range(B)))
    per_row = wsc["bytes"] / B
    t0 = time.perf_counter()
    n = 0
    while True:
        _oracle_score_step(oracle, h)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    gbs = n * B * per_row / dt / 1e9
    return {"value": round(gbs, 3), "unit": "GB/s",
            "cores": min(oracle.default_threads(), B * wsc["Hkv"]), "kind": "oracle",
            "sample": f"{n} full passes of all {B} requests (scores + top-k) in {dt:.1f} s"}


def run_long_context(args, local):
    """1M-token layer, reported per stage (not part of the headline step): 4 x 1,048,576-token
    decode (score + top-k, sparse page table, paged decode, k 32) and a 32768-token prefill chunk
    on a 1,048,576-token prefix (score + top-k over every chunk row, then sparse attention with
    contiguous K/V and with the prefix read through a page table)."""
    import block_sparse_attention_msa_gb300 as msa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    msa.load(build_if_missing=True)
    pk = peaks()
    out = {}
    # --small (profiling captures only): one 131072-token request, an 8192-token chunk on a
    # 131072-token prefix
    w = workloads.long_context_decode(dev, seed=5, **(dict(B=1, seq_len=131072) if args.small else {}))
    ws_ = msa.Workspace()

    def timed(fn, reps):
        # device time of `reps` back-to-back calls: a spin kernel queued first keeps the GPU
        # busy while the host enqueues them, so calls shorter than their host-side cost are
        # timed by their kernels, not by the launch rate
        for _ in range(2):
            fn()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        torch.cuda._sleep(int(4e6))
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    B, Hkv, Di, k = w["B"], w["Hkv"], w["Di"], w["topk"]
    ids, _ = msa.index_score_topk(w["q_idx"], w["k_idx_pages"], w["page_table"], w["seq_lens"], 1, k,
                                  workspace=ws_)
    fpt, lens = msa.build_sparse_page_table(ids, w["page_table"], w["seq_lens"], 1, w["num_pages"])
    ms_s = timed(lambda: msa.index_score_topk(w["q_idx"], w["k_idx_pages"], w["page_table"],
                                              w["seq_lens"], 1, k, workspace=ws_), max(3, args.steps))
    ms_pt = timed(lambda: msa.build_sparse_page_table(ids, w["page_table"], w["seq_lens"], 1,
                                                      w["num_pages"]), max(3, args.steps))
    ms_d = timed(lambda: msa.paged_sparse_decode(w["q"], w["k_cache"], w["v_cache"], fpt, lens,
                                                 workspace=ws_), max(3, args.steps))
    kidx_bytes = int(w["seq_lens"].to(torch.int64).sum()) * Hkv * Di * 2
    kv_bytes = int(lens.to(torch.int64).sum()) * w["D"] * 2 * 2
    out["decode_score_topk"] = {"ms": round(ms_s, 4), "GB/s": round(kidx_bytes / ms_s / 1e6, 1),
                                "frac_hbm": round(kidx_bytes / ms_s / 1e6 / pk["hbm_gbs"], 4)}
    out["decode_page_table_ms"] = round(ms_pt, 4)
    # the same selection with its page table built in the scorer's tail (one launch)
    ms_sf = timed(lambda: msa.index_score_topk_page_table(w["q_idx"], w["k_idx_pages"],
                                                          w["page_table"], w["seq_lens"], 1, k,
                                                          workspace=ws_), max(3, args.steps))
    out["decode_score_topk_page_table_fused_ms"] = round(ms_sf, 4)
    out["decode_attention"] = {"ms": round(ms_d, 4), "GB/s": round(kv_bytes / ms_d / 1e6, 1),
                               "frac_hbm": round(kv_bytes / ms_d / 1e6 / pk["hbm_gbs"], 4)}
    del w, ids, fpt, lens
    torch.cuda.empty_cache()
    w = workloads.long_context_prefill(dev, seed=6, **(dict(T=8192, prefix=131072) if args.small else {}))
    T, S, P = w["T"], w["S"], w["P"]
    kidx_pages = w["k_idx"].view(P, 128, Hkv, Di)
    sl = torch.tensor([S], dtype=torch.int32, device=dev)
    ws2 = msa.Workspace()
    ids, _ = msa.index_score_topk(w["q_idx"], kidx_pages, w["page_table"], sl, T, k, workspace=ws2)
    ms_ps = timed(lambda: msa.index_score_topk(w["q_idx"], kidx_pages, w["page_table"], sl, T, k,
                                               workspace=ws2), 2)
    kk, vv = w["k"][:S], w["v"][:S]
    ms_pa = timed(lambda: msa.sparse_prefill(w["q"], kk, vv, ids, workspace=ws2), 3)
    q_pos = torch.arange(S - T, S, device=dev, dtype=torch.int64)
    score_flops = 2 * Di * Hkv * int((q_pos + 1).sum())  # every causal key of every row
    attn_flops = 4 * w["D"] * (w["Hq"] // Hkv) * int(visible_keys(ids, q_pos).sum())
    out["prefill_score_topk"] = {"ms": round(ms_ps, 3), "TFLOP/s": round(score_flops / ms_ps / 1e9, 1),
                                 "flops": score_flops}
    out["prefill_attention"] = {"ms": round(ms_pa, 3), "TFLOP/s": round(attn_flops / ms_pa / 1e9, 1),
                                "frac_bf16": round(attn_flops / ms_pa / 1e9 / pk["bf16_tflops"], 4),
                                "frac_bf16_sustained": round(attn_flops / ms_pa / 1e9
                                                             / pk["bf16_tflops_sustained"], 4),
                                "flops": attn_flops}
    # the same chunk with the prefix read from the paged cache through its page table (the
    # chunk's K/V viewed as [P, 128, Hkv, D] pages; a block's rows have the same layout as in
    # the contiguous form, only the block's base comes from the table)
    kc = w["k"].view(P, 128, Hkv, w["D"])
    vc = w["v"].view(P, 128, Hkv, w["D"])
    pt = w["page_table"][0].contiguous()
    ms_pp = timed(lambda: msa.sparse_prefill_paged(w["q"], kc, vc, pt, ids, S, workspace=ws2), 3)
    out["prefill_attention_paged"] = {"ms": round(ms_pp, 3),
                                      "TFLOP/s": round(attn_flops / ms_pp / 1e9, 1),
                                      "frac_bf16": round(attn_flops / ms_pp / 1e9 / pk["bf16_tflops"], 4),
                                      "frac_bf16_sustained": round(attn_flops / ms_pp / 1e9
                                                                   / pk["bf16_tflops_sustained"], 4)}
    return out


def run_reference(args, ws, rank, local):
    if rank != 0:
        return
    import oracle
    oracle.build()
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    wsc = workloads.decode_scoring(dev, seed=2)
    B = wsc["B"]
    wsc["bytes"] = int(wsc["seq_lens"].to(torch.int64).sum().item()) * wsc["Hkv"] * wsc["Di"] * 2 \
        + wsc["q_idx"].numel() * 2 + wsc["page_table"].numel() * 4 + B * wsc["Hkv"] * wsc["topk"] * 8
    h = _host_scoring(wsc, list(range(B)))
    for _ in range(args.warmup):
        _oracle_score_step(oracle, h)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_score_step(oracle, h)
    dt = time.perf_counter() - t0
    ms = dt / args.steps * 1e3
    gbs = wsc["bytes"] / (ms * 1e-3) / 1e9
    cores = min(oracle.default_threads(), B * wsc["Hkv"])
    line = {"metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "impl": "reference",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded)",
            "config": {"workload": HEADLINE_WORKLOAD, "parallelism": "cpu oracle"},
            "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step scores and selects all {B} requests"},
            "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--stages", default="score,decode,prefill",
                    help="comma list of stages to run (profiling captures)")
    ap.add_argument("--long-context", action="store_true",
                    help="also report the 1M-token layer's stages (takes about a minute)")
    ap.add_argument("--small", action="store_true",
                    help="smaller decode/prefill workloads (profiling captures only)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the multi-token and host-resident K/V stages")
    ap.add_argument("--no-host-stage", action="store_true",
                    help="skip the decode from host-resident K/V caches")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    ws, rank, local = dist_info()
    if ws > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, ws, rank, local)
        else:
            run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
