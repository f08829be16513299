"""Seeded synthetic inputs for the MSA layer, shaped like the five workloads it is measured on.

This module is the only code shared by the CUDA path's callers and the oracle's callers.
It contains no MSA arithmetic: it draws random tensors, page permutations and block
selections, and builds index tables. Block selections that stand in for "top-k of seeded
scores" are drawn directly with the same distribution (see ``sample_selection``).

Every generator takes a ``seed`` and a torch ``device``. The stream of numbers depends on
the device (torch's CPU and CUDA generators differ), so a test draws the inputs once and
copies them to the other side; nothing compares two draws made on different devices.

Workload recipes (sizes in the docstrings of the named workloads below):
  * tiny_layer: 1 sequence of 2048 tokens, Hq=8, Hkv=2, D=128, Di=64, k=4, causal
          prefill then 16 decode steps, contiguous pages (identity page table).
  * decode_scoring: B=8 x 60032 tokens, Hkv=8, Di=128, k=16, 8 planted
          high-affinity blocks per (request, group), random page permutation.
  * causal_prefill (block-major sparse prefill): T=32768 causal, Hq=64, Hkv=8, D=128, k=16 with
          clustered selections (~75% of the queries of a 128-query span share 12 blocks).
  * paged_decode: B=64, context ~U[8K,128K], Hq=64, Hkv=8, D=128, k=16.
  * long_context_decode / long_context_prefill (1M-token layer): 4 decode requests at 1,048,576 tokens (k=32) and a 32768-token
          prefill chunk after a 1,048,576-token prefix (k=32).
"""
from __future__ import annotations

import math

import torch

BLOCK = 128


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, gen: torch.Generator, device, scale: float = 1.0,
               chunk_elems: int = 1 << 28) -> torch.Tensor:
    """N(0, scale^2) samples rounded to bf16, drawn in chunks to bound temporaries."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk_elems):
        e = min(flat.numel(), s + chunk_elems)
        x = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        flat[s:e] = x.to(torch.bfloat16)
    return out


def paged_layout(seq_lens, gen: torch.Generator, device, shuffle: bool = True):
    """Page table for requests of the given lengths: each request gets ceil(len/128) pages.

    Returns (page_table [B, max_blocks] int32, num_pages). Pages are a random permutation
    of 0..num_pages-1 when ``shuffle``, else consecutive per request. Unused entries are 0.
    """
    seq_lens = [int(s) for s in seq_lens]
    nblk = [(s + BLOCK - 1) // BLOCK for s in seq_lens]
    num_pages = sum(nblk)
    max_blocks = max(nblk)
    if shuffle:
        perm = torch.randperm(num_pages, generator=gen, device=device).to(torch.int32)
    else:
        perm = torch.arange(num_pages, device=device, dtype=torch.int32)
    table = torch.zeros((len(seq_lens), max_blocks), dtype=torch.int32, device=device)
    start = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[start:start + n]
        start += n
    return table, num_pages


def sample_selection(q_pos: torch.Tensor, Hkv: int, topk: int, gen: torch.Generator,
                     shared: torch.Tensor | None = None,
                     boosted: torch.Tensor | None = None) -> torch.Tensor:
    """Draw block selections [R, Hkv, topk] int32 with the structure of MSA's top-k.

    Row r (query position q_pos[r]) keeps the sink block 0 and its local block
    q_pos//128, then topk-2 further causal blocks chosen uniformly without replacement
    from 1..local-1 -- except that a boosted (row, group) first takes the blocks of its
    ``shared`` set (a [R, Hkv, n_shared] tensor of candidate ids, -1 = none). Ids are
    ascending, then -1 padding when fewer causal blocks exist.

    This has the distribution of the top-k rule applied to iid continuous block scores in
    which the shared blocks of boosted rows get a bonus that ranks them above every other
    candidate, without computing any score.
    """
    device = q_pos.device
    R = q_pos.numel()
    local = (q_pos // BLOCK).to(torch.int64)
    nmax = int(local.max().item()) + 1
    ids = torch.arange(nmax, device=device)
    # priority: uniform noise in [0,1) for candidates 1..local-1; -1 for non-candidates
    pri = torch.rand((R, Hkv, nmax), generator=gen, device=device)
    cand = (ids[None, :] >= 1) & (ids[None, :] < local[:, None])  # [R, nmax]
    pri = torch.where(cand[:, None, :], pri, torch.full_like(pri, -1.0))
    if shared is not None and boosted is not None:
        sh = shared.to(torch.int64)
        valid = (sh >= 0) & boosted[..., None]
        bonus = torch.zeros_like(pri)
        bonus.scatter_(2, sh.clamp(min=0), valid.to(pri.dtype) * 2.0)
        pri = torch.where(pri >= 0, pri + bonus, pri)
    m = topk - 2
    if nmax >= 1 and m > 0:
        top_pri, top_id = torch.topk(pri, k=min(m, nmax), dim=2)
        top_id = torch.where(top_pri >= 0, top_id, torch.full_like(top_id, -1))
    else:
        top_id = torch.full((R, Hkv, 0), -1, dtype=torch.int64, device=device)
    sink = torch.zeros((R, Hkv, 1), dtype=torch.int64, device=device)
    loc = torch.where(local > 0, local, torch.full_like(local, -1))[:, None, None].expand(R, Hkv, 1)
    allids = torch.cat([sink, loc, top_id], dim=2)
    pad = topk - allids.shape[2]
    if pad > 0:
        allids = torch.cat([allids, torch.full((R, Hkv, pad), -1, dtype=torch.int64,
                                               device=device)], dim=2)
    # ascending ids with -1 padding last
    key = torch.where(allids >= 0, allids, torch.full_like(allids, 1 << 40))
    key, _ = torch.sort(key, dim=2)
    out = torch.where(key >= (1 << 40), torch.full_like(key, -1), key)
    return out.to(torch.int32).contiguous()


# ----------------------------------------------------------------------------- workloads

def index_workload(seq_lens, N: int, Hkv: int, Di: int, seed: int, device,
                   n_planted: int = 0, shuffle: bool = True):
    """Query index rows and a paged K-index cache.

    q_idx [B*N, Hkv, Di] bf16 ~N(0,1); k_idx_pages [P, 128, Hkv, Di] bf16 ~N(0,1);
    page_table random permutation. With ``n_planted`` > 0, for each (request, group)
    that many distinct blocks drawn from 1..nblk-2 get 2*q_idx (of the request's last
    query row) added to every token's key index: high-affinity blocks.
    Returns a dict; ``planted`` is [B, Hkv, n_planted] int64 (or None).
    """
    gen = _gen(seed, device)
    B = len(seq_lens)
    page_table, num_pages = paged_layout(seq_lens, gen, device, shuffle)
    q_idx = randn_bf16((B * N, Hkv, Di), gen, device)
    k_idx = randn_bf16((num_pages, BLOCK, Hkv, Di), gen, device)
    planted = None
    if n_planted > 0:
        planted = torch.empty((B, Hkv, n_planted), dtype=torch.int64, device=device)
        for b, s in enumerate(seq_lens):
            nb = (int(s) + BLOCK - 1) // BLOCK
            assert nb - 2 >= n_planted
            for g in range(Hkv):
                pick = torch.randperm(nb - 2, generator=gen, device=device)[:n_planted] + 1
                planted[b, g] = pick
                qv = q_idx[b * N + N - 1, g].to(torch.float32)
                for j in pick.tolist():
                    p = int(page_table[b, j].item())
                    blk = k_idx[p, :, g, :].to(torch.float32) + 2.0 * qv[None, :]
                    k_idx[p, :, g, :] = blk.to(torch.bfloat16)
    return {
        "q_idx": q_idx, "k_idx_pages": k_idx, "page_table": page_table,
        "seq_lens": torch.tensor([int(s) for s in seq_lens], dtype=torch.int32, device=device),
        "num_pages": num_pages, "B": B, "N": N, "Hkv": Hkv, "Di": Di, "planted": planted,
        "max_seq_len": max(int(s) for s in seq_lens),
    }


def decode_workload(seq_lens, N: int, Hq: int, Hkv: int, D: int, topk: int, seed: int,
                    device, shuffle: bool = True):
    """Paged K/V caches, decode queries and sampled block selections.

    q [B*N, Hq, D] bf16 ~N(0,1)/sqrt(D) (pre-scaled); k_cache, v_cache [P, 128, Hkv, D]
    bf16 ~N(0,1); block_ids [B*N, Hkv, topk] drawn by ``sample_selection``.
    """
    gen = _gen(seed, device)
    B = len(seq_lens)
    page_table, num_pages = paged_layout(seq_lens, gen, device, shuffle)
    q = randn_bf16((B * N, Hq, D), gen, device, scale=1.0 / math.sqrt(D))
    k_cache = randn_bf16((num_pages, BLOCK, Hkv, D), gen, device)
    v_cache = randn_bf16((num_pages, BLOCK, Hkv, D), gen, device)
    sl = torch.tensor([int(s) for s in seq_lens], dtype=torch.int64, device=device)
    q_pos = (sl[:, None] - N + torch.arange(N, device=device)[None, :]).reshape(-1)
    block_ids = sample_selection(q_pos, Hkv, topk, gen)
    return {
        "q": q, "k_cache": k_cache, "v_cache": v_cache, "page_table": page_table,
        "seq_lens": sl.to(torch.int32), "block_ids": block_ids, "num_pages": num_pages,
        "B": B, "N": N, "Hq": Hq, "Hkv": Hkv, "D": D, "topk": topk,
    }


def prefill_workload(T: int, S_kv: int, Hq: int, Hkv: int, D: int, topk: int, seed: int,
                     device, share_frac: float = 0.75, n_shared: int = 12):
    """Contiguous K/V, a chunk of T queries at positions S_kv-T.., clustered selections.

    q [T, Hq, D] bf16 ~N(0,1)/sqrt(D); k, v [S_kv, Hkv, D] bf16 ~N(0,1). For each
    (128-query span, group) a shared set of ``n_shared`` non-forced causal blocks is drawn;
    each (query, group) is boosted with probability ``share_frac`` and then keeps the
    shared set (plus random blocks); see ``sample_selection``.
    """
    gen = _gen(seed, device)
    q = randn_bf16((T, Hq, D), gen, device, scale=1.0 / math.sqrt(D))
    k = randn_bf16((S_kv, Hkv, D), gen, device)
    v = randn_bf16((S_kv, Hkv, D), gen, device)
    q_pos = torch.arange(S_kv - T, S_kv, device=device, dtype=torch.int64)
    span = (q_pos // BLOCK)
    spans = torch.unique(span)
    shared = torch.full((T, Hkv, n_shared), -1, dtype=torch.int64, device=device)
    if n_shared > 0:
        for s in spans.tolist():
            ncand = s - 1  # blocks 1..s-1 are the non-forced causal blocks of this span
            if ncand < 1:
                continue
            rows = (span == s).nonzero().flatten()
            for g in range(Hkv):
                pick = torch.randperm(ncand, generator=gen, device=device)[:n_shared] + 1
                shared[rows, g, :pick.numel()] = pick
    boosted = torch.rand((T, Hkv), generator=gen, device=device) < share_frac
    block_ids = sample_selection(q_pos, Hkv, topk, gen, shared=shared, boosted=boosted)
    return {"q": q, "k": k, "v": v, "block_ids": block_ids, "T": T, "S_kv": S_kv, "Hq": Hq,
            "Hkv": Hkv, "D": D, "topk": topk}


def layer_workload(T: int, Hq: int, Hkv: int, D: int, Di: int, seed: int, device,
                   decode_steps: int = 0):
    """A whole layer's inputs for one sequence with contiguous pages (identity table).

    Tokens 0..T+decode_steps-1 each have q (pre-scaled), k, v, q_idx, k_idx drawn once.
    The caches are paged with page p holding tokens 128p..128p+127, so the same storage
    serves the contiguous prefill view [S, Hkv, D] and the paged view [P, 128, Hkv, D].
    """
    gen = _gen(seed, device)
    S = T + decode_steps
    P = (S + BLOCK - 1) // BLOCK
    cap = P * BLOCK
    q = randn_bf16((S, Hq, D), gen, device, scale=1.0 / math.sqrt(D))
    k = randn_bf16((cap, Hkv, D), gen, device)
    v = randn_bf16((cap, Hkv, D), gen, device)
    q_idx = randn_bf16((S, Hkv, Di), gen, device)
    k_idx = randn_bf16((cap, Hkv, Di), gen, device)
    return {"q": q, "k": k, "v": v, "q_idx": q_idx, "k_idx": k_idx, "T": T, "S": S, "P": P,
            "Hq": Hq, "Hkv": Hkv, "D": D, "Di": Di,
            "page_table": torch.arange(P, dtype=torch.int32, device=device)[None, :]}


# ----------------------------------------------------------------------------- named configs

def tiny_layer(device, seed: int = 0):
    """Tiny layer: 2048 tokens (16 blocks), Hq=8, Hkv=2, D=128, Di=64, k=4, 16 decode steps."""
    w = layer_workload(2048, 8, 2, 128, 64, seed, device, decode_steps=16)
    w["topk"] = 4
    return w


DECODE_SCORING = dict(B=8, seq_len=60032, Hkv=8, Di=128, topk=16, n_planted=8)


def decode_scoring(device, seed: int = 2, B: int | None = None, seq_len: int | None = None):
    """Decode index scoring: 8 requests x 60032 tokens (469 blocks), Hkv=8, Di=128, k=16."""
    B = B or DECODE_SCORING["B"]
    seq_len = seq_len or DECODE_SCORING["seq_len"]
    w = index_workload([seq_len] * B, 1, DECODE_SCORING["Hkv"], DECODE_SCORING["Di"], seed, device,
                       n_planted=DECODE_SCORING["n_planted"])
    w["topk"] = DECODE_SCORING["topk"]
    return w


CAUSAL_PREFILL = dict(T=32768, Hq=64, Hkv=8, D=128, topk=16)


def causal_prefill(device, seed: int = 3, T: int | None = None):
    """Block-major sparse prefill: 32768-token causal chunk, Hq=64, Hkv=8, D=128, k=16."""
    T = T or CAUSAL_PREFILL["T"]
    return prefill_workload(T, T, CAUSAL_PREFILL["Hq"], CAUSAL_PREFILL["Hkv"], CAUSAL_PREFILL["D"], CAUSAL_PREFILL["topk"], seed, device)


PAGED_DECODE = dict(B=64, lo=8192, hi=131072, Hq=64, Hkv=8, D=128, topk=16)


def paged_decode_seq_lens(seed: int, B: int, lo: int, hi: int):
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


def paged_decode(device, seed: int = 4, B: int | None = None):
    """Paged sparse decode: 64 requests, context ~U[8192, 131072], Hq=64, Hkv=8, D=128, k=16."""
    B = B or PAGED_DECODE["B"]
    lens = paged_decode_seq_lens(seed, B, PAGED_DECODE["lo"], PAGED_DECODE["hi"])
    return decode_workload(lens, 1, PAGED_DECODE["Hq"], PAGED_DECODE["Hkv"], PAGED_DECODE["D"], PAGED_DECODE["topk"], seed, device)


LONG_CONTEXT = dict(B=4, seq_len=1 << 20, Hq=64, Hkv=8, D=128, Di=128, topk=32, T_prefill=32768)


def paged_layer_workload(seq_lens, Hq: int, Hkv: int, D: int, Di: int, seed: int, device,
                         shuffle: bool = True):
    """Decode-time layer state for B requests sharing one page table: paged K-index, K and V
    caches [P, 128, Hkv, *] bf16 ~N(0,1), and one query row per request (q pre-scaled, q_idx)."""
    gen = _gen(seed, device)
    B = len(seq_lens)
    page_table, num_pages = paged_layout(seq_lens, gen, device, shuffle)
    q = randn_bf16((B, Hq, D), gen, device, scale=1.0 / math.sqrt(D))
    q_idx = randn_bf16((B, Hkv, Di), gen, device)
    k_idx = randn_bf16((num_pages, BLOCK, Hkv, Di), gen, device)
    k_cache = randn_bf16((num_pages, BLOCK, Hkv, D), gen, device)
    v_cache = randn_bf16((num_pages, BLOCK, Hkv, D), gen, device)
    return {"q": q, "q_idx": q_idx, "k_idx_pages": k_idx, "k_cache": k_cache, "v_cache": v_cache,
            "page_table": page_table, "num_pages": num_pages,
            "seq_lens": torch.tensor([int(s) for s in seq_lens], dtype=torch.int32, device=device),
            "B": B, "Hq": Hq, "Hkv": Hkv, "D": D, "Di": Di}


def chunk_prefill_workload(prefix: int, T: int, Hq: int, Hkv: int, D: int, Di: int, seed: int,
                           device):
    """A T-token prefill chunk after a `prefix`-token context of one sequence: contiguous K, V and
    K-index for all S = prefix + T tokens (the K-index is also the paged cache with the identity
    page table), queries q / q_idx for the chunk only."""
    gen = _gen(seed, device)
    S = prefix + T
    P = (S + BLOCK - 1) // BLOCK
    cap = P * BLOCK
    q = randn_bf16((T, Hq, D), gen, device, scale=1.0 / math.sqrt(D))
    q_idx = randn_bf16((T, Hkv, Di), gen, device)
    k = randn_bf16((cap, Hkv, D), gen, device)
    v = randn_bf16((cap, Hkv, D), gen, device)
    k_idx = randn_bf16((cap, Hkv, Di), gen, device)
    return {"q": q, "q_idx": q_idx, "k": k, "v": v, "k_idx": k_idx, "S": S, "T": T, "P": P,
            "Hq": Hq, "Hkv": Hkv, "D": D, "Di": Di,
            "page_table": torch.arange(P, dtype=torch.int32, device=device)[None, :]}


def long_context_decode(device, seed: int = 5, B: int | None = None, seq_len: int | None = None):
    """1M-token decode: 4 requests x 1,048,576 tokens, Hq 64, Hkv 8, D 128, Di 128, k 32."""
    c = LONG_CONTEXT
    w = paged_layer_workload([seq_len or c["seq_len"]] * (B or c["B"]), c["Hq"], c["Hkv"], c["D"],
                             c["Di"], seed, device)
    w["topk"] = c["topk"]
    return w


def long_context_prefill(device, seed: int = 6, T: int | None = None, prefix: int | None = None):
    """32768-token prefill chunk after a 1,048,576-token prefix, Hq 64, Hkv 8, D 128, Di 128, k 32."""
    c = LONG_CONTEXT
    w = chunk_prefill_workload(prefix if prefix is not None else c["seq_len"], T or c["T_prefill"],
                               c["Hq"], c["Hkv"], c["D"], c["Di"], seed, device)
    w["topk"] = c["topk"]
    return w
