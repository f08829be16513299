// Stage 1 of MSA: index scoring with a fused per-block max, and top-k block selection.
//
// Together AI MiniMax-M3 serving article, section "The index scorer becomes the decode
// critical path": every decode query compares its query-side index vector with the
// key-side index vectors of all candidate 128-token blocks, each block is reduced to one
// score and only the top blocks are kept. The shape is a small query index against a long
// key index; the pages stage each 128-token K-index page with asynchronous copies, prefetch
// the next page, take bf16 dot products and reduce each page to one block score.
//
// GB300 design. At decode the scorer is a streaming read of the whole paged K-index (one
// byte read per flop), so it is written for HBM bandwidth, not for tensor cores:
//  * one persistent CTA per SM walks a contiguous range of the batch's (request, page)
//    list; a producer warp streams each page through a ring of TMA stages (256 index rows
//    of all KV groups per stage, 128-byte swizzle so that 32 lanes reading 32 different
//    rows hit 32 different bank groups);
//  * each consumer thread owns one (token, group) row per stage and takes its full dot
//    product with every query row of the request in fp32 (exact bf16 products), keeping a
//    running max per query row; a shuffle + shared-memory reduction turns the page into
//    one score per (query row, group);
//  * the top-k is fused: the CTA that completes a request's last page (an atomic ticket
//    per request, no spinning) selects the blocks of every (query row, group) of that
//    request with a warp-level radix select.
// Long query chunks (prefill, N > 8) are a dense contraction and run on the tensor cores
// (tcgen05, accumulators in tensor memory), writing every visible block score; the same warp
// top-k follows in a separate launch.
#include "common.cuh"
#include "host_util.h"
#include "kernels.h"
#include "page_table_row.cuh"

MSA_DEFINE_ERROR_WORD(score)

namespace msa {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kStageRows = 256;
constexpr int kTopkMax = 64;

struct TopkScratch {
  uint32_t hist[256];
  int32_t sel[kTopkMax];
};

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Top-k of one (query row, group), executed by one full warp.
// s: the row's block scores (global, written by other CTAs: read with ld.global.cg).
// Blocks 0 and `local` are forced; the remaining slots take blocks 1..local-1 by score
// descending with ties to the lower id (radix select on order-preserving keys, then the
// lowest ids among the keys equal to the threshold). Writes ids ascending, -1 padding.
// KR > 0 (a warp running one top-k at the tail of the decode scorer, where its latency is
// exposed): rows of up to 1 + 32*KR blocks keep their candidate keys in registers (lane l's
// k-th key is block 1 + l + 32k), longer rows request 8 keys per lane before counting them.
// KR = 0 (the multi-row top-k kernel, which hides latency with many resident warps): each
// pass reads the keys one per lane per step, keeping the register count and occupancy low.
// Every pass checks j < local, so padding keys are never counted.
template <int KR>
__device__ void warp_topk(const float* __restrict__ s, int local, int topk, int32_t* ids_out,
                          float* sc_out, TopkScratch& ws) {
  const int lane = threadIdx.x & 31;
  const uint32_t full = 0xffffffffu;
  const int nforced = local > 0 ? 2 : 1;
  const int ncand = local > 1 ? local - 1 : 0;
  int m = topk - nforced;
  if (m > ncand) m = ncand;
  if (m < 0) m = 0;
  if (lane == 0) {
    ws.sel[0] = 0;
    if (local > 0) ws.sel[1] = local;
  }
  if (m == ncand) {
    for (int j = 1 + lane; j < local; j += 32) ws.sel[nforced + j - 1] = j;
  } else if (m > 0) {
    // A row that fits is read once into registers (all loads in flight together); a longer
    // row is re-read per pass, 8 keys per lane requested before any is counted.
    const bool in_regs = KR > 0 && ncand <= 32 * KR;
    uint32_t kr[KR > 0 ? KR : 1];
    if (in_regs) {
#pragma unroll
      for (int k = 0; k < KR; ++k) {
        const int j = 1 + lane + 32 * k;
        kr[k] = j < local ? float_key(__ldcg(s + j)) : 0u;
      }
    }
    uint32_t prefix = 0, pmask = 0;
    int remaining = m;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int b = lane; b < 256; b += 32) ws.hist[b] = 0;
      __syncwarp();
      if (in_regs) {
#pragma unroll
        for (int k = 0; k < KR; ++k) {
          const int j = 1 + lane + 32 * k;
          if (j < local && (kr[k] & pmask) == prefix) atomicAdd(&ws.hist[(kr[k] >> shift) & 255u], 1u);
        }
      } else if (KR == 0) {
        for (int j = 1 + lane; j < local; j += 32) {
          const uint32_t key = float_key(__ldcg(s + j));
          if ((key & pmask) == prefix) atomicAdd(&ws.hist[(key >> shift) & 255u], 1u);
        }
      } else {
        for (int j0 = 1; j0 < local; j0 += 32 * 8) {
          uint32_t kb[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int j = j0 + lane + 32 * u;
            kb[u] = j < local ? float_key(__ldcg(s + j)) : 0u;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int j = j0 + lane + 32 * u;
            if (j < local && (kb[u] & pmask) == prefix) atomicAdd(&ws.hist[(kb[u] >> shift) & 255u], 1u);
          }
        }
      }
      __syncwarp();
      // lane l owns digits 255-8l .. 248-8l (descending)
      int c[8], sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        c[q] = (int)ws.hist[255 - (lane * 8 + q)];
        sum += c[q];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(full, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - sum;
      const uint32_t bal = __ballot_sync(full, excl < remaining && incl >= remaining);
      const int src = __ffs(bal) - 1;
      int digit = 0, above = 0;
      if (lane == src) {
        int acc = excl;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (acc + c[q] >= remaining) {
            digit = 255 - (lane * 8 + q);
            above = acc;
            break;
          }
          acc += c[q];
        }
      }
      digit = __shfl_sync(full, digit, src);
      above = __shfl_sync(full, above, src);
      remaining -= above;
      prefix |= (uint32_t)digit << shift;
      pmask |= 255u << shift;
      __syncwarp();
    }
    // prefix is the threshold key; take every key above it and the `remaining` lowest
    // ids among the keys equal to it (ids ascending: 32 consecutive ids per step).
    int base = nforced, eq_seen = 0;
    for (int j0 = 1, k = 0; j0 < local; j0 += 32, ++k) {
      const int j = j0 + lane;
      uint32_t key = 0u;
      if (in_regs) {
#pragma unroll
        for (int t = 0; t < KR; ++t) key = t == k ? kr[t] : key;
      } else {
        key = j < local ? float_key(__ldcg(s + j)) : 0u;
      }
      const bool gt = j < local && key > prefix;
      const bool eq = j < local && key == prefix;
      const uint32_t eqm = __ballot_sync(full, eq);
      const int eqrank = eq_seen + __popc(eqm & lanemask_lt());
      const bool take = gt || (eq && eqrank < remaining);
      const uint32_t tm = __ballot_sync(full, take);
      const int dst = base + __popc(tm & lanemask_lt());
      if (take && dst < kTopkMax) ws.sel[dst] = j;
      base += __popc(tm);
      eq_seen += __popc(eqm);
    }
  }
  __syncwarp();
  const int nsel = nforced + m;
  // rank sort of the (distinct) kept ids, then write ids and their scores
  for (int k = lane; k < topk; k += 32) {
    if (k < nsel) {
      const int e = ws.sel[k];
      int rank = 0;
      for (int q = 0; q < nsel; ++q) rank += ws.sel[q] < e;
      ids_out[rank] = e;
      if (sc_out) sc_out[rank] = __ldcg(s + e);
    } else {
      ids_out[k] = -1;
      if (sc_out) sc_out[k] = -INFINITY;
    }
  }
  __syncwarp();
}

struct DecodeSmemLayout {
  uint32_t stage_bytes, q_off, red_off, topk_off, bar_off, misc_off, total;
};

__host__ __device__ inline DecodeSmemLayout decode_layout(int N, int Hkv, int Di, int nstage) {
  DecodeSmemLayout L;
  const int rows = kStageRows < 128 * Hkv ? kStageRows : 128 * Hkv;
  L.stage_bytes = (uint32_t)(rows * Di * 2);
  uint32_t off = L.stage_bytes * (uint32_t)nstage;           // stages at offset 0 (1024-aligned)
  L.q_off = off;
  off += (uint32_t)(N * Hkv * (Di + 4) * 4);
  L.red_off = off;
  off += (uint32_t)(2 * kConsumerWarps * N * Hkv * 4);  // double-buffered by page parity
  off = (off + 15u) & ~15u;
  L.topk_off = off;
  off += (uint32_t)(kConsumerWarps * sizeof(TopkScratch));
  off = (off + 7u) & ~7u;
  L.bar_off = off;
  off += (uint32_t)(2 * nstage * 8);
  L.misc_off = off;
  off += 64;
  L.total = off + 1024;  // slack for aligning the base to 1024 bytes
  return L;
}

struct DecodeKParams {
  const uint16_t* q_idx;
  const int32_t* page_table;
  const int32_t* seq_lens;
  int32_t B, N, Hkv, max_blocks, topk, nstage;
  int64_t num_pages;
  int32_t* block_ids;
  float* sel_scores;
  float* scores;
  int32_t* tickets;
  int32_t* fpt;        // optional: flat page table [B*N*Hkv, topk] built in the tail (row a3)
  int32_t* fpt_lens;   // optional: [B*N*Hkv]
};

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

template <int DI, int NQ>
__global__ void __launch_bounds__(kThreads, 1)
    score_decode_kernel(const __grid_constant__ CUtensorMap kmap, const DecodeKParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int Hkv = p.Hkv, N = p.N, nstage = p.nstage;
  const DecodeSmemLayout L = decode_layout(N, Hkv, DI, nstage);
  float* sq = reinterpret_cast<float*>(smem + L.q_off);
  float* sred = reinterpret_cast<float*>(smem + L.red_off);
  TopkScratch* stopk = reinterpret_cast<TopkScratch*>(smem + L.topk_off);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty_bar = full_bar + nstage;
  int32_t* misc = reinterpret_cast<int32_t*>(smem + L.misc_off);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rows = kStageRows < 128 * Hkv ? kStageRows : 128 * Hkv;
  const int stages_per_page = (128 * Hkv) / rows;
  const int tok_per_stage = rows / Hkv;

  // ---- range of (request, page) items of this CTA: warp 0 scans the request lengths
  if (warp == 0) {
    int total = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      bool bad = false;
      const int nb = b < p.B ? (clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) + 127) / 128 : 0;
      if (bad && blockIdx.x == 0) msa_record_error(kErrBadBlock);
      total += __reduce_add_sync(0xffffffffu, nb);
    }
    const int per = (total + (int)gridDim.x - 1) / (int)gridDim.x;
    const int p0 = min(total, (int)blockIdx.x * per);
    const int p1 = min(total, p0 + per);
    // locate the request holding item p0
    int run = 0, b_start = p.B, j_start = 0;
    for (int b0 = 0; b0 < p.B && b_start == p.B; b0 += 32) {
      const int b = b0 + lane;
      bool bad = false;
      const int nb = b < p.B ? (clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) + 127) / 128 : 0;
      int incl = nb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - nb;
      const uint32_t hit = __ballot_sync(0xffffffffu, b < p.B && run + excl <= p0 && p0 < run + incl);
      if (hit) {
        const int src = __ffs(hit) - 1;
        b_start = b0 + src;
        j_start = p0 - run - __shfl_sync(0xffffffffu, excl, src);
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      misc[0] = p0;
      misc[1] = p1;
      misc[2] = b_start;
      misc[3] = j_start;
      misc[5] = 0;  // set to 1 by any consumer whose bounded wait gave up
    }
  }
  if (tid == kConsumers) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    mbar_fence_init();
  }
  __syncthreads();
  const int p0 = misc[0], p1 = misc[1];
  if (p0 >= p1) return;

  if (warp == kConsumerWarps) {
    // ================================ producer warp
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      int b = misc[2], j = misc[3];
      bool bad = false;
      int nb = (clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) + 127) / 128;
      uint32_t it = 0;
      for (int item = p0; item < p1; ++item) {
        int32_t page = p.page_table[(int64_t)b * p.max_blocks + j];
        if (page < 0 || page >= p.num_pages) {
          msa_record_error(kErrBadPage);
          page = 0;
        }
        for (int sp = 0; sp < stages_per_page; ++sp, ++it) {
          const uint32_t slot = it % nstage;
          if (it >= (uint32_t)nstage && !mbar_wait(&empty_bar[slot], ((it / nstage) - 1) & 1)) {
            msa_record_error(kErrTimeout);
            // let the copies already issued land before the CTA exits (bounded)
            for (uint32_t k = it - nstage + 1; k < it; ++k)
              mbar_wait(&full_bar[k % nstage], (k / nstage) & 1);
            return;
          }
          uint8_t* dst = smem + slot * L.stage_bytes;
          mbar_expect_tx(&full_bar[slot], L.stage_bytes);
          const int32_t row = (int32_t)((int64_t)page * 128 * Hkv + (int64_t)sp * rows);
          tma_load_2d(dst, &kmap, &full_bar[slot], 0, row);
          if (DI == 128) tma_load_2d(dst + rows * 128, &kmap, &full_bar[slot], 64, row);
        }
        if (++j == nb) {
          j = 0;
          ++b;
          if (b < p.B) nb = (clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) + 127) / 128;
        }
      }
      // wait for the copies still in flight before the CTA may exit
      for (uint32_t k = (it > (uint32_t)nstage ? it - nstage : 0); k < it; ++k)
        if (!mbar_wait(&empty_bar[k % nstage], (k / nstage) & 1)) msa_record_error(kErrTimeout);
    }
    return;
  }

  // ================================== consumer warps
  int b = misc[2], j = misc[3];
  bool bad = false;
  int nb = (clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) + 127) / 128;
  int cur_b = -1, done_pages = 0, page_par = 0;
  int qpos[NQ];
  uint32_t it = 0;
  const int g = tid % Hkv;
  const bool has_row = tid < rows;

  auto finish_request = [&](int rb, int count) {
    // make this CTA's block scores of request rb visible device-wide, then publish its share
    if (tid < N * Hkv) __threadfence();
    consumer_sync();
    if (tid == 0) {
      bool bad_r = false;
      const int nbr = (clamp_seq(p.seq_lens, rb, N, p.max_blocks, bad_r) + 127) / 128;
      const int old = atomicAdd(&p.tickets[rb], count);
      misc[4] = (old + count == nbr) ? 1 : 0;
    }
    consumer_sync();
    if (misc[4]) {
      __threadfence();
      for (int item = warp; item < N * Hkv; item += kConsumerWarps) {
        const int i = item / Hkv, gg = item % Hkv;
        const int64_t r = (int64_t)rb * N + i;
        bool bad_r = false;
        const int qp = clamp_seq(p.seq_lens, rb, N, p.max_blocks, bad_r) - N + i;
        const int64_t orow = (r * Hkv + gg) * p.topk;
        warp_topk<16>(p.scores + (r * Hkv + gg) * p.max_blocks, qp / 128, p.topk, p.block_ids + orow,
                  p.sel_scores ? p.sel_scores + orow : nullptr, stopk[warp]);
        if (p.fpt) {
          // the sparse page table row of the selection just written (same warp: ordered by
          // the warp barrier)
          __syncwarp();
          const uint32_t err = warp_flat_page_table_row(
              p.block_ids + orow, p.page_table + (int64_t)rb * p.max_blocks, qp, Hkv, gg, p.topk,
              p.max_blocks, p.num_pages, p.fpt + orow, p.fpt_lens + r * Hkv + gg);
          if (err) msa_record_error(err);
        }
      }
    }
    consumer_sync();
  };

  for (int item = p0; item < p1; ++item) {
    if (b != cur_b) {
      if (cur_b >= 0) finish_request(cur_b, done_pages);
      cur_b = b;
      done_pages = 0;
      // query index rows of request b -> fp32 shared memory (rows padded by 4 floats)
      const uint16_t* qsrc = p.q_idx + (int64_t)b * N * Hkv * DI;
      for (int e = tid; e < N * Hkv * DI; e += kConsumers) {
        const int row = e / DI, d = e % DI;
        sq[row * (DI + 4) + d] = __uint_as_float((uint32_t)qsrc[e] << 16);
      }
#pragma unroll
      for (int i = 0; i < NQ; ++i)
        qpos[i] = clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) - N + i;
      consumer_sync();
    }
    float rm[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) rm[i] = -INFINITY;

    for (int sp = 0; sp < stages_per_page; ++sp, ++it) {
      const uint32_t slot = it % nstage;
      // A failed wait is recorded and the thread keeps following the same barriers as
      // the others; the CTA leaves the loop together after the page-end barrier.
      const bool ok = mbar_wait(&full_bar[slot], (it / nstage) & 1);
      if (!ok) {
        msa_record_error(kErrTimeout);
        misc[5] = 1;
      }
      if (ok && has_row) {
        const uint8_t* st = smem + slot * L.stage_bytes;
        const int tok = sp * tok_per_stage + tid / Hkv;
        const int pos = j * 128 + tok;
        float acc[NQ];
#pragma unroll
        for (int i = 0; i < NQ; ++i) acc[i] = 0.0f;
#pragma unroll
        for (int h = 0; h < DI / 64; ++h) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 kv = *reinterpret_cast<const uint4*>(st + h * rows * 128 + sw128(tid, c));
            float kf[8] = {bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y),
                           bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w)};
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
              if (i < N) {
                const float* qr = sq + (i * Hkv + g) * (DI + 4) + h * 64 + c * 8;
                const float4 qa = *reinterpret_cast<const float4*>(qr);
                const float4 qb = *reinterpret_cast<const float4*>(qr + 4);
                acc[i] = fmaf(qa.x, kf[0], acc[i]);
                acc[i] = fmaf(qa.y, kf[1], acc[i]);
                acc[i] = fmaf(qa.z, kf[2], acc[i]);
                acc[i] = fmaf(qa.w, kf[3], acc[i]);
                acc[i] = fmaf(qb.x, kf[4], acc[i]);
                acc[i] = fmaf(qb.y, kf[5], acc[i]);
                acc[i] = fmaf(qb.z, kf[6], acc[i]);
                acc[i] = fmaf(qb.w, kf[7], acc[i]);
              }
            }
          }
        }
#pragma unroll
        for (int i = 0; i < NQ; ++i)
          if (i < N && pos <= qpos[i]) rm[i] = fmaxf(rm[i], acc[i]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[slot]);
    }
    // ---- page end: max over the page's tokens for each (query row, group)
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      if (i < N) {
        float v = rm[i];
        for (int off = 16; off >= Hkv; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
        if (lane < Hkv) sred[((page_par * kConsumerWarps + warp) * N + i) * Hkv + lane] = v;
      }
    }
    consumer_sync();
    if (misc[5]) return;  // uniform: read by every consumer after the same barrier
    if (tid < N * Hkv) {
      float v = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w)
        v = fmaxf(v, sred[(page_par * kConsumerWarps + w) * N * Hkv + tid]);
      const int i = tid / Hkv, gg = tid % Hkv;
      const int64_t r = (int64_t)b * N + i;
      p.scores[(r * Hkv + gg) * p.max_blocks + j] = v;
    }
    page_par ^= 1;  // the other half of sred is free: its readers passed this page's barrier
    ++done_pages;
    if (++j == nb) {
      j = 0;
      ++b;
      if (b < p.B) nb = (clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) + 127) / 128;
    }
  }
  if (cur_b >= 0) finish_request(cur_b, done_pages);
}

// ---------------------------------------------------------------------------------------
// Multi-row scorer (N > 8: a prefill chunk, or many draft rows) on the tensor cores.
//
// The scores of one (request, group) are the product of the request's query-index rows
// (N x Di) with the transposed key-index rows of every visible block, reduced by a max over
// each block's 128 keys: a dense contraction, so it runs as tcgen05 MMAs with the accumulator
// in tensor memory. A work item is (request, group, chunk of kScoreChunk = 4 consecutive
// blocks). Its 4 key blocks (512 keys) stay in shared memory while the query rows that can see
// them stream through in 128-row tiles; one tile is two M=128, N=256 MMA groups into the two
// halves of tensor memory. Each key-index row is read from HBM once; the query rows of a
// (request, group) are re-read from L2 by every chunk (all CTAs sweep the same request and
// group at the same time).
//
// Warp 0 issues the TMA copies, warp 1 the MMAs, and warps 2..9 form two epilogue
// warpgroups: warpgroup h drains accumulator half h (blocks 2h and 2h+1 of the chunk), one
// query row per thread, applies the causal mask on the row's own (local) block and writes one
// max per block. While one half is drained the MMAs of the other half run.
constexpr int kScoreChunk = 4;                            // key blocks per work item
constexpr int kScThreads = 320;
constexpr int kScQStages = 3;

template <int DI>
struct ScoreTcLayout {
  static constexpr uint32_t kBox = 128 * 64 * 2;           // 128 rows x 64 channels = 16 KB
  static constexpr int kBoxes = DI / 64;
  static constexpr uint32_t kQTile = kBoxes * kBox;
  static constexpr uint32_t kKHalfBox = kScoreChunk * kBox;  // one 64-channel box of 4 blocks
  static constexpr uint32_t kOffK = 0;
  static constexpr uint32_t kOffQ = kBoxes * kKHalfBox;
  static constexpr uint32_t kOffBar = kOffQ + kScQStages * kQTile;
  static constexpr size_t kSmem = 1024 + kOffBar + 256;
};

struct ScoreTcBars {
  uint64_t k_full, k_empty;
  uint64_t q_full[kScQStages], q_empty[kScQStages];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_base;
  int32_t fail;
};

struct ScoreTcParams {
  const int32_t* page_table;
  const int32_t* seq_lens;
  int32_t B, N, Hkv, max_blocks, max_chunks;
  int64_t num_pages;
  float* scores;
};

// Query-row tiles of work item (b, c): rows whose position can see a key of blocks
// 4c..4c+3, in 128-row tiles counted from the request's first row. Returns the tile count.
__device__ __forceinline__ int item_tiles(const ScoreTcParams& p, int b, int c, int seq, int& t_lo) {
  const int nblk = (seq + 127) / 128;
  if (c * kScoreChunk >= nblk) return 0;
  const int first_row = c * kScoreChunk * 128 - (seq - p.N);  // first row seeing the chunk
  t_lo = first_row <= 0 ? 0 : first_row / 128;
  const int t_end = (p.N + 127) / 128;
  return t_end - t_lo;
}

__device__ __forceinline__ bool sc_wait(uint64_t* bar, uint32_t parity, volatile int32_t* fail) {
  if (*fail) return false;
  if (mbar_wait(bar, parity)) return true;
  msa_record_error(kErrTimeout);
  *fail = 1;
  return false;
}

template <int DI>
__global__ void __launch_bounds__(kScThreads, 1)
    score_rows_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                         const __grid_constant__ CUtensorMap kmap, const ScoreTcParams p) {
  using L = ScoreTcLayout<DI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  ScoreTcBars& Bz = *reinterpret_cast<ScoreTcBars*>(smem + L::kOffBar);
  volatile int32_t* fail = &Bz.fail;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t n_items = (int64_t)p.B * p.Hkv * p.max_chunks;

  if (tid == 0) {
    mbar_init(&Bz.k_full, 1);
    mbar_init(&Bz.k_empty, 1);
    for (int q = 0; q < kScQStages; ++q) {
      mbar_init(&Bz.q_full[q], 1);
      mbar_init(&Bz.q_empty[q], 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&Bz.acc_full[h], 1);
      mbar_init(&Bz.acc_empty[h], 4);
    }
    Bz.fail = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&Bz.tmem_base)), "n"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = Bz.tmem_base;
  const uint32_t sbase = smem_u32(smem);

  // Items in (request, group, chunk) order, dealt round-robin: all CTAs work on the chunks of
  // one (request, group) at a time, so its query rows stay in L2.
  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      int items_done = 0, tiles_done = 0;
      for (int64_t it = blockIdx.x; it < n_items && !*fail; it += gridDim.x) {
        const int c = (int)(it % p.max_chunks);
        const int g = (int)((it / p.max_chunks) % p.Hkv);
        const int b = (int)(it / ((int64_t)p.max_chunks * p.Hkv));
        bool bad = false;
        const int seq = clamp_seq(p.seq_lens, b, p.N, p.max_blocks, bad);
        if (bad && g == 0 && c == 0) msa_record_error(kErrBadBlock);
        int t_lo = 0;
        const int nt = item_tiles(p, b, c, seq, t_lo);
        if (nt <= 0) continue;
        if (items_done > 0 && !sc_wait(&Bz.k_empty, (items_done - 1) & 1, fail)) break;
        const int nblk = (seq + 127) / 128;
        const int j0 = c * kScoreChunk;
        const int nvalid = min(kScoreChunk, nblk - j0);
        mbar_expect_tx(&Bz.k_full, (uint32_t)(nvalid * L::kBoxes) * L::kBox);
        for (int s = 0; s < nvalid; ++s) {
          int32_t page = p.page_table[(int64_t)b * p.max_blocks + j0 + s];
          if (page < 0 || page >= p.num_pages) {
            msa_record_error(kErrBadPage);
            page = 0;
          }
          for (int h = 0; h < L::kBoxes; ++h)
            tma_load_3d(smem + L::kOffK + h * L::kKHalfBox + s * L::kBox, &kmap, &Bz.k_full,
                        h * 64, g, page * 128);
        }
        for (int t = 0; t < nt; ++t, ++tiles_done) {
          const int qs = tiles_done % kScQStages;
          if (tiles_done >= kScQStages &&
              !sc_wait(&Bz.q_empty[qs], (tiles_done / kScQStages - 1) & 1, fail))
            break;
          mbar_expect_tx(&Bz.q_full[qs], L::kQTile);
          const int row = b * p.N + (t_lo + t) * 128;
          for (int h = 0; h < L::kBoxes; ++h)
            tma_load_3d(smem + L::kOffQ + qs * L::kQTile + h * L::kBox, &qmap, &Bz.q_full[qs],
                        h * 64, g, row);
        }
        ++items_done;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(128, 256, 0, 0);  // Q (K-major) x K (K-major)
      int items_done = 0, tiles_done = 0;
      for (int64_t it = blockIdx.x; it < n_items && !*fail; it += gridDim.x) {
        const int c = (int)(it % p.max_chunks);
        const int b = (int)(it / ((int64_t)p.max_chunks * p.Hkv));
        bool bad = false;
        const int seq = clamp_seq(p.seq_lens, b, p.N, p.max_blocks, bad);
        int t_lo = 0;
        const int nt = item_tiles(p, b, c, seq, t_lo);
        if (nt <= 0) continue;
        if (!sc_wait(&Bz.k_full, items_done & 1, fail)) break;
        for (int t = 0; t < nt; ++t, ++tiles_done) {
          const int qs = tiles_done % kScQStages;
          if (!sc_wait(&Bz.q_full[qs], (tiles_done / kScQStages) & 1, fail)) break;
          const uint32_t qa = sbase + L::kOffQ + qs * L::kQTile;
          for (int h = 0; h < 2; ++h) {
            if (tiles_done > 0 && !sc_wait(&Bz.acc_empty[h], (tiles_done - 1) & 1, fail)) break;
            tmem_fence_after();
            const uint32_t ka = sbase + L::kOffK + h * 2 * L::kBox;  // blocks 2h, 2h+1
#pragma unroll
            for (int kk = 0; kk < DI / 16; ++kk) {
              const uint32_t a_off = (kk >> 2) * L::kBox + (kk & 3) * 32;
              const uint32_t b_off = (kk >> 2) * L::kKHalfBox + (kk & 3) * 32;
              umma_bf16(tmem + h * 256, umma_desc_sw128(qa + a_off, 16, 1024),
                        umma_desc_sw128(ka + b_off, 16, 1024), idesc, kk > 0);
            }
            umma_commit(&Bz.acc_full[h]);
          }
          if (*fail) break;
          umma_commit(&Bz.q_empty[qs]);
        }
        if (*fail) break;
        umma_commit(&Bz.k_empty);
        ++items_done;
      }
    }
    __syncwarp();
  } else {
    // ================================================================ epilogue (warps 2..9)
    const int h = (warp - 2) >> 2;                    // accumulator half = warpgroup
    const int row = 32 * (warp & 3) + lane;           // tile row = TMEM lane
    const uint32_t acc = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + h * 256;
    int tiles_done = 0;
    for (int64_t it = blockIdx.x; it < n_items && !*fail; it += gridDim.x) {
      const int c = (int)(it % p.max_chunks);
      const int g = (int)((it / p.max_chunks) % p.Hkv);
      const int b = (int)(it / ((int64_t)p.max_chunks * p.Hkv));
      bool bad = false;
      const int seq = clamp_seq(p.seq_lens, b, p.N, p.max_blocks, bad);
      int t_lo = 0;
      const int nt = item_tiles(p, b, c, seq, t_lo);
      if (nt <= 0) continue;
      const int nblk = (seq + 127) / 128;
      for (int t = 0; t < nt; ++t, ++tiles_done) {
        if (!sc_wait(&Bz.acc_full[h], tiles_done & 1, fail)) break;
        tmem_fence_after();
        const int i = (t_lo + t) * 128 + row;          // row within the request
        const int qp = seq - p.N + i;                  // its query position
        float best[2];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          float v[128];
#pragma unroll
          for (int x = 0; x < 4; ++x) tmem_ld32(acc + s * 128 + x * 32, v + x * 32);
          tmem_wait_ld();
          if (s == 1) {  // both blocks are in registers: hand the accumulator half back
            tmem_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&Bz.acc_empty[h]);
          }
          const int j = c * kScoreChunk + 2 * h + s;
          // causal mask: only the row's own block holds keys after the query
          const int lim = qp - j * 128;                // last visible column
          if (lim < 127) {
#pragma unroll
            for (int x = 0; x < 128; ++x)
              if (x > lim) v[x] = -INFINITY;
          }
          float m8[8];
#pragma unroll
          for (int r = 0; r < 8; ++r) m8[r] = v[r];
#pragma unroll
          for (int x = 8; x < 128; ++x) m8[x & 7] = fmaxf(m8[x & 7], v[x]);
          best[s] = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                          fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        }
        if (i < p.N) {
          const int64_t r = (int64_t)b * p.N + i;
          float* dst = p.scores + (r * p.Hkv + g) * p.max_blocks;
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const int j = c * kScoreChunk + 2 * h + s;
            if (j < nblk && j * 128 <= qp) dst[j] = best[s];
          }
        }
      }
    }
  }
  // ------------------------------------------------------------------ teardown
  tmem_fence_before();
  __syncthreads();
  if (warp == 1) {
    tmem_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(512)
                 : "memory");
  }
}

__global__ void __launch_bounds__(256) topk_rows_kernel(const ScoreArgs a) {
  __shared__ TopkScratch ws[8];
  const int warp = threadIdx.x >> 5;
  const int64_t item = (int64_t)blockIdx.x * 8 + warp;
  const int64_t R = (int64_t)a.B * a.N;
  if (item >= R * a.Hkv) return;
  const int64_t r = item / a.Hkv;
  const int b = (int)(r / a.N);
  bool bad = false;
  const int qp = clamp_seq(a.seq_lens, b, a.N, a.max_blocks, bad) - a.N + (int)(r % a.N);
  warp_topk<0>(a.scores + item * a.max_blocks, qp / 128, a.topk, a.block_ids + item * a.topk,
            a.sel_scores ? a.sel_scores + item * a.topk : nullptr, ws[warp]);
}

// ---------------------------------------------------------------------------------------
// Multi-token decode scorer (2 <= N <= 16 query rows per request) on the tensor cores.
//
// The pages' AB-swapped tile: the 128-token key-index block is the MMA's M side and the
// request's query rows, padded to 16, its N side. Every (page, group) of the K-index is one
// 128 x Di tile, brought by TMA ({64 channels, 1 group, 128 tokens} boxes, 128-byte swizzle)
// into a ring of stages and read once from HBM whatever N is; one MMA group of Di/16 steps
// (M 128, N 16) writes its 128 x 16 fp32 scores into a slot of tensor memory. An epilogue
// warpgroup (one token per thread) applies the causal mask of the request's last block and
// reduces each query row's column to the block max with a transposing butterfly (16 shuffles
// per warp for 16 columns), and one score per (query row, group, block) is written. The
// CUDA-core scorer re-reads every query row from shared memory for every key row, which caps
// it at about a quarter of the HBM bandwidth at N = 8.
//
// Work: the batch's (request, page) list in contiguous ranges, one persistent CTA per SM, the
// page's Hkv groups in order. Roles: warp 0 loads (TMA), warp 1 issues the MMAs (one elected
// lane of the converged warp), warps 2-5 drain tensor memory. The top-k of the N*Hkv rows of
// every request follows in the multi-row top-k kernel, one warp per row over the whole GPU:
// left to the CTA that finishes a request's last page (as the one-row scorer does) the
// N*Hkv top-ks of a request run on four warps of one SM while the others are idle.
constexpr int kTdThreads = 192;
constexpr int kTdEpi = 4;           // epilogue warps (128 tensor-memory lanes)
constexpr int kTdAcc = 4;           // accumulator slots of 16 columns
constexpr int kTdNPad = 16;         // query rows per MMA (N of the instruction)

struct TdLayout {
  uint32_t stage_bytes, q_bytes, off_q, off_red, off_bar, off_misc, total;
  int nstage;
};

__host__ __device__ inline TdLayout td_layout(int Hkv, int Di, int nstage) {
  TdLayout L;
  L.nstage = nstage;
  L.stage_bytes = (uint32_t)(128 * Di * 2);                   // one (page, group) tile
  L.q_bytes = (uint32_t)(Hkv * (Di / 64) * kTdNPad * 128);    // 16 rows x 64 channels per box
  uint32_t off = L.stage_bytes * (uint32_t)nstage;            // stages first (1024-aligned)
  L.off_q = off;
  off += L.q_bytes;
  L.off_red = off;
  off += (uint32_t)(2 * kTdEpi * kTdNPad * 4);                // per-warp column maxima, x2
  off = (off + 7u) & ~7u;
  L.off_bar = off;
  off += (uint32_t)(8 * (2 * nstage + 2 + 2 * kTdAcc));
  L.off_misc = off;
  off += 64;
  L.total = off + 1024;
  return L;
}

struct TdParams {
  const int32_t* page_table;
  const int32_t* seq_lens;
  int32_t B, N, Hkv, Di, max_blocks, nstage;
  int64_t num_pages;
  float* scores;
};

// Barrier of the epilogue warps, returning whether any epilogue thread passed `flag` (one decision for all).
__device__ __forceinline__ bool td_epi_sync_or(bool flag) {
  uint32_t any;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 2, %2, q;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(any)
      : "r"((uint32_t)flag), "n"(kTdEpi * 32)
      : "memory");
  return any != 0;
}

// Max over the warp's 32 rows of each of 16 columns: afterwards lanes 2c and 2c+1 hold the max
// of column c (each step halves the columns a lane keeps and exchanges the other half).
__device__ __forceinline__ float warp_colmax16(float (&v)[16], int lane) {
  float w8[8], w4[4], w2[2];
  const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float give = u16 ? v[c] : v[c + 8], keep = u16 ? v[c + 8] : v[c];
    w8[c] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, 16));
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float give = u8 ? w8[c] : w8[c + 4], keep = u8 ? w8[c + 4] : w8[c];
    w4[c] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, 8));
  }
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const float give = u4 ? w4[c] : w4[c + 2], keep = u4 ? w4[c + 2] : w4[c];
    w2[c] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, 4));
  }
  const float give = u2 ? w2[0] : w2[1], keep = u2 ? w2[1] : w2[0];
  float w = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, 2));
  return fmaxf(w, __shfl_xor_sync(0xffffffffu, w, 1));
}

template <int DI>
__global__ void __launch_bounds__(kTdThreads, 1)
    score_tc_decode_kernel(const __grid_constant__ CUtensorMap qmap,
                           const __grid_constant__ CUtensorMap kmap, const TdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const TdLayout L = td_layout(p.Hkv, DI, p.nstage);
  const int nstage = p.nstage, Hkv = p.Hkv, N = p.N;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_bar);
  uint64_t* empty = full + nstage;
  uint64_t* q_full = empty + nstage;
  uint64_t* q_empty = q_full + 1;
  uint64_t* acc_full = q_empty + 1;
  uint64_t* acc_empty = acc_full + kTdAcc;
  int32_t* misc = reinterpret_cast<int32_t*>(smem + L.off_misc);
  float* red = reinterpret_cast<float*>(smem + L.off_red);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- the CTA's contiguous range of (request, page) items: warp 0 scans the lengths
  if (warp == 0) {
    int total = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      bool bad = false;
      const int nb = b < p.B ? (clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) + 127) / 128 : 0;
      if (bad && blockIdx.x == 0) msa_record_error(kErrBadBlock);
      total += __reduce_add_sync(0xffffffffu, nb);
    }
    const int per = (total + (int)gridDim.x - 1) / (int)gridDim.x;
    const int p0 = min(total, (int)blockIdx.x * per);
    const int p1 = min(total, p0 + per);
    int run = 0, b_start = p.B, j_start = 0;
    for (int b0 = 0; b0 < p.B && b_start == p.B; b0 += 32) {
      const int b = b0 + lane;
      bool bad = false;
      const int nb = b < p.B ? (clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) + 127) / 128 : 0;
      int incl = nb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - nb;
      const uint32_t hit = __ballot_sync(0xffffffffu, b < p.B && run + excl <= p0 && p0 < run + incl);
      if (hit) {
        const int src = __ffs(hit) - 1;
        b_start = b0 + src;
        j_start = p0 - run - __shfl_sync(0xffffffffu, excl, src);
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      misc[0] = p0;
      misc[1] = p1;
      misc[2] = b_start;
      misc[3] = j_start;
      misc[5] = 0;  // set when a bounded wait gives up
    }
  }
  if (tid == 32) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, kTdEpi);
    for (int a = 0; a < kTdAcc; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kTdEpi);
    }
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(misc + 8)), "n"(kTdAcc * kTdNPad)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = (uint32_t)misc[8];
  const int p0 = misc[0], p1 = misc[1];
  const uint32_t sbase = smem_u32(smem);
  volatile int32_t* fail = misc + 5;
  auto wait_ok = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_wait(bar, parity)) return true;
    msa_record_error(kErrTimeout);
    *fail = 1;
    return false;
  };

  if (p0 < p1) {
    if (warp == 0) {
      // ================================================================ producer
      if (lane == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&qmap);
        int b = misc[2], j = misc[3], qloads = 0;
        bool bad = false;
        int nb = (clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) + 127) / 128;
        uint32_t it = 0;
        bool ok = true;
        for (int item = p0; item < p1 && ok; ++item) {
          if (item == p0 || j == 0) {
            // the request's query-index rows (16 from its first row; the MMA reads N of them)
            if (qloads > 0 && !wait_ok(q_empty, (qloads - 1) & 1)) break;
            mbar_expect_tx(q_full, L.q_bytes);
            for (int g = 0; g < Hkv; ++g)
              for (int h = 0; h < DI / 64; ++h)
                tma_load_3d(smem + L.off_q + (g * (DI / 64) + h) * (kTdNPad * 128), &qmap, q_full,
                            h * 64, g, b * N);
            ++qloads;
          }
          int32_t page = p.page_table[(int64_t)b * p.max_blocks + j];
          if (page < 0 || page >= p.num_pages) {
            msa_record_error(kErrBadPage);
            page = 0;
          }
          for (int g = 0; g < Hkv; ++g, ++it) {
            const uint32_t s = it % nstage;
            if (it >= (uint32_t)nstage && !wait_ok(&empty[s], ((it / nstage) - 1) & 1)) {
              ok = false;
              break;
            }
            uint8_t* dst = smem + s * L.stage_bytes;
            mbar_expect_tx(&full[s], L.stage_bytes);
#pragma unroll
            for (int h = 0; h < DI / 64; ++h)
              tma_load_3d(dst + h * 16384, &kmap, &full[s], h * 64, g, page * 128);
          }
          if (++j == nb) {
            j = 0;
            ++b;
            if (b < p.B) nb = (clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) + 127) / 128;
          }
        }
        // the copies still in flight land before the CTA may exit
        for (uint32_t k = it > (uint32_t)nstage ? it - nstage : 0; k < it; ++k)
          mbar_wait(&empty[k % nstage], (k / nstage) & 1);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ================================================================ MMA issuer
      const uint32_t idesc = umma_idesc_bf16(128, kTdNPad, 0, 0);
      int b = misc[2], j = misc[3], qloads = 0;
      bool bad = false;
      int nb = (clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) + 127) / 128;
      uint32_t it = 0;
      bool ok = true;
      for (int item = p0; item < p1 && ok; ++item) {
        if (item == p0 || j == 0) {
          ok = __all_sync(0xffffffffu, wait_ok(q_full, qloads & 1));
          ++qloads;
        }
        for (int g = 0; g < Hkv && ok; ++g, ++it) {
          const uint32_t s = it % nstage, a = it % kTdAcc;
          ok = __all_sync(0xffffffffu, wait_ok(&full[s], (it / nstage) & 1)) &&
               (it < (uint32_t)kTdAcc ||
                __all_sync(0xffffffffu, wait_ok(&acc_empty[a], ((it / kTdAcc) - 1) & 1)));
          if (!ok) break;
          tmem_fence_after();
          const uint64_t ad = umma_desc_sw128(sbase + s * L.stage_bytes, 16, 1024);
          const uint64_t bd = umma_desc_sw128(sbase + L.off_q + g * (DI / 64) * (kTdNPad * 128), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < DI / 16; ++kk) {
            // 16 channels per step: 32 bytes into a 128-byte row, 16 KB (A) / 2 KB (B) per half
            const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
            const uint32_t boff = (kk >> 2) * (kTdNPad * 128) + (kk & 3) * 32;
            umma_bf16_elect(tmem + a * kTdNPad, ad + (aoff >> 4), bd + (boff >> 4), idesc, kk > 0);
          }
          umma_commit_elect(&acc_full[a]);
          umma_commit_elect(&empty[s]);  // the stage is free once the group has read it
        }
        if (++j == nb) {
          j = 0;
          ++b;
          if (b < p.B) nb = (clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) + 127) / 128;
        }
      }
      __syncwarp();
    } else {
      // ================================================================ epilogue + top-k
      // a warp reads the tensor-memory lanes of its sub-partition: 32 * (warp % 4) ..
      const int ew = warp & 3;
      const int erow = ew * 32 + lane;                // token of the block = accumulator row
      const uint32_t lane_addr = (uint32_t)(32 * ew) << 16;
      int b = misc[2], j = misc[3], cur_b = -1, par = 0, qloads = 0;
      bool bad = false;
      int nb = (clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) + 127) / 128;
      uint32_t it = 0;
      bool ok = true, failed = false;  // failed: agreed by all epilogue threads at a barrier
      for (int item = p0; item < p1 && !failed; ++item) {
        if (b != cur_b) {
          cur_b = b;
          if (qloads > 0 && lane == 0) mbar_arrive(q_empty);  // the previous request's rows
          ++qloads;
        }
        bool bad_s = false;
        const int seq = clamp_seq(p.seq_lens, b, N, p.max_blocks, bad_s);
        const int pos = j * 128 + erow;
        for (int g = 0; g < Hkv; ++g, ++it) {
          const uint32_t a = it % kTdAcc;
          // warp-uniform: the tensor-memory load below is warp-collective
          ok = __all_sync(0xffffffffu, ok && wait_ok(&acc_full[a], (it / kTdAcc) & 1));
          float v[16];
          if (ok) {
            tmem_fence_after();
            uint32_t raw[16];
            tmem_ld16(tmem + lane_addr + a * kTdNPad, raw);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = __uint_as_float(raw[c]);
          }
          tmem_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[a]);
          // causal mask: row c sits at position seq - N + c
#pragma unroll
          for (int c = 0; c < 16; ++c)
            if (!ok || c >= N || pos > seq - N + c) v[c] = -INFINITY;
          const float m = warp_colmax16(v, lane);
          if ((lane & 1) == 0) red[(par * kTdEpi + ew) * kTdNPad + (lane >> 1)] = m;
          // a wait that gave up is agreed here, so every epilogue warp leaves after the same item
          failed = td_epi_sync_or(!ok);
          const int tid_e = tid - 64;
          if (!failed && tid_e < N) {
            float mx = -INFINITY;
#pragma unroll
            for (int w = 0; w < kTdEpi; ++w) mx = fmaxf(mx, red[(par * kTdEpi + w) * kTdNPad + tid_e]);
            const int64_t r = (int64_t)b * N + tid_e;
            p.scores[(r * Hkv + g) * p.max_blocks + j] = mx;
          }
          par ^= 1;
        }
        if (failed) break;
        if (++j == nb) {
          j = 0;
          ++b;
          if (b < p.B) nb = (clamp_seq(p.seq_lens, b, N, p.max_blocks, bad) + 127) / 128;
        }
      }
    }
  }
  // ------------------------------------------------------------------ teardown
  tmem_fence_before();
  __syncthreads();
  if (warp == 1) {
    tmem_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "n"(kTdAcc * kTdNPad)
                 : "memory");
  }
}

constexpr size_t kSmemMax = 232448;  // opt-in shared memory per block on sm_100/sm_103

}  // namespace

size_t score_decode_smem_bytes(int N, int Hkv, int Di, int* nstage) {
  for (int ns = 4; ns >= 2; --ns) {
    const DecodeSmemLayout L = decode_layout(N, Hkv, Di, ns);
    if (L.total <= kSmemMax) {
      if (nstage) *nstage = ns;
      return L.total;
    }
  }
  if (nstage) *nstage = 0;
  return 0;
}

cudaError_t launch_score_decode(const ScoreArgs& a, cudaStream_t stream) {
  int nstage = 0;
  const size_t smem = score_decode_smem_bytes(a.N, a.Hkv, a.Di, &nstage);
  if (nstage < 2) return cudaErrorInvalidValue;
  const int rows = kStageRows < 128 * a.Hkv ? kStageRows : 128 * a.Hkv;
  CUtensorMap map;
  const uint64_t dims[2] = {(uint64_t)a.Di, (uint64_t)a.num_pages * 128 * a.Hkv};
  const uint64_t strides[1] = {(uint64_t)a.Di * 2};
  const uint32_t box[2] = {64, (uint32_t)rows};
  if (!encode_bf16_map(&map, a.k_idx, 2, dims, strides, box, true)) return cudaErrorInvalidValue;
  DecodeKParams p;
  p.q_idx = a.q_idx;
  p.page_table = a.page_table;
  p.seq_lens = a.seq_lens;
  p.B = a.B;
  p.N = a.N;
  p.Hkv = a.Hkv;
  p.max_blocks = a.max_blocks;
  p.topk = a.topk;
  p.nstage = nstage;
  p.num_pages = a.num_pages;
  p.block_ids = a.block_ids;
  p.sel_scores = a.sel_scores;
  p.scores = a.scores;
  p.tickets = a.tickets;
  p.fpt = a.fpt;
  p.fpt_lens = a.fpt_lens;
  const int grid = sm_count();
  auto launch = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, stream>>>(map, p);
    return cudaSuccess;
  };
  const int nq = a.N <= 1 ? 1 : a.N <= 2 ? 2 : a.N <= 4 ? 4 : 8;
  cudaError_t e;
  if (a.Di == 128)
    e = nq == 1 ? launch(score_decode_kernel<128, 1>) : nq == 2 ? launch(score_decode_kernel<128, 2>)
        : nq == 4 ? launch(score_decode_kernel<128, 4>) : launch(score_decode_kernel<128, 8>);
  else
    e = nq == 1 ? launch(score_decode_kernel<64, 1>) : nq == 2 ? launch(score_decode_kernel<64, 2>)
        : nq == 4 ? launch(score_decode_kernel<64, 4>) : launch(score_decode_kernel<64, 8>);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int score_tc_decode_stages(int Hkv, int Di) {
  for (int ns = 6; ns >= 2; --ns)
    if (td_layout(Hkv, Di, ns).total <= kSmemMax) return ns;
  return 0;
}

cudaError_t launch_score_tc_decode(const ScoreArgs& a, cudaStream_t stream) {
  const int nstage = score_tc_decode_stages(a.Hkv, a.Di);
  if (nstage < 2 || a.N > kTdNPad) return cudaErrorInvalidValue;
  CUtensorMap qmap, kmap;
  const uint64_t qdims[3] = {(uint64_t)a.Di, (uint64_t)a.Hkv, (uint64_t)a.B * a.N};
  const uint64_t kdims[3] = {(uint64_t)a.Di, (uint64_t)a.Hkv, (uint64_t)a.num_pages * 128};
  const uint64_t strides[2] = {(uint64_t)a.Di * 2, (uint64_t)a.Hkv * a.Di * 2};
  const uint32_t qbox[3] = {64, 1, (uint32_t)kTdNPad};
  const uint32_t kbox[3] = {64, 1, 128};
  if (!encode_bf16_map(&qmap, a.q_idx, 3, qdims, strides, qbox, true) ||
      !encode_bf16_map(&kmap, a.k_idx, 3, kdims, strides, kbox, true))
    return cudaErrorInvalidValue;
  TdParams p;
  p.page_table = a.page_table;
  p.seq_lens = a.seq_lens;
  p.B = a.B;
  p.N = a.N;
  p.Hkv = a.Hkv;
  p.Di = a.Di;
  p.max_blocks = a.max_blocks;
  p.nstage = nstage;
  p.num_pages = a.num_pages;
  p.scores = a.scores;
  const size_t smem = td_layout(a.Hkv, a.Di, nstage).total;
  auto launch = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<sm_count(), kTdThreads, smem, stream>>>(qmap, kmap, p);
    return cudaGetLastError();
  };
  return a.Di == 128 ? launch(score_tc_decode_kernel<128>) : launch(score_tc_decode_kernel<64>);
}

cudaError_t launch_score_rows(const ScoreArgs& a, cudaStream_t stream) {
  CUtensorMap qmap, kmap;
  const uint64_t qdims[3] = {(uint64_t)a.Di, (uint64_t)a.Hkv, (uint64_t)a.B * a.N};
  const uint64_t kdims[3] = {(uint64_t)a.Di, (uint64_t)a.Hkv, (uint64_t)a.num_pages * 128};
  const uint64_t strides[2] = {(uint64_t)a.Di * 2, (uint64_t)a.Hkv * a.Di * 2};
  const uint32_t box[3] = {64, 1, 128};
  if (!encode_bf16_map(&qmap, a.q_idx, 3, qdims, strides, box, true) ||
      !encode_bf16_map(&kmap, a.k_idx, 3, kdims, strides, box, true))
    return cudaErrorInvalidValue;
  ScoreTcParams p;
  p.page_table = a.page_table;
  p.seq_lens = a.seq_lens;
  p.B = a.B;
  p.N = a.N;
  p.Hkv = a.Hkv;
  p.max_blocks = a.max_blocks;
  p.max_chunks = (a.max_blocks + kScoreChunk - 1) / kScoreChunk;
  p.num_pages = a.num_pages;
  p.scores = a.scores;
  const int64_t items = (int64_t)a.B * a.Hkv * p.max_chunks;
  const int grid = (int)(items < sm_count() ? items : sm_count());
  auto launch = [&](auto kern, size_t smem) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kScThreads, smem, stream>>>(qmap, kmap, p);
    return cudaGetLastError();
  };
  return a.Di == 128 ? launch(score_rows_tc_kernel<128>, ScoreTcLayout<128>::kSmem)
                     : launch(score_rows_tc_kernel<64>, ScoreTcLayout<64>::kSmem);
}

cudaError_t launch_topk_rows(const ScoreArgs& a, cudaStream_t stream) {
  const int64_t items = (int64_t)a.B * a.N * a.Hkv;
  topk_rows_kernel<<<(unsigned)((items + 7) / 8), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace msa
