// KV-block-major sparse prefill: bucketing, block-major attention partials, LSE merge.
//
// Together AI MiniMax-M3 serving article, section "KV-block-major sparse attention reduces
// redundant KV movement" (Japanese translation: "KV-block-major sparse attention"): many
// query tokens choose the same KV blocks, so a query-major kernel moves the same KV block
// from HBM to on-chip memory again and again. Remapping the work from {q, kv block} to
// {kv block, q} makes the KV block the outer loop: it is loaded once and serves every
// query that chose it. Each block then yields only a partial output, and a Log-Sum-Exp
// reduction rescales and sums the partials of the selected blocks.
//
// GB300 design.
//  (a) Bucketing inverts block_ids [T, Hkv, k] into lists of (query, slot) entries per
//      (group, query window, block): a count pass, a scan per (group, window) segment, a scan
//      over segments, a scatter, then one 16-byte descriptor per work tile.
//  (b) Work tile = (group g, block j, up to 128/G queries of the list) = 128 query-head rows,
//      on tcgen05: S = Q K^T and O = P V with accumulators in tensor memory, query rows
//      gathered by TMA, the K/V block loaded once per list; one bf16 partial O and its fp32
//      LSE per (query, group, slot) and head (see the attention section below).
//  (c) The LSE merge (page_table_merge.cu) reduces the partials of each (query, head).
// With G in {8, 16}, the slots that many queries of a 2*128/G-query pair share are taken out
// first and computed query-major (prefill_dense.cu); (a)-(b) then run on the remainder.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"
#include "pair_deal.cuh"
#include "softmax_math.cuh"

MSA_DEFINE_ERROR_WORD(pre)

namespace msa {

namespace {

// ------------------------------------------------------------------------------ bucketing
// The selections were counted into their lists by the selection kernel (prefill_dense.cu),
// which also kept each selection's place in its list (epos). Two kernels finish the lists:
// offsets per (group, window) segment with the tile descriptors, then the placement of every
// entry at its list's offset plus its place, with no atomics. Rows are (query, group) pairs,
// row = t*Hkv + g; the host checks that T*Hkv*topk fits in int32.

// Block-wide exclusive scan of one int per thread; returns the block total via *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? warp_sums[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) warp_sums[lane] = wi - w;
    if (lane == 31) warp_sums[32] = wi;
  }
  __syncthreads();
  const int out = warp_sums[warp] + incl - v;
  *total = warp_sums[32];
  __syncthreads();
  return out;
}

constexpr int kListThreads = 1024;

// One CTA per (group, window) segment. Every CTA sums the counts of all segments (a few
// thousand lists) to find its own segment's first entry and first tile, so no CTA waits for
// another; then it scans its own lists: offsets (relative to the segment) and tiles of `qpt`
// queries, and writes one descriptor (list, first entry, valid queries) per tile when `desc`
// is given. CTA 0 also writes the grand totals at index nseg.
__global__ void __launch_bounds__(kListThreads)
    bucket_lists_kernel(const int32_t* __restrict__ counts, int32_t nseg, int32_t nblk,
                        int32_t qpt, int32_t* __restrict__ offsets,
                        int32_t* __restrict__ tile_local, int32_t* __restrict__ group_base,
                        int32_t* __restrict__ seg_tile_base, int4* __restrict__ desc,
                        const int32_t* __restrict__ dcnt, int64_t npairs, int32_t deal_grid,
                        int32_t deal_rpw, int32_t* __restrict__ porder) {
  // blocks past the segments deal the query-major pairs, one window each (same launch)
  if (blockIdx.x >= (unsigned)nseg) {
    pair_deal_window(dcnt, npairs, deal_grid, deal_rpw, porder, (int64_t)blockIdx.x - nseg);
    return;
  }
  extern __shared__ int32_t seg_tot[];  // [2 * nseg]: entries, tiles per segment
  __shared__ int warp_sums[33];
  __shared__ int32_t s_base[2];
  const int seg = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int sg = warp; sg < nseg; sg += kListThreads / 32) {
    int c = 0, t = 0;
    for (int j = lane; j < nblk; j += 32) {
      const int v = counts[(int64_t)sg * nblk + j];
      c += v;
      t += (v + qpt - 1) / qpt;
    }
    c = __reduce_add_sync(0xffffffffu, c);
    t = __reduce_add_sync(0xffffffffu, t);
    if (lane == 0) {
      seg_tot[sg] = c;
      seg_tot[nseg + sg] = t;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int bc = 0, bt = 0, ac = 0, at = 0;
    for (int sg = 0; sg < nseg; ++sg) {
      if (sg == seg) {
        bc = ac;
        bt = at;
      }
      ac += seg_tot[sg];
      at += seg_tot[nseg + sg];
    }
    s_base[0] = bc;
    s_base[1] = bt;
    group_base[seg] = bc;
    seg_tile_base[seg] = bt;
    if (seg == 0) {
      group_base[nseg] = ac;
      seg_tile_base[nseg] = at;
    }
  }
  int carry = 0, tile_carry = 0;
  for (int j0 = 0; j0 < nblk; j0 += kListThreads) {
    const int j = j0 + threadIdx.x;
    const int c = j < nblk ? counts[(int64_t)seg * nblk + j] : 0;
    const int nt = (c + qpt - 1) / qpt;
    int tot_c, tot_t;
    const int ex_c = block_exclusive_scan(c, warp_sums, &tot_c);
    const int ex_t = block_exclusive_scan(nt, warp_sums, &tot_t);
    if (j < nblk) {
      offsets[(int64_t)seg * (nblk + 1) + j] = carry + ex_c;
      tile_local[(int64_t)seg * (nblk + 1) + j] = tile_carry + ex_t;
    }
    carry += tot_c;
    tile_carry += tot_t;
  }
  if (threadIdx.x == 0) {
    offsets[(int64_t)seg * (nblk + 1) + nblk] = carry;
    tile_local[(int64_t)seg * (nblk + 1) + nblk] = tile_carry;
  }
  if (!desc) return;
  __syncthreads();  // this CTA's offsets are visible to all its threads
  // one warp per list, lanes over the list's tiles
  for (int j = warp; j < nblk; j += kListThreads / 32) {
    const int32_t* off = offsets + (int64_t)seg * (nblk + 1) + j;
    const int32_t* tl = tile_local + (int64_t)seg * (nblk + 1) + j;
    const int first = s_base[0] + off[0], lcnt = off[1] - off[0];
    const int t0 = s_base[1] + tl[0], nt = tl[1] - tl[0];
    for (int q = lane; q < nt; q += 32)
      desc[t0 + q] = make_int4(seg * nblk + j, first + q * qpt, min(qpt, lcnt - q * qpt), 0);
  }
}

// One thread per (query, group) row: each counted selection (t, slot) goes to its list's first
// entry plus its place in the list.
__global__ void bucket_place_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ epos,
                                    int32_t rows, int32_t Hkv, int32_t topk, int32_t nblk,
                                    int32_t win, int32_t nwin, const int32_t* __restrict__ offsets,
                                    const int32_t* __restrict__ group_base,
                                    int32_t* __restrict__ entries, bool vec4) {
  for (int32_t row = blockIdx.x * blockDim.x + threadIdx.x; row < rows;
       row += gridDim.x * blockDim.x) {
    const int32_t t = row / Hkv;
    const int32_t g = row - t * Hkv;
    const int64_t seg = (int64_t)g * nwin + t / win;  // (group, window) segment
    const int32_t base = group_base[seg];
    const int32_t* off = offsets + seg * (nblk + 1);
    auto place = [&](int s, int32_t j, int32_t e) {
      if (j >= 0 && j < nblk) entries[base + off[j] + e] = t * topk + s;
    };
    if (vec4) {  // the row's ids and places four at a time
      for (int s = 0; s < topk; s += 4) {
        const int4 j4 = reinterpret_cast<const int4*>(ids + (int64_t)row * topk + s)[0];
        const int4 e4 = reinterpret_cast<const int4*>(epos + (int64_t)row * topk + s)[0];
        place(s, j4.x, e4.x);
        place(s + 1, j4.y, e4.y);
        place(s + 2, j4.z, e4.z);
        place(s + 3, j4.w, e4.w);
      }
    } else {
      for (int s = 0; s < topk; ++s) place(s, ids[row * topk + s], epos[row * topk + s]);
    }
  }
}

// ------------------------------------------------------------------------------ attention
// One CTA per SM (tcgen05 path). Warp 0 gathers the query rows (TMA), warp 2 loads the K/V
// blocks (TMA), warp 1 owns tensor memory and issues the MMAs, two softmax warpgroups (warps
// 4-7: even tiles, warps 8-11: odd tiles; one row per thread) run softmax and the epilogue.
constexpr int kThreads = 384;
constexpr int kRows = 128;                       // query-head rows per tile (MMA M)
constexpr uint32_t kBox = 128 * 64 * 2;          // 128 rows x 64 channels bf16 = 16 KB
constexpr uint32_t kTileBytes = 2 * kBox;        // Q tile, P tile, K block or V block: 32 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kTmemCols = 512;              // S[2] at 0/128, O[2] at 256/384
constexpr int kChunk = 4;                        // consecutive tiles per CTA per round
constexpr uint32_t kIssuerNap = 100;             // ns an idle MMA issuer blocks on a barrier
constexpr int kLaunchRegs = 168;                 // registers per thread at launch (384 threads)
constexpr int kRegsLow = 88;                     // warps 0-3 after the split
constexpr int kRegsHigh = 208;                   // softmax warpgroups after the split

// shared-memory carve-up (offsets from a 1024-aligned base): a 3-deep ring of gathered
// query tiles hides the latency of the scattered row gathers; two K/V block buffers let the
// next block load while the previous one is still in use. S and O live in tensor memory
// (double buffered); P (bf16) is written over the first 64 columns of its S buffer.
constexpr int kQStages = 3;
constexpr uint32_t kOffQ = 0;                                  // Q[kQStages]
constexpr uint32_t kOffKV = kQStages * kTileBytes;             // {K, V}[2]
constexpr uint32_t kOffBar = (kQStages + 4) * kTileBytes;
constexpr size_t kSmemBytes = 1024 + kOffBar + 256;

struct Bars {
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t s_full[2], p_full[2], o_full[2], o_free[2];
  uint64_t kv_full[2], kv_empty[2];
  uint32_t tmem_base;
  int32_t fail;
};

struct PreKParams {
  const int32_t* entries;
  const int4* desc;                // per-tile (list, first entry, valid queries)
  const int32_t* tile_offsets;
  int32_t Hkv, G, topk, nblk, qpt, nwin;
  // 1: the query map is 5-D {64 channels, 8 heads, 2 channel halves, G/8, query-group} and one
  // copy brings a query's G head rows as whole 8-row swizzle atoms (both channel halves, 2 KB
  // per 8 heads); 0: two 3-D copies per query, one per channel half.
  int32_t q_atoms;
  int64_t q_start;
  const int32_t* page_table;      // null: contiguous K/V; else the page of each block
  int64_t num_pages;
  uint16_t* part_o;               // chunk-major [16][part_rows][8] bf16
  int64_t part_rows;               // T*Hkv*topk*G
  float* part_lse;
};

// Tile descriptor: list gj = g*nblk + j, first entry of the tile, valid query slots.
__device__ __forceinline__ int4 load_desc(const PreKParams& p, int64_t tile) {
  return __ldg(p.desc + tile);
}

__device__ __forceinline__ bool wait_or_fail(uint64_t* bar, uint32_t parity, volatile int32_t* fail) {
  if (*fail) return false;
  if (mbar_wait(bar, parity)) return true;
  msa_record_error(kErrTimeout);
  *fail = 1;
  return false;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_block_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                            const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const PreKParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars& B = *reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int32_t* fail = &B.fail;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Tiles are dealt round-robin in chunks of kChunk: CTA c takes tiles
  // (r * gridDim + c) * kChunk + q, so all CTAs sweep the (group, window)-ordered tile list
  // together and the current window's query rows and K/V blocks stay in L2.
  const int64_t nseg = (int64_t)p.Hkv * p.nwin;
  const int64_t total = p.tile_offsets[nseg * (p.nblk + 1) + nseg];  // sum of segment tiles
  const int64_t round_tiles = (int64_t)gridDim.x * kChunk;
  const int64_t full_rounds = total / round_tiles;
  const int64_t rem = total - full_rounds * round_tiles;
  const int64_t mine_rem = rem - (int64_t)blockIdx.x * kChunk;
  const int n = (int)(full_rounds * kChunk + (mine_rem <= 0 ? 0 : (mine_rem < kChunk ? mine_rem : kChunk)));
  if (n == 0) return;  // uniform for the CTA
  auto tile_of = [&](int i) -> int64_t {
    return ((int64_t)(i / kChunk) * gridDim.x + blockIdx.x) * kChunk + (i % kChunk);
  };
  const int64_t lists_per_group = (int64_t)p.nwin * p.nblk;

  if (tid == 0) {
    for (int q = 0; q < kQStages; ++q) {
      mbar_init(&B.q_full[q], 1);
      mbar_init(&B.q_empty[q], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&B.s_full[b], 1);
      mbar_init(&B.p_full[b], 4);
      mbar_init(&B.o_full[b], 1);
      mbar_init(&B.o_free[b], 4);
      mbar_init(&B.kv_full[b], 1);
      mbar_init(&B.kv_empty[b], 1);
    }
    B.fail = 0;
    mbar_fence_init();
  }
  if (warp == 1) {  // the whole warp allocates the tensor memory, then gives up the permit
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&B.tmem_base)), "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = B.tmem_base;
  const uint32_t sbase = smem_u32(smem);

  // Register split: the producer / issuer warpgroup needs few registers, each softmax thread
  // holds a 128-column row. The launcher checks that the kernel was built with kLaunchRegs
  // registers per thread, so the split adds up to exactly what the launch allocated.
  static_assert(128 * kRegsLow + 256 * kRegsHigh == kThreads * kLaunchRegs, "register split");
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == 0 || warp == 3) {
      // ================================================================ query producers
      // Warps 0 and 3 gather the query rows of alternate tiles (warp 0 the even ones): each
      // lane copies up to kMaxQPerLane query slots of the tile (lane, lane+32, ...) with one
      // tensor copy per query. A warp's tensor copies issue one after another, about a
      // hundred cycles each under load (measured), so one warp alone bounds the tile rate.
      // Descriptors are read two of the warp's tiles ahead and entries one, so that no
      // global-memory latency sits between two tiles' copies.
      if (lane == 0 && warp == 0) tma_prefetch_desc(&qmap);
      if (lane == 0 && warp == 3) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
      }
      constexpr int kMaxQPerLane = 4;  // qpt = 128/G <= 128
      const int qw = warp == 0 ? 0 : 1;
      const int4 dz = make_int4(0, 0, 0, 0);
      auto load_entries = [&](const int4 d, int32_t (&e)[kMaxQPerLane]) {
  #pragma unroll
        for (int r = 0; r < kMaxQPerLane; ++r) {
          const int q = lane + 32 * r;
          e[r] = q < d.z ? p.entries[d.y + q] : -1;
        }
      };
      int4 dc = qw < n ? load_desc(p, tile_of(qw)) : dz;              // tile i
      int4 dn = qw + 2 < n ? load_desc(p, tile_of(qw + 2)) : dz;      // tile i+2
      int4 dnn = qw + 4 < n ? load_desc(p, tile_of(qw + 4)) : dz;     // tile i+4
      int32_t ec[kMaxQPerLane], en[kMaxQPerLane];
      load_entries(dc, ec);
      load_entries(dn, en);
      for (int i = qw; i < n; i += 2) {
        const int qs = i % kQStages;
        if (i >= kQStages && !wait_or_fail(&B.q_empty[qs], (i / kQStages - 1) & 1, fail)) break;
        const int g = (int)(dc.x / lists_per_group);
        uint8_t* qdst = smem + kOffQ + qs * kTileBytes;
        if (lane == 0) mbar_expect_tx(&B.q_full[qs], (uint32_t)(dc.z * p.G * 256));
        __syncwarp();
  #pragma unroll
        for (int r = 0; r < kMaxQPerLane; ++r) {
          const int q = lane + 32 * r;
          if (q < dc.z) {
            const int t = ec[r] / p.topk;
            if (p.q_atoms) {
              tma_load_5d(qdst + q * p.G * 256, &qmap, &B.q_full[qs], 0, 0, 0, 0, t * p.Hkv + g);
            } else {
              tma_load_3d(qdst + q * p.G * 128, &qmap, &B.q_full[qs], 0, g * p.G, t);
              tma_load_3d(qdst + kBox + q * p.G * 128, &qmap, &B.q_full[qs], 64, g * p.G, t);
            }
          }
        }
        // shift the read-ahead by one of this warp's tiles
        dc = dn;
        dn = dnn;
  #pragma unroll
        for (int r = 0; r < kMaxQPerLane; ++r) ec[r] = en[r];
        load_entries(i + 4 < n ? dnn : dz, en);
        dnn = i + 6 < n ? load_desc(p, tile_of(i + 6)) : dz;
      }
      __syncwarp();
    } else if (warp == 2) {
      // ================================================================ K/V producer
      // Walks the same tile sequence and loads the K and V block of every new list into the
      // next of the two K/V buffers, as soon as that buffer's previous list has finished its
      // last O MMA. Kept apart from the query gathers so that waiting for a buffer never
      // delays the query rows of the tiles in between. Descriptors are read 32 at a time.
      int loaded_gj = -1, kv_loads = 0;
      for (int base = 0; base < n && !*fail; base += 32) {
        const int mine = base + lane;
        const int gj_l = mine < n ? load_desc(p, tile_of(mine)).x : -1;
        const int cnt = n - base < 32 ? n - base : 32;
        for (int t = 0; t < cnt; ++t) {
          const int gj = __shfl_sync(0xffffffffu, gj_l, t);
          if (gj == loaded_gj) continue;
          const int c = kv_loads & 1;
          if (lane == 0) {
            // load kv_loads goes to buffer kv_loads & 1, free once the last tile of load
            // kv_loads - 2 has finished its O MMA
            if (kv_loads < 2 || wait_or_fail(&B.kv_empty[c], ((kv_loads - 2) >> 1) & 1, fail)) {
              const int g = (int)(gj / lists_per_group), j = gj % p.nblk;
              uint8_t* kvb = smem + kOffKV + c * 2 * kTileBytes;
              mbar_expect_tx(&B.kv_full[c], 4 * kBox);
              bool bad = false;
              const int tok = kv_block_row(p.page_table, p.num_pages, j, bad);
              if (bad) msa_record_error(kErrBadPage);
              tma_load_3d(kvb, &kmap, &B.kv_full[c], 0, g, tok);
              tma_load_3d(kvb + kBox, &kmap, &B.kv_full[c], 64, g, tok);
              tma_load_3d(kvb + kTileBytes, &vmap, &B.kv_full[c], 0, g, tok);
              tma_load_3d(kvb + kTileBytes + kBox, &vmap, &B.kv_full[c], 64, g, tok);
            }
          }
          if (__shfl_sync(0xffffffffu, (int)*fail, 0)) break;
          ++kv_loads;
          loaded_gj = gj;
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ================================================================ MMA issuer
      // Order S(0), S(1), then O(k), S(k+2) for k = 0, 1, ...: S(k+2) writes the tensor memory
      // that P(k) occupies, so it follows O(k). A ready O is issued before a ready S: the
      // warpgroup whose P is ready waits on that O for its epilogue, while the one the next S
      // serves is usually still in its own epilogue. An idle issuer blocks in hardware on the
      // next O's barrier for at most kIssuerNap ns before re-checking, so it reacts to either
      // within a few hundred cycles. All state stays in registers.
      // The whole warp runs the loop in lockstep (barrier states agreed by a vote) and one
      // elected lane issues each MMA and commit: a converged warp keeps the MMA operands in
      // uniform registers, where a lone lane would move them over before every instruction.
      {
        auto ready = [&](uint64_t* bar, uint32_t parity) {
          return __all_sync(0xffffffffu, mbar_test(bar, parity));
        };
        const uint32_t idesc_s = umma_idesc_bf16(128, 128, 0, 0);  // Q (K-major) x K (K-major)
        const uint32_t idesc_o = umma_idesc_bf16(128, 128, 0, 1);  // P (tmem) x V (MN-major)
        int kv_gj = -1, kv_loads = 0;
        // list and K/V buffer of the tile whose S is in tensor-memory buffer 0 / 1
        int gj0 = -1, gj1 = -1, kvb0 = 0, kvb1 = 0;
        int next_gj = load_desc(p, tile_of(0)).x;
        int after_gj = n > 1 ? load_desc(p, tile_of(1)).x : -2;
        int si = 0, oi = 0;
        uint32_t idle = 0;
        while (oi < n && !__any_sync(0xffffffffu, *fail != 0)) {
          // ---- O(oi): needs P(oi) and the epilogue of oi-2 done with its O buffer
          if (oi < si) {
            const int b = oi & 1;
            if (ready(&B.p_full[b], (oi >> 1) & 1) &&
                (oi < 2 || ready(&B.o_free[b], ((oi - 2) >> 1) & 1))) {
              tmem_fence_after();
              const int c = b ? kvb1 : kvb0;
              const uint32_t va = sbase + kOffKV + c * 2 * kTileBytes + kTileBytes;
  #pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint64_t bd = umma_desc_sw128(va + kk * 2048, kBox, 1024);
                umma_bf16_ts_elect(tmem + 256 + b * 128, tmem + b * 128 + kk * 8, bd, idesc_o, kk > 0);
              }
              umma_commit_elect(&B.o_full[b]);
              // the list of tile oi+1 (its S is issued, or it is the next S) tells whether tile
              // oi is the last one on this K/V load
              const int gj_after = oi + 1 < si ? (b ? gj0 : gj1) : (oi + 1 < n ? next_gj : -2);
              if (gj_after != (b ? gj1 : gj0)) umma_commit_elect(&B.kv_empty[c]);
              ++oi;
              idle = 0;
              continue;
            }
          }
          // ---- S(si): needs O(si-2) issued (this warp issues in order, and the tensor pipe runs
          // one thread's MMAs in issue order, so O(si-2) has read P(si-2) before S(si) writes
          // there; the commit that signals S(si) covers O(si-2)), its queries and its K/V block
          if (si < n && oi >= si - 1) {
            const int b = si & 1, qs = si % kQStages;
            const bool kv_new = next_gj != kv_gj;
            if ((!kv_new || ready(&B.kv_full[kv_loads & 1], (kv_loads >> 1) & 1)) &&
                ready(&B.q_full[qs], (si / kQStages) & 1)) {
              tmem_fence_after();
              if (kv_new) {
                ++kv_loads;
                kv_gj = next_gj;
              }
              const int c = (kv_loads - 1) & 1;
              const uint32_t qa = sbase + kOffQ + qs * kTileBytes;
              const uint32_t ka = sbase + kOffKV + c * 2 * kTileBytes;
  #pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                // query tile: per channel half, 8-row atoms 1 KB apart (two copies per query) or
                // 2 KB apart with the halves interleaved (one copy per query)
                const uint32_t qoff = p.q_atoms ? (kk >> 2) * 1024 + (kk & 3) * 32
                                                : (kk >> 2) * kBox + (kk & 3) * 32;
                const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
                umma_bf16_elect(tmem + b * 128, umma_desc_sw128(qa + qoff, 16, p.q_atoms ? 2048 : 1024),
                                umma_desc_sw128(ka + off, 16, 1024), idesc_s, kk > 0);
              }
              umma_commit_elect(&B.s_full[b]);
              umma_commit_elect(&B.q_empty[qs]);
              if (b) {
                gj1 = next_gj;
                kvb1 = c;
              } else {
                gj0 = next_gj;
                kvb0 = c;
              }
              ++si;
              next_gj = after_gj;  // descriptors are read two tiles ahead
              if (si + 1 < n) after_gj = load_desc(p, tile_of(si + 1)).x;
              idle = 0;
              continue;
            }
          }
          // ---- nothing ready: block briefly on the next O's P
          if (oi < si) mbar_try_wait_hint(&B.p_full[oi & 1], (oi >> 1) & 1, kIssuerNap);
          else __nanosleep(32);
          if (++idle > kWaitLimit) {
            msa_record_error(kErrTimeout);
            *fail = 1;
          }
        }
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
    // ================================================================ softmax + epilogue
    // Warpgroup wg handles tiles k = wg, wg+2, ... with S[wg], P[wg], O[wg].
    const int wg = (warp - 4) >> 2;
    const int row = (tid - 128) & 127;         // tile row = TMEM lane
    const uint32_t lane_addr = (uint32_t)(32 * (warp & 3)) << 16;
    const int G = p.G;
    const int qi = row / G, h = row % G;
    // software prefetch: descriptors two of this warpgroup's tiles ahead, entry one ahead
    int4 d_next = wg < n ? load_desc(p, tile_of(wg)) : make_int4(0, 0, 0, 0);
    int4 d_next2 = wg + 2 < n ? load_desc(p, tile_of(wg + 2)) : d_next;
    int32_t e_next = qi < d_next.z ? p.entries[d_next.y + qi] : -1;
    const uint32_t s_tmem = tmem + lane_addr + wg * 128;
    const uint32_t o_tmem = tmem + lane_addr + 256 + wg * 128;
    for (int k = wg; k < n; k += 2) {
      const int use = k >> 1;  // this warpgroup's use count of its buffers
      const int4 d = d_next;
      const int32_t ent = e_next;
      if (k + 2 < n) {
        e_next = qi < d_next2.z ? p.entries[d_next2.y + qi] : -1;
        d_next = d_next2;
        if (k + 4 < n) d_next2 = load_desc(p, tile_of(k + 4));
      }
      const int j = d.x % p.nblk;
      // ---------------- softmax of tile k
      if (!wait_or_fail(&B.s_full[wg], use & 1, fail)) break;
      tmem_fence_after();
      float v[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_tmem + c * 32, v + c * 32);
      tmem_wait_ld();
      // causal mask: key j*128 + col is visible to the query iff it is <= the query position
      const int64_t qpos = ent >= 0 ? p.q_start + ent / p.topk : -1;
      const int64_t lim64 = qpos - (int64_t)j * 128;  // last visible column
      // an empty query slot of the tile gets P = 0 through its exponent (scale 0, offset -inf)
      if (ent >= 0 && lim64 < 127) {
        const int lim = lim64 < -1 ? -1 : (int)lim64;
#pragma unroll
        for (int x = 0; x < 128; ++x)
          if (x > lim) v[x] = -INFINITY;
      }
      // row max: three-input max over column pairs, four independent chains
      float m4[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
      for (int x = 4; x < 128; x += 2) m4[(x >> 1) & 3] = max3(m4[(x >> 1) & 3], v[x], v[x + 1]);
      const float mx = ent >= 0 ? fmaxf(max3(m4[0], m4[1], m4[2]), m4[3]) : -INFINITY;
      const float mscaled = (mx == -INFINITY ? 0.f : mx) * kLog2e;
      const float sc = ent >= 0 ? kLog2e : 0.f;
      const float off = ent >= 0 ? -mscaled : -INFINITY;
      // p = 2^(s*log2e - max*log2e): the scaling in packed pairs, the exponent on the SFU
      float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int x = 0; x < 128; x += 2) {
        fma2(v[x], v[x + 1], v[x], v[x + 1], sc, sc, off, off);
        v[x] = ex2(v[x]);
        v[x + 1] = ex2(v[x + 1]);
        add2(l8[(x >> 1) & 3], l8[4 + ((x >> 1) & 3)], v[x], v[x + 1]);
      }
      // P row (bf16 pairs) into the first 64 columns of this tile's S buffer: the A operand
      // of the O MMA
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t pk[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) pk[x] = pack_bf16x2(v[h2 * 64 + 2 * x], v[h2 * 64 + 2 * x + 1]);
        tmem_st32(s_tmem + h2 * 32, pk);
      }
      tmem_wait_st();
      tmem_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.p_full[wg]);
      const float l = ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
      // ---------------- epilogue of tile k: normalised bf16 partial + fp32 LSE
      // Partials are stored chunk-major, part_o[c][row][8] with row = ((t*Hkv+g)*k+slot)*G+h:
      // the G rows of one query are adjacent, so a warp store covers 128-byte segments.
      if (!wait_or_fail(&B.o_full[wg], use & 1, fail)) break;
      tmem_fence_after();
      const float inv = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(o_tmem + c * 32, v + c * 32);
      tmem_wait_ld();
      tmem_fence_before();
      if (ent >= 0) {
        const int64_t t = ent / p.topk;
        const int64_t prow_idx = ((t * p.Hkv + d.x / lists_per_group) * p.topk + ent % p.topk) * G + h;
        __stcs(p.part_lse + prow_idx, l > 0.f ? mx + __logf(l) : -INFINITY);
        uint4* dst = reinterpret_cast<uint4*>(p.part_o) + prow_idx;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          uint4 u;
#pragma unroll
          for (int e = 0; e < 8; e += 2) mul2(v[c * 8 + e], v[c * 8 + e + 1], inv, inv);
          u.x = pack_bf16x2(v[c * 8 + 0], v[c * 8 + 1]);
          u.y = pack_bf16x2(v[c * 8 + 2], v[c * 8 + 3]);
          u.z = pack_bf16x2(v[c * 8 + 4], v[c * 8 + 5]);
          u.w = pack_bf16x2(v[c * 8 + 6], v[c * 8 + 7]);
          __stcs(dst + (int64_t)c * p.part_rows, u);  // read once, by the merge
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.o_free[wg]);
    }
  }
  // ------------------------------------------------------------------ teardown
  tmem_fence_before();
  __syncthreads();
  if (warp == 1) {
    tmem_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols)
                 : "memory");
  }
}

}  // namespace

cudaError_t launch_bucket_lists(const int32_t* ids, const int32_t* epos, int32_t T, int32_t Hkv,
                                int32_t topk, int32_t nblk, int32_t win, int32_t qpt,
                                const int32_t* counts, int32_t* offsets, int32_t* entries,
                                int32_t* group_base, int32_t* tile_offsets, int4* desc,
                                const int32_t* dcnt, int64_t npairs, int32_t* porder,
                                cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const int32_t nwin = (T + win - 1) / win;
  const int32_t nseg = Hkv * nwin;  // (group, window) segments
  // tile_offsets holds the segment-local tile prefix [nseg][nblk+1], then the segment tile
  // bases [nseg+1]
  int32_t* tile_local = tile_offsets;
  int32_t* seg_tile_base = tile_offsets + (size_t)nseg * (nblk + 1);
  const size_t smem = 8 * (size_t)nseg;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(bucket_lists_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // the query-major pairs' deal in extra blocks, one per window
  const PairDeal deal = dcnt && npairs > 0 ? pair_deal_geometry(npairs) : PairDeal{1, 1, 0, 0};
  bucket_lists_kernel<<<(unsigned)(nseg + deal.nwin), kListThreads, smem, stream>>>(
      counts, nseg, nblk, qpt, offsets, tile_local, group_base, seg_tile_base, desc, dcnt, npairs,
      (int32_t)deal.grid, deal.rpw, porder);
  const int32_t rows = T * Hkv;  // T*Hkv*topk fits in int32 (checked by the callers)
  const int rgrid = (int)std::max<int64_t>(1, std::min<int64_t>((rows + 255) / 256, (int64_t)sm_count() * 8));
  const bool vec4 = topk % 4 == 0 && (reinterpret_cast<uintptr_t>(ids) & 15) == 0 &&
                    (reinterpret_cast<uintptr_t>(epos) & 15) == 0;
  bucket_place_kernel<<<rgrid, 256, 0, stream>>>(ids, epos, rows, Hkv, topk, nblk, win, nwin,
                                                 offsets, group_base, entries, vec4);
  return cudaGetLastError();
}

cudaError_t launch_bucket(const int32_t* block_ids, int32_t T, int32_t Hkv, int32_t topk,
                          int32_t nblk, int32_t win, int32_t qpt, int32_t* offsets,
                          int32_t* entries, int32_t* counts, int32_t* group_base,
                          int32_t* tile_offsets, int32_t* epos, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const int32_t nwin = (T + win - 1) / win;
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)Hkv * nwin * nblk, stream);
  if (e != cudaSuccess) return e;
  e = launch_select_count(block_ids, T, (int64_t)nblk * 128, Hkv, 1, topk, nblk, win,
                          DenseWorkspace{}, counts, epos, stream);
  if (e != cudaSuccess) return e;
  return launch_bucket_lists(block_ids, epos, T, Hkv, topk, nblk, win, qpt, counts, offsets,
                             entries, group_base, tile_offsets, nullptr, nullptr, 0, nullptr,
                             stream);
}

cudaError_t launch_sparse_prefill(const PrefillArgs& a, cudaStream_t stream) {
  const int G = a.Hq / a.Hkv;
  const int qpt = kRows / G;
  const PrefillWorkspace W = prefill_ws_layout(a.T, a.Hkv, a.topk, a.nblk, G, true);
  int32_t* counts = reinterpret_cast<int32_t*>(a.workspace + W.counts);
  int32_t* group_base = reinterpret_cast<int32_t*>(a.workspace + W.group_base);
  int32_t* tile_offsets = reinterpret_cast<int32_t*>(a.workspace + W.tile_offsets);
  int32_t* offsets = reinterpret_cast<int32_t*>(a.workspace + W.offsets);
  int32_t* entries = reinterpret_cast<int32_t*>(a.workspace + W.entries);
  uint16_t* part_o = reinterpret_cast<uint16_t*>(a.workspace + W.part_o);
  float* part_lse = reinterpret_cast<float*>(a.workspace + W.part_lse);
  int4* tile_desc = reinterpret_cast<int4*>(a.workspace + W.tile_desc);
  int32_t* epos = reinterpret_cast<int32_t*>(a.workspace + W.epos);
  const int32_t win = prefill_window(a.T, a.nblk, a.topk, G);
  const int32_t nwin = prefill_nwin(a.T, a.nblk, a.topk, G);
  // G 8 / 16: the slots shared by many queries of a query pair are computed query-major; the
  // block-major pass and the merge's slot skipping then use the residual selections
  const bool hybrid = prefill_hybrid(G);
  DenseWorkspace dw{};
  const int32_t* ids = a.block_ids;
  if (hybrid) {
    dw.qperm = reinterpret_cast<int32_t*>(a.workspace + W.qperm);
    dw.porder = reinterpret_cast<int32_t*>(a.workspace + W.porder);
    dw.residual = reinterpret_cast<int32_t*>(a.workspace + W.residual);
    dw.dcnt = reinterpret_cast<int32_t*>(a.workspace + W.dcnt);
    dw.dblk = reinterpret_cast<int32_t*>(a.workspace + W.dblk);
    dw.dmask = reinterpret_cast<uint32_t*>(a.workspace + W.dmask);
    dw.part_o = reinterpret_cast<uint16_t*>(a.workspace + W.dense_o);
    dw.part_lse = reinterpret_cast<float*>(a.workspace + W.dense_lse);
    ids = dw.residual;
  }
  // (a) selection (query order, shared blocks) and the count of the block-major selections in
  // one kernel; the lists' offsets with the tile descriptors; the placement of the entries
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)a.Hkv * nwin * a.nblk, stream);
  if (e != cudaSuccess) return e;
  e = launch_select_count(a.block_ids, a.T, a.S_kv, a.Hkv, G, a.topk, a.nblk, win, dw, counts,
                          epos, stream);
  if (e != cudaSuccess) return e;
  // the list offsets, with the query-major pairs' deal to the CTAs in the same launch
  e = launch_bucket_lists(ids, epos, a.T, a.Hkv, a.topk, a.nblk, win, qpt, counts, offsets,
                          entries, group_base, tile_offsets, tile_desc, hybrid ? dw.dcnt : nullptr,
                          hybrid ? prefill_pairs(a.T, a.Hkv, G) : 0, dw.porder, stream);
  if (e != cudaSuccess) return e;

  CUtensorMap qmap, kmap, vmap;
  // Query rows, preferably as one copy per query: dims {channel in half, head mod 8, half,
  // head / 8, t*Hkv + g} (the half's stride is below the head's, so the box lands as
  // [G/8][half][8 heads][64 channels]); otherwise two 3-D copies per query.
  int32_t q_atoms = 0;
  if (G % 8 == 0) {
    const uint64_t q5dims[5] = {64, 8, 2, (uint64_t)G / 8, (uint64_t)a.T * a.Hkv};
    const uint64_t q5strides[4] = {(uint64_t)a.D * 2, 128, (uint64_t)8 * a.D * 2,
                                   (uint64_t)G * a.D * 2};
    const uint32_t q5box[5] = {64, 8, 2, (uint32_t)G / 8, 1};
    q_atoms = encode_bf16_map(&qmap, a.q, 5, q5dims, q5strides, q5box, true) ? 1 : 0;
  }
  const uint64_t qdims[3] = {(uint64_t)a.D, (uint64_t)a.Hq, (uint64_t)a.T};
  const uint64_t qstrides[2] = {(uint64_t)a.D * 2, (uint64_t)a.Hq * a.D * 2};
  const uint32_t qbox[3] = {64, (uint32_t)G, 1};
  const uint64_t kv_rows = a.page_table ? (uint64_t)a.num_pages * 128 : (uint64_t)a.S_kv;
  const uint64_t dims[3] = {(uint64_t)a.D, (uint64_t)a.Hkv, kv_rows};
  const uint64_t strides[2] = {(uint64_t)a.D * 2, (uint64_t)a.Hkv * a.D * 2};
  const uint32_t box[3] = {64, 1, 128};
  if ((!q_atoms && !encode_bf16_map(&qmap, a.q, 3, qdims, qstrides, qbox, true)) ||
      !encode_bf16_map(&kmap, a.k, 3, dims, strides, box, true) ||
      !encode_bf16_map(&vmap, a.v, 3, dims, strides, box, true))
    return cudaErrorInvalidValue;
  PreKParams p;
  p.entries = entries;
  p.desc = tile_desc;
  p.tile_offsets = tile_offsets;
  p.Hkv = a.Hkv;
  p.G = G;
  p.topk = a.topk;
  p.nblk = a.nblk;
  p.qpt = qpt;
  p.nwin = nwin;
  p.q_atoms = q_atoms;
  p.q_start = a.S_kv - a.T;
  p.page_table = a.page_table;
  p.num_pages = a.num_pages;
  p.part_o = part_o;
  p.part_rows = (int64_t)a.T * a.Hkv * a.topk * G;
  p.part_lse = part_lse;
  e = cudaFuncSetAttribute(prefill_block_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  // the in-kernel register split assumes exactly kLaunchRegs registers per thread at launch
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, prefill_block_tc_kernel);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  prefill_block_tc_kernel<<<sm_count(), kThreads, kSmemBytes, stream>>>(qmap, kmap, vmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (hybrid) {
    e = launch_dense_attention(qmap, kmap, vmap, q_atoms, a.T, a.S_kv, a.Hkv, G, a.page_table,
                               a.num_pages, dw, stream);
    if (e != cudaSuccess) return e;
  }
  return launch_lse_merge_chunked(part_o, part_lse, ids, hybrid ? dw.part_o : nullptr,
                                  hybrid ? dw.part_lse : nullptr, (int64_t)a.T * a.Hkv, a.topk, G,
                                  a.o, a.lse, stream);
}

}  // namespace msa
