// Query-major part of the sparse prefill: the KV blocks that many queries of a query pair
// share are computed with the queries as the outer loop, the scattered remainder stays
// block-major (prefill.cu).
//
// Together AI MiniMax-M3 serving article, section "KV-block-major sparse attention reduces
// redundant KV movement": the block-major remap exists because queries that chose the same
// KV block would otherwise each move it from HBM; its cost is one partial output per
// selection and a Log-Sum-Exp reduction over them. Where neighbouring queries choose the
// same blocks (the sink, the local block, a shared set), a query-major pass moves each such
// block once for all of them as well, and accumulates their output across blocks without
// partials. The combination is exact: every selection is computed once, by one of the two
// passes, and the merge (row a7) combines the query-major partial with the block-major ones.
//
// GB300 design.
//  (o, a) select_count_kernel, one CTA per (group, 128-query span): orders the span's queries
//      so that those choosing the span's popular blocks (chosen by at least half of the span)
//      come first, so that queries sharing blocks fill the same tiles; then, per pair of
//      128/G-query tiles (consecutive slots of that order), keeps the blocks chosen by at least
//      half of the pair's queries (at most kMaxDense, ascending) with a bit mask of the queries
//      that chose each, writes the residual selections (the shared ones replaced by -1) and
//      counts each residual selection into its block-major list.
//  (b) prefill_dense_tc_kernel, one persistent CTA per SM over the pairs: the two tiles of a
//      pair share each K/V block load; per block S = Q K^T and O += P V run on tcgen05 with
//      S, P and O in tensor memory; one softmax warpgroup per tile keeps a running row max and
//      sum (rows of queries that did not choose the block get P = 0; O and the sum are
//      rescaled only when the max grows by more than 2^8), and writes one bf16 partial and its
//      LSE per (query, head) after the pair's last block.
#include <climits>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"
#include "pair_deal.cuh"
#include "softmax_math.cuh"

MSA_DEFINE_ERROR_WORD(dense)

namespace msa {

namespace {

// ------------------------------------------------------------------------------ selection
// The ids a pair can choose are at most the local block of its span's last query (nb blocks);
// they are counted in windows of hw <= kHistBlocks blocks (hw: the chunk's block count, capped):
// a query mask per block in shared memory, filled with shared atomics (a block's count is its
// mask's popcount: a query chooses a block at most once), then a prefix scan over the window
// ranks the dense blocks in ascending order.
constexpr int kHistBlocks = 16384;

// Query of pair slot `pos` of group g (-1: past the chunk). Without an order, slot = query.
__device__ __forceinline__ int64_t slot_query(const int32_t* qperm, int64_t npos, int g,
                                              int64_t pos, int32_t T) {
  if (!qperm) return pos < T ? pos : -1;
  return qperm[(int64_t)g * npos + pos];
}

constexpr int kSpan = 128;

struct SelectParams {
  const int32_t* block_ids;  // [T, Hkv, topk]
  int32_t T, Hkv, topk;
  int64_t q_start;
  // query-major selection (G 8 / 16)
  bool hybrid, ordered;
  int32_t nb_max;            // blocks of the whole key range (ordering histogram)
  int32_t qpt, ppg, thr, hw;
  int64_t npos;
  int32_t* qperm;            // [Hkv, npos]
  int32_t* residual;         // [T, Hkv, topk]
  int32_t* dcnt;             // [pairs]
  int32_t* dblk;             // [pairs, kMaxDense]
  uint32_t* dmask;           // [pairs, kMaxDense]
  float* part_lse;           // [T*Hkv*G] query-major LSE, -inf until written
  int32_t G;
  // bucketing of the remaining (block-major) selections
  int32_t nblk, win, nwin;
  int32_t ph;                // per-warp pair histogram length (0: windowed CTA-wide selection)
  int32_t* counts;           // [Hkv*nwin, nblk], zero on entry
  int32_t* epos;             // [T, Hkv, topk]: place of each counted selection in its list
  bool vec4;                 // topk % 4 == 0 and block_ids 16-byte aligned: rows move as int4
};

// Blocks per pair histogram for the one-warp-per-pair selection (smaller key ranges); longer
// key ranges take the CTA-wide windowed selection.
constexpr int kPairHist = 1024;
// A row's ids are loaded, and its list counts taken, kIdBatch at a time: the loads (and the
// atomics, whose returned place is stored) are all in flight before any result is used.
constexpr int kIdBatch = 16;

// Writes j[0..n) (a batch of one row's slots) to dst[at..]: four at a time when the batch is
// whole and the rows are int4-aligned.
__device__ __forceinline__ void store_batch(const SelectParams& p, int32_t* dst, int64_t at,
                                            const int32_t (&j)[kIdBatch], int n) {
  if (p.vec4 && n >= kIdBatch) {
#pragma unroll
    for (int q = 0; q < kIdBatch / 4; ++q)
      reinterpret_cast<int4*>(dst + at)[q] = make_int4(j[4 * q], j[4 * q + 1], j[4 * q + 2], j[4 * q + 3]);
  } else {
#pragma unroll
    for (int u = 0; u < kIdBatch; ++u)
      if (u < n) dst[at + u] = j[u];
  }
}

// Loads slots k0.. of selection row `row` (a batch; -1 past topk or for an invalid row).
__device__ __forceinline__ void load_batch(const SelectParams& p, int64_t row, int k0, bool valid,
                                           int32_t (&j)[kIdBatch]) {
  if (p.vec4 && k0 + kIdBatch <= p.topk) {
    const int4* src = reinterpret_cast<const int4*>(p.block_ids + row * p.topk + k0);
#pragma unroll
    for (int q = 0; q < kIdBatch / 4; ++q) {
      const int4 v = valid ? src[q] : make_int4(-1, -1, -1, -1);
      j[4 * q] = v.x;
      j[4 * q + 1] = v.y;
      j[4 * q + 2] = v.z;
      j[4 * q + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int u = 0; u < kIdBatch; ++u)
      j[u] = valid && k0 + u < p.topk ? p.block_ids[row * p.topk + k0 + u] : -1;
  }
}

// Counts up to kIdBatch selections (ids j[], -1 = none; `n` of them valid slots) of one row into
// their lists; each one's place in its list goes to epos[at + u] (-1 for a slot not counted).
__device__ __forceinline__ void count_batch(const SelectParams& p, const int32_t (&j)[kIdBatch],
                                            int64_t list0, int64_t at, int n) {
  int32_t pos[kIdBatch];
#pragma unroll
  for (int u = 0; u < kIdBatch; ++u) {
    pos[u] = -1;
    if (u < n && j[u] >= 0) {
      if (j[u] < p.nblk) pos[u] = atomicAdd(&p.counts[list0 + j[u]], 1);
      else msa_record_error(kErrBadBlock);
    }
  }
  store_batch(p, p.epos, at, pos, n);
}

// One CTA per (group g, 128-query span), one thread per query of the span. The span's ids are
// staged in shared memory once.
//  (o) [hybrid, ordered] the span's block histogram; each query's number of selections among
//      the blocks chosen by at least half of the span; a stable rank by that number descending
//      gives the slot order (qperm): consecutive slots form the pairs of 2*128/G queries.
//  (a) [hybrid] per pair of the span: the blocks chosen by at least half of the pair's queries
//      (at most kMaxDense, ascending) with a query bit mask each; the pair's selections of those
//      blocks are replaced by -1 in `residual`. One warp per pair (key ranges of at most
//      kPairHist blocks), else the whole CTA per pair in windows of hw blocks.
//  (c) each remaining selection (t, slot) of block j is counted into list (g, t/win, j), and its
//      place in that list is kept in `epos` (the bucketing places it there once the lists'
//      offsets are known).
__global__ void __launch_bounds__(kSpan)
    select_count_kernel(const SelectParams p) {
  extern __shared__ __align__(16) uint8_t sel_smem[];
  // slot order: per warp, the number of its queries with each score key (score + 1, 0..topk+1),
  // and per key the number of the span's queries with a larger key
  constexpr int kKeys = 96;  // > topk + 1 for topk <= 64
  __shared__ int32_t key_cnt[kSpan / 32][kKeys];
  __shared__ int32_t key_above[kKeys];
  __shared__ int32_t s_query[kSpan];   // query of each slot of the span (-1: none)
  __shared__ int16_t s_row[kSpan];     // span row (t - span start) of each slot
  __shared__ int32_t warp_sum[kSpan / 32];
  const int r = threadIdx.x, lane = r & 31, warp = r >> 5;
  const int g = (int)(blockIdx.x % p.Hkv);
  const int64_t span = blockIdx.x / p.Hkv;
  const int64_t t_me = span * kSpan + r;
  const bool valid = t_me < p.T;
  const int nvalid = (int)min((int64_t)kSpan, (int64_t)p.T - span * kSpan);
  const int64_t row_me = t_me * p.Hkv + g;
  if (!p.hybrid) {
    // (c) only: count the selections of this thread's query
    if (!valid) return;
    const int64_t list0 = ((int64_t)g * p.nwin + t_me / p.win) * p.nblk;
    for (int k0 = 0; k0 < p.topk; k0 += kIdBatch) {
      int32_t j[kIdBatch];
      load_batch(p, row_me, k0, true, j);
      count_batch(p, j, list0, row_me * p.topk + k0, p.topk - k0);
    }
    return;
  }
  // the span's selections [topk][kSpan] (slot-major: a warp's rows fall in distinct banks;
  // residuals are written over them in (a)), then the histograms of (o) and (a)
  int32_t* s_ids = reinterpret_cast<int32_t*>(sel_smem);
  uint8_t* hist = sel_smem + (size_t)kSpan * p.topk * 4;
  for (int k0 = 0; k0 < p.topk; k0 += kIdBatch) {
    int32_t j[kIdBatch];  // a row's ids requested together, then stored
    load_batch(p, row_me, k0, valid, j);
#pragma unroll
    for (int u = 0; u < kIdBatch; ++u)
      if (k0 + u < p.topk) s_ids[(k0 + u) * kSpan + r] = j[u];
  }
  // ---------------- (o) slot order of the span
  if (p.ordered) {
    uint32_t* span_cnt = reinterpret_cast<uint32_t*>(hist);  // [nb_max]
    for (int j = r; j < p.nb_max; j += kSpan) span_cnt[j] = 0u;
    for (int j = r; j < (kSpan / 32) * kKeys; j += kSpan) (&key_cnt[0][0])[j] = 0;
    __syncthreads();
    for (int k = 0; k < p.topk; ++k) {
      const int32_t j = s_ids[k * kSpan + r];
      if (j >= 0 && j < p.nb_max) atomicAdd(&span_cnt[j], 1u);
    }
    __syncthreads();
    int sc = -1;  // slots past the chunk sort last
    if (valid) {
      sc = 0;
      for (int k = 0; k < p.topk; ++k) {
        const int32_t j = s_ids[k * kSpan + r];
        if (j >= 0 && j < p.nb_max && 2 * (int)span_cnt[j] >= nvalid) ++sc;
      }
    }
    // stable rank by score, descending: the queries with a larger score, then those with the
    // same score and a lower span row (earlier warps' counts, then lower lanes of this warp)
    const int key = sc + 1;
    const uint32_t same = __match_any_sync(0xffffffffu, key);
    const int below = __popc(same & ((1u << lane) - 1u));
    if (below == 0) key_cnt[warp][key] = __popc(same);
    __syncthreads();
    if (warp == 0) {
      // key_above[k] = number of queries with key > k (suffix sums over three 32-key groups)
      int t3[3], x3[3];
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        const int k = lane + 32 * c;
        t3[c] = 0;
#pragma unroll
        for (int w = 0; w < kSpan / 32; ++w) t3[c] += key_cnt[w][k];
        x3[c] = t3[c];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_down_sync(0xffffffffu, x3[c], o);
          if (lane + o < 32) x3[c] += y;
        }
      }
      const int tot1 = __shfl_sync(0xffffffffu, x3[1], 0), tot2 = __shfl_sync(0xffffffffu, x3[2], 0);
      key_above[lane] = x3[0] - t3[0] + tot1 + tot2;
      key_above[lane + 32] = x3[1] - t3[1] + tot2;
      key_above[lane + 64] = x3[2] - t3[2];
    }
    __syncthreads();
    int rank = key_above[key] + below;
    for (int w = 0; w < warp; ++w) rank += key_cnt[w][key];
    s_query[rank] = valid ? (int32_t)t_me : -1;
    s_row[rank] = (int16_t)r;
    p.qperm[(int64_t)g * p.npos + span * kSpan + rank] = valid ? (int32_t)t_me : -1;
  } else {
    s_query[r] = valid ? (int32_t)t_me : -1;
    s_row[r] = (int16_t)r;
  }
  __syncthreads();  // slot order and staged ids (the histogram space is reused below)
  // ---------------- (a) shared blocks of each pair of the span
  const int nq = 2 * p.qpt;
  const int pairs = kSpan / nq;
  const int64_t nb = (p.q_start + span * kSpan + nvalid - 1) / 128 + 1;  // blocks the span sees
  for (int rr = r; rr < kSpan * p.G / 4; rr += kSpan) {  // G 8 / 16: four heads per store
    const int32_t t = s_query[rr / (p.G / 4)];
    if (t >= 0)
      reinterpret_cast<float4*>(p.part_lse + ((int64_t)t * p.Hkv + g) * p.G)[rr % (p.G / 4)] =
          make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  }
  if (p.ph > 0 && nb <= p.ph) {
    // one warp per pair (pairs of 32 slots) or per two pairs (16 slots): lane = slot of the pair
    const int ppw = pairs / (kSpan / 32);  // pairs per warp: 1 or 2
    uint32_t* msk = reinterpret_cast<uint32_t*>(hist) + warp * p.ph;
    int16_t* rnk = reinterpret_cast<int16_t*>(hist + (kSpan / 32) * p.ph * 4) + warp * p.ph;
    for (int i = 0; i < ppw; ++i) {
      const int pi = warp * ppw + i;  // pair within the span
      const int64_t pslot = span * pairs + pi;
      const bool live = pslot < p.ppg;  // uniform for the warp
      if (!live) break;
      const int64_t pair = (int64_t)g * p.ppg + pslot;
      for (int j = lane; j < nb; j += 32) msk[j] = 0u;
      __syncwarp();
      const bool mine = lane < nq;
      const int slot = pi * nq + lane;
      const int srow = mine ? s_row[slot] : 0;
      const bool qv = mine && s_query[slot] >= 0;
      if (qv)
        for (int k = 0; k < p.topk; ++k) {
          const int32_t id = s_ids[k * kSpan + srow];
          if (id >= 0 && id < nb) atomicOr(&msk[id], 1u << lane);
        }
      __syncwarp();
      // ascending ranks of the dense blocks, 32 blocks per step
      int ranked = 0;
      for (int j0 = 0; j0 < nb; j0 += 32) {
        const int j = j0 + lane;
        const uint32_t m = j < nb ? msk[j] : 0u;
        const bool dense = __popc(m) >= p.thr;
        const uint32_t bal = __ballot_sync(0xffffffffu, dense);
        const int rank = ranked + __popc(bal & ((1u << lane) - 1u));
        int16_t rk = -1;
        if (dense && rank < kMaxDense) {
          p.dblk[pair * kMaxDense + rank] = j;
          p.dmask[pair * kMaxDense + rank] = m;
          rk = (int16_t)rank;
        }
        if (j < nb) rnk[j] = rk;
        ranked += __popc(bal);
      }
      if (lane == 0) p.dcnt[pair] = ranked < kMaxDense ? ranked : kMaxDense;
      __syncwarp();
      // the pair's residual selections: the dense ones leave, the others stay
      if (qv)
        for (int k = 0; k < p.topk; ++k) {
          const int32_t id = s_ids[k * kSpan + srow];
          if (id >= 0 && id < nb && rnk[id] >= 0) s_ids[k * kSpan + srow] = -1;
        }
      __syncwarp();
    }
  } else {
    uint32_t* msk = reinterpret_cast<uint32_t*>(hist);           // [hw]
    int16_t* rnk = reinterpret_cast<int16_t*>(hist + 4 * p.hw);  // [hw] dense rank or -1
    const int n = nq * p.topk;
    for (int i = 0; i < pairs; ++i) {
      const int64_t pslot = span * pairs + i;
      if (pslot >= p.ppg) break;
      const int64_t pair = (int64_t)g * p.ppg + pslot;
      int ranked = 0;  // dense blocks ranked in earlier windows
      for (int64_t base = 0; base < nb; base += p.hw) {
        const int w = (int)min((int64_t)p.hw, nb - base);
        for (int j = r; j < w; j += kSpan) msk[j] = 0u;
        __syncthreads();
        for (int e = r; e < n; e += kSpan) {
          const int q = e / p.topk, slot = i * nq + q;
          if (s_query[slot] < 0) continue;
          const int64_t id = s_ids[(e % p.topk) * kSpan + s_row[slot]];
          if (id >= base && id < base + w) atomicOr(&msk[id - base], 1u << q);
        }
        __syncthreads();
        const int per = (w + kSpan - 1) / kSpan;
        const int j0 = r * per, j1 = min(w, j0 + per);
        int local = 0;
        for (int j = j0; j < j1; ++j) local += __popc(msk[j]) >= p.thr ? 1 : 0;
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (lane == 31) warp_sum[warp] = incl;
        __syncthreads();
        int rank = ranked + incl - local, total = 0;
        for (int v = 0; v < kSpan / 32; ++v) {
          if (v < warp) rank += warp_sum[v];
          total += warp_sum[v];
        }
        for (int j = j0; j < j1; ++j) {
          const uint32_t m = msk[j];
          int16_t rk = -1;
          if (__popc(m) >= p.thr) {
            if (rank < kMaxDense) {
              p.dblk[pair * kMaxDense + rank] = (int32_t)(base + j);
              p.dmask[pair * kMaxDense + rank] = m;
              rk = (int16_t)rank;
            }
            ++rank;
          }
          rnk[j] = rk;
        }
        __syncthreads();
        for (int e = r; e < n; e += kSpan) {
          const int q = e / p.topk, slot = i * nq + q;
          if (s_query[slot] < 0) continue;
          int32_t* at = &s_ids[(e % p.topk) * kSpan + s_row[slot]];
          const int32_t id = *at;
          if (id >= base && id < base + w && rnk[id - base] >= 0) *at = -1;
        }
        ranked += total;
        __syncthreads();  // the window's arrays are reused by the next window / pair
      }
      if (r == 0) p.dcnt[pair] = ranked < kMaxDense ? ranked : kMaxDense;
    }
  }
  __syncthreads();  // every pair's residuals are in s_ids
  // ---------------- (c) count the remaining selections of this thread's query into their lists
  if (!valid) return;
  const int64_t list0 = ((int64_t)g * p.nwin + t_me / p.win) * p.nblk;
  for (int k0 = 0; k0 < p.topk; k0 += kIdBatch) {
    int32_t j[kIdBatch];
#pragma unroll
    for (int u = 0; u < kIdBatch; ++u) j[u] = k0 + u < p.topk ? s_ids[(k0 + u) * kSpan + r] : -1;
    store_batch(p, p.residual, row_me * p.topk + k0, j, p.topk - k0);
    count_batch(p, j, list0, row_me * p.topk + k0, p.topk - k0);
  }
}

}  // namespace

// Per-warp pair histogram length: the chunk's key blocks, when they are few enough.
int32_t pair_hist_len(int64_t S_kv) {
  const int64_t nbk = (S_kv + 127) / 128;
  return nbk <= kPairHist ? (int32_t)((nbk + 7) / 8 * 8) : 0;
}

// Shared memory of select_count_kernel: the span's ids, then the larger of the ordering
// histogram and the pair histograms.
size_t select_count_smem_bytes(int64_t S_kv, int32_t G, int32_t topk) {
  const int64_t nbk = (S_kv + 127) / 128;
  const int64_t hw = std::min<int64_t>(kHistBlocks, nbk);
  const int64_t nb_max = std::min<int64_t>(nbk, INT32_MAX);
  if (!prefill_hybrid(G)) return 16;
  const int32_t ph = pair_hist_len(S_kv);
  size_t h = ph > 0 ? (size_t)(kSpan / 32) * ph * 6 : (size_t)6 * hw;
  if (nb_max <= kHistBlocks) h = std::max(h, (size_t)4 * nb_max);
  return (size_t)kSpan * topk * 4 + (h + 15) / 16 * 16;
}

cudaError_t launch_select_count(const int32_t* block_ids, int32_t T, int64_t S_kv, int32_t Hkv,
                                int32_t G, int32_t topk, int32_t nblk, int32_t win,
                                const DenseWorkspace& w, int32_t* counts, int32_t* epos,
                                cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  SelectParams p{};
  p.block_ids = block_ids;
  p.T = T;
  p.Hkv = Hkv;
  p.topk = topk;
  p.q_start = S_kv - T;
  p.hybrid = prefill_hybrid(G) && w.residual != nullptr;
  p.G = G;
  p.qpt = 128 / G;
  p.ppg = (int32_t)((T + 2 * p.qpt - 1) / (2 * p.qpt));
  p.thr = std::max(2, (2 * p.qpt + 1) / 2);  // at least half of the pair's queries
  const int64_t nbk = (S_kv + 127) / 128;
  // the window covers every block of the chunk when it fits (one pass), else kHistBlocks
  p.hw = (int32_t)std::min<int64_t>(kHistBlocks, nbk);
  // pair order: while the key range's block counts fit in shared memory, else slot = query
  p.nb_max = (int32_t)std::min<int64_t>(nbk, INT32_MAX);
  p.ordered = p.nb_max <= kHistBlocks;
  p.npos = prefill_qpos(T);
  p.qperm = w.qperm;
  p.residual = w.residual;
  p.dcnt = w.dcnt;
  p.dblk = w.dblk;
  p.dmask = w.dmask;
  p.part_lse = w.part_lse;
  p.nblk = nblk;
  p.win = win;
  p.nwin = (T + win - 1) / win;
  p.counts = counts;
  p.epos = epos;
  p.vec4 = (topk % 4) == 0 && (reinterpret_cast<uintptr_t>(block_ids) & 15) == 0;
  p.ph = pair_hist_len(S_kv);
  const size_t smem = p.hybrid ? select_count_smem_bytes(S_kv, G, topk) : 16;
  cudaError_t e = cudaFuncSetAttribute(select_count_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t nspan = (T + kSpan - 1) / kSpan;
  select_count_kernel<<<(unsigned)(Hkv * nspan), kSpan, smem, stream>>>(p);
  return cudaGetLastError();
}

namespace {

// ------------------------------------------------------------------------------ attention
constexpr int kThreads = 384;
constexpr uint32_t kBox = 128 * 64 * 2;          // 128 rows x 64 channels bf16 = 16 KB
constexpr uint32_t kTileBytes = 2 * kBox;        // a query tile, a K block or a V block: 32 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.0f;                 // log2 headroom before O is rescaled
constexpr uint32_t kTmemCols = 512;              // S_A, S_B at 0 / 128; O_A, O_B at 256 / 384
constexpr uint32_t kIssuerNap = 100;             // ns an idle MMA issuer blocks on a barrier
constexpr int kLaunchRegs = 168;
constexpr int kRegsLow = 88;
constexpr int kRegsHigh = 208;

// shared memory (offsets from a 1024-aligned base): the pair's two query tiles, a two-deep
// ring of K/V blocks, barriers
constexpr uint32_t kOffQ = 0;                    // Q_A, Q_B
constexpr uint32_t kOffKV = 2 * kTileBytes;      // {K, V}[2]
constexpr uint32_t kOffBar = 6 * kTileBytes;
// blocks of the CTA's pair in each round (0: no pair or no shared block), one byte per round
constexpr int kMaxRounds = 8192;
constexpr uint32_t kOffCnt = kOffBar + 256;
constexpr size_t kSmemBytes = 1024 + kOffCnt + kMaxRounds;

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t kv_full[2], kv_empty[2];
  uint64_t s_full[2], p_full[2], o_full[2], o_free[2];
  uint32_t tmem_base;
  int32_t fail;
};

struct DenseKParams {
  const int32_t* qperm;  // query of each pair slot, or null (slot = query)
  int64_t npos;
  const int32_t* dcnt;
  const int32_t* dblk;
  const uint32_t* dmask;
  int32_t T, Hkv, G, qpt, ppg, q_atoms;
  int64_t npairs, q_start;
  int64_t pair0;              // first pair of this launch (launches cover kMaxRounds rounds)
  const int32_t* porder;      // pair of each (round, CTA) slot, -1: none
  int64_t nslots;             // slots in porder: whole rounds of gridDim.x
  const int32_t* page_table;  // null: contiguous K/V; else the page of each block
  int64_t num_pages;
  uint16_t* part_o;   // chunk-major [16][part_rows][8] bf16
  int64_t part_rows;  // T*Hkv*G
  float* part_lse;    // [T*Hkv*G]
};

__device__ __forceinline__ bool wait_or_fail(uint64_t* bar, uint32_t parity, volatile int32_t* fail) {
  if (*fail) return false;
  if (mbar_wait(bar, parity)) return true;
  msa_record_error(kErrTimeout);
  *fail = 1;
  return false;
}

// The pair of this CTA in round r (-1: none), from the deal written by pair_deal_window.
__device__ __forceinline__ int64_t cta_pair(const DenseKParams& p, int64_t r) {
  const int64_t idx = p.pair0 + r * gridDim.x + blockIdx.x;
  return idx < p.nslots ? p.porder[idx] : -1;
}


__global__ void __launch_bounds__(kThreads, 1)
    prefill_dense_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                            const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const DenseKParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars& B = *reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int32_t* fail = &B.fail;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // pairs p = blockIdx.x + r*gridDim.x with at least one dense block, in (group, query) order
  if (tid == 0) {
    mbar_init(&B.q_full, 1);
    mbar_init(&B.q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&B.kv_full[b], 1);
      mbar_init(&B.kv_empty[b], 1);
      mbar_init(&B.s_full[b], 1);
      mbar_init(&B.p_full[b], 4);
      mbar_init(&B.o_full[b], 1);
      mbar_init(&B.o_free[b], 4);
    }
    B.fail = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&B.tmem_base)), "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  {
    const int nr = (int)min((int64_t)kMaxRounds, (p.nslots - p.pair0) / gridDim.x);
    for (int r = tid; r < nr; r += kThreads) {
      const int64_t pr = cta_pair(p, r);
      const int c = pr < 0 ? 0 : p.dcnt[pr];
      smem[kOffCnt + r] = (uint8_t)(c < 0 ? 0 : (c > kMaxDense ? kMaxDense : c));
    }
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = B.tmem_base;
  const uint32_t sbase = smem_u32(smem);
  const int G = p.G, qpt = p.qpt;
  const int rounds = (int)min((int64_t)kMaxRounds, (p.nslots - p.pair0) / gridDim.x);
  uint8_t* rcnt = smem + kOffCnt;  // blocks of this CTA's pair of round r

  static_assert(128 * kRegsLow + 256 * kRegsHigh == kThreads * kLaunchRegs, "register split");
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == 0) {
      // ============================================================== producer (whole warp)
      // lane q gathers query q of the pair; lane 0 loads the K/V blocks
      if (lane == 0) {
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
      }
      int pairs_done = 0, kv_loads = 0;
      for (int r = 0; r < rounds && !*fail; ++r) {
        const int L = rcnt[r];
        if (L == 0) continue;
        const int64_t pr = cta_pair(p, r);
        const int g = (int)(pr / p.ppg);
        const int64_t t0 = (pr % p.ppg) * 2 * qpt;  // first pair slot
        const int64_t tq = lane < 2 * qpt ? slot_query(p.qperm, p.npos, g, t0 + lane, p.T) : -1;
        const int nvalid = __popc(__ballot_sync(0xffffffffu, tq >= 0));
        // the pair's block ids, one per lane (read before any wait)
        const int32_t blk_l = lane < L ? p.dblk[pr * kMaxDense + lane] : 0;
        const int32_t blk_h = lane + 32 < L ? p.dblk[pr * kMaxDense + lane + 32] : 0;
        if (pairs_done > 0 && !wait_or_fail(&B.q_empty, (pairs_done - 1) & 1, fail)) break;
        if (lane == 0) mbar_expect_tx(&B.q_full, (uint32_t)(nvalid * G * 256));
        __syncwarp();
        if (tq >= 0) {
          const int64_t t = tq;
          uint8_t* qdst = smem + kOffQ + (lane / qpt) * kTileBytes;
          const int q = lane % qpt;
          if (p.q_atoms) {
            tma_load_5d(qdst + q * G * 256, &qmap, &B.q_full, 0, 0, 0, 0, (int32_t)(t * p.Hkv + g));
          } else {
            tma_load_3d(qdst + q * G * 128, &qmap, &B.q_full, 0, g * G, (int32_t)t);
            tma_load_3d(qdst + kBox + q * G * 128, &qmap, &B.q_full, 64, g * G, (int32_t)t);
          }
        }
        for (int j = 0; j < L; ++j) {
          const int c = kv_loads & 1;
          const int32_t blk = __shfl_sync(0xffffffffu, j < 32 ? blk_l : blk_h, j & 31);
          if (lane == 0) {
            // load kv_loads goes to buffer kv_loads & 1, free once both O MMAs of load
            // kv_loads - 2 have completed
            if (kv_loads < 2 || wait_or_fail(&B.kv_empty[c], ((kv_loads - 2) >> 1) & 1, fail)) {
              bool bad = false;
              const int tok = kv_block_row(p.page_table, p.num_pages, blk, bad);
              if (bad) msa_record_error(kErrBadPage);
              uint8_t* kvb = smem + kOffKV + c * 2 * kTileBytes;
              mbar_expect_tx(&B.kv_full[c], 4 * kBox);
              tma_load_3d(kvb, &kmap, &B.kv_full[c], 0, g, tok);
              tma_load_3d(kvb + kBox, &kmap, &B.kv_full[c], 64, g, tok);
              tma_load_3d(kvb + kTileBytes, &vmap, &B.kv_full[c], 0, g, tok);
              tma_load_3d(kvb + kTileBytes + kBox, &vmap, &B.kv_full[c], 64, g, tok);
            }
          }
          if (__shfl_sync(0xffffffffu, (int)*fail, 0)) break;
          ++kv_loads;
        }
        ++pairs_done;
      }
      __syncwarp();
    } else if (warp == 1) {
      // ============================================================== MMA issuer
      // Per warpgroup X (tile A = 0, B = 1) and block n of the CTA's block sequence:
      //   O_X(n) needs P_X(n) and, on a pair's first block, the epilogue of the previous pair
      //   done with O_X; S_X(n+1) needs K/V(n+1), the pair's queries and O_X(n) issued.
      //   S_X(n+1) overwrites the tensor memory from which O_X(n) reads P_X(n): it is issued
      //   after O_X(n) from this one warp, and the tensor pipe runs the MMAs of one thread in
      //   issue order, so O_X(n) has read P_X(n) before S_X(n+1) writes there (the results are
      //   checked against the oracle); the commit that signals S_X(n+1) also covers O_X(n), so
      //   a softmax that sees S_X(n+1) may rescale O_X. K/V buffer n%2 is released after both
      //   O(n), the query tiles after both S of a pair's last block. A ready O goes first.
      // The whole warp runs this loop in lockstep (barrier states agreed by a vote) and one
      // elected lane issues each MMA and commit. The tensor pipe takes one group at a time,
      // holding the warp inside an MMA issue until it has room, so the decision between two
      // issues must be short: pair boundaries come from the per-round block counts in shared
      // memory and every other piece of state lives in registers.
      {
        const uint32_t idesc_s = umma_idesc_bf16(128, 128, 0, 0);
        const uint32_t idesc_o = umma_idesc_bf16(128, 128, 0, 1);
        const uint32_t qhalf = p.q_atoms ? 1024 : kBox;
        const uint32_t qsbo = p.q_atoms ? 2048 : 1024;
        int total = 0;
        for (int r = 0; r < rounds; ++r) total += rcnt[r];
        // per X: blocks issued, blocks left in the current pair, pair ordinal, round cursor
        int sN[2] = {0, 0}, s_left[2] = {0, 0}, s_pi[2] = {-1, -1}, s_r[2] = {-1, -1};
        int oN[2] = {0, 0}, o_left[2] = {0, 0}, o_pi[2] = {-1, -1}, o_r[2] = {-1, -1};
        bool o_first[2] = {true, true};
        auto ready = [&](uint64_t* bar, uint32_t parity) {
          return __all_sync(0xffffffffu, mbar_test(bar, parity));
        };
        auto next_round = [&](int r) {
          do { ++r; } while (r < rounds && rcnt[r] == 0);
          return r;
        };
        uint32_t idle = 0;
        while (oN[0] < total || oN[1] < total) {
          bool progress = false;
#pragma unroll
          for (int X = 0; X < 2; ++X) {
            // ---- O_X(oN[X])
            if (oN[X] < sN[X]) {
              if (o_left[X] == 0) {  // block oN[X] starts the next pair
                o_r[X] = next_round(o_r[X]);
                o_left[X] = o_r[X] < rounds ? rcnt[o_r[X]] : 0;
                ++o_pi[X];
                o_first[X] = true;
              }
              const int n = oN[X];
              if (ready(&B.p_full[X], n & 1) &&
                  (!o_first[X] || o_pi[X] == 0 || ready(&B.o_free[X], (o_pi[X] - 1) & 1))) {
                tmem_fence_after();
                const int c = n & 1;
                const uint64_t bd0 =
                    umma_desc_sw128(sbase + kOffKV + c * 2 * kTileBytes + kTileBytes, kBox, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                  umma_bf16_ts_elect(tmem + 256 + X * 128, tmem + X * 128 + kk * 8,
                                     bd0 + kk * (2048 >> 4), idesc_o,
                                     (!o_first[X] || kk > 0) ? 1u : 0u);
                umma_commit_elect(&B.o_full[X]);
                ++oN[X];
                if (oN[1 - X] >= oN[X]) umma_commit_elect(&B.kv_empty[c]);  // both O(n) issued
                --o_left[X];
                o_first[X] = false;
                progress = true;
              }
            }
            // ---- S_X(sN[X])
            if (sN[X] < total && oN[X] >= sN[X]) {
              if (s_left[X] == 0) {
                s_r[X] = next_round(s_r[X]);
                s_left[X] = s_r[X] < rounds ? rcnt[s_r[X]] : 0;
                ++s_pi[X];
              }
              const int n = sN[X];
              if (ready(&B.kv_full[n & 1], (n >> 1) & 1) && ready(&B.q_full, s_pi[X] & 1)) {
                tmem_fence_after();
                const uint64_t qd0 = umma_desc_sw128(sbase + kOffQ + X * kTileBytes, 16, qsbo);
                const uint64_t kd0 = umma_desc_sw128(sbase + kOffKV + (n & 1) * 2 * kTileBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                  const uint32_t qoff = (kk >> 2) * qhalf + (kk & 3) * 32;
                  const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
                  umma_bf16_elect(tmem + X * 128, qd0 + (qoff >> 4), kd0 + (off >> 4), idesc_s,
                                  kk > 0);
                }
                umma_commit_elect(&B.s_full[X]);
                ++sN[X];
                // the pair's last block: once both tiles' S of it are issued (the two tiles run
                // the same block sequence) the query tiles are free
                if (--s_left[X] == 0 && sN[1 - X] >= sN[X]) umma_commit_elect(&B.q_empty);
                progress = true;
              }
            }
          }
          if (progress) {
            idle = 0;
          } else {
            const int X = oN[0] <= oN[1] ? 0 : 1;
            if (oN[X] < sN[X]) mbar_try_wait_hint(&B.p_full[X], oN[X] & 1, kIssuerNap);
            else __nanosleep(32);
            // every lane leaves together: the flag is agreed by a vote (read now and then: it
            // is only set when another role's wait has timed out)
            const bool failed = __any_sync(0xffffffffu, *fail != 0);
            if (++idle > kWaitLimit || failed) {
              if (!failed && lane == 0) msa_record_error(kErrTimeout);
              *fail = 1;
              break;
            }
          }
        }
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
    // ================================================================ softmax + epilogue
    const int X = (warp - 4) >> 2;                 // tile A (warps 4-7) or B (warps 8-11)
    const int row = (tid - 128) & 127;             // tile row = TMEM lane
    const uint32_t lane_addr = (uint32_t)(32 * (warp & 3)) << 16;
    const int qi = row / G, h = row % G;
    const uint32_t s_tmem = tmem + lane_addr + X * 128;
    const uint32_t o_tmem = tmem + lane_addr + 256 + X * 128;
    const uint32_t qbit = 1u << (X * qpt + qi);
    int n = 0, pairs_done = 0;
    for (int r = 0; r < rounds && !*fail; ++r) {
      const int L = rcnt[r];
      if (L == 0) continue;
      const int64_t pr = cta_pair(p, r);
      const int g = (int)(pr / p.ppg);
      const int64_t t = slot_query(p.qperm, p.npos, g, (pr % p.ppg) * 2 * qpt + X * qpt + qi, p.T);
      const bool valid = t >= 0;
      const int64_t pos = p.q_start + t;
      float m_run = -INFINITY, l = 0.f;             // running max (log2 units) and sum
      uint32_t mask_next = p.dmask[pr * kMaxDense];
      int blk_next = p.dblk[pr * kMaxDense];
      for (int j = 0; j < L; ++j, ++n) {
        const uint32_t mbits = mask_next;
        const int blk = blk_next;
        if (j + 1 < L) {
          mask_next = p.dmask[pr * kMaxDense + j + 1];
          blk_next = p.dblk[pr * kMaxDense + j + 1];
        }
        const bool sel = valid && (mbits & qbit) != 0u;
        if (!wait_or_fail(&B.s_full[X], n & 1, fail)) break;
        tmem_fence_after();
        float v[128];
        float factor = 1.f;
        bool need = false;
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(s_tmem + c * 32, v + c * 32);
        tmem_wait_ld();
        // causal mask on the query's own block; a row whose query did not choose this block
        // gets P = 0 through its exponent (scale 0, offset -inf) instead of a mask
        const int64_t lim64 = pos - (int64_t)blk * 128;  // last visible column
        if (sel && lim64 < 127) {
          const int lim = lim64 < -1 ? -1 : (int)lim64;
#pragma unroll
          for (int x = 0; x < 128; ++x)
            if (x > lim) v[x] = -INFINITY;
        }
        float m4[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
        for (int x = 4; x < 128; x += 2) m4[(x >> 1) & 3] = max3(m4[(x >> 1) & 3], v[x], v[x + 1]);
        const float m2 = sel ? fmaxf(max3(m4[0], m4[1], m4[2]), m4[3]) * kLog2e : -INFINITY;
        if (m_run == -INFINITY) {
          m_run = m2;  // the row's O is still zero
        } else if (m2 > m_run + kRescale) {
          factor = ex2(m_run - m2);
          need = true;
          m_run = m2;
          l *= factor;
        }
        const float sc = sel ? kLog2e : 0.f;
        const float off = sel ? -m_run : -INFINITY;
        float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int x = 0; x < 128; x += 2) {
          fma2(v[x], v[x + 1], v[x], v[x + 1], sc, sc, off, off);
          v[x] = ex2(v[x]);
          v[x + 1] = ex2(v[x + 1]);
          add2(l8[(x >> 1) & 3], l8[4 + ((x >> 1) & 3)], v[x], v[x + 1]);
        }
        l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
        // P row (bf16 pairs) into the first 64 columns of the tile's S buffer
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t pk[32];
#pragma unroll
          for (int x = 0; x < 32; ++x) pk[x] = pack_bf16x2(v[h2 * 64 + 2 * x], v[h2 * 64 + 2 * x + 1]);
          tmem_st32(s_tmem + h2 * 32, pk);
        }
        if (__any_sync(0xffffffffu, need)) {
          // the row max grew by more than 2^8: rescale O once O(n-1) has completed
          if (!wait_or_fail(&B.o_full[X], (n - 1) & 1, fail)) break;
          tmem_fence_after();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float o[32];
            tmem_ld32(o_tmem + c * 32, o);
            tmem_wait_ld();
            uint32_t ob[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) ob[x] = __float_as_uint(o[x] * factor);
            tmem_st32(o_tmem + c * 32, ob);
          }
        }
        tmem_wait_st();
        tmem_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.p_full[X]);
      }
      if (*fail) break;
      // ---------------- epilogue of the pair: normalised bf16 partial + fp32 LSE per row
      if (!wait_or_fail(&B.o_full[X], (n - 1) & 1, fail)) break;
      tmem_fence_after();
      float v[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(o_tmem + c * 32, v + c * 32);
      tmem_wait_ld();
      tmem_fence_before();
      if (valid) {
        const int64_t prow = (t * p.Hkv + g) * G + h;
        __stcs(p.part_lse + prow, l > 0.f ? (m_run + __log2f(l)) * kLn2 : -INFINITY);
        const float inv = l > 0.f ? 1.0f / l : 0.f;
        uint4* dst = reinterpret_cast<uint4*>(p.part_o) + prow;
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
      if (lane == 0) mbar_arrive(&B.o_free[X]);
      ++pairs_done;
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

cudaError_t launch_dense_attention(const CUtensorMap& qmap, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, int32_t q_atoms, int32_t T,
                                   int64_t S_kv, int32_t Hkv, int32_t G,
                                   const int32_t* page_table, int64_t num_pages,
                                   const DenseWorkspace& w, cudaStream_t stream) {
  DenseKParams p;
  p.qperm = (S_kv + 127) / 128 <= kHistBlocks ? w.qperm : nullptr;  // as launch_dense_select
  p.npos = prefill_qpos(T);
  p.dcnt = w.dcnt;
  p.dblk = w.dblk;
  p.dmask = w.dmask;
  p.T = T;
  p.Hkv = Hkv;
  p.G = G;
  p.qpt = 128 / G;
  p.ppg = (int32_t)((T + 2 * p.qpt - 1) / (2 * p.qpt));
  p.q_atoms = q_atoms;
  p.npairs = (int64_t)Hkv * p.ppg;
  p.q_start = S_kv - T;
  p.page_table = page_table;
  p.num_pages = num_pages;
  p.part_o = w.part_o;
  p.part_rows = (int64_t)T * Hkv * G;
  p.part_lse = w.part_lse;
  if (p.npairs <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(prefill_dense_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, prefill_dense_tc_kernel);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  const PairDeal pd = pair_deal_geometry(p.npairs);
  const int64_t grid = pd.grid;
  p.porder = w.porder;
  p.nslots = pd.nslots;
  // one launch per kMaxRounds rounds of pairs (the per-round counts live in shared memory)
  for (int64_t pair0 = 0; pair0 < p.nslots; pair0 += grid * kMaxRounds) {
    p.pair0 = pair0;
    prefill_dense_tc_kernel<<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(qmap, kmap, vmap, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace msa
