// Sparse page table (decode) and the Log-Sum-Exp merge of partial attention outputs.
//
// Page table -- Together AI MiniMax-M3 serving article, section "MSA needs a new
// paged-attention integration": at decode a page table is built from the selected blocks,
// the KV-group dimension is flattened into the batch, and a strided view of the KV cache
// gives each flattened row its own pages (page address steps by D to select the virtual
// page start, tokens step by Hkv*D). Because the number of selected blocks is bounded the
// mapping kernel is tiny: one warp per flattened row, one lane per slot.
//
// LSE merge -- same article, section "KV-block-major sparse attention reduces redundant KV
// movement": every KV block yields a partial O, and a Log-Sum-Exp reduction rescales and
// sums the partials. The same merge finishes the decode, whose warps each leave one partial
// per row segment in the slot of the segment's first page. One warp per (unit, head): lanes
// own 4 consecutive channels, partials are read once, coalesced, and the result is written as
// bf16 with its fp32 LSE. (The prefill's chunk-major partials have their own merge below.)
#include <algorithm>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"
#include "page_table_row.cuh"

MSA_DEFINE_ERROR_WORD(ptm)

namespace msa {

namespace {

__global__ void __launch_bounds__(256)
    page_table_kernel(const int32_t* __restrict__ block_ids, const int32_t* __restrict__ page_table,
                      const int32_t* __restrict__ seq_lens, int32_t B, int32_t N, int32_t Hkv,
                      int32_t topk, int32_t max_blocks, int64_t num_pages,
                      int32_t* __restrict__ fpt, int32_t* __restrict__ lens) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t f = (int64_t)blockIdx.x * 8 + warp;
  if (f >= (int64_t)B * N * Hkv) return;
  const int64_t r = f / Hkv;
  const int g = (int)(f % Hkv);
  const int64_t b = r / N;
  bool bad = false;
  const int q_pos = clamp_seq(seq_lens, (int)b, N, max_blocks, bad) - N + (int)(r % N);
  if (bad && lane == 0 && g == 0) msa_record_error(kErrBadBlock);
  const uint32_t err = warp_flat_page_table_row(block_ids + f * topk, page_table + b * max_blocks,
                                                q_pos, Hkv, g, topk, max_blocks, num_pages,
                                                fpt + f * topk, lens + f);
  if (err) msa_record_error(err);
}

// One warp per (unit u, head e). Lane s < S loads partial s's LSE (and skip id) and turns it
// into a weight; the partial rows are then streamed with independent 16-byte loads (bf16: a
// half-warp covers one 256-byte row, two partials per step; fp32: one 512-byte row per step).
template <bool BF16>
__global__ void __launch_bounds__(256)
    lse_merge_kernel(const void* __restrict__ o_parts, const float* __restrict__ lse_parts,
                     const int32_t* __restrict__ skip_ids, int64_t U, int32_t S, int32_t G,
                     int32_t D, uint16_t* __restrict__ o, float* __restrict__ lse) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * 8 + warp;  // = u*G + e
  if (item >= U * G) return;
  const int64_t u = item / G;
  const int e = (int)(item % G);
  // lane owns partials `lane` and `lane + 32` (S <= 64); absent or skipped ones weigh 0
  float my_l[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int s = lane + 32 * h;
    my_l[h] = -INFINITY;
    if (s < S && (!skip_ids || skip_ids[u * S + s] >= 0)) my_l[h] = lse_parts[(u * S + s) * G + e];
  }
  const float m = warp_max(fmaxf(my_l[0], my_l[1]));
  float wts[2];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    wts[h] = (m == -INFINITY || my_l[h] == -INFINITY) ? 0.f : __expf(my_l[h] - m);
  const float my_w = wts[0];
  const float total = warp_sum(wts[0] + wts[1]);
  const float inv = total > 0.f ? 1.0f / total : 0.f;
  const int64_t orow = (u * G + e) * (int64_t)D;
  if (BF16 && D == 128 && S <= 32) {
    const int half = lane >> 4, c = lane & 15;  // channels c*8 .. c*8+7
    const uint16_t* base = reinterpret_cast<const uint16_t*>(o_parts);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int s0 = 0; s0 < S; s0 += 2) {
      const int s = s0 + half;
      const float w = __shfl_sync(0xffffffffu, my_w, s < 32 ? s : 0);
      if (s < S && w != 0.f) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4*>(base + ((u * S + s) * G + e) * 128) + c);
        acc[0] = fmaf(w, bf16_lo(v.x), acc[0]);
        acc[1] = fmaf(w, bf16_hi(v.x), acc[1]);
        acc[2] = fmaf(w, bf16_lo(v.y), acc[2]);
        acc[3] = fmaf(w, bf16_hi(v.y), acc[3]);
        acc[4] = fmaf(w, bf16_lo(v.z), acc[4]);
        acc[5] = fmaf(w, bf16_hi(v.z), acc[5]);
        acc[6] = fmaf(w, bf16_lo(v.w), acc[6]);
        acc[7] = fmaf(w, bf16_hi(v.w), acc[7]);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 16);
    if (half == 0) {
      uint4 out;
      out.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      out.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      out.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
      out.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
      *reinterpret_cast<uint4*>(o + orow + c * 8) = out;
    }
  } else {
    // generic path: lanes own 4 consecutive channels; the partials that carry weight stream
    // sixteen at a time with all their loads in flight (a row's partials are independent, so a
    // warp pays one memory round trip per sixteen of them, not one per partial)
    const uint64_t vm = (uint64_t)__ballot_sync(0xffffffffu, wts[0] != 0.f) |
                        ((uint64_t)__ballot_sync(0xffffffffu, wts[1] != 0.f) << 32);
    for (int d0 = 0; d0 < D; d0 += 128) {
      const int d = d0 + lane * 4;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      uint64_t rest = vm;
      while (rest) {
        constexpr int kBatch = 16;
        int sl[kBatch];
        float w8[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          sl[k] = -1;
          if (rest) {
            sl[k] = __ffsll((long long)rest) - 1;
            rest &= rest - 1;
          }
          const float wsel = sl[k] >= 32 ? wts[1] : wts[0];
          w8[k] = __shfl_sync(0xffffffffu, wsel, sl[k] & 31);
          if (sl[k] < 0) w8[k] = 0.f;
        }
        float4 v[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (sl[k] >= 0 && d < D) {
            const int64_t row = ((u * S + sl[k]) * G + e) * (int64_t)D;
            if (BF16) {
              const uint2 b = __ldcs(reinterpret_cast<const uint2*>(
                  reinterpret_cast<const uint16_t*>(o_parts) + row + d));
              v[k] = make_float4(bf16_lo(b.x), bf16_hi(b.x), bf16_lo(b.y), bf16_hi(b.y));
            } else {
              v[k] = __ldcs(reinterpret_cast<const float4*>(
                  reinterpret_cast<const float*>(o_parts) + row + d));
            }
          }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          acc[0] = fmaf(w8[k], v[k].x, acc[0]);
          acc[1] = fmaf(w8[k], v[k].y, acc[1]);
          acc[2] = fmaf(w8[k], v[k].z, acc[2]);
          acc[3] = fmaf(w8[k], v[k].w, acc[3]);
        }
      }
      if (d < D) {
        uint2 out;
        out.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        out.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2*>(o + orow + d) = out;
      }
    }
  }
  if (lse && lane == 0) lse[u * G + e] = total > 0.f ? m + __logf(total) : -INFINITY;
}

// Prefill merge over chunk-major partials: part_o[c][row][8] bf16 with c = 16 channel chunks
// and row = (u*S + s)*G + e; one warp per unit u (all G heads) at a time, persistent over the
// units. Lane slot idx = lane + 32*r covers head idx % G and chunk idx / G, so for a fixed r
// the lanes of one chunk plane read the G adjacent rows of a partial: 16*G contiguous bytes.
// The stream is latency-bound, so the dependent round trips per unit are few: the ids, every
// slot's LSE and the query-major LSE of the warp's next unit are requested while the current
// unit's partials stream (into registers, moved to shared memory at the top of the next unit);
// the valid partials, the query-major one (dense_o / dense_lse, one per unit and head) first,
// stream NB at a time with all their loads in flight, into accumulators kept relative to a
// running max that are rescaled when the max grows.
template <int G>
__device__ __forceinline__ void merge_fma(float (&acc)[(G * 16 + 31) / 32][8], float w,
                                          const uint4 (&v)[(G * 16 + 31) / 32]) {
#pragma unroll
  for (int r = 0; r < (G * 16 + 31) / 32; ++r) {
    acc[r][0] = fmaf(w, bf16_lo(v[r].x), acc[r][0]);
    acc[r][1] = fmaf(w, bf16_hi(v[r].x), acc[r][1]);
    acc[r][2] = fmaf(w, bf16_lo(v[r].y), acc[r][2]);
    acc[r][3] = fmaf(w, bf16_hi(v[r].y), acc[r][3]);
    acc[r][4] = fmaf(w, bf16_lo(v[r].z), acc[r][4]);
    acc[r][5] = fmaf(w, bf16_hi(v[r].z), acc[r][5]);
    acc[r][6] = fmaf(w, bf16_lo(v[r].w), acc[r][6]);
    acc[r][7] = fmaf(w, bf16_hi(v[r].w), acc[r][7]);
  }
}

// The first round trip of unit u: ids (S <= 64), the S*G <= 32*NL slot LSEs (NL per lane),
// the query-major LSE.
template <int NL>
struct MergeHead {
  int id0, id1;
  float ld;
  float lse[NL];
};
template <int G, int NL>
__device__ __forceinline__ void merge_head_load(MergeHead<NL>& m, int64_t u, int64_t U, int S,
                                                const int32_t* __restrict__ ids,
                                                const float* __restrict__ lse_parts,
                                                const float* __restrict__ dense_lse, int lane) {
  const bool in = u < U;
  const int SG = S * G;
  m.id0 = in && lane < S ? __ldg(ids + u * S + lane) : -1;
  m.id1 = in && lane + 32 < S ? __ldg(ids + u * S + lane + 32) : -1;
  m.ld = in && dense_lse ? __ldg(dense_lse + u * G + lane % G) : -INFINITY;
#pragma unroll
  for (int k = 0; k < NL; ++k) {
    const int i = lane + 32 * k;
    m.lse[k] = in && i < SG ? __ldg(lse_parts + u * SG + i) : -INFINITY;
  }
}

template <int G, int NL>
__global__ void __launch_bounds__(256, G >= 16 || NL > 8 ? 1 : 2)
    lse_merge_chunked_kernel(const uint4* __restrict__ part_o, int64_t part_rows,
                             const float* __restrict__ lse_parts, const int32_t* __restrict__ ids,
                             const uint4* __restrict__ dense_o, const float* __restrict__ dense_lse,
                             int64_t U, int32_t S, uint16_t* __restrict__ o, float* __restrict__ lse) {
  constexpr int R = (G * 16 + 31) / 32;  // chunk slots per lane
  constexpr int NB = R >= 8 ? 2 : 3;     // partials per batch of loads
  __shared__ float s_lse[8][NL * 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = lane % G;
  const int SG = S * G;
  float* wl = s_lse[warp];
  const int64_t stride = (int64_t)gridDim.x * 8;
  int64_t u = (int64_t)blockIdx.x * 8 + warp;
  MergeHead<NL> nxt;
  merge_head_load<G, NL>(nxt, u, U, S, ids, lse_parts, dense_lse, lane);
  for (; u < U; u += stride) {
    // this unit's head (requested during the previous unit) into shared memory and a mask
    const MergeHead<NL> cur = nxt;
    __syncwarp();  // the previous unit is done reading its LSEs
#pragma unroll
    for (int k = 0; k < NL; ++k) wl[lane + 32 * k] = cur.lse[k];
    uint64_t vmask = (uint64_t)__ballot_sync(0xffffffffu, cur.id0 >= 0) |
                     ((uint64_t)__ballot_sync(0xffffffffu, cur.id1 >= 0) << 32);
    __syncwarp();
    // the next unit's head, in flight while this unit's partials stream
    merge_head_load<G, NL>(nxt, u + stride, U, S, ids, lse_parts, dense_lse, lane);
    float acc[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int x = 0; x < 8; ++x) acc[r][x] = 0.f;
    float m = -INFINITY, total = 0.f;  // acc and total are relative to e^m
    bool dense_pending = dense_lse != nullptr;
    while (vmask || dense_pending) {
      const uint4* base[NB];
      int64_t rstride[NB];
      float l[NB];
#pragma unroll
      for (int k = 0; k < NB; ++k) {
        base[k] = nullptr;
        rstride[k] = 0;
        l[k] = -INFINITY;
        if (dense_pending) {
          dense_pending = false;
          base[k] = dense_o + u * G + e;
          rstride[k] = U * G;
          l[k] = cur.ld;
        } else if (vmask) {
          const int s = __ffsll((long long)vmask) - 1;
          vmask &= vmask - 1;
          base[k] = part_o + (u * S + s) * G + e;
          rstride[k] = part_rows;
          l[k] = wl[s * G + e];
        }
      }
      uint4 v[NB][R];
#pragma unroll
      for (int k = 0; k < NB; ++k)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int idx = lane + 32 * r;
          v[k][r] = base[k] && idx < G * 16 ? __ldcs(base[k] + (int64_t)(idx / G) * rstride[k])
                                           : make_uint4(0u, 0u, 0u, 0u);
        }
      float mx = l[0];
#pragma unroll
      for (int k = 1; k < NB; ++k) mx = fmaxf(mx, l[k]);
      if (mx == -INFINITY) continue;
      if (mx > m) {
        const float sc = m == -INFINITY ? 0.f : __expf(m - mx);
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int x = 0; x < 8; ++x) acc[r][x] *= sc;
        total *= sc;
        m = mx;
      }
#pragma unroll
      for (int k = 0; k < NB; ++k) {
        // a partial with LSE -inf contributes nothing; its rows may never have been written
        if (l[k] != -INFINITY) {
          const float w = __expf(l[k] - m);
          total += w;
          merge_fma<G>(acc, w, v[k]);
        }
      }
    }
    const float inv = total > 0.f ? 1.0f / total : 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int idx = lane + 32 * r;
      if (idx < G * 16) {
        uint4 out;
        out.x = pack_bf16x2(acc[r][0] * inv, acc[r][1] * inv);
        out.y = pack_bf16x2(acc[r][2] * inv, acc[r][3] * inv);
        out.z = pack_bf16x2(acc[r][4] * inv, acc[r][5] * inv);
        out.w = pack_bf16x2(acc[r][6] * inv, acc[r][7] * inv);
        *reinterpret_cast<uint4*>(o + (u * G + e) * 128 + (idx / G) * 8) = out;
      }
    }
    if (lse && lane < G) lse[u * G + e] = total > 0.f ? m + __logf(total) : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_lse_merge_chunked(const void* part_o, const float* lse_parts,
                                     const int32_t* ids, const void* dense_o,
                                     const float* dense_lse, int64_t U, int32_t S, int32_t G,
                                     uint16_t* o, float* lse, cudaStream_t stream) {
  if (U <= 0) return cudaSuccess;
  if (S > 64 || G > 16 || (int64_t)S * G > 1024) return cudaErrorInvalidValue;
  const int sg = S * G;
  const int nl = sg <= 128 ? 4 : sg <= 256 ? 8 : 32;
  const int per_sm = G >= 16 || nl > 8 ? 1 : 2;
  const unsigned grid = (unsigned)std::min<int64_t>((U + 7) / 8, (int64_t)sm_count() * per_sm);
  const int64_t rows = U * S * G;
  const uint4* po = reinterpret_cast<const uint4*>(part_o);
  const uint4* pd = reinterpret_cast<const uint4*>(dense_o);
#define MSA_MERGE_LAUNCH(GG, NN)                                                               \
  lse_merge_chunked_kernel<GG, NN><<<grid, 256, 0, stream>>>(po, rows, lse_parts, ids, pd, \
                                                              dense_lse, U, S, o, lse)
#define MSA_MERGE_G(GG)                   \
  if (nl == 4) MSA_MERGE_LAUNCH(GG, 4);   \
  else if (nl == 8) MSA_MERGE_LAUNCH(GG, 8); \
  else MSA_MERGE_LAUNCH(GG, 32);
  switch (G) {
    case 1: MSA_MERGE_G(1) break;
    case 2: MSA_MERGE_G(2) break;
    case 4: MSA_MERGE_G(4) break;
    case 8: MSA_MERGE_G(8) break;
    case 16: MSA_MERGE_G(16) break;
    default: return cudaErrorInvalidValue;
  }
#undef MSA_MERGE_G
#undef MSA_MERGE_LAUNCH
  return cudaGetLastError();
}

cudaError_t launch_build_page_table(const int32_t* block_ids, const int32_t* page_table,
                                   const int32_t* seq_lens, int32_t B, int32_t N, int32_t Hkv,
                                   int32_t topk, int32_t max_blocks, int64_t num_pages,
                                   int32_t* fpt, int32_t* lens, cudaStream_t stream) {
  const int64_t rows = (int64_t)B * N * Hkv;
  page_table_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
      block_ids, page_table, seq_lens, B, N, Hkv, topk, max_blocks, num_pages, fpt, lens);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const void* o_parts, bool parts_bf16, const float* lse_parts,
                             const int32_t* skip_ids, int64_t U, int32_t S, int32_t G, int32_t D,
                             uint16_t* o, float* lse, cudaStream_t stream) {
  const int64_t items = U * G;
  const unsigned grid = (unsigned)((items + 7) / 8);
  if (parts_bf16)
    lse_merge_kernel<true>
        <<<grid, 256, 0, stream>>>(o_parts, lse_parts, skip_ids, U, S, G, D, o, lse);
  else
    lse_merge_kernel<false>
        <<<grid, 256, 0, stream>>>(o_parts, lse_parts, skip_ids, U, S, G, D, o, lse);
  return cudaGetLastError();
}

}  // namespace msa
