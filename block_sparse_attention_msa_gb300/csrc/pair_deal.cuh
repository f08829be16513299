// The deal of the query-major pairs to the query-major kernel's persistent CTAs: its geometry
// (host) and the work of one window (device), run by extra blocks of the list-offsets kernel.
#pragma once

#include <stdint.h>

#include <algorithm>

#include "host_util.h"
#include "kernels.h"

namespace msa {

// The persistent CTAs, and windows of a power-of-two number of rounds (at most 8, at most 1024
// pairs; a divisor of kMaxRounds, so that no window straddles two launches of the kernel).
struct PairDeal {
  int64_t grid;
  int32_t rpw;
  int64_t nwin, nslots;
};
inline PairDeal pair_deal_geometry(int64_t npairs) {
  PairDeal d;
  d.grid = std::min<int64_t>(std::min<int64_t>(npairs, sm_count()), kMaxPairGrid);
  d.rpw = 1;
  while (d.rpw < 8 && 2 * d.rpw * d.grid <= 1024) d.rpw *= 2;
  const int64_t W = d.rpw * d.grid;
  d.nwin = (npairs + W - 1) / W;
  d.nslots = d.nwin * W;
  return d;
}

// Deal of the pairs to the persistent CTAs, by one block of 1024 threads per window `wi` of
// `rounds_per_window` rounds (rounds_per_window * grid consecutive pairs, at most the block size): a CTA's time is close
// to proportional to its blocks, and a plain round-robin deal leaves some CTAs about 8 % more
// blocks than the mean, which the kernel's end waits for. Within the window the pairs are
// ranked by block count (descending; ties by pair index) and rank i goes to round i / grid,
// place i % grid on even rounds and grid - 1 - i % grid on odd ones, so that each CTA's sum is
// near the window's mean; the places map to CTAs turned by 97 per window. Windows keep the
// pairs that run at once near one another in the chunk, which keeps their K/V blocks in L2.
// Slots past the last pair get -1.
__device__ __forceinline__ void pair_deal_window(const int32_t* __restrict__ dcnt, int64_t npairs,
                                                 int32_t grid, int32_t rounds_per_window,
                                                 int32_t* __restrict__ porder, int64_t wi) {
  __shared__ int32_t cnt[32][kMaxDense + 1];  // per warp and block count: pairs, then prefix
  __shared__ int32_t base[kMaxDense + 1];     // per block count: first rank
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int W = rounds_per_window * grid;
  const int64_t w0 = wi * W;
  for (int i = tid; i < 32 * (kMaxDense + 1); i += blockDim.x) (&cnt[0][0])[i] = 0;
  __syncthreads();
  const bool valid = tid < W && w0 + tid < npairs;
  int L = -1;
  if (valid) {
    const int c = dcnt[w0 + tid];
    L = c < 0 ? 0 : (c > kMaxDense ? kMaxDense : c);
  }
  const unsigned peers = __match_any_sync(0xffffffffu, L);
  const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
  if (valid && rank_in_warp == 0) cnt[warp][L] = __popc(peers);
  __syncthreads();
  if (tid <= kMaxDense) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = cnt[w][tid];
      cnt[w][tid] = run;
      run += c;
    }
    base[tid] = run;
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int b = kMaxDense; b >= 0; --b) {
      const int c = base[b];
      base[b] = acc;
      acc += c;
    }
  }
  __syncthreads();
  if (tid < W) {
    const int nvalid = (int)min((int64_t)W, npairs - w0);
    // valid pairs take ranks [0, nvalid), the empty ranks [nvalid, W) get no pair
    const int rank = valid ? base[L] + cnt[warp][L] + rank_in_warp : tid;
    if (valid || tid >= nvalid) {
      const int rl = rank / grid, place = rank % grid;
      // the snake, turned by a stride prime to the grid from one window to the next, so that
      // the heaviest pair of every window (rank 0) does not always land on the same CTA
      const int cta = (int)(((rl & 1 ? grid - 1 - place : place) + wi * 97) % grid);
      porder[w0 + (int64_t)rl * grid + cta] = valid ? (int32_t)(w0 + tid) : -1;
    }
  }
}

}  // namespace msa
