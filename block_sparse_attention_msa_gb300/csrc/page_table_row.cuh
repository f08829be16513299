// One flattened row of the sparse page table (row a3), computed by one warp: shared by the
// stand-alone page-table kernel and the decode scorer's tail, so both produce the same table.
//
// Together AI MiniMax-M3 serving article, section "MSA needs a new paged-attention
// integration": the selected blocks of flattened row f = r*Hkv + g become virtual pages of the
// per-head strided view, page p of group g at p*128*Hkv + g; the row's length counts the valid
// tokens of its selected blocks (all 128 of a full block, up to the query in its local block).
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace msa {

// ids: the row's topk block ids (-1 = none); pt_row: the request's page table; q_pos: the row's
// query position. Writes fpt_row[0..topk) and, from lane 0, *len. Returns error bits
// (kErrBadBlock, kErrBadPage) for the caller to record; a bad entry becomes -1.
__device__ __forceinline__ uint32_t warp_flat_page_table_row(
    const int32_t* ids, const int32_t* __restrict__ pt_row, int q_pos, int32_t Hkv, int32_t g,
    int32_t topk, int32_t max_blocks, int64_t num_pages, int32_t* fpt_row, int32_t* len) {
  const int lane = threadIdx.x & 31;
  const int local = q_pos / MSA_BLOCK_TOKENS;
  uint32_t err = 0;
  int n = 0;
  for (int i = lane; i < topk; i += 32) {
    const int32_t j = ids[i];
    int32_t v = -1;
    if (j >= 0) {
      if (j > local || j >= max_blocks) {
        err |= kErrBadBlock;
      } else {
        const int32_t pg = pt_row[j];
        if (pg < 0 || pg >= num_pages) {
          err |= kErrBadPage;
        } else {
          v = (int32_t)((int64_t)pg * MSA_BLOCK_TOKENS * Hkv + g);
          n += (j == local) ? (q_pos % MSA_BLOCK_TOKENS) + 1 : MSA_BLOCK_TOKENS;
        }
      }
    }
    fpt_row[i] = v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  if (lane == 0) *len = n;
  return err;
}

}  // namespace msa
