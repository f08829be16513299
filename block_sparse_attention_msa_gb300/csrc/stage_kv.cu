// KV residency split: the paged K/V cache stays in host memory, and only the blocks a decode
// step selected are copied to a device staging cache before the paged decode.
//
// Together AI MiniMax-M3 serving article, section "The index scorer becomes the decode critical
// path" (the index scorer reads a small key index for every block; only the selected blocks'
// K/V are needed by the attention), and section "MSA needs a new paged-attention integration"
// (the selection becomes a page table over the strided per-head view).
//
// GB300 design. Host memory is read directly by the kernel (pinned memory is mapped into the
// device address space and reached over NVLink-C2C on a Grace host): one CTA per selected
// (flattened row f = r*Hkv + g, slot i) copies the 128 token rows of group g of that block,
// K and V, into staging page r*topk + i, group slot g. The staging cache has the layout of the
// paged cache ([R*topk, 128, Hkv, D]) and every (r, i) page is filled by its Hkv rows, so the
// paged decode runs on it unchanged with the staging page table written here.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

MSA_DEFINE_ERROR_WORD(stage)

namespace msa {

namespace {

constexpr int kStageThreads = 256;
constexpr int kChunksPerRow = 128 * 2 / 16;          // D = 128 bf16 = 256 bytes = 16 x 16 B
constexpr int kRowChunks = 128 * kChunksPerRow;     // 128 rows of one block: 2048 x 16 B

__global__ void __launch_bounds__(kStageThreads)
    stage_kv_kernel(const uint4* __restrict__ k_src, const uint4* __restrict__ v_src,
                    int64_t num_pages, const int32_t* __restrict__ fpt, int32_t Hkv,
                    int32_t topk, uint4* __restrict__ k_dst, uint4* __restrict__ v_dst,
                    int32_t* __restrict__ stage_fpt) {
  const int64_t sel = blockIdx.x;  // (f, i)
  const int64_t f = sel / topk;
  const int i = (int)(sel % topk);
  const int64_t r = f / Hkv;
  const int g = (int)(f % Hkv);
  const int32_t v = fpt[sel];
  const int64_t s = r * topk + i;  // staging page
  // a virtual page of the strided view is p*128*Hkv + g with p < num_pages
  const int64_t page_span = (int64_t)128 * Hkv;
  const bool bad = v >= 0 && ((int64_t)v / page_span >= num_pages || (int64_t)v % page_span != g);
  if (threadIdx.x == 0) {
    if (bad) msa_record_error(kErrBadPage);
    stage_fpt[sel] = (v < 0 || bad) ? -1 : (int32_t)(s * 128 * Hkv + g);
  }
  if (v < 0 || bad) return;
  // source row tau of the strided view: element (v, tau, d) at v*D + tau*Hkv*D + d; the
  // destination is staging element [s, tau, g, d]. Chunks are 16 bytes (8 channels).
  const int64_t src0 = (int64_t)v * kChunksPerRow;
  const int64_t dst0 = (s * 128 * Hkv + g) * kChunksPerRow;
  constexpr int kPer = kRowChunks / kStageThreads;  // 8 chunks of K and 8 of V per thread
  uint4 kk[kPer], vv[kPer];
#pragma unroll
  for (int c = 0; c < kPer; ++c) {
    const int e = threadIdx.x + c * kStageThreads;
    const int tau = e / kChunksPerRow, ch = e % kChunksPerRow;
    const int64_t off = src0 + (int64_t)tau * Hkv * kChunksPerRow + ch;
    kk[c] = __ldcs(k_src + off);
    vv[c] = __ldcs(v_src + off);
  }
#pragma unroll
  for (int c = 0; c < kPer; ++c) {
    const int e = threadIdx.x + c * kStageThreads;
    const int tau = e / kChunksPerRow, ch = e % kChunksPerRow;
    const int64_t off = dst0 + (int64_t)tau * Hkv * kChunksPerRow + ch;
    k_dst[off] = kk[c];
    v_dst[off] = vv[c];
  }
}

}  // namespace

cudaError_t launch_stage_kv(const uint16_t* k_src, const uint16_t* v_src, int64_t num_pages,
                            const int32_t* fpt, int32_t R, int32_t Hkv, int32_t topk,
                            uint16_t* k_dst, uint16_t* v_dst, int32_t* stage_fpt,
                            cudaStream_t stream) {
  const int64_t n = (int64_t)R * Hkv * topk;
  if (n <= 0) return cudaSuccess;
  stage_kv_kernel<<<(unsigned)n, kStageThreads, 0, stream>>>(
      reinterpret_cast<const uint4*>(k_src), reinterpret_cast<const uint4*>(v_src), num_pages, fpt,
      Hkv, topk, reinterpret_cast<uint4*>(k_dst), reinterpret_cast<uint4*>(v_dst), stage_fpt);
  return cudaGetLastError();
}

}  // namespace msa
