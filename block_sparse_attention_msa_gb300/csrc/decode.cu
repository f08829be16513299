// Paged sparse decode attention over the strided per-head view of the KV cache.
//
// Together AI MiniMax-M3 serving article, section "MSA needs a new paged-attention
// integration": the KV-group dimension is flattened into the batch and each flattened row
// reads its selected pages through a strided view of one physical KV tensor (page address
// steps by D, tokens by Hkv*D). Here that view is a 3-D TMA tensor map over the cache
// [num_pages*128 tokens][Hkv][D]: one box {64 channels, 1 group, 128 tokens} is exactly one
// per-head page half, so each virtual page v = p*128*Hkv + g becomes the TMA coordinate
// (0|64, g, 128*p) and the hardware performs the deinterleaving gather.
//
// GB300 design. Decode attention is HBM-bound (every K/V byte is used by the G heads of one
// group only), so the kernel is built to keep HBM busy:
//  * work items are (flattened row, split of `pages_per_split` pages); a persistent grid of
//    one CTA per SM walks its items while a producer warp streams K and V pages through a
//    3-stage, 64 KB-per-stage TMA ring (128-byte swizzle);
//  * 8 consumer warps each take 16 tokens of every page; the G heads of the group form the
//    16-row side of warp-level bf16 MMAs (QK^T and PV, fp32 accumulate) so that tensor
//    cores, not the FMA pipe, absorb the 4 flops per byte; softmax is online per warp;
//  * the warps' (m, l, O) are merged in shared memory and each item writes one fp32 partial
//    and its LSE; the LSE-merge kernel combines the splits of a row.
#include <algorithm>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"

MSA_DEFINE_ERROR_WORD(dec)

namespace msa {

namespace {

constexpr int kWarps = 8;
constexpr int kConsumers = kWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr uint32_t kBox = 128 * 64 * 2;        // one box: 128 tokens x 64 channels bf16
constexpr uint32_t kStage = 4 * kBox;          // K lo/hi + V lo/hi = 64 KB
constexpr int kMaxStages = 3;
constexpr float kLog2e = 1.4426950408889634f;

struct DecKParams {
  const uint16_t* q;
  const int32_t* fpt;
  const int32_t* lens;
  int32_t Hkv, G, topk, nsplit, pps, nstage;
  int64_t n_items, num_pages;
  float* part_o;
  float* part_lse;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

struct Smem {
  float m[kWarps][16];
  float l[kWarps][16];
  float o[16][128];
  int32_t flag;
};

__global__ void __launch_bounds__(kThreads, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecKParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int nstage = p.nstage;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + nstage * kStage);
  uint64_t* empty_bar = full_bar + kMaxStages;
  Smem& S = *reinterpret_cast<Smem*>(smem + nstage * kStage + 2 * kMaxStages * 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == kConsumers) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kWarps);
    }
    mbar_fence_init();
  }
  if (tid == 0) S.flag = 0;
  __syncthreads();

  const int cap = p.topk * 128;
  if (warp == kWarps) {
    // ===================================== producer
    if (lane != 0) return;
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    const int64_t vpp = (int64_t)128 * p.Hkv;  // virtual pages per physical page
    uint32_t it = 0;
    for (int64_t item = blockIdx.x; item < p.n_items; item += gridDim.x) {
      const int64_t f = item / p.nsplit;
      const int s = (int)(item % p.nsplit);
      const int len = min(max(p.lens[f], 0), cap);
      const int npages = (len + 127) / 128;
      const int pbeg = s * p.pps, pend = min(npages, pbeg + p.pps);
      for (int pi = pbeg; pi < pend; ++pi, ++it) {
        const int64_t v = p.fpt[f * p.topk + pi];
        int64_t page = v >= 0 ? v / vpp : -1;
        int32_t g = v >= 0 ? (int32_t)(v % vpp) : -1;
        if (v < 0 || page >= p.num_pages || g >= p.Hkv) {
          msa_record_error(kErrBadPage);
          page = 0;
          g = 0;
        }
        const uint32_t slot = it % nstage;
        if (it >= (uint32_t)nstage && !mbar_wait(&empty_bar[slot], ((it / nstage) - 1) & 1)) {
          msa_record_error(kErrTimeout);
          // let the copies already issued land before the CTA exits (bounded)
          for (uint32_t k = it - nstage + 1; k < it; ++k) mbar_wait(&full_bar[k % nstage], (k / nstage) & 1);
          return;
        }
        uint8_t* st = smem + slot * kStage;
        mbar_expect_tx(&full_bar[slot], kStage);
        const int32_t tok = (int32_t)(page * 128);
        tma_load_3d(st, &kmap, &full_bar[slot], 0, g, tok);
        tma_load_3d(st + kBox, &kmap, &full_bar[slot], 64, g, tok);
        tma_load_3d(st + 2 * kBox, &vmap, &full_bar[slot], 0, g, tok);
        tma_load_3d(st + 3 * kBox, &vmap, &full_bar[slot], 64, g, tok);
      }
    }
    for (uint32_t k = (it > (uint32_t)nstage ? it - nstage : 0); k < it; ++k)
      if (!mbar_wait(&empty_bar[k % nstage], (k / nstage) & 1)) msa_record_error(kErrTimeout);
    return;
  }

  // ======================================= consumers
  const int gid = lane >> 2, tig = lane & 3;
  const int G = p.G;
  const int tb = warp * 16;  // this warp's tokens inside every page
  uint32_t it = 0;
  for (int64_t item = blockIdx.x; item < p.n_items; item += gridDim.x) {
    const int64_t f = item / p.nsplit;
    const int s = (int)(item % p.nsplit);
    const int len = min(max(p.lens[f], 0), cap);
    const int npages = (len + 127) / 128;
    const int pbeg = s * p.pps, pend = min(npages, pbeg + p.pps);
    const int64_t pidx = f * p.nsplit + s;
    if (pend <= pbeg) {
      if (tid < G) p.part_lse[pidx * G + tid] = -INFINITY;
      continue;
    }
    // Q fragments (A operand, 16 rows = heads of the group, zero rows beyond G)
    uint32_t qa[8][4];
    const uint16_t* qrow0 = p.q + (f * G + gid) * 128;
    const uint16_t* qrow1 = p.q + (f * G + gid + 8) * 128;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int d = ks * 16 + tig * 2;
      qa[ks][0] = gid < G ? *reinterpret_cast<const uint32_t*>(qrow0 + d) : 0u;
      qa[ks][1] = gid + 8 < G ? *reinterpret_cast<const uint32_t*>(qrow1 + d) : 0u;
      qa[ks][2] = gid < G ? *reinterpret_cast<const uint32_t*>(qrow0 + d + 8) : 0u;
      qa[ks][3] = gid + 8 < G ? *reinterpret_cast<const uint32_t*>(qrow1 + d + 8) : 0u;
    }
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    for (int e = tid; e < 16 * 128; e += kConsumers) (&S.o[0][0])[e] = 0.f;

    for (int pi = pbeg; pi < pend; ++pi, ++it) {
      const uint32_t slot = it % nstage;
      const bool ok = mbar_wait(&full_bar[slot], (it / nstage) & 1);
      if (!ok) {
        msa_record_error(kErrTimeout);
        S.flag = 1;
      }
      if (ok) {
        const uint32_t kb = smem_u32(smem + slot * kStage);
        const uint32_t vb = kb + 2 * kBox;
        // ---- S = Q K^T for tokens tb..tb+15 (two n-tiles of 8 tokens)
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          const int mi = lane >> 3;
          const uint32_t tok = tb + (mi >> 1) * 8 + (lane & 7);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t dc = 2 * ks + (mi & 1);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(kb + (dc >> 3) * kBox + sw128(tok, dc & 7), b0, b1, b2, b3);
            mma_bf16_16816(sc[0], qa[ks], b0, b1);
            mma_bf16_16816(sc[1], qa[ks], b2, b3);
          }
        }
        // ---- mask tokens past the row's visible length, online softmax
        const int n0 = pi * 128 + tb;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (n0 + nt * 8 + tig * 2 + (c & 1) >= len) sc[nt][c] = -INFINITY;
        float mx[2];
        mx[0] = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        mx[1] = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
          mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        }
        float scale[2], mref[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float mnew = fmaxf(mrow[r], mx[r]);
          mref[r] = mnew == -INFINITY ? 0.f : mnew;
          scale[r] = ex2((mrow[r] - mref[r]) * kLog2e);
          mrow[r] = mnew;
        }
        float ps[2] = {0.f, 0.f};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int r = c >> 1;
            sc[nt][c] = ex2((sc[nt][c] - mref[r]) * kLog2e);
            ps[r] += sc[nt][c];
          }
#pragma unroll
        for (int r = 0; r < 2; ++r) lrow[r] = lrow[r] * scale[r] + ps[r];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          o[i][0] *= scale[0];
          o[i][1] *= scale[0];
          o[i][2] *= scale[1];
          o[i][3] *= scale[1];
        }
        // ---- O += P V (P from the S accumulators, V via transposed ldmatrix)
        uint32_t pa[4];
        pa[0] = pack_bf16x2(sc[0][0], sc[0][1]);
        pa[1] = pack_bf16x2(sc[0][2], sc[0][3]);
        pa[2] = pack_bf16x2(sc[1][0], sc[1][1]);
        pa[3] = pack_bf16x2(sc[1][2], sc[1][3]);
        {
          const int mi = lane >> 3;
          const uint32_t tok = tb + (mi & 1) * 8 + (lane & 7);
#pragma unroll
          for (int nd = 0; nd < 16; nd += 2) {
            const uint32_t dc = nd + (mi >> 1);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(vb + (dc >> 3) * kBox + sw128(tok, dc & 7), b0, b1, b2, b3);
            mma_bf16_16816(o[nd], pa, b0, b1);
            mma_bf16_16816(o[nd + 1], pa, b2, b3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[slot]);
    }
    // ---- merge the 8 warps' partial softmax states
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
      lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
    }
    if (tig == 0) {
      S.m[warp][gid] = mrow[0];
      S.m[warp][gid + 8] = mrow[1];
      S.l[warp][gid] = lrow[0];
      S.l[warp][gid + 8] = lrow[1];
    }
    consumer_sync();
    if (S.flag) return;
    float wgt[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = gid + 8 * r;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, S.m[w][row]);
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w)
        if (S.m[w][row] != -INFINITY) L += S.l[w][row] * ex2((S.m[w][row] - M) * kLog2e);
      wgt[r] = (mrow[r] == -INFINITY || L <= 0.f) ? 0.f : ex2((mrow[r] - M) * kLog2e) / L;
      if (warp == 0 && tig == 0 && row < G)
        p.part_lse[pidx * G + row] = L > 0.f ? M + __logf(L) : -INFINITY;
    }
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      const int col = nd * 8 + tig * 2;
      if (gid < G) {
        atomicAdd(&S.o[gid][col], o[nd][0] * wgt[0]);
        atomicAdd(&S.o[gid][col + 1], o[nd][1] * wgt[0]);
      }
      if (gid + 8 < G) {
        atomicAdd(&S.o[gid + 8][col], o[nd][2] * wgt[1]);
        atomicAdd(&S.o[gid + 8][col + 1], o[nd][3] * wgt[1]);
      }
    }
    consumer_sync();
    float* dst = p.part_o + pidx * G * 128;
    for (int e = tid * 4; e < G * 128; e += kConsumers * 4)
      *reinterpret_cast<float4*>(dst + e) = *reinterpret_cast<const float4*>(&S.o[0][0] + e);
    consumer_sync();
  }
}

}  // namespace

void decode_split(int32_t topk, int32_t* nsplit, int32_t* pages_per_split) {
  const int pps = 4;
  *pages_per_split = pps;
  *nsplit = (topk + pps - 1) / pps;
}

cudaError_t launch_paged_decode(const DecodeArgs& a, cudaStream_t stream) {
  CUtensorMap kmap, vmap;
  const uint64_t dims[3] = {(uint64_t)a.D, (uint64_t)a.Hkv, (uint64_t)a.num_pages * 128};
  const uint64_t strides[2] = {(uint64_t)a.D * 2, (uint64_t)a.Hkv * a.D * 2};
  const uint32_t box[3] = {64, 1, 128};
  if (!encode_bf16_map(&kmap, a.k_cache, 3, dims, strides, box, true) ||
      !encode_bf16_map(&vmap, a.v_cache, 3, dims, strides, box, true))
    return cudaErrorInvalidValue;
  DecKParams p;
  p.q = a.q;
  p.fpt = a.fpt;
  p.lens = a.lens;
  p.Hkv = a.Hkv;
  p.G = a.Hq / a.Hkv;
  p.topk = a.topk;
  p.nsplit = a.nsplit;
  p.pps = a.pages_per_split;
  p.nstage = kMaxStages;
  p.n_items = (int64_t)a.R * a.Hkv * a.nsplit;
  p.num_pages = a.num_pages;
  p.part_o = a.part_o;
  p.part_lse = a.part_lse;
  const size_t smem = 1024 + kMaxStages * kStage + 2 * kMaxStages * 8 + sizeof(Smem);
  cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(p.n_items, sm_count());
  paged_decode_kernel<<<(unsigned)grid, kThreads, smem, stream>>>(kmap, vmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_lse_merge(a.part_o, false, a.part_lse, nullptr, (int64_t)a.R * a.Hkv, a.nsplit,
                          p.G, a.D, a.o, a.lse, stream);
}

}  // namespace msa
