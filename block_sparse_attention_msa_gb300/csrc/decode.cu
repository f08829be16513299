// Paged sparse decode attention over the strided per-head view of the KV cache.
//
// Together AI MiniMax-M3 serving article, section "MSA needs a new paged-attention
// integration": the KV-group dimension is flattened into the batch and each flattened row
// reads its selected pages through a strided view of one physical KV tensor (page address
// steps by D, tokens by Hkv*D). A virtual page v = p*128*Hkv + g of that view is the 128 token
// rows of group g in physical page p: 256 contiguous bytes of K (and of V) per token, at a
// stride of Hkv*D*2 bytes.
//
// GB300 design. Decode attention is HBM-bound (every K/V byte is used by the G heads of one
// group only), so the kernel is built to keep HBM busy with no synchronisation between warps:
//  * the (row, selected page) units of the whole batch are split into equal contiguous ranges,
//    one per warp of a persistent grid (8 warps per SM);
//  * a warp walks its range in steps of 16 tokens, fetching each step's K and V rows itself
//    with 16-byte cp.async (lanes 0-15 and 16-31 read two 256-byte rows per instruction) into
//    its own 3-stage ring, two steps ahead of the math, so its loads never wait for another
//    warp; 16-byte loads of this strided pattern run at the copy bandwidth;
//  * the G heads of the group form the 16-row side of warp-level bf16 MMAs (QK^T and PV, fp32
//    accumulate) so that tensor cores, not the FMA pipe, absorb the 4 flops per byte; softmax
//    is online across the warp's steps of a row;
//  * where its range leaves a row, the warp writes that row's partial (normalised fp32 O and
//    LSE) into the slot of the first page it covered; the other slots of its range hold LSE
//    -inf, and the LSE-merge kernel combines a row's slots. The result does not depend on warp
//    timing.
#include <cooperative_groups.h>

#include <algorithm>
#include <climits>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"

MSA_DEFINE_ERROR_WORD(dec)

namespace msa {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
constexpr uint32_t kHalf = 16 * 128;   // 16 tokens x 64 channels bf16, 128-byte swizzled
constexpr uint32_t kStep = 4 * kHalf;  // K lo/hi + V lo/hi = 8 KB
constexpr int kWin = 4;                // register windows of 4 x 32 entries
constexpr float kLog2e = 1.4426950408889634f;

struct DecKParams {
  const uint16_t* q;
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  const int32_t* fpt;
  const int32_t* lens;
  int32_t Hkv, G, topk;
  int64_t rows, units, num_pages;  // rows = R*Hkv, units = rows*topk
  float* part_o;                   // [rows, topk, G, 128]
  float* part_lse;                 // [rows, topk, G]
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A warp-uniform, forward-moving view of a 32-bit array through registers: lane l holds
// a[base + 32*j + l]; reading an index past the window reloads it from that index.
struct RegWindow {
  int64_t base;
  int32_t val[kWin];
  __device__ __forceinline__ int32_t get(const int32_t* a, int64_t n, int64_t i, int lane) {
    if (i < base || i >= base + 32 * kWin) {
      base = i;
#pragma unroll
      for (int j = 0; j < kWin; ++j) {
        const int64_t k = i + 32 * j + lane;
        val[j] = k < n ? __ldg(a + k) : 0;
      }
    }
    const int o = (int)(i - base), j = o >> 5;
    int32_t x = val[0];
#pragma unroll
    for (int t = 1; t < kWin; ++t) x = j == t ? val[t] : x;
    return __shfl_sync(0xffffffffu, x, o & 31);
  }
};

// A warp's walk over its unit range [u, u1): unit u = f*topk + pi is page pi of row f; pages
// past the row's visible length are skipped; each page is ceil(tokens/16) steps c.
struct Steps {
  int64_t u, u1, f;
  int len, npg, c, nc;
  bool valid;
  RegWindow lw;
  __device__ __forceinline__ void start(int64_t u0, int64_t uend) {
    u = u0 - 1;
    u1 = uend;
    f = -1;
    len = npg = c = nc = 0;
    lw.base = LLONG_MIN / 2;
  }
  __device__ __forceinline__ void advance(const DecKParams& p, int cap, int lane) {
    if (++c < nc) return;
    for (;;) {
      ++u;
      if (u >= u1) {
        valid = false;
        return;
      }
      const int64_t fu = u / p.topk;
      if (fu != f) {
        f = fu;
        len = min(max(lw.get(p.lens, p.rows, fu, lane), 0), cap);
        npg = (len + 127) >> 7;
      }
      const int pi = (int)(u - f * p.topk);
      if (pi >= npg) {  // the rest of this row has no visible tokens
        u = (f + 1) * p.topk - 1;
        continue;
      }
      c = 0;
      nc = (min(128, len - pi * 128) + 15) >> 4;
      valid = true;
      return;
    }
  }
};

// Copies tokens t0..t0+15 of K and V of virtual page v into a step buffer: channel half c/8 of
// token row r, 16-byte chunk c%8, lands at (c/8)*kHalf + sw128(r, c%8) (K) and 2*kHalf past
// that (V). An invalid page id is recorded and replaced by page 0, group 0.
__device__ __forceinline__ void load_step(uint32_t st, const DecKParams& p, int32_t v, int t0,
                                          int lane) {
  const int64_t vpp = (int64_t)128 * p.Hkv;  // virtual pages per physical page
  int64_t page = v >= 0 ? v / vpp : -1;
  int64_t g = v >= 0 ? v % vpp : -1;
  if (v < 0 || page >= p.num_pages || g >= p.Hkv) {
    if (lane == 0) msa_record_error(kErrBadPage);
    page = 0;
    g = 0;
  }
  const int64_t row0 = (page * 128 + t0) * p.Hkv + g;  // D-element row of token t0, group g
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int idx = lane + 32 * j;
    const int r = idx >> 4, c = idx & 15;
    const int64_t off = (row0 + (int64_t)r * p.Hkv) * 128 + c * 8;
    const uint32_t d = (c >> 3) * kHalf + sw128(r, c & 7);
    cp_async16(st + d, p.k_cache + off);
    cp_async16(st + 2 * kHalf + d, p.v_cache + off);
  }
}

// One warp's walk over the units [u0, u1) through its ring of kStages step buffers (ring: the
// shared-memory address of the warp's buffers). At the end of each row segment it calls
// emit(f, slot_row, o, lrow, mrow, gid, tig) with the segment's unnormalised O fragments (rows
// gid / gid + 8 = heads, columns nd*8 + tig*2 + {0, 1}), the row sums (already reduced over
// the quad) and the row maxima; the walk's copies of that segment have all landed by then.
template <class Emit>
__device__ __forceinline__ void walk_units(const DecKParams& p, uint32_t ring, int64_t u0,
                                           int64_t u1, int lane, Emit&& emit) {
  const int cap = p.topk * 128;
  const int G = p.G;
  Steps cur, pf;
  cur.start(u0, u1);
  pf.start(u0, u1);
  RegWindow vw;
  vw.base = LLONG_MIN / 2;
  // the range's first page ids are requested before the row lengths that the walk needs
  // first, so the two round trips overlap
  if (u0 < u1) (void)vw.get(p.fpt, p.units, u0, lane);
  cur.advance(p, cap, lane);
  pf.advance(p, cap, lane);
  // prefetch the first kStages - 1 steps (one commit group per step; empty groups past the
  // end keep the count uniform)
#pragma unroll
  for (int k = 0; k < kStages - 1; ++k) {
    if (pf.valid) {
      const int32_t v = vw.get(p.fpt, p.units, pf.u, lane);
      load_step(ring + k * kStep, p, v, pf.c * 16, lane);
      pf.advance(p, cap, lane);
    }
    cp_async_commit();
  }

  const int gid = lane >> 2, tig = lane & 3;
  uint32_t it = 0;
  while (cur.valid) {
    // ---- a row segment: row f from unit cur.u on
    const int64_t f = cur.f;
    const int64_t slot_row = cur.u;  // the segment's first page: its partial's slot
    const int len = cur.len;
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

    do {
      // step it + kStages - 1 of the walk goes into the buffer step it - 1 used
      if (pf.valid) {
        const int32_t v = vw.get(p.fpt, p.units, pf.u, lane);
        load_step(ring + ((it + kStages - 1) % kStages) * kStep, p, v, pf.c * 16, lane);
        pf.advance(p, cap, lane);
      }
      cp_async_commit();
      cp_async_wait<kStages - 1>();  // step it has landed
      __syncwarp();
      const uint32_t kb = ring + (it % kStages) * kStep;
      const uint32_t vb = kb + 2 * kHalf;
      // ---- S = Q K^T for the step's 16 tokens (two n-tiles of 8 tokens)
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int mi = lane >> 3;
        const uint32_t tok = (mi >> 1) * 8 + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t dc = 2 * ks + (mi & 1);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(kb + (dc >> 3) * kHalf + sw128(tok, dc & 7), b0, b1, b2, b3);
          mma_bf16_16816(sc[0], qa[ks], b0, b1);
          mma_bf16_16816(sc[1], qa[ks], b2, b3);
        }
      }
      // ---- mask tokens past the row's visible length, online softmax
      const int n0 = (int)(cur.u - f * p.topk) * 128 + cur.c * 16;
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
        const uint32_t tok = (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int nd = 0; nd < 16; nd += 2) {
          const uint32_t dc = nd + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(vb + (dc >> 3) * kHalf + sw128(tok, dc & 7), b0, b1, b2, b3);
          mma_bf16_16816(o[nd], pa, b0, b1);
          mma_bf16_16816(o[nd + 1], pa, b2, b3);
        }
      }
      __syncwarp();  // every lane is done with the buffer before it is refilled
      ++it;
      cur.advance(p, cap, lane);
    } while (cur.valid && cur.f == f);

    // ---- the segment's partial
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
      lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
    }
    emit(f, slot_row, o, lrow, mrow, gid, tig);
  }
  cp_async_wait<0>();
}

// Writes a segment's partial as normalised fp32 rows dst[head][128] and its LSE per head.
__device__ __forceinline__ void store_partial(float* dst, float* lse_dst, const float (&o)[16][4],
                                              const float (&lrow)[2], const float (&mrow)[2],
                                              int G, int gid, int tig) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = gid + 8 * r;
    if (row >= G) continue;
    const float inv = lrow[r] > 0.f ? 1.0f / lrow[r] : 0.f;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd)
      *reinterpret_cast<float2*>(dst + row * 128 + nd * 8 + tig * 2) =
          make_float2(o[nd][2 * r] * inv, o[nd][2 * r + 1] * inv);
    if (tig == 0) lse_dst[row] = lrow[r] > 0.f ? mrow[r] + __logf(lrow[r]) : -INFINITY;
  }
}

__global__ void __launch_bounds__(kThreads, 1) paged_decode_kernel(const DecKParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ring = smem_u32(smem) + warp * kStages * kStep;
  const int G = p.G;
  const int64_t nw = (int64_t)gridDim.x * kWarps, wg = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t u0 = p.units * wg / nw, u1 = p.units * (wg + 1) / nw;

  // every slot of the range starts empty; a row segment's partial overwrites its first slot
  for (int64_t i = u0 * G + lane; i < u1 * G; i += 32) p.part_lse[i] = -INFINITY;
  __syncwarp();
  walk_units(p, ring, u0, u1, lane,
             [&](int64_t, int64_t slot_row, const float (&o)[16][4], const float (&lrow)[2],
                 const float (&mrow)[2], int gid, int tig) {
               store_partial(p.part_o + slot_row * G * 128, p.part_lse + slot_row * G, o, lrow,
                             mrow, G, gid, tig);
             });
}

// Few rows (a small batch at long context): a cluster of kClusterCtas CTAs per flattened row.
// Its 32 warps split the row's selected pages into contiguous ranges and walk them as above;
// each warp then leaves its normalised partial and LSEs in its own (now idle) ring buffer, and
// after a cluster barrier every CTA merges a share of the row's (head, channel) outputs from
// all 32 partials through distributed shared memory. No partial goes to HBM and no merge
// kernel follows.
constexpr int kClusterCtas = 4;

__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kThreads, 1)
    paged_decode_cluster_kernel(const DecKParams p, uint16_t* __restrict__ o_out,
                                float* __restrict__ lse_out) {
  namespace cg = cooperative_groups;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  cg::cluster_group cluster = cg::this_cluster();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster.block_rank();
  const int64_t f = blockIdx.x / kClusterCtas;  // flattened row (request, group)
  const int G = p.G;
  constexpr int kParts = kClusterCtas * kWarps;
  const int wi = rank * kWarps + warp;
  const int64_t u0 = f * p.topk + (int64_t)p.topk * wi / kParts;
  const int64_t u1 = f * p.topk + (int64_t)p.topk * (wi + 1) / kParts;
  // a warp's partial, once its walk is over: O [G][128] fp32, then its G LSEs
  constexpr uint32_t kWarpBytes = kStages * kStep;
  float* part = reinterpret_cast<float*>(smem + warp * kWarpBytes);
  float* part_lse = part + 16 * 128;
  bool emitted = false;
  walk_units(p, smem_u32(smem) + warp * kWarpBytes, u0, u1, lane,
             [&](int64_t, int64_t, const float (&o)[16][4], const float (&lrow)[2],
                 const float (&mrow)[2], int gid, int tig) {
               cp_async_wait<0>();
               __syncwarp();  // the ring's last step is read: it becomes the partial's space
               store_partial(part, part_lse, o, lrow, mrow, G, gid, tig);
               emitted = true;
             });
  if (!emitted) {  // no visible page in the range: O = 0, LSE -inf
    cp_async_wait<0>();
    __syncwarp();
    for (int i = lane; i < G * 128; i += 32) part[i] = 0.f;
    for (int h = lane; h < G; h += 32) part_lse[h] = -INFINITY;
  }
  cluster.sync();  // every warp's partial is in its CTA's shared memory
  // the row's merge weights, one warp per head, lane j = partial j: w[h][j] = e^(lse_j - lse)
  // (0 for an empty range), kept in this CTA (behind warp 0's partial, which stays readable)
  float* wts = reinterpret_cast<float*>(smem + 12 * 1024);
  static_assert(kParts == 32, "one lane per partial");
  for (int h = warp; h < G; h += kWarps) {
    const float* pl = cluster.map_shared_rank(
        reinterpret_cast<float*>(smem + (lane % kWarps) * kWarpBytes) + 16 * 128, lane / kWarps);
    const float l = pl[h];
    const float m = warp_max(l);
    const float e = (m == -INFINITY || l == -INFINITY) ? 0.f : __expf(l - m);
    const float total = warp_sum(e);
    wts[h * 32 + lane] = total > 0.f ? e / total : 0.f;
    if (lane == 0 && lse_out && rank == (h % kClusterCtas))
      lse_out[f * G + h] = total > 0.f ? m + __logf(total) : -INFINITY;
  }
  __syncthreads();
  // (head, channel) outputs of the row, dealt over the cluster's threads: 32 independent
  // remote loads each
  for (int item = rank * kThreads + (int)threadIdx.x; item < G * 128;
       item += kClusterCtas * kThreads) {
    const int h = item >> 7, ch = item & 127;
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kParts; ++j) {
      const float* pj = cluster.map_shared_rank(
          reinterpret_cast<float*>(smem + (j % kWarps) * kWarpBytes), j / kWarps);
      acc = fmaf(wts[h * 32 + j], pj[h * 128 + ch], acc);
    }
    o_out[(f * G + h) * 128 + ch] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
  }
  cluster.sync();  // no CTA leaves while another still reads its shared memory
}

}  // namespace

cudaError_t launch_paged_decode(const DecodeArgs& a, cudaStream_t stream) {
  DecKParams p;
  p.q = a.q;
  p.k_cache = a.k_cache;
  p.v_cache = a.v_cache;
  p.fpt = a.fpt;
  p.lens = a.lens;
  p.Hkv = a.Hkv;
  p.G = a.Hq / a.Hkv;
  p.topk = a.topk;
  p.rows = (int64_t)a.R * a.Hkv;
  p.units = p.rows * a.topk;
  p.num_pages = a.num_pages;
  p.part_o = a.part_o;
  p.part_lse = a.part_lse;
  if (a.nslots != a.topk) return cudaErrorInvalidValue;  // one slot per selected page
  const size_t smem = 1024 + (size_t)kWarps * kStages * kStep;
  cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (p.units <= 0) return cudaSuccess;
  if (p.rows * kClusterCtas <= sm_count()) {
    // few rows: one cluster per row merges in distributed shared memory
    e = cudaFuncSetAttribute(paged_decode_cluster_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    paged_decode_cluster_kernel<<<(unsigned)(p.rows * kClusterCtas), kThreads, smem, stream>>>(
        p, a.o, a.lse);
    return cudaGetLastError();
  }
  const int64_t grid = std::min<int64_t>((p.units + kWarps - 1) / kWarps, sm_count());
  paged_decode_kernel<<<(unsigned)grid, kThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_lse_merge(a.part_o, false, a.part_lse, nullptr, p.rows, a.nslots, p.G, a.D,
                          a.o, a.lse, stream);
}
}  // namespace msa
