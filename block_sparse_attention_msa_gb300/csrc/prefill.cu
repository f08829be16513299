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
//  (a) Bucketing inverts block_ids [T, Hkv, k] into per-(group, block) lists of
//      (query, slot) entries: a count pass (shared atomics would not help: the lists are
//      global), one single-CTA scan that also lays out fixed-size work tiles, and a scatter.
//  (b) Work tile = (group g, block j, up to 128/G queries from the list) = 128 query-head
//      rows. A persistent grid of one CTA per SM walks a contiguous range of the global tile
//      list, so consecutive tiles of a CTA share (g, j): the K/V block (64 KB, loaded with
//      two 3-D TMA boxes per tensor straight out of [S_kv, Hkv, D]) stays in shared memory
//      across them, while the gathered query rows of the next tile stream in with cp.async
//      behind the current tile's math. Each of 8 warps owns 16 rows (bf16 MMA, fp32
//      accumulate): S = Q K^T over the 128 keys, causal mask, softmax, O = P V, and writes a
//      bf16 partial O and its fp32 LSE per (query, group, slot) and head.
//  (c) The LSE merge (page_table_merge.cu) reduces the <= k partials of each (query, head).
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"

MSA_DEFINE_ERROR_WORD(pre)

namespace msa {

namespace {

// ------------------------------------------------------------------------------ bucketing
__global__ void bucket_count_kernel(const int32_t* __restrict__ block_ids, int64_t n, int32_t Hkv,
                                    int32_t topk, int32_t nblk, int32_t* __restrict__ counts) {
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int32_t j = block_ids[idx];
    if (j < 0) continue;
    if (j >= nblk) {
      msa_record_error(kErrBadBlock);
      continue;
    }
    const int g = (int)((idx / topk) % Hkv);
    atomicAdd(&counts[(int64_t)g * nblk + j], 1);
  }
}

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

// One CTA: per-group exclusive offsets of the lists, the group bases, the global tile
// offsets (tiles of `qpt` queries per list), and counts reset to zero for the scatter.
__global__ void __launch_bounds__(1024)
    bucket_scan_kernel(int32_t* __restrict__ counts, int32_t Hkv, int32_t nblk, int32_t qpt,
                       int32_t* __restrict__ offsets, int32_t* __restrict__ group_base,
                       int32_t* __restrict__ tile_offsets) {
  __shared__ int warp_sums[33];
  int tile_carry = 0, base = 0;
  for (int g = 0; g < Hkv; ++g) {
    int carry = 0;
    for (int j0 = 0; j0 < nblk; j0 += blockDim.x) {
      const int j = j0 + threadIdx.x;
      const int c = j < nblk ? counts[(int64_t)g * nblk + j] : 0;
      const int nt = (c + qpt - 1) / qpt;
      int tot_c, tot_t;
      const int ex_c = block_exclusive_scan(c, warp_sums, &tot_c);
      const int ex_t = block_exclusive_scan(nt, warp_sums, &tot_t);
      if (j < nblk) {
        offsets[(int64_t)g * (nblk + 1) + j] = carry + ex_c;
        tile_offsets[(int64_t)g * nblk + j] = tile_carry + ex_t;
        counts[(int64_t)g * nblk + j] = 0;
      }
      carry += tot_c;
      tile_carry += tot_t;
    }
    if (threadIdx.x == 0) {
      offsets[(int64_t)g * (nblk + 1) + nblk] = carry;
      group_base[g] = base;
    }
    base += carry;
  }
  if (threadIdx.x == 0) {
    group_base[Hkv] = base;
    tile_offsets[(int64_t)Hkv * nblk] = tile_carry;
  }
}

__global__ void bucket_scatter_kernel(const int32_t* __restrict__ block_ids, int64_t n,
                                      int32_t Hkv, int32_t topk, int32_t nblk,
                                      const int32_t* __restrict__ offsets,
                                      const int32_t* __restrict__ group_base,
                                      int32_t* __restrict__ cursor, int32_t* __restrict__ entries) {
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int32_t j = block_ids[idx];
    if (j < 0 || j >= nblk) continue;
    const int64_t t = idx / ((int64_t)topk * Hkv);
    const int g = (int)((idx / topk) % Hkv);
    const int slot = (int)(idx % topk);
    const int pos = group_base[g] + offsets[(int64_t)g * (nblk + 1) + j] +
                    atomicAdd(&cursor[(int64_t)g * nblk + j], 1);
    entries[pos] = (int32_t)(t * topk + slot);
  }
}

// ------------------------------------------------------------------------------ attention
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 128;                       // query-head rows per tile
constexpr uint32_t kBox = 128 * 64 * 2;          // 128 rows x 64 channels bf16 = 16 KB
constexpr uint32_t kQBytes = 2 * kBox;           // one Q tile (two channel halves)
constexpr uint32_t kKVBytes = 4 * kBox;          // K lo/hi + V lo/hi
constexpr float kLog2e = 1.4426950408889634f;

struct PreKParams {
  const uint16_t* q;
  int32_t T, Hq, Hkv, G, topk, nblk, qpt;
  int64_t S_kv;
  const int32_t* offsets;
  const int32_t* group_base;
  const int32_t* entries;
  const int32_t* tile_offsets;
  uint16_t* part_o;
  float* part_lse;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Cursor over the global tile list: tile `tile` belongs to list gj = g*nblk + j, chunk c.
struct TileCursor {
  int64_t tile;
  int gj;
  int c;
};

__device__ __forceinline__ void cursor_seek(const int32_t* tile_offsets, int n_gj, int64_t tile,
                                            TileCursor& cur) {
  int lo = 0, hi = n_gj - 1;  // largest gj with tile_offsets[gj] <= tile and a nonempty list
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_offsets[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  while (lo + 1 < n_gj && tile_offsets[lo + 1] <= tile) ++lo;  // skip empty lists
  cur.tile = tile;
  cur.gj = lo;
  cur.c = (int)(tile - tile_offsets[lo]);
}

__device__ __forceinline__ void cursor_next(const int32_t* tile_offsets, int n_gj, TileCursor& cur) {
  ++cur.tile;
  ++cur.c;
  while (cur.gj < n_gj && tile_offsets[cur.gj + 1] <= cur.tile) {
    ++cur.gj;
    cur.c = 0;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_partials_kernel(const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const PreKParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* kv = smem;                         // K lo, K hi, V lo, V hi
  uint8_t* qbuf = smem + kKVBytes;            // two Q tiles
  uint64_t* kv_bar = reinterpret_cast<uint64_t*>(qbuf + 2 * kQBytes);
  int32_t* s_ent = reinterpret_cast<int32_t*>(kv_bar + 1);  // [2][128] entry per query slot

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_gj = p.Hkv * p.nblk;
  const int64_t total = p.tile_offsets[n_gj];
  const int64_t per = (total + gridDim.x - 1) / gridDim.x;
  const int64_t t0 = (int64_t)blockIdx.x * per;
  const int64_t t1 = t0 + per < total ? t0 + per : total;
  if (t0 >= t1) return;
  if (tid == 0) {
    mbar_init(kv_bar, 1);
    mbar_fence_init();
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  __syncthreads();

  const int G = p.G, qpt = p.qpt;
  const int64_t q_start = p.S_kv - p.T;
  // gather of one Q tile: thread -> (row = tid/2, channel half = tid%2), 8 x 16 bytes
  auto issue_q = [&](const TileCursor& cur, int buf) {
    const int g = cur.gj / p.nblk;
    const int gbase = p.group_base[g];
    const int32_t* off = p.offsets + (int64_t)g * (p.nblk + 1) + (cur.gj % p.nblk);
    const int lbeg = off[0], lcnt = off[1] - off[0];
    const int r = tid >> 1, half = tid & 1;
    const int qi = r / G, h = r % G;
    const int li = cur.c * qpt + qi;
    int32_t ent = -1;
    if (qi < qpt && li < lcnt) ent = p.entries[gbase + lbeg + li];
    if (h == 0 && half == 0 && qi < qpt) s_ent[buf * 128 + qi] = ent;
    uint8_t* dstb = qbuf + buf * kQBytes + half * kBox;
    if (ent >= 0) {
      const int64_t t = ent / p.topk;
      const uint16_t* src = p.q + ((t * p.Hq + (int64_t)g * G + h) * 128 + half * 64);
#pragma unroll
      for (int c = 0; c < 8; ++c) cp_async16(smem_u32(dstb + sw128(r, c)), src + c * 8);
    } else {
#pragma unroll
      for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(dstb + sw128(r, c)) = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
  };

  TileCursor cur;
  cursor_seek(p.tile_offsets, n_gj, t0, cur);
  int loaded_gj = -1;
  uint32_t kv_phase = 0;
  int buf = 0;
  issue_q(cur, 0);
  const int gid = lane >> 2, tig = lane & 3;

  for (int64_t tile = t0; tile < t1; ++tile) {
    const int g = cur.gj / p.nblk, j = cur.gj % p.nblk;
    // K/V block of this tile (shared by the CTA's consecutive tiles of the same list)
    if (cur.gj != loaded_gj) {
      if (tid == 0) {
        // the previous block was read through the generic proxy; order those reads before
        // the asynchronous-proxy (TMA) writes that replace it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(kv_bar, kKVBytes);
        tma_load_3d(kv, &kmap, kv_bar, 0, g, j * 128);
        tma_load_3d(kv + kBox, &kmap, kv_bar, 64, g, j * 128);
        tma_load_3d(kv + 2 * kBox, &vmap, kv_bar, 0, g, j * 128);
        tma_load_3d(kv + 3 * kBox, &vmap, kv_bar, 64, g, j * 128);
      }
      if (!mbar_wait(kv_bar, kv_phase)) {
        msa_record_error(kErrTimeout);
        cp_async_wait_all();
        return;  // every thread times out on the same phase
      }
      kv_phase ^= 1;
      loaded_gj = cur.gj;
    }
    // prefetch the next tile's queries into the other buffer
    TileCursor nxt = cur;
    cursor_next(p.tile_offsets, n_gj, nxt);
    cp_async_wait_all();
    __syncthreads();  // Q tile `buf` and s_ent[buf] visible to all
    if (tile + 1 < t1) issue_q(nxt, buf ^ 1);

    // ---------------- compute: warp owns rows 16*warp .. +15 of the tile
    const uint32_t qb = smem_u32(qbuf + buf * kQBytes);
    const uint32_t kb = smem_u32(kv), vb = kb + 2 * kBox;
    float sc[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
    {
      const int mi = lane >> 3;
      const uint32_t arow = warp * 16 + (mi & 1) * 8 + (lane & 7);
      const uint32_t brow = (mi >> 1) * 8 + (lane & 7);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t a[4];
        const uint32_t adc = 2 * ks + (mi >> 1);
        ldmatrix_x4(qb + (adc >> 3) * kBox + sw128(arow, adc & 7), a[0], a[1], a[2], a[3]);
        const uint32_t bdc = 2 * ks + (mi & 1);
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(kb + (bdc >> 3) * kBox + sw128(np * 16 + brow, bdc & 7), b0, b1, b2, b3);
          mma_bf16_16816(sc[2 * np], a, b0, b1);
          mma_bf16_16816(sc[2 * np + 1], a, b2, b3);
        }
      }
    }
    // causal mask: row -> query slot -> position
    int64_t qpos[2];
    int32_t ent[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = warp * 16 + gid + 8 * r;
      ent[r] = (row / G < qpt) ? s_ent[buf * 128 + row / G] : -1;
      qpos[r] = ent[r] >= 0 ? q_start + ent[r] / p.topk : -1;
    }
    const int64_t kpos0 = (int64_t)j * 128;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int r = c >> 1;
        const int64_t kp = kpos0 + nt * 8 + tig * 2 + (c & 1);
        if (kp > qpos[r]) sc[nt][c] = -INFINITY;
        mx[r] = fmaxf(mx[r], sc[nt][c]);
      }
    float lsum[2] = {0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    const float mref[2] = {mx[0] == -INFINITY ? 0.f : mx[0], mx[1] == -INFINITY ? 0.f : mx[1]};
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int r = c >> 1;
        sc[nt][c] = ex2((sc[nt][c] - mref[r]) * kLog2e);
        lsum[r] += sc[nt][c];
      }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      lsum[r] += __shfl_xor_sync(0xffffffffu, lsum[r], 1);
      lsum[r] += __shfl_xor_sync(0xffffffffu, lsum[r], 2);
    }
    // O = P V
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    {
      const int mi = lane >> 3;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t pa[4];
        pa[0] = pack_bf16x2(sc[2 * kk][0], sc[2 * kk][1]);
        pa[1] = pack_bf16x2(sc[2 * kk][2], sc[2 * kk][3]);
        pa[2] = pack_bf16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        pa[3] = pack_bf16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
        const uint32_t tok = kk * 16 + (mi & 1) * 8 + (lane & 7);
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
    // epilogue: normalised bf16 partial + fp32 LSE per (entry, head)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (ent[r] < 0) continue;
      const int row = warp * 16 + gid + 8 * r;
      const int h = row % G;
      const int64_t t = ent[r] / p.topk;
      const int slot = ent[r] % p.topk;
      const int64_t pidx = ((t * p.Hkv + g) * p.topk + slot) * G + h;
      const float inv = lsum[r] > 0.f ? 1.0f / lsum[r] : 0.f;
      uint16_t* dst = p.part_o + pidx * 128;
#pragma unroll
      for (int nd = 0; nd < 16; ++nd)
        *reinterpret_cast<uint32_t*>(dst + nd * 8 + tig * 2) =
            pack_bf16x2(o[nd][2 * r] * inv, o[nd][2 * r + 1] * inv);
      if (tig == 0) p.part_lse[pidx] = lsum[r] > 0.f ? mx[r] + __logf(lsum[r]) : -INFINITY;
    }
    __syncthreads();  // everyone done with Q tile `buf` (and K/V) before they are reused
    buf ^= 1;
    cur = nxt;
  }
  cp_async_wait_all();
}

}  // namespace

cudaError_t launch_bucket(const int32_t* block_ids, int32_t T, int32_t Hkv, int32_t topk,
                          int32_t nblk, int32_t qpt, int32_t* offsets, int32_t* entries,
                          int32_t* counts, int32_t* group_base, int32_t* tile_offsets,
                          cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)Hkv * nblk, stream);
  if (e != cudaSuccess) return e;
  const int64_t n = (int64_t)T * Hkv * topk;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, (int64_t)sm_count() * 8));
  bucket_count_kernel<<<grid, 256, 0, stream>>>(block_ids, n, Hkv, topk, nblk, counts);
  bucket_scan_kernel<<<1, 1024, 0, stream>>>(counts, Hkv, nblk, qpt, offsets, group_base,
                                             tile_offsets);
  bucket_scatter_kernel<<<grid, 256, 0, stream>>>(block_ids, n, Hkv, topk, nblk, offsets,
                                                  group_base, counts, entries);
  return cudaGetLastError();
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
  cudaError_t e = launch_bucket(a.block_ids, a.T, a.Hkv, a.topk, a.nblk, qpt, offsets, entries,
                                counts, group_base, tile_offsets, stream);
  if (e != cudaSuccess) return e;

  CUtensorMap kmap, vmap;
  const uint64_t dims[3] = {(uint64_t)a.D, (uint64_t)a.Hkv, (uint64_t)a.S_kv};
  const uint64_t strides[2] = {(uint64_t)a.D * 2, (uint64_t)a.Hkv * a.D * 2};
  const uint32_t box[3] = {64, 1, 128};
  if (!encode_bf16_map(&kmap, a.k, 3, dims, strides, box, true) ||
      !encode_bf16_map(&vmap, a.v, 3, dims, strides, box, true))
    return cudaErrorInvalidValue;
  PreKParams p;
  p.q = a.q;
  p.T = a.T;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = G;
  p.topk = a.topk;
  p.nblk = a.nblk;
  p.qpt = qpt;
  p.S_kv = a.S_kv;
  p.offsets = offsets;
  p.group_base = group_base;
  p.entries = entries;
  p.tile_offsets = tile_offsets;
  p.part_o = part_o;
  p.part_lse = part_lse;
  const size_t smem = 1024 + kKVBytes + 2 * kQBytes + 8 + 2 * 128 * 4;
  e = cudaFuncSetAttribute(prefill_partials_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  prefill_partials_kernel<<<sm_count(), kThreads, smem, stream>>>(kmap, vmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_lse_merge(part_o, true, part_lse, a.block_ids, (int64_t)a.T * a.Hkv, a.topk, G,
                          a.D, a.o, a.lse, stream);
}

}  // namespace msa
