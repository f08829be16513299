// Internal launcher interface between the C ABI (msa_api.cu) and the kernel translation
// units. Every launcher only queues work on `stream` and returns the launch status.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace msa {

// ------------------------------------------------------------------ stage 1
struct ScoreArgs {
  const uint16_t* q_idx;       // [B*N, Hkv, Di]
  const uint16_t* k_idx;       // [num_pages, 128, Hkv, Di]
  const int32_t* page_table;   // [B, max_blocks]
  const int32_t* seq_lens;     // [B]
  int32_t B, N, Hkv, Di, max_blocks, topk;
  int64_t num_pages;
  int32_t* block_ids;          // [B*N, Hkv, topk]
  float* sel_scores;           // [B*N, Hkv, topk] or null
  float* scores;               // workspace [B*N, Hkv, max_blocks]
  int32_t* tickets;            // workspace [B], cleared by the launcher before each call
  int32_t* fpt = nullptr;      // optional: sparse page table [B*N*Hkv, topk] (decode scorer's
  int32_t* fpt_lens = nullptr; //   tail builds it with the selection) and lengths [B*N*Hkv]
};
// Streaming scorer for N <= kDecodeMaxN with the top-k fused into the last CTA per request.
constexpr int kDecodeMaxN = 8;
cudaError_t launch_score_decode(const ScoreArgs& a, cudaStream_t stream);
// Multi-token decode scorer (2 <= N <= kDecodeTcMaxN) on the tensor cores, writing every
// visible block score (the top-k kernel follows).
constexpr int kDecodeTcMaxN = 16;
cudaError_t launch_score_tc_decode(const ScoreArgs& a, cudaStream_t stream);
int score_tc_decode_stages(int Hkv, int Di);
// Generic scorer (any N) writing every block score, followed by the top-k kernel.
cudaError_t launch_score_rows(const ScoreArgs& a, cudaStream_t stream);
cudaError_t launch_topk_rows(const ScoreArgs& a, cudaStream_t stream);
size_t score_decode_smem_bytes(int N, int Hkv, int Di, int* nstage);

// ------------------------------------------------------------------ page table
cudaError_t launch_build_page_table(const int32_t* block_ids, const int32_t* page_table,
                                   const int32_t* seq_lens, int32_t B, int32_t N, int32_t Hkv,
                                   int32_t topk, int32_t max_blocks, int64_t num_pages,
                                   int32_t* fpt, int32_t* lens, cudaStream_t stream);

// ------------------------------------------------------------------ paged decode
struct DecodeArgs {
  const uint16_t* q;           // [R, Hq, D]
  const uint16_t* k_cache;     // [num_pages, 128, Hkv, D]
  const uint16_t* v_cache;
  const int32_t* fpt;          // [R*Hkv, topk]
  const int32_t* lens;         // [R*Hkv]
  int32_t R, Hq, Hkv, D, topk;
  int64_t num_pages;
  uint16_t* o;                 // [R, Hq, D]
  float* lse;                  // [R, Hq] or null
  float* part_o;               // workspace [R*Hkv, nslots, G, D]
  float* part_lse;             // workspace [R*Hkv, nslots, G]
  int32_t nslots;              // partial slots per flattened row: decode_slots(topk)
};
// One partial slot per selected page: a warp whose unit range starts a row segment at page i
// writes slot i.
inline int32_t decode_slots(int32_t topk) { return topk; }
cudaError_t launch_paged_decode(const DecodeArgs& a, cudaStream_t stream);

// ------------------------------------------------------------------ KV residency split
// Copies the K/V rows of every selected (row f, slot i) from the (host-resident) paged caches
// into staging page (f/Hkv)*topk + i, group f%Hkv, of k_dst/v_dst [R*topk, 128, Hkv, D], and
// writes the staging flat page table [R*Hkv, topk] (-1 where fpt is -1).
cudaError_t launch_stage_kv(const uint16_t* k_src, const uint16_t* v_src, int64_t num_pages,
                            const int32_t* fpt, int32_t R, int32_t Hkv, int32_t topk,
                            uint16_t* k_dst, uint16_t* v_dst, int32_t* stage_fpt,
                            cudaStream_t stream);

// ------------------------------------------------------------------ LSE merge
// skip_ids: optional [U, S]; partial s of unit u is ignored when skip_ids[u*S+s] < 0.
cudaError_t launch_lse_merge(const void* o_parts, bool parts_bf16, const float* lse_parts,
                             const int32_t* skip_ids, int64_t U, int32_t S, int32_t G, int32_t D,
                             uint16_t* o, float* lse, cudaStream_t stream);

// Prefill merge of chunk-major partials part_o[16][U*S*G][8] bf16 (row = (u*S+s)*G+e); a
// partial s of unit u is skipped when ids[u*S+s] < 0 (never written). Optionally one more
// partial per (unit, head): dense_o chunk-major [16][U*G][8], dense_lse [U*G] (-inf = none).
// G in {1,2,4,8,16}.
cudaError_t launch_lse_merge_chunked(const void* part_o, const float* lse_parts,
                                     const int32_t* ids, const void* dense_o,
                                     const float* dense_lse, int64_t U, int32_t S, int32_t G,
                                     uint16_t* o, float* lse, cudaStream_t stream);

// ------------------------------------------------------------------ prefill
// Workspace carve-up shared by the C ABI (size query) and the launcher. Offsets in bytes,
// each 256-byte aligned.
// Query-major part (G in {8, 16}): pairs of 128/G-query tiles, at most kMaxDense shared blocks each.
constexpr int kMaxDense = 64;
// Most persistent CTAs of the query-major kernel (the pair deal pads the pairs to whole rounds).
constexpr int kMaxPairGrid = 1024;
inline bool prefill_hybrid(int32_t G) { return G == 8 || G == 16; }
inline int64_t prefill_pairs(int64_t T, int32_t Hkv, int32_t G) {
  const int64_t q2 = 2 * (128 / G);
  return (int64_t)Hkv * ((T + q2 - 1) / q2);
}
// Pair slots per group: the chunk's queries in 128-query spans (a pair never crosses a span).
inline int64_t prefill_qpos(int64_t T) { return (T + 127) / 128 * 128; }
struct PrefillWorkspace {
  size_t counts, group_base, tile_offsets, offsets, entries, epos, part_o, part_lse, tile_desc;
  size_t residual, dcnt, dblk, dmask, dense_o, dense_lse, qperm, porder, total;  // query-major (G 8, 16)
};
inline size_t ws_align(size_t x) { return (x + 255) & ~size_t(255); }
// Prefill work lists are per (group, query window, KV block): queries are cut into windows so
// that the tiles of one window -- whose query rows stay in L2 -- run together. The window is the
// smallest power of two from 2048 at which a list holds about `target` selections on average
// (window * topk >= target * nblk), or the whole chunk: with many blocks (a long prefix)
// short windows would leave tiles half empty and reload a K/V block for every few queries.
// The target counts all selections: 64 when every selection is block-major, 512 when the
// query-major pass (G 8, 16) first takes the shared blocks (about two thirds of them in the
// clustered workloads), so that the residual lists still fill their tiles.
constexpr int32_t kListTarget = 64;
constexpr int32_t kListTargetHybrid = 512;
inline int32_t prefill_window(int64_t T, int32_t nblk, int32_t topk, int32_t G) {
  const int64_t target = prefill_hybrid(G) ? kListTargetHybrid : kListTarget;
  int64_t w = 2048;
  while (w < T && w * topk < target * nblk) w *= 2;
  return (int32_t)w;
}
inline int32_t prefill_nwin(int64_t T, int32_t nblk, int32_t topk, int32_t G) {
  const int64_t w = prefill_window(T, nblk, topk, G);
  return (int32_t)((T + w - 1) / w);
}
inline PrefillWorkspace prefill_ws_layout(int64_t T, int32_t Hkv, int32_t topk, int32_t nblk,
                                          int32_t G, bool attention) {
  PrefillWorkspace w{};
  const size_t lists = (size_t)Hkv * (attention ? prefill_nwin(T, nblk, topk, G) : 1) * nblk;
  const size_t groups = lists / nblk;
  size_t off = 0;
  w.counts = off;       off = ws_align(off + 4 * lists);
  w.group_base = off;   off = ws_align(off + 4 * (groups + 1));
  w.tile_offsets = off; off = ws_align(off + 4 * (groups * (nblk + 1) + groups + 1));
  const size_t sel = (size_t)T * Hkv * topk;
  w.epos = off;         off = ws_align(off + 4 * sel);
  if (attention) {
    w.offsets = off;    off = ws_align(off + 4 * groups * (nblk + 1));
    w.entries = off;    off = ws_align(off + 4 * sel);
    w.part_o = off;     off = ws_align(off + 2 * sel * G * 128);
    w.part_lse = off;   off = ws_align(off + 4 * sel * G);
    // one 16-byte descriptor per work tile of 128/G queries: at most sel/(128/G) + lists
    w.tile_desc = off;  off = ws_align(off + 16 * (sel * G / 128 + lists + 1));
    if (prefill_hybrid(G)) {
      const size_t pairs = (size_t)prefill_pairs(T, Hkv, G);
      const size_t rows = (size_t)T * Hkv * G;
      w.residual = off;   off = ws_align(off + 4 * sel);
      w.dcnt = off;       off = ws_align(off + 4 * pairs);
      w.dblk = off;       off = ws_align(off + 4 * pairs * kMaxDense);
      w.dmask = off;      off = ws_align(off + 4 * pairs * kMaxDense);
      w.dense_o = off;    off = ws_align(off + 2 * rows * 128);
      w.dense_lse = off;  off = ws_align(off + 4 * rows);
      w.qperm = off;      off = ws_align(off + 4 * (size_t)Hkv * prefill_qpos(T));
      w.porder = off;     off = ws_align(off + 4 * (pairs + kMaxPairGrid));
    }
  }
  w.total = off;
  return w;
}
// Query-major part of the prefill (G in {8, 16}): per pair of 128/G-query tiles, the blocks
// chosen by at least half of the pair's queries (ascending, at most kMaxDense) with a bit mask of
// the queries that chose each; the residual selections go to the block-major pass.
struct DenseWorkspace {
  int32_t* qperm;      // [Hkv, prefill_qpos(T)]: query of each pair slot (-1: none)
  int32_t* porder;     // [pairs + kMaxPairGrid]: pair of each (round, CTA) of the query-major
                       // kernel (-1: none), written by its launcher
  int32_t* residual;   // [T, Hkv, k]
  int32_t* dcnt;       // [pairs]
  int32_t* dblk;       // [pairs, kMaxDense]
  uint32_t* dmask;     // [pairs, kMaxDense]
  uint16_t* part_o;    // chunk-major [16][T*Hkv*G][8] bf16
  float* part_lse;     // [T*Hkv*G]
};
// Row of the K/V tensor map that holds token 0 of block j: j*128 for contiguous K/V, else the
// block's page * 128 (an out-of-range page is reported through `bad` and read as page 0).
__device__ __forceinline__ int32_t kv_block_row(const int32_t* page_table, int64_t num_pages,
                                                int32_t j, bool& bad) {
  if (!page_table) return j * 128;
  const int32_t pg = page_table[j];
  bad = pg < 0 || pg >= num_pages;
  return (bad ? 0 : pg) * 128;
}
// (a) of the prefill in one kernel per (group, 128-query span): the query order and the shared
// blocks of each pair (G 8 / 16, when w.residual is set), then the count of every remaining
// selection into its (group, query window, block) list, with its place in the list in `epos`.
// `counts` [Hkv * nwin, nblk] must be zero on entry.
cudaError_t launch_select_count(const int32_t* block_ids, int32_t T, int64_t S_kv, int32_t Hkv,
                                int32_t G, int32_t topk, int32_t nblk, int32_t win,
                                const DenseWorkspace& w, int32_t* counts, int32_t* epos,
                                cudaStream_t stream);
cudaError_t launch_dense_attention(const CUtensorMap& qmap, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, int32_t q_atoms, int32_t T,
                                   int64_t S_kv, int32_t Hkv, int32_t G,
                                   const int32_t* page_table, int64_t num_pages,
                                   const DenseWorkspace& w, cudaStream_t stream);

// (a) bucketing; tiles of `qpt` queries are laid out for the attention kernel.
// List of selection (t, slot) of group g: ((g * nwin + t / win) * nblk + j); the per-list
// offsets are relative to their (group, window) segment, segments in (g, w) order.
// launch_bucket_lists finishes lists counted by launch_select_count (offsets, tile descriptors
// when `desc` is set, entries; with `dcnt` also the query-major pairs' deal into `porder`, in
// extra blocks); launch_bucket runs all of it on plain selections.
cudaError_t launch_bucket_lists(const int32_t* ids, const int32_t* epos, int32_t T, int32_t Hkv,
                                int32_t topk, int32_t nblk, int32_t win, int32_t qpt,
                                const int32_t* counts, int32_t* offsets, int32_t* entries,
                                int32_t* group_base, int32_t* tile_offsets, int4* desc,
                                const int32_t* dcnt, int64_t npairs, int32_t* porder,
                                cudaStream_t stream);
cudaError_t launch_bucket(const int32_t* block_ids, int32_t T, int32_t Hkv, int32_t topk,
                          int32_t nblk, int32_t win, int32_t qpt, int32_t* offsets,
                          int32_t* entries, int32_t* counts, int32_t* group_base,
                          int32_t* tile_offsets, int32_t* epos, cudaStream_t stream);
struct PrefillArgs {
  const uint16_t* q;           // [T, Hq, D]
  const uint16_t* k;           // [S_kv, Hkv, D], or paged [num_pages, 128, Hkv, D]
  const uint16_t* v;
  const int32_t* page_table;   // null (contiguous K/V) or [nblk]: page of each 128-token block
  int64_t num_pages;
  const int32_t* block_ids;    // [T, Hkv, topk]
  int32_t T, Hq, Hkv, D, topk, nblk;
  int64_t S_kv;
  uint16_t* o;                 // [T, Hq, D]
  float* lse;                  // [T, Hq] or null
  uint8_t* workspace;          // carved by prefill_ws_layout(..., attention = true)
};
cudaError_t launch_sparse_prefill(const PrefillArgs& a, cudaStream_t stream);

// ------------------------------------------------------------------ device errors
cudaError_t read_device_errors(uint32_t* word);

}  // namespace msa
