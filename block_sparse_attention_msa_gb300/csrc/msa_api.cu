// The C ABI of libmsa_gb300.so (declared in include/msa.h): host-side argument checks,
// workspace carving and dispatch to the kernel launchers. Nothing here allocates memory,
// synchronises or reads device data, except msa_device_error (a diagnostic).
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "host_util.h"
#include "kernels.h"
#include "msa.h"

cudaError_t msa_read_error_score(uint32_t* w);
cudaError_t msa_read_error_ptm(uint32_t* w);
cudaError_t msa_read_error_dec(uint32_t* w);
cudaError_t msa_read_error_pre(uint32_t* w);
cudaError_t msa_read_error_dense(uint32_t* w);
cudaError_t msa_read_error_stage(uint32_t* w);

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return MSA_OK;
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(MSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool pow2_upto(int32_t x, int32_t hi) { return x >= 1 && x <= hi && (x & (x - 1)) == 0; }

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

constexpr int64_t kInt32Max = 2147483647;

size_t score_ws_scores_bytes(int32_t B, int32_t N, int32_t Hkv, int32_t max_blocks) {
  return msa::ws_align((size_t)B * N * Hkv * max_blocks * sizeof(float));
}

}  // namespace

extern "C" {

const char* msa_last_error(void) { return g_last_error.c_str(); }

const char* msa_version(void) { return "0.1.0"; }

// ------------------------------------------------------------------------------ stage 1
size_t msa_index_score_topk_workspace_size(int32_t B, int32_t N, int32_t Hkv, int32_t max_blocks) {
  if (B <= 0 || N <= 0 || Hkv <= 0 || max_blocks <= 0) return 0;
  return score_ws_scores_bytes(B, N, Hkv, max_blocks) + msa::ws_align((size_t)B * sizeof(int32_t));
}

// Host checks of a stage-1 call's tensors and sizes (not its workspace), before any CUDA
// call: shared by the workspace and the scratch-array entry points, so that both report the
// same error for the same arguments.
static int check_score_args(const char* name, const uint16_t* q_idx, const uint16_t* k_idx_pages,
                            const int32_t* page_table, const int32_t* seq_lens, int32_t B,
                            int32_t N, int32_t Hkv, int32_t Di, int32_t max_blocks,
                            int64_t num_pages, int32_t topk, const int32_t* block_ids) {
  if (!q_idx || !k_idx_pages || !page_table || !seq_lens || !block_ids)
    return fail(MSA_ERR_ARG, "%s: null tensor pointer", name);
  if (B < 0 || N < 0 || max_blocks <= 0 || num_pages <= 0)
    return fail(MSA_ERR_ARG, "%s: B=%d N=%d max_blocks=%d num_pages=%lld", name, B, N,
                max_blocks, (long long)num_pages);
  if (topk < 2 || topk > 64)
    return fail(MSA_ERR_UNSUPPORTED, "%s: topk=%d outside [2, 64]", name, topk);
  if (!pow2_upto(Hkv, 16)) return fail(MSA_ERR_UNSUPPORTED, "%s: Hkv=%d", name, Hkv);
  if (Di != 64 && Di != 128) return fail(MSA_ERR_UNSUPPORTED, "%s: Di=%d", name, Di);
  if (num_pages * 128 * Hkv > kInt32Max)
    return fail(MSA_ERR_UNSUPPORTED, "%s: num_pages*128*Hkv exceeds int32", name);
  if ((int64_t)max_blocks * 128 > kInt32Max || (int64_t)B * N > kInt32Max)
    return fail(MSA_ERR_SHAPE, "%s: sizes exceed int32", name);
  if ((int64_t)N > (int64_t)max_blocks * 128)
    return fail(MSA_ERR_SHAPE, "%s: N=%d exceeds max_blocks*128", name, N);
  return MSA_OK;
}

static int index_score_topk_impl(const char* name, const uint16_t* q_idx,
                                 const uint16_t* k_idx_pages, const int32_t* page_table,
                                 const int32_t* seq_lens, int32_t B, int32_t N, int32_t Hkv,
                                 int32_t Di, int32_t max_blocks, int64_t num_pages, int32_t topk,
                                 int32_t* block_ids, float* scores, int32_t* fpt,
                                 int32_t* fpt_lens, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  if (B == 0 || N == 0) return ok();
  const int rc = check_score_args(name, q_idx, k_idx_pages, page_table, seq_lens, B, N, Hkv, Di,
                                  max_blocks, num_pages, topk, block_ids);
  if (rc != MSA_OK) return rc;
  const size_t need = msa_index_score_topk_workspace_size(B, N, Hkv, max_blocks);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return fail(MSA_ERR_WORKSPACE,
                "%s: workspace %p of %zu bytes (need %zu, 256-byte aligned)", name, workspace,
                workspace_bytes, need);
  msa::ScoreArgs a;
  a.q_idx = q_idx;
  a.k_idx = k_idx_pages;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.B = B;
  a.N = N;
  a.Hkv = Hkv;
  a.Di = Di;
  a.max_blocks = max_blocks;
  a.topk = topk;
  a.num_pages = num_pages;
  a.block_ids = block_ids;
  a.sel_scores = scores;
  a.fpt = fpt;
  a.fpt_lens = fpt_lens;
  // workspace: per-request tickets [B] int32 first, then the block scores
  a.tickets = reinterpret_cast<int32_t*>(workspace);
  a.scores = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                      msa::ws_align((size_t)B * sizeof(int32_t)));
  int nstage = 0;
  msa::score_decode_smem_bytes(N, Hkv, Di, &nstage);
  // one query row per request: the CUDA-core streaming scorer, with the top-k (and the page
  // table) fused into its last CTA per request; 2..16 rows: the tensor-core decode scorer (the
  // key index read once for all rows); longer chunks: the multi-row scorer. The last two are
  // followed by the top-k kernel (one warp per row) and, when asked for, the page-table kernel.
  const bool streaming = N == 1 && nstage >= 2;
  const bool tc_decode = N >= 2 && N <= msa::kDecodeTcMaxN && msa::score_tc_decode_stages(Hkv, Di) >= 2;
  if (streaming) {
    // the fused top-k counts finished pages per request from zero
    cudaError_t e = cudaMemsetAsync(a.tickets, 0, (size_t)B * sizeof(int32_t), as_stream(stream));
    if (e == cudaSuccess) e = msa::launch_score_decode(a, as_stream(stream));
    return cuda_status(e, name);
  }
  cudaError_t e = tc_decode ? msa::launch_score_tc_decode(a, as_stream(stream))
                            : msa::launch_score_rows(a, as_stream(stream));
  if (e == cudaSuccess) e = msa::launch_topk_rows(a, as_stream(stream));
  if (e == cudaSuccess && fpt)
    e = msa::launch_build_page_table(block_ids, page_table, seq_lens, B, N, Hkv, topk, max_blocks,
                                     num_pages, fpt, fpt_lens, as_stream(stream));
  return cuda_status(e, name);
}

int msa_index_score_topk(const uint16_t* q_idx, const uint16_t* k_idx_pages,
                         const int32_t* page_table, const int32_t* seq_lens, int32_t B,
                         int32_t N, int32_t Hkv, int32_t Di, int32_t max_blocks,
                         int64_t num_pages, int32_t topk, int32_t* block_ids, float* scores,
                         void* workspace, size_t workspace_bytes, void* stream) {
  return index_score_topk_impl("msa_index_score_topk", q_idx, k_idx_pages, page_table, seq_lens,
                               B, N, Hkv, Di, max_blocks, num_pages, topk, block_ids, scores,
                               nullptr, nullptr, workspace, workspace_bytes, stream);
}

int msa_index_score_topk_page_table(const uint16_t* q_idx, const uint16_t* k_idx_pages,
                                    const int32_t* page_table, const int32_t* seq_lens, int32_t B,
                                    int32_t N, int32_t Hkv, int32_t Di, int32_t max_blocks,
                                    int64_t num_pages, int32_t topk, int32_t* block_ids,
                                    float* scores, int32_t* flat_page_table, int32_t* flat_kv_lens,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (B != 0 && N != 0 && (!flat_page_table || !flat_kv_lens))
    return fail(MSA_ERR_ARG, "msa_index_score_topk_page_table: null page-table output");
  return index_score_topk_impl("msa_index_score_topk_page_table", q_idx, k_idx_pages, page_table,
                               seq_lens, B, N, Hkv, Di, max_blocks, num_pages, topk, block_ids,
                               scores, flat_page_table, flat_kv_lens, workspace, workspace_bytes,
                               stream);
}

// ------------------------------------------------------------------------------ page table
int msa_build_sparse_page_table(const int32_t* block_ids, const int32_t* page_table,
                                const int32_t* seq_lens, int32_t B, int32_t N, int32_t Hkv,
                                int32_t topk, int32_t max_blocks, int64_t num_pages,
                                int32_t* flat_page_table, int32_t* flat_kv_lens, void* stream) {
  if (B == 0 || N == 0) return ok();
  if (!block_ids || !page_table || !seq_lens || !flat_page_table || !flat_kv_lens)
    return fail(MSA_ERR_ARG, "msa_build_sparse_page_table: null tensor pointer");
  if (B < 0 || N < 0 || max_blocks <= 0 || num_pages <= 0 || topk < 1 || topk > 64)
    return fail(MSA_ERR_ARG, "msa_build_sparse_page_table: B=%d N=%d topk=%d max_blocks=%d", B, N,
                topk, max_blocks);
  if (!pow2_upto(Hkv, 16))
    return fail(MSA_ERR_UNSUPPORTED, "msa_build_sparse_page_table: Hkv=%d", Hkv);
  if (num_pages * 128 * Hkv > kInt32Max)
    return fail(MSA_ERR_UNSUPPORTED, "msa_build_sparse_page_table: num_pages*128*Hkv exceeds int32");
  if ((int64_t)N > (int64_t)max_blocks * 128)
    return fail(MSA_ERR_SHAPE, "msa_build_sparse_page_table: N=%d exceeds max_blocks*128", N);
  return cuda_status(msa::launch_build_page_table(block_ids, page_table, seq_lens, B, N, Hkv, topk,
                                                  max_blocks, num_pages, flat_page_table,
                                                  flat_kv_lens, as_stream(stream)),
                     "msa_build_sparse_page_table");
}

// ------------------------------------------------------------------------------ KV staging
int msa_stage_selected_kv(const uint16_t* k_cache, const uint16_t* v_cache, int64_t num_pages,
                          const int32_t* flat_page_table, int32_t R, int32_t Hkv, int32_t D,
                          int32_t topk, uint16_t* k_stage, uint16_t* v_stage,
                          int32_t* stage_page_table, void* stream) {
  if (R == 0) return ok();
  if (!k_cache || !v_cache || !flat_page_table || !k_stage || !v_stage || !stage_page_table)
    return fail(MSA_ERR_ARG, "msa_stage_selected_kv: null pointer");
  if (R < 0 || num_pages <= 0 || topk < 1 || topk > 64)
    return fail(MSA_ERR_ARG, "msa_stage_selected_kv: R=%d num_pages=%lld topk=%d", R,
                (long long)num_pages, topk);
  if (D != 128) return fail(MSA_ERR_UNSUPPORTED, "msa_stage_selected_kv: D=%d (only 128)", D);
  if (!pow2_upto(Hkv, 16)) return fail(MSA_ERR_UNSUPPORTED, "msa_stage_selected_kv: Hkv=%d", Hkv);
  if (num_pages * 128 * Hkv > kInt32Max || (int64_t)R * topk * 128 * Hkv > kInt32Max)
    return fail(MSA_ERR_UNSUPPORTED, "msa_stage_selected_kv: pages*128*Hkv exceeds int32");
  return cuda_status(msa::launch_stage_kv(k_cache, v_cache, num_pages, flat_page_table, R, Hkv,
                                          topk, k_stage, v_stage, stage_page_table,
                                          as_stream(stream)),
                     "msa_stage_selected_kv");
}

// ------------------------------------------------------------------------------ decode
size_t msa_paged_sparse_decode_workspace_size(int32_t R, int32_t Hq, int32_t Hkv, int32_t topk) {
  if (R <= 0 || Hq <= 0 || Hkv <= 0 || topk <= 0) return 0;
  const size_t units = (size_t)R * Hq * msa::decode_slots(topk);  // (row, group, slot, head)
  return msa::ws_align(units * 128 * sizeof(float)) + msa::ws_align(units * sizeof(float));
}

int msa_paged_sparse_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                            const int32_t* flat_page_table, const int32_t* flat_kv_lens,
                            int32_t R, int32_t Hq, int32_t Hkv, int32_t D, int32_t topk,
                            int64_t num_pages, uint16_t* o, float* lse, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (R == 0) return ok();
  if (!q || !k_cache || !v_cache || !flat_page_table || !flat_kv_lens || !o)
    return fail(MSA_ERR_ARG, "msa_paged_sparse_decode: null tensor pointer");
  if (R < 0 || num_pages <= 0 || topk < 1 || topk > 64)
    return fail(MSA_ERR_ARG, "msa_paged_sparse_decode: R=%d topk=%d num_pages=%lld", R, topk,
                (long long)num_pages);
  if (D != 128) return fail(MSA_ERR_UNSUPPORTED, "msa_paged_sparse_decode: D=%d (only 128)", D);
  if (!pow2_upto(Hkv, 16) || Hq % Hkv != 0 || !pow2_upto(Hq / Hkv, 16))
    return fail(MSA_ERR_UNSUPPORTED, "msa_paged_sparse_decode: Hq=%d Hkv=%d", Hq, Hkv);
  if (num_pages * 128 * Hkv > kInt32Max)
    return fail(MSA_ERR_UNSUPPORTED, "msa_paged_sparse_decode: num_pages*128*Hkv exceeds int32");
  const size_t need = msa_paged_sparse_decode_workspace_size(R, Hq, Hkv, topk);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return fail(MSA_ERR_WORKSPACE,
                "msa_paged_sparse_decode: workspace %p of %zu bytes (need %zu, 256-byte aligned)",
                workspace, workspace_bytes, need);
  msa::DecodeArgs a;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.fpt = flat_page_table;
  a.lens = flat_kv_lens;
  a.R = R;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.topk = topk;
  a.num_pages = num_pages;
  a.o = o;
  a.lse = lse;
  a.nslots = msa::decode_slots(topk);
  const size_t units = (size_t)R * Hq * a.nslots;
  a.part_o = reinterpret_cast<float*>(workspace);
  a.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                        msa::ws_align(units * 128 * sizeof(float)));
  return cuda_status(msa::launch_paged_decode(a, as_stream(stream)), "msa_paged_sparse_decode");
}

// ------------------------------------------------------------------------------ prefill
size_t msa_sparse_prefill_workspace_size(int32_t T, int64_t S_kv, int32_t Hq, int32_t Hkv,
                                         int32_t topk) {
  if (T <= 0 || S_kv <= 0 || Hq <= 0 || Hkv <= 0 || topk <= 0 || Hq % Hkv) return 0;
  const int32_t nblk = (int32_t)((S_kv + 127) / 128);
  return msa::prefill_ws_layout(T, Hkv, topk, nblk, Hq / Hkv, true).total;
}

static int sparse_prefill_impl(const char* name, const uint16_t* q, const uint16_t* k,
                               const uint16_t* v, const int32_t* page_table, int64_t num_pages,
                               const int32_t* block_ids, int32_t T, int64_t S_kv, int32_t Hq,
                               int32_t Hkv, int32_t D, int32_t topk, uint16_t* o, float* lse,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (T == 0) return ok();
  if (!q || !k || !v || !block_ids || !o) return fail(MSA_ERR_ARG, "%s: null tensor pointer", name);
  if (T < 0 || S_kv < T || topk < 1 || topk > 64)
    return fail(MSA_ERR_ARG, "%s: T=%d S_kv=%lld topk=%d", name, T, (long long)S_kv, topk);
  if (S_kv > kInt32Max - 128) return fail(MSA_ERR_UNSUPPORTED, "%s: S_kv too large", name);
  if (D != 128) return fail(MSA_ERR_UNSUPPORTED, "%s: D=%d (only 128)", name, D);
  if (!pow2_upto(Hkv, 16) || Hq % Hkv != 0 || !pow2_upto(Hq / Hkv, 16))
    return fail(MSA_ERR_UNSUPPORTED, "%s: Hq=%d Hkv=%d", name, Hq, Hkv);
  if ((int64_t)T * Hkv * topk > kInt32Max)
    return fail(MSA_ERR_UNSUPPORTED, "%s: T*Hkv*topk exceeds int32", name);
  if (page_table && (num_pages <= 0 || num_pages * 128 > kInt32Max))
    return fail(MSA_ERR_ARG, "%s: num_pages=%lld", name, (long long)num_pages);
  const size_t need = msa_sparse_prefill_workspace_size(T, S_kv, Hq, Hkv, topk);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return fail(MSA_ERR_WORKSPACE, "%s: workspace %p of %zu bytes (need %zu, 256-byte aligned)",
                name, workspace, workspace_bytes, need);
  msa::PrefillArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.page_table = page_table;
  a.num_pages = num_pages;
  a.block_ids = block_ids;
  a.T = T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.topk = topk;
  a.nblk = (int32_t)((S_kv + 127) / 128);
  a.S_kv = S_kv;
  a.o = o;
  a.lse = lse;
  a.workspace = static_cast<uint8_t*>(workspace);
  return cuda_status(msa::launch_sparse_prefill(a, as_stream(stream)), name);
}

int msa_sparse_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const int32_t* block_ids, int32_t T, int64_t S_kv, int32_t Hq,
                       int32_t Hkv, int32_t D, int32_t topk, uint16_t* o, float* lse,
                       void* workspace, size_t workspace_bytes, void* stream) {
  return sparse_prefill_impl("msa_sparse_prefill", q, k, v, nullptr, 0, block_ids, T, S_kv, Hq,
                             Hkv, D, topk, o, lse, workspace, workspace_bytes, stream);
}

int msa_sparse_prefill_paged(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                             const int32_t* page_table, int64_t num_pages,
                             const int32_t* block_ids, int32_t T, int64_t S_kv, int32_t Hq,
                             int32_t Hkv, int32_t D, int32_t topk, uint16_t* o, float* lse,
                             void* workspace, size_t workspace_bytes, void* stream) {
  if (T != 0 && !page_table) return fail(MSA_ERR_ARG, "msa_sparse_prefill_paged: null page table");
  return sparse_prefill_impl("msa_sparse_prefill_paged", q, k_cache, v_cache, page_table,
                             num_pages, block_ids, T, S_kv, Hq, Hkv, D, topk, o, lse, workspace,
                             workspace_bytes, stream);
}

size_t msa_prefill_bucket_workspace_size(int32_t T, int32_t Hkv, int32_t topk, int32_t nblk) {
  if (T < 0 || Hkv <= 0 || topk <= 0 || nblk <= 0) return 0;
  return msa::prefill_ws_layout(T, Hkv, topk, nblk, 1, false).total;
}

int msa_prefill_bucket(const int32_t* block_ids, int32_t T, int32_t Hkv, int32_t topk,
                       int32_t nblk, int32_t* offsets, int32_t* entries, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (!block_ids || !offsets || !entries)
    return fail(MSA_ERR_ARG, "msa_prefill_bucket: null tensor pointer");
  if (T < 0 || Hkv <= 0 || Hkv > 16 || topk < 1 || topk > 64 || nblk <= 0)
    return fail(MSA_ERR_ARG, "msa_prefill_bucket: T=%d Hkv=%d topk=%d nblk=%d", T, Hkv, topk, nblk);
  if ((int64_t)T * Hkv * topk > kInt32Max)
    return fail(MSA_ERR_UNSUPPORTED, "msa_prefill_bucket: T*Hkv*topk exceeds int32");
  if (T == 0)  // every list is empty
    return cuda_status(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (size_t)Hkv * (nblk + 1),
                                       as_stream(stream)),
                       "msa_prefill_bucket");
  const size_t need = msa_prefill_bucket_workspace_size(T, Hkv, topk, nblk);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return fail(MSA_ERR_WORKSPACE, "msa_prefill_bucket: workspace of %zu bytes (need %zu)",
                workspace_bytes, need);
  const msa::PrefillWorkspace W = msa::prefill_ws_layout(T, Hkv, topk, nblk, 1, false);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return cuda_status(
      msa::launch_bucket(block_ids, T, Hkv, topk, nblk, T, 128, offsets, entries,
                         reinterpret_cast<int32_t*>(ws + W.counts),
                         reinterpret_cast<int32_t*>(ws + W.group_base),
                         reinterpret_cast<int32_t*>(ws + W.tile_offsets),
                         reinterpret_cast<int32_t*>(ws + W.epos), as_stream(stream)),
      "msa_prefill_bucket");
}

int msa_lse_merge(const void* o_parts, int32_t parts_bf16, const float* lse_parts, int64_t U,
                  int32_t S, int32_t G, int32_t D, uint16_t* o, float* lse, void* stream) {
  if (U == 0) return ok();
  if (!o_parts || !lse_parts || !o) return fail(MSA_ERR_ARG, "msa_lse_merge: null tensor pointer");
  if (U < 0 || S < 1 || G < 1 || D < 4 || D % 4 != 0)
    return fail(MSA_ERR_ARG, "msa_lse_merge: U=%lld S=%d G=%d D=%d", (long long)U, S, G, D);
  if (reinterpret_cast<uintptr_t>(o_parts) & 15)
    return fail(MSA_ERR_ARG, "msa_lse_merge: o_parts must be 16-byte aligned");
  return cuda_status(msa::launch_lse_merge(o_parts, parts_bf16 != 0, lse_parts, nullptr, U, S, G,
                                           D, o, lse, as_stream(stream)),
                     "msa_lse_merge");
}

// ------------------------------------------------------------------------------ scoring without
// a caller workspace
//
// Scratch of msa_index_score_topk_noalloc: one fixed array in device memory, created when
// the library's module is first used on a device (CUDA loads modules lazily) and held until
// the process exits or the device is reset. Host code only sees a host-side stand-in for it,
// so its device address is looked up per device (below).
static __device__ __align__(256) unsigned char g_noalloc_score_scratch[MSA_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device. It is resolved on the first
// call on a device, and again on every call whose stream is not being captured: a device
// reset (cudaDeviceReset) unloads the module, and the array may sit elsewhere once the module
// is loaded again. During a capture the address cached by the last call outside one is used.
int noalloc_scratch(cudaStream_t stream, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e, "msa_index_score_topk_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(MSA_ERR_UNSUPPORTED, "msa_index_score_topk_noalloc: device %d", dev);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return cuda_status(e, "msa_index_score_topk_noalloc: cudaStreamIsCapturing");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev] || cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_score_scratch);
    if (e != cudaSuccess || !p)
      return cuda_status(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                         "msa_index_score_topk_noalloc: cudaGetSymbolAddress");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MSA_OK;
}
}  // namespace

int msa_index_score_topk_noalloc(const uint16_t* q_idx, const uint16_t* k_idx_pages,
                                 const int32_t* page_table, const int32_t* seq_lens, int32_t B,
                                 int32_t N, int32_t Hkv, int32_t Di, int32_t max_blocks,
                                 int64_t num_pages, int32_t topk, int32_t* block_ids,
                                 float* scores, void* stream) {
  if (B == 0 || N == 0) return ok();
  const int rc_args = check_score_args("msa_index_score_topk_noalloc", q_idx, k_idx_pages,
                                       page_table, seq_lens, B, N, Hkv, Di, max_blocks, num_pages,
                                       topk, block_ids);
  if (rc_args != MSA_OK) return rc_args;
  const size_t need = msa_index_score_topk_workspace_size(B, N, Hkv, max_blocks);
  if (need > (size_t)MSA_NOALLOC_SCRATCH_BYTES)
    return fail(MSA_ERR_UNSUPPORTED,
                "msa_index_score_topk_noalloc: this call needs %zu bytes of scratch but the "
                "built-in scratch holds %zu (B*N*Hkv*max_blocks too large); call "
                "msa_index_score_topk with a workspace instead",
                need, (size_t)MSA_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  const int rc = noalloc_scratch(as_stream(stream), &scratch);
  if (rc != MSA_OK) return rc;
  // Same checks, kernels and per-call clearing of the ticket counters as the workspace
  // entry point; the scratch array simply stands in for the workspace.
  return msa_index_score_topk(q_idx, k_idx_pages, page_table, seq_lens, B, N, Hkv, Di,
                              max_blocks, num_pages, topk, block_ids, scores, scratch,
                              (size_t)MSA_NOALLOC_SCRATCH_BYTES, stream);
}

// ------------------------------------------------------------------------------ diagnostics
int msa_device_error(uint32_t* word) {
  if (!word) return fail(MSA_ERR_ARG, "msa_device_error: null output pointer");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_status(e, "msa_device_error");
  uint32_t all = 0, w = 0;
  cudaError_t (*readers[])(uint32_t*) = {msa_read_error_score, msa_read_error_ptm,
                                         msa_read_error_dec, msa_read_error_pre,
                                         msa_read_error_dense, msa_read_error_stage};
  for (auto rd : readers) {
    w = 0;
    e = rd(&w);
    if (e != cudaSuccess) return cuda_status(e, "msa_device_error");
    all |= w;
  }
  *word = all;
  if (all) return fail(MSA_ERR_DEVICE, "device error word 0x%x", all);
  return ok();
}

}  // extern "C"
