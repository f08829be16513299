/*
 * msa.h -- C ABI of the GB300 (sm_103a) MiniMax Sparse Attention (MSA) layer library,
 *          libmsa_gb300.so.
 *
 * MSA runs one attention layer in two stages: stage 1 scores every 128-token KV block per
 * KV group and keeps the top-k blocks; stage 2 runs dense causal GQA attention between
 * the query tokens and only the kept blocks (Together AI MiniMax-M3 serving article,
 * section "MiniMax Sparse Attention changes the serving problem").
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Block = page = 128 tokens (MSA_BLOCK). Positions are 0-based. A query at position t
 *    sees keys 0..t; its local block is t/128; block 0 is the sink block.
 *  - GQA: Hq query heads, Hkv KV groups, G = Hq/Hkv heads per group; head h belongs to
 *    group h/G. One index head per KV group (index dim Di).
 *  - bf16 tensors are passed as uint16_t* (raw bf16 bit patterns); int32 tables as
 *    int32_t*; fp32 as float*. Every tensor is dense, row-major, in the layout stated: the
 *    calls take plain pointers and cannot see strides, so a strided view must be made
 *    contiguous by the caller (the Python binding checks this and raises).
 *  - Query rows: request b of a batch of B requests holds N query rows r = b*N + i
 *    (i = 0..N-1) at positions seq_lens[b] - N + i, i.e. the last N tokens of the request,
 *    whose K/V/K-index are already in the cache. Decode is N = 1; multi-token decode
 *    (speculative verify) is N = 2..16; a prefill chunk of one request is B = 1, N = T.
 *  - q is pre-scaled by 1/sqrt(D): the kernels apply no softmax scale. LSE is the natural
 *    log-sum-exp of the scaled scores, fp32.
 *
 * Ownership, synchronisation and errors
 * -------------------------------------
 *  - Every pointer argument except the ones marked "host" is DEVICE memory owned by the
 *    caller, valid until the work queued on `stream` has finished. The library allocates
 *    nothing: calls that need scratch take a caller-provided `workspace` of at least the
 *    size reported by the matching *_workspace_size() function.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy
 *    default stream). They never synchronise and never read device data on the host.
 *  - Return value: MSA_OK (0) or a negative MSA_ERR_* code. Argument checks run on the host
 *    before anything is queued; on error nothing is queued and msa_last_error() returns a
 *    thread-local message. A CUDA launch failure returns MSA_ERR_CUDA.
 *  - Device-side checks: page ids, block ids and sequence lengths read from device tables
 *    are range-checked inside the kernels before any address is formed from them. A bad
 *    value is never dereferenced: a page id out of range is read as page 0 (page 0, group
 *    0 for a virtual page of the strided view), a sequence length above max_blocks*128 is
 *    clamped to it, and a sparse page-table entry whose block or page is invalid becomes
 *    -1. Each case sets a bit of a device error word that msa_device_error() reads back
 *    (that call synchronises).
 *
 * Supported values: D = 128; Di in {64, 128}; G in {1, 2, 4, 8, 16} with Hkv*G = Hq;
 * Hkv in {1, 2, 4, 8, 16}; 2 <= topk <= 64.
 */
#ifndef MSA_GB300_H
#define MSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MSA_API __attribute__((visibility("default")))
#else
#define MSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define MSA_BLOCK 128

enum {
  MSA_OK = 0,
  MSA_ERR_ARG = -1,          /* null pointer or value out of range */
  MSA_ERR_SHAPE = -2,        /* inconsistent sizes */
  MSA_ERR_UNSUPPORTED = -3,  /* a size outside the supported set above */
  MSA_ERR_WORKSPACE = -4,    /* workspace missing, too small or misaligned */
  MSA_ERR_CUDA = -5,         /* a CUDA runtime call or launch failed */
  MSA_ERR_DEVICE = -6        /* msa_device_error(): a kernel recorded a bad id or timeout */
};

/* ------------------------------------------------------------------------------------
 * Stage 1 -- index scoring and top-k block selection.
 *
 * Passages: Together AI MiniMax-M3 serving article, section "The index scorer becomes the
 * decode critical path" (each query-side index vector is compared with the key-side index
 * vectors of the candidate blocks; each 128-token block is reduced to one score; only the
 * top blocks are kept; every request and KV group has its own candidate range and mask);
 * the Japanese translation, section "Decode Index Scoring Kernel Optimization" (bf16 dot
 * products, one score per page).
 *
 * For every query row r and KV group g:
 *   score[r,g,j] = max over tokens pos = 128*j + tau <= q_pos(r) of
 *                  sum_d q_idx[r,g,d] * k_idx[page_table[b,j], tau, g, d]   (fp32 accumulate)
 *   for the causal blocks j = 0 .. q_pos(r)/128. Selection: the sink block 0 and the local
 *   block q_pos/128 are always kept and count toward topk; the remaining slots take the
 *   other causal blocks by score descending, ties to the lower block id. Output ids are
 *   ascending, then -1 padding when fewer than topk causal blocks exist.
 *
 *   q_idx        [B*N, Hkv, Di] bf16
 *   k_idx_pages  [num_pages, 128, Hkv, Di] bf16 -- the paged key-index cache
 *   page_table   [B, max_blocks] int32 -- page of block j of request b (j < ceil(seq_len/128))
 *   seq_lens     [B] int32, N <= seq_lens[b] <= max_blocks*128
 *   block_ids    [B*N, Hkv, topk] int32 (out)
 *   scores       [B*N, Hkv, topk] fp32 (out, may be NULL): score of each kept block,
 *                -inf for padding
 *   workspace    >= msa_index_score_topk_workspace_size(B, N, Hkv, max_blocks) bytes,
 *                256-byte aligned, any contents (the call clears what it counts from).
 *                Calls that may run concurrently need separate workspaces.
 * ------------------------------------------------------------------------------------ */
MSA_API size_t msa_index_score_topk_workspace_size(int32_t B, int32_t N, int32_t Hkv, int32_t max_blocks);

MSA_API int msa_index_score_topk(const uint16_t* q_idx, const uint16_t* k_idx_pages,
                         const int32_t* page_table, const int32_t* seq_lens, int32_t B,
                         int32_t N, int32_t Hkv, int32_t Di, int32_t max_blocks,
                         int64_t num_pages, int32_t topk, int32_t* block_ids, float* scores,
                         void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * msa_index_score_topk followed by msa_build_sparse_page_table on its selection, in one
 * call: for N = 1 the warp that selects a row's blocks in the scorer's last CTA for the
 * request also writes the row's sparse page table and length, so no separate launch and no
 * round trip of block_ids sits between the selection and the paged decode; for N > 1 the
 * page-table kernel follows the top-k kernel within the call.
 *
 * Passages: as msa_index_score_topk and msa_build_sparse_page_table (Together AI MiniMax-M3
 * serving article, sections "The index scorer becomes the decode critical path" and "MSA
 * needs a new paged-attention integration"; the pages list top-k and the page-table build
 * among the small kernels around the attention).
 *
 *   arguments as msa_index_score_topk, plus
 *   flat_page_table [B*N*Hkv, topk] int32 (out), flat_kv_lens [B*N*Hkv] int32 (out), exactly
 *   as msa_build_sparse_page_table(block_ids, page_table, seq_lens, ...) would write them.
 * Returns MSA_ERR_ARG for a null page-table output; otherwise as msa_index_score_topk.
 * ------------------------------------------------------------------------------------ */
MSA_API int msa_index_score_topk_page_table(const uint16_t* q_idx, const uint16_t* k_idx_pages,
                                            const int32_t* page_table, const int32_t* seq_lens,
                                            int32_t B, int32_t N, int32_t Hkv, int32_t Di,
                                            int32_t max_blocks, int64_t num_pages, int32_t topk,
                                            int32_t* block_ids, float* scores,
                                            int32_t* flat_page_table, int32_t* flat_kv_lens,
                                            void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Sparse page table for paged decode.
 *
 * Passage: Together AI MiniMax-M3 serving article, section "MSA needs a new paged-attention
 * integration" (a page table is built from the selected blocks at decode; the KV-group
 * dimension is flattened into the batch; a strided view of the KV-cache tensor gives each
 * flattened row its own pages: the page address steps by D to select the virtual page
 * start and tokens step by Hkv*D, deinterleaving one physical tensor into per-head pages).
 *
 * Flattened row f = r*Hkv + g. Virtual page of physical page p for group g:
 *   v = p*128*Hkv + g;  element (v, tau, d) of the view is cache[v*D + tau*Hkv*D + d],
 *   i.e. cache[p, tau, g, d] of a [num_pages, 128, Hkv, D] tensor.
 *   flat_page_table[f, i] = virtual page of the i-th kept block (ascending), -1 after.
 *   flat_kv_lens[f]       = visible tokens: 128 per kept block below the local block plus
 *                           q_pos%128 + 1 for the local block.
 *
 *   block_ids   [B*N, Hkv, topk] int32 (from msa_index_score_topk)
 *   page_table  [B, max_blocks] int32; seq_lens [B] int32
 *   flat_page_table [B*N*Hkv, topk] int32 (out); flat_kv_lens [B*N*Hkv] int32 (out)
 * Requires num_pages*128*Hkv < 2^31 (virtual page ids are int32).
 * ------------------------------------------------------------------------------------ */
MSA_API int msa_build_sparse_page_table(const int32_t* block_ids, const int32_t* page_table,
                                const int32_t* seq_lens, int32_t B, int32_t N, int32_t Hkv,
                                int32_t topk, int32_t max_blocks, int64_t num_pages,
                                int32_t* flat_page_table, int32_t* flat_kv_lens, void* stream);

/* ------------------------------------------------------------------------------------
 * KV residency split: copy only the selected blocks' K/V to the device.
 *
 * Passages: Together AI MiniMax-M3 serving article, sections "The index scorer becomes the
 * decode critical path" (the scorer reads the small key index of every block; the attention
 * needs only the selected blocks) and "MSA needs a new paged-attention integration" (the
 * selection as a page table over the strided per-head view).
 *
 * The paged caches may live in host memory (pinned, so that the device can read it: on a
 * Grace host over NVLink-C2C) while the key index and the scorer stay on the device. For every
 * flattened row f = r*Hkv + g and slot i with flat_page_table[f, i] = p*128*Hkv + g >= 0, the
 * 128 token rows of group g of page p are copied from k_cache / v_cache to staging page
 * r*topk + i, group slot g, of k_stage / v_stage, and stage_page_table[f, i] = (r*topk + i)*
 * 128*Hkv + g (-1 where the input is -1). msa_paged_sparse_decode(q, k_stage, v_stage,
 * stage_page_table, flat_kv_lens, R, Hq, Hkv, D, topk, R*topk, ...) then gives the same result
 * as on the full caches.
 *
 *   k_cache, v_cache [num_pages, 128, Hkv, D] bf16 (device or device-readable host memory)
 *   flat_page_table  [R*Hkv, topk] int32 (from msa_build_sparse_page_table)
 *   k_stage, v_stage [R*topk, 128, Hkv, D] bf16 device (out; rows of unselected slots untouched)
 *   stage_page_table [R*Hkv, topk] int32 device (out)
 * A virtual page outside the caches or of another group is recorded in the device error
 * word (kErrBadPage) and staged as -1.
 * ------------------------------------------------------------------------------------ */
MSA_API int msa_stage_selected_kv(const uint16_t* k_cache, const uint16_t* v_cache,
                                  int64_t num_pages, const int32_t* flat_page_table, int32_t R,
                                  int32_t Hkv, int32_t D, int32_t topk, uint16_t* k_stage,
                                  uint16_t* v_stage, int32_t* stage_page_table, void* stream);

/* ------------------------------------------------------------------------------------
 * Paged sparse decode attention over the strided per-head view.
 *
 * Passages: Together AI MiniMax-M3 serving article, sections "MSA needs a new
 * paged-attention integration" (flattened rows with per-row page tables over one shared
 * KV tensor) and "MiniMax Sparse Attention changes the serving problem" (stage two: dense
 * attention between the queries and the selected blocks).
 *
 * For flattened row f = r*Hkv + g and each of its G heads h = g*G + e:
 *   s_n = q[r,h,:] . K_view(f, n),  n < flat_kv_lens[f], where K_view(f, n) is token n%128
 *   of virtual page flat_page_table[f, n/128]; o[r,h,:] = softmax(s) . V_view; lse[r,h].
 *
 *   q        [R, Hq, D] bf16 (R = B*N query rows)
 *   k_cache, v_cache [num_pages, 128, Hkv, D] bf16
 *   flat_page_table [R*Hkv, topk] int32; flat_kv_lens [R*Hkv] int32, each in [1, topk*128]
 *   o        [R, Hq, D] bf16 (out); lse [R, Hq] fp32 (out, may be NULL)
 *   workspace >= msa_paged_sparse_decode_workspace_size(R, Hq, Hkv, topk) bytes
 *             (one partial slot per selected page; no zero-fill needed)
 * With few flattened rows (4 * R * Hkv <= the device's SM count, e.g. a small batch at long
 * context) each row is computed by one cluster of 4 CTAs whose partials are merged in
 * distributed shared memory; the workspace is then not touched.
 * The result depends only on the inputs (no run-to-run variation).
 * ------------------------------------------------------------------------------------ */
MSA_API size_t msa_paged_sparse_decode_workspace_size(int32_t R, int32_t Hq, int32_t Hkv, int32_t topk);

MSA_API int msa_paged_sparse_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                            const int32_t* flat_page_table, const int32_t* flat_kv_lens,
                            int32_t R, int32_t Hq, int32_t Hkv, int32_t D, int32_t topk,
                            int64_t num_pages, uint16_t* o, float* lse, void* workspace,
                            size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * KV-block-major sparse prefill with a Log-Sum-Exp merge.
 *
 * Passages: Together AI MiniMax-M3 serving article, section "KV-block-major sparse
 * attention reduces redundant KV movement" (the work mapping {q, kv block} becomes
 * {kv block, q}: the KV block is the outer loop, loaded once and used for every query
 * token that chose it; each block yields a partial O and a Log-Sum-Exp reduction rescales
 * and sums the partials); Japanese translation, section "KV-block-major sparse attention".
 *
 * Queries t = 0..T-1 sit at positions q_start + t with q_start = S_kv - T. For head h of
 * group g, query t attends to keys pos <= q_start + t in the blocks block_ids[t, g, :]
 * (-1 entries ignored). Steps, all on the GPU: (a) invert the selections into per-(group,
 * block) query lists, (b) block-major attention writing one partial (O, lse) per
 * (query, group, slot), (c) merge the partials of each (query, head). With G = Hq/Hkv of 8
 * or 16, the queries of each 128-query span are first ranked by how many of their blocks at
 * least half of the span chose, and consecutive ranks form pairs of 128/G-query tiles; the
 * blocks that at least half of a pair chose are taken out and computed query-major (one
 * partial per (query, head) for all of them); (a)-(b) run on the remaining selections and
 * (c) merges both. Every selection is computed exactly once.
 *
 *   q     [T, Hq, D] bf16; k, v [S_kv, Hkv, D] bf16 (contiguous K/V of the sequence)
 *   block_ids [T, Hkv, topk] int32, each id -1 or a causal block of its query
 *   o     [T, Hq, D] bf16 (out); lse [T, Hq] fp32 (out, may be NULL)
 *   workspace >= msa_sparse_prefill_workspace_size(T, S_kv, Hq, Hkv, topk) bytes
 *             (no zero-fill needed)
 * ------------------------------------------------------------------------------------ */
MSA_API size_t msa_sparse_prefill_workspace_size(int32_t T, int64_t S_kv, int32_t Hq, int32_t Hkv,
                                         int32_t topk);

MSA_API int msa_sparse_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const int32_t* block_ids, int32_t T, int64_t S_kv, int32_t Hq,
                       int32_t Hkv, int32_t D, int32_t topk, uint16_t* o, float* lse,
                       void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * msa_sparse_prefill over a paged K/V cache: a prefill chunk against a prefix that is
 * already in the paged cache (chunked prefill), the K/V of every block read through the
 * page table as in the paged decode.
 *
 * Passages: as msa_sparse_prefill; the paged cache and its page table as in
 * msa_paged_sparse_decode (Together AI MiniMax-M3 serving article, section "MSA needs a new
 * paged-attention integration").
 *
 *   k_cache, v_cache [num_pages, 128, Hkv, D] bf16
 *   page_table [ceil(S_kv/128)] int32: the page holding tokens 128*j .. 128*j+127 of the
 *              sequence; each in [0, num_pages) (an out-of-range page is read as page 0 and
 *              recorded in the device error word); num_pages*128 <= 2^31-1
 *   everything else, the result and the workspace as msa_sparse_prefill.
 * Returns MSA_ERR_ARG for a null page table.
 * ------------------------------------------------------------------------------------ */
MSA_API int msa_sparse_prefill_paged(const uint16_t* q, const uint16_t* k_cache,
                                     const uint16_t* v_cache, const int32_t* page_table,
                                     int64_t num_pages, const int32_t* block_ids, int32_t T,
                                     int64_t S_kv, int32_t Hq, int32_t Hkv, int32_t D,
                                     int32_t topk, uint16_t* o, float* lse, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Step (a) of msa_sparse_prefill on its own: invert the selections.
 *
 * Passage: as msa_sparse_prefill ({q, kv block} -> {kv block, q}).
 * For each group g and block j < nblk, the list of entries t*topk + i with
 * block_ids[t, g, i] == j. offsets[g*(nblk+1) + j] is the start of list (g, j) inside
 * group g's segment and offsets[g*(nblk+1) + nblk] the group total; group g's segment of
 * `entries` starts at the sum of the earlier groups' totals. The order inside one list is
 * unspecified (the attention results do not depend on it).
 *
 *   block_ids [T, Hkv, topk] int32; offsets [Hkv, nblk+1] int32 (out);
 *   entries   [T*Hkv*topk] int32 (out; only the first sum-of-totals entries are written)
 *   workspace >= msa_prefill_bucket_workspace_size(T, Hkv, topk, nblk) bytes (no zero-fill
 *             needed)
 * ------------------------------------------------------------------------------------ */
MSA_API size_t msa_prefill_bucket_workspace_size(int32_t T, int32_t Hkv, int32_t topk, int32_t nblk);

MSA_API int msa_prefill_bucket(const int32_t* block_ids, int32_t T, int32_t Hkv, int32_t topk,
                       int32_t nblk, int32_t* offsets, int32_t* entries, void* workspace,
                       size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Step (c) of msa_sparse_prefill on its own (the decode finishes its per-page slots with the
 * same merge): merge partial attention outputs with their log-sum-exp weights.
 *
 * Passage: Together AI MiniMax-M3 serving article, section "KV-block-major sparse
 * attention reduces redundant KV movement" (a Log-Sum-Exp based reduction rescales and
 * sums the partial outputs of the selected blocks).
 *
 * For unit u < U and head e < G:  lse = log sum_s exp(lse_parts[u,s,e]);
 *   o[u,e,:] = sum_s exp(lse_parts[u,s,e] - lse) * o_parts[u,s,e,:]; partials whose lse is
 *   -inf carry no weight; a unit with no finite partial gives o = 0, lse = -inf.
 *   o_parts   [U, S, G, D], bf16 when parts_bf16 != 0 else fp32; lse_parts [U, S, G] fp32
 *   o         [U, G, D] bf16 (out); lse [U, G] fp32 (out, may be NULL)
 * With U = T*Hkv and G = Hq/Hkv the output is exactly the [T, Hq, D] layout.
 * ------------------------------------------------------------------------------------ */
MSA_API int msa_lse_merge(const void* o_parts, int32_t parts_bf16, const float* lse_parts, int64_t U,
                  int32_t S, int32_t G, int32_t D, uint16_t* o, float* lse, void* stream);

/* ------------------------------------------------------------------------------------
 * Stage 1 without a caller workspace.
 *
 * The pages have no counterpart to this call: it exists for callers that cannot provide
 * device scratch memory. Examples are a plugin inside a host framework that owns all
 * device memory and gives its plugins no allocator, or a decode loop that must not call
 * cudaMalloc because the allocation would synchronise the device and stall the stream.
 *
 * Same arguments, results and errors as msa_index_score_topk, minus the workspace. The
 * scratch is a fixed array of MSA_NOALLOC_SCRATCH_BYTES (8 MiB) of device memory inside the
 * library. Every GPU on which the library is loaded holds this array until the process
 * exits. The call allocates nothing (no cudaMalloc, no cudaFree, no allocating library
 * routine).
 *  - Limit: the call needs msa_index_score_topk_workspace_size(B, N, Hkv, max_blocks)
 *    <= MSA_NOALLOC_SCRATCH_BYTES, i.e. about B*N*Hkv*max_blocks <= 2 million block
 *    scores. Larger calls return MSA_ERR_UNSUPPORTED before anything is queued.
 *  - Set-up: the first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current and caches it; every later call whose
 *    stream is not being captured looks it up again, so that a device reset (which unloads
 *    the module; the array may move when it is loaded again) leaves no stale address behind.
 *    Make the first call on each device, and the first call after a device reset, before
 *    any stream capture begins.
 *  - Sharing: every call on a device uses the same array, which keeps the previous call's
 *    contents. Each call clears the counters it needs at zero (an asynchronous memset on
 *    `stream`). Calls whose execution may overlap on the GPU (different streams, no
 *    ordering between them) race on the array and give undefined results. Order such
 *    calls, or give each of them a workspace through msa_index_score_topk.
 * ------------------------------------------------------------------------------------ */
#define MSA_NOALLOC_SCRATCH_BYTES (8u << 20)

MSA_API int msa_index_score_topk_noalloc(const uint16_t* q_idx, const uint16_t* k_idx_pages,
                                         const int32_t* page_table, const int32_t* seq_lens,
                                         int32_t B, int32_t N, int32_t Hkv, int32_t Di,
                                         int32_t max_blocks, int64_t num_pages, int32_t topk,
                                         int32_t* block_ids, float* scores, void* stream);

/* ------------------------------------------------------------------------------------
 * Diagnostics.
 * ------------------------------------------------------------------------------------ */
/* Thread-local message of the last failing call on this host thread ("" if none). */
MSA_API const char* msa_last_error(void);

/* Synchronises the current device, returns the device error word recorded by the kernels
 * (0 = none; bit 0 = out-of-range page id, bit 1 = out-of-range block id, bit 2 = a bounded
 * wait timed out) in *word (host pointer) and clears it. Returns MSA_OK, or MSA_ERR_DEVICE
 * when the word was non-zero, or MSA_ERR_CUDA. Not for the hot path. */
MSA_API int msa_device_error(uint32_t* word);

/* Library version as "major.minor.patch" (host string, static storage). */
MSA_API const char* msa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MSA_GB300_H */
