/*
 * MSA CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct host implementation of MiniMax Sparse Attention (MSA)
 * for one attention layer. Only the test suite, the smoke check and the benchmark's CPU
 * baseline leg may call it; the CUDA library never links, includes or calls anything here,
 * and this file includes nothing from the CUDA library.
 *
 * Sources (web pages, cited by title and section):
 *   [Together-M3]  "Serving MiniMax-M3 on Together AI: sparse attention, paged decode and
 *                   multimodal inference" (ai-pulse-lab.com, Chinese), sections
 *                   "MiniMax Sparse Attention changes the serving problem",
 *                   "KV-block-major sparse attention reduces redundant KV movement",
 *                   "MSA needs a new paged-attention integration",
 *                   "The index scorer becomes the decode critical path".
 *   [Together-JP]  "Serving MiniMax-M3 for efficient inference" (news.ainew.jp, Japanese),
 *                   sections "KV-block-major sparse attention", "Integrating MSA with paged
 *                   attention", "Decode Index Scoring Kernel Optimization".
 *   [SGLang-M3.1]  "SGLang and Miles Add Day-0 Support for MiniMax M3.1 Flash",
 *                   section "Miles Day-0 Support" (16 blocks of 128 per KV head).
 *
 * Conventions where the pages are silent (each reading is listed in the design notes):
 *   - block = page = 128 tokens; query head h belongs to KV group g = h / (Hq/Hkv);
 *   - one index head per KV group; positions are 0-based; a query at position t sees
 *     keys 0..t; its local block is t/128; block 0 is the sink;
 *   - block score = max over the block's valid tokens of the bf16 x bf16 dot product,
 *     accumulated in fp32 in index order (the scorer's precision is bf16 products);
 *   - top-k: sink and local block forced; the rest by (score desc, block id asc);
 *     ids emitted ascending, padded with -1;
 *   - attention arithmetic in fp64; q is pre-scaled (no softmax scale); LSE natural log.
 *
 * Data types: bf16 values travel as uint16_t bit patterns; every routine is reentrant
 * and works on caller-owned host memory. Row-parallel routines split their independent
 * output rows across POSIX threads; each output element is computed by one thread with
 * the same sequential arithmetic regardless of the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define MSA_BLOCK 128

/* ---------------------------------------------------------------- bf16 helpers */

static float bf16_to_f32(uint16_t x) {
  uint32_t u = (uint32_t)x << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round a double to the nearest bf16 (ties to even), directly from the double value:
 * write x = m * 2^e with 0.5 <= |m| < 1, keep 8 significant bits with nearbyint()
 * (round-half-even in the default rounding mode), rebuild the value, and read its
 * upper 16 bits as a float (the rebuilt value is exact in float). One rounding only. */
uint16_t oracle_round_bf16(double x) {
  if (isnan(x)) return 0x7fc0;
  if (isinf(x)) return x > 0 ? 0x7f80 : 0xff80;
  if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
  double y;
  if (fabs(x) < ldexp(1.0, -126)) {
    /* bf16 subnormal range: fixed quantum 2^-133 */
    y = ldexp(nearbyint(ldexp(x, 133)), -133);
  } else {
    int e;
    double m = frexp(x, &e);
    y = ldexp(nearbyint(ldexp(m, 8)), e - 8);
  }
  if (fabs(y) >= ldexp(1.0, 128)) return x > 0 ? 0x7f80 : 0xff80;
  float f = (float)y; /* exact */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

void oracle_round_bf16_array(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16(x[i]);
}

/* ---------------------------------------------------------------- threads */

typedef void (*row_fn)(void* ctx, int64_t row);
typedef struct {
  row_fn fn;
  void* ctx;
  int64_t n;
  int tid, nthreads;
} worker_arg;

static void* worker(void* p) {
  worker_arg* a = (worker_arg*)p;
  for (int64_t i = a->tid; i < a->n; i += a->nthreads) a->fn(a->ctx, i);
  return NULL;
}

static void parallel_rows(int64_t n, int nthreads, row_fn fn, void* ctx) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
  pthread_t th[256];
  worker_arg args[256];
  for (int i = 0; i < nthreads; ++i) {
    args[i].fn = fn; args[i].ctx = ctx; args[i].n = n;
    args[i].tid = i; args[i].nthreads = nthreads;
  }
  for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, &args[i]);
  worker(&args[0]);
  for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
}

/* ---------------------------------------------------------------- stage 1: block scores
 *
 * [Together-M3] "The index scorer becomes the decode critical path": each decode query's
 * query-side index vector is compared with the key-side index vectors of every candidate
 * block; each 128-token block is compressed to one score. [Together-JP] "Decode Index
 * Scoring Kernel Optimization": dot products in bfloat16, one score per page; every
 * request and KV group has its own candidate range and mask.
 *
 * Query rows: request b holds N query rows r = b*N + i (i = 0..N-1) at positions
 * q_pos = seq_lens[b] - N + i (the last N tokens of the request, already in the cache).
 * Inputs:
 *   q_idx        [B*N, Hkv, Di] bf16
 *   k_idx_pages  [num_pages, 128, Hkv, Di] bf16; token (b, pos) of group g lives at
 *                page page_table[b, pos/128], slot pos%128
 *   page_table   [B, max_blocks] int32
 * Output, for each listed row: scores[row_slot, g, j] for j < max_blocks:
 *   max over tokens pos = 128*j + tau (tau < 128, pos <= q_pos) of
 *   sum_d q_idx[r,g,d] * k_idx[page, tau, g, d] (fp32, d ascending); -inf when the block
 *   has no valid token (j > q_pos/128).
 */
typedef struct {
  const uint16_t *q_idx, *k_idx;
  const int32_t *page_table, *seq_lens;
  int N, Hkv, Di, max_blocks;
  const int64_t* rows;
  float* scores;
} score_ctx;

/* One work item = one (listed row, group): item = slot*Hkv + g, so that a few long rows
 * (decode: one row per request) still spread over every host thread. */
static void score_row(void* p, int64_t item) {
  score_ctx* c = (score_ctx*)p;
  int64_t slot = item / c->Hkv;
  int g = (int)(item % c->Hkv);
  int64_t r = c->rows ? c->rows[slot] : slot;
  int64_t b = r / c->N;
  int64_t i = r % c->N;
  int64_t q_pos = (int64_t)c->seq_lens[b] - c->N + i;
  {
    const uint16_t* q = c->q_idx + (r * c->Hkv + g) * c->Di;
    float* out = c->scores + (slot * c->Hkv + g) * c->max_blocks;
    for (int j = 0; j < c->max_blocks; ++j) {
      float best = -INFINITY;
      if (q_pos >= 0 && (int64_t)j <= q_pos / MSA_BLOCK) {
        int64_t page = c->page_table[b * c->max_blocks + j];
        for (int tau = 0; tau < MSA_BLOCK; ++tau) {
          int64_t pos = (int64_t)j * MSA_BLOCK + tau;
          if (pos > q_pos) break;
          const uint16_t* k = c->k_idx + ((page * MSA_BLOCK + tau) * c->Hkv + g) * c->Di;
          float acc = 0.0f;
          for (int d = 0; d < c->Di; ++d) acc += bf16_to_f32(q[d]) * bf16_to_f32(k[d]);
          if (acc > best) best = acc;
        }
      }
      out[j] = best;
    }
  }
}

int oracle_block_scores(const uint16_t* q_idx, const uint16_t* k_idx_pages,
                        const int32_t* page_table, const int32_t* seq_lens, int B, int N,
                        int Hkv, int Di, int max_blocks, const int64_t* rows, int64_t nrows,
                        float* scores, int nthreads) {
  if (!q_idx || !k_idx_pages || !page_table || !seq_lens || !scores) return -1;
  if (B <= 0 || N <= 0 || Hkv <= 0 || Di <= 0 || max_blocks <= 0) return -1;
  if (!rows) nrows = (int64_t)B * N;
  score_ctx c = {q_idx, k_idx_pages, page_table, seq_lens, N, Hkv, Di, max_blocks, rows, scores};
  parallel_rows(nrows * Hkv, nthreads, score_row, &c);
  return 0;
}

/* ---------------------------------------------------------------- stage 1: top-k
 *
 * [Together-M3] "MiniMax Sparse Attention changes the serving problem": stage one keeps,
 * per KV group, the K most relevant blocks. Readings held fixed: block 0 (sink) and the
 * query's local block q_pos/128 are always kept and count toward k; the remaining
 * k - #forced slots take the other causal blocks (1 .. local-1) by score descending,
 * ties to the lower block id; the kept ids are written ascending, then -1 padding.
 * sel_scores holds each kept block's score (forced ones included), -inf for padding.
 */
typedef struct {
  int id;
  float s;
} cand;

static int cand_cmp(const void* a, const void* b) {
  const cand* x = (const cand*)a;
  const cand* y = (const cand*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->id > y->id) - (x->id < y->id);
}

static int int_cmp(const void* a, const void* b) {
  int x = *(const int*)a, y = *(const int*)b;
  return (x > y) - (x < y);
}

int oracle_topk(const float* scores, const int64_t* q_pos, int64_t nrows, int Hkv,
                int max_blocks, int topk, int32_t* block_ids, float* sel_scores) {
  if (!scores || !q_pos || !block_ids || topk < 2 || max_blocks <= 0) return -1;
  cand* cands = (cand*)malloc(sizeof(cand) * (size_t)max_blocks);
  int* kept = (int*)malloc(sizeof(int) * (size_t)topk);
  if (!cands || !kept) { free(cands); free(kept); return -1; }
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t local = q_pos[r] / MSA_BLOCK;
    for (int g = 0; g < Hkv; ++g) {
      const float* s = scores + (r * Hkv + g) * max_blocks;
      int nk = 0;
      kept[nk++] = 0;
      if (local > 0) kept[nk++] = (int)local;
      int nc = 0;
      for (int j = 1; j < local; ++j) { cands[nc].id = j; cands[nc].s = s[j]; ++nc; }
      qsort(cands, (size_t)nc, sizeof(cand), cand_cmp);
      for (int c = 0; c < nc && nk < topk; ++c) kept[nk++] = cands[c].id;
      qsort(kept, (size_t)nk, sizeof(int), int_cmp);
      int32_t* ids = block_ids + (r * Hkv + g) * topk;
      for (int i = 0; i < topk; ++i) {
        ids[i] = i < nk ? kept[i] : -1;
        if (sel_scores)
          sel_scores[(r * Hkv + g) * topk + i] = i < nk ? s[kept[i]] : -INFINITY;
      }
    }
  }
  free(cands);
  free(kept);
  return 0;
}

/* ---------------------------------------------------------------- sparse page table
 *
 * [Together-M3] "MSA needs a new paged-attention integration": at decode a page table is
 * built from the selected blocks, the KV-group dimension is flattened into the batch, and
 * a strided view of the KV-cache tensor hands each flattened row its own pages: the page
 * address steps by D to pick the virtual page start and tokens step by Hkv*D, which
 * deinterleaves one physical tensor [num_pages, 128, Hkv, D] into per-head pages.
 *
 * Flattened row f = r*Hkv + g (query row r, KV group g). Virtual page of physical page p
 * for group g: v = p*128*Hkv + g, so element (v, tau, d) of the view sits at
 * v*D + tau*Hkv*D + d == ((p*128 + tau)*Hkv + g)*D + d.
 * flat_page_table[f, i] = virtual page of the i-th kept block (ascending), -1 after.
 * flat_kv_lens[f] = tokens visible to the query in the kept blocks: 128 per kept block
 * below the local block plus (q_pos % 128) + 1 for the local block.
 */
int oracle_build_sparse_page_table(const int32_t* block_ids, const int32_t* page_table,
                                   const int32_t* seq_lens, int B, int N, int Hkv, int topk,
                                   int max_blocks, int32_t* flat_page_table,
                                   int32_t* flat_kv_lens) {
  if (!block_ids || !page_table || !seq_lens || !flat_page_table || !flat_kv_lens) return -1;
  for (int64_t r = 0; r < (int64_t)B * N; ++r) {
    int64_t b = r / N;
    int64_t q_pos = (int64_t)seq_lens[b] - N + (r % N);
    int64_t local = q_pos / MSA_BLOCK;
    for (int g = 0; g < Hkv; ++g) {
      int64_t f = r * Hkv + g;
      int64_t len = 0;
      for (int i = 0; i < topk; ++i) {
        int32_t j = block_ids[f * topk + i];
        if (j < 0) { flat_page_table[f * topk + i] = -1; continue; }
        int64_t p = page_table[b * max_blocks + j];
        flat_page_table[f * topk + i] = (int32_t)(p * MSA_BLOCK * Hkv + g);
        len += (j == local) ? (q_pos % MSA_BLOCK) + 1 : MSA_BLOCK;
      }
      flat_kv_lens[f] = (int32_t)len;
    }
  }
  return 0;
}

/* ---------------------------------------------------------------- softmax attention core
 *
 * [Together-M3] "MiniMax Sparse Attention changes the serving problem": stage two runs
 * dense attention between the query tokens and the selected blocks. Given the list of
 * visible key rows, this is ordinary softmax attention: s_n = q . k_n (q pre-scaled),
 * m = max s, l = sum exp(s - m), o = sum exp(s_n - m) v_n / l, lse = m + log l.
 * Two passes in fp64. n == 0 gives o = 0 and lse = -inf.
 */
static void attend(const uint16_t* q, const uint16_t* const* keys, const uint16_t* const* vals,
                   int64_t n, int D, double* s_buf, double* o, double* lse) {
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (n == 0) { *lse = -INFINITY; return; }
  double m = -INFINITY;
  for (int64_t i = 0; i < n; ++i) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += (double)bf16_to_f32(q[d]) * (double)bf16_to_f32(keys[i][d]);
    s_buf[i] = acc;
    if (acc > m) m = acc;
  }
  double l = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    double p = exp(s_buf[i] - m);
    l += p;
    for (int d = 0; d < D; ++d) o[d] += p * (double)bf16_to_f32(vals[i][d]);
  }
  for (int d = 0; d < D; ++d) o[d] /= l;
  *lse = m + log(l);
}

/* ---------------------------------------------------------------- sparse decode (logical)
 *
 * The plain definition of MSA decode attention for query row r = b*N + i and head h:
 * attend over the keys at positions pos (ascending) that lie in the group's kept blocks
 * and satisfy pos <= q_pos, reading K/V through the request's page table
 * (k_cache[page_table[b, pos/128], pos%128, g, :]).
 * units: list of r*Hq + h to compute (NULL = all R*Hq); outputs o[unit_slot, D], lse[unit_slot].
 */
typedef struct {
  const uint16_t *q, *k, *v;
  const int32_t *page_table, *seq_lens, *block_ids;
  int N, Hq, Hkv, D, topk, max_blocks;
  const int64_t* units;
  double *o, *lse;
} dec_ctx;

static void dec_unit(void* p, int64_t slot) {
  dec_ctx* c = (dec_ctx*)p;
  int64_t u = c->units ? c->units[slot] : slot;
  int64_t r = u / c->Hq;
  int h = (int)(u % c->Hq);
  int g = h / (c->Hq / c->Hkv);
  int64_t b = r / c->N;
  int64_t q_pos = (int64_t)c->seq_lens[b] - c->N + (r % c->N);
  int64_t cap = (int64_t)c->topk * MSA_BLOCK;
  const uint16_t** keys = (const uint16_t**)malloc(sizeof(void*) * (size_t)cap);
  const uint16_t** vals = (const uint16_t**)malloc(sizeof(void*) * (size_t)cap);
  double* s_buf = (double*)malloc(sizeof(double) * (size_t)cap);
  int64_t n = 0;
  const int32_t* ids = c->block_ids + (r * c->Hkv + g) * c->topk;
  for (int i = 0; i < c->topk; ++i) {
    int32_t j = ids[i];
    if (j < 0) continue;
    int64_t page = c->page_table[b * c->max_blocks + j];
    for (int tau = 0; tau < MSA_BLOCK; ++tau) {
      int64_t pos = (int64_t)j * MSA_BLOCK + tau;
      if (pos > q_pos) break;
      int64_t off = ((page * MSA_BLOCK + tau) * c->Hkv + g) * c->D;
      keys[n] = c->k + off;
      vals[n] = c->v + off;
      ++n;
    }
  }
  attend(c->q + u * c->D, keys, vals, n, c->D, s_buf, c->o + slot * c->D, c->lse + slot);
  free(keys); free(vals); free(s_buf);
}

int oracle_sparse_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                         const int32_t* page_table, const int32_t* seq_lens,
                         const int32_t* block_ids, int B, int N, int Hq, int Hkv, int D,
                         int topk, int max_blocks, const int64_t* units, int64_t nunits,
                         double* o, double* lse, int nthreads) {
  if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !block_ids || !o || !lse) return -1;
  if (Hkv <= 0 || Hq % Hkv != 0) return -1;
  if (!units) nunits = (int64_t)B * N * Hq;
  dec_ctx c = {q, k_cache, v_cache, page_table, seq_lens, block_ids, N, Hq, Hkv, D, topk,
               max_blocks, units, o, lse};
  parallel_rows(nunits, nthreads, dec_unit, &c);
  return 0;
}

/* ---------------------------------------------------------------- paged decode through the
 * strided view
 *
 * The same attention read the way the pages describe the paged kernel's input: flattened
 * row f = r*Hkv + g has its own page table; its n-th visible token is slot n%128 of
 * virtual page flat_page_table[f, n/128], whose elements sit at v*D + tau*Hkv*D + d of
 * the cache viewed as a flat array.
 * q [R, Hq, D] (head h of row r is row f = r*Hkv + h/G, member h%G), units as above.
 */
typedef struct {
  const uint16_t *q, *k, *v;
  const int32_t *fpt, *lens;
  int Hq, Hkv, D, topk;
  const int64_t* units;
  double *o, *lse;
} flat_ctx;

static void flat_unit(void* p, int64_t slot) {
  flat_ctx* c = (flat_ctx*)p;
  int64_t u = c->units ? c->units[slot] : slot;
  int64_t r = u / c->Hq;
  int h = (int)(u % c->Hq);
  int64_t f = r * c->Hkv + h / (c->Hq / c->Hkv);
  int64_t n = c->lens[f];
  const uint16_t** keys = (const uint16_t**)malloc(sizeof(void*) * (size_t)(n > 0 ? n : 1));
  const uint16_t** vals = (const uint16_t**)malloc(sizeof(void*) * (size_t)(n > 0 ? n : 1));
  double* s_buf = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  for (int64_t t = 0; t < n; ++t) {
    int64_t vpage = c->fpt[f * c->topk + t / MSA_BLOCK];
    int64_t off = vpage * c->D + (t % MSA_BLOCK) * (int64_t)c->Hkv * c->D;
    keys[t] = c->k + off;
    vals[t] = c->v + off;
  }
  attend(c->q + u * c->D, keys, vals, n, c->D, s_buf, c->o + slot * c->D, c->lse + slot);
  free(keys); free(vals); free(s_buf);
}

int oracle_paged_decode_flat(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                             const int32_t* flat_page_table, const int32_t* flat_kv_lens,
                             int64_t R, int Hq, int Hkv, int D, int topk, const int64_t* units,
                             int64_t nunits, double* o, double* lse, int nthreads) {
  if (!q || !k_cache || !v_cache || !flat_page_table || !flat_kv_lens || !o || !lse) return -1;
  if (Hkv <= 0 || Hq % Hkv != 0) return -1;
  if (!units) nunits = R * Hq;
  flat_ctx c = {q, k_cache, v_cache, flat_page_table, flat_kv_lens, Hq, Hkv, D, topk, units, o, lse};
  parallel_rows(nunits, nthreads, flat_unit, &c);
  return 0;
}

/* ---------------------------------------------------------------- sparse prefill
 *
 * [Together-M3] "KV-block-major sparse attention reduces redundant KV movement": in
 * prefill each query token attends densely to its group's selected blocks. The plain
 * definition, for query t (position q_start + t, q_start = S_kv - T) and head h of group
 * g: attend over the keys pos in the kept blocks (ascending) with pos <= q_start + t,
 * from contiguous k, v [S_kv, Hkv, D].
 * units: list of t*Hq + h (NULL = all T*Hq).
 */
typedef struct {
  const uint16_t *q, *k, *v;
  const int32_t* block_ids;
  int64_t T, S;
  int Hq, Hkv, D, topk;
  const int64_t* units;
  double *o, *lse;
} pre_ctx;

static void pre_unit(void* p, int64_t slot) {
  pre_ctx* c = (pre_ctx*)p;
  int64_t u = c->units ? c->units[slot] : slot;
  int64_t t = u / c->Hq;
  int h = (int)(u % c->Hq);
  int g = h / (c->Hq / c->Hkv);
  int64_t q_pos = c->S - c->T + t;
  int64_t cap = (int64_t)c->topk * MSA_BLOCK;
  const uint16_t** keys = (const uint16_t**)malloc(sizeof(void*) * (size_t)cap);
  const uint16_t** vals = (const uint16_t**)malloc(sizeof(void*) * (size_t)cap);
  double* s_buf = (double*)malloc(sizeof(double) * (size_t)cap);
  int64_t n = 0;
  const int32_t* ids = c->block_ids + (t * c->Hkv + g) * c->topk;
  for (int i = 0; i < c->topk; ++i) {
    int32_t j = ids[i];
    if (j < 0) continue;
    for (int tau = 0; tau < MSA_BLOCK; ++tau) {
      int64_t pos = (int64_t)j * MSA_BLOCK + tau;
      if (pos > q_pos || pos >= c->S) break;
      int64_t off = (pos * c->Hkv + g) * c->D;
      keys[n] = c->k + off;
      vals[n] = c->v + off;
      ++n;
    }
  }
  attend(c->q + u * c->D, keys, vals, n, c->D, s_buf, c->o + slot * c->D, c->lse + slot);
  free(keys); free(vals); free(s_buf);
}

int oracle_sparse_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const int32_t* block_ids, int64_t T, int64_t S_kv, int Hq, int Hkv,
                          int D, int topk, const int64_t* units, int64_t nunits, double* o,
                          double* lse, int nthreads) {
  if (!q || !k || !v || !block_ids || !o || !lse) return -1;
  if (Hkv <= 0 || Hq % Hkv != 0 || T > S_kv) return -1;
  if (!units) nunits = T * Hq;
  pre_ctx c = {q, k, v, block_ids, T, S_kv, Hq, Hkv, D, topk, units, o, lse};
  parallel_rows(nunits, nthreads, pre_unit, &c);
  return 0;
}

/* ---------------------------------------------------------------- block-major partials and
 * the Log-Sum-Exp merge
 *
 * [Together-M3] "KV-block-major sparse attention reduces redundant KV movement" and
 * [Together-JP] "KV-block-major sparse attention": with the KV block as the outer loop each
 * block yields only a partial output; a Log-Sum-Exp reduction rescales and sums the
 * partials. The procedure itself is missing from the extracted pages, so the textbook
 * definition is used:
 *   partial of block j:  o_j = sum_{n in j} exp(s_n - m_j) v_n / l_j, lse_j = m_j + log l_j
 *   merge:  lse = log sum_j exp(lse_j);  o = sum_j exp(lse_j - lse) o_j
 * Blocks with no visible key have lse_j = -inf and weight 0.
 */
int oracle_prefill_block_partial(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 int64_t T, int64_t S_kv, int Hq, int Hkv, int D, int64_t t,
                                 int h, int32_t block, double* o, double* lse) {
  if (!q || !k || !v || !o || !lse || Hkv <= 0 || Hq % Hkv != 0) return -1;
  int g = h / (Hq / Hkv);
  int64_t q_pos = S_kv - T + t;
  const uint16_t* keys[MSA_BLOCK];
  const uint16_t* vals[MSA_BLOCK];
  double s_buf[MSA_BLOCK];
  int64_t n = 0;
  for (int tau = 0; tau < MSA_BLOCK; ++tau) {
    int64_t pos = (int64_t)block * MSA_BLOCK + tau;
    if (pos > q_pos || pos >= S_kv) break;
    keys[n] = k + (pos * Hkv + g) * D;
    vals[n] = v + (pos * Hkv + g) * D;
    ++n;
  }
  attend(q + (t * Hq + h) * D, keys, vals, n, D, s_buf, o, lse);
  return 0;
}

/* Merge n partials (o_parts [n, D] as float, lse_parts [n] as float) into o[D], lse. */
int oracle_lse_merge(const float* o_parts, const float* lse_parts, int n, int D, double* o,
                     double* lse) {
  if (!o_parts || !lse_parts || !o || !lse || n < 0) return -1;
  double m = -INFINITY;
  for (int i = 0; i < n; ++i) if (lse_parts[i] > m) m = lse_parts[i];
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (n == 0 || m == -INFINITY) { *lse = -INFINITY; return 0; }
  double total = 0.0;
  for (int i = 0; i < n; ++i) total += exp((double)lse_parts[i] - m);
  double out_lse = m + log(total);
  for (int i = 0; i < n; ++i) {
    double w = exp((double)lse_parts[i] - out_lse);
    for (int d = 0; d < D; ++d) o[d] += w * (double)o_parts[(int64_t)i * D + d];
  }
  *lse = out_lse;
  return 0;
}

/* ---------------------------------------------------------------- prefill bucketing
 *
 * [Together-M3] "KV-block-major sparse attention reduces redundant KV movement": the work
 * mapping {q, kv block} becomes {kv block, q}. The inversion of the selection lists: for
 * every KV group g and block j, the (query t, slot i) pairs with block_ids[t, g, i] == j,
 * in increasing (t, i) order. counts[g, j] is the list length; offsets[g*(nblk+1) + j] the
 * exclusive prefix within group g (offsets[g, nblk] = total of group g); entries hold
 * t*topk + i, group g's lists starting at group_base[g] = sum of earlier groups' totals.
 */
int oracle_prefill_buckets(const int32_t* block_ids, int64_t T, int Hkv, int topk, int nblk,
                           int32_t* offsets, int32_t* entries) {
  if (!block_ids || !offsets || !entries || nblk <= 0) return -1;
  int64_t base = 0;
  for (int g = 0; g < Hkv; ++g) {
    int32_t* off = offsets + (int64_t)g * (nblk + 1);
    for (int j = 0; j <= nblk; ++j) off[j] = 0;
    for (int64_t t = 0; t < T; ++t)
      for (int i = 0; i < topk; ++i) {
        int32_t j = block_ids[(t * Hkv + g) * topk + i];
        if (j >= 0 && j < nblk) off[j + 1] += 1;
      }
    for (int j = 0; j < nblk; ++j) off[j + 1] += off[j];
    int64_t* cursor = (int64_t*)calloc((size_t)nblk, sizeof(int64_t));
    if (!cursor) return -1;
    for (int64_t t = 0; t < T; ++t)
      for (int i = 0; i < topk; ++i) {
        int32_t j = block_ids[(t * Hkv + g) * topk + i];
        if (j < 0 || j >= nblk) continue;
        entries[base + off[j] + cursor[j]] = (int32_t)(t * topk + i);
        cursor[j] += 1;
      }
    free(cursor);
    base += off[nblk];
  }
  return 0;
}
