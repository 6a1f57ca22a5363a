/*
 * sparse_mla_oracle.c -- CPU fp64 oracle for the sparse MLA attention forward (DSA top-k).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the reference that the CUDA path is checked
 * against.  Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
 * load it; the product path never does.  It shares no code, header or table with the CUDA
 * path.
 *
 * What it computes is the plain definition of the masked sparse softmax attention that the
 * pages describe, written out directly in double precision:
 *
 *   FlashMLA PR #196, "Problem" / "Fix": each query row attends to its own list of top-k
 *     KV indices into one shared latent KV (h_kv = 1); an index is valid iff
 *     0 <= idx < s_kv; invalid entries may sit anywhere in the row and are masked.
 *   FlashMLA PR #196, "Correctness notes": a row with no valid index gives O = 0,
 *     lse = +inf, max_logits = -inf.
 *   FlashMLA PR #216, "Summary": an optional per-row topk_length bounds the row; only slots
 *     below it take part, and the tail beyond it is never used for addressing.
 *   FlashMLA PR #198, "Summary" item 2: the per-head attention sink is a value-less virtual
 *     key folded into the softmax denominator.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - K = kv[:, :d_qk] and V = kv[:, :d_v] come from the same row (h_kv = 1 latent KV).
 *   - logits are sm_scale * q.k; max_logits is the max of those scaled logits (natural units).
 *   - lse is the natural-log log-sum-exp of the scaled logits over the valid slots; the sink
 *     is NOT included in lse or max_logits, only in O's denominator.
 *   - the sink is a logit in the same units as the scaled logits (not multiplied by sm_scale).
 *   - topk_length is clamped to [0, topk]; indices are slots, so a duplicated index counts
 *     twice.
 *
 * Inputs q / kv are bf16 bit patterns (uint16); every bf16 value is exact in double.
 * Build: gcc -O2 -fopenmp -shared -fPIC (no fast-math: plain IEEE double arithmetic).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof(f));
  return (double)f;
}

/* Effective length of a row: topk_length clamped to [0, topk] when given, else topk
 * (FlashMLA PR #216, "Summary"). */
static int64_t row_length(const int32_t* topk_length, int64_t t, int topk) {
  if (!topk_length) return topk;
  int64_t L = topk_length[t];
  if (L < 0) L = 0;
  if (L > topk) L = topk;
  return L;
}

/* One query row t, all heads.  `kv_row_of(j)` resolves slot j to a kv row pointer or NULL
 * when the slot is invalid.  Scratch `logit` and `w` hold topk doubles. */
typedef const uint16_t* (*kv_resolver)(const void* ctx, int64_t t, int32_t idx);

static void attend_row(const uint16_t* q_row /* [h_q, d_qk] */, const int32_t* idx_row /* [topk] */,
                       int64_t L, kv_resolver resolve, const void* ctx, int64_t t,
                       const float* attn_sink, double sm_scale, int h_q, int d_qk, int d_v,
                       double* out_row /* [h_q, d_v] */, double* lse_row, double* max_row,
                       const uint16_t** rows_buf, double* logit, double* w) {
  /* gather the valid slots of [0, L) */
  int64_t n = 0;
  for (int64_t j = 0; j < L; ++j) {
    const uint16_t* r = resolve(ctx, t, idx_row[j]);
    if (r) rows_buf[n++] = r;
  }
  for (int h = 0; h < h_q; ++h) {
    double* o = out_row + (int64_t)h * d_v;
    if (n == 0) {
      /* FlashMLA PR #196, "Correctness notes": empty row -> 0 / +inf / -inf, with or
       * without a sink. */
      for (int d = 0; d < d_v; ++d) o[d] = 0.0;
      lse_row[h] = INFINITY;
      max_row[h] = -INFINITY;
      continue;
    }
    const uint16_t* qh = q_row + (int64_t)h * d_qk;
    double m = -INFINITY;
    for (int64_t s = 0; s < n; ++s) {
      double dot = 0.0;
      for (int d = 0; d < d_qk; ++d) dot += bf16_to_double(qh[d]) * bf16_to_double(rows_buf[s][d]);
      logit[s] = sm_scale * dot;
      if (logit[s] > m) m = logit[s];
    }
    double se = 0.0;
    for (int64_t s = 0; s < n; ++s) {
      w[s] = exp(logit[s] - m);
      se += w[s];
    }
    double den = se;
    if (attn_sink) den += exp((double)attn_sink[h] - m); /* value-less virtual key */
    for (int d = 0; d < d_v; ++d) {
      double acc = 0.0;
      for (int64_t s = 0; s < n; ++s) acc += w[s] * bf16_to_double(rows_buf[s][d]);
      o[d] = acc / den;
    }
    lse_row[h] = m + log(se);
    max_row[h] = m;
  }
}

/* ------------------------------------------------------------------ flat (one shared KV) */
typedef struct {
  const uint16_t* kv;
  int64_t s_kv;
  int d_qk;
} flat_ctx;

static const uint16_t* flat_resolve(const void* vctx, int64_t t, int32_t idx) {
  const flat_ctx* c = (const flat_ctx*)vctx;
  (void)t;
  if (idx < 0 || (int64_t)idx >= c->s_kv) return NULL; /* validity predicate 0 <= idx < s_kv */
  return c->kv + (int64_t)idx * c->d_qk;
}

/* ------------------------------------------------------------------ paged KV cache */
typedef struct {
  const uint16_t* kv_pool;      /* [pool_rows, d_qk] */
  const int32_t* block_table;   /* [n_req, max_blocks] */
  const int32_t* seqlens_k;     /* [n_req] or NULL */
  int64_t s_kv_per_req, pool_rows;
  int max_blocks, page_block, s_q_per_req, d_qk;
} paged_ctx;

/* Token position idx of the request that query row t belongs to, resolved to its pool row
 * (FlashMLA PR #216, "Summary": indices are token positions of the request, and a position
 * that is not valid is never used as an address).  Reading of the paged layout: a position
 * counts only if it lies in the request (0 <= idx < its length), its page lies inside the
 * request's block-table row, the table entry is a page (not negative), and the resulting row
 * lies inside the pool.  Anything else is an invalid slot, like -1 in the flat form. */
static const uint16_t* paged_resolve(const void* vctx, int64_t t, int32_t idx) {
  const paged_ctx* c = (const paged_ctx*)vctx;
  int64_t b = t / c->s_q_per_req;
  int64_t len = c->seqlens_k ? (int64_t)c->seqlens_k[b] : c->s_kv_per_req;
  if (idx < 0 || (int64_t)idx >= len) return NULL; /* token position must lie in the request */
  int64_t blk = idx / c->page_block;
  if (blk >= c->max_blocks) return NULL;           /* page beyond the request's table row */
  int64_t page = c->block_table[b * c->max_blocks + blk];
  if (page < 0) return NULL;                       /* unmapped page */
  int64_t row = page * c->page_block + idx % c->page_block;
  if (row >= c->pool_rows) return NULL;            /* row off the end of the pool */
  return c->kv_pool + row * c->d_qk;
}

static int run_rows(const uint16_t* q, const int32_t* indices, const int32_t* topk_length,
                    const float* attn_sink, double sm_scale, int64_t s_q, int h_q, int d_qk,
                    int d_v, int topk, const int64_t* rows, int64_t n_rows, double* out,
                    double* lse, double* max_logits, int n_threads, kv_resolver resolve,
                    const void* ctx) {
  if (!rows) n_rows = s_q;
  int bad = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif
#pragma omp parallel
  {
    const uint16_t** rows_buf = (const uint16_t**)malloc(sizeof(void*) * (size_t)(topk > 0 ? topk : 1));
    double* logit = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1));
    double* w = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1));
    if (!rows_buf || !logit || !w) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t i = 0; i < n_rows; ++i) {
        int64_t t = rows ? rows[i] : i;
        if (t < 0 || t >= s_q) {
#pragma omp atomic write
          bad = 1;
          continue;
        }
        int64_t L = row_length(topk_length, t, topk);
        attend_row(q + t * (int64_t)h_q * d_qk, indices + t * (int64_t)topk, L, resolve, ctx, t,
                   attn_sink, sm_scale, h_q, d_qk, d_v, out + i * (int64_t)h_q * d_v,
                   lse + i * (int64_t)h_q, max_logits + i * (int64_t)h_q, rows_buf, logit, w);
      }
    }
    free(rows_buf);
    free(logit);
    free(w);
  }
  return bad ? -1 : 0;
}

/* Sparse MLA forward over one shared latent KV [s_kv, 1, d_qk].
 * q [s_q, h_q, d_qk] bf16, indices [s_q, 1, topk] int32, topk_length [s_q] or NULL,
 * attn_sink [h_q] fp32 or NULL.  Outputs (double) are written for the rows listed in `rows`
 * (n_rows of them, in that order), or for every row when `rows` is NULL:
 * out [n_rows, h_q, d_v], lse / max_logits [n_rows, h_q].  Returns 0, or -1 on a bad row id
 * or allocation failure. */
int smla_oracle_fwd(const uint16_t* q, const uint16_t* kv, const int32_t* indices,
                    const int32_t* topk_length, const float* attn_sink, double sm_scale,
                    int64_t s_q, int64_t s_kv, int h_q, int d_qk, int d_v, int topk,
                    const int64_t* rows, int64_t n_rows, double* out, double* lse,
                    double* max_logits, int n_threads) {
  flat_ctx ctx = {kv, s_kv, d_qk};
  return run_rows(q, indices, topk_length, attn_sink, sm_scale, s_q, h_q, d_qk, d_v, topk, rows,
                  n_rows, out, lse, max_logits, n_threads, flat_resolve, &ctx);
}

/* Same forward over a paged KV cache (FlashMLA PR #216, "Summary": indices are token
 * positions of the request; the cache is stored in pages of `page_block` tokens).  Query row
 * t belongs to request t / s_q_per_req; token position p of request b lives in pool row
 * block_table[b][p / page_block] * page_block + p % page_block of the pool's pool_rows rows.
 * Position p is valid iff 0 <= p < seqlens_k[b] (or s_kv_per_req when seqlens_k is NULL),
 * p / page_block < max_blocks, the table entry is >= 0 and the row is < pool_rows. */
int smla_oracle_fwd_paged(const uint16_t* q, const uint16_t* kv_pool, int64_t pool_rows,
                          const int32_t* block_table,
                          const int32_t* seqlens_k, int64_t s_kv_per_req, int max_blocks,
                          int page_block, int s_q_per_req, const int32_t* indices,
                          const int32_t* topk_length, const float* attn_sink, double sm_scale,
                          int64_t s_q, int h_q, int d_qk, int d_v, int topk, const int64_t* rows,
                          int64_t n_rows, double* out, double* lse, double* max_logits,
                          int n_threads) {
  if (page_block <= 0 || s_q_per_req <= 0 || max_blocks <= 0 || pool_rows < 0) return -1;
  paged_ctx ctx = {kv_pool, block_table, seqlens_k, s_kv_per_req, pool_rows, max_blocks,
                   page_block, s_q_per_req, d_qk};
  return run_rows(q, indices, topk_length, attn_sink, sm_scale, s_q, h_q, d_qk, d_v, topk, rows,
                  n_rows, out, lse, max_logits, n_threads, paged_resolve, &ctx);
}

/* Length a row would need so that every valid slot lies below it: one past the last slot j
 * with 0 <= idx[j] < s_kv, 0 when the row has none (FlashMLA PR #196, "Fix": the value a
 * tail scan for the last valid entry yields, used as topk_length). */
void smla_oracle_last_valid_length(const int32_t* indices, int64_t s_q, int topk, int64_t s_kv,
                                   int32_t* out) {
  for (int64_t t = 0; t < s_q; ++t) {
    int32_t L = 0;
    for (int j = topk - 1; j >= 0; --j) {
      int32_t v = indices[t * (int64_t)topk + j];
      if (v >= 0 && (int64_t)v < s_kv) {
        L = j + 1;
        break;
      }
    }
    out[t] = L;
  }
}
