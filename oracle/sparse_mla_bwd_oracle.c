/*
 * sparse_mla_bwd_oracle.c -- CPU fp64 oracle for the sparse MLA attention backward (DSA top-k).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the reference that the CUDA backward is checked
 * against.  Only the test suite and the benchmark's CPU-baseline leg may load it; the product
 * path never does.  It shares no code, header or table with the CUDA path (nor with the
 * forward oracle: it recomputes the forward it differentiates).
 *
 * What it computes: the gradients of  L = sum_{t,h,d} dO[t,h,d] * O[t,h,d]  with respect to
 * q, the shared latent kv and the per-head sink, where O is the sparse MLA forward of FlashMLA
 * PR #196 ("Problem" / "Fix": per-row top-k slots into one kv, invalid slots masked), with the
 * optional row length of PR #216 ("Summary") and the value-less sink of PR #198 ("Summary"
 * item 2).  FlashMLA PR #198 ("Summary" item 1) names this operation: the sparse MLA backward
 * for the absorbed shape, with dK / dV scattered into the shared latent rows and the sink's
 * gradient accumulated from the rowsum of dO * O.
 *
 * For one row t and head h, with the counted slots s (kv row r_s, key k_s = kv[r_s, :d_qk],
 * value v_s = kv[r_s, :d_v]) and logits l_s = sm_scale * <q_h, k_s>:
 *   Z      = sum_s exp(l_s) + [sink] exp(sink_h)          (softmax normaliser, sink included)
 *   p_s    = exp(l_s) / Z,   p_sink = exp(sink_h) / Z
 *   O_h    = sum_s p_s v_s
 *   dP_s   = <dO_h, v_s>,    D = sum_s p_s dP_s  (= <dO_h, O_h>)
 *   dS_s   = p_s (dP_s - D)                                (d L / d l_s)
 *   dq_h          = sm_scale * sum_s dS_s k_s
 *   dkv[r_s, :d_qk] += sm_scale * dS_s q_h                 (through the key)
 *   dkv[r_s, :d_v]  += p_s dO_h                            (through the value)
 *   dsink[h]        += -p_sink * D                         (d L / d sink_h)
 * A row without a counted slot has O = 0 (PR #196, "Correctness notes") and contributes
 * nothing.  Slots are counted, so a duplicated index contributes once per slot.
 *
 * Inputs arrive as doubles (the Python side converts bf16 bit patterns exactly), so the same
 * routine serves finite-difference checks on arbitrary real inputs.
 * Build: gcc -O2 -fopenmp -shared -fPIC (no fast-math: plain IEEE double arithmetic).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Row length: topk_length clamped to [0, topk] when given, else topk (PR #216, "Summary"). */
static int64_t bwd_row_length(const int32_t* topk_length, int64_t t, int topk) {
  if (!topk_length) return topk;
  int64_t len = topk_length[t];
  if (len < 0) len = 0;
  if (len > topk) len = topk;
  return len;
}

/* Gradients for one query row.  `slot_rows` receives the kv row of every counted slot; the
 * row's contributions to dkv go to `contrib` ([n_counted, d_qk], later added into dkv in slot
 * order) and to `dsink_row` ([h_q]). */
static int64_t grad_row(const double* q_row, const double* kv, const double* do_row,
                        const int32_t* idx_row, int64_t len, int64_t s_kv,
                        const float* attn_sink, double sm_scale, int h_q, int d_qk, int d_v,
                        double* dq_row, int64_t* slot_rows, double* contrib, double* dsink_row,
                        double* lg, double* pr, double* dp) {
  int64_t n = 0;
  for (int64_t j = 0; j < len; ++j) {
    int32_t v = idx_row[j];
    if (v >= 0 && (int64_t)v < s_kv) slot_rows[n++] = v; /* validity 0 <= idx < s_kv */
  }
  memset(dq_row, 0, sizeof(double) * (size_t)h_q * (size_t)d_qk);
  memset(contrib, 0, sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)d_qk);
  for (int h = 0; h < h_q; ++h) dsink_row[h] = 0.0;
  if (n == 0) return 0;
  for (int h = 0; h < h_q; ++h) {
    const double* qh = q_row + (int64_t)h * d_qk;
    const double* doh = do_row + (int64_t)h * d_v;
    double top = -INFINITY;
    for (int64_t s = 0; s < n; ++s) {
      const double* ks = kv + slot_rows[s] * d_qk;
      double acc = 0.0;
      for (int d = 0; d < d_qk; ++d) acc += qh[d] * ks[d];
      lg[s] = sm_scale * acc;
      if (lg[s] > top) top = lg[s];
    }
    /* normaliser with the sink as one more (value-less) term, shifted by the largest logit */
    double z = 0.0;
    for (int64_t s = 0; s < n; ++s) z += exp(lg[s] - top);
    double e_sink = attn_sink ? exp((double)attn_sink[h] - top) : 0.0;
    z += e_sink;
    double delta = 0.0;
    for (int64_t s = 0; s < n; ++s) {
      const double* vs = kv + slot_rows[s] * d_qk;
      pr[s] = exp(lg[s] - top) / z;
      double acc = 0.0;
      for (int d = 0; d < d_v; ++d) acc += doh[d] * vs[d];
      dp[s] = acc;
      delta += pr[s] * dp[s];
    }
    double* dqh = dq_row + (int64_t)h * d_qk;
    for (int64_t s = 0; s < n; ++s) {
      const double* ks = kv + slot_rows[s] * d_qk;
      double ds = pr[s] * (dp[s] - delta);
      double* cs = contrib + s * d_qk;
      for (int d = 0; d < d_qk; ++d) {
        dqh[d] += sm_scale * ds * ks[d];
        cs[d] += sm_scale * ds * qh[d];
      }
      for (int d = 0; d < d_v; ++d) cs[d] += pr[s] * doh[d];
    }
    dsink_row[h] = -(e_sink / z) * delta;
  }
  return n;
}

/* Sparse MLA backward over one shared latent kv [s_kv, d_qk].
 * q [s_q, h_q, d_qk], kv [s_kv, d_qk], dout [s_q, h_q, d_v] (doubles), indices [s_q, topk],
 * topk_length [s_q] or NULL, attn_sink [h_q] or NULL.
 * Writes dq [s_q, h_q, d_qk], dkv [s_kv, d_qk] and, when not NULL, dsink [h_q].
 * Returns 0, or -1 on an allocation failure. */
int smla_oracle_bwd(const double* q, const double* kv, const double* dout, const int32_t* indices,
                    const int32_t* topk_length, const float* attn_sink, double sm_scale,
                    int64_t s_q, int64_t s_kv, int h_q, int d_qk, int d_v, int topk, double* dq,
                    double* dkv, double* dsink, int n_threads) {
  int bad = 0;
  memset(dkv, 0, sizeof(double) * (size_t)s_kv * (size_t)d_qk);
  if (dsink)
    for (int h = 0; h < h_q; ++h) dsink[h] = 0.0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif
  /* rows in parallel; each row's kv / sink contributions are added in row order afterwards,
   * chunk by chunk, so the result does not depend on the thread count */
  const size_t width = (size_t)(topk > 0 ? topk : 1);
  /* rows per chunk: at most 64, with the per-chunk contribution buffer under ~256 MB */
  int64_t chunk = (int64_t)(((size_t)256 << 20) / (width * (size_t)(d_qk > 0 ? d_qk : 1) * sizeof(double)));
  if (chunk > 64) chunk = 64;
  if (chunk < 1) chunk = 1;
  int64_t* rows_all = (int64_t*)malloc(sizeof(int64_t) * (size_t)chunk * width);
  int64_t* n_all = (int64_t*)malloc(sizeof(int64_t) * (size_t)chunk);
  double* contrib_all = (double*)malloc(sizeof(double) * (size_t)chunk * width * (size_t)d_qk);
  double* dsink_all = (double*)malloc(sizeof(double) * (size_t)chunk * (size_t)h_q);
  if (!rows_all || !n_all || !contrib_all || !dsink_all) bad = 1;
  for (int64_t t0 = 0; t0 < s_q && !bad; t0 += chunk) {
    const int64_t t1 = t0 + chunk < s_q ? t0 + chunk : s_q;
#pragma omp parallel
    {
      double* lg = (double*)malloc(sizeof(double) * width);
      double* pr = (double*)malloc(sizeof(double) * width);
      double* dp = (double*)malloc(sizeof(double) * width);
      if (!lg || !pr || !dp) {
#pragma omp atomic write
        bad = 1;
      } else {
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = t0; t < t1; ++t) {
          const int64_t i = t - t0;
          n_all[i] = grad_row(q + t * (int64_t)h_q * d_qk, kv, dout + t * (int64_t)h_q * d_v,
                              indices + t * (int64_t)topk, bwd_row_length(topk_length, t, topk),
                              s_kv, attn_sink, sm_scale, h_q, d_qk, d_v,
                              dq + t * (int64_t)h_q * d_qk, rows_all + i * (int64_t)width,
                              contrib_all + i * (int64_t)width * d_qk, dsink_all + i * h_q, lg, pr,
                              dp);
        }
      }
      free(lg);
      free(pr);
      free(dp);
    }
    if (bad) break;
    for (int64_t t = t0; t < t1; ++t) {
      const int64_t i = t - t0;
      for (int64_t s = 0; s < n_all[i]; ++s) {
        double* dst = dkv + rows_all[i * (int64_t)width + s] * d_qk;
        const double* src = contrib_all + (i * (int64_t)width + s) * d_qk;
        for (int d = 0; d < d_qk; ++d) dst[d] += src[d];
      }
      if (dsink)
        for (int h = 0; h < h_q; ++h) dsink[h] += dsink_all[i * h_q + h];
    }
  }
  free(rows_all);
  free(n_all);
  free(contrib_all);
  free(dsink_all);
  return bad ? -1 : 0;
}
