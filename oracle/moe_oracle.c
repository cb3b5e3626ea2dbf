/*
 * MoE layer oracle: a plain, slow, obviously correct fp64 CPU implementation of one MoE layer's
 * expert computation, forward and backward. TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the benchmark's CPU-baseline leg call it; the CUDA library never does, and the two share no
 * code (no headers, helpers, tables or constants).
 *
 * What it follows ("Scalable Pretraining of Large MoE LMs on Aurora"):
 *   - brief, section 核心方法 (FastSparseMoE): per-expert token counting, index generation, and a
 *     grouped GEMM that merges the experts' FFNs;
 *   - summary page, section 关键设计: the experts are matrix multiplications plus an activation;
 *   - brief, sections 为什么值得记录 / 关键结果: forward and backward are both part of the module.
 * The pages leave the router, activation and layouts open; the readings taken here are:
 *   selection  S_t = the k experts with the largest logit, ordered by (logit desc, id asc); -0 == +0
 *   weights    w_{t,e} = exp(L[t,e] - m_t) / sum_{e' in S_t} exp(L[t,e'] - m_t)   (softmax, top-k, renorm)
 *   expert     a = Wg[e] x, b = Wu[e] x, h = silu(a) * b, y = Wd[e] h, silu(z) = z / (1 + exp(-z))
 *   output     out_t = sum_{e in S_t} w_{t,e} y_{t,e}
 *   backward   (S_t held fixed)  dw_{t,e} = <g_t, y_{t,e}>;
 *              dL[t,e] = w_{t,e} (dw_{t,e} - sum_{e' in S_t} w_{t,e'} dw_{t,e'}) on S_t, 0 elsewhere;
 *              dh = w_{t,e} Wd[e]^T g_t; da = dh * b * s(a)(1 + a(1 - s(a))); db = dh * silu(a);
 *              dx_t = sum_e Wg[e]^T da + Wu[e]^T db;
 *              dWg[e] += da x_t^T, dWu[e] += db x_t^T, dWd[e] += (w_{t,e} g_t) h^T.
 *   grouping   counts[e] = #slots routed to e; offsets = exclusive scan of counts; expert e's rows
 *              start at tile_offsets[e] * BM with tile_offsets = exclusive scan of ceil(counts/BM);
 *              within an expert rows follow increasing slot index t*k + j (stable).
 * Every sum runs in fp64 in the plain order of its definition. Inputs are read exactly as stored
 * (bf16 or fp32 widened to fp64). The experts are evaluated per token: no permutation or grouping
 * code is involved in the float results.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1, OR_F64 = 2 };

static double ld(const void *p, size_t i, int dt) {
  if (dt == OR_F32) return (double)((const float *)p)[i];
  if (dt == OR_F64) return ((const double *)p)[i];
  uint32_t u = (uint32_t)((const uint16_t *)p)[i] << 16; /* bf16 -> fp32 is exact */
  float v;
  memcpy(&v, &u, sizeof v);
  return (double)v;
}

static double sigm(double z) { return 1.0 / (1.0 + exp(-z)); }
static double silu(double z) { return z * sigm(z); }

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Top-k selection and renormalised softmax weights for every token. */
int oracle_route_topk(const void *logits, int l_dt, int T, int E, int k, int32_t *idx, double *w) {
  if (T < 0 || E <= 0 || k <= 0 || k > E) return -1;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    char used[1024];
    memset(used, 0, sizeof used);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      double bv = 0.0;
      for (int e = 0; e < E; ++e) {
        if (used[e]) continue;
        double v = ld(logits, (size_t)t * E + e, l_dt);
        if (best < 0 || v > bv) { best = e; bv = v; } /* strict '>' keeps the lower id on ties */
      }
      used[best] = 1;
      idx[(size_t)t * k + j] = best;
    }
    double m = ld(logits, (size_t)t * E + idx[(size_t)t * k], l_dt);
    double s = 0.0;
    for (int j = 0; j < k; ++j) s += exp(ld(logits, (size_t)t * E + idx[(size_t)t * k + j], l_dt) - m);
    for (int j = 0; j < k; ++j)
      w[(size_t)t * k + j] = exp(ld(logits, (size_t)t * E + idx[(size_t)t * k + j], l_dt) - m) / s;
  }
  return 0;
}

/* Token counting and index generation. rows_cap = length of token_of_row (filled with -1 first). */
int oracle_index(const int32_t *idx, int T, int k, int E, int BM, int32_t *counts, int32_t *offsets,
                 int32_t *tile_offsets, int32_t *row_of_slot, int32_t *token_of_row, int64_t rows_cap) {
  if (BM <= 0 || E <= 0) return -1;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t s = 0; s < (int64_t)T * k; ++s) {
    if (idx[s] < 0 || idx[s] >= E) return -2;
    counts[idx[s]] += 1;
  }
  offsets[0] = 0;
  tile_offsets[0] = 0;
  for (int e = 0; e < E; ++e) {
    offsets[e + 1] = offsets[e] + counts[e];
    tile_offsets[e + 1] = tile_offsets[e] + (counts[e] + BM - 1) / BM;
  }
  if ((int64_t)tile_offsets[E] * BM > rows_cap) return -3;
  for (int64_t r = 0; r < rows_cap; ++r) token_of_row[r] = -1;
  int64_t *next = (int64_t *)malloc(sizeof(int64_t) * (size_t)E);
  for (int e = 0; e < E; ++e) next[e] = (int64_t)tile_offsets[e] * BM;
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      int64_t s = (int64_t)t * k + j;
      int64_t r = next[idx[s]]++;
      row_of_slot[s] = (int32_t)r;
      token_of_row[r] = t;
    }
  free(next);
  return 0;
}

/* One expert applied to one token: fills a, b, h (length f) and y (length d). */
static void expert_fwd(int d, int f, const void *x, int x_dt, size_t xoff, const void *wgu, const void *wd,
                       int w_dt, int e, double *a, double *b, double *h, double *y) {
  size_t g0 = (size_t)e * 2 * f * d, u0 = g0 + (size_t)f * d, d0 = (size_t)e * d * f;
  for (int i = 0; i < f; ++i) {
    double sa = 0.0, sb = 0.0;
    for (int c = 0; c < d; ++c) {
      double xc = ld(x, xoff + c, x_dt);
      sa += ld(wgu, g0 + (size_t)i * d + c, w_dt) * xc;
      sb += ld(wgu, u0 + (size_t)i * d + c, w_dt) * xc;
    }
    a[i] = sa;
    b[i] = sb;
    h[i] = silu(sa) * sb;
  }
  if (y)
    for (int c = 0; c < d; ++c) {
      double s = 0.0;
      for (int i = 0; i < f; ++i) s += ld(wd, d0 + (size_t)c * f + i, w_dt) * h[i];
      y[c] = s;
    }
}

/*
 * Forward (and, if g != NULL, backward except the weight gradients) for a list of tokens.
 * tokens[n] (NULL = 0..T-1) selects which tokens; outputs are indexed by list position n:
 *   out [n_tok, d], y [n_tok, k, d] (optional), dx [n_tok, d], dlogits [n_tok, E], dw [n_tok, k].
 * idx/w are the routing of all T tokens (oracle_route_topk).
 */
int oracle_moe_tokens(int T, int d, int E, int k, int f, const void *x, int x_dt, const int32_t *idx,
                      const double *w, const void *wgu, const void *wd, int w_dt, const void *g, int g_dt,
                      const int64_t *tokens, int64_t n_tok, double *out, double *y_out, double *dx,
                      double *dlogits, double *dw_out) {
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || f <= 0) return -1;
  int bad = 0;
#pragma omp parallel
  {
    double *a = (double *)malloc(sizeof(double) * (size_t)f * 6);
    double *b = a + f, *h = b + f, *dh = h + f, *da = dh + f, *db = da + f;
    double *y = (double *)malloc(sizeof(double) * (size_t)d * k);
    double *dwl = (double *)malloc(sizeof(double) * (size_t)k);
#pragma omp for schedule(dynamic, 1)
    for (int64_t n = 0; n < n_tok; ++n) {
      int64_t t = tokens ? tokens[n] : n;
      if (t < 0 || t >= T) { bad = 1; continue; }
      size_t xoff = (size_t)t * d;
      double *o = out + (size_t)n * d;
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      for (int j = 0; j < k; ++j) {
        int e = idx[t * k + j];
        double wt = w[t * k + j];
        double *yj = y + (size_t)j * d;
        expert_fwd(d, f, x, x_dt, xoff, wgu, wd, w_dt, e, a, b, h, yj);
        for (int c = 0; c < d; ++c) o[c] += wt * yj[c];
        if (y_out) memcpy(y_out + ((size_t)n * k + j) * d, yj, sizeof(double) * (size_t)d);
      }
      if (!g) continue;
      /* routing backward */
      double sw = 0.0;
      for (int j = 0; j < k; ++j) {
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += ld(g, xoff + c, g_dt) * y[(size_t)j * d + c];
        dwl[j] = s;
        sw += w[t * k + j] * s;
      }
      if (dw_out)
        for (int j = 0; j < k; ++j) dw_out[(size_t)n * k + j] = dwl[j];
      if (dlogits) {
        double *dl = dlogits + (size_t)n * E;
        for (int e = 0; e < E; ++e) dl[e] = 0.0;
        for (int j = 0; j < k; ++j) dl[idx[t * k + j]] = w[t * k + j] * (dwl[j] - sw);
      }
      /* expert backward to the token */
      if (dx) {
        double *dxt = dx + (size_t)n * d;
        for (int c = 0; c < d; ++c) dxt[c] = 0.0;
        for (int j = 0; j < k; ++j) {
          int e = idx[t * k + j];
          double wt = w[t * k + j];
          size_t g0 = (size_t)e * 2 * f * d, u0 = g0 + (size_t)f * d, d0 = (size_t)e * d * f;
          expert_fwd(d, f, x, x_dt, xoff, wgu, wd, w_dt, e, a, b, h, NULL);
          for (int i = 0; i < f; ++i) {
            double s = 0.0;
            for (int c = 0; c < d; ++c) s += ld(wd, d0 + (size_t)c * f + i, w_dt) * ld(g, xoff + c, g_dt);
            dh[i] = wt * s;
            double sg = sigm(a[i]);
            da[i] = dh[i] * b[i] * sg * (1.0 + a[i] * (1.0 - sg));
            db[i] = dh[i] * silu(a[i]);
          }
          for (int c = 0; c < d; ++c) {
            double s = 0.0;
            for (int i = 0; i < f; ++i)
              s += ld(wgu, g0 + (size_t)i * d + c, w_dt) * da[i] + ld(wgu, u0 + (size_t)i * d + c, w_dt) * db[i];
            dxt[c] += s;
          }
        }
      }
    }
    free(a);
    free(y);
    free(dwl);
  }
  return bad ? -2 : 0;
}

/* Weight gradients of every expert over all T tokens: dwgu [E, 2f, d], dwd [E, d, f] (overwritten). */
int oracle_moe_dweights(int T, int d, int E, int k, int f, const void *x, int x_dt, const int32_t *idx,
                        const double *w, const void *wgu, const void *wd, int w_dt, const void *g, int g_dt,
                        double *dwgu, double *dwd) {
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || f <= 0) return -1;
#pragma omp parallel
  {
    double *a = (double *)malloc(sizeof(double) * (size_t)f * 6);
    double *b = a + f, *h = b + f, *dh = h + f, *da = dh + f, *db = da + f;
#pragma omp for schedule(dynamic, 1)
    for (int e = 0; e < E; ++e) {
      double *dg = dwgu + (size_t)e * 2 * f * d, *du = dg + (size_t)f * d, *dd = dwd + (size_t)e * d * f;
      memset(dg, 0, sizeof(double) * (size_t)2 * f * d);
      memset(dd, 0, sizeof(double) * (size_t)d * f);
      size_t d0 = (size_t)e * d * f;
      for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
          if (idx[t * k + j] != e) continue;
          double wt = w[t * k + j];
          size_t xoff = (size_t)t * d;
          expert_fwd(d, f, x, x_dt, xoff, wgu, wd, w_dt, e, a, b, h, NULL);
          for (int i = 0; i < f; ++i) {
            double s = 0.0;
            for (int c = 0; c < d; ++c) s += ld(wd, d0 + (size_t)c * f + i, w_dt) * ld(g, xoff + c, g_dt);
            dh[i] = wt * s;
            double sg = sigm(a[i]);
            da[i] = dh[i] * b[i] * sg * (1.0 + a[i] * (1.0 - sg));
            db[i] = dh[i] * silu(a[i]);
          }
          for (int i = 0; i < f; ++i)
            for (int c = 0; c < d; ++c) {
              double xc = ld(x, xoff + c, x_dt);
              dg[(size_t)i * d + c] += da[i] * xc;
              du[(size_t)i * d + c] += db[i] * xc;
            }
          for (int c = 0; c < d; ++c) {
            double gc = wt * ld(g, xoff + c, g_dt);
            for (int i = 0; i < f; ++i) dd[(size_t)c * f + i] += gc * h[i];
          }
        }
    }
    free(a);
  }
  return 0;
}

/*
 * Selected weight-gradient entries, each summed over all tokens routed to its expert.
 * Entry n is (mat[n], e[n], r[n], c[n]):
 *   mat 0: dWgu[e][r][c], r in [0, 2f) (rows < f are the gate, rows >= f the up projection), c in [0, d)
 *   mat 1: dWd[e][r][c],  r in [0, d), c in [0, f)
 */
int oracle_moe_dweight_entries(int T, int d, int E, int k, int f, const void *x, int x_dt, const int32_t *idx,
                               const double *w, const void *wgu, const void *wd, int w_dt, const void *g,
                               int g_dt, int64_t n_ent, const int32_t *mat, const int32_t *ent_e,
                               const int32_t *ent_r, const int32_t *ent_c, double *val) {
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t n = 0; n < n_ent; ++n) {
    int e = ent_e[n], r = ent_r[n], c = ent_c[n];
    if (e < 0 || e >= E || (mat[n] == 0 && (r < 0 || r >= 2 * f || c < 0 || c >= d)) ||
        (mat[n] == 1 && (r < 0 || r >= d || c < 0 || c >= f)) || (mat[n] != 0 && mat[n] != 1)) {
      bad = 1;
      continue;
    }
    size_t g0 = (size_t)e * 2 * f * d, u0 = g0 + (size_t)f * d, d0 = (size_t)e * d * f;
    double acc = 0.0;
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j) {
        if (idx[t * k + j] != e) continue;
        double wt = w[t * k + j];
        size_t xoff = (size_t)t * d;
        int i = (mat[n] == 0) ? (r % f) : c; /* the hidden unit this entry needs */
        double a = 0.0, b = 0.0;
        for (int q = 0; q < d; ++q) {
          double xq = ld(x, xoff + q, x_dt);
          a += ld(wgu, g0 + (size_t)i * d + q, w_dt) * xq;
          b += ld(wgu, u0 + (size_t)i * d + q, w_dt) * xq;
        }
        if (mat[n] == 1) {
          acc += wt * ld(g, xoff + r, g_dt) * (silu(a) * b);
        } else {
          double s = 0.0;
          for (int q = 0; q < d; ++q) s += ld(wd, d0 + (size_t)q * f + i, w_dt) * ld(g, xoff + q, g_dt);
          double dh = wt * s, sg = sigm(a);
          double dz = (r < f) ? dh * b * sg * (1.0 + a * (1.0 - sg)) : dh * silu(a);
          acc += dz * ld(x, xoff + c, x_dt);
        }
      }
    val[n] = acc;
  }
  return bad ? -2 : 0;
}

/*
 * The router, the step before the selection ("Scalable Pretraining of Large MoE LMs on Aurora",
 * summary page, section 关键设计: expert selection): a linear map from the token to one logit per
 * expert, L[t,e] = sum_c x[t,c] Wr[e,c], with Wr stored [E, d]. Its backward for a given dL is
 *   dx_r[t,c] = sum_e dL[t,e] Wr[e,c]      (added to the experts' dx_t by the layer)
 *   dWr[e,c]  = sum_t dL[t,e] x[t,c].
 * tok (n entries, NULL = all T tokens) lists the rows to evaluate; cols (NULL = all d) the columns
 * of dWr. Results are fp64, rows in list order.
 */
int oracle_router_logits(int T, int d, int E, const void *x, int x_dt, const void *wr, int w_dt, const int64_t *tok,
                         int64_t n, double *L) {
  if (T < 0 || d <= 0 || E <= 0) return -1;
  int bad = 0;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    int64_t t = tok ? tok[i] : i;
    if (t < 0 || t >= T) { bad = 1; continue; }
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int c = 0; c < d; ++c) s += ld(x, (size_t)t * d + c, x_dt) * ld(wr, (size_t)e * d + c, w_dt);
      L[(size_t)i * E + e] = s;
    }
  }
  return bad ? -2 : 0;
}

int oracle_router_dx(int T, int d, int E, const void *dl, int dl_dt, const void *wr, int w_dt, const int64_t *tok,
                     int64_t n, double *dx) {
  if (T < 0 || d <= 0 || E <= 0) return -1;
  int bad = 0;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    int64_t t = tok ? tok[i] : i;
    if (t < 0 || t >= T) { bad = 1; continue; }
    for (int c = 0; c < d; ++c) {
      double s = 0.0;
      for (int e = 0; e < E; ++e) s += ld(dl, (size_t)t * E + e, dl_dt) * ld(wr, (size_t)e * d + c, w_dt);
      dx[(size_t)i * d + c] = s;
    }
  }
  return bad ? -2 : 0;
}

int oracle_router_dw(int T, int d, int E, const void *x, int x_dt, const void *dl, int dl_dt, const int32_t *cols,
                     int64_t ncols, double *dw) {
  if (T < 0 || d <= 0 || E <= 0) return -1;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int e = 0; e < E; ++e)
    for (int64_t j = 0; j < ncols; ++j) {
      int c = cols ? cols[j] : (int)j;
      if (c < 0 || c >= d) { bad = 1; continue; }
      double s = 0.0;
      for (int t = 0; t < T; ++t) s += ld(dl, (size_t)t * E + e, dl_dt) * ld(x, (size_t)t * d + c, x_dt);
      dw[(size_t)e * ncols + j] = s;
    }
  return bad ? -2 : 0;
}
