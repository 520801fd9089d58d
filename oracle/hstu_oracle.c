/*
 * hstu_oracle.c -- plain, slow, FP64 CPU oracle for HSTU jagged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA path and the CUDA path never calls it.
 *
 * What it computes (HSTU, "Spatial Aggregation" and "Pointwise
 * Transformation", ai6s.net generative-recommendation survey, section 2.1.2,
 * equations (2) and (3), whose images did not survive extraction; the
 * formula used is the softmax-free pointwise form the prose describes):
 *
 *   for every sequence b and head h, for tokens i, j of that sequence:
 *     z_ij = alpha * <q_i, k_j> + rab_pos[h][bp(i,j)] + rab_time[h][bt(i,j)]
 *     A_ij = allowed(i,j) ? SiLU(z_ij) / N : 0          (no softmax)
 *     o_i  = sum_j A_ij v_j
 *   y_t = LayerNorm(concat_h o_t) (*) u_t                 (population variance,
 *                                                        no affine)
 *
 * Mask (ranking task, section 2.1.2: candidates are appended after the
 * history and must not interact with each other; the compound causal +
 * context/target mask of the wmrh.cn RecSDK page, "HSTU acceleration
 * operator" paragraph).  With n tokens, c context tokens in front and m
 * candidates at the end, h_end = n - m:
 *     j >= h_end : allowed iff i == j          (a candidate sees itself only
 *                                               among the candidates)
 *     j <  h_end : allowed iff j <= i or (i < c and j < c)
 *
 * Buckets:
 *     pos(i)   = min(i, h_end)        (all candidates share one position)
 *     bp(i,j)  = min(|pos(i) - pos(j)|, P - 1)
 *     bt(i,j)  = 0 if t_i == t_j, else min(Tb - 1, floor(log2 |t_i - t_j|) + 1)
 *
 * Backward: the chain rule of the above, with SiLU'(z) = s(z)(1 + z(1 - s(z))),
 * s the logistic sigmoid.
 *
 * Everything is double precision with plain loops; OpenMP (when compiled with
 * it) only splits independent (sequence, head, row) work.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- helpers */

static int64_t seq_len(const int64_t* off, int b) { return off[b + 1] - off[b]; }

static int64_t n_targets_of(const int32_t* nt, int b) { return nt ? nt[b] : 0; }
static int64_t n_contexts_of(const int32_t* nc, int b) { return nc ? nc[b] : 0; }

/* allowed(i, j) for one sequence: the compound mask described above. */
static int allowed(int64_t i, int64_t j, int64_t c, int64_t h_end) {
  if (j >= h_end) return i == j;
  return (j <= i) || (i < c && j < c);
}

static int64_t position_of(int64_t i, int64_t h_end) { return i < h_end ? i : h_end; }

static int pos_bucket(int64_t i, int64_t j, int64_t h_end, int P) {
  int64_t d = position_of(i, h_end) - position_of(j, h_end);
  if (d < 0) d = -d;
  return (int)(d < P - 1 ? d : P - 1);
}

/* floor(log2 delta) + 1 for delta > 0, 0 for delta == 0: the number of
 * binary digits of delta, counted by repeated halving. */
static int time_bucket(int64_t ti, int64_t tj, int Tb) {
  uint64_t d = ti >= tj ? (uint64_t)ti - (uint64_t)tj : (uint64_t)tj - (uint64_t)ti;
  int digits = 0;
  while (d > 0) { digits++; d >>= 1; }
  return digits < Tb - 1 ? digits : Tb - 1;
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }
static double silu(double z) { return z * sigmoid(z); }
static double silu_grad(double z) { double s = sigmoid(z); return s * (1.0 + z * (1.0 - s)); }

typedef struct {
  int B, H, dqk, dv, P, Tb;
  const int64_t* off; const int32_t* nt; const int32_t* nc; const int64_t* ts;
  const double* rab_pos; const double* rab_time;
  double alpha, N;
  const double *q, *k, *v;
} problem_t;

/* z_ij for global token rows gi = s0 + i, gj = s0 + j of head h. */
static double score(const problem_t* p, int h, int64_t s0, int64_t i, int64_t j, int64_t h_end) {
  const double* qi = p->q + ((s0 + i) * p->H + h) * p->dqk;
  const double* kj = p->k + ((s0 + j) * p->H + h) * p->dqk;
  double dot = 0.0;
  for (int e = 0; e < p->dqk; ++e) dot += qi[e] * kj[e];
  double z = p->alpha * dot;
  if (p->rab_pos) z += p->rab_pos[h * p->P + pos_bucket(i, j, h_end, p->P)];
  if (p->rab_time && p->ts) z += p->rab_time[h * p->Tb + time_bucket(p->ts[s0 + i], p->ts[s0 + j], p->Tb)];
  return z;
}

/* ---------------------------------------------------------------- forward */

/* o[T,H,dv] for every row (row_mask == NULL) or the rows with row_mask[t] != 0.
 * Rows not selected are left untouched.  Returns 0, or -1 on invalid input. */
int hstu_oracle_fwd(int B, int H, int dqk, int dv,
                    const int64_t* offsets, const int32_t* num_targets, const int32_t* num_contexts,
                    const int64_t* timestamps, const double* rab_pos, int P, const double* rab_time, int Tb,
                    double alpha, double N,
                    const double* q, const double* k, const double* v,
                    double* o, const uint8_t* row_mask) {
  problem_t p = {B, H, dqk, dv, P, Tb, offsets, num_targets, num_contexts, timestamps,
                 rab_pos, rab_time, alpha, N, q, k, v};
  for (int b = 0; b < B; ++b) {
    int64_t n = seq_len(offsets, b);
    if (n < 0 || n_targets_of(num_targets, b) + n_contexts_of(num_contexts, b) > n) return -1;
  }
  int64_t T = offsets[B];
  int64_t work = T * (int64_t)H;
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t w = 0; w < work; ++w) {
    int64_t t = w / H; int h = (int)(w % H);
    if (row_mask && !row_mask[t]) continue;
    int b = 0;
    { int lo = 0, hi = B - 1; while (lo < hi) { int mid = (lo + hi + 1) / 2; if (offsets[mid] <= t) lo = mid; else hi = mid - 1; } b = lo; }
    int64_t s0 = offsets[b], n = seq_len(offsets, b), i = t - s0;
    int64_t c = n_contexts_of(num_contexts, b), h_end = n - n_targets_of(num_targets, b);
    double* oi = o + (t * H + h) * dv;
    for (int e = 0; e < dv; ++e) oi[e] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      if (!allowed(i, j, c, h_end)) continue;
      double a = silu(score(&p, h, s0, i, j, h_end)) / N;
      const double* vj = v + ((s0 + j) * H + h) * dv;
      for (int e = 0; e < dv; ++e) oi[e] += a * vj[e];
    }
  }
  return 0;
}

/* ------------------------------------------------------------- norm + gate */

/* Per token t over its F = H*dv features x = o[t, :]:
 *   norm == 1 (LayerNorm): mean = sum(x)/F, var = sum((x-mean)^2)/F,
 *                          rstd = 1/sqrt(var + eps), y = (x - mean) * rstd * u
 *   norm == 0 (none):      y = x * u
 * u == NULL means a gate of one.  mean/rstd may be NULL. */
int hstu_oracle_norm_gate(int64_t T, int F, int norm, double eps, const double* o, const double* u,
                          double* y, double* mean_out, double* rstd_out, const uint8_t* row_mask) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    if (row_mask && !row_mask[t]) continue;
    const double* x = o + t * F;
    double mean = 0.0, var = 0.0, rstd = 1.0;
    if (norm == 1) {
      for (int f = 0; f < F; ++f) mean += x[f];
      mean /= F;
      for (int f = 0; f < F; ++f) var += (x[f] - mean) * (x[f] - mean);
      var /= F;
      rstd = 1.0 / sqrt(var + eps);
    }
    for (int f = 0; f < F; ++f) {
      double xn = norm == 1 ? (x[f] - mean) * rstd : x[f];
      y[t * F + f] = u ? xn * u[t * F + f] : xn;
    }
    if (mean_out) mean_out[t] = mean;
    if (rstd_out) rstd_out[t] = rstd;
  }
  return 0;
}

/* Backward of the above given dy:  with xn the normalised x and g = dy * u,
 *   du = xn * dy
 *   LayerNorm: dx = rstd * (g - mean(g) - xn * mean(g * xn))
 *   none:      dx = g
 * (u == NULL: g = dy, du not written). */
int hstu_oracle_norm_gate_bwd(int64_t T, int F, int norm, double eps, const double* o, const double* u,
                              const double* dy, double* dx, double* du, const uint8_t* row_mask) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    if (row_mask && !row_mask[t]) continue;
    const double* x = o + t * F;
    double mean = 0.0, var = 0.0, rstd = 1.0;
    if (norm == 1) {
      for (int f = 0; f < F; ++f) mean += x[f];
      mean /= F;
      for (int f = 0; f < F; ++f) var += (x[f] - mean) * (x[f] - mean);
      var /= F;
      rstd = 1.0 / sqrt(var + eps);
    }
    double mg = 0.0, mgx = 0.0;
    for (int f = 0; f < F; ++f) {
      double xn = norm == 1 ? (x[f] - mean) * rstd : x[f];
      double g = u ? dy[t * F + f] * u[t * F + f] : dy[t * F + f];
      if (du) du[t * F + f] = xn * dy[t * F + f];
      mg += g; mgx += g * xn;
    }
    mg /= F; mgx /= F;
    for (int f = 0; f < F; ++f) {
      double xn = norm == 1 ? (x[f] - mean) * rstd : x[f];
      double g = u ? dy[t * F + f] * u[t * F + f] : dy[t * F + f];
      dx[t * F + f] = norm == 1 ? rstd * (g - mg - xn * mgx) : g;
    }
  }
  return 0;
}

/* --------------------------------------------------------------- backward */

/* Attention backward given dO = d(loss)/d(o) [T,H,dv].
 *   dv_j = sum_i A_ij dO_i
 *   dA_ij = <dO_i, v_j>,   dZ_ij = allowed ? dA_ij * SiLU'(z_ij) / N : 0
 *   dq_i = alpha * sum_j dZ_ij k_j,   dk_j = alpha * sum_i dZ_ij q_i
 *   d_rab_pos[h][bp] = sum of dZ over pairs in bucket bp, same for time.
 * dq rows are computed where q_rows[t] != 0 (all if NULL); dk/dv rows where
 * kv_rows[t] != 0 (all if NULL).  d_rab_* are only written when both masks are
 * NULL (they need every pair).  Any output pointer may be NULL to skip it. */
int hstu_oracle_attn_bwd(int B, int H, int dqk, int dv,
                         const int64_t* offsets, const int32_t* num_targets, const int32_t* num_contexts,
                         const int64_t* timestamps, const double* rab_pos, int P, const double* rab_time, int Tb,
                         double alpha, double N,
                         const double* q, const double* k, const double* v, const double* dO,
                         double* dq, double* dk, double* dvo, double* d_rab_pos, double* d_rab_time,
                         const uint8_t* q_rows, const uint8_t* kv_rows) {
  problem_t p = {B, H, dqk, dv, P, Tb, offsets, num_targets, num_contexts, timestamps,
                 rab_pos, rab_time, alpha, N, q, k, v};
  for (int b = 0; b < B; ++b) {
    int64_t n = seq_len(offsets, b);
    if (n < 0 || n_targets_of(num_targets, b) + n_contexts_of(num_contexts, b) > n) return -1;
  }
  int64_t T = offsets[B];
  int64_t work = T * (int64_t)H;

  /* pass 1: dq_i, one (row, head) at a time */
  if (dq) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t w = 0; w < work; ++w) {
      int64_t t = w / H; int h = (int)(w % H);
      if (q_rows && !q_rows[t]) continue;
      int b = 0;
      { int lo = 0, hi = B - 1; while (lo < hi) { int mid = (lo + hi + 1) / 2; if (offsets[mid] <= t) lo = mid; else hi = mid - 1; } b = lo; }
      int64_t s0 = offsets[b], n = seq_len(offsets, b), i = t - s0;
      int64_t c = n_contexts_of(num_contexts, b), h_end = n - n_targets_of(num_targets, b);
      double* dqi = dq + (t * H + h) * dqk;
      for (int e = 0; e < dqk; ++e) dqi[e] = 0.0;
      const double* doi = dO + (t * H + h) * dv;
      for (int64_t j = 0; j < n; ++j) {
        if (!allowed(i, j, c, h_end)) continue;
        const double* vj = v + ((s0 + j) * H + h) * dv;
        double dA = 0.0;
        for (int e = 0; e < dv; ++e) dA += doi[e] * vj[e];
        double dZ = dA * silu_grad(score(&p, h, s0, i, j, h_end)) / N;
        const double* kj = k + ((s0 + j) * H + h) * dqk;
        for (int e = 0; e < dqk; ++e) dqi[e] += alpha * dZ * kj[e];
      }
    }
  }

  /* pass 2: dk_j and dv_j, one (column, head) at a time */
  if (dk || dvo) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t w = 0; w < work; ++w) {
      int64_t t = w / H; int h = (int)(w % H);
      if (kv_rows && !kv_rows[t]) continue;
      int b = 0;
      { int lo = 0, hi = B - 1; while (lo < hi) { int mid = (lo + hi + 1) / 2; if (offsets[mid] <= t) lo = mid; else hi = mid - 1; } b = lo; }
      int64_t s0 = offsets[b], n = seq_len(offsets, b), j = t - s0;
      int64_t c = n_contexts_of(num_contexts, b), h_end = n - n_targets_of(num_targets, b);
      double* dkj = dk ? dk + (t * H + h) * dqk : NULL;
      double* dvj = dvo ? dvo + (t * H + h) * dv : NULL;
      if (dkj) for (int e = 0; e < dqk; ++e) dkj[e] = 0.0;
      if (dvj) for (int e = 0; e < dv; ++e) dvj[e] = 0.0;
      const double* vj = v + (t * H + h) * dv;
      for (int64_t i = 0; i < n; ++i) {
        if (!allowed(i, j, c, h_end)) continue;
        const double* doi = dO + ((s0 + i) * H + h) * dv;
        double z = score(&p, h, s0, i, j, h_end);
        if (dvj) {
          double a = silu(z) / N;
          for (int e = 0; e < dv; ++e) dvj[e] += a * doi[e];
        }
        if (dkj) {
          double dA = 0.0;
          for (int e = 0; e < dv; ++e) dA += doi[e] * vj[e];
          double dZ = dA * silu_grad(z) / N;
          const double* qi = q + ((s0 + i) * H + h) * dqk;
          for (int e = 0; e < dqk; ++e) dkj[e] += alpha * dZ * qi[e];
        }
      }
    }
  }

  /* pass 3: d-rab, every pair of every (sequence, head) */
  if ((d_rab_pos || d_rab_time) && !q_rows && !kv_rows) {
    if (d_rab_pos) memset(d_rab_pos, 0, sizeof(double) * (size_t)H * P);
    if (d_rab_time) memset(d_rab_time, 0, sizeof(double) * (size_t)H * Tb);
    int64_t tasks = (int64_t)B * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < tasks; ++w) {
      int b = (int)(w / H), h = (int)(w % H);
      int64_t s0 = offsets[b], n = seq_len(offsets, b);
      int64_t c = n_contexts_of(num_contexts, b), h_end = n - n_targets_of(num_targets, b);
      double* lp = (double*)calloc((size_t)P, sizeof(double));
      double* lt = (double*)calloc((size_t)Tb, sizeof(double));
      for (int64_t i = 0; i < n; ++i) {
        const double* doi = dO + ((s0 + i) * H + h) * dv;
        for (int64_t j = 0; j < n; ++j) {
          if (!allowed(i, j, c, h_end)) continue;
          const double* vj = v + ((s0 + j) * H + h) * dv;
          double dA = 0.0;
          for (int e = 0; e < dv; ++e) dA += doi[e] * vj[e];
          double dZ = dA * silu_grad(score(&p, h, s0, i, j, h_end)) / N;
          lp[pos_bucket(i, j, h_end, P)] += dZ;
          if (timestamps) lt[time_bucket(timestamps[s0 + i], timestamps[s0 + j], Tb)] += dZ;
        }
      }
#pragma omp critical
      {
        if (d_rab_pos && rab_pos) for (int e = 0; e < P; ++e) d_rab_pos[h * P + e] += lp[e];
        if (d_rab_time && rab_time && timestamps) for (int e = 0; e < Tb; ++e) d_rab_time[h * Tb + e] += lt[e];
      }
      free(lp); free(lt);
    }
  }
  return 0;
}

/* ------------------------------------------------------------- tile plan */

/* Brute-force tile classification for BM x BN tiles of every sequence:
 * counts the allowed, in-sequence pairs of the tile one by one.
 * class 0 = SKIP (no allowed pair), 2 = FULL (all BM*BN pairs in the sequence
 * and allowed), 1 = PARTIAL.  Tiles are listed sequence by sequence, q-block
 * major, k-block minor; out_* must hold oracle_tile_count() entries. */
int64_t hstu_oracle_tile_count(int B, const int64_t* offsets, int BM, int BN) {
  int64_t total = 0;
  for (int b = 0; b < B; ++b) {
    int64_t n = seq_len(offsets, b);
    total += ((n + BM - 1) / BM) * ((n + BN - 1) / BN);
  }
  return total;
}

int hstu_oracle_tile_classes(int B, const int64_t* offsets, const int32_t* num_targets,
                             const int32_t* num_contexts, int BM, int BN,
                             int32_t* out_b, int32_t* out_qb, int32_t* out_kb, int32_t* out_class,
                             int64_t* out_allowed) {
  int64_t idx = 0;
  for (int b = 0; b < B; ++b) {
    int64_t n = seq_len(offsets, b);
    int64_t c = n_contexts_of(num_contexts, b), h_end = n - n_targets_of(num_targets, b);
    for (int64_t qb = 0; qb * BM < n; ++qb) {
      for (int64_t kb = 0; kb * BN < n; ++kb) {
        int64_t count = 0;
        for (int64_t i = qb * BM; i < (qb + 1) * BM; ++i)
          for (int64_t j = kb * BN; j < (kb + 1) * BN; ++j)
            if (i < n && j < n && allowed(i, j, c, h_end)) count++;
        out_b[idx] = b; out_qb[idx] = (int32_t)qb; out_kb[idx] = (int32_t)kb;
        out_class[idx] = count == 0 ? 0 : (count == (int64_t)BM * BN ? 2 : 1);
        if (out_allowed) out_allowed[idx] = count;
        idx++;
      }
    }
  }
  return 0;
}

/* Number of allowed pairs of every sequence, counted one by one. */
int hstu_oracle_allowed_pairs(int B, const int64_t* offsets, const int32_t* num_targets,
                              const int32_t* num_contexts, int64_t* out) {
  for (int b = 0; b < B; ++b) {
    int64_t n = seq_len(offsets, b);
    int64_t c = n_contexts_of(num_contexts, b), h_end = n - n_targets_of(num_targets, b);
    int64_t count = 0;
    for (int64_t i = 0; i < n; ++i)
      for (int64_t j = 0; j < n; ++j)
        count += allowed(i, j, c, h_end);
    out[b] = count;
  }
  return 0;
}

/* Exported bucket functions, so tests can pin them to their definitions. */
int hstu_oracle_time_bucket(int64_t ti, int64_t tj, int Tb) { return time_bucket(ti, tj, Tb); }
int hstu_oracle_pos_bucket(int64_t i, int64_t j, int64_t h_end, int P) { return pos_bucket(i, j, h_end, P); }

int hstu_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
