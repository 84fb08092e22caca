/*
 * Exact-attention oracle: a plain, slow, fp64 CPU statement of what the fused
 * attention kernels compute.  TEST INFRASTRUCTURE ONLY: the tests, the smoke
 * check and the CPU-baseline leg of the benchmark call it; the product path
 * never does.  It shares no code, header or constant with the CUDA library.
 *
 * What it follows:
 *  - "FlashAttention-4: como Together AI acelero la atencion en GPU Blackwell",
 *    section "Por que el enfoque estandar ya no funciona": attention is the two
 *    products S = Q K^T and O = P V with a softmax between them.
 *  - "FlashAttention-3 (ES)", section "El problema del mecanismo de atencion":
 *    the softmax of the scores; the method is exact (tiling and fusion change
 *    where the numbers live, not what they are: section "FlashAttention y
 *    FlashAttention-2").
 *  - The pages do not print the scaled, masked form nor the backward formulas.
 *    The plainest reading, stated once here and used throughout:
 *        s_ij  = scale * sum_c q_ic k_jc
 *        vis   = (!causal) || (j <= i)              (lower-triangular mask)
 *        m_i   = max_{vis j} s_ij,  l_i = sum_{vis j} exp(s_ij - m_i)
 *        P_ij  = exp(s_ij - m_i) / l_i  (0 where not visible)
 *        O_i   = sum_j P_ij v_j,        LSE_i = m_i + ln(l_i)   (natural log)
 *    and, for L = sum(dO o O), by the chain rule through the softmax:
 *        dP_ij = dO_i . v_j,   D_i = dO_i . O_i,   dS_ij = P_ij (dP_ij - D_i)
 *        dQ_i  = scale sum_j dS_ij k_j
 *        dK_j  = scale sum_{h in group} sum_i dS_ij q_i
 *        dV_j  =       sum_{h in group} sum_i P_ij dO_i
 *  - Grouped-query attention: query head h reads key/value head
 *    h / (H / Hkv) (contiguous groups).
 *
 * Layouts (row-major, all double): q, o, dq, dO: [B, N, H, d];
 * k, v, dk, dv: [B, N, Hkv, d]; lse: [B, H, N].
 *
 * Each function loops in the order the formulas above are written; OpenMP
 * only splits independent rows (or independent key rows) across threads.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX4(b, n, h, c, N, Hx, d) ((((size_t)(b) * (N) + (n)) * (Hx) + (h)) * (d) + (c))

static double dot(const double *x, const double *y, int d) {
  double acc = 0.0;
  for (int c = 0; c < d; ++c) acc += x[c] * y[c];
  return acc;
}

static int visible(int i, int j, int causal) { return !causal || j <= i; }

/* Row statistics of one query row i of head (b, h): m_i and l_i, plus the
 * scores s_ij for every key j (written to s, -INFINITY where not visible). */
static void row_scores(const double *q, const double *k, int b, int h, int kh, int i,
                       int N, int H, int Hkv, int d, double scale, int causal,
                       double *s, double *m_out, double *l_out) {
  const double *qi = q + IDX4(b, i, h, 0, N, H, d);
  double m = -INFINITY;
  for (int j = 0; j < N; ++j) {
    if (visible(i, j, causal)) {
      s[j] = scale * dot(qi, k + IDX4(b, j, kh, 0, N, Hkv, d), d);
      if (s[j] > m) m = s[j];
    } else {
      s[j] = -INFINITY;
    }
  }
  double l = 0.0;
  for (int j = 0; j < N; ++j)
    if (visible(i, j, causal)) l += exp(s[j] - m);
  *m_out = m;
  *l_out = l;
}

/* Forward for the listed query rows (rows == NULL means every row 0..N-1).
 * o: [B, nrows, H, d], lse: [B, H, nrows], in the order of `rows`. */
void oracle_fwd_rows(const double *q, const double *k, const double *v,
                     int B, int H, int Hkv, int N, int d, double scale, int causal,
                     const int *rows, int nrows, double *o, double *lse) {
  const int g = H / Hkv;
  const long total = (long)B * H * nrows;
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 4)
    for (long t = 0; t < total; ++t) {
      const int r = (int)(t % nrows);
      const int h = (int)((t / nrows) % H);
      const int b = (int)(t / ((long)nrows * H));
      const int i = rows ? rows[r] : r;
      const int kh = h / g;
      double m, l;
      row_scores(q, k, b, h, kh, i, N, H, Hkv, d, scale, causal, s, &m, &l);
      double *oi = o + IDX4(b, r, h, 0, nrows, H, d);
      for (int c = 0; c < d; ++c) oi[c] = 0.0;
      for (int j = 0; j < N; ++j) {
        if (!visible(i, j, causal)) continue;
        const double p = exp(s[j] - m) / l;
        const double *vj = v + IDX4(b, j, kh, 0, N, Hkv, d);
        for (int c = 0; c < d; ++c) oi[c] += p * vj[c];
      }
      lse[((size_t)b * H + h) * nrows + r] = m + log(l);
    }
    free(s);
  }
}

void oracle_fwd(const double *q, const double *k, const double *v,
                int B, int H, int Hkv, int N, int d, double scale, int causal,
                double *o, double *lse) {
  oracle_fwd_rows(q, k, v, B, H, Hkv, N, d, scale, causal, NULL, N, o, lse);
}

/* Backward.  dq is produced for the listed query rows, dk and dv for the listed
 * key rows (NULL lists mean every row).  Shapes: dq [B, nq, H, d],
 * dk/dv [B, nkv, Hkv, d].  The forward statistics (LSE_i, O_i, D_i) of every
 * query row are recomputed here from the definition, in fp64. */
void oracle_bwd_rows(const double *q, const double *k, const double *v, const double *dO,
                     int B, int H, int Hkv, int N, int d, double scale, int causal,
                     const int *qrows, int nq, const int *kvrows, int nkv,
                     double *dq, double *dk, double *dv) {
  const int g = H / Hkv;
  double *lse = (double *)malloc(sizeof(double) * (size_t)B * H * N);
  double *D = (double *)malloc(sizeof(double) * (size_t)B * H * N);

  /* Step 1: for every query row, LSE_i and D_i = dO_i . O_i with O_i the fp64
   * forward output of that row. */
  {
    const long total = (long)B * H * N;
#pragma omp parallel
    {
      double *s = (double *)malloc(sizeof(double) * (size_t)N);
      double *oi = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 4)
      for (long t = 0; t < total; ++t) {
        const int i = (int)(t % N);
        const int h = (int)((t / N) % H);
        const int b = (int)(t / ((long)N * H));
        const int kh = h / g;
        double m, l;
        row_scores(q, k, b, h, kh, i, N, H, Hkv, d, scale, causal, s, &m, &l);
        for (int c = 0; c < d; ++c) oi[c] = 0.0;
        for (int j = 0; j < N; ++j) {
          if (!visible(i, j, causal)) continue;
          const double p = exp(s[j] - m) / l;
          const double *vj = v + IDX4(b, j, kh, 0, N, Hkv, d);
          for (int c = 0; c < d; ++c) oi[c] += p * vj[c];
        }
        lse[((size_t)b * H + h) * N + i] = m + log(l);
        D[((size_t)b * H + h) * N + i] = dot(dO + IDX4(b, i, h, 0, N, H, d), oi, d);
      }
      free(oi);
      free(s);
    }
  }

  /* Step 2: dQ_i = scale sum_j P_ij (dP_ij - D_i) k_j, with P_ij = exp(s_ij - LSE_i). */
  {
    const long total = (long)B * H * nq;
#pragma omp parallel for schedule(dynamic, 4)
    for (long t = 0; t < total; ++t) {
      const int r = (int)(t % nq);
      const int h = (int)((t / nq) % H);
      const int b = (int)(t / ((long)nq * H));
      const int i = qrows ? qrows[r] : r;
      const int kh = h / g;
      const double *qi = q + IDX4(b, i, h, 0, N, H, d);
      const double *doi = dO + IDX4(b, i, h, 0, N, H, d);
      const double Li = lse[((size_t)b * H + h) * N + i];
      const double Di = D[((size_t)b * H + h) * N + i];
      double *dqi = dq + IDX4(b, r, h, 0, nq, H, d);
      for (int c = 0; c < d; ++c) dqi[c] = 0.0;
      for (int j = 0; j < N; ++j) {
        if (!visible(i, j, causal)) continue;
        const double *kj = k + IDX4(b, j, kh, 0, N, Hkv, d);
        const double *vj = v + IDX4(b, j, kh, 0, N, Hkv, d);
        const double p = exp(scale * dot(qi, kj, d) - Li);
        const double ds = p * (dot(doi, vj, d) - Di);
        for (int c = 0; c < d; ++c) dqi[c] += scale * ds * kj[c];
      }
    }
  }

  /* Step 3: dK_j and dV_j, summed over the query heads of the group and over i. */
  {
    const long total = (long)B * Hkv * nkv;
#pragma omp parallel for schedule(dynamic, 4)
    for (long t = 0; t < total; ++t) {
      const int r = (int)(t % nkv);
      const int kh = (int)((t / nkv) % Hkv);
      const int b = (int)(t / ((long)nkv * Hkv));
      const int j = kvrows ? kvrows[r] : r;
      const double *kj = k + IDX4(b, j, kh, 0, N, Hkv, d);
      const double *vj = v + IDX4(b, j, kh, 0, N, Hkv, d);
      double *dkj = dk + IDX4(b, r, kh, 0, nkv, Hkv, d);
      double *dvj = dv + IDX4(b, r, kh, 0, nkv, Hkv, d);
      for (int c = 0; c < d; ++c) dkj[c] = dvj[c] = 0.0;
      for (int h = kh * g; h < (kh + 1) * g; ++h) {
        for (int i = 0; i < N; ++i) {
          if (!visible(i, j, causal)) continue;
          const double *qi = q + IDX4(b, i, h, 0, N, H, d);
          const double *doi = dO + IDX4(b, i, h, 0, N, H, d);
          const double p = exp(scale * dot(qi, kj, d) - lse[((size_t)b * H + h) * N + i]);
          const double ds = p * (dot(doi, vj, d) - D[((size_t)b * H + h) * N + i]);
          for (int c = 0; c < d; ++c) {
            dvj[c] += p * doi[c];
            dkj[c] += scale * ds * qi[c];
          }
        }
      }
    }
  }
  free(D);
  free(lse);
}

void oracle_bwd(const double *q, const double *k, const double *v, const double *dO,
                int B, int H, int Hkv, int N, int d, double scale, int causal,
                double *dq, double *dk, double *dv) {
  oracle_bwd_rows(q, k, v, dO, B, H, Hkv, N, d, scale, causal, NULL, N, NULL, N, dq, dk, dv);
}

/* Threads for this library's later parallel regions (n >= 1); for timing only. */
void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Number of OpenMP threads a parallel region of this library uses. */
int oracle_num_threads(void) {
  int n = 1;
#pragma omp parallel
  {
#pragma omp single
    {
#ifdef _OPENMP
      n = omp_get_num_threads();
#endif
    }
  }
  return n;
}
