/*
 * attention_oracle.c -- fp64 CPU oracle for exact attention, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or load
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header, table or helper with the CUDA
 * library; it is the plain definition of the operation written out in double
 * precision, so that a reader can check it against the source pages by eye.
 *
 * What it computes (per batch b, query head h, kv head g = h / (H / HKV)):
 *
 *   S_ij  = scale * sum_d Q[b,h,i,d] * K[b,g,j,d]
 *           -- rustytorch "flash_attention_forward.metal", kernel header comment
 *              (the output is the scaled-score row softmax applied to V)
 *   visible(i,j) = (!causal || j <= i) && (window == 0 || j >= i - window + 1)
 *           -- forge "flash_attention.metal", FlashParams comment (window keeps
 *              keys including self, 0 = full) and flash_attn_fwd's jmin / j_end;
 *              boostr "flash.wgsl", flash_attention_fwd_f32 start_k / end_k
 *   P_ij  = exp(S_ij - m_i) / sum_{k visible} exp(S_ik - m_i),  m_i = max_vis S_ij
 *   O_i   = sum_j P_ij V[b,g,j]
 *   LSE_i = m_i + log sum_{j visible} exp(S_ij - m_i)   (natural log)
 *           -- all three pages store this one float per query row
 *   Row with no visible key: O_i = 0, LSE_i = -inf, and P_i. = 0 in the backward.
 *
 * Backward, by the textbook chain rule through the softmax Jacobian (deliberately
 * NOT the rowsum(dO o O) identity that the GPU path uses):
 *   dP_ij = dO_i . V_j
 *   r_i   = sum_k P_ik dP_ik
 *   dS_ij = P_ij (dP_ij - r_i)
 *   dQ_i  = scale sum_j dS_ij K_j
 *   dK_j  = scale sum_{h in group} sum_i dS_ij Q_i
 *   dV_j  = sum_{h in group} sum_i P_ij dO_i
 *           -- forge "flash_attention.metal", kernels flash_attn_bwd_dq,
 *              flash_attn_bwd_dv, flash_attn_bwd_dk (gradients summed over the
 *              grouped query heads of each kv head)
 *
 * Every sum runs in a fixed order; each output element is produced by exactly one
 * OpenMP iteration, so the result does not depend on the thread count.
 *
 * Layout: Q, O, dO, dQ are [B, H, Sq, D]; K, V, dK, dV are [B, HKV, Sk, D];
 * LSE is [B, H, Sq]. All contiguous, row-major, double.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int B, H, HKV, Sq, Sk, D;
  double scale;
  int causal;
  int window;
} oracle_shape;

static int oracle_check(const oracle_shape* s) {
  if (s->B < 0 || s->H < 1 || s->HKV < 1 || s->Sq < 0 || s->Sk < 0 || s->D < 1) return -1;
  if (s->H % s->HKV != 0) return -1;
  if (s->window < 0 || (s->causal != 0 && s->causal != 1)) return -1;
  return 0;
}

static int visible(long i, long j, const oracle_shape* s) {
  if (s->causal && j > i) return 0;
  if (s->window > 0 && j < i - (long)s->window + 1) return 0;
  return 1;
}

static double dot(const double* a, const double* b, int n) {
  double acc = 0.0;
  for (int d = 0; d < n; ++d) acc += a[d] * b[d];
  return acc;
}

/* Softmax row of query i against the Sk keys of kv head Kg.
 * Writes the normalised probabilities into p[0..Sk) (0 where masked) and returns
 * the natural-log LSE of the row, or -inf if no key is visible. m_out / sum_out
 * receive the row max of S and sum_j exp(S_ij - m) for recomputation. */
static double softmax_row(const double* qi, const double* Kg, long i, const oracle_shape* s,
                          double* p, double* m_out, double* sum_out) {
  const int Sk = s->Sk, D = s->D;
  double m = -INFINITY;
  int any = 0;
  for (long j = 0; j < Sk; ++j) {
    if (!visible(i, j, s)) { p[j] = -INFINITY; continue; }
    p[j] = s->scale * dot(qi, Kg + j * (long)D, D);   /* S_ij */
    if (!any || p[j] > m) m = p[j];
    any = 1;
  }
  if (!any) {
    for (long j = 0; j < Sk; ++j) p[j] = 0.0;
    *m_out = -INFINITY;
    *sum_out = 0.0;
    return -INFINITY;
  }
  double sum = 0.0;
  for (long j = 0; j < Sk; ++j) {
    if (!visible(i, j, s)) { p[j] = 0.0; continue; }
    p[j] = exp(p[j] - m);
    sum += p[j];
  }
  for (long j = 0; j < Sk; ++j) p[j] /= sum;
  *m_out = m;
  *sum_out = sum;
  return m + log(sum);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Forward: O = softmax(scale Q K^T + mask) V and the per-row LSE. Returns 0, or -1
 * on an invalid shape. */
int oracle_attention_fwd(const double* Q, const double* K, const double* V, double* O, double* LSE,
                         int B, int H, int HKV, int Sq, int Sk, int D, double scale, int causal,
                         int window) {
  oracle_shape s = {B, H, HKV, Sq, Sk, D, scale, causal, window};
  if (oracle_check(&s)) return -1;
  const int rep = H / HKV;
  const long rows = (long)B * H * Sq;
  int fail = 0;
#pragma omp parallel
  {
    double* p = (double*)malloc(sizeof(double) * (Sk > 0 ? Sk : 1));
    if (!p) {
#pragma omp atomic write
      fail = 1;
    }
#pragma omp for schedule(dynamic, 16)
    for (long r = 0; r < rows; ++r) {
      if (!p) continue;
      const long i = r % Sq, bh = r / Sq, h = bh % H, b = bh / H, g = h / rep;
      const double* qi = Q + r * D;
      const double* Kg = K + ((long)b * HKV + g) * (long)Sk * D;
      const double* Vg = V + ((long)b * HKV + g) * (long)Sk * D;
      double m, sum;
      LSE[r] = softmax_row(qi, Kg, i, &s, p, &m, &sum);
      double* oi = O + r * D;
      for (int d = 0; d < D; ++d) oi[d] = 0.0;
      for (long j = 0; j < Sk; ++j) {
        if (p[j] == 0.0) continue;
        for (int d = 0; d < D; ++d) oi[d] += p[j] * Vg[j * (long)D + d];
      }
    }
    free(p);
  }
  return fail ? -2 : 0;
}

/* Backward through the softmax Jacobian. Inputs Q, K, V, dO; outputs dQ, dK, dV
 * (overwritten). O and LSE are not inputs: P is rebuilt from its definition.
 * Phase 1 walks query rows (dQ, and the row statistics m_i, sum_i, r_i);
 * phase 2 walks key rows of each kv head (dK, dV), recomputing P_ij and dS_ij
 * from those statistics. */
int oracle_attention_bwd(const double* Q, const double* K, const double* V, const double* dO,
                         double* dQ, double* dK, double* dV, int B, int H, int HKV, int Sq, int Sk,
                         int D, double scale, int causal, int window) {
  oracle_shape s = {B, H, HKV, Sq, Sk, D, scale, causal, window};
  if (oracle_check(&s)) return -1;
  const int rep = H / HKV;
  const long rows = (long)B * H * Sq;
  const long krows = (long)B * HKV * Sk;
  double* mrow = (double*)malloc(sizeof(double) * (rows > 0 ? rows : 1));
  double* srow = (double*)malloc(sizeof(double) * (rows > 0 ? rows : 1));
  double* rrow = (double*)malloc(sizeof(double) * (rows > 0 ? rows : 1));
  if (!mrow || !srow || !rrow) { free(mrow); free(srow); free(rrow); return -2; }
  int fail = 0;

  /* Phase 1: per query row i of head (b,h). */
#pragma omp parallel
  {
    double* p = (double*)malloc(sizeof(double) * (Sk > 0 ? Sk : 1));
    double* dp = (double*)malloc(sizeof(double) * (Sk > 0 ? Sk : 1));
    if (!p || !dp) {
#pragma omp atomic write
      fail = 1;
    }
#pragma omp for schedule(dynamic, 16)
    for (long r = 0; r < rows; ++r) {
      if (!p || !dp) continue;
      const long i = r % Sq, bh = r / Sq, h = bh % H, b = bh / H, g = h / rep;
      const double* Kg = K + ((long)b * HKV + g) * (long)Sk * D;
      const double* Vg = V + ((long)b * HKV + g) * (long)Sk * D;
      const double* doi = dO + r * D;
      softmax_row(Q + r * D, Kg, i, &s, p, &mrow[r], &srow[r]);
      double ri = 0.0;                       /* r_i = sum_k P_ik dP_ik */
      for (long j = 0; j < Sk; ++j) {
        dp[j] = (p[j] != 0.0) ? dot(doi, Vg + j * (long)D, D) : 0.0;
        ri += p[j] * dp[j];
      }
      rrow[r] = ri;
      double* dqi = dQ + r * D;
      for (int d = 0; d < D; ++d) dqi[d] = 0.0;
      for (long j = 0; j < Sk; ++j) {
        if (p[j] == 0.0) continue;
        const double ds = p[j] * (dp[j] - ri);
        for (int d = 0; d < D; ++d) dqi[d] += ds * Kg[j * (long)D + d];
      }
      for (int d = 0; d < D; ++d) dqi[d] *= scale;
    }
    free(p);
    free(dp);
  }

  /* Phase 2: per key row j of kv head (b,g), summing over the grouped query heads. */
#pragma omp parallel for schedule(dynamic, 16)
  for (long kr = 0; kr < krows; ++kr) {
    const long j = kr % Sk, bg = kr / Sk, g = bg % HKV, b = bg / HKV;
    const double* kj = K + kr * D;
    const double* vj = V + kr * D;
    double* dkj = dK + kr * D;
    double* dvj = dV + kr * D;
    for (int d = 0; d < D; ++d) { dkj[d] = 0.0; dvj[d] = 0.0; }
    for (int t = 0; t < rep; ++t) {
      const long h = g * rep + t;
      const long base = ((long)b * H + h) * Sq;
      for (long i = 0; i < Sq; ++i) {
        if (!visible(i, j, &s) || srow[base + i] == 0.0) continue;
        const double* qi = Q + (base + i) * D;
        const double* doi = dO + (base + i) * D;
        const double pij = exp(scale * dot(qi, kj, D) - mrow[base + i]) / srow[base + i];
        const double dpij = dot(doi, vj, D);
        const double ds = pij * (dpij - rrow[base + i]);
        for (int d = 0; d < D; ++d) {
          dkj[d] += ds * qi[d];
          dvj[d] += pij * doi[d];
        }
      }
    }
    for (int d = 0; d < D; ++d) dkj[d] *= scale;
  }
  free(mrow);
  free(srow);
  free(rrow);
  return fail ? -2 : 0;
}
