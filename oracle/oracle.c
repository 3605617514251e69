/*
 * Plain fp64 CPU oracle for the DeepSeek-sparse-attention lightning-indexer
 * backward.  TEST INFRASTRUCTURE ONLY: nothing on the product path may call,
 * link or load this file.  It shares no code with the CUDA library.
 *
 * Sources (cudnn-frontend pull-request pages):
 *   [P2] "dsa(indexer_backward): optimize SM100 gradient kernels - #730":
 *        walkthrough (kernel 1 writes the grad signal over attn_score and keeps
 *        index_score), benchmark-harness comment (fixture; ref_grads, the fp64
 *        chunked reference of the gemm_only semantics; the -1 / positive
 *        out-of-range padding-equivalence check).
 *   [P1] "dsa(indexer_backward): restore range_constexpr in 8 kernel_gemm
 *        epilogue loops - #549": kernel names and outputs (kernel_score_grad,
 *        kernel_gemm -> d_index_q, d_weights, d_index_k).
 *
 * Notation: t = query row, h = indexer head, j = slot in the row,
 * s = idx[t,j].  A slot is valid iff 0 <= s < S_k; every other id (-1 or a
 * positive out-of-range id) is padding and contributes nothing ([P2] harness,
 * padding-equivalence check).  Ids are local to their batch.
 *
 *   forward:    z[t,j,h] = sm_scale * (q[t,h,:] . k[s,:]);
 *               I[t,j] = sum_h w[t,h] relu(z)
 *   score-grad: p = softmax over valid j of I[t,:];  ahat = a / sum_valid a;
 *               dI[t,j] = grad_scale * (p_j - ahat_j) / S_q   (0 if invalid)
 *               -- the gradient of (grad_scale/S_q) sum_t KL(ahat_t || p_t);
 *               the pages name the inputs and the in-place output but print no
 *               formula, so this plain reading is taken.
 *   gemm stage: dW[t,h]  = sum_j dI relu(z)
 *               dz       = dI w[t,h] [z > 0] sm_scale
 *               dQ[t,h]  = sum_j dz k[s]
 *               dK[s]   += sum_{t,h} dz q[t,h]
 *               ([P2] ref_grads, with sm_scale = 1; the ReLU derivative at
 *               z = 0 is taken as 0, as the strict comparison there states.)
 *   sm_scale:   the logit scale of the [P2] harness, which runs with
 *               sm_scale = 1.0 and calls the kernel's scaling a runtime fold
 *               that is then a no-op.  Read as a factor inside the ReLU, the
 *               plain reading; dz is the chain rule through it.  For
 *               sm_scale > 0, relu(s x) = s relu(x), so I, dW, dQ and dK all
 *               scale by s; sm_scale = 1 gives the unscaled definitions
 *               exactly.
 *
 * Dense variant: every key s <= t is selected (S_q == S_k); scores are
 * indexed [t, s] and entries with s > t are zero.
 *
 * Layouts (row-major, contiguous): q [B,S_q,H,D] bf16 bits, k [B,S_k,D] bf16
 * bits, w [B,S_q,H] fp32, idx [B,S_q,topk] int32, scores [B,S_q,topk] fp32
 * (dense: [B,S,S]).  All arithmetic is in double; bf16 and fp32 inputs convert
 * to double exactly.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static int slot_valid(int32_t s, int S_k) { return s >= 0 && s < S_k; }

/* q or k as doubles (a plain exact widening). */
static double *widen_bf16(const uint16_t *x, size_t n) {
  double *y = (double *)malloc(n * sizeof(double));
  if (!y) return NULL;
  for (size_t i = 0; i < n; i++) y[i] = bf16_to_double(x[i]);
  return y;
}

static double dot(const double *a, const double *b, int n) {
  double s = 0.0;
  for (int i = 0; i < n; i++) s += a[i] * b[i];
  return s;
}

int oracle_set_threads(int n) {
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
}

/* ---------------------------------------------------------------- forward */

/* I[b,t,j] = sum_h w[b,t,h] * relu(q[b,t,h,:] . k[b,idx,:]) for valid slots,
 * 0 for padding.  The forward the backward recomputes ([P2] ref_grads builds
 * s = einsum(q, k_sel) the same way). */
int oracle_forward_sparse(const uint16_t *q16, const uint16_t *k16, const float *w,
                          const int32_t *idx, int B, int S_q, int S_k, int H, int D,
                          int topk, double sm_scale, double *I) {
  double *q = widen_bf16(q16, (size_t)B * S_q * H * D);
  double *k = widen_bf16(k16, (size_t)B * S_k * D);
  if (!q || !k) { free(q); free(k); return 1; }
  int64_t rows = (int64_t)B * S_q;
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t r = 0; r < rows; r++) {
    int64_t b = r / S_q;
    const double *qr = q + r * H * D;
    for (int j = 0; j < topk; j++) {
      int32_t s = idx[r * topk + j];
      double acc = 0.0;
      if (slot_valid(s, S_k)) {
        const double *kr = k + (b * S_k + s) * D;
        for (int h = 0; h < H; h++) {
          double z = sm_scale * dot(qr + (int64_t)h * D, kr, D);
          if (z > 0.0) acc += (double)w[r * H + h] * z;
        }
      }
      I[r * topk + j] = acc;
    }
  }
  free(q);
  free(k);
  return 0;
}

/* ------------------------------------------------------------- score-grad */

/* One row of the score-grad: n slots, validity given by valid[]. */
static void score_grad_row(const float *I, const float *a, const unsigned char *valid,
                           int n, double scale, double *dI) {
  double m = -INFINITY;
  double A = 0.0;
  int nv = 0;
  for (int j = 0; j < n; j++) {
    if (!valid[j]) continue;
    nv++;
    if ((double)I[j] > m) m = (double)I[j];
    A += (double)a[j];
  }
  if (nv == 0) {
    for (int j = 0; j < n; j++) dI[j] = 0.0;
    return;
  }
  double Z = 0.0;
  for (int j = 0; j < n; j++)
    if (valid[j]) Z += exp((double)I[j] - m);
  for (int j = 0; j < n; j++) {
    if (!valid[j]) { dI[j] = 0.0; continue; }
    double p = exp((double)I[j] - m) / Z;
    double ahat = (A != 0.0) ? (double)a[j] / A : 0.0;
    dI[j] = scale * (p - ahat);
  }
}

/* dI[b,t,j] = grad_scale * (softmax_valid(I[b,t,:])_j - a_j / sum_valid a) / S_q.
 * Kernel 1 of [P2] (walkthrough: the grad signal is written over attn_score,
 * index_score is left intact); [P1] names it kernel_score_grad. */
int oracle_score_grad_sparse(const float *index_score, const float *attn_score,
                             const int32_t *idx, int B, int S_q, int S_k, int topk,
                             double grad_scale, double *dI) {
  int64_t rows = (int64_t)B * S_q;
  double scale = grad_scale / (double)S_q;
  int bad = 0;
#pragma omp parallel
  {
    unsigned char *valid = (unsigned char *)malloc((size_t)topk);
    if (!valid) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(static)
      for (int64_t r = 0; r < rows; r++) {
        for (int j = 0; j < topk; j++) valid[j] = (unsigned char)slot_valid(idx[r * topk + j], S_k);
        score_grad_row(index_score + r * topk, attn_score + r * topk, valid, topk, scale,
                       dI + r * topk);
      }
      free(valid);
    }
  }
  return bad;
}

/* Dense rows: slot s of row t is valid iff s <= t. */
int oracle_score_grad_dense(const float *index_score, const float *attn_score, int B, int S,
                            double grad_scale, double *dI) {
  int64_t rows = (int64_t)B * S;
  double scale = grad_scale / (double)S;
  int bad = 0;
#pragma omp parallel
  {
    unsigned char *valid = (unsigned char *)malloc((size_t)S);
    if (!valid) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(static)
      for (int64_t r = 0; r < rows; r++) {
        int64_t t = r % S;
        for (int s = 0; s < S; s++) valid[s] = (unsigned char)(s <= t);
        score_grad_row(index_score + r * S, attn_score + r * S, valid, S, scale, dI + r * S);
      }
      free(valid);
    }
  }
  return bad;
}

/* -------------------------------------------------------------- gemm stage */

/* One query row of the gemm stage over an explicit key list.
 * keys[j] < 0 marks padding.  Accumulates dQ/dW for the row and, when dk is
 * non-NULL, the row's dK contribution into dk (a per-thread partial). */
static void gemm_row(const double *qr, const double *kb, const float *wr, const double *dIr,
                     const int32_t *keys, int n, int H, int D, double sm_scale, double *dqr,
                     double *dwr, double *dk) {
  for (int h = 0; h < H; h++) {
    dwr[h] = 0.0;
    for (int d = 0; d < D; d++) dqr[(int64_t)h * D + d] = 0.0;
  }
  for (int j = 0; j < n; j++) {
    int32_t s = keys[j];
    if (s < 0) continue;
    const double *kr = kb + (int64_t)s * D;
    double g = dIr[j];
    for (int h = 0; h < H; h++) {
      const double *qh = qr + (int64_t)h * D;
      double z = sm_scale * dot(qh, kr, D);
      if (!(z > 0.0)) continue;            /* relu(z) = 0 and [z > 0] = 0 */
      dwr[h] += g * z;                     /* dW += dI * relu(z) */
      double dz = g * (double)wr[h] * sm_scale;  /* dz = dI w [z > 0] sm_scale */
      double *dqh = dqr + (int64_t)h * D;
      for (int d = 0; d < D; d++) dqh[d] += dz * kr[d];  /* dQ[t,h] += dz k[s] */
      if (dk) {
        double *dks = dk + (int64_t)s * D;
        for (int d = 0; d < D; d++) dks[d] += dz * qh[d];  /* dK[s] += dz q[t,h] */
      }
    }
  }
}

/* Sums per-thread dK partials in thread order 0..n-1 (fixed order). */
static void sum_partials(double *dk, double *part, int nth, size_t n) {
  for (size_t i = 0; i < n; i++) dk[i] = 0.0;
  for (int th = 0; th < nth; th++)
    for (size_t i = 0; i < n; i++) dk[i] += part[(size_t)th * n + i];
}

/* Kernel 2 (kernel_gemm) of [P1]/[P2]: dQ, dW, dK from the grad signal dI.
 * [P2] ref_grads is the fp64 definition followed here, written as loops. */
int oracle_gemm_sparse(const uint16_t *q16, const uint16_t *k16, const float *w,
                       const double *dI, const int32_t *idx, int B, int S_q, int S_k,
                       int H, int D, int topk, double sm_scale, double *dq, double *dw,
                       double *dk) {
  double *q = widen_bf16(q16, (size_t)B * S_q * H * D);
  double *k = widen_bf16(k16, (size_t)B * S_k * D);
  int nth = omp_get_max_threads();
  size_t dkn = (size_t)B * S_k * D;
  double *part = (double *)calloc((size_t)nth * dkn, sizeof(double));
  if (!q || !k || !part) { free(q); free(k); free(part); return 1; }
  int64_t rows = (int64_t)B * S_q;
  int bad = 0;
#pragma omp parallel num_threads(nth)
  {
    int th = omp_get_thread_num();
    int32_t *keys = (int32_t *)malloc((size_t)topk * sizeof(int32_t));
    if (!keys) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(static)
      for (int64_t r = 0; r < rows; r++) {
        int64_t b = r / S_q;
        for (int j = 0; j < topk; j++) {
          int32_t s = idx[r * topk + j];
          keys[j] = slot_valid(s, S_k) ? s : -1;
        }
        gemm_row(q + r * H * D, k + b * S_k * D, w + r * H, dI + r * topk, keys, topk, H, D,
                 sm_scale, dq + r * H * D, dw + r * H, part + (size_t)th * dkn + (size_t)b * S_k * D);
      }
      free(keys);
    }
  }
  sum_partials(dk, part, nth, dkn);
  free(part);
  free(q);
  free(k);
  return bad;
}

/* dQ and dW for a list of global rows r = b*S_q + t only (no dK): lets a test
 * check sampled rows of a full-size problem one by one. */
int oracle_gemm_sparse_rows(const uint16_t *q16, const uint16_t *k16, const float *w,
                            const double *dI_rows, const int32_t *idx, int B, int S_q, int S_k,
                            int H, int D, int topk, double sm_scale, const int64_t *rows,
                            int nrows, double *dq, double *dw) {
  (void)B;
  int bad = 0;
#pragma omp parallel
  {
    double *qr = (double *)malloc((size_t)H * D * sizeof(double));
    double *kr = (double *)malloc((size_t)topk * D * sizeof(double));
    int32_t *keys = (int32_t *)malloc((size_t)topk * sizeof(int32_t));
    if (!qr || !kr || !keys) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int i = 0; i < nrows; i++) {
        int64_t r = rows[i];
        int64_t b = r / S_q;
        for (int x = 0; x < H * D; x++) qr[x] = bf16_to_double(q16[r * H * D + x]);
        /* Gather the selected key rows so gemm_row sees a compact key list. */
        for (int j = 0; j < topk; j++) {
          int32_t s = idx[r * topk + j];
          if (slot_valid(s, S_k)) {
            for (int d = 0; d < D; d++)
              kr[(int64_t)j * D + d] = bf16_to_double(k16[(b * S_k + s) * D + d]);
            keys[j] = j;
          } else {
            keys[j] = -1;
          }
        }
        gemm_row(qr, kr, w + r * H, dI_rows + (int64_t)i * topk, keys, topk, H, D, sm_scale,
                 dq + (int64_t)i * H * D, dw + (int64_t)i * H, NULL);
      }
    }
    free(qr);
    free(kr);
    free(keys);
  }
  return bad;
}

/* Dense forward: I[b,t,s] for s <= t, 0 above the diagonal. */
int oracle_forward_dense(const uint16_t *q16, const uint16_t *k16, const float *w, int B, int S,
                         int H, int D, double sm_scale, double *I) {
  double *q = widen_bf16(q16, (size_t)B * S * H * D);
  double *k = widen_bf16(k16, (size_t)B * S * D);
  if (!q || !k) { free(q); free(k); return 1; }
  int64_t rows = (int64_t)B * S;
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t r = 0; r < rows; r++) {
    int64_t b = r / S, t = r % S;
    for (int s = 0; s < S; s++) {
      double acc = 0.0;
      if (s <= t) {
        const double *kr = k + (b * S + s) * D;
        for (int h = 0; h < H; h++) {
          double z = sm_scale * dot(q + r * H * D + (int64_t)h * D, kr, D);
          if (z > 0.0) acc += (double)w[r * H + h] * z;
        }
      }
      I[r * S + s] = acc;
    }
  }
  free(q);
  free(k);
  return 0;
}

/* Dense gemm stage: every causal key s <= t is selected; dI is [B,S,S]. */
int oracle_gemm_dense(const uint16_t *q16, const uint16_t *k16, const float *w, const double *dI,
                      int B, int S, int H, int D, double sm_scale, double *dq, double *dw,
                      double *dk) {
  double *q = widen_bf16(q16, (size_t)B * S * H * D);
  double *k = widen_bf16(k16, (size_t)B * S * D);
  int nth = omp_get_max_threads();
  size_t dkn = (size_t)B * S * D;
  double *part = (double *)calloc((size_t)nth * dkn, sizeof(double));
  if (!q || !k || !part) { free(q); free(k); free(part); return 1; }
  int64_t rows = (int64_t)B * S;
  int bad = 0;
#pragma omp parallel num_threads(nth)
  {
    int th = omp_get_thread_num();
    int32_t *keys = (int32_t *)malloc((size_t)S * sizeof(int32_t));
    if (!keys) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(static)
      for (int64_t r = 0; r < rows; r++) {
        int64_t b = r / S, t = r % S;
        for (int s = 0; s < S; s++) keys[s] = (s <= t) ? s : -1;
        gemm_row(q + r * H * D, k + b * S * D, w + r * H, dI + r * S, keys, S, H, D, sm_scale,
                 dq + r * H * D, dw + r * H, part + (size_t)th * dkn + (size_t)b * S * D);
      }
      free(keys);
    }
  }
  sum_partials(dk, part, nth, dkn);
  free(part);
  free(q);
  free(k);
  return bad;
}

/* Dense dQ/dW for a list of global rows only. */
int oracle_gemm_dense_rows(const uint16_t *q16, const uint16_t *k16, const float *w,
                           const double *dI_rows, int B, int S, int H, int D, double sm_scale,
                           const int64_t *rows, int nrows, double *dq, double *dw) {
  (void)B;
  int bad = 0;
#pragma omp parallel
  {
    double *qr = (double *)malloc((size_t)H * D * sizeof(double));
    double *kb = (double *)malloc((size_t)S * D * sizeof(double));
    int32_t *keys = (int32_t *)malloc((size_t)S * sizeof(int32_t));
    if (!qr || !kb || !keys) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int i = 0; i < nrows; i++) {
        int64_t r = rows[i];
        int64_t b = r / S, t = r % S;
        for (int x = 0; x < H * D; x++) qr[x] = bf16_to_double(q16[r * H * D + x]);
        for (int64_t x = 0; x < (int64_t)S * D; x++) kb[x] = bf16_to_double(k16[b * S * D + x]);
        for (int s = 0; s < S; s++) keys[s] = (s <= t) ? s : -1;
        gemm_row(qr, kb, w + r * H, dI_rows + (int64_t)i * S, keys, S, H, D, sm_scale,
                 dq + (int64_t)i * H * D, dw + (int64_t)i * H, NULL);
      }
    }
    free(qr);
    free(kb);
    free(keys);
  }
  return bad;
}
