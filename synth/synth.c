/*
 * Seeded synthetic inputs for the indexer backward.  Shared by the tests, the
 * benchmark and the oracle's callers; it holds none of the method's
 * arithmetic (no forward, no score-grad, no gradients).
 *
 * Random numbers come from one counter-based generator: value(seed, stream,
 * counter) = splitmix64-finalizer(seed * C1 + stream * C2 + counter), with the
 * SplitMix64 constants of Steele, Lea and Flood ("Fast splittable
 * pseudorandom number generators", OOPSLA 2014) as used in Vigna's
 * splitmix64.c.  Every array draws from its own stream, so a value depends
 * only on (seed, stream, position) and not on threading or call order.
 *
 * Distributions (the fixture of the cudnn-frontend #730 benchmark harness and
 * the workloads it sweeps):
 *   normal        Box-Muller on two 53-bit uniforms;
 *   bf16          round-to-nearest-even from the fp32 value;
 *   topk ids      distinct uniform causal keys in [0, c(t)], c(t) =
 *                 floor(t*S_k/S_q), in random order (Floyd's sampling, then a
 *                 Fisher-Yates shuffle), -1 padding at the tail when the row
 *                 has fewer than topk causal keys;
 *   window ids    half of the slots drawn with replacement from the last
 *                 `window` causal keys, the rest distinct uniform from the keys
 *                 before the window, shuffled;
 *   target        normalised exp of N(0, var) logits over the valid slots,
 *                 0 on padded slots (a probability row).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static uint64_t mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t synth_u64(uint64_t seed, uint64_t stream, uint64_t ctr) {
  return mix64(seed * 0xD1B54A32D192ED03ull + stream * 0xABC98388FB8FAC03ull + ctr);
}

/* uniform in (0, 1]: never 0, so log() is finite */
static double unit_open0(uint64_t x) { return ((double)(x >> 11) + 1.0) * (1.0 / 9007199254740992.0); }
/* uniform in [0, 1) */
static double unit(uint64_t x) { return (double)(x >> 11) * (1.0 / 9007199254740992.0); }

/* uniform integer in [0, n) by the multiply-high method */
static uint64_t below(uint64_t x, uint64_t n) { return (uint64_t)(((unsigned __int128)x * n) >> 64); }

static double normal_at(uint64_t seed, uint64_t stream, uint64_t i) {
  double u1 = unit_open0(synth_u64(seed, stream, 2 * i));
  double u2 = unit(synth_u64(seed, stream, 2 * i + 1));
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

void synth_normal_f32(uint64_t seed, uint64_t stream, int64_t n, double mean, double std, float *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++) out[i] = (float)(mean + std * normal_at(seed, stream, (uint64_t)i));
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, int64_t n, double mean, double std, uint16_t *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++)
    out[i] = f32_to_bf16_rne((float)(mean + std * normal_at(seed, stream, (uint64_t)i)));
}

static int64_t causal_last(int64_t t, int64_t S_q, int64_t S_k) {
  int64_t c = (t * S_k) / S_q;
  return c < S_k - 1 ? c : S_k - 1;
}

/* Floyd's algorithm: m distinct values from [lo, lo+n) into out[0..m), using a
 * scratch bitmap of n bits; draws come from counters ctr, ctr+1, ... */
static void floyd(uint64_t seed, uint64_t stream, uint64_t ctr, int64_t lo, int64_t n, int64_t m,
                  unsigned char *seen, int32_t *out) {
  memset(seen, 0, (size_t)n);
  int64_t cnt = 0;
  for (int64_t jj = n - m; jj < n; jj++) {
    int64_t r = (int64_t)below(synth_u64(seed, stream, ctr++), (uint64_t)(jj + 1));
    int64_t pick = seen[r] ? jj : r;
    seen[pick] = 1;
    out[cnt++] = (int32_t)(lo + pick);
  }
}

static void shuffle(uint64_t seed, uint64_t stream, uint64_t ctr, int32_t *a, int64_t n) {
  for (int64_t i = n - 1; i > 0; i--) {
    int64_t j = (int64_t)below(synth_u64(seed, stream, ctr++), (uint64_t)(i + 1));
    int32_t tmp = a[i];
    a[i] = a[j];
    a[j] = tmp;
  }
}

/* Distinct ids per row in random order, -1 padding at the tail: from the
 * row's causal keys, or (uniform) from all S_k keys. */
static int topk_rows(uint64_t seed, uint64_t stream, int B, int S_q, int S_k, int topk, int uniform, int32_t *idx) {
  int64_t rows = (int64_t)B * S_q;
  int bad = 0;
#pragma omp parallel
  {
    unsigned char *seen = (unsigned char *)malloc((size_t)S_k);
    if (!seen) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (int64_t r = 0; r < rows; r++) {
        int64_t t = r % S_q;
        int64_t n = uniform ? S_k : causal_last(t, S_q, S_k) + 1;
        int64_t m = n < topk ? n : topk;
        int32_t *row = idx + r * topk;
        uint64_t base = (uint64_t)r << 24;
        floyd(seed, stream, base, 0, n, m, seen, row);
        shuffle(seed, stream, base + (1u << 23), row, m);
        for (int64_t j = m; j < topk; j++) row[j] = -1;
      }
      free(seen);
    }
  }
  return bad;
}

int synth_topk_causal(uint64_t seed, uint64_t stream, int B, int S_q, int S_k, int topk, int32_t *idx) {
  return topk_rows(seed, stream, B, S_q, S_k, topk, 0, idx);
}

/* Every row: min(topk, S_k) distinct ids drawn from all S_k keys. */
int synth_topk_uniform(uint64_t seed, uint64_t stream, int B, int S_q, int S_k, int topk, int32_t *idx) {
  return topk_rows(seed, stream, B, S_q, S_k, topk, 1, idx);
}

/* Local-window ids: rows with more than topk causal keys take topk/2 slots
 * with replacement from the last `window` causal keys and the rest distinct
 * from the keys before the window; shorter rows take every causal key. */
int synth_topk_window(uint64_t seed, uint64_t stream, int B, int S_q, int S_k, int topk, int window,
                      int32_t *idx) {
  int64_t rows = (int64_t)B * S_q;
  int bad = 0;
#pragma omp parallel
  {
    unsigned char *seen = (unsigned char *)malloc((size_t)S_k);
    if (!seen) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (int64_t r = 0; r < rows; r++) {
        int64_t t = r % S_q;
        int64_t c = causal_last(t, S_q, S_k);
        int64_t n = c + 1;
        int32_t *row = idx + r * topk;
        uint64_t base = (uint64_t)r << 24;
        if (n <= topk) {
          floyd(seed, stream, base, 0, n, n, seen, row);
          shuffle(seed, stream, base + (1u << 23), row, n);
          for (int64_t j = n; j < topk; j++) row[j] = -1;
          continue;
        }
        int64_t wlo = c - window + 1;
        if (wlo < 0) wlo = 0;
        int64_t before = wlo;                 /* keys [0, wlo) lie before the window */
        int64_t m_out = topk - topk / 2;      /* distinct picks outside the window */
        if (m_out > before) m_out = before;
        int64_t m_in = topk - m_out;          /* with-replacement picks inside it */
        floyd(seed, stream, base, 0, before, m_out, seen, row);
        for (int64_t j = 0; j < m_in; j++)
          row[m_out + j] = (int32_t)(wlo + (int64_t)below(synth_u64(seed, stream, base + (1u << 22) + j),
                                                         (uint64_t)(c - wlo + 1)));
        shuffle(seed, stream, base + (1u << 23), row, topk);
      }
      free(seen);
    }
  }
  return bad;
}

/* Target distribution per row: exp(logit) / sum over valid slots, logits
 * N(0, var); padded slots get 0.  valid(j) iff 0 <= idx < S_k. */
int synth_target_sparse(uint64_t seed, uint64_t stream, const int32_t *idx, int B, int S_q, int S_k,
                        int topk, double var, float *out) {
  int64_t rows = (int64_t)B * S_q;
  double sd = sqrt(var);
  int bad = 0;
#pragma omp parallel
  {
    double *e = (double *)malloc((size_t)topk * sizeof(double));
    if (!e) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(static)
      for (int64_t r = 0; r < rows; r++) {
        double m = -INFINITY, sum = 0.0;
        for (int j = 0; j < topk; j++) {
          e[j] = sd * normal_at(seed, stream, (uint64_t)(r * topk + j));
          int32_t s = idx[r * topk + j];
          if (s >= 0 && s < S_k && e[j] > m) m = e[j];
        }
        for (int j = 0; j < topk; j++) {
          int32_t s = idx[r * topk + j];
          e[j] = (s >= 0 && s < S_k) ? exp(e[j] - m) : 0.0;
          sum += e[j];
        }
        for (int j = 0; j < topk; j++) out[r * topk + j] = sum > 0.0 ? (float)(e[j] / sum) : 0.0f;
      }
      free(e);
    }
  }
  return bad;
}

/* Dense target rows: valid iff s <= t. */
int synth_target_dense(uint64_t seed, uint64_t stream, int B, int S, double var, float *out) {
  int64_t rows = (int64_t)B * S;
  double sd = sqrt(var);
  int bad = 0;
#pragma omp parallel
  {
    double *e = (double *)malloc((size_t)S * sizeof(double));
    if (!e) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(static)
      for (int64_t r = 0; r < rows; r++) {
        int64_t t = r % S;
        double m = -INFINITY, sum = 0.0;
        for (int s = 0; s <= t; s++) {
          e[s] = sd * normal_at(seed, stream, (uint64_t)(r * S + s));
          if (e[s] > m) m = e[s];
        }
        for (int s = 0; s <= t; s++) {
          e[s] = exp(e[s] - m);
          sum += e[s];
        }
        for (int s = 0; s < S; s++) out[r * S + s] = (s <= t) ? (float)(e[s] / sum) : 0.0f;
      }
      free(e);
    }
  }
  return bad;
}
