/*
 * Float64 CPU oracle for tree-verify MLA attention over a page_size=1 latent KV pool.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library's product path may include,
 * link or call this file; only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg use it. It shares no code, header, table or
 * constant with the CUDA library.
 *
 * What it computes (plain definition, no blocking, no split, no online softmax):
 * for every sequence b, tree node i < T and head h, the query row
 * q[(b*T + i)*H + h][0:576] attends to the visible token set
 *
 *   V(b, i) = { t : 0 <= t < L_b }  U  { L_b + j : j in anc*(i) }
 *
 * where L_b = seq_lens[b] is the prefix length and anc*(i) is node i followed by
 * its parent chain up to -1. Token t's latent row is kv[slot_table[b][t]][0:576]
 * (page_size=1: one token per slot, any slot for any token). With
 * s_t = scale * <q, k_t> over all 576 dims and v_t = k_t[0:512]:
 *
 *   m = max_t s_t,  Z = sum_t exp(s_t - m),  out = sum_t exp(s_t - m) v_t / Z,
 *   lse = m + ln Z.
 *
 * Passages followed (page title, section):
 *  - "The Moment of Certainty", The Final Piece / The Path Forward: the verify step
 *    checks the draft tree against the whole cache; the prefix needs no mask and
 *    only the small tree block takes the custom visibility mask.
 *  - "The GPU That Wasn't There", The Native Engine Thesis: a tree visibility
 *    bitmask over the draft block; the prefix part needs no masking.
 *  - "Diagnosing Latency-Bound Decode", The Technical Depth: MLA keeps one
 *    compressed latent row per token; page_size=1 gives each token its own page
 *    and the kernel gathers them one by one (The Reasoning, Step 4).
 *  - The pages give no dimensions: the row is 512 latent + 64 RoPE dims, V is
 *    the first 512 dims of the same row, scale 1/sqrt(192) (absorbed MLA form).
 *
 * Inputs are the exact bf16 bit patterns (uint16), widened exactly to double.
 * Build: gcc -O2 -fopenmp -shared -fPIC (no -ffast-math: the order of every sum
 * is the plain loop order).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Planted-mistake builds for the pin tests (default 0 = the oracle as defined).
 * Each nonzero value compiles one plausible mistake, so the tests can show that
 * their pins reject it: 1 node not visible to itself, 2 RoPE dims dropped from
 * the score, 3 values read from the wrong columns, 4 every tree node visible,
 * 5 lse without the max term, 6 scale applied twice, 7 heads and nodes swapped
 * in the query row index. */
#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_TREE -2
#define ORACLE_ERR_SLOT -3
#define ORACLE_ERR_NOMEM -4

static double widen_bf16(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* anc*(i) as a bit set over node indices: node i itself plus every ancestor.
 * Requires parent[i] in [-1, i) (topological order), T <= 64. */
int oracle_ancestor_masks(int32_t T, const int32_t *parent, uint64_t *mask) {
  if (T < 1 || T > 64) return ORACLE_ERR_ARG;
  for (int32_t i = 0; i < T; ++i) {
    int32_t p = parent[i];
    if (p < -1 || p >= i) return ORACLE_ERR_TREE;
    mask[i] = ((uint64_t)1 << i) | (p >= 0 ? mask[p] : 0);
#if ORACLE_MUTATION == 1
    mask[i] = (p >= 0 ? (((uint64_t)1 << p) | mask[p]) : 0);
#endif
  }
  return ORACLE_OK;
}

/* Is logical position t visible to node i of a sequence with prefix L? */
static int visible(int64_t t, int64_t L, int32_t T, uint64_t anc_i) {
  if (t < L) return 1;
#if ORACLE_MUTATION == 4
  (void)anc_i;
  if (t < L + T) return 1;
#endif
  if (t < L + T) return (int)((anc_i >> (t - L)) & 1u);
  return 0;
}

typedef struct {
  int32_t B, T, H, d_latent, d_rope;
  const int32_t *seq_lens, *slot_table, *tree_parent;
  int64_t stride, num_slots;
  const uint16_t *q, *kv;
  double scale;
  int64_t pos_begin, pos_end; /* only positions in [pos_begin, pos_end) take part */
} problem_t;

/* One query row: out[0:d_latent] and lse; weights (optional) per logical position. */
static int one_row(const problem_t *P, const uint64_t *masks, int64_t row, double *out,
                   double *lse, double *weights, double *scores) {
  const int32_t dk = P->d_latent + P->d_rope;
  const int32_t dv = P->d_latent;
  const int64_t bi = row / P->H; /* b*T + i */
  const int32_t b = (int32_t)(bi / P->T);
  const int32_t i = (int32_t)(bi % P->T);
  const int64_t L = P->seq_lens[b];
  const int64_t N = L + P->T;
  const uint64_t anc = masks[(int64_t)b * P->T + i];
#if ORACLE_MUTATION == 7
  const uint16_t *qr = P->q + (((int64_t)b * P->H + row % P->H) * P->T + i) * dk;
#else
  const uint16_t *qr = P->q + row * dk;
#endif
  const int32_t *tab = P->slot_table + (int64_t)b * P->stride;

  /* pass 1: scores of visible tokens, and their maximum */
  double m = -INFINITY;
  for (int64_t t = 0; t < N; ++t) {
    scores[t] = -INFINITY;
    if (t < P->pos_begin || t >= P->pos_end || !visible(t, L, P->T, anc)) continue;
    int64_t slot = tab[t];
    if (slot < 0 || slot >= P->num_slots) return ORACLE_ERR_SLOT;
    const uint16_t *k = P->kv + slot * dk;
    double dot = 0.0;
#if ORACLE_MUTATION == 2
    for (int32_t d = 0; d < P->d_latent; ++d) dot += widen_bf16(qr[d]) * widen_bf16(k[d]);
#else
    for (int32_t d = 0; d < dk; ++d) dot += widen_bf16(qr[d]) * widen_bf16(k[d]);
#endif
    scores[t] = P->scale * dot;
#if ORACLE_MUTATION == 6
    scores[t] *= P->scale;
#endif
    if (scores[t] > m) m = scores[t];
  }
  for (int32_t d = 0; d < dv; ++d) out[d] = 0.0;
  if (m == -INFINITY) { /* nothing visible in the window */
    *lse = -INFINITY;
    if (weights)
      for (int64_t t = 0; t < N; ++t) weights[t] = 0.0;
    return ORACLE_OK;
  }
  /* pass 2: Z and the unnormalised weighted sum of values */
  double Z = 0.0;
  for (int64_t t = 0; t < N; ++t) {
    if (scores[t] == -INFINITY) continue;
    double e = exp(scores[t] - m);
    Z += e;
#if ORACLE_MUTATION == 3
    const uint16_t *v = P->kv + (int64_t)tab[t] * dk + P->d_rope;
#else
    const uint16_t *v = P->kv + (int64_t)tab[t] * dk;
#endif
    for (int32_t d = 0; d < dv; ++d) out[d] += e * widen_bf16(v[d]);
  }
  for (int32_t d = 0; d < dv; ++d) out[d] /= Z;
  *lse = m + log(Z);
#if ORACLE_MUTATION == 5
  *lse = log(Z);
#endif
  if (weights)
    for (int64_t t = 0; t < N; ++t) weights[t] = scores[t] == -INFINITY ? 0.0 : exp(scores[t] - m) / Z;
  return ORACLE_OK;
}

static int build_masks(const problem_t *P, uint64_t *masks) {
  for (int32_t b = 0; b < P->B; ++b) {
    int rc = oracle_ancestor_masks(P->T, P->tree_parent + (int64_t)b * P->T, masks + (int64_t)b * P->T);
    if (rc) return rc;
  }
  return ORACLE_OK;
}

/*
 * Exact attention for the listed rows (rows == NULL: all B*T*H rows, in order).
 * out: [num_rows, d_latent] float64; lse: [num_rows] float64.
 * Only positions in [pos_begin, pos_end) take part (pass 0, INT64_MAX for the
 * whole visible set); rows with nothing visible get lse = -inf and out = 0.
 */
int oracle_verify(int32_t B, int32_t T, int32_t H, int32_t d_latent, int32_t d_rope,
                  const int32_t *seq_lens, const int32_t *slot_table, int64_t stride,
                  const int32_t *tree_parent, const uint16_t *q, const uint16_t *kv,
                  int64_t num_slots, double scale, const int64_t *rows, int64_t num_rows,
                  int64_t pos_begin, int64_t pos_end, double *out, double *lse,
                  int32_t num_threads) {
  if (B < 1 || T < 1 || T > 64 || H < 1 || d_latent < 1 || d_rope < 0) return ORACLE_ERR_ARG;
  problem_t P = {B, T, H, d_latent, d_rope, seq_lens, slot_table, tree_parent, stride, num_slots,
                 q, kv, scale, pos_begin, pos_end};
  int64_t max_N = 0;
  for (int32_t b = 0; b < B; ++b) {
    if (seq_lens[b] < 0 || (int64_t)seq_lens[b] + T > stride) return ORACLE_ERR_ARG;
    if ((int64_t)seq_lens[b] + T > max_N) max_N = (int64_t)seq_lens[b] + T;
  }
  uint64_t *masks = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)B * T);
  if (!masks) return ORACLE_ERR_NOMEM;
  int rc = build_masks(&P, masks);
  if (rc) { free(masks); return rc; }
  const int64_t total = rows ? num_rows : (int64_t)B * T * H;
  int err = ORACLE_OK;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#else
  (void)num_threads;
#endif
#pragma omp parallel
  {
    double *scores = (double *)malloc(sizeof(double) * (size_t)max_N);
    if (!scores) {
#pragma omp atomic write
      err = ORACLE_ERR_NOMEM;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t n = 0; n < total; ++n) {
      if (!scores) continue;
      int64_t row = rows ? rows[n] : n;
      if (row < 0 || row >= (int64_t)B * T * H) {
#pragma omp atomic write
        err = ORACLE_ERR_ARG;
        continue;
      }
      int r = one_row(&P, masks, row, out + n * d_latent, lse + n, NULL, scores);
      if (r) {
#pragma omp atomic write
        err = r;
      }
    }
    free(scores);
  }
  free(masks);
  return err;
}

/* Softmax weights of one row over logical positions 0..N_b-1 (0 where invisible). */
int oracle_row_weights(int32_t B, int32_t T, int32_t H, int32_t d_latent, int32_t d_rope,
                       const int32_t *seq_lens, const int32_t *slot_table, int64_t stride,
                       const int32_t *tree_parent, const uint16_t *q, const uint16_t *kv,
                       int64_t num_slots, double scale, int64_t row, double *weights) {
  problem_t P = {B, T, H, d_latent, d_rope, seq_lens, slot_table, tree_parent, stride, num_slots,
                 q, kv, scale, 0, INT64_MAX};
  if (row < 0 || row >= (int64_t)B * T * H) return ORACLE_ERR_ARG;
  uint64_t *masks = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)B * T);
  if (!masks) return ORACLE_ERR_NOMEM;
  int rc = build_masks(&P, masks);
  if (rc) { free(masks); return rc; }
  int32_t b = (int32_t)(row / H / T);
  int64_t N = (int64_t)seq_lens[b] + T;
  double *scores = (double *)malloc(sizeof(double) * (size_t)N);
  double *out = (double *)malloc(sizeof(double) * (size_t)d_latent);
  double lse;
  rc = (scores && out) ? one_row(&P, masks, row, out, &lse, weights, scores) : ORACLE_ERR_NOMEM;
  free(scores);
  free(out);
  free(masks);
  return rc;
}

/*
 * Merge S partial results of the same rows, each normalised over its own part
 * of the visible set: lse = ln sum_s exp(lse_s); out = sum_s exp(lse_s - lse) o_s.
 * Parts with lse_s = -inf carry no weight. part_o: [S, rows, d_v]; part_lse: [S, rows].
 */
int oracle_combine(int32_t S, int64_t rows, int32_t d_v, const double *part_o,
                   const double *part_lse, double *out, double *lse) {
  if (S < 1 || rows < 0 || d_v < 1) return ORACLE_ERR_ARG;
  for (int64_t r = 0; r < rows; ++r) {
    double m = -INFINITY;
    for (int32_t s = 0; s < S; ++s)
      if (part_lse[s * rows + r] > m) m = part_lse[s * rows + r];
    for (int32_t d = 0; d < d_v; ++d) out[r * d_v + d] = 0.0;
    if (m == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double Z = 0.0;
    for (int32_t s = 0; s < S; ++s) Z += exp(part_lse[s * rows + r] - m);
    lse[r] = m + log(Z);
    for (int32_t s = 0; s < S; ++s) {
      double w = exp(part_lse[s * rows + r] - lse[r]);
      if (w == 0.0) continue;
      for (int32_t d = 0; d < d_v; ++d) out[r * d_v + d] += w * part_o[((int64_t)s * rows + r) * d_v + d];
    }
  }
  return ORACLE_OK;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
