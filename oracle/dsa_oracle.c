/*
 * dsa_oracle.c -- plain CPU oracle for the DSA indexer's sparse index
 * selection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: it is used by tests/ and by the CPU legs of bench.py.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * Source: "onnx-runtime-ep-cuda 0.1.0-dev.6, src/kernels/dsa_index_select.rs",
 * module doc (the op: head-weighted, ReLU'd, scaled dot products plus the
 * additive f32 bias; allowed iff bias > -1e30; the top min(#allowed, top_k)
 * positions by (score desc, index asc); emitted ascending by position and
 * right-padded with -1; NaN canonicalised to the positive quiet NaN before
 * ordering; ordering is f32 total order) and the score kernel's stated
 * arithmetic (fp32, multiply and add each rounded separately, the dot product
 * over head_dim ascending, then the weighted sum over heads ascending).
 *
 * The page fixes the precision (fp32, in that order) because its output is
 * an index set: the oracle therefore computes in fp32 exactly as stated, and
 * must be compiled without floating-point contraction (-ffp-contract=off).
 *
 * Shapes (row-major, contiguous), rows = B * S, row = b * S + s:
 *   query   [B, S, H, D]   f32 (16-bit inputs widened exactly)
 *   key     [B, T, D]      f32
 *   weights [B, S, H]      f32
 *   bias    [B, 1, S, T]   f32
 *   out     [B, 1, S, top_k] int64
 * For row (b, s) and key t:
 *   allowed = bias[row, t] > -1e30
 *   dot_h   = sum_{d ascending} q[row, h, d] * k[b, t, d]
 *   score   = (sum_{h ascending} max(scale * dot_h, 0) * (w[row, h] * weights_scale))
 *             + bias[row, t];   NaN -> +NaN (0x7fc00000)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Positive quiet NaN with no payload. */
static float canonical_nan(void) {
  const uint32_t bits = 0x7fc00000u;
  float f;
  memcpy(&f, &bits, sizeof f);
  return f;
}

/* Score of one (row, key) cell, in the page's fp32 order. */
static float cell_score(const float *q, const float *k, const float *w, float bias, int64_t H, int64_t D,
                        float scale, float weights_scale) {
  float weighted = 0.0f;
  for (int64_t h = 0; h < H; ++h) {
    float dot = 0.0f;
    for (int64_t d = 0; d < D; ++d) {
      const float prod = q[h * D + d] * k[d];
      dot = dot + prod;
    }
    float scored = scale * dot;
    scored = scored > 0.0f ? scored : 0.0f; /* ReLU; a NaN dot gives 0 */
    const float wprod = w[h] * weights_scale;
    const float term = scored * wprod;
    weighted = weighted + term;
  }
  float score = weighted + bias;
  if (isnan(score)) score = canonical_nan();
  return score;
}

/*
 * Scores and allowed flags of every cell: scores[row * T + t] (-inf where not
 * allowed), allowed[row * T + t] in {0, 1}.  Returns 0.
 */
int oracle_dsa_scores(const float *query, const float *key, const float *weights, const float *bias,
                      float *scores, unsigned char *allowed, int64_t B, int64_t S, int64_t H, int64_t D,
                      int64_t T, float scale, float weights_scale) {
  for (int64_t b = 0; b < B; ++b)
    for (int64_t s = 0; s < S; ++s) {
      const int64_t row = b * S + s;
      for (int64_t t = 0; t < T; ++t) {
        const float bt = bias[row * T + t];
        const int ok = bt > -1e30f;
        allowed[row * T + t] = (unsigned char)ok;
        scores[row * T + t] =
            ok ? cell_score(query + row * H * D, key + (b * T + t) * D, weights + row * H, bt, H, D, scale,
                            weights_scale)
               : -INFINITY;
      }
    }
  return 0;
}

/*
 * f32 total order (IEEE 754 totalOrder as Rust's f32::total_cmp defines
 * it): negative NaNs < -inf < negative numbers < -0 < +0 < positive numbers
 * < +inf < positive NaNs.  Returns -1, 0 or 1.  Written from the definition
 * (sign, class and magnitude), not from a bit transform.
 */
static int total_cmp(float a, float b) {
  const int na = isnan(a), nb = isnan(b);
  const int sa = signbit(a) != 0, sb = signbit(b) != 0;
  if (na || nb) {
    /* a NaN sits beyond every number on its sign's side */
    const int ra = na ? (sa ? -2 : 2) : 0;
    const int rb = nb ? (sb ? -2 : 2) : 0;
    if (ra != rb) return ra < rb ? -1 : 1;
    if (na && nb) {
      /* two NaNs of one sign: by payload magnitude, reversed when negative */
      uint32_t ia, ib;
      memcpy(&ia, &a, sizeof ia);
      memcpy(&ib, &b, sizeof ib);
      ia &= 0x7fffffffu;
      ib &= 0x7fffffffu;
      if (ia == ib) return 0;
      return ((ia < ib) != sa) ? -1 : 1;
    }
    return 0; /* unreachable: ra != rb when exactly one is NaN */
  }
  if (a < b) return -1;
  if (a > b) return 1;
  /* equal numerically: only the zeros differ in order */
  if (a == 0.0f && sa != sb) return sa ? -1 : 1;
  return 0;
}

typedef struct {
  float score;
  int64_t index;
} cand_t;

/* Descending score, then ascending index. */
static int cand_order(const void *x, const void *y) {
  const cand_t *a = (const cand_t *)x, *b = (const cand_t *)y;
  const int c = total_cmp(a->score, b->score);
  if (c != 0) return -c;
  return (a->index > b->index) - (a->index < b->index);
}

static int index_order(const void *x, const void *y) {
  const int64_t a = *(const int64_t *)x, b = *(const int64_t *)y;
  return (a > b) - (a < b);
}

/*
 * Selection of one row: the allowed keys sorted by (score desc, index asc),
 * the first min(#allowed, top_k) kept, emitted ascending, padded with -1.
 */
static int select_row(const float *scores, const unsigned char *allowed, int64_t T, int64_t top_k,
                      int64_t *out) {
  cand_t *c = (cand_t *)malloc((size_t)(T > 0 ? T : 1) * sizeof(cand_t));
  if (!c) return 1;
  int64_t n = 0;
  for (int64_t t = 0; t < T; ++t)
    if (allowed[t]) {
      c[n].score = scores[t];
      c[n].index = t;
      ++n;
    }
  qsort(c, (size_t)n, sizeof(cand_t), cand_order);
  const int64_t keep = n < top_k ? n : top_k;
  for (int64_t i = 0; i < keep; ++i) out[i] = c[i].index;
  qsort(out, (size_t)keep, sizeof(int64_t), index_order);
  for (int64_t i = keep; i < top_k; ++i) out[i] = -1;
  free(c);
  return 0;
}

/* Selection of every row from given scores / allowed flags. */
int oracle_dsa_select(const float *scores, const unsigned char *allowed, int64_t *out, int64_t rows, int64_t T,
                      int64_t top_k) {
  for (int64_t r = 0; r < rows; ++r)
    if (select_row(scores + r * T, allowed + r * T, T, top_k, out + r * top_k)) return 1;
  return 0;
}

/*
 * The whole op for a list of rows (row = b * S + s): scores and selection,
 * out[i * top_k ...] for rows[i].  Returns 0, or 1 on a bad row / allocation.
 */
int oracle_dsa_rows(const float *query, const float *key, const float *weights, const float *bias,
                    const int64_t *rows, int64_t n_rows, int64_t *out, int64_t B, int64_t S, int64_t H,
                    int64_t D, int64_t T, int64_t top_k, float scale, float weights_scale) {
  float *sc = (float *)malloc((size_t)(T > 0 ? T : 1) * sizeof(float));
  unsigned char *al = (unsigned char *)malloc((size_t)(T > 0 ? T : 1));
  if (!sc || !al) {
    free(sc);
    free(al);
    return 1;
  }
  int rc = 0;
  for (int64_t i = 0; i < n_rows && rc == 0; ++i) {
    const int64_t row = rows[i];
    if (row < 0 || row >= B * S) {
      rc = 1;
      break;
    }
    const int64_t b = row / S;
    for (int64_t t = 0; t < T; ++t) {
      const float bt = bias[row * T + t];
      al[t] = (unsigned char)(bt > -1e30f);
      sc[t] = al[t] ? cell_score(query + row * H * D, key + (b * T + t) * D, weights + row * H, bt, H, D,
                                 scale, weights_scale)
                    : -INFINITY;
    }
    rc = select_row(sc, al, T, top_k, out + i * top_k);
  }
  free(sc);
  free(al);
  return rc;
}
