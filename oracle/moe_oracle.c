/*
 * CPU oracle for the W8A8 MoE expert layer -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library.  The product path (the CUDA library) never calls it and
 * shares no code, header or table with it.
 *
 * Source of the method: the PTO-ISA MegaMoE operator page ("pto-isa megamoe
 * operator", kernels/manual/a2a3/dispatch_mega_combine/overview), whose
 * "key implementation logic" section splits MegaMoe::Process() into seven
 * stages (FrontReorder, Dispatch, GMM1, SwiGLU, GMM2, Combine, Unpermute).
 * Each function below cites the stage section it restates.  With one rank the
 * cross-rank parts of FrontReorder/Dispatch/Combine (count exchange, remote
 * windows) are the identity and are not modelled.
 *
 * Precision is the pages' own: binary16 tokens and stage outputs, int8
 * quantised operands, exact integer accumulation, fp32 for the scale
 * arithmetic.  Every fp32 operation is a separate IEEE operation (the library
 * is built with -ffp-contract=off); every binary16 rounding is round to
 * nearest even.  Readings of points the page leaves open:
 *   - sort order: ascending expert id, ties by ascending route id (stable);
 *     route id r = token * topK + slot.
 *   - an expert id outside [0, E) marks the route invalid: it is placed after
 *     all valid routes (ascending r), counted in no expert, and its
 *     expandedRowIdx is -1 so that Unpermute skips it.
 *   - cumsum[e] is the inclusive prefix over experts of tokensPerExpert.
 *   - token quant rounds half away from zero (CAST_ROUND), clamps to
 *     [-127, 127]; an all-zero row gets scale 0 and all-zero codes.
 *   - requant multiplies by 127/amax computed once, rounds half to even
 *     (CAST_RINT), clamps to [-127, 127]; amax 0 gives scale 0, codes 0.
 *   - GMM epilogue: binary16(float(acc) * channel_scale); the per-token scales
 *     are applied later, in SwiGLU (pts1) and Combine (pts2).
 *   - silu acts on the first half of the GMM1 row, the second half multiplies.
 *   - silu(v) = v / (1 + e) with e = exp(-v) evaluated in double and rounded
 *     to fp32 (portable across libms).
 *   - Unpermute: fp32 accumulator starting at 0, slots in order 0..topK-1,
 *     each step a multiply then an add (no fused multiply-add).
 *   - every fp32 -> binary16 stage conversion (GMM epilogues, Combine,
 *     Unpermute) rounds to nearest even and saturates at +-65504: the page
 *     does not say what the output-type cast does on overflow, and with the
 *     workloads' value ranges Combine's D = C2 * pts2 exceeds the binary16
 *     range for about 1% of its elements at K=7168, I=2048.
 * Function: all of the layer.  Pins: tests/test_oracle.py.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#include <omp.h>

/* ------------------------------------------------------------------ */
/* binary16 <-> fp32 (compiler _Float16: IEEE conversions, RNE)        */
/* ------------------------------------------------------------------ */
static inline float h2f(uint16_t b) {
  _Float16 h;
  memcpy(&h, &b, 2);
  return (float)h;
}
static inline uint16_t f2h_ieee(float f) {
  _Float16 h = (_Float16)f;
  uint16_t b;
  memcpy(&b, &h, 2);
  return b;
}
/* Stage-output conversion: round to nearest even, saturating to the largest
 * finite binary16 (65504) instead of overflowing to infinity. */
#define F16_MAX_FINITE 65504.0f
static inline uint16_t f2h(float f) {
  if (f > F16_MAX_FINITE) f = F16_MAX_FINITE;
  if (f < -F16_MAX_FINITE) f = -F16_MAX_FINITE;
  return f2h_ieee(f);
}

void oracle_f16_to_f32(int64_t n, const uint16_t* in, float* out) {
  for (int64_t i = 0; i < n; i++) out[i] = h2f(in[i]);
}
void oracle_f32_to_f16(int64_t n, const float* in, uint16_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = f2h_ieee(in[i]);
}
void oracle_f32_to_f16_sat(int64_t n, const float* in, uint16_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = f2h(in[i]);
}

static inline int clamp127(int v) { return v > 127 ? 127 : (v < -127 ? -127 : v); }

/* round half away from zero */
static inline int round_half_away(float v) { return (int)roundf(v); }

/* round half to even, written out: floor, then compare the remainder with 1/2 */
static inline int round_half_even(float v) {
  float f = floorf(v);
  float rem = v - f; /* exact: v and f are within one binade step */
  int i = (int)f;
  if (rem > 0.5f) return i + 1;
  if (rem < 0.5f) return i;
  return (i % 2 == 0) ? i : i + 1;
}

/* ------------------------------------------------------------------ */
/* FrontReorder, Phase 1 + Phase 2a/2b + Phase 4 (one rank):           */
/* sort routes expert-major, count per expert, invert the permutation, */
/* prefix-sum the counts.                                               */
/* ------------------------------------------------------------------ */
/* Returns the number of invalid routes (expert id outside [0, E)). */
int oracle_route_sort(int M, int topK, int E, const int32_t* expert_idx,
                      int32_t* sorted_src_route, int32_t* expanded_row_idx,
                      int32_t* tokens_per_expert, int32_t* cumsum) {
  const int R = M * topK;
  int d = 0;
  /* stable sort by expert id: sweep experts in order, routes in order */
  for (int e = 0; e < E; e++) {
    int cnt = 0;
    for (int r = 0; r < R; r++) {
      if (expert_idx[r] == e) {
        sorted_src_route[d] = r;
        expanded_row_idx[r] = d;
        d++;
        cnt++;
      }
    }
    tokens_per_expert[e] = cnt;
    cumsum[e] = d; /* inclusive prefix */
  }
  int invalid = 0;
  for (int r = 0; r < R; r++) {
    if (expert_idx[r] < 0 || expert_idx[r] >= E) {
      sorted_src_route[d++] = r;
      expanded_row_idx[r] = -1;
      invalid++;
    }
  }
  return invalid;
}

/* ------------------------------------------------------------------ */
/* FrontReorder, Phase 2c: per-token dynamic quant, once per token.    */
/* scale = rowmax|x| / 127 ; q = CAST_ROUND(x / scale)                  */
/* ------------------------------------------------------------------ */
void oracle_quant_tokens(int M, int K, const uint16_t* x, int8_t* xq, float* pts1) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < M; t++) {
    const uint16_t* row = x + (size_t)t * K;
    float amax = 0.0f;
    for (int k = 0; k < K; k++) {
      float a = fabsf(h2f(row[k]));
      if (a > amax) amax = a;
    }
    float scale = amax / 127.0f;
    pts1[t] = scale;
    for (int k = 0; k < K; k++) {
      int q = 0;
      if (amax > 0.0f) q = clamp127(round_half_away(h2f(row[k]) / scale));
      xq[(size_t)t * K + k] = (int8_t)q;
    }
  }
}

/* ------------------------------------------------------------------ */
/* Dispatch + GMM1 for one expanded row d (route r, token t, expert e): */
/*   acc[n] = sum_k xq[t,k] * w1[e][n][k]      (exact integer)          */
/*   C1[d,n] = binary16( float(acc[n]) * s1[e][n] )   (TSTORE_FP)       */
/* ------------------------------------------------------------------ */
static void gmm_row(int Kd, int N, const int8_t* a, const int8_t* w, const float* s,
                    int32_t* acc_out, uint16_t* c_out) {
  for (int n = 0; n < N; n++) {
    const int8_t* wr = w + (size_t)n * Kd;
    int32_t acc = 0;
    for (int k = 0; k < Kd; k++) acc += (int32_t)a[k] * (int32_t)wr[k];
    if (acc_out) acc_out[n] = acc;
    c_out[n] = f2h((float)acc * s[n]);
  }
}

/* GMM1 over all valid expanded rows.  w1: [E][2I][K], s1: [E][2I].
 * acc1 (nullable): int32 [R_valid][2I]; c1: binary16 [R_valid][2I]. */
void oracle_gmm1(int M, int K, int I, int E, int topK, const int8_t* xq,
                 const int32_t* sorted_src_route, const int32_t* expert_idx,
                 const int8_t* w1, const float* s1, int R_valid, int32_t* acc1, uint16_t* c1) {
  (void)M; (void)E;
  const int N = 2 * I;
#pragma omp parallel for schedule(dynamic, 1)
  for (int d = 0; d < R_valid; d++) {
    int r = sorted_src_route[d];
    int t = r / topK, e = expert_idx[r];
    gmm_row(K, N, xq + (size_t)t * K, w1 + (size_t)e * N * K, s1 + (size_t)e * N,
            acc1 ? acc1 + (size_t)d * N : NULL, c1 + (size_t)d * N);
  }
}

/* ------------------------------------------------------------------ */
/* SwiGLU for one row: dequant, silu(first half) * second half,         */
/* per-row dynamic requant (section "4. SwiGLU").                      */
/* ------------------------------------------------------------------ */
static inline float silu_f32(float v) {
  float e = (float)exp(-(double)v);
  return v / (1.0f + e);
}

static void swiglu_row(int I, const uint16_t* c1row, float pts1, int8_t* q2row, float* pts2,
                       float* y /* scratch [I] */) {
  float amax = 0.0f;
  for (int j = 0; j < I; j++) {
    float h_gate = h2f(c1row[j]) * pts1;
    float h_up = h2f(c1row[j + I]) * pts1;
    y[j] = silu_f32(h_gate) * h_up;
    float a = fabsf(y[j]);
    if (a > amax) amax = a;
  }
  if (amax > 0.0f) {
    *pts2 = amax / 127.0f;
    float inv = 127.0f / amax;
    for (int j = 0; j < I; j++) q2row[j] = (int8_t)clamp127(round_half_even(y[j] * inv));
  } else {
    *pts2 = 0.0f;
    for (int j = 0; j < I; j++) q2row[j] = 0;
  }
}

/* rows d in [0, R_valid): c1 [R_valid][2I] -> q2 [R_valid][I], pts2 [R_valid].
 * pts1 is per token; the row's token is sorted_src_route[d] / topK. */
void oracle_swiglu_quant(int R_valid, int I, int topK, const uint16_t* c1, const float* pts1,
                         const int32_t* sorted_src_route, int8_t* q2, float* pts2) {
#pragma omp parallel
  {
    float* y = (float*)malloc(sizeof(float) * (size_t)I);
#pragma omp for schedule(static)
    for (int d = 0; d < R_valid; d++) {
      int t = sorted_src_route[d] / topK;
      swiglu_row(I, c1 + (size_t)d * 2 * I, pts1[t], q2 + (size_t)d * I, pts2 + d, y);
    }
    free(y);
  }
}

/* ------------------------------------------------------------------ */
/* GMM2 (section "5. GMM2"): acc[k] = sum_i q2[d,i] * w2[e][k][i];      */
/* C2[d,k] = binary16(float(acc) * s2[e][k]).  w2: [E][K][I].          */
/* ------------------------------------------------------------------ */
void oracle_gmm2(int K, int I, int topK, const int8_t* q2, const int32_t* sorted_src_route,
                 const int32_t* expert_idx, const int8_t* w2, const float* s2, int R_valid,
                 int32_t* acc2, uint16_t* c2) {
  (void)topK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int d = 0; d < R_valid; d++) {
    int e = expert_idx[sorted_src_route[d]];
    gmm_row(I, K, q2 + (size_t)d * I, w2 + (size_t)e * K * I, s2 + (size_t)e * K,
            acc2 ? acc2 + (size_t)d * K : NULL, c2 + (size_t)d * K);
  }
}

/* ------------------------------------------------------------------ */
/* Combine ("6. Combine"): D[d,k] = binary16(float(C2[d,k]) * pts2[d])  */
/* Unpermute ("7. Unpermute"): out[t,k] = binary16( fp32 sum over slots */
/*   of float(D[expandedRowIdx[t*topK+j], k]) * probs[t,j] )            */
/* ------------------------------------------------------------------ */
void oracle_combine(int R_valid, int K, const uint16_t* c2, const float* pts2, uint16_t* dmat) {
#pragma omp parallel for schedule(static)
  for (int d = 0; d < R_valid; d++)
    for (int k = 0; k < K; k++)
      dmat[(size_t)d * K + k] = f2h(h2f(c2[(size_t)d * K + k]) * pts2[d]);
}

void oracle_unpermute(int M, int K, int topK, const uint16_t* dmat, const int32_t* expanded_row_idx,
                      const float* probs, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < M; t++) {
    for (int k = 0; k < K; k++) {
      float acc = 0.0f;
      for (int j = 0; j < topK; j++) {
        int d = expanded_row_idx[t * topK + j];
        if (d < 0) continue; /* invalid route */
        float weighted = h2f(dmat[(size_t)d * K + k]) * probs[t * topK + j];
        acc = acc + weighted;
      }
      out[(size_t)t * K + k] = f2h(acc);
    }
  }
}

/* ------------------------------------------------------------------ */
/* Whole layer (MegaMoe::Process on one rank).  Intermediates are      */
/* written when their pointer is non-NULL (sizes for R = M*topK rows). */
/* Returns the number of invalid routes.                                */
/* ------------------------------------------------------------------ */
int oracle_layer_fwd(int M, int K, int I, int E, int topK, const uint16_t* x,
                     const int32_t* expert_idx, const float* probs, const int8_t* w1,
                     const float* s1, const int8_t* w2, const float* s2, uint16_t* out,
                     int32_t* o_sorted, int32_t* o_expanded, int32_t* o_tpe, int32_t* o_cumsum,
                     int8_t* o_xq, float* o_pts1, uint16_t* o_c1, int8_t* o_q2, float* o_pts2,
                     uint16_t* o_c2) {
  const int R = M * topK;
  int32_t* sorted = o_sorted ? o_sorted : (int32_t*)malloc(sizeof(int32_t) * (size_t)R);
  int32_t* expanded = o_expanded ? o_expanded : (int32_t*)malloc(sizeof(int32_t) * (size_t)R);
  int32_t* tpe = o_tpe ? o_tpe : (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  int32_t* cs = o_cumsum ? o_cumsum : (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  int8_t* xq = o_xq ? o_xq : (int8_t*)malloc((size_t)M * K);
  float* pts1 = o_pts1 ? o_pts1 : (float*)malloc(sizeof(float) * (size_t)M);
  uint16_t* c1 = o_c1 ? o_c1 : (uint16_t*)malloc(sizeof(uint16_t) * (size_t)R * 2 * I);
  int8_t* q2 = o_q2 ? o_q2 : (int8_t*)malloc((size_t)R * I);
  float* pts2 = o_pts2 ? o_pts2 : (float*)malloc(sizeof(float) * (size_t)R);
  uint16_t* c2 = o_c2 ? o_c2 : (uint16_t*)malloc(sizeof(uint16_t) * (size_t)R * K);
  uint16_t* dm = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)R * K);

  int invalid = oracle_route_sort(M, topK, E, expert_idx, sorted, expanded, tpe, cs);
  int R_valid = R - invalid;
  oracle_quant_tokens(M, K, x, xq, pts1);
  oracle_gmm1(M, K, I, E, topK, xq, sorted, expert_idx, w1, s1, R_valid, NULL, c1);
  oracle_swiglu_quant(R_valid, I, topK, c1, pts1, sorted, q2, pts2);
  oracle_gmm2(K, I, topK, q2, sorted, expert_idx, w2, s2, R_valid, NULL, c2);
  oracle_combine(R_valid, K, c2, pts2, dm);
  oracle_unpermute(M, K, topK, dm, expanded, probs, out);

  free(dm);
  if (!o_sorted) free(sorted);
  if (!o_expanded) free(expanded);
  if (!o_tpe) free(tpe);
  if (!o_cumsum) free(cs);
  if (!o_xq) free(xq);
  if (!o_pts1) free(pts1);
  if (!o_c1) free(c1);
  if (!o_q2) free(q2);
  if (!o_pts2) free(pts2);
  if (!o_c2) free(c2);
  return invalid;
}

/* ------------------------------------------------------------------ */
/* The layer's output for a sample of tokens.  A token's output row    */
/* depends only on its own routes, so each sampled token runs its topK */
/* routes through GMM1 -> SwiGLU -> GMM2 -> Combine, then Unpermute,   */
/* with exactly the per-row operations of the full pipeline above.     */
/* Used where the full layer would take the CPU too long.               */
/* ------------------------------------------------------------------ */
void oracle_layer_tokens(int M, int K, int I, int E, int topK, const uint16_t* x,
                         const int32_t* expert_idx, const float* probs, const int8_t* w1,
                         const float* s1, const int8_t* w2, const float* s2, int n_tok,
                         const int32_t* tokens, uint16_t* out_rows /* [n_tok][K] */) {
  (void)M;
  const int N = 2 * I;
#pragma omp parallel
  {
    int8_t* xq = (int8_t*)malloc((size_t)K);
    uint16_t* c1 = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)N);
    int8_t* q2 = (int8_t*)malloc((size_t)I);
    uint16_t* c2 = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)K);
    float* y = (float*)malloc(sizeof(float) * (size_t)I);
    float* acc = (float*)malloc(sizeof(float) * (size_t)K);
#pragma omp for schedule(dynamic, 1)
    for (int i = 0; i < n_tok; i++) {
      int t = tokens[i];
      float pts1;
      oracle_quant_tokens(1, K, x + (size_t)t * K, xq, &pts1);
      for (int k = 0; k < K; k++) acc[k] = 0.0f;
      for (int j = 0; j < topK; j++) {
        int e = expert_idx[t * topK + j];
        if (e < 0 || e >= E) continue;
        float pts2;
        gmm_row(K, N, xq, w1 + (size_t)e * N * K, s1 + (size_t)e * N, NULL, c1);
        swiglu_row(I, c1, pts1, q2, &pts2, y);
        gmm_row(I, K, q2, w2 + (size_t)e * K * I, s2 + (size_t)e * K, NULL, c2);
        for (int k = 0; k < K; k++) {
          float dval = h2f(f2h(h2f(c2[k]) * pts2));
          float weighted = dval * probs[t * topK + j];
          acc[k] = acc[k] + weighted;
        }
      }
      for (int k = 0; k < K; k++) out_rows[(size_t)i * K + k] = f2h(acc[k]);
    }
    free(xq); free(c1); free(q2); free(c2); free(y); free(acc);
  }
}

/* Threads an OpenMP region of this library runs on (diagnostics: the benchmark
 * reports how many host cores the oracle used).  No arithmetic. */
int oracle_max_threads(void) { return omp_get_max_threads(); }

/* Threads the following OpenMP regions of this library use (the benchmark's
 * single-thread baseline sets 1, then restores the previous count).  No arithmetic. */
void oracle_set_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
