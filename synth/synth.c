/*
 * Seeded synthetic inputs for the W8A8 MoE expert layer.
 *
 * This file holds no arithmetic of the layer itself: it only draws the inputs
 * (tokens, routing, routing probabilities, int8 weights, per-channel scales).
 * Both the CPU oracle and the CUDA path receive the bytes produced here.
 *
 * Generator: counter-based SplitMix64 (Steele, Lea, Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014).  Draw i of stream s is
 *     mix64(key(seed, s) + (i + 1) * 0x9E3779B97F4A7C15)
 * where mix64 is SplitMix64's output function and key() is mix64 of the seed
 * and the stream id.  Being counter-based, every element is independent of
 * the thread that computes it, so the output is identical for any thread
 * count and on any host (x86_64 or aarch64).
 */
#include <stdint.h>
#include <math.h>
#include <string.h>
#include <stdlib.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(mix64(seed * GOLDEN + 0x5851F42D4C957F2DULL) ^ (stream * 0xD1B54A32D192ED03ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

/* uniform double in (0, 1): 53 random bits, never exactly 0 */
static inline double unif01(uint64_t r) { return ((double)(r >> 11) + 0.5) * (1.0 / 9007199254740992.0); }

/* standard normal by Box-Muller from draws 2i and 2i+1 */
static inline double normal_at(uint64_t key, uint64_t i) {
  double u1 = unif01(draw(key, 2 * i)), u2 = unif01(draw(key, 2 * i + 1));
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
}

/* Gumbel(0,1) */
static inline double gumbel_at(uint64_t key, uint64_t i) { return -log(-log(unif01(draw(key, i)))); }

/* IEEE binary16 bits of a float, round to nearest even (input generation only). */
static uint16_t f32_to_f16_bits(float f) {
  _Float16 h = (_Float16)f;
  uint16_t b;
  memcpy(&b, &h, 2);
  return b;
}

/* x[n]: binary16 bits of N(0,1) draws */
void synth_normal_f16(uint64_t seed, uint64_t stream, int64_t n, uint16_t* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++) out[i] = f32_to_f16_bits((float)normal_at(key, (uint64_t)i));
}

/* int8 uniform over the 255 integers [-127, 127]; two values per 64-bit draw
 * (multiply-shift of each 32-bit half onto [0, 255)). */
void synth_int8_sym127(uint64_t seed, uint64_t stream, int64_t n, int8_t* out) {
  uint64_t key = stream_key(seed, stream);
  int64_t pairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < pairs; p++) {
    uint64_t r = draw(key, (uint64_t)p);
    uint32_t lo = (uint32_t)r, hi = (uint32_t)(r >> 32);
    out[2 * p] = (int8_t)((int)(((uint64_t)lo * 255u) >> 32) - 127);
    if (2 * p + 1 < n) out[2 * p + 1] = (int8_t)((int)(((uint64_t)hi * 255u) >> 32) - 127);
  }
}

/* fp32 uniform on [lo, hi) */
void synth_uniform_f32(uint64_t seed, uint64_t stream, int64_t n, double lo, double hi, float* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++) out[i] = (float)(lo + (hi - lo) * unif01(draw(key, (uint64_t)i)));
}

/*
 * Routing.  For each token, topK distinct experts are drawn without
 * replacement from the categorical distribution softmax(logit[t, :]) by the
 * Gumbel-top-k method (keys logit + Gumbel, take the k largest; the order of
 * the chosen experts is the draw order, i.e. descending key; ties, which have
 * probability zero, go to the lower expert id).
 *
 * mode 0 "uniform": logit = 0 for every expert.
 * mode 1 "biased" : logit[t,e] = g[t,e] + b[e], g ~ N(0,1), b ~ N(0, 0.5^2).
 * mode 2 "zipf"   : logit[t,e] = log p[e], p[perm[i]] proportional to 1/(i+1)^s,
 *                   perm a seeded random permutation of the experts.
 *
 * Probabilities: mode 1 takes the softmax of the chosen experts' logits g+b;
 * modes 0 and 2 take the softmax of fresh N(0,1) logits over the k slots.
 * They are not renormalised further by the layer.
 */
void synth_routing(uint64_t seed, int M, int E, int topK, int mode, double zipf_s,
                   int32_t* expert_idx, float* probs) {
  uint64_t kg = stream_key(seed, 6), kl = stream_key(seed, 7), kb = stream_key(seed, 8);
  uint64_t kp = stream_key(seed, 9), kperm = stream_key(seed, 10);
  double* base = (double*)malloc(sizeof(double) * (size_t)E);
  for (int e = 0; e < E; e++) base[e] = 0.0;
  if (mode == 1) {
    for (int e = 0; e < E; e++) base[e] = 0.5 * normal_at(kb, (uint64_t)e);
  } else if (mode == 2) {
    int* perm = (int*)malloc(sizeof(int) * (size_t)E);
    for (int e = 0; e < E; e++) perm[e] = e;
    for (int i = E - 1; i > 0; i--) { /* Fisher-Yates */
      int j = (int)(((draw(kperm, (uint64_t)i) >> 11) * (uint64_t)(i + 1)) >> 53);
      int tmp = perm[i]; perm[i] = perm[j]; perm[j] = tmp;
    }
    for (int i = 0; i < E; i++) base[perm[i]] = -zipf_s * log((double)(i + 1));
    free(perm);
  }
#pragma omp parallel for schedule(static)
  for (int t = 0; t < M; t++) {
    double keyv[64];
    int chosen[64];
    double logit_c[64];
    int k = topK;
    for (int j = 0; j < k; j++) { keyv[j] = -INFINITY; chosen[j] = -1; logit_c[j] = 0.0; }
    for (int e = 0; e < E; e++) {
      uint64_t idx = (uint64_t)t * (uint64_t)E + (uint64_t)e;
      double lg = base[e];
      if (mode == 1) lg += normal_at(kl, idx);
      double kv = lg + gumbel_at(kg, idx);
      /* insert into the descending top-k list (strictly greater: lower e wins ties) */
      if (kv > keyv[k - 1]) {
        int p = k - 1;
        while (p > 0 && kv > keyv[p - 1]) { keyv[p] = keyv[p - 1]; chosen[p] = chosen[p - 1]; logit_c[p] = logit_c[p - 1]; p--; }
        keyv[p] = kv; chosen[p] = e; logit_c[p] = lg;
      }
    }
    double z[64], mx = -INFINITY, sum = 0.0;
    for (int j = 0; j < k; j++) {
      z[j] = (mode == 1) ? logit_c[j] : normal_at(kp, (uint64_t)t * (uint64_t)k + (uint64_t)j);
      if (z[j] > mx) mx = z[j];
    }
    for (int j = 0; j < k; j++) { z[j] = exp(z[j] - mx); sum += z[j]; }
    for (int j = 0; j < k; j++) {
      expert_idx[(size_t)t * k + j] = chosen[j];
      probs[(size_t)t * k + j] = (float)(z[j] / sum);
    }
  }
  free(base);
}
