// SwiGLU + dynamic requant arithmetic of one expanded row (PTO-ISA MegaMoE operator
// page, "4. SwiGLU"), shared by the SwiGLU kernel (elementwise.cu) and the SwiGLU
// fused into the tcgen05 GMM1 (gemm_tc.cu), so both produce the same bits:
//   h = float(c1) * pts1,  y_j = silu(h_j) * h_{j+I},  silu(v) = v / (1 + exp(-v))
//   pts2 = max|y| / 127,   q_j = round-half-even(y_j * (127 / max|y|))
// The up half's token scale pts1 is left out of y: it scales the whole row, so the
// codes y * 127 / max|y| keep their values (to an ulp or two) and only pts2 takes
// it back.  exp and the division in silu use the MUFU fast paths (ex2 / rcp, a few
// ulp): SwiGLU is instruction-bound and the requantised codes tolerate it.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace moe {

// Requant codes read off a float: for |v| < 127.5, r = fl(v + kCodeMagic) is
// kCodeMagic + q with q = v rounded to the nearest integer, ties to even (the float
// spacing in [2^23, 2^24) is 1 and kCodeMagic is even), and r's bits are 0x4B406480 + q:
// the low half-word, 0x6480 + q, is the binary16 1152 + q (the mantissa of 1024) and
// its low byte 0x80 + q is q's two's-complement byte with the top bit flipped.
constexpr float kCodeMagic = 12608640.0f;  // 1.5 * 2^23 + 0x6480

// Two such code floats -> the binary16 pair (q0, q1): their low half-words, minus 1152.
__device__ __forceinline__ uint32_t code_bits_to_half2(uint32_t b0, uint32_t b1) {
  uint32_t r;
  asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(__byte_perm(b0, b1, 0x5410)), "r"(0x64806480u));
  return r;
}

// y of one gate/up pair (the token scale p1 applied to the gate only).
__device__ __forceinline__ float swiglu_y(__half gate, __half up, float p1) {
  const float hg = __fmul_rn(__half2float(gate), p1);
  const float silu = __fdividef(hg, __fadd_rn(1.0f, __expf(-hg)));
  return __fmul_rn(silu, __half2float(up));
}

// The row's code multiplier and pts2 from max|y| (0 and 0 for an all-zero row:
// every y * inv is then +-0 and its code 0).
__device__ __forceinline__ float swiglu_inv(float amax) { return amax > 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f; }
__device__ __forceinline__ float swiglu_pts2(float amax, float p1) {
  return amax > 0.0f ? __fdiv_rn(__fmul_rn(amax, p1), 127.0f) : 0.0f;
}

// Eight y -> their eight codes as binary16 (r = fl(y * inv + kCodeMagic), one rounding
// of the exact product: |y| <= amax keeps |y * inv| below 127 * (1 + 2^-23) < 127.5,
// so no clamp) and, in *l1, the sum of their |q| (binary16 integers up to 8 * 127 are
// exact; read off the bits of s + 1024 = 0x6400 + s).  `r_out`, if given, receives the
// code floats (their bits hold the int8 codes, see kCodeMagic).
__device__ __forceinline__ int4 swiglu_codes8(const float (&y)[8], float inv, int* l1, float* r_out = nullptr) {
  float r[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) r[j] = __fmaf_rn(y[j], inv, kCodeMagic);
  union {
    int4 v;
    uint32_t u[4];
    __half2 h2[4];
  } hc;
#pragma unroll
  for (int j = 0; j < 4; ++j) hc.u[j] = code_bits_to_half2(__float_as_uint(r[2 * j]), __float_as_uint(r[2 * j + 1]));
  if (l1) {
    __half2 a = __habs2(hc.h2[0]);
#pragma unroll
    for (int j = 1; j < 4; ++j) a = __hadd2(a, __habs2(hc.h2[j]));
    const __half s = __hadd(__hadd(__low2half(a), __high2half(a)), __ushort_as_half(0x6400));
    *l1 = (int)__half_as_ushort(s) - 0x6400;
  }
  if (r_out) {
#pragma unroll
    for (int j = 0; j < 8; ++j) r_out[j] = r[j];
  }
  return hc.v;
}

}  // namespace moe
