// ExpCast-FP8 (paper §3.3 Eq 7): the E4M3 probability byte written straight
// from the log-domain score, c(u) = clip_[0,120](RNE(8(u+8) + 56 + beta)),
// beta = -0.35.  With u = (a*acc - M) / 8, where `acc` is the raw QK^T
// accumulator, a = 8 log2(e) sQ sK / sqrt(d) and M = 8 x (running row max in
// the log2 domain), the code is clip(RNE(fma(a, acc, b))) with b = 119.65 - M.
#pragma once
#include "common.cuh"

namespace vca {

constexpr float kExpCastBias = 119.65f;  // 8*8 + 56 + beta, beta = -0.35

// Reference form: one FMA, the clip, then RNE by adding 1.5 * 2^23 (the fp32
// adder rounds to the integer grid); the code is the low byte.
__device__ __forceinline__ uint32_t expcast_code(float acc, float a, float b) {
  float t = __fmaf_rn(a, acc, b);
  t = fminf(fmaxf(t, 0.0f), 120.0f);  // NaN -> 0
  return __float_as_uint(__fadd_rn(t, 12582912.0f)) & 0xFFu;
}

// When the kernel form gives exactly the reference form's byte, for scores
// with a * acc <= M (M the running maximum, scaled by 8, log2 domain; a > 0,
// the product of positive scales):
//   - |M| < 2^20: t = fma(a, acc, 119.65 - M) stays below 120.5 (the rounding
//     of a * max and of 119.65 - M each add at most 2^-4), so the upper clip
//     never acts;
//   - a > 0: a masked key (acc = -inf) gives t = -inf, not NaN;
//   - no score of the row is NaN (those rows take the reference form).
__device__ __forceinline__ bool expcast_fast_is_exact(float M, float a) {
  return fabsf(M) < 1048576.0f && a > 0.0f;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmax3_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of a row's 128 scores (fp32 bit patterns): eight chains of
// three-input max.  NaN scores are ignored (max.f32 returns the other operand).
__device__ __forceinline__ float row_max128(const uint32_t (&s)[128]) {
  float m8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    m8[i] = fmaxf(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
#pragma unroll
  for (int c = 16; c < 128; c += 16)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      m8[i] = fmax3(m8[i], __uint_as_float(s[c + 2 * i]), __uint_as_float(s[c + 2 * i + 1]));
  return fmaxf(fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5])),
               fmaxf(m8[6], m8[7]));
}

// The same maximum, also telling whether the row holds a NaN score: one pass
// of NaN-propagating max (the common case), the NaN-ignoring pass only for a
// row that has one.
__device__ __forceinline__ float row_max128_flag(const uint32_t (&s)[128], bool& has_nan) {
  float m8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    m8[i] = fmax3_nan(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]),
                      __uint_as_float(s[2 * i + 1]));
#pragma unroll
  for (int c = 16; c < 128; c += 16)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      m8[i] = fmax3_nan(m8[i], __uint_as_float(s[c + 2 * i]), __uint_as_float(s[c + 2 * i + 1]));
  const float m = fmax3_nan(fmax3_nan(m8[0], m8[1], m8[2]), fmax3_nan(m8[3], m8[4], m8[5]),
                            fmax3_nan(m8[6], m8[7], m8[7]));
  has_nan = m != m;
  return has_nan ? row_max128(s) : m;
}

// The ExpCast bytes of one row of a 128-key block relative to the running
// maximum Mn (>= a * every score), four per word in the A-operand layout of
// the value product (byte k of word c is key 4c + k).
// Kernel form, two scores per step: one paired FMA gives t = fma(a, acc,
// 119.65 - Mn) exactly as the reference form does; multiplying by 2^-149
// (paired) rounds t to the integer grid of fp32 subnormals with ties to even,
// so the bits of the product are RNE(t) for 0 <= t < 2^23, and a sign bit
// for t < 0 (or -inf); the saturating pack to unsigned bytes maps those to 0.
// 1.5 instructions per score.  Rows the fast form is not exact for take the
// reference form.
__device__ __forceinline__ void expcast_row_bytes(const uint32_t (&s)[128], float a, float Mn,
                                                  bool has_nan, uint32_t (&w)[32]) {
  const float b = kExpCastBias - Mn;
  if (!has_nan && expcast_fast_is_exact(Mn, a)) {
    const uint64_t a2 = ((uint64_t)__float_as_uint(a) << 32) | __float_as_uint(a);
    const uint64_t b2 = ((uint64_t)__float_as_uint(b) << 32) | __float_as_uint(b);
    const uint64_t tiny = 0x0000000100000001ull;  // 2^-149, twice
#pragma unroll
    for (int c = 0; c < 128; c += 4) {
      uint64_t t01, t23, u01, u23;
      asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(t01)
          : "l"(((uint64_t)s[c + 1] << 32) | s[c]), "l"(a2), "l"(b2));
      asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(t23)
          : "l"(((uint64_t)s[c + 3] << 32) | s[c + 2]), "l"(a2), "l"(b2));
      asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(u01) : "l"(t01), "l"(tiny));
      asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(u23) : "l"(t23), "l"(tiny));
      uint32_t hi, word;
      asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(hi)
          : "r"((uint32_t)(u23 >> 32)), "r"((uint32_t)u23), "r"(0u));
      asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(word)
          : "r"((uint32_t)(u01 >> 32)), "r"((uint32_t)u01), "r"(hi));
      w[c / 4] = word;
    }
  } else {
#pragma unroll
    for (int c = 0; c < 128; c += 4)
      w[c / 4] = expcast_code(__uint_as_float(s[c]), a, b) |
                 (expcast_code(__uint_as_float(s[c + 1]), a, b) << 8) |
                 (expcast_code(__uint_as_float(s[c + 2]), a, b) << 16) |
                 (expcast_code(__uint_as_float(s[c + 3]), a, b) << 24);
  }
}

// Keys at and past `valid` of the last block are masked: score -inf, byte 0.
__device__ __forceinline__ void mask_tail128(uint32_t (&s)[128], int valid) {
#pragma unroll
  for (int c = 0; c < 128; ++c)
    if (c >= valid) s[c] = 0xFF800000u;
}

}  // namespace vca
