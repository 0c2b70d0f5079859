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

// Kernel form on a pair: the FMA is evaluated on the 1/128-scaled operands
// with saturation to [0, 1] (exact, scaling by a power of two commutes with
// rounding), which clips below at 0; adding 1.5 * 2^16 rounds 128 t' to the
// integer grid (ulp 2^-7), so the low byte of the sum is RNE(t).  The upper
// clip at 120 can only act when |M| >= 2^20 (see expcast_fast_is_exact).
// Returns the two fp32 bit patterns 0x47C00000 + code.
__device__ __forceinline__ uint2 expcast_pair_bits(float acc0, float acc1, float a128,
                                                   float b128) {
  float t0, t1;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(t0) : "f"(a128), "f"(acc0), "f"(b128));
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(t1) : "f"(a128), "f"(acc1), "f"(b128));
  uint64_t in = ((uint64_t)__float_as_uint(t1) << 32) | __float_as_uint(t0), out;
  const uint64_t magic = ((uint64_t)0x47C00000u << 32) | 0x47C00000u;  // 98304.0f x2
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(out) : "l"(in), "l"(magic));
  return make_uint2((uint32_t)out, (uint32_t)(out >> 32));
}

// When the pair form gives exactly the reference form's byte, for scores with
// a * acc <= M (M the running maximum, scaled by 8, log2 domain):
//   - |M| < 2^20: t = fma(a, acc, 119.65 - M) stays below 120.5 (the rounding
//     of a * max and of 119.65 - M each add at most 2^-4), so the upper clip
//     never acts;
//   - a = 0 or a >= 2^-119: a * 2^-7 is exact (not subnormal).  (b * 2^-7 is
//     always exact: 119.65 - M is 0 or at least 2^-18 in magnitude.)
__device__ __forceinline__ bool expcast_fast_is_exact(float M, float a) {
  return fabsf(M) < 1048576.0f && (a == 0.0f || a >= 1.50463277e-36f /* 2^-119 */);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
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

// The ExpCast bytes of one row of a 128-key block relative to the running
// maximum Mn (>= a * every score), four per word in the A-operand layout of
// the value product (byte k of word c is key 4c + k).  The pair form when it
// is exact, else the reference form.
__device__ __forceinline__ void expcast_row_bytes(const uint32_t (&s)[128], float a, float Mn,
                                                  uint32_t (&w)[32]) {
  const float b = kExpCastBias - Mn;
  if (expcast_fast_is_exact(Mn, a)) {
    const float a128 = a * 0.0078125f, b128 = b * 0.0078125f;
#pragma unroll
    for (int c = 0; c < 128; c += 4) {
      const uint2 e0 = expcast_pair_bits(__uint_as_float(s[c]), __uint_as_float(s[c + 1]), a128,
                                         b128);
      const uint2 e1 = expcast_pair_bits(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]),
                                         a128, b128);
      w[c / 4] = __byte_perm(__byte_perm(e0.x, e0.y, 0x0040), __byte_perm(e1.x, e1.y, 0x0040),
                             0x5410);
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
