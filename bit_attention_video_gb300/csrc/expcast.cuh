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

// With M the running maximum (scaled by 8, log2 domain), the fast form needs
// no upper clip when t = fma(a, acc, 119.65 - M) provably stays below 120.5.
__device__ __forceinline__ bool expcast_fast_is_exact(float M) { return fabsf(M) < 1048576.0f; }

}  // namespace vca
