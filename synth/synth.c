/*
 * Seeded synthetic inputs shaped like the video-DiT attention workloads of
 * "VC-Attention" (arXiv 2609.15810, §4.1 and Appx A: post-RoPE Q, K, V of
 * Wan2.2-class models).  The captured tensors are not available, so these
 * generators stand in for them.  This module holds none of the method's
 * arithmetic; it only produces bf16 inputs that both the CUDA library and
 * the CPU oracle consume.
 *
 * Every value is a pure function of (seed, tensor tag, index): a counter-
 * based SplitMix64 hash gives uniforms, Box-Muller gives normals.  Any slice
 * can therefore be regenerated independently, in any thread order.
 *
 *   Q, K : N(0,1) + a per-(b,h) per-channel offset drawn from N(0, 2).
 *   V    : a mixture of C Gaussian clusters per (b,h): centres N(0,1) per
 *          channel, spread 0.3, labels uniform per token (so the token order
 *          is scrambled); 1% of tokens are outliers whose 4 distinct,
 *          independently drawn channels are multiplied by 30.
 * Outputs are bf16 bit patterns, [B, H, N, d] row-major.
 */
#include <math.h>
#include <stdint.h>

enum { TAG_QVAL = 1, TAG_QOFF, TAG_KVAL, TAG_KOFF, TAG_VCENT, TAG_VNOISE, TAG_VLABEL,
       TAG_VOUT, TAG_VOUTCH };

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t seed, uint64_t tag, uint64_t idx) {
  return mix64(mix64(seed ^ (tag * 0xD1B54A32D192ED03ULL)) + (idx + 1) * 0x9E3779B97F4A7C15ULL);
}

static inline double uniform_open(uint64_t r) { /* (0, 1) */
  return ((double)(r >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline double normal(uint64_t seed, uint64_t tag, uint64_t idx) {
  double u1 = uniform_open(draw(seed, tag, 2 * idx));
  double u2 = uniform_open(draw(seed, tag, 2 * idx + 1));
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

static inline uint16_t to_bf16(double x) {
  float f = (float)x;
  union { float f; uint32_t u; } v = {f};
  uint32_t keep = v.u >> 16, drop = v.u & 0xFFFFu;
  if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u))) keep += 1;
  return (uint16_t)keep;
}

/* which: 0 = Q, 1 = K */
void synth_qk(uint16_t* out, int B, int H, int N, int d, uint64_t seed, int which) {
  const uint64_t tv = which ? TAG_KVAL : TAG_QVAL, to = which ? TAG_KOFF : TAG_QOFF;
  const int64_t rows = (int64_t)B * H * N;
#pragma omp parallel for schedule(static)
  for (int64_t row = 0; row < rows; ++row) {
    const int64_t bh = row / N;
    for (int c = 0; c < d; ++c) {
      double off = sqrt(2.0) * normal(seed, to, (uint64_t)(bh * d + c));
      double x = normal(seed, tv, (uint64_t)(row * d + c)) + off;
      out[row * d + c] = to_bf16(x);
    }
  }
}

void synth_v(uint16_t* out, int B, int H, int N, int d, int clusters, uint64_t seed) {
  const int64_t rows = (int64_t)B * H * N;
#pragma omp parallel for schedule(static)
  for (int64_t row = 0; row < rows; ++row) {
    const int64_t bh = row / N;
    const int label = (int)(draw(seed, TAG_VLABEL, (uint64_t)row) % (uint64_t)clusters);
    const int outlier = draw(seed, TAG_VOUT, (uint64_t)row) < (uint64_t)(0.01 * 18446744073709551616.0);
    int och[4] = {-1, -1, -1, -1};
    if (outlier) {
      int have = 0;
      for (uint64_t i = 0; have < 4; ++i) {
        int c = (int)(draw(seed, TAG_VOUTCH, (uint64_t)row * 64 + i) % (uint64_t)d);
        int dup = 0;
        for (int j = 0; j < have; ++j) dup |= (och[j] == c);
        if (!dup) och[have++] = c;
      }
    }
    for (int c = 0; c < d; ++c) {
      double centre = normal(seed, TAG_VCENT, (uint64_t)((bh * clusters + label) * d + c));
      double x = centre + 0.3 * normal(seed, TAG_VNOISE, (uint64_t)(row * d + c));
      if (outlier && (c == och[0] || c == och[1] || c == och[2] || c == och[3])) x *= 30.0;
      out[row * d + c] = to_bf16(x);
    }
  }
}

/* Number of outlier tokens and the label of each token of one (b,h), so tests
 * can check the recipe (1% outliers, uniform labels) without re-deriving it. */
void synth_v_labels(int32_t* labels, uint8_t* is_outlier, int B, int H, int N, int clusters,
                    uint64_t seed, int b, int h) {
  for (int t = 0; t < N; ++t) {
    uint64_t row = ((uint64_t)b * H + h) * N + t;
    labels[t] = (int32_t)(draw(seed, TAG_VLABEL, row) % (uint64_t)clusters);
    is_outlier[t] = draw(seed, TAG_VOUT, row) < (uint64_t)(0.01 * 18446744073709551616.0);
  }
}
