// VC-Attention CPU oracle — TEST INFRASTRUCTURE ONLY (see oracle.h).
//
// Written from the paper "VC-Attention: Value Smoothing and Softmax Casting
// for Low-bit Attention" (arXiv 2609.15810).  Each function names the section
// or equation it restates.  Single-threaded, unoptimised, fp64 wherever the
// method does not fix a narrower type.  Must be compiled with
// -ffp-contract=off so that every fp32 step rounds exactly once.

#include "oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

namespace {

const double kLog2e = 1.4426950408889634073599246810019;

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------

// Value of every non-negative finite E4M3 code, in code order (increasing).
// Byte = s eeee mmm, bias 7: normal 2^(e-7)(1+m/8), subnormal 2^-6 (m/8).
double e4m3_value(int c) {
  int e = (c >> 3) & 15, m = c & 7;
  if (e == 0) return std::ldexp(m / 8.0, -6);
  return std::ldexp(1.0 + m / 8.0, e - 7);
}

// E2M1: s ee m, bias 1: normal 2^(e-1)(1+m/2), subnormal m/2.
double e2m1_value(int c) {
  int e = (c >> 1) & 3, m = c & 1;
  if (e == 0) return m * 0.5;
  return std::ldexp(1.0 + m / 2.0, e - 1);
}

// Round a non-negative magnitude to the nearest of the increasing grid
// value(0..top), ties to the even code.  Magnitudes at or above value(top)
// saturate to top.  The midpoint comparison is exact in double because every
// grid value and every float input is a short dyadic rational.
template <typename F>
int round_to_grid(double a, int top, F value) {
  if (a >= value(top)) return top;
  int lo = 0, hi = top;  // invariant: value(lo) <= a < value(hi)
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (value(mid) <= a) lo = mid; else hi = mid;
  }
  double mid = 0.5 * (value(lo) + value(hi));
  if (a < mid) return lo;
  if (a > mid) return hi;
  return (lo % 2 == 0) ? lo : hi;
}

// ---------------------------------------------------------------------------
// SplitMix64 (Steele, Lea, Flood: "Fast splittable pseudorandom number
// generators", OOPSLA 2014), the generator that draws k-means seeds.
// ---------------------------------------------------------------------------
struct SplitMix64 {
  uint64_t state;
  uint64_t next() {
    state += 0x9E3779B97F4A7C15ULL;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
  }
};

// Round-half-to-even of the rational s/n, n > 0, in exact integer arithmetic.
int64_t div_round_half_even(int64_t s, int64_t n) {
  int64_t q = s / n, rem = s % n;
  if (rem < 0) { q -= 1; rem += n; }  // floor division, 0 <= rem < n
  if (2 * rem > n) return q + 1;
  if (2 * rem < n) return q;
  return (q % 2 == 0) ? q : q + 1;
}

// Sum of Bv fp32 values by the fixed pairwise tree: element r is added to
// element r + Bv/2, then r + Bv/4, ... .  Bv is a power of two.
float tree_sum(std::vector<float> w) {
  for (size_t stride = w.size() / 2; stride >= 1; stride /= 2)
    for (size_t r = 0; r < stride; ++r) w[r] = w[r] + w[r + stride];
  return w[0];
}

inline float bf(uint16_t b) { return orc_bf16_to_f32(b); }

int num_blocks(int N, int Bv) { return (N + Bv - 1) / Bv; }

// Per-block fp32 scale of an 8-bit operand: amax / 448, or 1 for an all-zero
// block (the E4M3 maximum is 448).
float e4m3_scale(float amax) { return amax > 0.0f ? amax / 448.0f : 1.0f; }

// NVFP4 global scale: amax / (448 * 6), so that the largest 16-block gets the
// largest UE4M3 block scale and E2M1 elements reach 6.
float nvfp4_global_scale(float amax) { return amax > 0.0f ? amax / 2688.0f : 1.0f; }

// Quantise a run of 16 fp32 values to NVFP4 with global scale g: block scale
// UE4M3(amax16 / (6 g)), elements E2M1(x / (scale * g)).
void nvfp4_block(const float* x, int stride, float g, uint8_t* codes, int cstride,
                 uint8_t* scale_out) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(x[i * stride]));
  float denom = 6.0f * g;
  uint8_t sc = orc_e4m3_encode(amax / denom);
  float scv = (float)orc_e4m3_decode(sc);
  *scale_out = sc;
  for (int i = 0; i < 16; ++i) {
    if (scv == 0.0f) { codes[i * cstride] = 0; continue; }
    float step = scv * g;
    codes[i * cstride] = orc_e2m1_encode(x[i * stride] / step);
  }
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// Formats (paper §3.3: E4M3 byte = s eeee mmm, value 2^(e-7)(1+m/8);
// Appx A: NVFP4 = E2M1 elements under a per-16 E4M3 microscale)
// ---------------------------------------------------------------------------
float orc_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

uint16_t orc_f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if (std::isnan(f)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t keep = u >> 16, drop = u & 0xFFFFu;
  if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u))) keep += 1;  // RNE
  return (uint16_t)keep;
}

double orc_e4m3_decode(uint8_t c) {
  if ((c & 0x7F) == 0x7F) return NAN;
  double v = e4m3_value(c & 0x7F);
  return (c & 0x80) ? -v : v;
}

uint8_t orc_e4m3_encode(float x) {
  if (std::isnan(x)) return 0x7F;
  uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  int c = round_to_grid(std::fabs((double)x), 126, e4m3_value);  // 126 = 448
  return (uint8_t)(sign | c);
}

double orc_e2m1_decode(uint8_t c) {
  double v = e2m1_value(c & 7);
  return (c & 8) ? -v : v;
}

uint8_t orc_e2m1_encode(float x) {
  if (std::isnan(x)) return 0;
  uint8_t sign = std::signbit(x) ? 8 : 0;
  int c = round_to_grid(std::fabs((double)x), 7, e2m1_value);  // 7 = 6.0
  return (uint8_t)(sign | c);
}

void orc_e4m3_encode_array(const float* x, uint8_t* out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(x[i]);
}

void orc_e2m1_encode_array(const float* x, uint8_t* out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = orc_e2m1_encode(x[i]);
}

// ---------------------------------------------------------------------------
// ExpCast-FP8, paper §3.3 Eq 7
// ---------------------------------------------------------------------------
int orc_expcast_code(double u) {
  const double beta = -0.35;
  double v = 8.0 * (u + 8.0) + 56.0 + beta;
  if (std::isnan(v)) return 0;
  double r = std::nearbyint(v);  // default rounding mode: ties to even
  if (r < 0.0) r = 0.0;
  if (r > 120.0) r = 120.0;
  return (int)r;
}

int orc_expcast_code_f32(float acc, float a, float b) {
  float t = std::fmaf(a, acc, b);  // one rounding
  if (std::isnan(t)) return 0;
  float r = std::nearbyintf(t);
  if (r < 0.0f) r = 0.0f;
  if (r > 120.0f) r = 120.0f;
  return (int)r;
}

void orc_expcast_f32_array(const float* acc, const float* a, const float* b, uint8_t* out,
                           size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_expcast_code_f32(acc[i], a[i], b[i]);
}

// ---------------------------------------------------------------------------
// V-Smooth, paper §3.2 (Eq 3, Eq 4) and §3.4 / Appx B
// ---------------------------------------------------------------------------
void orc_kmeans_init_indices(uint64_t seed, int b, int h, int H, int N, int k, int32_t* idx) {
  SplitMix64 g{seed ^ (0x9E3779B97F4A7C15ULL * (uint64_t)(b * H + h + 1))};
  int have = 0;
  while (have < k) {
    int32_t cand = (int32_t)(g.next() % (uint64_t)N);
    bool dup = false;
    for (int i = 0; i < have; ++i) dup = dup || (idx[i] == cand);
    if (!dup) idx[have++] = cand;
  }
}

// Features: the value tokens on a symmetric int8 grid with one scale per head,
// s = amax / 127 (1 for an all-zero head), x = clamp(RNE(v / s), -127, 127).
static float kmeans_features(const uint16_t* v, int N, int d, std::vector<int>& x) {
  float amax = 0.0f;
  for (size_t i = 0; i < (size_t)N * d; ++i) amax = std::max(amax, std::fabs(bf(v[i])));
  const float s = amax > 0.0f ? amax / 127.0f : 1.0f;
  x.assign((size_t)N * d, 0);
  for (size_t i = 0; i < (size_t)N * d; ++i) {
    float q = std::nearbyintf(bf(v[i]) / s);
    x[i] = (int)std::min(127.0f, std::max(-127.0f, q));
  }
  return s;
}

// Lloyd iterations: assign to the nearest centroid (squared Euclidean
// distance, lowest index on ties), then move each centroid to the
// round-half-even integer mean of its members; an empty cluster keeps its
// centroid.  The labels are those of the last assignment.
static void kmeans_lloyd(const std::vector<int>& x, int N, int d, int k, int iters,
                         std::vector<int>& c, int32_t* labels) {
  for (int it = 0; it < iters; ++it) {
    for (int t = 0; t < N; ++t) {
      int64_t best = 0;
      int bestm = -1;
      for (int m = 0; m < k; ++m) {
        int64_t dist = 0;
        for (int j = 0; j < d; ++j) {
          int64_t diff = (int64_t)x[(size_t)t * d + j] - c[(size_t)m * d + j];
          dist += diff * diff;
        }
        if (bestm < 0 || dist < best) { best = dist; bestm = m; }
      }
      labels[t] = bestm;
    }
    std::vector<int64_t> sum((size_t)k * d, 0), cnt(k, 0);
    for (int t = 0; t < N; ++t) {
      cnt[labels[t]] += 1;
      for (int j = 0; j < d; ++j) sum[(size_t)labels[t] * d + j] += x[(size_t)t * d + j];
    }
    for (int m = 0; m < k; ++m)
      if (cnt[m] > 0)
        for (int j = 0; j < d; ++j)
          c[(size_t)m * d + j] = (int)div_round_half_even(sum[(size_t)m * d + j], cnt[m]);
  }
}

void orc_kmeans(const uint16_t* v, const orc_head_cfg* cfg, int8_t* x_out, float* grid_scale_out,
                int32_t* labels, int8_t* centroids) {
  const int N = cfg->N, d = cfg->d, k = cfg->k;
  std::vector<int> x;
  const float s = kmeans_features(v, N, d, x);
  if (x_out)
    for (size_t i = 0; i < x.size(); ++i) x_out[i] = (int8_t)x[i];
  *grid_scale_out = s;

  // Initial centroids: k distinct tokens chosen by SplitMix64.
  std::vector<int32_t> idx(k);
  orc_kmeans_init_indices(cfg->seed, cfg->b, cfg->h, cfg->H, N, k, idx.data());
  std::vector<int> c((size_t)k * d);
  for (int m = 0; m < k; ++m)
    for (int j = 0; j < d; ++j) c[(size_t)m * d + j] = x[(size_t)idx[m] * d + j];
  kmeans_lloyd(x, N, d, k, cfg->iters, c, labels);
  for (size_t i = 0; i < c.size(); ++i) centroids[i] = (int8_t)c[i];
}

void orc_kmeans_warm(const uint16_t* v, const orc_head_cfg* cfg, const int8_t* prev_centroids,
                     float prev_grid_scale, int8_t* x_out, float* grid_scale_out,
                     int32_t* labels, int8_t* centroids) {
  const int N = cfg->N, d = cfg->d, k = cfg->k;
  std::vector<int> x;
  const float s = kmeans_features(v, N, d, x);
  if (x_out)
    for (size_t i = 0; i < x.size(); ++i) x_out[i] = (int8_t)x[i];
  *grid_scale_out = s;

  // The previous step's centroids, kept at the same place in value units:
  // on the new grid c = clamp(RNE(c_prev * (s_prev / s)), -127, 127), the
  // ratio and the product each rounded to fp32.
  const float r = prev_grid_scale / s;
  std::vector<int> c((size_t)k * d);
  for (size_t i = 0; i < c.size(); ++i) {
    const float t = std::nearbyintf((float)prev_centroids[i] * r);
    c[i] = (int)std::min(127.0f, std::max(-127.0f, t));
  }
  kmeans_lloyd(x, N, d, k, cfg->iters, c, labels);
  for (size_t i = 0; i < c.size(); ++i) centroids[i] = (int8_t)c[i];
}

void orc_stable_argsort(const int32_t* labels, int N, int k, int32_t* perm) {
  std::vector<int64_t> start(k + 1, 0);
  for (int t = 0; t < N; ++t) start[labels[t] + 1] += 1;
  for (int m = 0; m < k; ++m) start[m + 1] += start[m];
  for (int t = 0; t < N; ++t) perm[start[labels[t]]++] = t;
}

void orc_hadamard128(const float* x, float* y) {
  // The normalised Sylvester-Hadamard transform y = x H / sqrt(128), H[i][j] =
  // (-1)^popcount(i & j), as the fast transform: butterflies on pairs
  // (i, i + s) with i & s = 0 for s = 1, 2, ..., 64 in that order, each
  // (a, b) -> (a + b, a - b) in fp32, then one fp32 multiply by the fp32
  // value of 1/sqrt(128).
  float t[128];
  for (int i = 0; i < 128; ++i) t[i] = x[i];
  for (int s = 1; s < 128; s <<= 1)
    for (int i = 0; i < 128; ++i)
      if ((i & s) == 0) {
        const float a = t[i], b = t[i + s];
        t[i] = a + b;
        t[i + s] = a - b;
      }
  const float scale = (float)(1.0 / std::sqrt(128.0));
  for (int i = 0; i < 128; ++i) y[i] = t[i] * scale;
}

void orc_block_demean(const uint16_t* vperm, int N, int d, int Bv, uint16_t* mu, float* r) {
  const int nb = num_blocks(N, Bv);
  for (int j = 0; j < nb; ++j) {
    const int nj = std::min(Bv, N - j * Bv);
    for (int c = 0; c < d; ++c) {
      std::vector<float> w(Bv, 0.0f);
      for (int i = 0; i < nj; ++i) w[i] = bf(vperm[(size_t)(j * Bv + i) * d + c]);
      float mean = tree_sum(w) / (float)nj;
      uint16_t m16 = orc_f32_to_bf16(mean);
      mu[(size_t)j * d + c] = m16;
      for (int i = 0; i < Bv; ++i) {
        size_t row = (size_t)j * Bv + i;
        r[row * d + c] = (i < nj) ? bf(vperm[row * d + c]) - bf(m16) : 0.0f;
      }
    }
  }
}

namespace {

// Shared front half of both preparations: grouping, the permutation, and the
// key channel mean (Appx B: the K pass fuses the centring statistics).
struct Front {
  std::vector<int32_t> perm;
  std::vector<uint16_t> kbar;
  std::vector<float> kp;  // permuted, centred keys, fp32 [Npad*d], zero padding
  std::vector<uint16_t> vperm;  // permuted values, bf16 [N*d]
};

// naive: the comparison kernel that smooths nothing (sequence order, no key
// centring): pi is the identity and kbar is 0.
void front_half(const uint16_t* k, const uint16_t* v, const orc_head_cfg* cfg,
                const int32_t* perm_in, int32_t* labels, int8_t* centroids, float* grid_scale,
                Front& f, bool naive = false) {
  const int N = cfg->N, d = cfg->d, Bv = cfg->Bv, nb = num_blocks(N, Bv);
  const size_t Npad = (size_t)nb * Bv;
  f.perm.assign(N, 0);
  if (naive) {
    for (int i = 0; i < N; ++i) f.perm[i] = i;
  } else if (perm_in) {
    std::copy(perm_in, perm_in + N, f.perm.begin());
  } else {
    orc_kmeans(v, cfg, nullptr, grid_scale, labels, centroids);
    orc_stable_argsort(labels, N, cfg->k, f.perm.data());
  }
  // Key channel mean: fp32 tree sum per block of the original order, the block
  // sums added in block order in fp64, divided by N, rounded to fp32 then bf16.
  f.kbar.assign(d, 0);
  for (int c = 0; c < d && !naive; ++c) {
    double total = 0.0;
    for (int j = 0; j < nb; ++j) {
      std::vector<float> w(Bv, 0.0f);
      for (int i = 0; i < Bv && j * Bv + i < N; ++i) w[i] = bf(k[(size_t)(j * Bv + i) * d + c]);
      total += (double)tree_sum(w);
    }
    f.kbar[c] = orc_f32_to_bf16((float)(total / (double)N));
  }
  // K' = K[pi] - kbar  (Eq 3, then the mean subtraction of Appx B)
  f.kp.assign(Npad * d, 0.0f);
  for (int i = 0; i < N; ++i)
    for (int c = 0; c < d; ++c)
      f.kp[(size_t)i * d + c] = bf(k[(size_t)f.perm[i] * d + c]) - bf(f.kbar[c]);
  // V' = V[pi]
  f.vperm.assign((size_t)N * d, 0);
  for (int i = 0; i < N; ++i)
    for (int c = 0; c < d; ++c) f.vperm[(size_t)i * d + c] = v[(size_t)f.perm[i] * d + c];
}

// Per-block E4M3 quantisation of rows [Npad*d] (fp32, zero padding).
void quant_rows_e4m3(const float* x, int N, int d, int Bv, uint8_t* codes, float* scales) {
  const int nb = num_blocks(N, Bv);
  for (int j = 0; j < nb; ++j) {
    float amax = 0.0f;
    for (int i = 0; i < Bv && j * Bv + i < N; ++i)
      for (int c = 0; c < d; ++c) amax = std::max(amax, std::fabs(x[(size_t)(j * Bv + i) * d + c]));
    float s = e4m3_scale(amax);
    scales[j] = s;
    for (int i = 0; i < Bv; ++i) {
      size_t row = (size_t)j * Bv + i;
      for (int c = 0; c < d; ++c)
        codes[row * d + c] = (j * Bv + i < N) ? orc_e4m3_encode(x[row * d + c] / s) : 0;
    }
  }
}

// The value operand: block means and residual (Eq 4), or, on the steps after
// the grouping window (§3.4 "Amortized grouping schedule"), the permuted values
// themselves with every mean zero.
void split_values(const std::vector<uint16_t>& vperm, int N, int d, int Bv, bool demean,
                  uint16_t* mu, float* r) {
  if (demean) {
    orc_block_demean(vperm.data(), N, d, Bv, mu, r);
    return;
  }
  const int nb = num_blocks(N, Bv);
  std::fill(mu, mu + (size_t)nb * d, (uint16_t)0);
  std::fill(r, r + (size_t)nb * Bv * d, 0.0f);
  for (size_t i = 0; i < (size_t)N * d; ++i) r[i] = bf(vperm[i]);
}

// The QK Hadamard rotation of every row of x [rows*128] in place (Appx B: the Q
// and K kernels fuse it before quantising), as hadamard128 below.
void rotate_rows(float* x, size_t rows) {
  for (size_t i = 0; i < rows; ++i) orc_hadamard128(x + i * 128, x + i * 128);
}

void prepare8(const uint16_t* q, const uint16_t* k, const uint16_t* v, const orc_head_cfg* cfg,
              const int32_t* perm_in, bool demean, orc_prep8_out* out, bool naive = false,
              bool hadamard = false) {
  const int N = cfg->N, d = cfg->d, Bv = cfg->Bv, nb = num_blocks(N, Bv);
  const size_t Npad = (size_t)nb * Bv;
  Front f;
  front_half(k, v, cfg, perm_in, out->labels, out->centroids, out->grid_scale, f, naive);
  std::copy(f.perm.begin(), f.perm.end(), out->perm);
  std::copy(f.kbar.begin(), f.kbar.end(), out->kbar);

  // Q: per-block E4M3, Q keeps its order (Eq 3).
  std::vector<float> qf(Npad * d, 0.0f);
  for (size_t i = 0; i < (size_t)N * d; ++i) qf[i] = bf(q[i]);
  if (hadamard) {
    rotate_rows(qf.data(), N);
    rotate_rows(f.kp.data(), N);
  }
  quant_rows_e4m3(qf.data(), N, d, Bv, out->qhat, out->sq);
  // K': per-block E4M3 of the permuted, centred keys.
  quant_rows_e4m3(f.kp.data(), N, d, Bv, out->khat, out->sk);

  // V: block demeaning (Eq 4) and per-channel E4M3 of the residual (§3.2);
  // the means are stored divided by the channel scale (Appx B).
  std::vector<float> r(Npad * d);
  split_values(f.vperm, N, d, Bv, demean, out->mu, r.data());
  for (int c = 0; c < d; ++c) {
    float amax = 0.0f;
    for (int i = 0; i < N; ++i) amax = std::max(amax, std::fabs(r[(size_t)i * d + c]));
    out->sv[c] = e4m3_scale(amax);
  }
  for (int c = 0; c < d; ++c)
    for (size_t i = 0; i < Npad; ++i)
      out->rhatT[(size_t)c * Npad + i] =
          (i < (size_t)N) ? orc_e4m3_encode(r[i * d + c] / out->sv[c]) : 0;
  for (int j = 0; j < nb; ++j)
    for (int c = 0; c < d; ++c)
      out->mutilde[(size_t)j * d + c] = bf(out->mu[(size_t)j * d + c]) / out->sv[c];
}

void prepare4(const uint16_t* q, const uint16_t* k, const uint16_t* v, const orc_head_cfg* cfg,
              const int32_t* perm_in, bool demean, orc_prep4_out* out, bool hadamard = false,
              bool naive = false) {
  const int N = cfg->N, d = cfg->d, Bv = cfg->Bv, nb = num_blocks(N, Bv);
  const size_t Npad = (size_t)nb * Bv;
  Front f;
  front_half(k, v, cfg, perm_in, out->labels, out->centroids, out->grid_scale, f, naive);
  std::copy(f.perm.begin(), f.perm.end(), out->perm);
  std::copy(f.kbar.begin(), f.kbar.end(), out->kbar);

  // Q and K': NVFP4 with blocks of 16 along the head dimension (the QK^T
  // reduction dimension) and one global scale per head.
  std::vector<float> qf(Npad * d, 0.0f);
  for (size_t i = 0; i < (size_t)N * d; ++i) qf[i] = bf(q[i]);
  if (hadamard) {
    rotate_rows(qf.data(), N);
    rotate_rows(f.kp.data(), N);
  }
  float qa = 0.0f, ka = 0.0f;
  for (size_t i = 0; i < (size_t)N * d; ++i) {
    qa = std::max(qa, std::fabs(qf[i]));
    ka = std::max(ka, std::fabs(f.kp[i]));
  }
  *out->gq = nvfp4_global_scale(qa);
  *out->gk = nvfp4_global_scale(ka);
  for (size_t row = 0; row < Npad; ++row)
    for (int cb = 0; cb < d / 16; ++cb) {
      size_t o = row * d + (size_t)cb * 16;
      nvfp4_block(&qf[o], 1, *out->gq, &out->q4[o], 1, &out->q4s[o / 16]);
      nvfp4_block(&f.kp[o], 1, *out->gk, &out->k4[o], 1, &out->k4s[o / 16]);
    }
  // V: the same block demeaning; the residual in NVFP4 with blocks of 16
  // along tokens (the PV reduction dimension); means stay unscaled (Appx B).
  std::vector<float> r(Npad * d);
  split_values(f.vperm, N, d, Bv, demean, out->mu, r.data());
  float ra = 0.0f;
  for (size_t i = 0; i < (size_t)N * d; ++i) ra = std::max(ra, std::fabs(r[i]));
  *out->gr = nvfp4_global_scale(ra);
  for (int c = 0; c < d; ++c)
    for (size_t tb = 0; tb < Npad / 16; ++tb) {
      size_t o = (size_t)c * Npad + tb * 16;
      nvfp4_block(&r[tb * 16 * d + c], d, *out->gr, &out->r4T[o], 1, &out->r4s[o / 16]);
    }
}

}  // namespace

void orc_prepare8(const uint16_t* q, const uint16_t* k, const uint16_t* v, const orc_head_cfg* cfg,
                  const int32_t* perm_in, orc_prep8_out* out) {
  prepare8(q, k, v, cfg, perm_in, true, out);
}
void orc_prepare4(const uint16_t* q, const uint16_t* k, const uint16_t* v, const orc_head_cfg* cfg,
                  const int32_t* perm_in, orc_prep4_out* out) {
  prepare4(q, k, v, cfg, perm_in, true, out);
}
void orc_prepare8_plain(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const orc_head_cfg* cfg, const int32_t* perm, orc_prep8_out* out) {
  prepare8(q, k, v, cfg, perm, false, out);
}
void orc_prepare4_plain(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const orc_head_cfg* cfg, const int32_t* perm, orc_prep4_out* out) {
  prepare4(q, k, v, cfg, perm, false, out);
}
void orc_prepare8_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const orc_head_cfg* cfg, const int32_t* perm_in, unsigned opts,
                     orc_prep8_out* out) {
  prepare8(q, k, v, cfg, perm_in, (opts & (ORC_PLAIN | ORC_NAIVE)) == 0, out,
           (opts & ORC_NAIVE) != 0, (opts & ORC_HADAMARD) != 0);
}
void orc_prepare4_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const orc_head_cfg* cfg, const int32_t* perm_in, unsigned opts,
                     orc_prep4_out* out) {
  prepare4(q, k, v, cfg, perm_in, (opts & (ORC_PLAIN | ORC_NAIVE)) == 0, out,
           (opts & ORC_HADAMARD) != 0, (opts & ORC_NAIVE) != 0);
}
void orc_prepare8_hadamard(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const orc_head_cfg* cfg, const int32_t* perm_in, orc_prep8_out* out) {
  prepare8(q, k, v, cfg, perm_in, true, out, false, true);
}
void orc_prepare4_hadamard(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const orc_head_cfg* cfg, const int32_t* perm_in, orc_prep4_out* out) {
  prepare4(q, k, v, cfg, perm_in, true, out, true);
}
void orc_prepare8_naive(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const orc_head_cfg* cfg, orc_prep8_out* out) {
  prepare8(q, k, v, cfg, nullptr, false, out, true);
}

// ---------------------------------------------------------------------------
// Attention
// ---------------------------------------------------------------------------
void orc_attention_exact(const uint16_t* q, const uint16_t* k, const uint16_t* v, int N, int d,
                         const int32_t* rows, int nrows, double* out) {
  const double inv = 1.0 / std::sqrt((double)d);
  std::vector<double> s(N);
  for (int ri = 0; ri < nrows; ++ri) {
    const int i = rows[ri];
    double mx = -INFINITY;
    for (int t = 0; t < N; ++t) {
      double acc = 0.0;
      for (int c = 0; c < d; ++c) acc += (double)bf(q[(size_t)i * d + c]) * bf(k[(size_t)t * d + c]);
      s[t] = acc * inv;
      mx = std::max(mx, s[t]);
    }
    double l = 0.0;
    std::vector<double> o(d, 0.0);
    for (int t = 0; t < N; ++t) {
      double p = std::exp(s[t] - mx);
      l += p;
      for (int c = 0; c < d; ++c) o[c] += p * bf(v[(size_t)t * d + c]);
    }
    for (int c = 0; c < d; ++c) out[(size_t)ri * d + c] = o[c] / l;
  }
}

// The conventional probability byte that ExpCast replaces (§3.3): the
// exponential, then the E4M3 cast, with the same 2^8 scale as the ExpCast
// byte: E4M3_RNE(2^(u + 8)), u <= 0 the log2-domain score minus the maximum.
static uint8_t exp_cast_code(double u) { return orc_e4m3_encode((float)std::exp2(u + 8.0)); }

// Eq 1 with the split numerator of Eq 6, over tiles of Bv keys, in fp64.
void orc_attention_recurrence(const double* q, const double* kp, const double* r, const double* mu,
                              int N, int d, int Bv, int pmode, const int32_t* rows, int nrows,
                              double* out) {
  const int nb = num_blocks(N, Bv);
  const double inv = 1.0 / std::sqrt((double)d);
  for (int ri = 0; ri < nrows; ++ri) {
    const int i = rows[ri];
    double m = -INFINITY, l = 0.0;
    std::vector<double> A(d, 0.0);
    for (int j = 0; j < nb; ++j) {
      const int k0 = j * Bv, k1 = std::min(N, k0 + Bv);
      std::vector<double> t(k1 - k0);
      double mt = -INFINITY;
      for (int kk = k0; kk < k1; ++kk) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += q[(size_t)i * d + c] * kp[(size_t)kk * d + c];
        t[kk - k0] = acc * inv * kLog2e;  // log2-domain score
        mt = std::max(mt, t[kk - k0]);
      }
      const double mnew = std::max(m, mt);
      const double alpha = std::exp2(m - mnew);  // 0 on the first tile
      double rsum = 0.0;
      std::vector<double> pv(d, 0.0);
      for (int kk = k0; kk < k1; ++kk) {
        const double u = t[kk - k0] - mnew;
        const double p = pmode == 0   ? std::exp2(u)
                         : pmode == 1 ? orc_e4m3_decode((uint8_t)orc_expcast_code(u))
                                      : orc_e4m3_decode(exp_cast_code(u));
        rsum += p;
        for (int c = 0; c < d; ++c) pv[c] += p * r[(size_t)kk * d + c];
      }
      for (int c = 0; c < d; ++c) A[c] = alpha * A[c] + pv[c] + rsum * mu[(size_t)j * d + c];
      l = alpha * l + rsum;
      m = mnew;
    }
    for (int c = 0; c < d; ++c) out[(size_t)ri * d + c] = A[c] / l;
  }
}

static void attention8(const orc_prep8_out* P, int N, int d, const int32_t* rows, int nrows,
                       bool expcast, uint16_t* out, double* out64) {
  const int Bv = 128, nb = num_blocks(N, Bv);
  const size_t Npad = (size_t)nb * Bv;
  const double inv = 1.0 / std::sqrt((double)d);
  // Dequantised codes (scales applied below, where the kernel applies them).
  std::vector<double> kd(Npad * d), rd(Npad * d);
  for (size_t i = 0; i < Npad * d; ++i) kd[i] = orc_e4m3_decode(P->khat[i]);
  for (int c = 0; c < d; ++c)
    for (size_t i = 0; i < Npad; ++i) rd[i * d + c] = orc_e4m3_decode(P->rhatT[(size_t)c * Npad + i]);
  for (int ri = 0; ri < nrows; ++ri) {
    const int i = rows[ri];
    const double sq = P->sq[i / Bv];
    std::vector<double> qd(d);
    for (int c = 0; c < d; ++c) qd[c] = orc_e4m3_decode(P->qhat[(size_t)i * d + c]);
    double m = -INFINITY, l = 0.0;
    std::vector<double> A(d, 0.0);  // in units of the per-channel value scale sv
    for (int j = 0; j < nb; ++j) {
      const int k0 = j * Bv, k1 = std::min(N, k0 + Bv);
      std::vector<double> t(k1 - k0);
      double mt = -INFINITY;
      for (int kk = k0; kk < k1; ++kk) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += qd[c] * kd[(size_t)kk * d + c];
        t[kk - k0] = acc * sq * (double)P->sk[j] * inv * kLog2e;
        mt = std::max(mt, t[kk - k0]);
      }
      const double mnew = std::max(m, mt);
      const double alpha = std::exp2(m - mnew);
      double rsum = 0.0;
      std::vector<double> pv(d, 0.0);
      for (int kk = k0; kk < k1; ++kk) {
        // Eq 7: the probability byte, read as E4M3 (it carries the 2^8 scale);
        // or the conventional exponential and cast
        const double u = t[kk - k0] - mnew;
        const double w = orc_e4m3_decode(expcast ? (uint8_t)orc_expcast_code(u) : exp_cast_code(u));
        rsum += w;
        for (int c = 0; c < d; ++c) pv[c] += w * rd[(size_t)kk * d + c];
      }
      // Eq 6: A <- alpha A + P_q R_q + r mu^T (mu pre-divided by sv), l <- alpha l + r
      for (int c = 0; c < d; ++c)
        A[c] = alpha * A[c] + pv[c] + rsum * (double)P->mutilde[(size_t)j * d + c];
      l = alpha * l + rsum;
      m = mnew;
    }
    for (int c = 0; c < d; ++c) {
      const double o = (double)P->sv[c] * A[c] / l;
      if (out64) out64[(size_t)ri * d + c] = o;
      out[(size_t)ri * d + c] = orc_f32_to_bf16((float)o);
    }
  }
}

void orc_attention8(const orc_prep8_out* P, int N, int d, const int32_t* rows, int nrows,
                    uint16_t* out, double* out64) {
  attention8(P, N, d, rows, nrows, true, out, out64);
}
void orc_attention8_exp(const orc_prep8_out* P, int N, int d, const int32_t* rows, int nrows,
                        uint16_t* out, double* out64) {
  attention8(P, N, d, rows, nrows, false, out, out64);
}

void orc_attention4(const orc_prep4_out* P, int N, int d, const int32_t* rows, int nrows,
                    uint16_t* out, double* out64) {
  const int Bv = 128, nb = num_blocks(N, Bv);
  const size_t Npad = (size_t)nb * Bv;
  const double inv = 1.0 / std::sqrt((double)d);
  const double gq = *P->gq, gk = *P->gk, gr = *P->gr;
  std::vector<double> kd(Npad * d), rd(Npad * d);
  for (size_t i = 0; i < Npad * d; ++i)
    kd[i] = orc_e2m1_decode(P->k4[i]) * orc_e4m3_decode(P->k4s[i / 16]) * gk;
  for (int c = 0; c < d; ++c)
    for (size_t i = 0; i < Npad; ++i) {
      size_t o = (size_t)c * Npad + i;
      rd[i * d + c] = orc_e2m1_decode(P->r4T[o]) * orc_e4m3_decode(P->r4s[o / 16]) * gr;
    }
  for (int ri = 0; ri < nrows; ++ri) {
    const int i = rows[ri];
    std::vector<double> qd(d);
    for (int c = 0; c < d; ++c) {
      size_t o = (size_t)i * d + c;
      qd[c] = orc_e2m1_decode(P->q4[o]) * orc_e4m3_decode(P->q4s[o / 16]) * gq;
    }
    double m = -INFINITY, l = 0.0;
    std::vector<double> A(d, 0.0);
    for (int j = 0; j < nb; ++j) {
      const int k0 = j * Bv, k1 = std::min(N, k0 + Bv);
      std::vector<double> t(Bv, -INFINITY);
      double mt = -INFINITY;
      for (int kk = k0; kk < k1; ++kk) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += qd[c] * kd[(size_t)kk * d + c];
        t[kk - k0] = acc * inv * kLog2e;
        mt = std::max(mt, t[kk - k0]);
      }
      const double mnew = std::max(m, mt);
      const double alpha = std::exp2(m - mnew);
      // Conventional exponential; r and l use the unquantised probabilities.
      std::vector<double> p(Bv, 0.0);
      double rsum = 0.0;
      for (int kk = 0; kk < k1 - k0; ++kk) { p[kk] = std::exp2(t[kk] - mnew); rsum += p[kk]; }
      // P in NVFP4: the row scaled so its maximum is 448*6, blocks of 16 keys.
      std::vector<double> pq(Bv, 0.0);
      for (int b16 = 0; b16 < Bv / 16; ++b16) {
        double amax = 0.0;
        for (int e = 0; e < 16; ++e) amax = std::max(amax, 2688.0 * p[b16 * 16 + e]);
        const uint8_t sc = orc_e4m3_encode((float)(amax / 6.0));
        const double scv = orc_e4m3_decode(sc);
        for (int e = 0; e < 16; ++e) {
          if (scv == 0.0) continue;
          const uint8_t code = orc_e2m1_encode((float)(2688.0 * p[b16 * 16 + e] / scv));
          pq[b16 * 16 + e] = orc_e2m1_decode(code) * scv / 2688.0;
        }
      }
      std::vector<double> pv(d, 0.0);
      for (int kk = k0; kk < k1; ++kk)
        for (int c = 0; c < d; ++c) pv[c] += pq[kk - k0] * rd[(size_t)kk * d + c];
      for (int c = 0; c < d; ++c)
        A[c] = alpha * A[c] + pv[c] + rsum * (double)orc_bf16_to_f32(P->mu[(size_t)j * d + c]);
      l = alpha * l + rsum;
      m = mnew;
    }
    for (int c = 0; c < d; ++c) {
      const double o = A[c] / l;
      if (out64) out64[(size_t)ri * d + c] = o;
      out[(size_t)ri * d + c] = orc_f32_to_bf16((float)o);
    }
  }
}

}  // extern "C"
