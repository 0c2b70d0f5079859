// V-Smooth preprocessing kernels (paper §3.2 Eq 3-4, §3.4 "Fused
// preprocessing", Appx B).  All are memory-bound passes except the k-means
// assignment.  Every floating-point step that decides a stored code is a
// single IEEE operation written with an explicit-rounding intrinsic, and every
// floating-point sum has a fixed order, so codes, scales and means are
// reproducible bit for bit.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "prep.h"

namespace vca {
namespace {

__device__ __forceinline__ bool prep_skip(const int* status) {
  return *(volatile const int*)status != 0;
}

__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide max over blockDim.x threads (multiple of 32, <= 1024).
__device__ float block_max(float v, float* red) {
  v = warp_max(v);
  const int w = threadIdx.x / 32, nw = blockDim.x / 32;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float m = 0.0f;
  for (int i = 0; i < nw; ++i) m = fmaxf(m, red[i]);
  return m;
}

// Per-block fp32 E4M3 scale: amax / 448, or 1 for an all-zero block.
__device__ __forceinline__ float e4m3_scale(float amax) {
  return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

// SplitMix64 (Steele, Lea & Flood 2014).
__device__ __forceinline__ uint64_t splitmix64_next(uint64_t& s) {
  s += 0x9E3779B97F4A7C15ull;
  uint64_t z = s;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// ---------------------------------------------------------------------------
// state header / reuse check
// ---------------------------------------------------------------------------
// reuse: 0 fresh grouping, 1 cached permutation, 2 grouping warm-started from
// the cached centroids, 3 cached permutation without block demeaning (modes
// 1-3 need a grouping of the same problem), 4 the naive comparison
// preparation (sequence order, no smoothing; leaves no grouping behind)
__global__ void header_kernel(uint32_t* hdr, int* status, int B, int H, int N, int d, int k,
                              int bits, int reuse) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  if (reuse >= 1 && reuse <= 3) {
    const bool match = hdr[0] == kStateMagic && hdr[1] == (uint32_t)B && hdr[2] == (uint32_t)H &&
                       hdr[3] == (uint32_t)N && hdr[4] == (uint32_t)d && hdr[5] == (uint32_t)k &&
                       hdr[6] == (uint32_t)bits && hdr[7] == 1u;
    *status = match ? 0 : kStatNoPerm;
    if (match) {
      if (reuse == 2) hdr[7] = 0;  // permutation being recomputed
      hdr[8] = 0;                  // operands being rewritten
    }
    return;
  }
  hdr[0] = kStateMagic;
  hdr[1] = B; hdr[2] = H; hdr[3] = N; hdr[4] = d; hdr[5] = k; hdr[6] = bits;
  hdr[7] = 0;  // permutation cached
  hdr[8] = 0;  // operands ready
  *status = 0;
}

__global__ void header_done_kernel(uint32_t* hdr, const int* status, int set_perm) {
  if (threadIdx.x != 0 || blockIdx.x != 0 || prep_skip(status)) return;
  if (set_perm) hdr[7] = 1;
  hdr[8] = 1;
}

// perm[bh][i] = i: sequence order (the naive comparison preparation)
__global__ void identity_perm_kernel(int32_t* perm, int N, const int* status) {
  if (prep_skip(status)) return;
  const size_t bh = blockIdx.y;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x)
    perm[bh * N + i] = i;
}

__global__ void zero_kernel(uint32_t* p, size_t words) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < words;
       i += (size_t)gridDim.x * blockDim.x)
    p[i] = 0;
}

// ---------------------------------------------------------------------------
// k-means on the int8 feature grid (paper §3.2 "Value-guided permutation")
// ---------------------------------------------------------------------------
// grid (chunks, BH): max |V| of each head, as the uint bits of a non-negative float.
__global__ void head_amax_kernel(const uint16_t* v, uint32_t* amax_bits, size_t per_head,
                                 const int* status) {
  __shared__ float red[32];
  if (prep_skip(status)) return;
  const size_t bh = blockIdx.y;
  const uint4* src = reinterpret_cast<const uint4*>(v + bh * per_head);
  const size_t n16 = per_head / 8;
  float m = 0.0f;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16;
       i += (size_t)gridDim.x * blockDim.x) {
    uint4 w = src[i];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      m = fmaxf(m, fabsf(__uint_as_float(ws[e] << 16)));
      m = fmaxf(m, fabsf(__uint_as_float(ws[e] & 0xFFFF0000u)));
    }
  }
  m = block_max(m, red);
  if (threadIdx.x == 0) atomicMax(&amax_bits[bh], __float_as_uint(m));
}

// x = clamp(RNE(v / s), -127, 127), s = amax / 127 (1 if amax = 0), stored
// as int8 or, for the tensor-core Lloyd iterations, as fp16 (exact).
template <bool kHalf>
__global__ void features_kernel(const uint16_t* v, const uint32_t* amax_bits, float* grid_scale,
                                void* x, size_t per_head, const int* status) {
  if (prep_skip(status)) return;
  const size_t bh = blockIdx.y;
  const float amax = __uint_as_float(amax_bits[bh]);
  const float s = amax > 0.0f ? __fdiv_rn(amax, 127.0f) : 1.0f;
  if (blockIdx.x == 0 && threadIdx.x == 0) grid_scale[bh] = s;
  const uint4* src = reinterpret_cast<const uint4*>(v + bh * per_head);
  const size_t n8 = per_head / 8;
  // RNE(v / s) from the bracketing products v rlo <= RN(v / s) <= v rhi (in
  // magnitude; rlo, rhi = (1/s)(1 -/+ 2^-20) rounded): integer rounding is
  // monotone, so equal integers at both ends are the quotient's; each end is
  // rounded to the integer grid by adding 1.5 * 2^23 (|v / s| <= 127).
  const float r = __frcp_rn(s);
  const float rlo = __fmul_rn(r, 1.0f - 0x1p-20f), rhi = __fmul_rn(r, 1.0f + 0x1p-20f);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8;
       i += (size_t)gridDim.x * blockDim.x) {
    uint4 w = src[i];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    uint32_t out[2] = {0, 0}, out16[4] = {0, 0, 0, 0};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t bits = (e & 1) ? (ws[e / 2] & 0xFFFF0000u) : (ws[e / 2] << 16);
      const float xv = __uint_as_float(bits);
      const float a = __fadd_rn(__fmul_rn(xv, rlo), 12582912.0f);
      const float b = __fadd_rn(__fmul_rn(xv, rhi), 12582912.0f);
      int q = a == b ? (int)(__float_as_uint(a) - 0x4B400000u) : __float2int_rn(__fdiv_rn(xv, s));
      q = max(-127, min(127, q));
      if constexpr (kHalf) {
        const uint32_t hb = __half_as_ushort(__int2half_rn(q));
        out16[e / 2] |= hb << (16 * (e % 2));
      } else {
        out[e / 4] |= ((uint32_t)(q & 0xFF)) << (8 * (e % 4));
      }
    }
    if constexpr (kHalf)
      reinterpret_cast<uint4*>(static_cast<uint16_t*>(x) + bh * per_head)[i] =
          make_uint4(out16[0], out16[1], out16[2], out16[3]);
    else
      reinterpret_cast<uint2*>(static_cast<int8_t*>(x) + bh * per_head)[i] =
          make_uint2(out[0], out[1]);
  }
}

// grid BH, 128 threads: initial centroids = features of k distinct tokens drawn
// by SplitMix64 from seed ^ (0x9E3779B97F4A7C15 * (bh + 1)); zero the sums.
// Warp 0 draws: every lane steps the same generator, the lanes test the
// candidate against a share of the accepted indices each, and a candidate
// is accepted when no lane finds it (the draws and acceptances of a single
// thread testing them in turn).  The k rows are then copied in 16-byte
// chunks (d = 128).
template <bool kHalf>
__global__ void kmeans_init_kernel(const void* x, int8_t* cent, int32_t* sums, int32_t* counts,
                                   uint64_t seed, int N, int k, int d, int* status) {
  __shared__ int32_t idx[256];
  if (prep_skip(status)) return;
  const int bh = blockIdx.x, lane = threadIdx.x % 32;
  if (threadIdx.x < 32) {
    uint64_t st = seed ^ (0x9E3779B97F4A7C15ull * (uint64_t)(bh + 1));
    int have = 0;
    // k <= N distinct draws; the bound only guards against a corrupted k
    for (long long tries = 0; have < k && tries < (1ll << 26); ++tries) {
      const int32_t cand = (int32_t)(splitmix64_next(st) % (uint64_t)N);
      bool dup = false;
      for (int i = lane; i < have; i += 32) dup |= (idx[i] == cand);
      if (!__any_sync(0xffffffffu, dup)) {
        if (lane == 0) idx[have] = cand;
        ++have;
        __syncwarp();
      }
    }
    if (lane == 0 && have < k) atomicOr(status, kStatBadArg);
  }
  __syncthreads();
  const int chunks = d / 16;
  for (int i = threadIdx.x; i < k * chunks; i += blockDim.x) {
    const int m = i / chunks, c16 = i % chunks;
    uint4 w;
    if constexpr (kHalf) {
      // 16 fp16 features (exact integers) -> 16 int8
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) +
                                                        ((size_t)bh * N + idx[m]) * d) + 2 * c16;
      uint32_t o[4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 in = src[h];
        const uint32_t iw[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          uint32_t word = 0;
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            const uint32_t hw = iw[2 * e + f / 2] >> (16 * (f % 2));
            const int q = __half2int_rn(__ushort_as_half((uint16_t)(hw & 0xFFFFu)));
            word |= ((uint32_t)(q & 0xFF)) << (8 * f);
          }
          o[2 * h + e] = word;
        }
      }
      w = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      w = reinterpret_cast<const uint4*>(static_cast<const int8_t*>(x) +
                                         ((size_t)bh * N + idx[m]) * d)[c16];
    }
    reinterpret_cast<uint4*>(cent + ((size_t)bh * k + m) * d)[c16] = w;
  }
  int4* s4 = reinterpret_cast<int4*>(sums + (size_t)bh * k * d);
  for (int i = threadIdx.x; i < k * d / 4; i += blockDim.x) s4[i] = make_int4(0, 0, 0, 0);
  for (int m = threadIdx.x; m < k; m += blockDim.x) counts[(size_t)bh * k + m] = 0;
}

// grid BH, 128 threads: warm start (paper §3.2, "Unbalanced clusters cost
// little": each step starts from the previous step's centroids).  The cached
// centroids, on the grid of the cached scale s', move to this call's grid
// s = amax / 127 at the same value-space position: c = clamp(RNE(c (s' / s)),
// -127, 127), the ratio and the product rounded to fp32.  Runs before the
// features kernel overwrites s'; zeroes the sums.
__global__ void kmeans_warm_kernel(const uint32_t* amax_bits, const float* grid_scale,
                                   int8_t* cent, int32_t* sums, int32_t* counts, int k, int d,
                                   const int* status) {
  if (prep_skip(status)) return;
  const int bh = blockIdx.x;
  const float amax = __uint_as_float(amax_bits[bh]);
  const float s = amax > 0.0f ? __fdiv_rn(amax, 127.0f) : 1.0f;
  const float r = __fdiv_rn(grid_scale[bh], s);
  for (int i = threadIdx.x; i < k * d; i += blockDim.x) {
    int8_t* c = cent + (size_t)bh * k * d + i;
    const int t = __float2int_rn(__fmul_rn((float)*c, r));
    *c = (int8_t)max(-127, min(127, t));
    sums[(size_t)bh * k * d + i] = 0;
  }
  for (int m = threadIdx.x; m < k; m += blockDim.x) counts[(size_t)bh * k + m] = 0;
}

// grid (ceil(N / kAssignTokens), BH), 256 threads.  Phase 1: every token's
// nearest centroid by exact integer distance ||c||^2 - 2 x.c (the token's own
// norm is common to all centroids), lowest index on ties.  Phase 2: the tile's
// per-cluster channel sums in shared memory (one thread per channel, tokens in
// order, no atomics), then one global atomic add per (cluster, channel).
constexpr int kAssignTokens = 1024;
// Shared words of the assign kernel for k clusters and `groups` accumulators.
inline size_t assign_smem_bytes(int k, int groups) {
  return (size_t)(k * 32 + k + kAssignTokens + groups * (k * 128 + k)) * 4;
}
__global__ void __launch_bounds__(256) kmeans_assign_kernel(const int8_t* x, const int8_t* cent,
                                                            int32_t* labels, int32_t* sums,
                                                            int32_t* counts, int N, int k,
                                                            int groups, const int* status) {
  extern __shared__ int32_t sm[];
  int32_t* cw = sm;                      // centroids as packed int8x4 words [k][32]
  int32_t* cnorm = cw + k * 32;          // [k]
  int32_t* lab = cnorm + k;              // [kAssignTokens]
  int32_t* acc = lab + kAssignTokens;    // [groups][k*128 sums + k counts]
  if (prep_skip(status)) return;
  const int bh = blockIdx.y, t0 = blockIdx.x * kAssignTokens;
  const int ntok = min(kAssignTokens, N - t0);
  const int32_t* cg = reinterpret_cast<const int32_t*>(cent + (size_t)bh * k * 128);
  for (int i = threadIdx.x; i < k * 32; i += blockDim.x) cw[i] = cg[i];
  for (int i = threadIdx.x; i < groups * (k * 128 + k); i += blockDim.x) acc[i] = 0;
  __syncthreads();
  for (int m = threadIdx.x; m < k; m += blockDim.x) {
    int32_t n2 = 0;
    for (int w = 0; w < 32; ++w) n2 = __dp4a(cw[m * 32 + w], cw[m * 32 + w], n2);
    cnorm[m] = n2;
  }
  __syncthreads();
  const int8_t* xh = x + ((size_t)bh * N + t0) * 128;
  for (int t = threadIdx.x; t < ntok; t += blockDim.x) {
    int32_t xw[32];
    const int4* row = reinterpret_cast<const int4*>(xh + (size_t)t * 128);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      int4 v = row[q];
      xw[4 * q] = v.x; xw[4 * q + 1] = v.y; xw[4 * q + 2] = v.z; xw[4 * q + 3] = v.w;
    }
    int best = 0x7FFFFFFF, bestm = 0;
    for (int m = 0; m < k; ++m) {
      int32_t dot = 0;
#pragma unroll
      for (int w = 0; w < 32; ++w) dot = __dp4a(xw[w], cw[m * 32 + w], dot);
      const int dist = cnorm[m] - 2 * dot;
      if (dist < best) { best = dist; bestm = m; }
    }
    lab[t] = bestm;
    labels[(size_t)bh * N + t0 + t] = bestm;
  }
  __syncthreads();
  // phase 2: `groups` groups of 128 threads (one per channel), each over a
  // contiguous share of the tile's tokens, in token order
  const int g = threadIdx.x / 128, c = threadIdx.x % 128;
  if (g < groups) {
    int32_t* a = acc + g * (k * 128 + k);
    const int share = (ntok + groups - 1) / groups, lo = g * share, hi = min(ntok, lo + share);
    for (int t = lo; t < hi; ++t) {
      const int z = lab[t];
      a[z * 128 + c] += (int32_t)xh[(size_t)t * 128 + c];
      if (c == 0) a[k * 128 + z] += 1;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < k * 128 + k; i += blockDim.x) {
    int32_t s = 0;
    for (int gg = 0; gg < groups; ++gg) s += acc[gg * (k * 128 + k) + i];
    if (s != 0) {
      if (i < k * 128) atomicAdd(&sums[(size_t)bh * k * 128 + i], s);
      else atomicAdd(&counts[(size_t)bh * k + (i - k * 128)], s);
    }
  }
}

// One Lloyd iteration on the tensor cores, for k <= 128.  grid (chunks, BH),
// 256 threads; a CTA owns a run of 128-token tiles [tile0, tile0 + nt) of one
// head.  The features are fp16 (the int8 grid values, exact) and accumulate
// in fp32 (exact: every dot product and every per-CTA sum of at most
// kPipeMaxTiles tiles stays below 2^24).  Per tile:
//   D_a = X C^T       (M = 128 tokens, N = kpad centroids, K = 128 channels)
//   label_t = argmin_m ||c_m||^2 - 2 D_a[t, m]  (lowest index on ties)
//   D_u += X^T H      (M = 128 channels, N = kpad clusters, K = 128 tokens)
// with H the one-hot label matrix.  The producer TMA-loads each fp16 tile as
// two 128-byte-swizzled atoms (channels 0-63, 64-127) straight into one of nx
// X buffers; that image is the K-major A operand of the first product and the
// MN-major A operand of the second, and is reloaded once the second product
// of its tile is done.  H is stored K-major as H^T.
// Warp roles: warp 0 TMA producer; warp 1 MMA issuer and TMEM owner; warps
// 4-7, one token row per thread (the TMEM lane), take each tile's argmin and
// write its one-hot column while the products of the neighbouring tiles run.
// H^T and D_a are triple-buffered, and the cluster-sum product of tile t - 2
// follows the assign product of tile t, so the argmin of a tile has two
// products' time before its one-hot columns are needed.  The CTA's cluster
// sums D_u and counts are added to the global sums once at the end.
// Each product is 8 instructions of K = 16 at N = kpad <= 128, which take
// about as long as N = 144 ones: the tensor time of a tile is about 16 x 70
// cycles, and at k = 64 the fp16 features read from HBM cost about as much.
constexpr int kPipeMaxTiles = 1024;                   // 1024 * 128 * 127 < 2^24
constexpr int kPipeMaxX = 5;
// shared memory: X fp16 nx x 32 KB | H^T fp16 3 x kpad x 256 B | centroids fp16
// kpad x 256 B.  H^T[b] holds two 128-byte-swizzled atoms of kpad rows
// (tokens 0-63, 64-127).
constexpr uint32_t kPipeStaticSmem = 2048;            // the kernel's static shared memory, rounded up
__host__ __device__ inline uint32_t kpipe_h(int nx) { return nx * 32768u; }
__host__ __device__ inline uint32_t kpipe_c(int nx, int kpad) {
  return kpipe_h(nx) + 3u * 256u * (uint32_t)kpad;
}
inline size_t kmeans_pipe_smem_bytes(int kpad, int nx) {
  return kpipe_c(nx, kpad) + (size_t)kpad * 256 + 1024;
}

// barrier indices
enum { KB_XFULL = 0, KB_DA = KB_XFULL + kPipeMaxX, KB_HREADY = KB_DA + 3, KB_UDONE = KB_HREADY + 3,
       KB_CNT = KB_UDONE + kPipeMaxX, KB_DRAIN = KB_CNT + 1, KB_COUNT = KB_DRAIN + 1 };

constexpr int kPipeThreads = 256;
__global__ void __launch_bounds__(kPipeThreads, 1)
    kmeans_assign_pipe_kernel(const __grid_constant__ CUtensorMap tmX, const int8_t* cent,
                              int32_t* labels, int32_t* sums, int32_t* counts, int N, int k,
                              int kpad, int tiles_per_cta, int nx, int* status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t bars[KB_COUNT];
  __shared__ int abort_flag;
  __shared__ int32_t cnt[128];
  __shared__ float cnorm[128];  // ||c_m||^2, an integer below 2^24
  if (prep_skip(status)) return;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int bh = blockIdx.y;
  const int tile0 = blockIdx.x * tiles_per_cta;
  const int nt = min(tiles_per_cta, (N + 127) / 128 - tile0);
  if (nt <= 0) return;  // uniform over the CTA
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t kPX = 0, kPH = kpipe_h(nx), kPC = kpipe_c(nx, kpad);
  const uint32_t hatom = (uint32_t)kpad * 128;    // one H^T atom: kpad rows x 128 B
  const uint32_t hbuf = 2 * hatom;
  // D_a[b] at b * kpad (b < 3); the argmin reads max(64, kpad rounded up to
  // 32) columns from there, so D_u starts past what D_a[2]'s reader touches
  const uint32_t col_u = 2u * (uint32_t)kpad + (uint32_t)(kpad <= 64 ? 64 : (kpad + 31) / 32 * 32);
  const uint32_t ncols = col_u + (uint32_t)kpad <= 256 ? 256 : 512;
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), ncols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < KB_COUNT; ++i) {
      const bool workers = (i >= KB_HREADY && i < KB_HREADY + 3) || i == KB_CNT;
      mbar_init(bar(i), workers ? 128 : 1);
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tensormap(&tmX);
  }
  // centroids -> fp16, K-major 128-byte swizzle: two atoms of kpad rows x 64
  // channels; rows k..kpad-1 are zero
  const int8_t* cg = cent + (size_t)bh * k * 128;
  for (int i = tid; i < kpad * 16; i += kPipeThreads) {  // one 16-byte chunk (8 channels) per step
    const int m = i / 16, c8 = i % 16, atom = c8 / 8, ch = c8 % 8;
    uint32_t w[4] = {0, 0, 0, 0};
    if (m < k) {
      const uint2 src = *reinterpret_cast<const uint2*>(cg + (size_t)m * 128 + c8 * 8);
      i8x4_to_f16x4(src.x, w[0], w[1]);
      i8x4_to_f16x4(src.y, w[2], w[3]);
    }
    *reinterpret_cast<uint4*>(sm + kPC + atom * kpad * 128 + m * 128 + ((ch ^ (m & 7)) << 4)) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
  for (int m = tid; m < 128; m += kPipeThreads) {
    cnt[m] = 0;
    int32_t n2 = 0;
    if (m < k)
      for (int c = 0; c < 128; ++c) {
        const int v = cg[(size_t)m * 128 + c];
        n2 += v * v;
      }
    cnorm[m] = (float)n2;
  }
  // the one-hot buffers start at zero; a worker later clears only the entry
  // it set three tiles before
  for (int i = tid; i < (int)(3 * hbuf / 16); i += kPipeThreads)
    reinterpret_cast<uint4*>(sm + kPH)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    int issued = 0;
    for (int t = 0; t < nt; ++t) {
      const int xi = t % nx;
      // X[xi] was last read by the cluster-sum product of tile t - nx
      if (t >= nx) ok = mbar_wait(bar(KB_UDONE + xi), ((t / nx) - 1) & 1, &abort_flag, status);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (lane == 0) {
        const uint32_t xb = base + kPX + xi * 32768;
        const int row = bh * N + (tile0 + t) * 128;
        mbar_expect_tx(bar(KB_XFULL + xi), 32768);
        tma_load_2d(xb, &tmX, bar(KB_XFULL + xi), 0, row);            // channels 0-63
        tma_load_2d(xb + 16384, &tmX, bar(KB_XFULL + xi), 64, row);   // channels 64-127
      }
      ++issued;
    }
    if (lane == 0 && abort_flag) {
      // let the copies in flight land before the CTA exits
      const uint64_t t0 = globaltimer();
      for (int t = max(0, issued - nx); t < issued; ++t)
        while (!mbar_try_wait(bar(KB_XFULL + t % nx), (t / nx) & 1) &&
               globaltimer() - t0 < kWaitLimitNs) {
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // per step t: assign(t) once tile t has landed, update(t-2) once its
    // one-hot columns are written
    const uint32_t ia = idesc_f16(128, kpad), iu = idesc_f16(128, kpad, false, true);
    bool ok = true;
    for (int t = 0; t <= nt + 1 && ok; ++t) {
      if (t < nt) {
        const int b = t % 3, xi = t % nx;
        ok = mbar_wait(bar(KB_XFULL + xi), (t / nx) & 1, &abort_flag, status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const uint32_t xb = base + kPX + xi * 32768;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t o = (s / 4) * 16384 + (s % 4) * 32;
          const uint32_t oc = (s / 4) * kpad * 128 + (s % 4) * 32;
          mma_f16_ss_w(tmem + b * kpad, desc_k_sw128(xb + o), desc_k_sw128(base + kPC + oc), ia,
                       s > 0);
        }
        mma_commit_w(bar(KB_DA + b));
      }
      if (t >= 2) {
        const int u = t - 2, b = u % 3;
        ok = mbar_wait(bar(KB_HREADY + b), (u / 3) & 1, &abort_flag, status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const uint32_t xb = base + kPX + (u % nx) * 32768, hb = base + kPH + b * hbuf;
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_f16_ss_w(tmem + col_u, make_desc(xb + s * 2048, 16384, 1024, 2),
                       desc_k_sw128(hb + (s / 4) * hatom + (s % 4) * 32), iu, (u > 0 || s > 0));
        mma_commit_w(bar(KB_UDONE + u % nx));
      }
    }
    // every issued product completes before the CTA releases its tensor memory
    mma_commit_w(bar(KB_DRAIN));
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar(KB_DRAIN), 0) && globaltimer() - t0 < kWaitLimitNs) {
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ argmin workers
    const int wt = tid - 128, quarter = warp - 4;  // token row / cluster row = TMEM lane
    const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
    int old_lab[3] = {-1, -1, -1};  // the entry this thread set in H^T[b] three tiles before
    bool ok = true;
    // used when kpad <= 64: ||c_m||^2 + 2^23 + 2^21 for a cluster, 1.5 * 2^24 past k
    float cn[64];
#pragma unroll
    for (int m = 0; m < 64; ++m) cn[m] = m < k ? cnorm[m & 127] + 10485760.0f : 25165824.0f;
    for (int u = 0; u < nt && ok; ++u) {
      {
        // tile u: argmin of this token's row of D_a, then its one-hot column
        const int b = u % 3;
        ok = mbar_wait(bar(KB_DA + b), (u / 3) & 1, &abort_flag, status);
        // H^T[b] was last read by the cluster-sum product of tile u - 3
        if (ok && u >= 3) ok = mbar_wait(bar(KB_UDONE + (u - 3) % nx), ((u - 3) / nx) & 1, &abort_flag, status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const uint32_t trow = tmem + lanes + b * kpad;
        // distances ||c||^2 - 2 x.c are integers below 2^24: exact in fp32;
        // the strict comparison keeps the lowest index on ties
        float best = INFINITY;
        int bestm = 0;
        if (kpad <= 64) {
          // one packed key per cluster, minimised over a tree.  With x and c
          // in [-127, 127]^128, d = ||c||^2 - 2 x.c lies in [-||x||^2,
          // 6193536] and ||x||^2 <= 2064512, so f = d + 2^23 + 2^21 is an
          // integer in [2^23, 2^24): exact in fp32, its low 23 bits are
          // f - 2^23, and (bits(f) << 6) + m orders by (d, m), lowest index
          // on ties.  A zero centroid row past k gives f = 1.5 * 2^24 (key
          // >= 0xE0000000, above every cluster's); columns past kpad hold
          // other data and are forced to the largest key.
          uint32_t v[64];
          tmem_ld32(trow, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          if (kpad > 32) {
            tmem_ld32(trow + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          } else {
#pragma unroll
            for (int m = 32; m < 64; ++m) v[m] = 0u;
          }
          tmem_ld_wait();
          uint32_t key[64];
#pragma unroll
          for (int m = 0; m < 64; ++m)
            key[m] = (__float_as_uint(fmaf(-2.0f, __uint_as_float(v[m]), cn[m])) << 6) + (uint32_t)m;
          if (kpad < 64) {
#pragma unroll
            for (int m = 16; m < 64; ++m)
              if (m >= kpad) key[m] = 0xFFFFFFFFu;
          }
#pragma unroll
          for (int s = 32; s >= 1; s >>= 1)
#pragma unroll
            for (int m = 0; m < s; ++m) key[m] = min(key[m], key[m + s]);
          bestm = (int)(key[0] & 63u);
        } else {
          for (int c0 = 0; c0 < kpad; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(trow + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const int m = c0 + c;
              if (m < k) {
                const float dist = fmaf(-2.0f, __uint_as_float(v[c]), cnorm[m]);
                if (dist < best) { best = dist; bestm = m; }
              }
            }
          }
        }
        const int token = (tile0 + u) * 128 + wt;
        uint8_t* hb = sm + kPH + b * hbuf;
        // H^T[m][token] at (token / 64) * hatom + m * 128 B, 16-byte chunk
        // (token % 64) / 8 swizzled with m % 8, element token % 8
        auto hoff = [&](int m) {
          return (wt / 64) * hatom + m * 128 + ((((wt % 64) / 8) ^ (m & 7)) << 4) + (wt % 8) * 2;
        };
        if (old_lab[b] >= 0) *reinterpret_cast<uint16_t*>(hb + hoff(old_lab[b])) = 0;
        old_lab[b] = -1;
        if (token < N) {
          labels[(size_t)bh * N + token] = bestm;
          atomicAdd(&cnt[bestm], 1);
          *reinterpret_cast<uint16_t*>(hb + hoff(bestm)) = 0x3C00;  // 1.0 (fp16)
          old_lab[b] = bestm;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(KB_HREADY + b));
      }
    }
    // the CTA's cluster sums (TMEM lane c = channel c, column m = cluster m)
    // and counts
    mbar_arrive(bar(KB_CNT));
    if (ok) ok = mbar_wait(bar(KB_UDONE + (nt - 1) % nx), ((nt - 1) / nx) & 1, &abort_flag, status);
    if (ok) ok = mbar_wait(bar(KB_CNT), 0, &abort_flag, status);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int c = wt;
      for (int m0 = 0; m0 < kpad; m0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lanes + col_u + m0, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int m = m0 + i;
          const int sv = (int)__uint_as_float(v[i]);
          if (m < k && sv) atomicAdd(&sums[((size_t)bh * k + m) * 128 + c], sv);
        }
      }
      if (wt < k && cnt[wt]) atomicAdd(&counts[(size_t)bh * k + wt], cnt[wt]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// Round-half-even of s / n (n > 0) in exact integer arithmetic.
__device__ __forceinline__ int div_rne(int s, int n) {
  int q = s / n, r = s % n;
  if (r < 0) { q -= 1; r += n; }
  if (2 * r > n || (2 * r == n && (q & 1))) q += 1;
  return q;
}

// grid (BH, k), 128 threads: centroid = RNE integer mean of its members; an
// empty cluster keeps its centroid.  Clears the sums for the next iteration.
__global__ void kmeans_update_kernel(int8_t* cent, int32_t* sums, int32_t* counts, int k,
                                     const int* status) {
  if (prep_skip(status)) return;
  const int bh = blockIdx.x, m = blockIdx.y, c = threadIdx.x;
  const size_t o = ((size_t)bh * k + m) * 128 + c;
  const int n = counts[(size_t)bh * k + m];
  if (n > 0) cent[o] = (int8_t)div_rne(sums[o], n);
  sums[o] = 0;
  __syncthreads();
  if (c == 0) counts[(size_t)bh * k + m] = 0;
}

// ---------------------------------------------------------------------------
// Stable counting sort of the labels: pi = argsort(z) (paper Eq 3)
// ---------------------------------------------------------------------------
constexpr int kSortChunk = 2048;
// grid (chunks, BH): hist[bh][label][chunk]
__global__ void sort_hist_kernel(const int32_t* labels, int32_t* hist, int N, int k, int nchunk,
                                 const int* status) {
  __shared__ int32_t h[256];
  if (prep_skip(status)) return;
  const int bh = blockIdx.y, ch = blockIdx.x;
  for (int i = threadIdx.x; i < k; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int t0 = ch * kSortChunk, t1 = min(N, t0 + kSortChunk);
  for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
    const int z = labels[(size_t)bh * N + t];
    if (index_ok(z, k, status)) atomicAdd(&h[z], 1);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < k; i += blockDim.x)
    hist[((size_t)bh * k + i) * nchunk + ch] = h[i];
}

// grid BH, 256 threads: hist -> exclusive offsets in (label, chunk) order.
__global__ void sort_scan_kernel(int32_t* hist, int k, int nchunk, const int* status) {
  __shared__ int32_t tot[256];
  if (prep_skip(status)) return;
  const int bh = blockIdx.x;
  int32_t* hh = hist + (size_t)bh * k * nchunk;
  for (int m = threadIdx.x; m < k; m += blockDim.x) {
    int s = 0;
    for (int c = 0; c < nchunk; ++c) s += hh[m * nchunk + c];
    tot[m] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int m = 0; m < k; ++m) { const int t = tot[m]; tot[m] = run; run += t; }
  }
  __syncthreads();
  for (int m = threadIdx.x; m < k; m += blockDim.x) {
    int run = tot[m];
    for (int c = 0; c < nchunk; ++c) { const int t = hh[m * nchunk + c]; hh[m * nchunk + c] = run; run += t; }
  }
}

// grid (chunks, BH), 256 threads: stable scatter.  Tokens of a chunk are taken
// in rounds of 256 in order; within a round a token's rank among equal labels
// comes from warp match masks and per-warp counts.
__global__ void __launch_bounds__(256) sort_scatter_kernel(const int32_t* labels,
                                                           const int32_t* offs, int32_t* perm,
                                                           int N, int k, int nchunk,
                                                           const int* status) {
  __shared__ int32_t base[256];
  __shared__ int32_t wcnt[8][256];
  if (prep_skip(status)) return;
  const int bh = blockIdx.y, ch = blockIdx.x, w = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int m = threadIdx.x; m < k; m += blockDim.x)
    base[m] = offs[((size_t)bh * k + m) * nchunk + ch];
  const int t0 = ch * kSortChunk, t1 = min(N, t0 + kSortChunk);
  for (int r0 = t0; r0 < t1; r0 += 256) {
    for (int i = threadIdx.x; i < 8 * 256; i += blockDim.x) (&wcnt[0][0])[i] = 0;
    __syncthreads();
    const int t = r0 + threadIdx.x;
    const int zt = t < t1 ? labels[(size_t)bh * N + t] : -1;
    const bool valid = t < t1 && index_ok(zt, k, status);
    const int z = valid ? zt : -1 - lane;  // unique per invalid lane
    const unsigned same = __match_any_sync(0xffffffffu, z);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (valid && rank == 0) wcnt[w][z] = __popc(same);
    __syncthreads();
    if (valid) {
      int pos = base[z] + rank;
      for (int ww = 0; ww < w; ++ww) pos += wcnt[ww][z];
      if (index_ok(pos, N, status)) perm[(size_t)bh * N + pos] = t;
    }
    __syncthreads();
    for (int m = threadIdx.x; m < k; m += blockDim.x) {
      int s = 0;
      for (int ww = 0; ww < 8; ++ww) s += wcnt[ww][m];
      base[m] += s;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Quantizers (8-bit)
// ---------------------------------------------------------------------------
// Load 64 consecutive bf16 of a row into fp32.
__device__ __forceinline__ void load64(const uint16_t* src, float (&f)[64]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint4 w = s[q];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[q * 8 + 2 * e] = __uint_as_float(ws[e] << 16);
      f[q * 8 + 2 * e + 1] = __uint_as_float(ws[e] & 0xFFFF0000u);
    }
  }
}
// The QK Hadamard rotation of one 128-channel row held by a lane pair (lane
// parity h holds channels 64h .. 64h+63): the fast transform, butterflies
// (a, b) -> (a + b, a - b) on channels (i, i + s), i & s = 0, for s = 1 .. 32
// inside a lane and s = 64 across the pair (the even lane keeps a + b, the odd
// one a - b), then one multiply by fp32(1/sqrt(128)).  The whole warp calls it.
__device__ __forceinline__ void hadamard128_pair(float (&f)[64], int h) {
#pragma unroll
  for (int s = 1; s < 64; s <<= 1)
#pragma unroll
    for (int i = 0; i < 64; ++i)
      if ((i & s) == 0) {
        const float a = f[i], b = f[i + s];
        f[i] = __fadd_rn(a, b);
        f[i + s] = __fsub_rn(a, b);
      }
  constexpr float kInvSqrt128 = 0x1.6a09e6p-4f;  // fp32(1/sqrt(128))
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const float o = __shfl_xor_sync(0xffffffffu, f[i], 1);
    f[i] = __fmul_rn(h == 0 ? __fadd_rn(f[i], o) : __fsub_rn(o, f[i]), kInvSqrt128);
  }
}

// The same rotation of one row held by a half-warp (lane c8 = lane % 16 holds
// channels 8 c8 .. 8 c8 + 7): the butterflies of strides 1, 2, 4 inside a
// lane and 8, 16, 32, 64 across lanes c8 ^ 1, ^ 2, ^ 4, ^ 8 (the lower lane
// keeps a + b, the upper one a - b), in that order, then the multiply by
// fp32(1/sqrt(128)): the operations of hadamard128_pair on every value.
__device__ __forceinline__ void hadamard128_rows(float (&f)[8], int c8) {
#pragma unroll
  for (int s = 1; s < 8; s <<= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((i & s) == 0) {
        const float a = f[i], b = f[i + s];
        f[i] = __fadd_rn(a, b);
        f[i + s] = __fsub_rn(a, b);
      }
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {
    const bool upper = (c8 & m) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, f[i], m);
      f[i] = upper ? __fsub_rn(o, f[i]) : __fadd_rn(f[i], o);
    }
  }
  constexpr float kInvSqrt128 = 0x1.6a09e6p-4f;  // fp32(1/sqrt(128))
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], kInvSqrt128);
}

// Step u of a row-mapped block kernel (half-warp = one row, lane c8 = 8
// channels): the 8 values of row j * 128 + 16 u + t / 16 (0 past N), gathered
// through perm and centred by kbar (as fp32 words c) when given, rotated
// when kRot.
template <bool kRot>
__device__ __forceinline__ void load_row8(const uint16_t* x, const int32_t* perm, bool centre,
                                          const float (&c)[8], int bh, int j, int u, int t,
                                          int N, float (&v)[8], const int* status) {
  const int c8 = t % 16, row = j * 128 + u * 16 + t / 16;
#pragma unroll
  for (int e = 0; e < 8; ++e) v[e] = 0.0f;
  const int src = row < N ? (perm ? perm[(size_t)bh * N + row] : row) : -1;
  if (row < N && index_ok(src, N, status)) {
    const uint4 w = *reinterpret_cast<const uint4*>(x + ((size_t)bh * N + src) * 128 + c8 * 8);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[2 * e] = __uint_as_float(ws[e] << 16);
      v[2 * e + 1] = __uint_as_float(ws[e] & 0xFFFF0000u);
    }
    if (centre)
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = __fsub_rn(v[e], c[e]);
  }
  if constexpr (kRot) hadamard128_rows(v, c8);
}

// E4M3 codes (RNE, saturating) of the correctly rounded quotients x / s,
// mostly without dividing.  With r the rounded reciprocal of s, the products
// x rlo and x rhi (rlo, rhi = r (1 -/+ 2^-20) rounded) carry at most three
// roundings of 2^-24 each, so they bracket the rounded quotient in
// magnitude; the E4M3 cast is monotone in magnitude, so when both ends give
// the same code it is the quotient's.  Otherwise (a quotient within about
// 2^-20 of an E4M3 rounding boundary, rare) the division runs exactly.
struct QuotBracket {
  float s, rlo, rhi;
};
__device__ __forceinline__ QuotBracket quot_bracket(float s) {
  const float r = __frcp_rn(s);
  return {s, __fmul_rn(r, 1.0f - 0x1p-20f), __fmul_rn(r, 1.0f + 0x1p-20f)};
}
// the rare exact path, out of line so that the common one keeps few registers
__device__ __noinline__ uint32_t e4m3x2_div(float x0, float x1, float s) {
  return f32x2_to_e4m3x2(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
}
__device__ __forceinline__ uint32_t e4m3x2_quot(float x0, float x1, const QuotBracket& q) {
  const uint32_t lo = f32x2_to_e4m3x2(__fmul_rn(x0, q.rlo), __fmul_rn(x1, q.rlo));
  const uint32_t hi = f32x2_to_e4m3x2(__fmul_rn(x0, q.rhi), __fmul_rn(x1, q.rhi));
  if (lo == hi) return lo;
  return e4m3x2_div(x0, x1, q.s);
}

__device__ __forceinline__ void store64_e4m3(uint8_t* dst, const float (&f)[64], float s) {
  const QuotBracket qb = quot_bracket(s);
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = q * 16 + e * 4;
      const uint32_t lo = e4m3x2_quot(f[i], f[i + 1], qb);
      const uint32_t hi = e4m3x2_quot(f[i + 2], f[i + 3], qb);
      w[e] = lo | (hi << 16);
    }
    d[q] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Eight E4M3 codes (one uint2) of the correctly rounded quotients x / s.
__device__ __forceinline__ uint2 e4m3x8_quot(const float (&x)[8], const QuotBracket& qb) {
  return make_uint2(e4m3x2_quot(x[0], x[1], qb) | (e4m3x2_quot(x[2], x[3], qb) << 16),
                    e4m3x2_quot(x[4], x[5], qb) | (e4m3x2_quot(x[6], x[7], qb) << 16));
}

// grid (nb, BH), 256 threads, without the rotation: per 128-token block
// sQ = amax / 448 and Q^ = E4M3(Q / sQ).  Step q (0..7) of thread t covers
// the 8 values at q * 2048 + 8 t of the block (16 rows per step, each
// half-warp one whole row), so every load and store instruction of a warp
// moves one contiguous span; the values stay packed bf16 in registers.
__global__ void __launch_bounds__(256, 4) quant_q8_rows_kernel(const uint16_t* q, uint8_t* qhat,
                                                              float* sq, int N, int Npad, int nb,
                                                              const int* status) {
  __shared__ float red[8];
  if (prep_skip(status)) return;
  const int bh = blockIdx.y, j = blockIdx.x, t = threadIdx.x;
  uint4 w[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int row = j * 128 + u * 16 + t / 16;
    w[u] = row < N ? *reinterpret_cast<const uint4*>(q + ((size_t)bh * N + row) * 128 + (t % 16) * 8)
                   : make_uint4(0u, 0u, 0u, 0u);
  }
  float m = 0.0f;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    m = max3f(m, fabsf(bf_lo(w[u].x)), fabsf(bf_hi(w[u].x)));
    m = max3f(m, fabsf(bf_lo(w[u].y)), fabsf(bf_hi(w[u].y)));
    m = max3f(m, fabsf(bf_lo(w[u].z)), fabsf(bf_hi(w[u].z)));
    m = max3f(m, fabsf(bf_lo(w[u].w)), fabsf(bf_hi(w[u].w)));
  }
  const float s = e4m3_scale(block_max(m, red));
  if (t == 0) sq[(size_t)bh * nb + j] = s;
  const QuotBracket qb = quot_bracket(s);
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int row = j * 128 + u * 16 + t / 16;
    const float x[8] = {bf_lo(w[u].x), bf_hi(w[u].x), bf_lo(w[u].y), bf_hi(w[u].y),
                        bf_lo(w[u].z), bf_hi(w[u].z), bf_lo(w[u].w), bf_hi(w[u].w)};
    *reinterpret_cast<uint2*>(qhat + ((size_t)bh * Npad + row) * 128 + (t % 16) * 8) =
        e4m3x8_quot(x, qb);
  }
}

// grid (nb, BH), 256 threads: per 128-token block, sQ = amax / 448 and
// Q^ = E4M3(Q / sQ).  Thread t covers row t/2, channels 64*(t%2) ..., so a
// lane pair holds the row that hadamard128_pair rotates: the launch path of
// the QK rotation (quant_q8_rows_kernel serves the unrotated one).
__global__ void __launch_bounds__(256, 3) quant_q8_kernel(const uint16_t* q, uint8_t* qhat, float* sq,
                                                       int N, int Npad, int nb, int hadamard,
                                                       const int* status) {
  __shared__ float red[8];
  if (prep_skip(status)) return;
  const int bh = blockIdx.y, j = blockIdx.x;
  const int r = threadIdx.x / 2, h = threadIdx.x % 2, row = j * 128 + r;
  float f[64];
  if (row < N) load64(q + ((size_t)bh * N + row) * 128 + h * 64, f);
  else
    for (int i = 0; i < 64; ++i) f[i] = 0.0f;
  if (hadamard) hadamard128_pair(f, h);
  float m = 0.0f;
  for (int i = 0; i < 64; ++i) m = fmaxf(m, fabsf(f[i]));
  const float s = e4m3_scale(block_max(m, red));
  if (threadIdx.x == 0) sq[(size_t)bh * nb + j] = s;
  store64_e4m3(qhat + ((size_t)bh * Npad + row) * 128 + h * 64, f, s);
}

// Fixed pairwise tree over 128 values: v[r] += v[r + 64], then + 32, ... .
__device__ __forceinline__ float tree128(float (&v)[128]) {
#pragma unroll
  for (int s = 64; s >= 1; s >>= 1)
#pragma unroll
    for (int r = 0; r < s; ++r) v[r] = __fadd_rn(v[r], v[r + s]);
  return v[0];
}

// grid (nb, BH), 256 threads: fp32 tree sum of each block of the original key
// order.  The block is staged in shared memory with coalesced 16-byte loads
// of whole rows (zero rows past N); threads 0..127 then sum one channel each.
__global__ void __launch_bounds__(256) key_block_sum_kernel(const uint16_t* k, float* ksum, int N,
                                                            int nb, const int* status) {
  __shared__ __align__(16) uint16_t tile[128][128];
  if (prep_skip(status)) return;
  const int bh = blockIdx.y, j = blockIdx.x, c = threadIdx.x;
  {
    // thread t: 16-byte chunk t % 16 of rows t / 16 + 16u, all eight loads in flight
    const int c16 = threadIdx.x % 16, r0 = threadIdx.x / 16;
    uint4 w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int row = j * 128 + r0 + 16 * u;
      w[u] = row < N ? *reinterpret_cast<const uint4*>(k + ((size_t)bh * N + row) * 128 + c16 * 8)
                     : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4*>(&tile[r0 + 16 * u][c16 * 8]) = w[u];
  }
  __syncthreads();
  if (c >= 128) return;
  float v[128];
#pragma unroll
  for (int r = 0; r < 128; ++r) v[r] = bf16_bits_to_f32(tile[r][c]);
  ksum[((size_t)bh * nb + j) * 128 + c] = tree128(v);
}

// grid BH, 128 threads: kbar = bf16(fp32(sum of block sums in block order, in
// fp64, / N)).
__global__ void key_mean_kernel(const float* ksum, uint16_t* kbar, int N, int nb,
                                const int* status) {
  if (prep_skip(status)) return;
  const int bh = blockIdx.x, c = threadIdx.x;
  double t = 0.0;
  for (int j = 0; j < nb; ++j) t = __dadd_rn(t, (double)ksum[((size_t)bh * nb + j) * 128 + c]);
  kbar[(size_t)bh * 128 + c] = f32_to_bf16_bits(__double2float_rn(__ddiv_rn(t, (double)N)));
}

// grid (nb, BH), 256 threads, without the rotation: K' = K[pi] - kbar,
// per-block E4M3, with the access pattern of quant_q8_rows_kernel (each
// half-warp gathers one whole row; a thread's 8 channels, and their kbar,
// are the same in every step).
__global__ void __launch_bounds__(256, 4) quant_k8_rows_kernel(const uint16_t* k,
                                                              const int32_t* perm,
                                                              const uint16_t* kbar, uint8_t* khat,
                                                              float* sk, int N, int Npad, int nb,
                                                              const int* status) {
  __shared__ float red[8];
  if (prep_skip(status)) return;
  const int bh = blockIdx.y, j = blockIdx.x, t = threadIdx.x;
  const uint4 kb = *reinterpret_cast<const uint4*>(kbar + (size_t)bh * 128 + (t % 16) * 8);
  const float c[8] = {bf_lo(kb.x), bf_hi(kb.x), bf_lo(kb.y), bf_hi(kb.y),
                      bf_lo(kb.z), bf_hi(kb.z), bf_lo(kb.w), bf_hi(kb.w)};
  uint4 w[8];
  bool valid[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int row = j * 128 + u * 16 + t / 16;
    valid[u] = row < N;
    const int src = valid[u] ? perm[(size_t)bh * N + row] : -1;
    if (valid[u] && index_ok(src, N, status)) {
      w[u] = *reinterpret_cast<const uint4*>(k + ((size_t)bh * N + src) * 128 + (t % 16) * 8);
    } else {
      w[u] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  auto vals = [&](int u, float (&x)[8]) {
    const uint32_t ww[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = valid[u] ? __fsub_rn(bf_lo(ww[e]), c[2 * e]) : 0.0f;
      x[2 * e + 1] = valid[u] ? __fsub_rn(bf_hi(ww[e]), c[2 * e + 1]) : 0.0f;
    }
  };
  float m = 0.0f;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    float x[8];
    vals(u, x);
#pragma unroll
    for (int e = 0; e < 8; e += 2) m = max3f(m, fabsf(x[e]), fabsf(x[e + 1]));
  }
  const float s = e4m3_scale(block_max(m, red));
  if (t == 0) sk[(size_t)bh * nb + j] = s;
  const QuotBracket qb = quot_bracket(s);
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int row = j * 128 + u * 16 + t / 16;
    float x[8];
    vals(u, x);
    *reinterpret_cast<uint2*>(khat + ((size_t)bh * Npad + row) * 128 + (t % 16) * 8) =
        e4m3x8_quot(x, qb);
  }
}

// grid (nb, BH), 256 threads: K' = K[pi] - kbar, per-block E4M3, a lane pair
// per row as in quant_q8_kernel (the QK rotation's launch path;
// quant_k8_rows_kernel serves the unrotated one).
__global__ void __launch_bounds__(256, 3) quant_k8_kernel(const uint16_t* k, const int32_t* perm,
                                                       const uint16_t* kbar, uint8_t* khat,
                                                       float* sk, int N, int Npad, int nb,
                                                       int hadamard, const int* status) {
  __shared__ float red[8];
  if (prep_skip(status)) return;
  const int bh = blockIdx.y, j = blockIdx.x;
  const int r = threadIdx.x / 2, h = threadIdx.x % 2, row = j * 128 + r;
  float f[64];
  const int src = row < N ? perm[(size_t)bh * N + row] : -1;
  if (row < N && index_ok(src, N, status)) {
    load64(k + ((size_t)bh * N + src) * 128 + h * 64, f);
    const uint16_t* kb = kbar + (size_t)bh * 128 + h * 64;
    for (int i = 0; i < 64; ++i) f[i] = __fsub_rn(f[i], bf16_bits_to_f32(kb[i]));
  } else {
    for (int i = 0; i < 64; ++i) f[i] = 0.0f;
  }
  if (hadamard) hadamard128_pair(f, h);
  float m = 0.0f;
  for (int i = 0; i < 64; ++i) m = fmaxf(m, fabsf(f[i]));
  const float s = e4m3_scale(block_max(m, red));
  if (threadIdx.x == 0) sk[(size_t)bh * nb + j] = s;
  store64_e4m3(khat + ((size_t)bh * Npad + row) * 128 + h * 64, f, s);
}

// Gather the 128 permuted rows of block j (bf16, zero rows past N) into shared
// memory, with the 256 threads the callers launch: thread t loads 16-byte
// chunk t % 16 of rows t / 16 + 16u, u = 0..7, so each group of 16 lanes reads
// one whole 256-byte row.  The eight indices are read first and the eight
// rows next, so a thread has all its loads in flight at once.
__device__ __forceinline__ void gather_block(const uint16_t* v, const int32_t* perm, int bh, int j,
                                             int N, uint16_t (*tile)[128], const int* status) {
  const int c16 = threadIdx.x % 16, r0 = threadIdx.x / 16;
  int src[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int row = j * 128 + r0 + 16 * u;
    src[u] = row < N ? perm[(size_t)bh * N + row] : -1;
  }
  uint4 w[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    w[u] = make_uint4(0, 0, 0, 0);
    if (j * 128 + r0 + 16 * u < N && index_ok(src[u], N, status))
      w[u] = *reinterpret_cast<const uint4*>(v + ((size_t)bh * N + src[u]) * 128 + c16 * 8);
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4*>(&tile[r0 + 16 * u][c16 * 8]) = w[u];
}

// grid (nb, BH), 256 threads: block mean (Eq 4) of V' = V[pi]: fp32 tree sum
// over the 128 rows (row r + row r+64, then +32, ...; padded rows 0) / n_j,
// rounded to bf16; and the per-block residual channel maxima.  Threads
// 0..127 own one channel each.  Without demeaning (the steps after the
// grouping window, paper §3.4) every mean is 0 and the residual is V'.
__global__ void __launch_bounds__(256) vpass1_kernel(const uint16_t* v, const int32_t* perm,
                                                     uint16_t* mu, float* vamax, int N, int nb,
                                                     int demean, const int* status) {
  __shared__ __align__(16) uint16_t tile[128][128];
  if (prep_skip(status)) return;
  const int bh = blockIdx.y, j = blockIdx.x, c = threadIdx.x;
  const int nj = min(128, N - j * 128);
  gather_block(v, perm, bh, j, N, tile, status);
  __syncthreads();
  if (c >= 128) return;
  float x[128];
#pragma unroll
  for (int r = 0; r < 128; ++r) x[r] = bf16_bits_to_f32(tile[r][c]);
  const float mean = __fdiv_rn(tree128(x), (float)nj);
  const uint16_t m16 = demean ? f32_to_bf16_bits(mean) : (uint16_t)0;
  const float mf = bf16_bits_to_f32(m16);
  float amax = 0.0f;
  for (int r = 0; r < nj; ++r) amax = fmaxf(amax, fabsf(__fsub_rn(bf16_bits_to_f32(tile[r][c]), mf)));
  mu[((size_t)bh * nb + j) * 128 + c] = m16;
  vamax[((size_t)bh * nb + j) * 128 + c] = amax;
}

// grid BH, 256 threads: sv[c] = (max over blocks of the residual channel
// maxima) / 448, or 1 for an all-zero channel.
__global__ void vreduce_kernel(const float* vamax, float* sv, int nb, const int* status) {
  __shared__ float part[2][128];
  if (prep_skip(status)) return;
  const int bh = blockIdx.x, c = threadIdx.x % 128, half = threadIdx.x / 128;
  float m = 0.0f;
  for (int j = half; j < nb; j += 2) m = fmaxf(m, vamax[((size_t)bh * nb + j) * 128 + c]);
  part[half][c] = m;
  __syncthreads();
  if (half == 0) sv[(size_t)bh * 128 + c] = e4m3_scale(fmaxf(part[0][c], part[1][c]));
}

// grid (nb, BH), 256 threads (threads t and t + 128 share channel t % 128,
// 64 tokens each): R = V' - mu, R^ = E4M3(R / sv) written transposed (tokens
// fastest) through a swizzled shared tile, so each channel's 128 codes leave
// as one line; mutilde = mu / sv and the mean operand of the restoration MMA.  Blocks form groups of kGroup aligned
// to the last block (block j is slot (j + gpad) % kGroup of group
// (j + gpad) / kGroup); per group two 128 (channel) x 16 (K) bf16 K-major
// chunks without swizzle, element (c, k) at (c/8)*256 + (k/8)*128 + (c%8)*16
// + (k%8)*2: chunk 0 holds bf16(mutilde), chunk 1 the bf16 of the remainder;
// the operand is zeroed beforehand, so K columns kGroup..15 and leading empty
// slots stay 0.
__global__ void __launch_bounds__(256) vpass2_kernel(const uint16_t* v, const int32_t* perm,
                                                     const uint16_t* mu, const float* sv,
                                                     uint8_t* rhatT, float* mutilde,
                                                     uint8_t* mside, int N, int Npad, int nb,
                                                     int ngroups, int gpad, const int* status) {
  __shared__ __align__(16) uint16_t tile[128][128];
  __shared__ __align__(16) uint8_t codes[128 * 128];  // [channel][token], 16-byte chunks swizzled
  if (prep_skip(status)) return;
  const int bh = blockIdx.y, j = blockIdx.x;
  // threads t and t + 128 share channel c = t % 128, tokens 64 hh .. 64 hh + 63
  const int c = threadIdx.x % 128, hh = threadIdx.x / 128;
  gather_block(v, perm, bh, j, N, tile, status);
  __syncthreads();
  const size_t o = ((size_t)bh * nb + j) * 128 + c;
  const float mf = bf16_bits_to_f32(mu[o]);
  const float s = sv[(size_t)bh * 128 + c];
  const QuotBracket qb = quot_bracket(s);
#pragma unroll 2
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float y[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = hh * 64 + q * 16 + e * 4 + u;
        y[u] = (j * 128 + r < N) ? __fsub_rn(bf16_bits_to_f32(tile[r][c]), mf) : 0.0f;
      }
      w[e] = e4m3x2_quot(y[0], y[1], qb) | (e4m3x2_quot(y[2], y[3], qb) << 16);
    }
    const int chunk = (hh * 4 + q) ^ (c & 7);
    *reinterpret_cast<uint4*>(codes + c * 128 + chunk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __syncthreads();
  // each group of 8 threads stores one channel's 128 codes as one line
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = threadIdx.x + 256 * k, cc = i / 8, ch = i % 8;
    const uint4 w = *reinterpret_cast<const uint4*>(codes + cc * 128 + ((ch ^ (cc & 7)) * 16));
    *reinterpret_cast<uint4*>(rhatT + ((size_t)bh * 128 + cc) * Npad + (size_t)j * 128 + ch * 16) = w;
  }
  if (hh != 0) return;
  const float mt = __fdiv_rn(mf, s);
  mutilde[o] = mt;
  const uint16_t hi = f32_to_bf16_bits(mt);
  const uint16_t lo = f32_to_bf16_bits(__fsub_rn(mt, bf16_bits_to_f32(hi)));
  const int g = (j + gpad) / kGroup, k = (j + gpad) % kGroup;
  uint8_t* tile_g = mside + ((size_t)bh * ngroups + g) * kGroupBytes;
  const uint32_t off = (c / 8) * 256 + (c % 8) * 16 + (k / 8) * 128 + (k % 8) * 2;
  *reinterpret_cast<uint16_t*>(tile_g + off) = hi;
  *reinterpret_cast<uint16_t*>(tile_g + kGroupBytes / 2 + off) = lo;
}

// ---------------------------------------------------------------------------
// Quantizers (4-bit, NVFP4; Appx B "At 4 bits the NVFP4 microscales ...")
// ---------------------------------------------------------------------------
// Per-head NVFP4 global scale: amax / (448 * 6), so the largest 16-block gets
// the largest UE4M3 scale and its E2M1 elements reach 6; 1 for a zero tensor.
__device__ __forceinline__ float nvfp4_global(float amax) {
  return amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
}

// 16 values under global scale g: block scale UE4M3(amax / (6 g)) (returned),
// elements E2M1(x / (scale g)) packed into 8 bytes (element 2i low nibble).
__device__ __forceinline__ uint32_t nvfp4_16(const float* x, float g, uint2& packed) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(x[i]));
  const uint32_t sc = f32_to_e4m3(__fdiv_rn(m, __fmul_rn(6.0f, g)));
  const float scv = e4m3_to_f32((uint8_t)sc);
  uint32_t w[2] = {0u, 0u};
  if (scv > 0.0f) {
    // E2M1 codes of the rounded quotients x / step through the same
    // bracketing products as the E4M3 quantisers (the E2M1 cast is monotone
    // in magnitude too)
    const float step = __fmul_rn(scv, g);
    const float r = __frcp_rn(step);
    const float rlo = __fmul_rn(r, 1.0f - 0x1p-20f), rhi = __fmul_rn(r, 1.0f + 0x1p-20f);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      uint32_t c = f32x2_to_e2m1x2(__fmul_rn(x[i], rlo), __fmul_rn(x[i + 1], rlo));
      if (c != f32x2_to_e2m1x2(__fmul_rn(x[i], rhi), __fmul_rn(x[i + 1], rhi)))
        c = f32x2_to_e2m1x2(__fdiv_rn(x[i], step), __fdiv_rn(x[i + 1], step));
      w[i / 8] |= c << (4 * (i % 8));
    }
  }
  packed = make_uint2(w[0], w[1]);
  return sc;
}

// Byte offset of the scales of row m, blocks 4s..4s+3, in a 1024-byte scale
// tile (the order the tensor core reads: (kb/4)*512 + (m%32)*16 + (m/32)*4 + kb%4).
__device__ __forceinline__ uint32_t scale_tile_off(int m, int s) {
  return (uint32_t)(s * 512 + (m % 32) * 16 + (m / 32) * 4);
}


// grid (chunks, BH): max |K - kbar| of each head (the set of K' rows does not
// depend on the order), as the uint bits of a non-negative float.
__global__ void k4_amax_kernel(const uint16_t* k, const uint16_t* kbar, uint32_t* amax_bits,
                               size_t per_head, const int* status) {
  __shared__ float red[32];
  if (prep_skip(status)) return;
  const size_t bh = blockIdx.y;
  const uint4* src = reinterpret_cast<const uint4*>(k + bh * per_head);
  const uint16_t* kb = kbar + bh * 128;
  const size_t n8 = per_head / 8;
  float m = 0.0f;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint4 w = src[i];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    const int c0 = (int)((i * 8) % 128);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      m = fmaxf(m, fabsf(__fsub_rn(__uint_as_float(ws[e] << 16), bf16_bits_to_f32(kb[c0 + 2 * e]))));
      m = fmaxf(m, fabsf(__fsub_rn(__uint_as_float(ws[e] & 0xFFFF0000u),
                                   bf16_bits_to_f32(kb[c0 + 2 * e + 1]))));
    }
  }
  m = block_max(m, red);
  if (threadIdx.x == 0) atomicMax(&amax_bits[bh], __float_as_uint(m));
}

// grid (nb, BH), 256 threads: max |x H / sqrt(128)| over the rows of a head
// (x = Q, or K - kbar when kbar is given), with the row mapping of the
// block quantisers; as the uint bits of a non-negative float.
__global__ void __launch_bounds__(256) rot_amax_rows_kernel(const uint16_t* x, const uint16_t* kbar,
                                                            uint32_t* amax_bits, int N,
                                                            const int* status) {
  __shared__ float red[8];
  if (prep_skip(status)) return;
  const int bh = blockIdx.y, j = blockIdx.x, t = threadIdx.x, c8 = t % 16;
  float c[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
  if (kbar) {
    const uint4 kb = *reinterpret_cast<const uint4*>(kbar + (size_t)bh * 128 + c8 * 8);
    const uint32_t kw[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      c[2 * e] = __uint_as_float(kw[e] << 16);
      c[2 * e + 1] = __uint_as_float(kw[e] & 0xFFFF0000u);
    }
  }
  float m = 0.0f;
#pragma unroll 2
  for (int u = 0; u < 8; ++u) {
    float v[8];
    load_row8<true>(x, nullptr, kbar != nullptr, c, bh, j, u, t, N, v, status);
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[e]));
  }
  m = block_max(m, red);
  if (t == 0) atomicMax(&amax_bits[bh], __float_as_uint(m));
}


// grid BH, 256 threads: the three global scales gq, gk, gr of a head (gr from
// the per-block residual channel maxima).
__global__ void g4_kernel(const uint32_t* amax_q, const uint32_t* amax_k, const float* vamax,
                          float* g4, int nb, const int* status) {
  __shared__ float red[8];
  if (prep_skip(status)) return;
  const int bh = blockIdx.x;
  float m = 0.0f;
  for (size_t i = threadIdx.x; i < (size_t)nb * 128; i += 256)
    m = fmaxf(m, vamax[(size_t)bh * nb * 128 + i]);
  m = block_max(m, red);
  if (threadIdx.x == 0) {
    g4[bh * 4 + 0] = nvfp4_global(__uint_as_float(amax_q[bh]));
    g4[bh * 4 + 1] = nvfp4_global(__uint_as_float(amax_k[bh]));
    g4[bh * 4 + 2] = nvfp4_global(m);
    g4[bh * 4 + 3] = 0.0f;
  }
}

// Eight values of a 16-element NVFP4 block held by a lane pair (lane parity
// p holds elements 8p .. 8p+7) under global scale g: the block scale from the
// pair's maximum, then E2M1 codes of the eight values (value 2i in the low
// nibble), the same arithmetic as nvfp4_16.  Returns the scale; the whole
// warp calls it.
__device__ __forceinline__ uint32_t nvfp4_8_pair(const float (&x)[8], float g, uint32_t& packed) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[i]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  const uint32_t sc = f32_to_e4m3(__fdiv_rn(m, __fmul_rn(6.0f, g)));
  const float scv = e4m3_to_f32((uint8_t)sc);
  uint32_t w = 0u;
  if (scv > 0.0f) {
    const float step = __fmul_rn(scv, g);
    const float r = __frcp_rn(step);
    const float rlo = __fmul_rn(r, 1.0f - 0x1p-20f), rhi = __fmul_rn(r, 1.0f + 0x1p-20f);
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      uint32_t c = f32x2_to_e2m1x2(__fmul_rn(x[i], rlo), __fmul_rn(x[i + 1], rlo));
      if (c != f32x2_to_e2m1x2(__fmul_rn(x[i], rhi), __fmul_rn(x[i + 1], rhi)))
        c = f32x2_to_e2m1x2(__fdiv_rn(x[i], step), __fdiv_rn(x[i + 1], step));
      w |= c << (4 * i);
    }
  }
  packed = w;
  return sc;
}

// grid (nb, BH), 256 threads, without the rotation: Q (or K' = K[pi] - kbar
// when perm is given) in NVFP4, blocks of 16 along d.  Step u of thread t
// covers channels 8 (t % 16) .. +7 of row 16 u + t / 16 of the block, so
// each half-warp loads one whole row and stores its 64 code bytes; a lane
// pair holds one 16-element block and the even lane stores its scale.
template <bool kRot>
__global__ void __launch_bounds__(256) quant_4_rows_kernel(const uint16_t* x, const int32_t* perm,
                                                           const uint16_t* kbar, const float* g4,
                                                           int gidx, uint8_t* codes,
                                                           uint8_t* scales, size_t scale_stride,
                                                           int N, int Npad, int nb,
                                                           const int* status) {
  if (prep_skip(status)) return;
  const int bh = blockIdx.y, j = blockIdx.x, t = threadIdx.x, c8 = t % 16;
  const float g = g4[bh * 4 + gidx];
  float c[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
  if (kbar) {
    const uint4 kb = *reinterpret_cast<const uint4*>(kbar + (size_t)bh * 128 + c8 * 8);
    const uint32_t kw[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      c[2 * e] = __uint_as_float(kw[e] << 16);
      c[2 * e + 1] = __uint_as_float(kw[e] & 0xFFFF0000u);
    }
  }
  uint8_t* stile = scales + (size_t)(bh * nb + j) * scale_stride;
#pragma unroll 2
  for (int u = 0; u < 8; ++u) {
    const int m = u * 16 + t / 16, row = j * 128 + m;
    float v[8];
    load_row8<kRot>(x, perm, kbar != nullptr, c, bh, j, u, t, N, v, status);
    uint32_t pk;
    const uint32_t sc = nvfp4_8_pair(v, g, pk);
    *reinterpret_cast<uint32_t*>(codes + ((size_t)bh * Npad + row) * 64 + c8 * 4) = pk;
    if ((c8 & 1) == 0) {
      const int b = c8 / 2;  // block 0..7 of the row
      stile[(b / 4) * 512 + (m % 32) * 16 + (m / 32) * 4 + b % 4] = (uint8_t)sc;
    }
  }
}



// grid (nb, BH), 256 threads (0..127 own a channel): R = V' - mu in NVFP4,
// blocks of 16 tokens, written transposed (tokens fastest) with the scales in
// the second tile of the block's K'/R scale pair; and the block mean into the
// 4-bit mean operand (group (j + gpad) / 4, slot u = (j + gpad) % 4, K rows
// 2u, 2u+1, 8+2u, 9+2u; element (c, k) at (c/8)*256 + (k/8)*128 + (c%8)*16 +
// (k%8)*2; zeroed beforehand, so empty leading slots stay 0).
__global__ void __launch_bounds__(256) vpass2_4_kernel(const uint16_t* v, const int32_t* perm,
                                                       const uint16_t* mu, const float* g4,
                                                       uint8_t* r4T, uint8_t* kr4s,
                                                       uint8_t* mside, int N, int Npad, int nb,
                                                       int ngroups, int gpad, const int* status) {
  __shared__ __align__(16) uint16_t tile[128][128];
  if (prep_skip(status)) return;
  const int bh = blockIdx.y, j = blockIdx.x, c = threadIdx.x;
  gather_block(v, perm, bh, j, N, tile, status);
  __syncthreads();
  if (c >= 128) return;
  const size_t o = ((size_t)bh * nb + j) * 128 + c;
  const uint16_t m16 = mu[o];
  const float mf = bf16_bits_to_f32(m16);
  const float g = g4[bh * 4 + 2];
  uint8_t* dst = r4T + ((size_t)bh * 128 + c) * (Npad / 2) + (size_t)j * 64;
  uint32_t sc[2] = {0u, 0u};
#pragma unroll 1
  for (int kb = 0; kb < 8; ++kb) {
    float x[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int r = kb * 16 + u;
      x[u] = (j * 128 + r < N) ? __fsub_rn(bf16_bits_to_f32(tile[r][c]), mf) : 0.0f;
    }
    uint2 pk;
    sc[kb / 4] |= nvfp4_16(x, g, pk) << (8 * (kb % 4));
    *reinterpret_cast<uint2*>(dst + kb * 8) = pk;
  }
  uint8_t* st = kr4s + ((size_t)bh * nb + j) * 2 * kScaleTileBytes + kScaleTileBytes;
  *reinterpret_cast<uint32_t*>(st + scale_tile_off(c, 0)) = sc[0];
  *reinterpret_cast<uint32_t*>(st + scale_tile_off(c, 1)) = sc[1];
  const int grp = (j + gpad) / kGroup4, u = (j + gpad) % kGroup4;
  uint8_t* tg = mside + ((size_t)bh * ngroups + grp) * kGroup4Bytes + (c / 8) * 256 + (c % 8) * 16;
  const int ks[4] = {2 * u, 2 * u + 1, 8 + 2 * u, 9 + 2 * u};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<uint16_t*>(tg + (ks[i] / 8) * 128 + (ks[i] % 8) * 2) = m16;
}

inline int grid_chunks(size_t work, int per_block, int cap) {
  return (int)std::max<size_t>(1, std::min<size_t>((work + per_block - 1) / per_block, cap));
}

}  // namespace

// ---------------------------------------------------------------------------
// host: the preparation chain
// ---------------------------------------------------------------------------
// Header, grouping (skipped when the cached permutation is reused; started
// from the cached centroids when warm) and the key channel mean: the part of
// the chain both bit widths share.
static int launch_front(const PrepArgs& a, int bits, cudaStream_t st) {
  const int BH = a.B * a.H, N = a.N, nb = a.nb, k = a.k;
  const size_t per_head = (size_t)N * 128;
  uint8_t* S = a.state;
  const vca_state_layout& L = a.L;
  int* status = reinterpret_cast<int*>(S + L.status);
  uint32_t* hdr = reinterpret_cast<uint32_t*>(S + L.header);
  const uint16_t* kk = a.k_in;
  const uint16_t* v = a.v;
  int32_t* labels = reinterpret_cast<int32_t*>(S + L.labels);
  int32_t* perm = reinterpret_cast<int32_t*>(S + L.perm);

  header_kernel<<<1, 32, 0, st>>>(hdr, status, a.B, a.H, N, 128, k, bits, a.reuse);
  if (a.reuse == 0 || a.reuse == 2) {
    uint32_t* amax_bits = reinterpret_cast<uint32_t*>(S + L.grid);
    float* gscale = reinterpret_cast<float*>(S + L.grid) + BH;
    // features: fp16 for the tensor-core iterations (k <= 128), else int8
    void* x = S + L.features;
    const bool half_features = k <= 128;
    int8_t* cent = reinterpret_cast<int8_t*>(S + L.centroids);
    int32_t* sums = reinterpret_cast<int32_t*>(S + L.sums);
    int32_t* counts = sums + (size_t)BH * k * 128;
    zero_kernel<<<1, 256, 0, st>>>(amax_bits, BH);
    const int ch = grid_chunks(per_head / 8, 256 * 8, 1024);
    head_amax_kernel<<<dim3(ch, BH), 256, 0, st>>>(v, amax_bits, per_head, status);
    if (a.reuse == 2)
      kmeans_warm_kernel<<<BH, 128, 0, st>>>(amax_bits, gscale, cent, sums, counts, k, 128,
                                             status);
    if (half_features)
      features_kernel<true><<<dim3(ch, BH), 256, 0, st>>>(v, amax_bits, gscale, x, per_head, status);
    else
      features_kernel<false><<<dim3(ch, BH), 256, 0, st>>>(v, amax_bits, gscale, x, per_head, status);
    if (a.reuse == 0) {
      if (half_features)
        kmeans_init_kernel<true><<<BH, 128, 0, st>>>(x, cent, sums, counts, a.seed, N, k, 128, status);
      else
        kmeans_init_kernel<false><<<BH, 128, 0, st>>>(x, cent, sums, counts, a.seed, N, k, 128, status);
    }
    if (k <= 128) {
      // tensor-core Lloyd iteration (the cluster-sum product has M = 128 rows):
      // each CTA takes a run of tiles of one head, runs sized to fill whole
      // waves of the SMs (and short enough for exact fp32 sums)
      const int kpad = (k + 15) / 16 * 16;
      // nx >= 3: the producer reloads X[t % nx] after the cluster-sum product
      // of tile t - nx, which is issued two steps after that tile's assign
      int nx = kPipeMaxX;
      while (nx > 3 && kmeans_pipe_smem_bytes(kpad, nx) + kPipeStaticSmem > 232448) --nx;
      if (kmeans_pipe_smem_bytes(kpad, nx) + kPipeStaticSmem > 232448) return VCA_ERR_UNSUPPORTED;
      const size_t psmem = kmeans_pipe_smem_bytes(kpad, nx);
      cudaFuncSetAttribute(kmeans_assign_pipe_kernel,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem);
      // fp16 rows of 128 channels; a box is one 128-byte swizzle atom
      // (64 channels x 128 tokens)
      CUtensorMap tmx;
      if (!make_tmap_2d(&tmx, x, 2, 128, (uint64_t)BH * N, 256, 64, 128, 128)) return VCA_ERR_CUDA;
      int dev = 0, nsm = 152;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
      const int T = (N + 127) / 128;
      int tpc = std::min(T, kPipeMaxTiles);
      double best = 1e300;
      for (int c = 1; c <= 4 * nsm; ++c) {
        const int run = (T + c - 1) / c;
        if (run <= kPipeMaxTiles) {
          const double waves = std::ceil((double)((T + run - 1) / run) * BH / nsm);
          const double cost = waves * (run + 4);  // + the per-CTA set-up, in tiles
          if (cost < best) { best = cost; tpc = run; }
        }
        if (run == 1) break;
      }
      const dim3 grid((T + tpc - 1) / tpc, BH);
      for (int it = 0; it < a.iters; ++it) {
        kmeans_assign_pipe_kernel<<<grid, kPipeThreads, psmem, st>>>(tmx, cent, labels, sums, counts, N,
                                                             k, kpad, tpc, nx, status);
        kmeans_update_kernel<<<dim3(BH, k), 128, 0, st>>>(cent, sums, counts, k, status);
      }
    } else {
      const int groups = k <= 96 ? 2 : 1;
      const size_t asmem = assign_smem_bytes(k, groups);
      cudaFuncSetAttribute(kmeans_assign_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)asmem);
      const int tiles = (N + kAssignTokens - 1) / kAssignTokens;
      for (int it = 0; it < a.iters; ++it) {
        kmeans_assign_kernel<<<dim3(tiles, BH), 256, asmem, st>>>(
            static_cast<const int8_t*>(x), cent, labels, sums, counts, N, k, groups, status);
        kmeans_update_kernel<<<dim3(BH, k), 128, 0, st>>>(cent, sums, counts, k, status);
      }
    }
    // stable counting sort; the k-means sums buffer is reused for the histogram
    const int nchunk = (N + kSortChunk - 1) / kSortChunk;
    int32_t* hist = reinterpret_cast<int32_t*>(S + L.ksum);  // [BH][k][nchunk] fits in ksum
    sort_hist_kernel<<<dim3(nchunk, BH), 256, 0, st>>>(labels, hist, N, k, nchunk, status);
    sort_scan_kernel<<<BH, 256, 0, st>>>(hist, k, nchunk, status);
    sort_scatter_kernel<<<dim3(nchunk, BH), 256, 0, st>>>(labels, hist, perm, N, k, nchunk,
                                                          status);
  }
  uint16_t* kbar = reinterpret_cast<uint16_t*>(S + L.kbar);
  if (a.reuse == 4) {
    // naive: sequence order and no key centring (kbar = 0)
    identity_perm_kernel<<<dim3(grid_chunks((size_t)N, 256, 64), BH), 256, 0, st>>>(perm, N,
                                                                                   status);
    zero_kernel<<<1, 256, 0, st>>>(reinterpret_cast<uint32_t*>(kbar), (size_t)BH * 64);
    return VCA_OK;
  }
  float* ksum = reinterpret_cast<float*>(S + L.ksum);
  key_block_sum_kernel<<<dim3(nb, BH), 256, 0, st>>>(kk, ksum, N, nb, status);
  key_mean_kernel<<<BH, 128, 0, st>>>(ksum, kbar, N, nb, status);
  return VCA_OK;
}

int launch_prepare8(const PrepArgs& a, cudaStream_t st) {
  const int BH = a.B * a.H, N = a.N, nb = a.nb, Npad = a.Npad;
  uint8_t* S = a.state;
  const vca_state_layout& L = a.L;
  int* status = reinterpret_cast<int*>(S + L.status);
  uint32_t* hdr = reinterpret_cast<uint32_t*>(S + L.header);
  const uint16_t* q = a.q;
  const uint16_t* kk = a.k_in;
  const uint16_t* v = a.v;
  const int32_t* perm = reinterpret_cast<const int32_t*>(S + L.perm);
  if (const int rc = launch_front(a, 8, st); rc != VCA_OK) return rc;
  uint8_t* qhat = S + L.qhat;
  float* sq = reinterpret_cast<float*>(S + L.sq);
  uint8_t* khat = S + L.khat;
  float* sk = reinterpret_cast<float*>(S + L.sk);
  const uint16_t* kbar = reinterpret_cast<const uint16_t*>(S + L.kbar);
  uint8_t* rhatT = S + L.rhatT;
  float* sv = reinterpret_cast<float*>(S + L.sv);
  uint16_t* mu = reinterpret_cast<uint16_t*>(S + L.mu);
  float* mut = reinterpret_cast<float*>(S + L.mutilde);
  uint8_t* mside = S + L.mside;
  float* vamax = reinterpret_cast<float*>(S + L.vamax);
  const int had = (a.flags & VCA_PREP_QK_HADAMARD) ? 1 : 0;
  if (had) {
    // the rotation needs each row in one lane pair
    quant_q8_kernel<<<dim3(nb, BH), 256, 0, st>>>(q, qhat, sq, N, Npad, nb, had, status);
    quant_k8_kernel<<<dim3(nb, BH), 256, 0, st>>>(kk, perm, kbar, khat, sk, N, Npad, nb, had,
                                                  status);
  } else {
    quant_q8_rows_kernel<<<dim3(nb, BH), 256, 0, st>>>(q, qhat, sq, N, Npad, nb, status);
    quant_k8_rows_kernel<<<dim3(nb, BH), 256, 0, st>>>(kk, perm, kbar, khat, sk, N, Npad, nb,
                                                      status);
  }
  vpass1_kernel<<<dim3(nb, BH), 256, 0, st>>>(v, perm, mu, vamax, N, nb,
                                              a.reuse != 3 && a.reuse != 4, status);
  vreduce_kernel<<<BH, 256, 0, st>>>(vamax, sv, nb, status);
  const int ngroups = (nb + kGroup - 1) / kGroup;
  zero_kernel<<<grid_chunks((size_t)BH * ngroups * kGroupBytes / 4, 256, 4096), 256, 0, st>>>(
      reinterpret_cast<uint32_t*>(mside), (size_t)BH * ngroups * kGroupBytes / 4);
  vpass2_kernel<<<dim3(nb, BH), 256, 0, st>>>(v, perm, mu, sv, rhatT, mut, mside, N, Npad, nb,
                                              ngroups, ngroups * kGroup - nb, status);
  header_done_kernel<<<1, 32, 0, st>>>(hdr, status, a.reuse == 0 || a.reuse == 2);
  return cudaGetLastError() == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}

int launch_prepare4(const PrepArgs& a, cudaStream_t st) {
  const int BH = a.B * a.H, N = a.N, nb = a.nb, Npad = a.Npad;
  const size_t per_head = (size_t)N * 128;
  uint8_t* S = a.state;
  const vca_state_layout& L = a.L;
  int* status = reinterpret_cast<int*>(S + L.status);
  uint32_t* hdr = reinterpret_cast<uint32_t*>(S + L.header);
  const uint16_t* q = a.q;
  const uint16_t* kk = a.k_in;
  const uint16_t* v = a.v;
  const int32_t* perm = reinterpret_cast<const int32_t*>(S + L.perm);
  if (const int rc = launch_front(a, 4, st); rc != VCA_OK) return rc;
  const uint16_t* kbar = reinterpret_cast<const uint16_t*>(S + L.kbar);
  uint16_t* mu = reinterpret_cast<uint16_t*>(S + L.mu);
  float* vamax = reinterpret_cast<float*>(S + L.vamax);
  float* g4 = reinterpret_cast<float*>(S + L.g4);
  uint8_t* mside = S + L.mside;
  // per-head |Q| and |K'| maxima in the key-sum scratch (free after the key mean)
  uint32_t* amax_q = reinterpret_cast<uint32_t*>(S + L.ksum);
  uint32_t* amax_k = amax_q + BH;
  zero_kernel<<<1, 256, 0, st>>>(amax_q, 2 * (size_t)BH);
  const int ch = grid_chunks(per_head / 8, 256 * 8, 1024);
  const int had = (a.flags & VCA_PREP_QK_HADAMARD) ? 1 : 0;
  if (had) {
    rot_amax_rows_kernel<<<dim3(nb, BH), 256, 0, st>>>(q, nullptr, amax_q, N, status);
    rot_amax_rows_kernel<<<dim3(nb, BH), 256, 0, st>>>(kk, kbar, amax_k, N, status);
  } else {
    head_amax_kernel<<<dim3(ch, BH), 256, 0, st>>>(q, amax_q, per_head, status);
    k4_amax_kernel<<<dim3(ch, BH), 256, 0, st>>>(kk, kbar, amax_k, per_head, status);
  }
  vpass1_kernel<<<dim3(nb, BH), 256, 0, st>>>(v, perm, mu, vamax, N, nb,
                                              a.reuse != 3 && a.reuse != 4, status);
  g4_kernel<<<BH, 256, 0, st>>>(amax_q, amax_k, vamax, g4, nb, status);
  if (had) {
    // the rotation needs each row in one lane pair
    quant_4_rows_kernel<true><<<dim3(nb, BH), 256, 0, st>>>(q, nullptr, nullptr, g4, 0, S + L.q4,
                                                            S + L.q4s, kScaleTileBytes, N, Npad,
                                                            nb, status);
    quant_4_rows_kernel<true><<<dim3(nb, BH), 256, 0, st>>>(kk, perm, kbar, g4, 1, S + L.k4,
                                                            S + L.kr4s, 2 * kScaleTileBytes, N,
                                                            Npad, nb, status);
  } else {
    quant_4_rows_kernel<false><<<dim3(nb, BH), 256, 0, st>>>(q, nullptr, nullptr, g4, 0, S + L.q4,
                                                             S + L.q4s, kScaleTileBytes, N, Npad,
                                                             nb, status);
    quant_4_rows_kernel<false><<<dim3(nb, BH), 256, 0, st>>>(kk, perm, kbar, g4, 1, S + L.k4,
                                                             S + L.kr4s, 2 * kScaleTileBytes, N,
                                                             Npad, nb, status);
  }
  const int ngroups = (nb + kGroup4 - 1) / kGroup4;
  zero_kernel<<<grid_chunks((size_t)BH * ngroups * kGroup4Bytes / 4, 256, 4096), 256, 0, st>>>(
      reinterpret_cast<uint32_t*>(mside), (size_t)BH * ngroups * kGroup4Bytes / 4);
  vpass2_4_kernel<<<dim3(nb, BH), 256, 0, st>>>(v, perm, mu, g4, S + L.r4T, S + L.kr4s, mside, N,
                                                Npad, nb, ngroups, ngroups * kGroup4 - nb, status);
  header_done_kernel<<<1, 32, 0, st>>>(hdr, status, a.reuse == 0 || a.reuse == 2);
  return cudaGetLastError() == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}

}  // namespace vca

// ---------------------------------------------------------------------------
// Grouping without caller-provided scratch
// ---------------------------------------------------------------------------
namespace vca {
namespace {

// Scratch of vca_kmeans_permutation_noalloc: a fixed array in this library's
// device image, present on every GPU that loads the library until the process
// exits.  Layout (bytes): [0,256) status word, [256,512) |V| maximum and grid
// scale, then the int8 features [kNoAllocMaxTokens x 128], the int8 centroids
// [256 x 128], the int32 cluster sums [256 x 128] and counts [256], and the
// sort histogram [256 x kNoAllocMaxTokens / kSortChunk].
constexpr size_t kNaOffStatus = 0, kNaOffAmax = 256, kNaOffX = 512;
constexpr size_t kNaOffCent = kNaOffX + (size_t)VCA_NOALLOC_MAX_TOKENS * 128;
constexpr size_t kNaOffSums = kNaOffCent + 256 * 128;
constexpr size_t kNaOffHist = kNaOffSums + (256 * 128 + 256) * 4;
constexpr size_t kNaBytes = kNaOffHist + 256 * (VCA_NOALLOC_MAX_TOKENS / kSortChunk) * 4;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNaBytes];

// Device address of the scratch array on each device (the host-side symbol is
// only a stand-in, not a device address).  Filled by the first call on a device.
constexpr int kMaxDevices = 64;
uint8_t* g_noalloc_ptr[kMaxDevices] = {};

}  // namespace

int* noalloc_status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return g_noalloc_ptr[dev] ? reinterpret_cast<int*>(g_noalloc_ptr[dev] + kNaOffStatus) : nullptr;
}

}  // namespace vca

extern "C" int vca_kmeans_permutation_noalloc(const void* v, int N, int d, int k_clusters,
                                              int iters, uint64_t seed, int b, int h, int H,
                                              int32_t* labels, int32_t* perm,
                                              vca_stream_t stream) {
  using namespace vca;
  if (!v || !labels || !perm) return VCA_ERR_INVALID_ARG;
  if (((uintptr_t)v & 15u) || ((uintptr_t)labels & 3u) || ((uintptr_t)perm & 3u))
    return VCA_ERR_INVALID_ARG;
  if (d != 128 || N < 1 || N > VCA_NOALLOC_MAX_TOKENS) return VCA_ERR_UNSUPPORTED;
  if (k_clusters < 1 || k_clusters > 256 || k_clusters > N) return VCA_ERR_UNSUPPORTED;
  if (iters < 1 || iters > 1000 || b < 0 || h < 0 || H < 1 || h >= H) return VCA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VCA_ERR_CUDA;
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return VCA_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
  }
  uint8_t* S = g_noalloc_ptr[dev];
  const cudaStream_t st = (cudaStream_t)stream;
  const int k = k_clusters;
  const size_t per_head = (size_t)N * 128;
  int* status = reinterpret_cast<int*>(S + kNaOffStatus);
  uint32_t* amax_bits = reinterpret_cast<uint32_t*>(S + kNaOffAmax);
  float* gscale = reinterpret_cast<float*>(S + kNaOffAmax + 4);
  int8_t* x = reinterpret_cast<int8_t*>(S + kNaOffX);
  int8_t* cent = reinterpret_cast<int8_t*>(S + kNaOffCent);
  int32_t* sums = reinterpret_cast<int32_t*>(S + kNaOffSums);
  int32_t* counts = sums + (size_t)k * 128;
  int32_t* hist = reinterpret_cast<int32_t*>(S + kNaOffHist);
  const uint16_t* vv = static_cast<const uint16_t*>(v);
  // The initial centroids of head (b, h) come from SplitMix64 seeded with
  // seed ^ (0x9E3779B97F4A7C15 * (b*H + h + 1)); the init kernel mixes in its
  // block index (0 here) the same way, so the seed is pre-mixed to match.
  const uint64_t G = 0x9E3779B97F4A7C15ull;
  const uint64_t seed_mixed = seed ^ (G * (uint64_t)((int64_t)b * H + h + 1)) ^ G;

  // the leftover contents of the previous call are cleared where needed:
  // status and maximum here, centroid sums and counts by the init kernel
  zero_kernel<<<1, 32, 0, st>>>(reinterpret_cast<uint32_t*>(S), 2 * 256 / 4);
  const int ch = grid_chunks(per_head / 8, 256 * 8, 1024);
  head_amax_kernel<<<dim3(ch, 1), 256, 0, st>>>(vv, amax_bits, per_head, status);
  features_kernel<false><<<dim3(ch, 1), 256, 0, st>>>(vv, amax_bits, gscale, x, per_head, status);
  kmeans_init_kernel<false><<<1, 128, 0, st>>>(x, cent, sums, counts, seed_mixed, N, k, 128, status);
  const int groups = k <= 96 ? 2 : 1;
  const size_t asmem = assign_smem_bytes(k, groups);
  if (cudaFuncSetAttribute(kmeans_assign_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)asmem) != cudaSuccess)
    return VCA_ERR_CUDA;
  const int tiles = (N + kAssignTokens - 1) / kAssignTokens;
  for (int it = 0; it < iters; ++it) {
    kmeans_assign_kernel<<<dim3(tiles, 1), 256, asmem, st>>>(x, cent, labels, sums, counts, N, k,
                                                             groups, status);
    kmeans_update_kernel<<<dim3(1, k), 128, 0, st>>>(cent, sums, counts, k, status);
  }
  const int nchunk = (N + kSortChunk - 1) / kSortChunk;
  sort_hist_kernel<<<dim3(nchunk, 1), 256, 0, st>>>(labels, hist, N, k, nchunk, status);
  sort_scan_kernel<<<1, 256, 0, st>>>(hist, k, nchunk, status);
  sort_scatter_kernel<<<dim3(nchunk, 1), 256, 0, st>>>(labels, hist, perm, N, k, nchunk, status);
  return cudaGetLastError() == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}

