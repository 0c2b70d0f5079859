// 4-bit (NVFP4) VC-Attention forward on tcgen05 block-scaled tensor cores
// (paper §3.1 Eq 1, §3.2 Eq 6, Appx A "Scope of ExpCast-FP8", Appx B).
//
// Q, the permuted centred keys K' and the transposed residual R^T are E2M1
// codes with one UE4M3 scale per 16 elements along the product's reduction
// dimension and one fp32 global scale per head (gq, gk, gr).  ExpCast does not
// apply at 4 bits (no affine log-to-code map exists for E2M1 under a
// microscale), so the softmax evaluates the exponential, and P is quantised to
// NVFP4 after scaling the row so that its maximum is 448 * 6 = 2688.
//
// One CTA owns two 128-row query tiles (A and B) of one (batch, head) and
// streams the key blocks through a TMA ring; both tiles consume each stage.
// Warp roles (12 warps):
//   warp 0      producer: the two Q tiles and their scales once; per stage K'_j,
//               R^T_j and their two scale tiles; the mean operand of each
//               group of 4 blocks (ring of 4)
//   warp 1      S issuer and TMEM owner: copies the Q scales once and the K'
//               scales of each block into tensor memory (tcgen05.cp), then
//               issues S_A(j), S_B(j), S_A(j+1), ... each after the other tile
//               loaded the shared S buffer; it polls its barriers (a
//               non-blocking test every ~128 ns), which holds back the softmax
//               warps of its sub-partition less than a suspended wait
//   warp 2      PV issuer: copies the R and P scales, issues PV_A(j), PV_B(j)
//               and the mean products, and releases the stages
//   warps 4-7   softmax + correction + epilogue of tile A, warps 8-11 of tile
//               B, one thread per query row (the row's 128 scores in registers)
// Every scale copy is issued by the warp whose products read it, so the copy
// and the products execute in issue order.
//
// Tensor memory (480 of 512 columns):
//   [0,128)     S = Q K'^T (raw, without gq gk), shared by the two tiles
//   [128,384)   the output accumulators A_A, A_B
//   [384,400)   Q scale factors of A, B (two K steps x 4 columns each)
//   [400,416)   P scale factors of A, B
//   [416,432)   a group's row-sum operand (bf16 hi, lo) of A, B
//   [432,448)   K' scale factors, two slots (blocks j % 2)
//   [448,464)   R scale factors, two slots
//
// Per key block j and tile (log2 domain, a = gq gk log2(e) / sqrt(d)):
//   M'  = max(M, a rowmax(S))
//   p'  = 2^(a S - M' + log2 2688)          so that p' <= 2688
//   r   = sum p'   (from the unquantised probabilities: Eq 6's r; block
//         sums of 16 in f16, accumulated in fp32)
//   P   = NVFP4(p'): scale UE4M3(max16 / 6), elements E2M1(p' / scale), each
//         element evaluated directly as 2^(a S - M' + log2 2688 - log2 scale)
//         (exponent in fp32, exponential in packed f16)
//   A  *= alpha = 2^(M - M'), l = alpha l + r
//   A  += P R_j          (block-scaled FP4 MMA; R = R-codes x scales, no gr)
//   A  += (r / gr) mu_j  (one BF16 K=16 MMA per group of 4 blocks; the bf16 hi
//                         and lo of each block's rescaled row sum meet the
//                         block's mean in K rows 2u, 2u+1)
// Epilogue: O = gr A / l (l in the same 2688-scaled units), bf16.
#include "common.cuh"
#include <cuda_fp16.h>
#include "prep.h"

namespace vca {
namespace {

constexpr int kStages = 8;
constexpr int kMeanBufs = 4;
constexpr uint32_t kStageBytes = 2 * kTile4Bytes + 2 * kScaleTileBytes;  // K', R^T, scales
constexpr uint32_t OFF_Q = 0;                                 // Q_A, Q_B
constexpr uint32_t OFF_QS = OFF_Q + 2 * kTile4Bytes;          // their scale tiles
constexpr uint32_t OFF_KV = OFF_QS + 2 * kScaleTileBytes;
constexpr uint32_t OFF_P = OFF_KV + kStages * kStageBytes;    // P_A, P_B
constexpr uint32_t OFF_PS = OFF_P + 2 * kTile4Bytes;          // their scale tiles
constexpr uint32_t OFF_BG = OFF_PS + 2 * kScaleTileBytes;
constexpr uint32_t OFF_BAR = OFF_BG + kMeanBufs * kGroup4Bytes;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;  // + alignment slack
constexpr int kThreads = 384;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(OFF_KV % 1024 == 0 && kStageBytes % 1024 == 0 && OFF_P % 1024 == 0,
              "swizzled tiles stay 1024-byte aligned");
static_assert(kGroup4 == 4, "four row-sum slots per group");

constexpr uint32_t TC_S = 0, TC_KS = 432, TC_RS = 448;
__device__ __forceinline__ uint32_t tc_acc(int X) { return 128u + 128u * X; }
__device__ __forceinline__ uint32_t tc_qs(int X) { return 384u + 8u * X; }
__device__ __forceinline__ uint32_t tc_ps(int X) { return 400u + 8u * X; }
__device__ __forceinline__ uint32_t tc_g(int X) { return 416u + 8u * X; }

struct Nvfp4Params {
  const uint8_t* q4s;     // [BH][nb][1024]
  const uint8_t* kr4s;    // [BH][nb][2048]
  const float* g4;        // [BH][4]
  const uint8_t* mside;   // [BH][ngroups][4096]
  const uint32_t* hdr;
  uint16_t* out;          // [BH][N][128]
  int* status;
  int B, H, N, nb, Npad, ngroups, gpad, npairs;
  float log2e_rsqrt_d;    // log2(e) / sqrt(128)
};

enum { B_QFULL = 0, B_KVFULL = 1, B_KVEMPTY = B_KVFULL + kStages, B_SFULL = B_KVEMPTY + kStages,
       B_SFREE = B_SFULL + 2, B_PFULL = B_SFREE + 2, B_PVDONE = B_PFULL + 2,
       B_DRAIN = B_PVDONE + 2, B_COUNT = B_DRAIN + 1 };

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ bool group_ends(int j, int nb, int gpad) {
  return j == nb - 1 || (j + gpad) % kGroup4 == kGroup4 - 1;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_nvfp4_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmR, const Nvfp4Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + B_COUNT * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_BAR + B_COUNT * 8 + 4);
  auto bar = [&](int i) { return base + OFF_BAR + 8u * (uint32_t)i; };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nb = p.nb, gpad = p.gpad;
  const int bh = blockIdx.x / p.npairs, qp = blockIdx.x % p.npairs;
  const bool has_b = 2 * qp + 1 < nb;   // the last pair of an odd nb has tile A only

  {
    const volatile uint32_t* h = p.hdr;
    const bool hdr_ok = h[0] == kStateMagic && h[1] == (uint32_t)p.B && h[2] == (uint32_t)p.H &&
                        h[3] == (uint32_t)p.N && h[6] == 4u && h[8] == 1u;
    if (!hdr_ok) {
      if (threadIdx.x == 0) atomicOr(p.status, kStatStateMismatch);
      return;
    }
    if (*(volatile int*)p.status != 0) return;
  }

  if (threadIdx.x == 0) {
    // "S read" and "P written": the 128 softmax threads of a tile; the drain:
    // both issuers; the rest: one arrival or a tcgen05 commit
    for (int i = 0; i < B_COUNT; ++i)
      mbar_init(bar(i), (i >= B_SFREE && i < B_PVDONE) ? 128 : (i == B_DRAIN ? 2 : 1));
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmR);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t i4 = idesc_nvf4(128, 128);
  const uint64_t dstage = kStageBytes >> 4, dhalf = 512 >> 4;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    if (lane == 0) {
      mbar_expect_tx(bar(B_QFULL), (has_b ? 2 : 1) * (kTile4Bytes + kScaleTileBytes));
      for (int X = 0; X < (has_b ? 2 : 1); ++X) {
        tma_load_2d(base + OFF_Q + X * kTile4Bytes, &tmQ, bar(B_QFULL), 0,
                    bh * p.Npad + (2 * qp + X) * 128);
        bulk_load(base + OFF_QS + X * kScaleTileBytes,
                  p.q4s + ((size_t)bh * nb + 2 * qp + X) * kScaleTileBytes, kScaleTileBytes,
                  bar(B_QFULL));
      }
    }
    int issued = 0;
    for (int j = 0; j < nb; ++j) {
      const int s = j % kStages;
      if (j >= kStages)
        ok = mbar_wait(bar(B_KVEMPTY + s), ((j / kStages) - 1) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (lane == 0) {
        const uint32_t st = base + OFF_KV + s * kStageBytes;
        const bool group_start = j == 0 || (j + gpad) % kGroup4 == 0;
        mbar_expect_tx(bar(B_KVFULL + s),
                       2 * kTile4Bytes + 2 * kScaleTileBytes + (group_start ? kGroup4Bytes : 0));
        tma_load_2d(st, &tmK, bar(B_KVFULL + s), 0, bh * p.Npad + j * 128);
        tma_load_2d(st + kTile4Bytes, &tmR, bar(B_KVFULL + s), j * 64, bh * 128);
        bulk_load(st + 2 * kTile4Bytes, p.kr4s + ((size_t)bh * nb + j) * 2 * kScaleTileBytes,
                  2 * kScaleTileBytes, bar(B_KVFULL + s));
        if (group_start) {
          // ring of kMeanBufs: the buffer of group g - kMeanBufs was last read
          // by a mean product issued before the release of stage j - kStages
          const int g = (j + gpad) / kGroup4;
          bulk_load(base + OFF_BG + (g % kMeanBufs) * kGroup4Bytes,
                    p.mside + ((size_t)bh * p.ngroups + g) * kGroup4Bytes, kGroup4Bytes,
                    bar(B_KVFULL + s));
        }
      }
      __syncwarp();
      ++issued;
    }
    if (lane == 0 && *abort_flag) {
      const uint64_t t0 = globaltimer();
      for (int j = max(0, issued - kStages); j < issued; ++j) {
        const int s = j % kStages;
        while (!mbar_try_wait(bar(B_KVFULL + s), (j / kStages) & 1) &&
               globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    const uint64_t dq0 = desc_k_sw64(base + OFF_Q), dqstep = kTile4Bytes >> 4;
    const uint64_t dk0 = desc_k_sw64(base + OFF_KV);
    const uint64_t dqs0 = desc_k_plain(base + OFF_QS, 512, 128);
    const uint64_t dks0 = desc_k_plain(base + OFF_KV + 2 * kTile4Bytes, 512, 128);
    const uint64_t dtile = kScaleTileBytes >> 4;
    bool ok = mbar_wait(bar(B_QFULL), 0, abort_flag, p.status);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      for (int X = 0; X < (has_b ? 2 : 1); ++X) {
        tmem_cp_32x128b_x4_w(tmem + tc_qs(X), dqs0 + X * dtile);
        tmem_cp_32x128b_x4_w(tmem + tc_qs(X) + 4, dqs0 + X * dtile + dhalf);
      }
    } else {
      ok = false;
    }
    // S_X(j); tile A's product also copies the block's K' scales (slot j % 2)
    auto issue_s = [&](int X, int j, bool kv_ready) {
      const int s = j % kStages;
      if (X == 0) {
        if (!kv_ready) {
          ok = mbar_wait(bar(B_KVFULL + s), (j / kStages) & 1, abort_flag, p.status);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; return; }
        }
        tc_fence_after();
        tmem_cp_32x128b_x4_w(tmem + TC_KS + 8 * (j & 1), dks0 + s * dstage);
        tmem_cp_32x128b_x4_w(tmem + TC_KS + 8 * (j & 1) + 4, dks0 + s * dstage + dhalf);
      } else {
        tc_fence_after();
      }
      const uint64_t dk = dk0 + s * dstage, dq = dq0 + X * dqstep;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        mma_nvf4_ss_w(tmem + TC_S, dq + 2 * kk, dk + 2 * kk, i4, tmem + tc_qs(X) + 4 * kk,
                      tmem + TC_KS + 8 * (j & 1) + 4 * kk, kk > 0);
      mma_commit_w(bar(B_SFULL + X));
    };
    auto wait_sfree = [&](int X, int j) {
      ok = mbar_wait_poll(bar(B_SFREE + X), j & 1, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
    };
    if (ok) issue_s(0, 0, false);
    if (ok && has_b) {
      wait_sfree(0, 0);
      if (ok) issue_s(1, 0, true);
    }
    for (int j = 0; ok && j + 1 < nb; ++j) {
      // the stage of block j+1 first (usually landed long before), so the wait
      // for the other tile is the last step before the product
      ok = mbar_wait_poll(bar(B_KVFULL + (j + 1) % kStages), ((j + 1) / kStages) & 1, abort_flag,
                          p.status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      wait_sfree(has_b ? 1 : 0, j);
      if (!ok) break;
      issue_s(0, j + 1, true);
      if (!ok) break;
      if (has_b) {
        wait_sfree(0, j + 1);
        if (!ok) break;
        issue_s(1, j + 1, true);
      }
    }
    mma_commit_w(bar(B_DRAIN));
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar(B_DRAIN), 0) && globaltimer() - t0 < kWaitLimitNs) {
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ PV issuer
    const uint64_t dp0 = desc_k_sw64(base + OFF_P), dpstep = kTile4Bytes >> 4;
    const uint64_t dr0 = desc_k_sw64(base + OFF_KV + kTile4Bytes);
    const uint64_t dps0 = desc_k_plain(base + OFF_PS, 512, 128), dtile = kScaleTileBytes >> 4;
    const uint64_t drs0 = desc_k_plain(base + OFF_KV + 2 * kTile4Bytes + kScaleTileBytes, 512, 128);
    const uint64_t dbg0 = desc_k_plain(base + OFF_BG, 128, 256), dgroup = kGroup4Bytes >> 4;
    const uint32_t i16 = idesc_bf16(128, 128);
    bool ok = true;
    auto issue_pv = [&](int X, int j) {
      ok = mbar_wait(bar(B_PFULL + X), j & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; return; }
      tc_fence_after();
      const int s = j % kStages;
      if (X == 0) {  // the block's R scales (slot j % 2), used by both tiles
        tmem_cp_32x128b_x4_w(tmem + TC_RS + 8 * (j & 1), drs0 + s * dstage);
        tmem_cp_32x128b_x4_w(tmem + TC_RS + 8 * (j & 1) + 4, drs0 + s * dstage + dhalf);
      }
      tmem_cp_32x128b_x4_w(tmem + tc_ps(X), dps0 + X * dtile);
      tmem_cp_32x128b_x4_w(tmem + tc_ps(X) + 4, dps0 + X * dtile + dhalf);
      const uint64_t dr = dr0 + s * dstage, dp = dp0 + X * dpstep;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        mma_nvf4_ss_w(tmem + tc_acc(X), dp + 2 * kk, dr + 2 * kk, i4, tmem + tc_ps(X) + 4 * kk,
                      tmem + TC_RS + 8 * (j & 1) + 4 * kk, (j > 0 || kk > 0));
      if (j > 0 && group_ends(j - 1, nb, gpad))
        mma_f16_ts_w(tmem + tc_acc(X), tmem + tc_g(X),
                     dbg0 + (((j - 1 + gpad) / kGroup4) % kMeanBufs) * dgroup, i16, 1);
      mma_commit_w(bar(B_PVDONE + X));
    };
    for (int j = 0; ok && j < nb; ++j) {
      issue_pv(0, j);
      if (!ok) break;
      if (has_b) issue_pv(1, j);
      if (!ok) break;
      mma_commit_w(bar(B_KVEMPTY + j % kStages));
    }
    // the last group's mean product, after the softmax wrote its row sums
    for (int X = 0; ok && X < (has_b ? 2 : 1); ++X) {
      ok = mbar_wait(bar(B_PFULL + X), nb & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      mma_f16_ts_w(tmem + tc_acc(X), tmem + tc_g(X),
                   dbg0 + (((nb - 1 + gpad) / kGroup4) % kMeanBufs) * dgroup, i16, 1);
      mma_commit_w(bar(B_PVDONE + X));
    }
    mma_commit_w(bar(B_DRAIN));
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar(B_DRAIN), 0) && globaltimer() - t0 < kWaitLimitNs) {
    }
  } else if (warp >= 4 && (warp < 8 || has_b)) {
    // ------------------------------------------------------------ softmax
    const int X = (warp - 4) / 4, quarter = warp % 4;
    const int qt = 2 * qp + X;
    const int row = quarter * 32 + lane;  // row within the query tile = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t acc = tl + tc_acc(X);
    const float gq = p.g4[(size_t)bh * 4], gk = p.g4[(size_t)bh * 4 + 1];
    const float gr = p.g4[(size_t)bh * 4 + 2];
    const float a = gq * gk * p.log2e_rsqrt_d;
    const float inv_gr = 1.0f / gr;
    const float kLog2P = 11.392317f;          // log2(2688)
    const int valid_last = p.N - (nb - 1) * 128;
    uint8_t* ptile = sm + OFF_P + X * kTile4Bytes;
    // this row's scale words: K step 0 (keys 0-63) and, 512 bytes on, step 1
    uint32_t* ps = reinterpret_cast<uint32_t*>(sm + OFF_PS + X * kScaleTileBytes +
                                               (row % 32) * 16 + (row / 32) * 4);
    float M = -INFINITY, l = 0.0f;
    float pend[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    bool ok = true;
    // the row-sum operand of a group: column u = bf16 (hi, lo) of the
    // rescaled row sum of slot u divided by gr; columns 4-7 (K 8..15) zero
    auto write_group = [&]() {
      uint32_t w[8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float x = pend[u] * inv_gr;
        const uint16_t hi = f32_to_bf16_bits(x);
        const uint16_t lo = f32_to_bf16_bits(x - bf16_bits_to_f32(hi));
        w[u] = (uint32_t)hi | ((uint32_t)lo << 16);
        w[4 + u] = 0u;
        pend[u] = 0.0f;
      }
      tmem_st8(tl + tc_g(X), w);
    };
    for (int j = 0; j < nb; ++j) {
      ok = mbar_wait(bar(B_SFULL + X), j & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      // all 128 scores of the row into registers, then release the S buffer
      uint32_t s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_ld32(tl + TC_S + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * c]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bar(B_SFREE + X));
      if (j == nb - 1 && valid_last < 128) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= valid_last) s[c] = 0xFF800000u;  // -inf: masked key -> probability 0
      }
      float mx16[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float m = fmaxf(__uint_as_float(s[16 * i]), __uint_as_float(s[16 * i + 15]));
#pragma unroll
        for (int c = 1; c < 15; c += 2)
          m = max3(m, __uint_as_float(s[16 * i + c]), __uint_as_float(s[16 * i + c + 1]));
        mx16[i] = m;
      }
      const float mx = fmaxf(fmaxf(max3(mx16[0], mx16[1], mx16[2]), max3(mx16[3], mx16[4], mx16[5])),
                             fmaxf(mx16[6], mx16[7]));
      const float Mn = fmaxf(M, a * mx);
      const float alpha = ex2(M - Mn);   // 0 on the first block
      const float nbias = kLog2P - Mn;
      // Per 16 keys: the block scale from the block maximum, then each code
      // straight from q = p' / scale = 2^(a s - M' + log2 2688 - log2 scale):
      // the exponent in fp32, then the exponential, the block sum and the
      // E2M1 cast on packed f16 pairs (f16 carries q <= 6 to 11 bits, far
      // finer than E2M1); the row sum r = sum p' is rebuilt as scale * sum q
      // per block of 16.  A block whose scale rounds to zero
      // holds probabilities below 2688 * 2^-10 / 6 of the maximum: codes 0,
      // and their negligible share of r is dropped.
      float rs = 0.0f;
      uint32_t pw[16];
      uint32_t sc4[2] = {0u, 0u};
      // the eight block scales first (eight independent chains)
      float scvs[8], nbis[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float amax = ex2(fmaf(mx16[i], a, nbias));
        const uint32_t sc = f32_to_e4m3(amax * (1.0f / 6.0f));
        const float scv = e4m3_to_f32((uint8_t)sc);
        float l2s;
        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l2s) : "f"(scv));
        scvs[i] = scv;
        nbis[i] = scv > 0.0f ? nbias - l2s : -INFINITY;
        sc4[i / 4] |= sc << (8 * (i % 4));
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float scv = scvs[i], nbi = nbis[i];
        // pairs of keys: the exponent in fp32 (one paired FMA), then the
        // exponential, the block sum and the E2M1 cast in packed f16
        uint32_t hsum = 0u;   // f16x2 partial sums of q
        uint32_t e[8];
        const uint64_t a2 = ((uint64_t)__float_as_uint(a) << 32) | __float_as_uint(a);
        const uint64_t b2 = ((uint64_t)__float_as_uint(nbi) << 32) | __float_as_uint(nbi);
#pragma unroll
        for (int c = 0; c < 16; c += 2) {
          const uint64_t s2 = ((uint64_t)s[16 * i + c + 1] << 32) | s[16 * i + c];
          uint64_t x2;
          asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(x2) : "l"(s2), "l"(a2), "l"(b2));
          uint32_t hx;
          asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hx) : "f"(__uint_as_float((uint32_t)(x2 >> 32))),
              "f"(__uint_as_float((uint32_t)x2)));
          asm("ex2.approx.f16x2 %0, %1;" : "=r"(e[c / 2]) : "r"(hx));
          asm("add.rn.f16x2 %0, %1, %2;" : "=r"(hsum) : "r"(hsum), "r"(e[c / 2]));
        }
        const float hlo = __half2float(__ushort_as_half((uint16_t)(hsum & 0xFFFFu)));
        const float hhi = __half2float(__ushort_as_half((uint16_t)(hsum >> 16)));
        rs = fmaf(hlo + hhi, scv, rs);
        // the E2M1 casts, four code bytes (eight keys) per word, byte k =
        // keys 2k, 2k+1 of the word
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
          asm("{\n.reg .b8 t0, t1, t2, t3;\n"
              "cvt.rn.satfinite.e2m1x2.f16x2 t0, %1;\ncvt.rn.satfinite.e2m1x2.f16x2 t1, %2;\n"
              "cvt.rn.satfinite.e2m1x2.f16x2 t2, %3;\ncvt.rn.satfinite.e2m1x2.f16x2 t3, %4;\n"
              "mov.b32 %0, {t0, t1, t2, t3};\n}"
              : "=r"(pw[2 * i + h2])
              : "r"(e[4 * h2]), "r"(e[4 * h2 + 1]), "r"(e[4 * h2 + 2]), "r"(e[4 * h2 + 3]));
      }
      if (j > 0) {
        ok = mbar_wait(bar(B_PVDONE + X), (j - 1) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      // P codes (64-byte swizzled K-major: 16-byte chunk c = keys 32c..32c+31)
      // and the row's eight P scales
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(ptile + off_sw64(row, c)) =
            make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
      ps[0] = sc4[0];
      ps[128] = sc4[1];
      fence_proxy_async_smem();
      if (j > 0) {
        if (__any_sync(0xffffffffu, alpha < 1.0f)) {
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(acc + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
            tmem_st32(acc + c0, v);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) pend[u] *= alpha;
        if (group_ends(j - 1, nb, gpad)) write_group();
      }
      l = l * alpha + rs;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (u == (j + gpad) % kGroup4) pend[u] = rs;
      M = Mn;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + X));
    }
    if (ok) {
      ok = mbar_wait(bar(B_PVDONE + X), (nb - 1) & 1, abort_flag, p.status);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        write_group();
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(B_PFULL + X));
        ok = mbar_wait(bar(B_PVDONE + X), nb & 1, abort_flag, p.status);
      } else {
        ok = false;
      }
    }
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int grow = qt * 128 + row;
      const float f = gr / l;
      uint16_t* orow = p.out + ((size_t)bh * p.N + grow) * 128;
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(acc + c0, v);
        tmem_ld_wait();
        if (grow < p.N) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint32_t pk[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float o0 = __uint_as_float(v[c + 2 * u]) * f;
              const float o1 = __uint_as_float(v[c + 2 * u + 1]) * f;
              pk[u] = (uint32_t)f32_to_bf16_bits(o0) | ((uint32_t)f32_to_bf16_bits(o1) << 16);
            }
            *reinterpret_cast<uint4*>(orow + c0 + c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int launch_attention_nvfp4(uint8_t* S, const vca_state_layout& L, int B, int H, int N, void* o,
                           cudaStream_t st) {
  const int BH = B * H, nb = (N + 127) / 128, Npad = nb * 128;
  CUtensorMap tq, tk, tr;
  if (!make_tmap_2d(&tq, S + L.q4, 1, 64, (uint64_t)BH * Npad, 64, 64, 128, 64) ||
      !make_tmap_2d(&tk, S + L.k4, 1, 64, (uint64_t)BH * Npad, 64, 64, 128, 64) ||
      !make_tmap_2d(&tr, S + L.r4T, 1, Npad / 2, (uint64_t)BH * 128, Npad / 2, 64, 128, 64))
    return VCA_ERR_CUDA;
  Nvfp4Params p;
  p.q4s = S + L.q4s;
  p.kr4s = S + L.kr4s;
  p.g4 = reinterpret_cast<const float*>(S + L.g4);
  p.mside = S + L.mside;
  p.hdr = reinterpret_cast<const uint32_t*>(S + L.header);
  p.out = reinterpret_cast<uint16_t*>(o);
  p.status = reinterpret_cast<int*>(S + L.status);
  p.B = B; p.H = H; p.N = N; p.nb = nb; p.Npad = Npad;
  p.ngroups = (nb + kGroup4 - 1) / kGroup4;
  p.gpad = p.ngroups * kGroup4 - nb;
  p.npairs = (nb + 1) / 2;
  p.log2e_rsqrt_d = (float)(1.4426950408889634 / sqrt(128.0));
  if (cudaFuncSetAttribute(attn_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes) != cudaSuccess)
    return VCA_ERR_CUDA;
  const long long grid = (long long)BH * p.npairs;
  if (grid > 0x7FFFFFFF) return VCA_ERR_UNSUPPORTED;
  attn_nvfp4_kernel<<<(unsigned)grid, kThreads, kSmemBytes, st>>>(tq, tk, tr, p);
  return cudaGetLastError() == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}

}  // namespace vca
