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
// One CTA owns one 128-row query tile of one (batch, head) and streams the key
// blocks through a TMA ring.  Warp roles as in the 8-bit kernel:
//   warp 0        producer: Q tile and its scales once; per stage K'_j, R^T_j
//                 and their two scale tiles; the mean operand of each group
//                 of 4 blocks (ring of 4)
//   warp 1        MMA issuer (warp-uniform, elected lane) and TMEM owner; it
//                 also copies every scale tile into tensor memory
//                 (tcgen05.cp), in order with the products that read it
//   warps 4-11    softmax + correction + epilogue: two threads per query row
//                 (keys / output channels 0-63 and 64-127)
//
// Tensor memory (480 of 512 columns):
//   [0,128), [128,256)  S_j = Q K'_j^T (raw, without gq gk) in buffer j % 2
//   [256,384)  the output accumulator A
//   [384,392)  Q scale factors (two K steps x 4 columns)
//   [392,400)  P scale factors
//   [400,408)  a group's row-sum operand (bf16 hi, lo) of the mean product
//   [416,480)  K' and R scale factors of block j in slot j % 4 (16 columns)
//
// Per key block j (log2 domain, a = gq gk log2(e) / sqrt(d)):
//   M'  = max(M, a rowmax(S))
//   p'  = 2^(a S - M' + log2 2688)          so that p' <= 2688
//   r   = sum p'   (fp32, from the unquantised probabilities: Eq 6's r)
//   P   = NVFP4(p'): scale UE4M3(max16 / 6), elements E2M1(p' / scale)
//   A  *= alpha = 2^(M - M'), l = alpha l + r
//   A  += P R_j          (block-scaled FP4 MMA; R = R-codes x scales, no gr)
//   A  += (r / gr) mu_j  (one BF16 K=16 MMA per group of 4 blocks; each of
//                         the two threads of a row contributes its own partial
//                         sums as separate K entries, hi/lo split)
// Epilogue: O = gr A / l (l in the same 2688-scaled units), bf16.
#include "common.cuh"
#include "prep.h"

namespace vca {
namespace {

constexpr int kStages = 8;
constexpr int kMeanBufs = 4;
constexpr uint32_t kStageBytes = 2 * kTile4Bytes + 2 * kScaleTileBytes;  // K', R^T, scales
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_QS = OFF_Q + kTile4Bytes;
constexpr uint32_t OFF_KV = OFF_QS + kScaleTileBytes;
constexpr uint32_t OFF_P = OFF_KV + kStages * kStageBytes;
constexpr uint32_t OFF_PS = OFF_P + kTile4Bytes;
constexpr uint32_t OFF_BG = OFF_PS + kScaleTileBytes;
constexpr uint32_t OFF_XCH = OFF_BG + kMeanBufs * kGroup4Bytes;  // partial row max, 2 x 2 x 128
constexpr uint32_t OFF_L = OFF_XCH + 2048;                       // partial row sums, 2 x 128
constexpr uint32_t OFF_BAR = OFF_L + 1024;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;  // + alignment slack
constexpr int kThreads = 384;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(OFF_KV % 1024 == 0 && kStageBytes % 1024 == 0 && OFF_P % 1024 == 0,
              "swizzled tiles stay 1024-byte aligned");
static_assert(kGroup4 == 4, "four row-sum slots per thread");

constexpr uint32_t TC_S = 0, TC_ACC = 256, TC_QS = 384, TC_PS = 392, TC_G = 400, TC_KRS = 416;

struct Nvfp4Params {
  const uint8_t* q4s;     // [BH][nb][1024]
  const uint8_t* kr4s;    // [BH][nb][2048]
  const float* g4;        // [BH][4]
  const uint8_t* mside;   // [BH][ngroups][4096]
  const uint32_t* hdr;
  uint16_t* out;          // [BH][N][128]
  int* status;
  int B, H, N, nb, Npad, ngroups, gpad;
  float log2e_rsqrt_d;    // log2(e) / sqrt(128)
};

enum { B_QFULL = 0, B_KVFULL = 1, B_KVEMPTY = B_KVFULL + kStages, B_SFULL = B_KVEMPTY + kStages,
       B_SFREE = B_SFULL + 2, B_PFULL = B_SFREE + 2, B_PVDONE = B_PFULL + 1,
       B_DRAIN = B_PVDONE + 1, B_XCH = B_DRAIN + 1, B_COUNT = B_XCH + 4 };

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
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
  const int bh = blockIdx.x / nb, qt = blockIdx.x % nb;

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
    // "S read" and "P written": all 256 softmax threads; the row-pair
    // exchange of each lane quarter: its two warps; the rest: one arrival
    // or a tcgen05 commit
    for (int i = 0; i < B_COUNT; ++i)
      mbar_init(bar(i), (i >= B_SFREE && i < B_PVDONE) ? 256 : (i >= B_XCH ? 64 : 1));
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    if (lane == 0) {
      mbar_expect_tx(bar(B_QFULL), kTile4Bytes + kScaleTileBytes);
      tma_load_2d(base + OFF_Q, &tmQ, bar(B_QFULL), 0, bh * p.Npad + qt * 128);
      bulk_load(base + OFF_QS, p.q4s + ((size_t)bh * nb + qt) * kScaleTileBytes, kScaleTileBytes,
                bar(B_QFULL));
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
    // ------------------------------------------------------------ MMA issuer
    const uint32_t i4 = idesc_nvf4(128, 128), i16 = idesc_bf16(128, 128);
    const uint64_t dq = desc_k_sw64(base + OFF_Q);
    const uint64_t dp = desc_k_sw64(base + OFF_P);
    const uint64_t dk0 = desc_k_sw64(base + OFF_KV);
    const uint64_t dr0 = desc_k_sw64(base + OFF_KV + kTile4Bytes);
    const uint64_t dstage = kStageBytes >> 4;
    // scale tiles: 32 rows x 16 bytes per K step, no swizzle
    const uint64_t dqs = desc_k_plain(base + OFF_QS, 512, 128);
    const uint64_t dps = desc_k_plain(base + OFF_PS, 512, 128);
    const uint64_t dks0 = desc_k_plain(base + OFF_KV + 2 * kTile4Bytes, 512, 128);
    const uint64_t dhalf = 512 >> 4, dtile = kScaleTileBytes >> 4;
    const uint64_t dbg0 = desc_k_plain(base + OFF_BG, 128, 256);
    const uint64_t dgroup = kGroup4Bytes >> 4;
    bool ok = mbar_wait_spin(bar(B_QFULL), 0, abort_flag, p.status);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      tmem_cp_32x128b_x4_w(tmem + TC_QS, dqs);
      tmem_cp_32x128b_x4_w(tmem + TC_QS + 4, dqs + dhalf);
    } else {
      ok = false;
    }
    auto issue_s = [&](int j) {
      const int s = j % kStages;
      ok = mbar_wait_spin(bar(B_KVFULL + s), (j / kStages) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; return; }
      tc_fence_after();
      const uint32_t krs = tmem + TC_KRS + 16 * (j % 4);
      const uint64_t ds = dks0 + s * dstage;
      tmem_cp_32x128b_x4_w(krs, ds);                       // K' scales, K step 0
      tmem_cp_32x128b_x4_w(krs + 4, ds + dhalf);           // K' scales, K step 1
      tmem_cp_32x128b_x4_w(krs + 8, ds + dtile);           // R scales, K step 0
      tmem_cp_32x128b_x4_w(krs + 12, ds + dtile + dhalf);  // R scales, K step 1
      const uint64_t dk = dk0 + s * dstage;
      const uint32_t d = tmem + TC_S + 128 * (j & 1);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        mma_nvf4_ss_w(d, dq + 2 * kk, dk + 2 * kk, i4, tmem + TC_QS + 4 * kk, krs + 4 * kk, kk > 0);
      mma_commit_w(bar(B_SFULL + (j & 1)));
    };
    auto issue_flush = [&](int g) {
      mma_f16_ts_w(tmem + TC_ACC, tmem + TC_G, dbg0 + (g % kMeanBufs) * dgroup, i16, 1);
    };
    for (int j = 0; ok && j < min(2, nb); ++j) issue_s(j);
    for (int j = 0; ok && j < nb; ++j) {
      ok = mbar_wait_spin(bar(B_PFULL), j & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      tmem_cp_32x128b_x4_w(tmem + TC_PS, dps);
      tmem_cp_32x128b_x4_w(tmem + TC_PS + 4, dps + dhalf);
      const uint64_t dr = dr0 + (j % kStages) * dstage;
      const uint32_t krs = tmem + TC_KRS + 16 * (j % 4);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        mma_nvf4_ss_w(tmem + TC_ACC, dp + 2 * kk, dr + 2 * kk, i4, tmem + TC_PS + 4 * kk,
                      krs + 8 + 4 * kk, (j > 0 || kk > 0));
      if (j > 0 && group_ends(j - 1, nb, gpad)) issue_flush((j - 1 + gpad) / kGroup4);
      mma_commit_w(bar(B_PVDONE));
      mma_commit_w(bar(B_KVEMPTY + j % kStages));
      if (j + 2 < nb) {
        ok = mbar_wait_spin(bar(B_SFREE + (j & 1)), (j >> 1) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        issue_s(j + 2);
      }
    }
    if (ok) {
      ok = mbar_wait_spin(bar(B_PFULL), nb & 1, abort_flag, p.status);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        issue_flush((nb - 1 + gpad) / kGroup4);
        mma_commit_w(bar(B_PVDONE));
      }
    }
    mma_commit_w(bar(B_DRAIN));
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar(B_DRAIN), 0) && globaltimer() - t0 < kWaitLimitNs) {
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int h = (warp - 4) / 4, quarter = warp % 4;
    const int row = quarter * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    // The two threads of a row exchange partial results through shared memory
    // and the quarter's mbarrier (bounded waits, so a stalled partner cannot
    // hang the CTA); phase j is block j, phase nb the final normaliser.
    const uint32_t xbar = bar(B_XCH + quarter);
    const float gq = p.g4[(size_t)bh * 4], gk = p.g4[(size_t)bh * 4 + 1];
    const float gr = p.g4[(size_t)bh * 4 + 2];
    const float a = gq * gk * p.log2e_rsqrt_d;
    const float inv_gr = 1.0f / gr;
    const float kLog2P = 11.392317f;          // log2(2688)
    const int valid_last = p.N - (nb - 1) * 128 - 64 * h;
    float* xch_base = reinterpret_cast<float*>(sm + OFF_XCH);
    uint8_t* ptile = sm + OFF_P;
    uint32_t* pscale = reinterpret_cast<uint32_t*>(sm + OFF_PS + h * 512 + (row % 32) * 16 +
                                                   (row / 32) * 4);
    float M = -INFINITY, l = 0.0f;
    float pend[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    bool ok = true;
    // the row-sum operand of a group: column 4h + u = bf16 (hi, lo) of this
    // thread's rescaled partial sum of slot u, divided by gr
    auto write_group = [&]() {
      uint32_t w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float x = pend[u] * inv_gr;
        const uint16_t hi = f32_to_bf16_bits(x);
        const uint16_t lo = f32_to_bf16_bits(x - bf16_bits_to_f32(hi));
        w[u] = (uint32_t)hi | ((uint32_t)lo << 16);
        pend[u] = 0.0f;
      }
      tmem_st4(tl + TC_G + 4 * h, w);
    };
    for (int j = 0; j < nb; ++j) {
      const uint32_t sbuf = tl + TC_S + 128 * (j & 1);
      ok = mbar_wait(bar(B_SFULL + (j & 1)), (j >> 1) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t s[64];
      tmem_ld32(sbuf + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_ld32(sbuf + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bar(B_SFREE + (j & 1)));
      if (j == nb - 1 && valid_last < 64) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= valid_last) s[c] = 0xFF800000u;  // -inf: masked key -> probability 0
      }
      float mx16[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float m = __uint_as_float(s[16 * i]);
#pragma unroll
        for (int c = 1; c < 16; ++c) m = fmaxf(m, __uint_as_float(s[16 * i + c]));
        mx16[i] = m;
      }
      float* xch = xch_base + (j & 1) * 256;
      xch[h * 128 + row] = fmaxf(fmaxf(mx16[0], mx16[1]), fmaxf(mx16[2], mx16[3]));
      mbar_arrive(xbar);
      ok = mbar_wait_spin(xbar, j & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      const float mx = fmaxf(xch[row], xch[128 + row]);
      const float Mn = fmaxf(M, a * mx);
      const float alpha = ex2(M - Mn);   // 0 on the first block
      const float nbias = kLog2P - Mn;
      // p' = 2688 * 2^(a s - M'), its sum, and the NVFP4 codes of each 16
      float rs = 0.0f;
      uint32_t pw[8];
      uint32_t sc4 = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float amax = ex2(fmaf(mx16[i], a, nbias));
        const uint32_t sc = f32_to_e4m3(amax * (1.0f / 6.0f));
        const float scv = e4m3_to_f32((uint8_t)sc);
        const float inv = scv > 0.0f ? 1.0f / scv : 0.0f;
        sc4 |= sc << (8 * i);
        uint32_t w0 = 0, w1 = 0;
#pragma unroll
        for (int c = 0; c < 16; c += 2) {
          const float p0 = ex2(fmaf(__uint_as_float(s[16 * i + c]), a, nbias));
          const float p1 = ex2(fmaf(__uint_as_float(s[16 * i + c + 1]), a, nbias));
          rs += p0 + p1;
          const uint32_t byte = f32x2_to_e2m1x2(p0 * inv, p1 * inv);
          if (c < 8) w0 |= byte << (4 * c);
          else w1 |= byte << (4 * (c - 8));
        }
        pw[2 * i] = w0;
        pw[2 * i + 1] = w1;
      }
      if (j > 0) {
        ok = mbar_wait(bar(B_PVDONE), (j - 1) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      // P codes (64-byte swizzled K-major, this half = 16-byte chunks 2h, 2h+1)
      // and the four P scales of this half
      *reinterpret_cast<uint4*>(ptile + off_sw64(row, 2 * h)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      *reinterpret_cast<uint4*>(ptile + off_sw64(row, 2 * h + 1)) =
          make_uint4(pw[4], pw[5], pw[6], pw[7]);
      *pscale = sc4;
      fence_proxy_async_smem();
      if (j > 0) {
        if (__any_sync(0xffffffffu, alpha < 1.0f)) {
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tl + TC_ACC + 64 * h + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
            tmem_st32(tl + TC_ACC + 64 * h + c0, v);
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
      mbar_arrive(bar(B_PFULL));
    }
    if (ok) {
      ok = mbar_wait(bar(B_PVDONE), (nb - 1) & 1, abort_flag, p.status);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        write_group();
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(B_PFULL));
        ok = mbar_wait(bar(B_PVDONE), nb & 1, abort_flag, p.status);
      } else {
        ok = false;
      }
    }
    // the row's normaliser: this half's sum plus the partner's
    float* lx = reinterpret_cast<float*>(sm + OFF_L);
    float ltot = 0.0f;
    if (__all_sync(0xffffffffu, ok)) {
      lx[h * 128 + row] = l;
      mbar_arrive(xbar);
      ok = mbar_wait_spin(xbar, nb & 1, abort_flag, p.status);
      ltot = lx[row] + lx[128 + row];
    }
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int grow = qt * 128 + row;
      const float f = gr / ltot;
      uint16_t* orow = p.out + ((size_t)bh * p.N + grow) * 128 + 64 * h;
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tl + TC_ACC + 64 * h + c0, v);
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
  p.log2e_rsqrt_d = (float)(1.4426950408889634 / sqrt(128.0));
  if (cudaFuncSetAttribute(attn_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes) != cudaSuccess)
    return VCA_ERR_CUDA;
  const long long grid = (long long)BH * nb;
  if (grid > 0x7FFFFFFF) return VCA_ERR_UNSUPPORTED;
  attn_nvfp4_kernel<<<(unsigned)grid, kThreads, kSmemBytes, st>>>(tq, tk, tr, p);
  return cudaGetLastError() == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}

}  // namespace vca
