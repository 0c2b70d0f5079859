// 8-bit VC-Attention forward (paper §3.1 Eq 1, §3.2 Eq 6, §3.3 Eq 7) on
// tcgen05 tensor cores.
//
// One CTA owns two 128-row query tiles of one (batch, head) and streams all
// key blocks j of the permuted, centred keys K' and the transposed residual
// R^T through a 3-stage TMA ring.  Warp roles:
//   warp 0        TMA producer (Q tiles once; K'_j, R^T_j and the per-block
//                 mean operand per stage)
//   warp 1        MMA issuer (one thread) and TMEM owner
//   warps 4-7     softmax + correction + epilogue of query tile 0
//   warps 8-11    the same for query tile 1
// Tensor memory (512 columns): tile t uses columns [256t, 256t+128) for
// S = Q^ K'^T (fp32) and [256t+128, 256t+256) for the output accumulator A.
//
// Per key block j and query tile t:
//   S   = Q^_t K'^_j^T                          FP8 MMA, 4 x K=32
//   M'  = max(M, a_j rowmax(S))                 exact running max (x8, log2)
//   c   = clip_[0,120](RNE(a_j S + 119.65 - M'))  ExpCast-FP8 bytes -> P^ (smem)
//   r   = sum of the E4M3 values of the bytes   (exactly what the MMA consumes)
//   A  *= alpha = 2^((M - M')/8) when M rises    (TMEM correction)
//   A  += P^ R^_j + r mutilde_j^T                FP8 MMA + one BF16 K=16 MMA
//   l   = alpha l + r
// Epilogue: O = sV (.) A / l in bf16, original query order (Q is not permuted).
#include "common.cuh"
#include "expcast.cuh"
#include "prep.h"

namespace vca {
namespace {

constexpr int kStages = 3;
constexpr uint32_t kStageBytes = 2 * kTileBytes + kSideTileBytes;  // K', R^T, mean operand
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_P = 2 * kTileBytes;
constexpr uint32_t OFF_KV = 4 * kTileBytes;
constexpr uint32_t OFF_AS = OFF_KV + kStages * kStageBytes;  // r operand, 2 x 4 KB
constexpr uint32_t OFF_SV = OFF_AS + 2 * kSideTileBytes;     // sV, 512 B
constexpr uint32_t OFF_BAR = OFF_SV + 512;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;  // + alignment slack

struct Fp8Params {
  const float* sq;        // [BH][nb]
  const float* sk;        // [BH][nb]
  const float* sv;        // [BH][128]
  const uint8_t* mside;   // [BH][nb][4096]
  const uint32_t* hdr;
  uint16_t* out;          // [BH][N][128]
  int* status;
  int B, H, N, nb, Npad, npairs;
  float qk_scale;         // 8 log2(e) / sqrt(128)
};

// barrier indices
enum { B_QFULL = 0, B_KVFULL = 1, B_KVEMPTY = B_KVFULL + kStages, B_SFULL = B_KVEMPTY + kStages,
       B_SFREE = B_SFULL + 2, B_PFULL = B_SFREE + 2, B_PVDONE = B_PFULL + 2, B_DRAIN = B_PVDONE + 2,
       B_COUNT = B_DRAIN + 1 };

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(384, 1)
    attn_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmR, const Fp8Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + B_COUNT * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_BAR + B_COUNT * 8 + 4);
  float* s_sv = reinterpret_cast<float*>(sm + OFF_SV);
  auto bar = [&](int i) { return base + OFF_BAR + 8u * (uint32_t)i; };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bh = blockIdx.x / p.npairs, pair = blockIdx.x % p.npairs;
  const int qt0 = 2 * pair;
  const int ntiles = min(2, p.nb - qt0);

  // Skip the launch if the blob is in an error state or not an 8-bit
  // preparation of this shape (uniform over the CTA).
  {
    const volatile uint32_t* h = p.hdr;
    const bool hdr_ok = h[0] == kStateMagic && h[1] == (uint32_t)p.B && h[2] == (uint32_t)p.H &&
                        h[3] == (uint32_t)p.N && h[6] == 8u && h[8] == 1u;
    if (!hdr_ok) {
      if (threadIdx.x == 0) atomicOr(p.status, kStatStateMismatch);
      return;
    }
    if (*(volatile int*)p.status != 0) return;
  }

  if (threadIdx.x == 0) {
    // producer/MMA barriers complete on one arrival (or a tcgen05 commit);
    // "S read" and "P written" complete when all 128 softmax threads arrive
    for (int i = 0; i < B_COUNT; ++i)
      mbar_init(bar(i), (i >= B_SFREE && i < B_PVDONE) ? 128 : 1);
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
  if (threadIdx.x >= 128 && threadIdx.x < 256) s_sv[threadIdx.x - 128] = p.sv[(size_t)bh * 128 + threadIdx.x - 128];
  // the constant (zero) K columns 8..15 of the r operand
  for (int i = threadIdx.x; i < 2 * (int)kSideTileBytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm + OFF_AS)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int qrow = bh * p.Npad + qt0 * 128;
      mbar_expect_tx(bar(B_QFULL), ntiles * kTileBytes);
      for (int t = 0; t < ntiles; ++t)
        tma_load_2d(base + OFF_Q + t * kTileBytes, &tmQ, bar(B_QFULL), 0, qrow + t * 128);
      int issued = 0;
      for (int j = 0; j < p.nb; ++j) {
        const int s = j % kStages;
        if (j >= kStages &&
            !mbar_wait(bar(B_KVEMPTY + s), ((j / kStages) - 1) & 1, abort_flag, p.status))
          break;
        const uint32_t st = base + OFF_KV + s * kStageBytes;
        mbar_expect_tx(bar(B_KVFULL + s), kStageBytes);
        tma_load_2d(st, &tmK, bar(B_KVFULL + s), 0, bh * p.Npad + j * 128);
        tma_load_2d(st + kTileBytes, &tmR, bar(B_KVFULL + s), j * 128, bh * 128);
        bulk_load(st + 2 * kTileBytes, p.mside + ((size_t)bh * p.nb + j) * kSideTileBytes,
                  kSideTileBytes, bar(B_KVFULL + s));
        ++issued;
      }
      if (*abort_flag) {
        // let the copies in flight land before the CTA exits
        const uint64_t t0 = globaltimer();
        for (int j = max(0, issued - kStages); j < issued; ++j) {
          const int s = j % kStages;
          while (!mbar_try_wait(bar(B_KVFULL + s), (j / kStages) & 1) &&
                 globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t i8 = idesc_f8(128, 128), i16 = idesc_bf16(128, 128);
      bool ok = mbar_wait(bar(B_QFULL), 0, abort_flag, p.status);
      for (int j = 0; ok && j <= p.nb; ++j) {
        if (j < p.nb) {
          const int s = j % kStages;
          if (!(ok = mbar_wait(bar(B_KVFULL + s), (j / kStages) & 1, abort_flag, p.status))) break;
          const uint32_t kt = base + OFF_KV + s * kStageBytes;
          for (int t = 0; t < ntiles; ++t) {
            if (j > 0 && !(ok = mbar_wait(bar(B_SFREE + t), (j - 1) & 1, abort_flag, p.status)))
              break;
            tc_fence_after();
            const uint32_t qa = base + OFF_Q + t * kTileBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f8_ss(tmem + 256 * t, desc_k_sw128(qa + 32 * kk), desc_k_sw128(kt + 32 * kk), i8,
                        kk > 0);
            mma_commit(bar(B_SFULL + t));
          }
          if (!ok) break;
        }
        if (j > 0) {
          const int jp = j - 1, sp = jp % kStages;
          const uint32_t st = base + OFF_KV + sp * kStageBytes;
          for (int t = 0; t < ntiles; ++t) {
            if (!(ok = mbar_wait(bar(B_PFULL + t), jp & 1, abort_flag, p.status))) break;
            tc_fence_after();
            const uint32_t pa = base + OFF_P + t * kTileBytes;
            const uint32_t acc = tmem + 256 * t + 128;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f8_ss(acc, desc_k_sw128(pa + 32 * kk), desc_k_sw128(st + kTileBytes + 32 * kk),
                        i8, (jp > 0 || kk > 0));
            // + r mutilde_j^T: [r_hi r_lo r_hi 0..] x [mu_hi; mu_hi; mu_lo; 0..]
            mma_f16_ss(acc, desc_k_plain(base + OFF_AS + t * kSideTileBytes, 128, 256),
                       desc_k_plain(st + 2 * kTileBytes, 128, 256), i16, 1);
            mma_commit(bar(B_PVDONE + t));
          }
          if (!ok) break;
          mma_commit(bar(B_KVEMPTY + sp));
        }
      }
      // all issued MMAs complete before the CTA releases its tensor memory
      mma_commit(bar(B_DRAIN));
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar(B_DRAIN), 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  } else if (warp >= 4 && (warp - 4) / 4 < ntiles) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) / 4, quarter = warp % 4;
    const int row = quarter * 32 + lane;  // row within the query tile = TMEM lane
    const uint32_t tS = tmem + ((uint32_t)(quarter * 32) << 16) + 256 * t;
    const uint32_t tA = tS + 128;
    const int qt = qt0 + t;
    const float a_q = p.qk_scale * p.sq[(size_t)bh * p.nb + qt];
    const int last_valid = p.N - (p.nb - 1) * 128;
    uint8_t* prow = sm + OFF_P + t * kTileBytes + row * 128;
    uint8_t* asrow = sm + OFF_AS + t * kSideTileBytes + (row / 8) * 256 + (row % 8) * 16;
    float M = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < p.nb; ++j) {
      ok = mbar_wait(bar(B_SFULL + t), j & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t s[128];
      tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
      tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bar(B_SFREE + t));

      if (j == p.nb - 1 && last_valid < 128) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= last_valid) s[c] = 0xFF800000u;  // -inf: masked key -> byte 0
      }
      const float a = a_q * __ldg(p.sk + (size_t)bh * p.nb + j);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; c += 2) mx = max3(mx, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
      const float Mn = fmaxf(M, a * mx);
      const float alpha = ex2((M - Mn) * 0.125f);  // 0 on the first block
      const float b = kExpCastBias - Mn;
      uint32_t w[32];
      float r;
      if (expcast_fast_is_exact(Mn)) {
        const float a128 = a * 0.0078125f, b128 = b * 0.0078125f;
        uint64_t rs = 0;  // two fp32 partial sums of the decoded bytes (x 2^-120)
#pragma unroll
        for (int c = 0; c < 128; c += 4) {
          const uint2 e0 = expcast_pair_bits(__uint_as_float(s[c]), __uint_as_float(s[c + 1]), a128, b128);
          const uint2 e1 = expcast_pair_bits(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]), a128, b128);
          // the fp32 pattern (code << 20) is the E4M3 value of the code x 2^-120,
          // subnormal codes included; (bits << 20) keeps exactly the code bits
          uint64_t d0 = ((uint64_t)(e0.y << 20) << 32) | (e0.x << 20);
          uint64_t d1 = ((uint64_t)(e1.y << 20) << 32) | (e1.x << 20);
          asm("add.rn.f32x2 %0, %0, %1;" : "+l"(rs) : "l"(d0));
          asm("add.rn.f32x2 %0, %0, %1;" : "+l"(rs) : "l"(d1));
          w[c / 4] = __byte_perm(__byte_perm(e0.x, e0.y, 0x0040), __byte_perm(e1.x, e1.y, 0x0040), 0x5410);
        }
        r = (__uint_as_float((uint32_t)rs) + __uint_as_float((uint32_t)(rs >> 32))) * 0x1p120f;
      } else {
        float rsum = 0.0f;
#pragma unroll
        for (int c = 0; c < 128; c += 4) {
          uint32_t cc[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            cc[u] = expcast_code(__uint_as_float(s[c + u]), a, b);
            rsum += __uint_as_float(cc[u] << 20);
          }
          w[c / 4] = cc[0] | (cc[1] << 8) | (cc[2] << 16) | (cc[3] << 24);
        }
        r = rsum * 0x1p120f;
      }

      if (j > 0) {
        ok = mbar_wait(bar(B_PVDONE + t), (j - 1) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      // P^ row into the 128-byte-swizzled K-major tile: 16-byte chunk c of row
      // `row` lives at chunk c ^ (row % 8)
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(prow + ((c ^ (row & 7)) << 4)) =
            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
      // r operand row: (r_hi, r_lo, r_hi, 0, ...) in bf16
      {
        const uint16_t rhi = f32_to_bf16_bits(r);
        const uint16_t rlo = f32_to_bf16_bits(r - bf16_bits_to_f32(rhi));
        *reinterpret_cast<uint4*>(asrow) =
            make_uint4((uint32_t)rhi | ((uint32_t)rlo << 16), (uint32_t)rhi, 0u, 0u);
      }
      // correction: rescale the accumulator row when the running max rose
      if (j > 0 && __any_sync(0xffffffffu, alpha < 1.0f)) {
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tA + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
          tmem_st32(tA + c0, v);
        }
        tmem_st_wait();
      }
      l = alpha * l + r;
      M = Mn;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + t));
    }
    if (ok) ok = mbar_wait(bar(B_PVDONE + t), (p.nb - 1) & 1, abort_flag, p.status);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int grow = qt * 128 + row;
      const float inv_l = 1.0f / l;
      uint16_t* orow = p.out + ((size_t)bh * p.N + grow) * 128;
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tA + c0, v);
        tmem_ld_wait();
        if (grow < p.N) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint32_t pk[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float o0 = __uint_as_float(v[c + 2 * u]) * s_sv[c0 + c + 2 * u] * inv_l;
              const float o1 = __uint_as_float(v[c + 2 * u + 1]) * s_sv[c0 + c + 2 * u + 1] * inv_l;
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

int launch_attention_fp8(uint8_t* S, const vca_state_layout& L, int B, int H, int N, void* o,
                         cudaStream_t st) {
  const int BH = B * H, nb = (N + 127) / 128, Npad = nb * 128;
  CUtensorMap tq, tk, tr;
  if (!make_tmap_2d(&tq, S + L.qhat, 1, 128, (uint64_t)BH * Npad, 128, 128, 128) ||
      !make_tmap_2d(&tk, S + L.khat, 1, 128, (uint64_t)BH * Npad, 128, 128, 128) ||
      !make_tmap_2d(&tr, S + L.rhatT, 1, Npad, (uint64_t)BH * 128, Npad, 128, 128))
    return VCA_ERR_CUDA;
  Fp8Params p;
  p.sq = reinterpret_cast<const float*>(S + L.sq);
  p.sk = reinterpret_cast<const float*>(S + L.sk);
  p.sv = reinterpret_cast<const float*>(S + L.sv);
  p.mside = S + L.mside;
  p.hdr = reinterpret_cast<const uint32_t*>(S + L.header);
  p.out = reinterpret_cast<uint16_t*>(o);
  p.status = reinterpret_cast<int*>(S + L.status);
  p.B = B; p.H = H; p.N = N; p.nb = nb; p.Npad = Npad;
  p.npairs = (nb + 1) / 2;
  p.qk_scale = (float)(8.0 * 1.4426950408889634 / sqrt(128.0));
  if (cudaFuncSetAttribute(attn_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes) != cudaSuccess)
    return VCA_ERR_CUDA;
  const long long grid = (long long)BH * p.npairs;
  if (grid > 0x7FFFFFFF) return VCA_ERR_UNSUPPORTED;
  attn_fp8_kernel<<<(unsigned)grid, 384, kSmemBytes, st>>>(tq, tk, tr, p);
  return cudaGetLastError() == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}

}  // namespace vca
