// BF16 reference attention on tcgen05 (the role BF16 FlashAttention-4 plays in
// the paper's §4.1 "Baselines": the denominator of every speedup).
//
// Same skeleton as the 8-bit kernel: one CTA owns two 128-row query tiles of
// one (batch, head); warp 0 streams K_j and V_j through a 2-stage TMA ring,
// warp 1 issues the MMAs, warps 4-7 / 8-11 run the online softmax of tile 0 /
// tile 1 with the exact running maximum (paper Eq 1).  The probabilities are
// rounded to bf16 and written into the S columns of tensor memory, and the
// PV product reads them from there (A operand in TMEM).  V is consumed in its
// natural [key][channel] layout as an MN-major B operand.
#include "common.cuh"
#include "prep.h"

namespace vca {
namespace {

constexpr int kStages = 2;
constexpr uint32_t kHalf = 16384;                  // 128 rows x 64 bf16
constexpr uint32_t kTile = 2 * kHalf;              // 128 x 128 bf16
constexpr uint32_t kStageBytes = 2 * kTile;        // K_j, V_j
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_KV = 2 * kTile;
constexpr uint32_t OFF_BAR = OFF_KV + kStages * kStageBytes;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;

enum { B_QFULL = 0, B_KVFULL = 1, B_KVEMPTY = B_KVFULL + kStages, B_SFULL = B_KVEMPTY + kStages,
       B_PFULL = B_SFULL + 2, B_PVDONE = B_PFULL + 2, B_DRAIN = B_PVDONE + 2,
       B_COUNT = B_DRAIN + 1 };

struct Bf16Params {
  uint16_t* out;
  int* status;
  int N, nb, npairs;
  float scale_log2;  // log2(e) / sqrt(128)
};

__device__ int g_bf16_status;  // status word used when the caller passes none

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__global__ void __launch_bounds__(384, 1)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const Bf16Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + B_COUNT * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_BAR + B_COUNT * 8 + 4);
  auto bar = [&](int i) { return base + OFF_BAR + 8u * (uint32_t)i; };
  int* status = p.status;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bh = blockIdx.x / p.npairs, pair = blockIdx.x % p.npairs;
  const int qt0 = 2 * pair, ntiles = min(2, p.nb - qt0);
  if (*(volatile int*)status != 0) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), (i == B_PFULL || i == B_PFULL + 1) ? 128 : 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
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
    if (lane == 0) {
      mbar_expect_tx(bar(B_QFULL), ntiles * kTile);
      for (int t = 0; t < ntiles; ++t)
        for (int h = 0; h < 2; ++h)
          tma_load_3d(base + OFF_Q + t * kTile + h * kHalf, &tmQ, bar(B_QFULL), 64 * h,
                      (qt0 + t) * 128, bh);
      int issued = 0;
      for (int j = 0; j < p.nb; ++j) {
        const int s = j % kStages;
        if (j >= kStages && !mbar_wait(bar(B_KVEMPTY + s), ((j / kStages) - 1) & 1, abort_flag, status))
          break;
        const uint32_t st = base + OFF_KV + s * kStageBytes;
        mbar_expect_tx(bar(B_KVFULL + s), kStageBytes);
        for (int h = 0; h < 2; ++h) {
          tma_load_3d(st + h * kHalf, &tmK, bar(B_KVFULL + s), 64 * h, j * 128, bh);
          tma_load_3d(st + kTile + h * kHalf, &tmV, bar(B_KVFULL + s), 64 * h, j * 128, bh);
        }
        ++issued;
      }
      if (*abort_flag) {
        const uint64_t t0 = globaltimer();
        for (int j = max(0, issued - kStages); j < issued; ++j)
          while (!mbar_try_wait(bar(B_KVFULL + j % kStages), (j / kStages) & 1) &&
                 globaltimer() - t0 < kWaitLimitNs) {
          }
      }
    }
  } else if (warp == 1) {
    // Warp-uniform loop; one elected lane issues each MMA and commit.
    {
      const uint32_t iqk = idesc_bf16(128, 128), ipv = idesc_bf16(128, 128, true);
      const uint64_t dq0 = desc_k_sw128(base + OFF_Q), dk0 = desc_k_sw128(base + OFF_KV);
      const uint64_t dv0 = make_desc(base + OFF_KV + kTile, kHalf, 1024, 2);
      const uint64_t dstage = kStageBytes >> 4, dtile = kTile >> 4, dhalf = kHalf >> 4;
      bool ok = mbar_wait_spin(bar(B_QFULL), 0, abort_flag, status);
      // Per tile: PV_j^t as soon as its probabilities are in TMEM, then S_{j+1}^t
      // once PV_j^t has consumed them (P aliases the S columns).  The tiles
      // alternate, so one tile's products overlap the other's softmax.
      auto issue_s = [&](int j, int t) {
        const uint64_t dk = dk0 + (j % kStages) * dstage, dq = dq0 + t * dtile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t o = (kk / 4) * dhalf + (kk % 4) * 2;
          mma_f16_ss_w(tmem + 256 * t, dq + o, dk + o, iqk, kk > 0);
        }
        mma_commit_w(bar(B_SFULL + t));
      };
      if (ok) ok = mbar_wait_spin(bar(B_KVFULL), 0, abort_flag, status);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        for (int t = 0; t < ntiles; ++t) issue_s(0, t);
      } else {
        ok = false;
      }
      for (int j = 0; ok && j < p.nb; ++j) {
        const uint64_t dv = dv0 + (j % kStages) * dstage;
        for (int t = 0; t < ntiles && ok; ++t) {
          ok = mbar_wait_spin(bar(B_PFULL + t), j & 1, abort_flag, status);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_f16_ts_w(tmem + 256 * t + 128, tmem + 256 * t + 8 * kk, dv + kk * (2048 >> 4), ipv,
                         (j > 0 || kk > 0));
          mma_commit_w(bar(B_PVDONE + t));
          if (j + 1 < p.nb) {
            const int s1 = (j + 1) % kStages;
            if (t == 0) ok = mbar_wait_spin(bar(B_KVFULL + s1), ((j + 1) / kStages) & 1, abort_flag, status);
            if (ok) ok = mbar_wait_spin(bar(B_PVDONE + t), j & 1, abort_flag, status);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            issue_s(j + 1, t);
          }
        }
        if (ok) mma_commit_w(bar(B_KVEMPTY + j % kStages));
      }
      mma_commit_w(bar(B_DRAIN));
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar(B_DRAIN), 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  } else if (warp >= 4 && (warp - 4) / 4 < ntiles) {
    const int t = (warp - 4) / 4, quarter = warp % 4, row = quarter * 32 + lane;
    const uint32_t tS = tmem + ((uint32_t)(quarter * 32) << 16) + 256 * t;
    const uint32_t tA = tS + 128;
    const int last_valid = p.N - (p.nb - 1) * 128;
    float M = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < p.nb; ++j) {
      ok = mbar_wait(bar(B_SFULL + t), j & 1, abort_flag, status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t s[128];
      tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
      tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
      tmem_ld_wait();
      if (j == p.nb - 1 && last_valid < 128) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= last_valid) s[c] = 0xFF800000u;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; c += 2) mx = max3f(mx, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
      const float Mn = fmaxf(M, mx * p.scale_log2);
      const float alpha = ex2f(M - Mn);
      float rs0 = 0.0f, rs1 = 0.0f;
      uint32_t pw[64];
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        const float p0 = ex2f(fmaf(__uint_as_float(s[c]), p.scale_log2, -Mn));
        const float p1 = ex2f(fmaf(__uint_as_float(s[c + 1]), p.scale_log2, -Mn));
        rs0 += p0;
        rs1 += p1;
        pw[c / 2] = pack_bf16x2(p0, p1);
      }
      // probabilities into the first 64 columns of this tile's S region
      tmem_st32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&pw[0]));
      tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pw[32]));
      if (j > 0) {
        ok = mbar_wait(bar(B_PVDONE + t), (j - 1) & 1, abort_flag, status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha < 1.0f)) {
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tA + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
            tmem_st32(tA + c0, v);
          }
        }
      }
      tmem_st_wait();
      l = alpha * l + (rs0 + rs1);
      M = Mn;
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + t));
    }
    if (ok) ok = mbar_wait(bar(B_PVDONE + t), (p.nb - 1) & 1, abort_flag, status);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int grow = (qt0 + t) * 128 + row;
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
            for (int u = 0; u < 4; ++u)
              pk[u] = pack_bf16x2(__uint_as_float(v[c + 2 * u]) * inv_l,
                                  __uint_as_float(v[c + 2 * u + 1]) * inv_l);
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

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, int N, int BH) {
  typedef CUresult (*Fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                         const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                         CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                         CUtensorMapFloatOOBfill);
  static Fn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !ptr)
      return false;
    fn = (Fn)ptr;
  }
  // [BH][N][128] bf16: rows past N inside a head read as zeros
  const cuuint64_t dims[3] = {128, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {256, (cuuint64_t)N * 256};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_attention_bf16(const void* q, const void* k, const void* v, int B, int H, int N,
                          void* o, int* status, cudaStream_t st) {
  const int BH = B * H, nb = (N + 127) / 128;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_bf16_3d(&tq, q, N, BH) || !make_tmap_bf16_3d(&tk, k, N, BH) ||
      !make_tmap_bf16_3d(&tv, v, N, BH))
    return VCA_ERR_CUDA;
  Bf16Params p;
  p.out = reinterpret_cast<uint16_t*>(o);
  if (!status && cudaGetSymbolAddress((void**)&status, g_bf16_status) != cudaSuccess)
    return VCA_ERR_CUDA;
  p.status = status;
  p.N = N;
  p.nb = nb;
  p.npairs = (nb + 1) / 2;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt(128.0));
  if (cudaFuncSetAttribute(attn_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes) != cudaSuccess)
    return VCA_ERR_CUDA;
  const long long grid = (long long)BH * p.npairs;
  if (grid > 0x7FFFFFFF) return VCA_ERR_UNSUPPORTED;
  attn_bf16_kernel<<<(unsigned)grid, 384, kSmemBytes, st>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}

}  // namespace vca
