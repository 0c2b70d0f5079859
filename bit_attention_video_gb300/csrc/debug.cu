// Test entry points: the ExpCast device function, the format encoders, and a
// single-tile tcgen05 product with each operand layout the kernels rely on.
#include "common.cuh"
#include "expcast.cuh"

namespace vca {
namespace {

__global__ void expcast_kernel(const float* acc, const float* a, const float* b, uint8_t* out,
                               size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    out[i] = (uint8_t)expcast_code(acc[i], a[i], b[i]);
}

// The softmax's per-row byte step of the 8-bit attention kernel, one thread
// per row of 128 scores: mask the keys at and past valid[r], Mn = max(M[r],
// a[r] * rowmax), then the ExpCast bytes relative to Mn (the same device
// functions the kernel calls).
__global__ void __launch_bounds__(64) expcast_rows_kernel(const float* s, const float* a,
                                                          const float* M, const int* valid,
                                                          uint8_t* codes, float* Mn_out,
                                                          size_t rows) {
  for (size_t r = blockIdx.x * (size_t)blockDim.x + threadIdx.x; r < rows;
       r += (size_t)gridDim.x * blockDim.x) {
    uint32_t sv[128];
#pragma unroll
    for (int c = 0; c < 128; ++c) sv[c] = __float_as_uint(s[r * 128 + c]);
    const int vl = valid[r];
    if (vl < 128) mask_tail128(sv, vl);
    const float ar = a[r];
    bool has_nan;
    const float Mn = fmaxf(M[r], ar * row_max128_flag(sv, has_nan));
    uint32_t w[32];
    expcast_row_bytes(sv, ar, Mn, has_nan, w);
    uint4* o = reinterpret_cast<uint4*>(codes + r * 128);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    Mn_out[r] = Mn;
  }
}

// Failure path of the bounded waits: one CTA whose two barriers are never
// arrived at.  Warp 0 waits on barrier 0 with the limit `limit_ns` (mode 0:
// the suspending wait, mode 1: the spinning wait of the MMA issuers) and,
// when it gives up, records the timeout and raises the CTA's abort flag;
// warp 1 waits on barrier 1 with the kernels' own one-second limit and must
// leave through that flag.  out[w] = 1 if warp w's wait returned false,
// out[2 + w] = its nanoseconds in the wait.  No copy is in flight.
__global__ void __launch_bounds__(64) wait_timeout_kernel(int mode, uint64_t limit_ns, int* status,
                                                          uint64_t* out) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const uint64_t t0 = globaltimer();
  bool ok;
  if (warp == 0)
    ok = mode == 0   ? mbar_wait(smem_u32(&bars[0]), 0, &abort_flag, status, limit_ns)
         : mode == 1 ? mbar_wait_spin(smem_u32(&bars[0]), 0, &abort_flag, status, limit_ns)
                     : mbar_wait_poll(smem_u32(&bars[0]), 0, &abort_flag, status, limit_ns);
  else
    ok = mbar_wait(smem_u32(&bars[1]), 0, &abort_flag, status);
  const uint64_t t1 = globaltimer();
  if (lane == 0) {
    out[warp] = ok ? 0u : 1u;
    out[2 + warp] = t1 - t0;
  }
}

__global__ void encode_kernel(const float* x, uint8_t* e4, uint8_t* e2, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    e4[i] = f32_to_e4m3(x[i]);
    e2[i] = f32x2_to_e2m1x2(x[i], 0.0f) & 0x0F;
  }
}

// Byte offset of element (r, k) of a K-major tile with 128-byte swizzle;
// `ebytes` bytes per element, 128/ebytes elements per swizzle atom column,
// atom columns `atom_stride` bytes apart.
__device__ uint32_t off_k_sw128(int r, int k, int ebytes, uint32_t atom_stride) {
  const int per_atom = 128 / ebytes;
  const int atom = k / per_atom, kb = (k % per_atom) * ebytes;
  return atom * atom_stride + r * 128 + ((((kb >> 4) ^ (r & 7)) << 4) | (kb & 15));
}
// MN-major, 128-byte swizzle, 16-bit elements: MN chunks of 64 `lbo` bytes
// apart, K rows of 128 bytes, 8-row groups of 1024 bytes.
__device__ uint32_t off_mn_sw128(int n, int k, uint32_t lbo) {
  const int chunk = n / 64, nb = (n % 64) * 2;
  return chunk * lbo + k * 128 + ((((nb >> 4) ^ (k & 7)) << 4) | (nb & 15));
}
// K-major, no swizzle: 8-row x 16-byte core matrices, LBO along K, SBO along M/N.
__device__ uint32_t off_k_plain(int r, int k, int ebytes, uint32_t lbo, uint32_t sbo) {
  const int kb = k * ebytes;
  return (r / 8) * sbo + (kb / 16) * lbo + (r % 8) * 16 + (kb % 16);
}

constexpr uint32_t kDbgSmem = 200 * 1024;
__device__ int g_debug_status;  // wait-timeout bits of the layout test kernel

__global__ void __launch_bounds__(128, 1)
    mma_kernel(int mode, const uint8_t* a, const uint8_t* b, float* d) {
  int* status = &g_debug_status;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t A = base, B = base + 65536;  // operand regions
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
  }
  for (uint32_t i = tid; i < kDbgSmem / 4; i += 128) reinterpret_cast<uint32_t*>(sm)[i] = 0;
  __syncthreads();

  const uint16_t* a16 = reinterpret_cast<const uint16_t*>(a);
  const uint16_t* b16 = reinterpret_cast<const uint16_t*>(b);
  // operands into shared memory
  if (mode == 0 || mode == 5 || mode == 6) {  // FP8 K-major swizzled, K = 128
    for (int i = tid; i < 128 * 128; i += 128) {
      int r = i / 128, k = i % 128;
      if (mode != 5) sm[(A - base) + off_k_sw128(r, k, 1, 16384)] = a[i];
      sm[(B - base) + off_k_sw128(r, k, 1, 16384)] = b[i];
    }
  }
  if (mode == 1 || mode == 4) {  // BF16 K-major swizzled, K = 128 (two atom columns)
    for (int i = tid; i < 128 * 128; i += 128) {
      int r = i / 128, k = i % 128;
      if (mode == 1) *reinterpret_cast<uint16_t*>(sm + (A - base) + off_k_sw128(r, k, 2, 16384)) = a16[i];
      *reinterpret_cast<uint16_t*>(sm + (B - base) + off_k_sw128(r, k, 2, 16384)) = b16[i];
    }
  }
  if (mode == 2) {  // A K-major swizzled K = 64; B MN-major swizzled
    for (int i = tid; i < 128 * 64; i += 128) {
      int r = i / 64, k = i % 64;
      *reinterpret_cast<uint16_t*>(sm + (A - base) + off_k_sw128(r, k, 2, 16384)) = a16[i];
      *reinterpret_cast<uint16_t*>(sm + (B - base) + off_mn_sw128(r, k, 8192)) = b16[i];
    }
  }
  if (mode == 3 || mode == 6) {  // BF16 K-major no swizzle, K = 16
    const uint16_t* as = mode == 6 ? reinterpret_cast<const uint16_t*>(a + 128 * 128) : a16;
    const uint16_t* bs = mode == 6 ? reinterpret_cast<const uint16_t*>(b + 128 * 128) : b16;
    const uint32_t A2 = mode == 6 ? A + 32768 : A, B2 = mode == 6 ? B + 32768 : B;
    for (int i = tid; i < 128 * 16; i += 128) {
      int r = i / 16, k = i % 16;
      *reinterpret_cast<uint16_t*>(sm + (A2 - base) + off_k_plain(r, k, 2, 128, 256)) = as[i];
      *reinterpret_cast<uint16_t*>(sm + (B2 - base) + off_k_plain(r, k, 2, 128, 256)) = bs[i];
    }
  }
  // Mode 7 (NVFP4): a and b each hold [128][64] packed E2M1 bytes (element 2i
  // in the low nibble) and then [128][8] UE4M3 scales, one per 16 elements.
  // Operands go to the 64-byte-swizzled K-major layout; the scales to the
  // layout the scale copy reads: for K step s, 512 bytes where row m, block
  // kb (of that step's four) sits at (m % 32) * 16 + (m / 32) * 4 + kb.
  constexpr uint32_t kSfA = 32768, kSfB = 33792;
  if (mode == 7) {
    for (int i = tid; i < 128 * 4; i += 128) {
      const int r = i / 4, c = i % 4;
      *reinterpret_cast<uint4*>(sm + (A - base) + off_sw64(r, c)) =
          *reinterpret_cast<const uint4*>(a + r * 64 + c * 16);
      *reinterpret_cast<uint4*>(sm + (B - base) + off_sw64(r, c)) =
          *reinterpret_cast<const uint4*>(b + r * 64 + c * 16);
    }
    for (int i = tid; i < 128 * 8; i += 128) {
      const int m = i / 8, kb = i % 8;
      const uint32_t o = (kb / 4) * 512 + (m % 32) * 16 + (m / 32) * 4 + kb % 4;
      sm[(A - base) + kSfA + o] = a[8192 + i];
      sm[(A - base) + kSfB + o] = b[8192 + i];
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

  // A operand in tensor memory (columns 128..): row r in lane r, K packed
  // little-endian into 32-bit columns (2 bf16 or 4 fp8 per column).
  if (mode == 4 || mode == 5) {
    const int r = warp * 32 + lane;
    const int ncol = mode == 4 ? 64 : 32;
    for (int c0 = 0; c0 < ncol; c0 += 32) {
      uint32_t w[32];
      for (int c = 0; c < 32; ++c) {
        if (mode == 4)
          w[c] = (uint32_t)a16[r * 128 + 2 * (c0 + c)] |
                 ((uint32_t)a16[r * 128 + 2 * (c0 + c) + 1] << 16);
        else
          w[c] = *reinterpret_cast<const uint32_t*>(a + r * 128 + 4 * (c0 + c));
      }
      tmem_st32(tmem + lane_base + 128 + c0, w);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (tid == 0 && mode != 7) {
    const uint32_t i8 = idesc_f8(128, 128), i16 = idesc_bf16(128, 128),
                   i16mn = idesc_bf16(128, 128, true);
    if (mode == 0 || mode == 6)
      for (int s = 0; s < 4; ++s)
        mma_f8_ss(tmem, desc_k_sw128(A + 32 * s), desc_k_sw128(B + 32 * s), i8, s > 0);
    if (mode == 1)
      for (int s = 0; s < 8; ++s) {
        uint32_t o = (s / 4) * 16384 + (s % 4) * 32;
        mma_f16_ss(tmem, desc_k_sw128(A + o), desc_k_sw128(B + o), i16, s > 0);
      }
    if (mode == 2)
      for (int s = 0; s < 4; ++s)
        mma_f16_ss(tmem, desc_k_sw128(A + 32 * s), make_desc(B + 2048 * s, 8192, 1024, 2), i16mn,
                   s > 0);
    if (mode == 3)
      mma_f16_ss(tmem, desc_k_plain(A, 128, 256), desc_k_plain(B, 128, 256), i16, 0);
    if (mode == 6)
      mma_f16_ss(tmem, desc_k_plain(A + 32768, 128, 256), desc_k_plain(B + 32768, 128, 256), i16,
                 1);
    if (mode == 4)
      for (int s = 0; s < 8; ++s) {
        uint32_t o = (s / 4) * 16384 + (s % 4) * 32;
        mma_f16_ts(tmem, tmem + 128 + 8 * s, desc_k_sw128(B + o), i16, s > 0);
      }
    if (mode == 5)
      for (int s = 0; s < 4; ++s)
        mma_f8_ts(tmem, tmem + 128 + 8 * s, desc_k_sw128(B + 32 * s), i8, s > 0);
    mma_commit(smem_u32(&bar));
  }
  if (mode == 7 && warp == 0) {
    // scale factors: A in columns 128.., B in columns 160.., four per K step
    for (int s = 0; s < 2; ++s) {
      tmem_cp_32x128b_x4_w(tmem + 128 + 4 * s, desc_k_plain(A + kSfA + 512 * s, 512, 128));
      tmem_cp_32x128b_x4_w(tmem + 160 + 4 * s, desc_k_plain(A + kSfB + 512 * s, 512, 128));
    }
    for (int s = 0; s < 2; ++s)
      mma_nvf4_ss_w(tmem, desc_k_sw64(A + 32 * s), desc_k_sw64(B + 32 * s), idesc_nvf4(128, 128),
                    tmem + 128 + 4 * s, tmem + 160 + 4 * s, s > 0);
    mma_commit_w(smem_u32(&bar));
  }
  __syncwarp();
  const bool ok = mbar_wait(smem_u32(&bar), 0, &abort_flag, status);
  tc_fence_after();
  if (ok) {
    const int r = warp * 32 + lane;
    for (int c0 = 0; c0 < 128; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_base + c0, v);
      tmem_ld_wait();
      for (int c = 0; c < 32; ++c) d[r * 128 + c0 + c] = __uint_as_float(v[c]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace
}  // namespace vca

using namespace vca;

extern "C" int vca_debug_expcast(const float* acc, const float* a, const float* b, uint8_t* out,
                                 size_t n, vca_stream_t stream) {
  if (n == 0) return VCA_OK;
  if (!acc || !a || !b || !out) return VCA_ERR_INVALID_ARG;
  int blocks = (int)std::min<size_t>((n + 255) / 256, 152 * 16);
  expcast_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(acc, a, b, out, n);
  return cudaGetLastError() == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}

extern "C" int vca_debug_expcast_rows(const float* s, const float* a, const float* M,
                                      const int* valid, uint8_t* codes, float* Mn, size_t rows,
                                      vca_stream_t stream) {
  if (rows == 0) return VCA_OK;
  if (!s || !a || !M || !valid || !codes || !Mn) return VCA_ERR_INVALID_ARG;
  if (((uintptr_t)codes & 15u) || rows > ((size_t)1 << 24)) return VCA_ERR_INVALID_ARG;
  const int blocks = (int)std::min<size_t>((rows + 63) / 64, 152 * 8);
  expcast_rows_kernel<<<blocks, 64, 0, (cudaStream_t)stream>>>(s, a, M, valid, codes, Mn, rows);
  return cudaGetLastError() == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}

extern "C" int vca_debug_wait_timeout(int mode, uint64_t limit_ns, int* status, uint64_t* out,
                                      vca_stream_t stream) {
  if (mode < 0 || mode > 2 || !status || !out) return VCA_ERR_INVALID_ARG;
  if (limit_ns == 0 || limit_ns > vca::kWaitLimitNs / 10) return VCA_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(mode, limit_ns, status, out);
  return cudaGetLastError() == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}

extern "C" int vca_debug_encode(const float* x, uint8_t* e4, uint8_t* e2, size_t n,
                                vca_stream_t stream) {
  if (n == 0) return VCA_OK;
  if (!x || !e4 || !e2) return VCA_ERR_INVALID_ARG;
  int blocks = (int)std::min<size_t>((n + 255) / 256, 152 * 16);
  encode_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(x, e4, e2, n);
  return cudaGetLastError() == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}

extern "C" int vca_debug_mma(int mode, const void* a, const void* b, float* d,
                             vca_stream_t stream) {
  if (mode < 0 || mode > 7 || !a || !b || !d) return VCA_ERR_INVALID_ARG;
  if (cudaFuncSetAttribute(mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kDbgSmem + 1024) != cudaSuccess)
    return VCA_ERR_CUDA;
  mma_kernel<<<1, 128, kDbgSmem + 1024, (cudaStream_t)stream>>>(
      mode, (const uint8_t*)a, (const uint8_t*)b, d);
  return cudaGetLastError() == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}
