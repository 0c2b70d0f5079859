// Shared device helpers for the VC-Attention sm_103a kernels: status codes,
// bounded mbarrier waits, TMA and tcgen05 (TMEM, UMMA) inline PTX, UMMA
// descriptors, and the E4M3 / E2M1 / bf16 conversions.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/vca.h"

namespace vca {

// ----------------------------------------------------------------------------
// Device status word (lives in the state blob).  Kernels OR error bits into it
// and skip their work once any bit is set.
// ----------------------------------------------------------------------------
enum : int {
  kStatTimeout = 1 << 0,      // a bounded wait expired (pipeline did not advance)
  kStatNoPerm = 1 << 1,       // reuse requested but the blob holds no matching permutation
  kStatStateMismatch = 1 << 2,  // the blob header does not match the call's shape
  kStatBadArg = 1 << 3,       // device-side argument check failed
};

// Wall-clock limit of every spin-wait in the pipelined kernels.  The longest
// legitimate wait is one pipeline stage (microseconds); one second means the
// pipeline is stuck, and the kernel gives up instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;

// Index checks of the debug build (compiled with -DVCA_DEBUG), standing in
// for a memory checker: an index that addresses memory and comes from data
// (a cached permutation, a label) is tested against its array's extent
// before use; one outside [0, n) records kStatBadArg in the status word and
// the access is skipped (a read gives zeros).  Release builds compile the
// test away.
#ifdef VCA_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif
__device__ __forceinline__ bool index_ok(long long i, long long n, const int* status) {
  if constexpr (kDebugChecks) {
    if (i < 0 || i >= n) {
      atomicOr(const_cast<int*>(status), kStatBadArg);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ----------------------------------------------------------------------------
// mbarrier
// ----------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of the phase of `parity` (a few cycles; try_wait costs
// over a hundred even on a completed phase).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same test, but the thread may be suspended up to `hint_ns` while the
// phase is incomplete (no busy spinning).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `parity` to complete, for at most `limit_ns`.  On
// expiry, or if another warp of the CTA already gave up (abort flag), returns
// false after recording the timeout in the device status word.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if ((n & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(status, kStatTimeout);
        return false;
      }
    }
  }
}

// The same bound, by non-blocking tests ~128 ns apart: the waiting warp holds
// no suspended try_wait.  The 4-bit attention's S issuer waits this way (its
// sub-partition's softmax warps then lose fewer cycles to it; 32-96 ns apart
// the tests cost them more, 256 ns and longer delay the hand-over).
__device__ __forceinline__ bool mbar_wait_poll(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, int* status,
                                               uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t n = 1;; ++n) {
    __nanosleep(128);
    if (mbar_test_wait(bar, parity)) return true;
    if ((n & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(status, kStatTimeout);
        return false;
      }
    }
  }
}

// mbar_wait for a phase that has usually completed already: the non-blocking
// test first.
__device__ __forceinline__ bool mbar_wait_likely(uint32_t bar, uint32_t parity,
                                                 volatile int* abort_flag, int* status) {
  return mbar_test_wait(bar, parity) || mbar_wait(bar, parity, abort_flag, status);
}

// The same bound, busy-polling without suspension: for the one thread whose
// reaction time is on the critical path (the MMA issuer).
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, int* status,
                                               uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(status, kStatTimeout);
        return false;
      }
    }
  }
}

// ----------------------------------------------------------------------------
// TMA (bulk tensor copies) and plain bulk copies, global -> shared
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// Make generic-proxy shared-memory writes visible to the async proxy (the
// tensor core reads operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f8f6f4 (E4M3 x E4M3 -> f32)
__device__ __forceinline__ void mma_f8_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accum) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
// kind::f16 with both operands from shared memory
__device__ __forceinline__ void mma_f16_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t accum) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
// kind::f16 with A from tensor memory
__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                           uint32_t accum) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
// kind::f8f6f4 with A from tensor memory
__device__ __forceinline__ void mma_f8_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                          uint32_t accum) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
// Warp-uniform forms: every lane of the warp executes the call with the same
// operands (so the compiler keeps them in uniform registers) and the lowest
// active lane, chosen by elect.sync, issues the instruction.
__device__ __forceinline__ void mma_f8_ss_w(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t accum) {
  asm volatile(
      "{\n.reg .pred p, q;\nelect.sync _|p, 0xffffffff;\nsetp.ne.u32 q, %4, 0;\n"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, q;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void mma_f8_ts_w(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t accum) {
  asm volatile(
      "{\n.reg .pred p, q;\nelect.sync _|p, 0xffffffff;\nsetp.ne.u32 q, %4, 0;\n"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, q;\n}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void mma_f16_ss_w(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                             uint32_t accum) {
  asm volatile(
      "{\n.reg .pred p, q;\nelect.sync _|p, 0xffffffff;\nsetp.ne.u32 q, %4, 0;\n"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, q;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void mma_f16_ts_w(uint32_t d, uint32_t a_tmem, uint64_t b,
                                             uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n.reg .pred p, q;\nelect.sync _|p, 0xffffffff;\nsetp.ne.u32 q, %4, 0;\n"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, q;\n}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
// kind::mxf4nvf4 block-scaled product (NVFP4): E2M1 x E2M1 -> f32 with one
// UE4M3 scale per 16 elements along K (scale_vec::4X: four scales per row for
// the K = 64 of one instruction).  Both operands come from shared memory; the
// scale factors of A and B sit in tensor memory (`sfa`, `sfb`).
__device__ __forceinline__ void mma_nvf4_ss_w(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t sfa, uint32_t sfb, uint32_t accum) {
  asm volatile(
      "{\n.reg .pred p, q;\nelect.sync _|p, 0xffffffff;\nsetp.ne.u32 q, %4, 0;\n"
      "@p tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
      "[%0], %1, %2, %3, [%5], [%6], q;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum), "r"(sfa), "r"(sfb)
      : "memory");
}
// Copy 32 rows x 16 bytes of shared memory (a no-swizzle K-major matrix,
// rows 16 bytes apart) into tensor memory columns [col, col+4), replicated
// into all four 32-lane quarters.  This is how block scale factors reach the
// tensor core: for a 128-row operand, lane l, column col+i holds the four
// scales of row 32 i + l.  Ordered with the MMAs the same thread issues.
__device__ __forceinline__ void tmem_cp_32x128b_x4_w(uint32_t taddr, uint64_t sdesc) {
  asm volatile(
      "{\n.reg .pred p;\nelect.sync _|p, 0xffffffff;\n"
      "@p tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n}" ::"r"(taddr),
      "l"(sdesc)
      : "memory");
}
// A whole K=128 FP8 product as four K=32 MMAs from one elected lane: the
// descriptors of steps 1-3 advance the start address by 32 bytes (+2 in the
// >>4 encoding).  `accum` decides only the first step.
__device__ __forceinline__ void mma4_f8_ss_w(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                             uint32_t accum) {
  asm volatile(
      "{\n.reg .pred p, q, t;\n.reg .b64 a1, a2, a3, b1, b2, b3;\n"
      "elect.sync _|p, 0xffffffff;\nsetp.ne.u32 q, %4, 0;\nsetp.eq.u32 t, 0, 0;\n"
      "add.s64 a1, %1, 2;\nadd.s64 a2, %1, 4;\nadd.s64 a3, %1, 6;\n"
      "add.s64 b1, %2, 2;\nadd.s64 b2, %2, 4;\nadd.s64 b3, %2, 6;\n"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, q;\n"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a1, b1, %3, t;\n"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a2, b2, %3, t;\n"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a3, b3, %3, t;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
// The same with A (four columns of bytes per step: 8 columns) in tensor memory.
__device__ __forceinline__ void mma4_f8_ts_w(uint32_t d, uint32_t a_tmem, uint64_t b,
                                             uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n.reg .pred p, q, t;\n.reg .b32 a1, a2, a3;\n.reg .b64 b1, b2, b3;\n"
      "elect.sync _|p, 0xffffffff;\nsetp.ne.u32 q, %4, 0;\nsetp.eq.u32 t, 0, 0;\n"
      "add.u32 a1, %1, 8;\nadd.u32 a2, %1, 16;\nadd.u32 a3, %1, 24;\n"
      "add.s64 b1, %2, 2;\nadd.s64 b2, %2, 4;\nadd.s64 b3, %2, 6;\n"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, q;\n"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a1], b1, %3, t;\n"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a2], b2, %3, t;\n"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a3], b3, %3, t;\n}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void mma_commit_w(uint32_t bar) {
  asm volatile(
      "{\n.reg .pred p;\nelect.sync _|p, 0xffffffff;\n"
      "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Instruction descriptor of kind::f16 / kind::f8f6f4 (dense, f32 accumulator).
//   bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format,
//   15 / 16 A / B major (0 = K-major, 1 = MN-major), 17-22 N>>3, 24-28 M>>4.
// Formats: kind::f8f6f4 E4M3 = 0; kind::f16 F16 = 0, BF16 = 1.
__host__ __device__ constexpr uint32_t idesc_f8(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major = false,
                                                 bool a_mn_major = false) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (a_mn_major ? (1u << 15) : 0u) |
         (b_mn_major ? (1u << 16) : 0u) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major ? (1u << 16) : 0u) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor of kind::mxf4nvf4 (block-scaled, f32 accumulator):
//   bits 4-5 B scale-factor id (0), 7-9 A format, 10-12 B format (E2M1 = 1),
//   15 / 16 A / B major (K-major only), 17-22 N>>3, 23 scale format
//   (0 = UE4M3), 24-28 M>>4, 29-30 A scale-factor id (0).
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (0u << 23) |
         ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor (tcgen05 form):
//   bits 0-13 start address >> 4, 16-29 leading byte offset >> 4,
//   32-45 stride byte offset >> 4, 46-47 version (1), 61-63 layout
//   (0 = no swizzle, 2 = 128-byte swizzle, 4 = 64-byte swizzle).
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(layout & 7u) << 61;
  return d;
}
// K-major tile of rows x 128 bytes, 128-byte swizzle, 8-row atoms of 1024 B
// (the layout a TMA load with CU_TENSOR_MAP_SWIZZLE_128B writes).
__device__ __forceinline__ uint64_t desc_k_sw128(uint32_t saddr) {
  return make_desc(saddr, 16, 1024, 2);
}
// K-major tile of rows x 64 bytes, 64-byte swizzle, 8-row atoms of 512 B
// (the layout a TMA load with CU_TENSOR_MAP_SWIZZLE_64B writes).
__device__ __forceinline__ uint64_t desc_k_sw64(uint32_t saddr) {
  return make_desc(saddr, 16, 512, 4);
}
// Byte offset of 16-byte chunk `c` (0..3) of row `r` in that layout.
__device__ __forceinline__ uint32_t off_sw64(int r, int c) {
  return (uint32_t)((r >> 3) * 512 + (r & 7) * 64 + ((c ^ ((r & 7) >> 1)) << 4));
}
// K-major, no swizzle: 8x16-byte core matrices; `lbo` steps along K, `sbo`
// steps along M/N.
__device__ __forceinline__ uint64_t desc_k_plain(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return make_desc(saddr, lbo, sbo, 0);
}

// 32 lanes x 32 columns of 32-bit values: thread i of the warp gets lane
// (warp's lane quarter + i), columns [col, col+32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// 32 lanes x 1 / 8 / 16 columns.
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
  return r;
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ----------------------------------------------------------------------------
// Number formats
// ----------------------------------------------------------------------------
// Two fp32 -> two E4M3 bytes (lo, hi), round to nearest even, saturate to +-448.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// four values, RNE with saturation, byte i = value i
__device__ __forceinline__ uint32_t f32x4_to_e4m3x4(float v0, float v1, float v2, float v3) {
  return (uint32_t)f32x2_to_e4m3x2(v0, v1) | ((uint32_t)f32x2_to_e4m3x2(v2, v3) << 16);
}
__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  return (uint8_t)(f32x2_to_e4m3x2(x, 0.0f) & 0xFF);
}
// Two fp32 -> two E2M1 codes packed in one byte (lo nibble = lo), RNE, +-6.
__device__ __forceinline__ uint8_t f32x2_to_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n.reg .b8 t;\ncvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\ncvt.u16.u8 %0, t;\n}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return (uint8_t)r;
}
// Value of an E4M3 byte (exact).  Via f16x2: E4M3 -> f16 is exact.
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  uint32_t h2;
  uint16_t in = c;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFF)));
}

// Four int8 (one word, byte i = element i) -> two f16x2 words, exactly:
// byte b is placed as the half 1024 + (b ^ 0x80) (exponent 10, so the low
// mantissa bits are the byte) and 1152 is subtracted.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x5140), b = __byte_perm(u, 0x64646464u, 0x5342);
  asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
  asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

}  // namespace vca
