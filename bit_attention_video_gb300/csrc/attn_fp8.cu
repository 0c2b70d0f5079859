// 8-bit VC-Attention forward (paper §3.1 Eq 1, §3.2 Eq 6, §3.3 Eq 7) on
// tcgen05 tensor cores.
//
// One CTA owns one 128-row query tile of one (batch, head) and streams all
// key blocks j of the permuted, centred keys K' and the transposed residual
// R^T through a TMA ring.  Warp roles:
//   warp 0        producer: TMA of the Q tile once; per stage K'_j, R^T_j and
//                 the 16 "slot" rows appended to R^T_j (written by the warp's
//                 lanes); the mean operand of each group of 8 blocks
//   warp 1        MMA issuer (warp-uniform loop, one elected lane issues;
//                 busy-polling) and TMEM owner
//   warps 4-11    softmax + correction + epilogue: two threads per query row
//                 (key columns 0-63 and 64-127, output columns 0-63 and
//                 64-127), which exchange the partial row maximum
//
// Tensor memory (448 of 512 columns):
//   [0,128), [128,256)  S_j = Q^ K'_j^T in buffer j % 2 (fp32)
//   [256,384)  the output accumulator A (128 channels)
//   [384,400)  two banks of 8 row-sum slots (see below), part of the same
//              accumulator, so the alpha rescaling covers them
//   [400,432)  P^_j (ExpCast bytes, 4 per column), the A operand of the product
//   [432,448)  a group's row-sum operand (bf16 hi, lo) of the mean product
//
// Per key block j:
//   S   = Q^ K'^_j^T                              FP8 MMA (N=128)
//   M'  = max(M, a_j rowmax(S))                   exact running max (x8, log2)
//   c   = clip_[0,120](RNE(a_j S + 119.65 - M'))  ExpCast-FP8 bytes -> TMEM
//   A  *= alpha = 2^((M - M')/8) when M rises     (TMEM correction)
//   A  += P^ [R^_j ; E_j]                          FP8 MMA (N=144), A from TMEM
// E_j (16 rows of K=128) is zero except row 8*bank + slot of block j, which is
// all ones: column 128 + 8 bank + slot of the product is the row sum r_j of
// exactly the bytes the product consumes.  Blocks form groups of 8 (aligned
// to the last block; only the first group can be partial) that alternate
// between the two banks.  After a group's last product the softmax reads its
// 8 slots rho (rescaled like the accumulator), adds them to l, clears the bank
// and writes rho as bf16 hi/lo to TMEM; three BF16 K=16 MMAs then add
// sum_g rho_g mutilde_g^T (Eq 6's mean term, hi/lo split of both factors).
// Epilogue: O = sV (.) A / l in bf16, original query order (Q is not permuted).
#include "common.cuh"
#include "expcast.cuh"
#include "prep.h"

namespace vca {
namespace {

constexpr int kStages = 5;
constexpr uint32_t kSlotRowsBytes = 16 * 128;                      // E_j: 16 rows x 128 keys
constexpr uint32_t kStageBytes = 2 * kTileBytes + kSlotRowsBytes;  // K'_j, R^T_j, E_j
constexpr uint32_t OFF_Q = 0;                                      // the query tile
constexpr uint32_t OFF_KV = kTileBytes;
constexpr uint32_t OFF_BG = OFF_KV + kStages * kStageBytes;    // mean operand, 2 buffers x 8 KB
constexpr uint32_t OFF_SV = OFF_BG + 2 * kGroupBytes;          // sV, 512 B
constexpr uint32_t OFF_XCH = OFF_SV + 512;                     // partial row max, 2 x 2 x 128 x 4 B
constexpr uint32_t OFF_BAR = OFF_XCH + 2048;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;  // + alignment slack
constexpr int kThreads = 384;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned");
static_assert(kGroup == 8, "eight row-sum slots per bank");

// TMEM columns
constexpr uint32_t TC_S = 0, TC_ACC = 256, TC_BANK = 384, TC_P = 400, TC_GHI = 432, TC_GLO = 440;

struct Fp8Params {
  const float* sq;        // [BH][nb]
  const float* sk;        // [BH][nb]
  const float* sv;        // [BH][128]
  const uint8_t* mside;   // [BH][ngroups][8192]
  const uint32_t* hdr;
  uint16_t* out;          // [BH][N][128]
  int* status;
  int B, H, N, nb, Npad, ngroups, gpad;
  float qk_scale;         // 8 log2(e) / sqrt(128)
};

// barrier indices
enum { B_QFULL = 0, B_KVFULL = 1, B_KVEMPTY = B_KVFULL + kStages, B_SFULL = B_KVEMPTY + kStages,
       B_SFREE = B_SFULL + 2, B_PFULL = B_SFREE + 2, B_PVDONE = B_PFULL + 1,
       B_DRAIN = B_PVDONE + 1, B_COUNT = B_DRAIN + 1 };

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

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// block j closes its mean group (slot kGroup - 1, or the last block)
__device__ __forceinline__ bool group_ends(int j, int nb, int gpad) {
  return j == nb - 1 || (j + gpad) % kGroup == kGroup - 1;
}

__global__ void __launch_bounds__(kThreads, 1)
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
  const int nb = p.nb, gpad = p.gpad;
  const int bh = blockIdx.x / nb, qt = blockIdx.x % nb;

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
    // "S read" and "P written" complete when all 256 softmax threads arrive
    for (int i = 0; i < B_COUNT; ++i)
      mbar_init(bar(i), (i >= B_SFREE && i < B_PVDONE) ? 256 : 1);
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
  if (threadIdx.x >= 128 && threadIdx.x < 256)
    s_sv[threadIdx.x - 128] = p.sv[(size_t)bh * 128 + threadIdx.x - 128];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    if (lane == 0) {
      mbar_expect_tx(bar(B_QFULL), kTileBytes);
      tma_load_2d(base + OFF_Q, &tmQ, bar(B_QFULL), 0, bh * p.Npad + qt * 128);
    }
    int issued = 0;
    for (int j = 0; j < nb; ++j) {
      const int s = j % kStages;
      if (j >= kStages) ok = mbar_wait(bar(B_KVEMPTY + s), ((j / kStages) - 1) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint32_t st = base + OFF_KV + s * kStageBytes;
      // E_j: 16 rows of 128 bytes (a 128-byte-swizzled tile whose rows are
      // uniform, so the swizzle does not move bytes); row 8*bank + slot is
      // 1.0 (0x38), the others 0.  Lane i writes 64 bytes.
      {
        const int slot_row = 8 * (((j + gpad) / kGroup) & 1) + (j + gpad) % kGroup;
        const uint32_t v = (lane / 2 == slot_row) ? 0x38383838u : 0u;
        uint4* e = reinterpret_cast<uint4*>(sm + OFF_KV + s * kStageBytes + 2 * kTileBytes) + lane * 4;
#pragma unroll
        for (int u = 0; u < 4; ++u) e[u] = make_uint4(v, v, v, v);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        const bool group_start = j == 0 || (j + gpad) % kGroup == 0;
        mbar_expect_tx(bar(B_KVFULL + s), 2 * kTileBytes + (group_start ? kGroupBytes : 0));
        tma_load_2d(st, &tmK, bar(B_KVFULL + s), 0, bh * p.Npad + j * 128);
        tma_load_2d(st + kTileBytes, &tmR, bar(B_KVFULL + s), j * 128, bh * 128);
        if (group_start) {
          const int g = (j + gpad) / kGroup;
          bulk_load(base + OFF_BG + (g & 1) * kGroupBytes,
                    p.mside + ((size_t)bh * p.ngroups + g) * kGroupBytes, kGroupBytes,
                    bar(B_KVFULL + s));
        }
      }
      ++issued;
    }
    if (lane == 0 && *abort_flag) {
      // let the copies in flight land before the CTA exits
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
    // The whole warp runs this loop (uniform control flow, operands in
    // uniform registers); one elected lane issues each MMA and commit.
    // S_0, S_1 up front; per block j, once P^_j is in TMEM: P^ [R^_j; E_j],
    // the mean product of a group closed by block j-1, and S_{j+2} into the
    // buffer the softmax released after reading S_j.
    {
      const uint32_t i8 = idesc_f8(128, 128), i8w = idesc_f8(128, 144),
                     i16 = idesc_bf16(128, 128);
      const uint64_t dq = desc_k_sw128(base + OFF_Q);
      const uint64_t dk0 = desc_k_sw128(base + OFF_KV);                  // stage 0 K'
      const uint64_t dr0 = desc_k_sw128(base + OFF_KV + kTileBytes);     // stage 0 [R^; E]
      const uint64_t dstage = kStageBytes >> 4;                          // per-stage step
      const uint64_t dbg0 = desc_k_plain(base + OFF_BG, 128, 256);
      const uint64_t dgroup = kGroupBytes >> 4, dhalf = (kGroupBytes / 2) >> 4;
      bool ok = mbar_wait_spin(bar(B_QFULL), 0, abort_flag, p.status);
      auto issue_s = [&](int j) {
        const int s = j % kStages;
        ok = mbar_wait_spin(bar(B_KVFULL + s), (j / kStages) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; return; }
        tc_fence_after();
        const uint64_t dk = dk0 + s * dstage;
        const uint32_t d = tmem + TC_S + 128 * (j & 1);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_f8_ss_w(d, dq + 2 * kk, dk + 2 * kk, i8, kk > 0);
        mma_commit_w(bar(B_SFULL + (j & 1)));
      };
      auto issue_flush = [&](int g) {
        // sum_g rho_g mutilde_g^T = rho_hi mu_hi + rho_lo mu_hi + rho_hi mu_lo
        const uint64_t bg = dbg0 + (g & 1) * dgroup;
        mma_f16_ts_w(tmem + TC_ACC, tmem + TC_GHI, bg, i16, 1);
        mma_f16_ts_w(tmem + TC_ACC, tmem + TC_GLO, bg, i16, 1);
        mma_f16_ts_w(tmem + TC_ACC, tmem + TC_GHI, bg + dhalf, i16, 1);
      };
      ok = __all_sync(0xffffffffu, ok);
      for (int j = 0; ok && j < min(2, nb); ++j) issue_s(j);
      for (int j = 0; ok && j < nb; ++j) {
        ok = mbar_wait_spin(bar(B_PFULL), j & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const uint64_t dr = dr0 + (j % kStages) * dstage;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f8_ts_w(tmem + TC_ACC, tmem + TC_P + 8 * kk, dr + 2 * kk, i8w, (j > 0 || kk > 0));
        if (j > 0 && group_ends(j - 1, nb, gpad)) issue_flush((j - 1 + gpad) / kGroup);
        mma_commit_w(bar(B_PVDONE));
        mma_commit_w(bar(B_KVEMPTY + j % kStages));
        if (j + 2 < nb) {
          ok = mbar_wait_spin(bar(B_SFREE + (j & 1)), (j >> 1) & 1, abort_flag, p.status);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          issue_s(j + 2);
        }
      }
      // the last group's mean product, after the softmax read its row sums
      if (ok) {
        ok = mbar_wait_spin(bar(B_PFULL), nb & 1, abort_flag, p.status);
        if (__all_sync(0xffffffffu, ok)) {
          tc_fence_after();
          issue_flush((nb - 1 + gpad) / kGroup);
          mma_commit_w(bar(B_PVDONE));
        }
      }
      // all issued MMAs complete before the CTA releases its tensor memory
      mma_commit_w(bar(B_DRAIN));
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar(B_DRAIN), 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int h = (warp - 4) / 4, quarter = warp % 4;
    const int row = quarter * 32 + lane;  // row within the query tile = TMEM lane
    const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
    const uint32_t tl = tmem + lanes;
    const uint32_t named = 1 + quarter;   // barrier of the two warps sharing these rows
    const float a_q = p.qk_scale * p.sq[(size_t)bh * nb + qt];
    const float* skp = p.sk + (size_t)bh * nb;
    const int valid_last = p.N - (nb - 1) * 128 - 64 * h;  // valid columns of this half, last block
    // [block parity][h][row]: the slot written in block j is not rewritten
    // before the partner has passed the barrier of block j + 1
    float* xch_base = reinterpret_cast<float*>(sm + OFF_XCH);
    float M = -INFINITY, l = 0.0f;
    float sk_next = __ldg(skp);
    bool ok = true;
    // After group g's last product: read its 8 row-sum slots (already rescaled
    // to the current maximum), add them to l, clear the bank (half 0) and
    // write the bf16 operand (half 0: hi, half 1: lo; slots 2c, 2c+1 in column
    // c, columns 4-7 = K 8..15 = 0).
    auto close_group = [&](int g) {
      const uint32_t bank = tl + TC_BANK + 8 * (g & 1);
      uint32_t v[8];
      tmem_ld8(bank, v);
      tmem_ld_wait();
      float rsum = 0.0f;
      uint32_t pk[8];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float r0 = __uint_as_float(v[2 * c]), r1 = __uint_as_float(v[2 * c + 1]);
        rsum += r0 + r1;
        uint16_t h0 = f32_to_bf16_bits(r0), h1 = f32_to_bf16_bits(r1);
        if (h) {
          h0 = f32_to_bf16_bits(r0 - bf16_bits_to_f32(h0));
          h1 = f32_to_bf16_bits(r1 - bf16_bits_to_f32(h1));
        }
        pk[c] = (uint32_t)h0 | ((uint32_t)h1 << 16);
      }
#pragma unroll
      for (int c = 4; c < 8; ++c) pk[c] = 0u;
      l += rsum;
      tmem_st8(tl + (h ? TC_GLO : TC_GHI), pk);
      // both halves have read the bank before half 0 clears it
      asm volatile("bar.sync %0, 64;" ::"r"(named) : "memory");
      if (h == 0) {
        uint32_t z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        tmem_st8(bank, z);
      }
    };
    for (int j = 0; j < nb; ++j) {
      const uint32_t sbuf = tl + TC_S + 128 * (j & 1);
      const float a = a_q * sk_next;
      if (j + 1 < nb) sk_next = __ldg(skp + j + 1);
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
          if (c >= valid_last) s[c] = 0xFF800000u;  // -inf: masked key -> byte 0
      }
      // partial row maximum (four chains), exchanged with the partner thread
      float m4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) m4[i] = fmaxf(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
#pragma unroll
      for (int c = 8; c < 64; c += 8)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          m4[i] = max3(m4[i], __uint_as_float(s[c + 2 * i]), __uint_as_float(s[c + 2 * i + 1]));
      float* xch = xch_base + (j & 1) * 256;
      xch[h * 128 + row] = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      asm volatile("bar.sync %0, 64;" ::"r"(named) : "memory");
      const float mx = fmaxf(xch[row], xch[128 + row]);
      const float Mn = fmaxf(M, a * mx);
      const float alpha = ex2((M - Mn) * 0.125f);  // 0 on the first block
      const float b = kExpCastBias - Mn;
      // this half's ExpCast bytes, four per 32-bit TMEM column (the A layout of
      // the product: byte k of column c is key 4c + k)
      uint32_t w[16];
      if (expcast_fast_is_exact(Mn)) {
        const float a128 = a * 0.0078125f, b128 = b * 0.0078125f;
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          const uint2 e0 = expcast_pair_bits(__uint_as_float(s[c]), __uint_as_float(s[c + 1]), a128, b128);
          const uint2 e1 = expcast_pair_bits(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]), a128, b128);
          w[c / 4] = __byte_perm(__byte_perm(e0.x, e0.y, 0x0040), __byte_perm(e1.x, e1.y, 0x0040), 0x5410);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; c += 4)
          w[c / 4] = expcast_code(__uint_as_float(s[c]), a, b) |
                     (expcast_code(__uint_as_float(s[c + 1]), a, b) << 8) |
                     (expcast_code(__uint_as_float(s[c + 2]), a, b) << 16) |
                     (expcast_code(__uint_as_float(s[c + 3]), a, b) << 24);
      }
      if (j > 0) {
        // the previous product read P^ and wrote the accumulator
        ok = mbar_wait(bar(B_PVDONE), (j - 1) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      tmem_st16(tl + TC_P + 16 * h, w);
      if (j > 0) {
        // correction: rescale this half of the accumulator row and this half's
        // row-sum bank when the running max rose
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
          uint32_t v8[8];
          tmem_ld8(tl + TC_BANK + 8 * h, v8);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 8; ++c) v8[c] = __float_as_uint(__uint_as_float(v8[c]) * alpha);
          tmem_st8(tl + TC_BANK + 8 * h, v8);
          tmem_st_wait();
          // both halves must finish rescaling before either reads a bank
          asm volatile("bar.sync %0, 64;" ::"r"(named) : "memory");
        }
        l *= alpha;
        if (group_ends(j - 1, nb, gpad)) close_group((j - 1 + gpad) / kGroup);
      }
      M = Mn;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL));
    }
    if (ok) {
      // the last group's row sums and mean product
      ok = mbar_wait(bar(B_PVDONE), (nb - 1) & 1, abort_flag, p.status);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        close_group((nb - 1 + gpad) / kGroup);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(B_PFULL));
        ok = mbar_wait(bar(B_PVDONE), nb & 1, abort_flag, p.status);
      } else {
        ok = false;
      }
    }
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int grow = qt * 128 + row;
      const float inv_l = 1.0f / l;
      uint16_t* orow = p.out + ((size_t)bh * p.N + grow) * 128 + 64 * h;
      const float* svh = s_sv + 64 * h;
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
              const float o0 = __uint_as_float(v[c + 2 * u]) * svh[c0 + c + 2 * u] * inv_l;
              const float o1 = __uint_as_float(v[c + 2 * u + 1]) * svh[c0 + c + 2 * u + 1] * inv_l;
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
  p.ngroups = (nb + kGroup - 1) / kGroup;
  p.gpad = p.ngroups * kGroup - nb;
  p.qk_scale = (float)(8.0 * 1.4426950408889634 / sqrt(128.0));
  if (cudaFuncSetAttribute(attn_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes) != cudaSuccess)
    return VCA_ERR_CUDA;
  const long long grid = (long long)BH * nb;
  if (grid > 0x7FFFFFFF) return VCA_ERR_UNSUPPORTED;
  attn_fp8_kernel<<<(unsigned)grid, kThreads, kSmemBytes, st>>>(tq, tk, tr, p);
  return cudaGetLastError() == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}

}  // namespace vca
