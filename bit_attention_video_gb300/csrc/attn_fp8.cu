// 8-bit VC-Attention forward (paper §3.1 Eq 1, §3.2 Eq 6, §3.3 Eq 7) on
// tcgen05 tensor cores.
//
// One CTA owns two 128-row query tiles (A and B) of one (batch, head) and
// streams all key blocks j of the permuted, centred keys K' and the
// transposed residual R^T through a TMA ring; both tiles consume each stage.
// Warp roles (12 warps):
//   warp 0        producer: TMA of the two Q tiles once; per stage K'_j, R^T_j
//                 and the 16 "slot" rows appended to R^T_j (written by the
//                 warp's lanes); the mean operand of each group of 8 blocks
//   warp 1        MMA issuer of the S products (alternating A, B) and TMEM
//                 owner; warp 2 MMA issuer of the PV products and the stage
//                 releases.  Warp-uniform loops, one elected lane issues,
//                 suspending waits.  An mbarrier test costs ~130 cycles even
//                 on a completed phase, so the two chains of waits run on
//                 two warps
//   warps 4-7     softmax + correction + epilogue of tile A, warps 8-11 of
//                 tile B: one thread per query row, which holds the row's 128
//                 scores in registers (so each SM sub-partition carries one
//                 softmax warp per tile beside the MMA or producer warp)
//
// Tensor memory (512 columns):
//   [0,128)    S = Q^ K'^T (fp32), one buffer shared by the two tiles: the
//              softmax releases it as soon as it has loaded its scores
//   per tile X at base 128 + 192 X:
//     [+0,+128)    the output accumulator A_X
//     [+128,+144)  two banks of 8 row-sum slots, part of the same accumulator
//     [+144,+176)  P^_X (ExpCast bytes, 4 per column): A operand of the product
//     [+176,+192)  a group's row-sum operand (bf16 hi, lo) of the mean product
// The MMA warp issues S_A(j+1) before PV_A(j) (P has its own columns), so a
// tile's next scores are ready when its softmax finishes a block, and the two
// tiles' softmaxes run concurrently, each handing the S buffer to the other.
//
// Per key block j and tile:
//   S   = Q^ K'^_j^T                              FP8 MMA (N=128)
//   M'  = max(M, a_j rowmax(S))                   exact running max (x8, log2)
//   c   = clip_[0,120](RNE(a_j S + 119.65 - M'))  ExpCast-FP8 bytes -> TMEM
//   A  *= alpha = 2^((M - M')/8) when M rises     (TMEM correction)
//   A  += P^ [R^_j ; E_j]                          FP8 MMA (N=144), A from TMEM
// E_j (16 rows of K=128) is zero except row 8*bank + slot of block j, which is
// all ones: column 128 + 8 bank + slot of the product is the row sum r_j of
// exactly the bytes the product consumes, at the maximum M_j of block j.
// Blocks form groups of 8 (aligned to the last block; only the first group can
// be partial) that alternate between the two banks; the correction rescales
// the banks with the accumulator.  After a group's last product the softmax
// reads its 8 slots (already at the current maximum), adds them to l, clears
// the bank and writes the slots as bf16 hi/lo to TMEM; three BF16 K=16 MMAs
// then add sum_g rho_g mutilde_g^T (Eq 6's mean term).
// Epilogue: O = sV (.) A / l in bf16, original query order (Q is not permuted).
//
// The same kernel with kExpCast = false writes the conventional bytes that
// ExpCast replaces, E4M3_RNE(2^((a S - M')/8 + 8)): the exponential on the
// MUFU, then the hardware E4M3 cast.  On a naive preparation this is the
// "Naive FP8" comparison kernel of §4.5 (Table 4); on a V-Smooth one, V-Smooth
// without ExpCast.
#include "common.cuh"
#include "expcast.cuh"
#include "prep.h"

namespace vca {
namespace {

constexpr int kStages = 5;
constexpr uint32_t kSlotRowsBytes = 16 * 128;                      // E_j: 16 rows x 128 keys
constexpr uint32_t kStageBytes = 2 * kTileBytes + kSlotRowsBytes;  // K'_j, R^T_j, E_j
constexpr uint32_t OFF_Q = 0;                                      // the two query tiles
constexpr uint32_t OFF_KV = 2 * kTileBytes;
constexpr uint32_t OFF_BG = OFF_KV + kStages * kStageBytes;    // mean operand, 2 buffers x 8 KB
constexpr uint32_t OFF_SV = OFF_BG + 2 * kGroupBytes;          // sV, 512 B
constexpr uint32_t OFF_BAR = OFF_SV + 512;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;  // + alignment slack
constexpr int kThreads = 384;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned");
static_assert(kGroup == 8, "eight row-sum slots per bank");

// TMEM columns
constexpr uint32_t TC_S = 0;
__device__ __forceinline__ uint32_t tc_acc(int X) { return 128u + 192u * X; }
__device__ __forceinline__ uint32_t tc_p(int X) { return tc_acc(X) + 144u; }
__device__ __forceinline__ uint32_t tc_ghi(int X) { return tc_acc(X) + 176u; }
__device__ __forceinline__ uint32_t tc_glo(int X) { return tc_acc(X) + 184u; }

struct Fp8Params {
  const float* sq;        // [BH][nb]
  const float* sk;        // [BH][nb]
  const float* sv;        // [BH][128]
  const uint8_t* mside;   // [BH][ngroups][8192]
  const uint32_t* hdr;
  uint16_t* out;          // [BH][N][128]
  int* status;
  int B, H, N, nb, Npad, ngroups, gpad, npairs;
  float qk_scale;         // 8 log2(e) / sqrt(128)
};

// barrier indices ([2]: per tile)
enum { B_QFULL = 0, B_KVFULL = 1, B_KVEMPTY = B_KVFULL + kStages, B_SFULL = B_KVEMPTY + kStages,
       B_SFREE = B_SFULL + 2, B_PFULL = B_SFREE + 2, B_PVDONE = B_PFULL + 2,
       B_DRAIN = B_PVDONE + 2, B_COUNT = B_DRAIN + 1 };

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
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
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

template <bool kExpCast>
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
  const int bh = blockIdx.x / p.npairs, qp = blockIdx.x % p.npairs;
  const bool has_b = 2 * qp + 1 < nb;   // the last pair of an odd nb has tile A only

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
    // "S read" and "P written": the 128 softmax threads of a tile; the
    // rest: one arrival or a tcgen05 commit
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
      mbar_expect_tx(bar(B_QFULL), (has_b ? 2 : 1) * kTileBytes);
      tma_load_2d(base + OFF_Q, &tmQ, bar(B_QFULL), 0, bh * p.Npad + 2 * qp * 128);
      if (has_b)
        tma_load_2d(base + OFF_Q + kTileBytes, &tmQ, bar(B_QFULL), 0, bh * p.Npad + (2 * qp + 1) * 128);
    }
    int issued = 0;
    for (int j = 0; j < nb; ++j) {
      const int s = j % kStages;
      if (j >= kStages)
        ok = mbar_wait(bar(B_KVEMPTY + s), ((j / kStages) - 1) & 1, abort_flag, p.status);
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
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // The whole warp runs this loop (uniform control flow, operands in
    // uniform registers); one elected lane issues each MMA and commit.
    // S issuer: S_A(0), S_B(0), S_A(1), S_B(1), ..., each after the other tile
    // loaded the shared S buffer.  PV issuer: PV_A(0), PV_B(0), PV_A(1), ...,
    // each after its tile wrote P; a PV follows its tile's use of the S
    // product that read the same stage, so its commit releases the stage.
    const uint32_t i8 = idesc_f8(128, 128), i8w = idesc_f8(128, 144), i16 = idesc_bf16(128, 128);
    const uint64_t dq0 = desc_k_sw128(base + OFF_Q);
    const uint64_t dqstep = kTileBytes >> 4;
    const uint64_t dk0 = desc_k_sw128(base + OFF_KV);                  // stage 0 K'
    const uint64_t dr0 = desc_k_sw128(base + OFF_KV + kTileBytes);     // stage 0 [R^; E]
    const uint64_t dstage = kStageBytes >> 4;                          // per-stage step
    const uint64_t dbg0 = desc_k_plain(base + OFF_BG, 128, 256);
    const uint64_t dgroup = kGroupBytes >> 4, dhalf = (kGroupBytes / 2) >> 4;
    bool ok = mbar_wait(bar(B_QFULL), 0, abort_flag, p.status);
    // S_X(j); tile B's S(j) reads the stage tile A's S(j) already waited for
    auto issue_s = [&](int X, int j, bool kv_ready = false) {
      const int s = j % kStages;
      if (X == 0 && !kv_ready) {
        ok = mbar_wait(bar(B_KVFULL + s), (j / kStages) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; return; }
      }
      tc_fence_after();
      const uint64_t dk = dk0 + s * dstage, dq = dq0 + X * dqstep;
      mma4_f8_ss_w(tmem + TC_S, dq, dk, i8, 0);
      mma_commit_w(bar(B_SFULL + X));
    };
    auto issue_pv = [&](int X, int j) {
      ok = mbar_wait(bar(B_PFULL + X), j & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; return; }
      tc_fence_after();
      const uint64_t dr = dr0 + (j % kStages) * dstage;
      mma4_f8_ts_w(tmem + tc_acc(X), tmem + tc_p(X), dr, i8w, j > 0);
      if (j > 0 && group_ends(j - 1, nb, gpad)) {
        // sum_g rho_g mutilde_g^T = rho_hi mu_hi + rho_lo mu_hi + rho_hi mu_lo
        const uint64_t bg = dbg0 + (((j - 1 + gpad) / kGroup) & 1) * dgroup;
        mma_f16_ts_w(tmem + tc_acc(X), tmem + tc_ghi(X), bg, i16, 1);
        mma_f16_ts_w(tmem + tc_acc(X), tmem + tc_glo(X), bg, i16, 1);
        mma_f16_ts_w(tmem + tc_acc(X), tmem + tc_ghi(X), bg + dhalf, i16, 1);
      }
      mma_commit_w(bar(B_PVDONE + X));
    };
    auto wait_sfree = [&](int X, int j) {
      ok = mbar_wait(bar(B_SFREE + X), j & 1, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
    };
    ok = __all_sync(0xffffffffu, ok);
    if (warp == 1) {
      // every S product, alternating A, B
      if (ok) issue_s(0, 0);
      if (ok && has_b) {
        wait_sfree(0, 0);
        if (ok) issue_s(1, 0);
      }
      for (int j = 0; ok && j + 1 < nb; ++j) {
        // the stage of block j+1 first (usually landed long before), so the
        // wait for the other tile is the last step before the product
        ok = mbar_wait(bar(B_KVFULL + (j + 1) % kStages), ((j + 1) / kStages) & 1, abort_flag,
                       p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        wait_sfree(has_b ? 1 : 0, j);
        if (!ok) break;
        issue_s(0, j + 1, true);
        if (!ok) break;
        if (has_b) {
          wait_sfree(0, j + 1);
          if (!ok) break;
          issue_s(1, j + 1);
        }
      }
    } else {
      // every PV product and the stage releases
      for (int j = 0; ok && j < nb; ++j) {
        issue_pv(0, j);
        if (!ok) break;
        if (has_b) issue_pv(1, j);
        if (!ok) break;
        mma_commit_w(bar(B_KVEMPTY + j % kStages));
      }
      for (int X = 0; ok && X < (has_b ? 2 : 1); ++X) {
        ok = mbar_wait(bar(B_PFULL + X), nb & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const uint64_t bg = dbg0 + (((nb - 1 + gpad) / kGroup) & 1) * dgroup;
        mma_f16_ts_w(tmem + tc_acc(X), tmem + tc_ghi(X), bg, i16, 1);
        mma_f16_ts_w(tmem + tc_acc(X), tmem + tc_glo(X), bg, i16, 1);
        mma_f16_ts_w(tmem + tc_acc(X), tmem + tc_ghi(X), bg + dhalf, i16, 1);
        mma_commit_w(bar(B_PVDONE + X));
      }
    }
    // all issued MMAs complete before the CTA releases its tensor memory
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
    const float a_q = p.qk_scale * p.sq[(size_t)bh * nb + qt];
    const float* skp = p.sk + (size_t)bh * nb;
    const int valid_last = p.N - (nb - 1) * 128;  // valid keys of the last block
    float M = -INFINITY, l = 0.0f;
    float sk_next = __ldg(skp);
    bool ok = true;
    // After group g's last product: read its 8 row-sum slots (already at the
    // current maximum), add them to l, clear the bank and write the bf16
    // operand (hi in the first 8 columns, lo in the next 8; slots 2c, 2c+1 in
    // column c, columns 4-7 = K 8..15 = 0).
    auto close_group = [&](int g) {
      const uint32_t bank = acc + 128 + 8 * (g & 1);
      uint32_t v[8];
      tmem_ld8(bank, v);
      tmem_ld_wait();
      float rsum = 0.0f;
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float r0 = __uint_as_float(v[2 * c]), r1 = __uint_as_float(v[2 * c + 1]);
        rsum += r0 + r1;
        const uint16_t h0 = f32_to_bf16_bits(r0), h1 = f32_to_bf16_bits(r1);
        const uint16_t l0 = f32_to_bf16_bits(r0 - bf16_bits_to_f32(h0));
        const uint16_t l1 = f32_to_bf16_bits(r1 - bf16_bits_to_f32(h1));
        pk[c] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        pk[8 + c] = (uint32_t)l0 | ((uint32_t)l1 << 16);
        pk[4 + c] = 0u;
        pk[12 + c] = 0u;
      }
      l += rsum;
      tmem_st16(tl + tc_ghi(X), pk);
      uint32_t z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      tmem_st8(bank, z);
    };
    for (int j = 0; j < nb; ++j) {
      const float a = a_q * sk_next;
      if (j + 1 < nb) sk_next = __ldg(skp + j + 1);
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
      if (j == nb - 1 && valid_last < 128) mask_tail128(s, valid_last);  // masked keys: byte 0
      bool has_nan;
      const float Mn = fmaxf(M, a * row_max128_flag(s, has_nan));
      const float alpha = ex2((M - Mn) * 0.125f);  // 0 on the first block
      // ExpCast bytes, four per 32-bit TMEM column (the A layout of the
      // product: byte k of column c is key 4c + k)
      uint32_t w[32];
      if constexpr (!kExpCast) {
        // x = (a S - M')/8 + 8 (one FMA; the /8 is exact), p = 2^x <= 256
        const float a8 = a * 0.125f, b8 = 8.0f - Mn * 0.125f;
#pragma unroll
        for (int c = 0; c < 128; c += 4) {
          const float p0 = ex2(fmaf(__uint_as_float(s[c]), a8, b8));
          const float p1 = ex2(fmaf(__uint_as_float(s[c + 1]), a8, b8));
          const float p2 = ex2(fmaf(__uint_as_float(s[c + 2]), a8, b8));
          const float p3 = ex2(fmaf(__uint_as_float(s[c + 3]), a8, b8));
          w[c / 4] = f32x4_to_e4m3x4(p0, p1, p2, p3);
        }
      } else {
        expcast_row_bytes(s, a, Mn, has_nan, w);
      }
      if (j > 0) {
        // the previous product read P^ and wrote the accumulator
        ok = mbar_wait(bar(B_PVDONE + X), (j - 1) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      tmem_st16(tl + tc_p(X), *reinterpret_cast<uint32_t(*)[16]>(&w[0]));
      tmem_st16(tl + tc_p(X) + 16, *reinterpret_cast<uint32_t(*)[16]>(&w[16]));
      if (j > 0) {
        // correction: rescale the accumulator row and both row-sum banks
        // when the running max rose
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
          uint32_t v16[16];
          tmem_ld16(acc + 128, v16);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) v16[c] = __float_as_uint(__uint_as_float(v16[c]) * alpha);
          tmem_st16(acc + 128, v16);
        }
        l *= alpha;
        if (group_ends(j - 1, nb, gpad)) close_group((j - 1 + gpad) / kGroup);
      }
      M = Mn;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + X));
    }
    if (ok) {
      // the last group's row sums and mean product
      ok = mbar_wait(bar(B_PVDONE + X), (nb - 1) & 1, abort_flag, p.status);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        close_group((nb - 1 + gpad) / kGroup);
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
      const float inv_l = 1.0f / l;
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
                         bool expcast, cudaStream_t st) {
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
  p.npairs = (nb + 1) / 2;
  p.qk_scale = (float)(8.0 * 1.4426950408889634 / sqrt(128.0));
  auto kernel = expcast ? attn_fp8_kernel<true> : attn_fp8_kernel<false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
      cudaSuccess)
    return VCA_ERR_CUDA;
  const long long grid = (long long)BH * p.npairs;
  if (grid > 0x7FFFFFFF) return VCA_ERR_UNSUPPORTED;
  kernel<<<(unsigned)grid, kThreads, kSmemBytes, st>>>(tq, tk, tr, p);
  return cudaGetLastError() == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}

}  // namespace vca
