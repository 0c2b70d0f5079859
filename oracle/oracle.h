/*
 * VC-Attention CPU oracle — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded C++17 restatement of what the VC-Attention
 * hot path computes ("VC-Attention: Value Smoothing and Softmax Casting for
 * Low-bit Attention", arXiv 2609.15810).  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or helper with the CUDA library, and never calls it.
 *
 * Precision: floating point is fp64 except where the method fixes a narrower
 * type (bf16 inputs, fp32 scales and means, E4M3/E2M1 codes), in which case
 * the fp32 step is written out with one IEEE rounding per operation
 * (the library is built with -ffp-contract=off so no FMA is formed silently).
 *
 * Parity status of each function is stated next to it.  "parity unpinned"
 * marks a function that no test ties to something other than itself.
 *
 * All arrays are caller-owned, contiguous, row-major.  bf16 values travel as
 * their uint16 bit patterns.  One call handles one (batch, head) unless stated.
 */
#ifndef VCA_ORACLE_H
#define VCA_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------- number formats (paper §3.3 "ExpCast-FP8", Appx A) ------- */
/* bf16 <-> fp32.  Encode is round-to-nearest-even.  Pinned against torch. */
float    orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16(float f);
/* E4M3 (bias 7, 3 mantissa bits, no inf, 0x7F/0xFF NaN): value of a byte and
 * round-to-nearest-even encode with saturation to +-448 (satfinite).
 * Pinned: format table, torch float8_e4m3fn for |x|<=448, midpoint ties. */
double   orc_e4m3_decode(uint8_t c);
uint8_t  orc_e4m3_encode(float x);
/* E2M1 (values 0,.5,1,1.5,2,3,4,6): 4-bit code in the low nibble, sign bit 3.
 * RNE with saturation to +-6.  Pinned: format table and midpoint ties. */
double   orc_e2m1_decode(uint8_t c);
uint8_t  orc_e2m1_encode(float x);
/* The same encoders over arrays. */
void     orc_e4m3_encode_array(const float* x, uint8_t* out, size_t n);
void     orc_e2m1_encode_array(const float* x, uint8_t* out, size_t n);

/* ---------------- ExpCast-FP8 (paper §3.3 Eq 7, Appx C/D) ----------------- */
/* Eq 7 literally, in fp64: c(u) = clip_[0,120](RNE(8(u+8)+56+beta)), beta=-0.35.
 * Pinned: worked example u=-1.60 -> 107 (value 88), 79.6% byte agreement over a
 * doubling, ratio range of Eq 11, TV bound of Eq 13. */
int      orc_expcast_code(double u);
/* The fp32 single-FMA form of Eq 7 that a kernel evaluates:
 * clip_[0,120](RNE(fmaf(a, acc, b))).  NaN maps to 0. */
int      orc_expcast_code_f32(float acc, float a, float b);
void     orc_expcast_f32_array(const float* acc, const float* a, const float* b,
                               uint8_t* out, size_t n);

/* ---------------- V-Smooth preprocessing, one (b,h) (paper §3.2, §3.4) ---- */
typedef struct {
  int N, d, k, iters, bits;   /* bits: 8 or 4 */
  int Bv;                     /* block rows, 128 in the method; tests may vary */
  uint64_t seed;
  int b, h, H;                /* position of this head, for the k-means seed */
} orc_head_cfg;

/* SplitMix64 (Steele, Lea & Flood 2014): the k-means initial indices.
 * Writes k distinct token indices.  Pinned by published SplitMix64 outputs. */
void orc_kmeans_init_indices(uint64_t seed, int b, int h, int H, int N, int k,
                             int32_t* idx_out);

/* k-means on the int8 grid of value features (paper §3.2 "Value-guided
 * permutation").  Outputs labels z[N] (last assignment), centroids[k*d] (after
 * the last update), grid scale.  Pinned: brute force on tiny inputs, k=1. */
void orc_kmeans(const uint16_t* v, const orc_head_cfg* cfg,
                int8_t* x_out /* N*d, may be NULL */, float* grid_scale_out,
                int32_t* labels_out, int8_t* centroids_out);

/* Warm-started k-means (paper §3.2, "Unbalanced clusters cost little": each
 * step starts from the previous step's centroids).  The previous centroids
 * (on the grid of scale prev_grid_scale) are moved to this head's grid at the
 * same value-space position, c = clamp(RNE(c_prev * (prev_grid_scale / s)),
 * -127, 127) with the ratio and the product rounded to fp32, then cfg->iters
 * Lloyd iterations run as in orc_kmeans.  With cfg->iters = 0 the outputs are
 * the moved centroids (labels untouched).  Pinned: exact halving when the
 * grid doubles, fixed point of a converged run, brute-force assignment. */
void orc_kmeans_warm(const uint16_t* v, const orc_head_cfg* cfg, const int8_t* prev_centroids,
                     float prev_grid_scale, int8_t* x_out /* may be NULL */,
                     float* grid_scale_out, int32_t* labels_out, int8_t* centroids_out);

/* The QK Hadamard rotation (paper Appx B; §4.1 "Baselines", the fused QK
 * Hadamard transform): y = x H / sqrt(128) for one 128-channel row, H the
 * Sylvester-Hadamard matrix, computed as the fast transform (butterflies with
 * stride 1, 2, ..., 64 in fp32, then an fp32 multiply by fp32(1/sqrt(128))).
 * y may alias x.  Pinned: scipy's Hadamard matrix in fp64, exact integer
 * inputs, orthogonality (QK^T unchanged). */
void orc_hadamard128(const float* x, float* y);

/* Stable counting sort of labels: perm[i] = source token of permuted row i. */
void orc_stable_argsort(const int32_t* labels, int N, int k, int32_t* perm_out);

/* Block demeaning of already-permuted rows (paper Eq 4) in fp32 with the
 * pairwise tree: mu[nb*d] (bf16 bits), R[Npad*d] (fp32, zero padding rows).
 * Bv is a parameter so the toy example of the pages (Bv=2) can pin it. */
void orc_block_demean(const uint16_t* vperm, int N, int d, int Bv,
                      uint16_t* mu_out, float* r_out);

/* Full 8-bit preparation of one head.  Output layouts:
 *   qhat [Npad*d] e4m3, sq [nb]; khat [Npad*d] e4m3 (permuted, centred),
 *   sk [nb], kbar [d] bf16; rhatT [d*Npad] e4m3, sv [d], mu [nb*d] bf16,
 *   mutilde [nb*d] fp32 (= mu / sv). */
typedef struct {
  int32_t* labels; int32_t* perm; int8_t* centroids; float* grid_scale;
  uint8_t* qhat; float* sq;
  uint8_t* khat; float* sk; uint16_t* kbar;
  uint8_t* rhatT; float* sv; uint16_t* mu; float* mutilde;
} orc_prep8_out;
void orc_prepare8(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                  const orc_head_cfg* cfg, const int32_t* perm_in /* NULL: run k-means */,
                  orc_prep8_out* out);

/* Full 4-bit (NVFP4) preparation of one head.  Codes are one E2M1 code per
 * byte (unpacked, for readability); block scales are UE4M3 bytes.
 *   q4 [Npad*d], q4s [Npad*d/16], gq; k4 [Npad*d], k4s [Npad*d/16], gk, kbar;
 *   r4T [d*Npad] (blocks of 16 along tokens), r4s [d*Npad/16], gr;
 *   mu [nb*d] bf16 (unscaled). */
typedef struct {
  int32_t* labels; int32_t* perm; int8_t* centroids; float* grid_scale;
  uint8_t* q4; uint8_t* q4s; float* gq;
  uint8_t* k4; uint8_t* k4s; float* gk; uint16_t* kbar;
  uint8_t* r4T; uint8_t* r4s; float* gr; uint16_t* mu;
} orc_prep4_out;
void orc_prepare4(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                  const orc_head_cfg* cfg, const int32_t* perm_in, orc_prep4_out* out);

/* The same preparations for the steps after the grouping window (paper §3.4
 * "Amortized grouping schedule": the plain low-bit kernel on the permutation
 * the window left behind): the given permutation (required), no block
 * demeaning, so every mean is zero and the value operand is V[pi] itself.
 * Pinned: zero means, value codes restated with torch casts, attention
 * equal to plain quantised attention without a mean term. */
void orc_prepare8_plain(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const orc_head_cfg* cfg, const int32_t* perm, orc_prep8_out* out);

/* The naive 8-bit preparation the pages compare against (§4.1 "Baselines":
 * an 8-bit kernel that rounds each operand to the nearest code per block and
 * smooths neither; §4.5 Table 4 "Naive FP8"): sequence order (pi = identity,
 * no grouping: labels, centroids and grid scale untouched), no key centring
 * (kbar = 0), no block demeaning (mu = 0); Q and K per 128-token block, V per
 * channel, all E4M3.  Pinned: codes restated with torch casts. */
void orc_prepare8_naive(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const orc_head_cfg* cfg, orc_prep8_out* out);

/* The preparations with the QK Hadamard rotation fused into the Q and K
 * quantisers (paper Appx B: Q fuses the rotation and quantisation; K fuses the
 * gather, the rotation, the mean subtraction and quantisation): every row of
 * Q and of K' = K[pi] - kbar is rotated by orc_hadamard128 before its scale
 * and codes are taken.  QK^T is unchanged in exact arithmetic; V is untouched.
 * Pinned: the codes restated from the rotated rows with torch casts. */
/* Every preparation above through one call: opts = ORC_PLAIN (no demeaning,
 * needs perm_in), ORC_NAIVE (sequence order, no smoothing; perm_in unused),
 * ORC_HADAMARD (the QK rotation), combinable. */
#define ORC_PLAIN 1u
#define ORC_NAIVE 2u
#define ORC_HADAMARD 4u
void orc_prepare8_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const orc_head_cfg* cfg, const int32_t* perm_in, unsigned opts,
                     orc_prep8_out* out);
void orc_prepare4_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const orc_head_cfg* cfg, const int32_t* perm_in, unsigned opts,
                     orc_prep4_out* out);
void orc_prepare8_hadamard(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const orc_head_cfg* cfg, const int32_t* perm_in, orc_prep8_out* out);
void orc_prepare4_hadamard(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const orc_head_cfg* cfg, const int32_t* perm_in, orc_prep4_out* out);
void orc_prepare4_plain(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const orc_head_cfg* cfg, const int32_t* perm, orc_prep4_out* out);

/* ---------------- attention (paper §3.1 Eq 1, §3.2 Eq 6, §3.3 Eq 7) ------- */
/* Exact softmax(QK^T/sqrt d)V in fp64 on the bf16 inputs of one head, for the
 * listed query rows.  out[nrows*d] fp64.  Pinned against numpy softmax. */
void orc_attention_exact(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         int N, int d, const int32_t* rows, int nrows, double* out);

/* The Eq 1 / Eq 6 recurrence on generic fp64 operands, for pins:
 *   keys kp[N*d], residual values r[N*d], block means mu[nb*d] (Bv rows),
 *   pmode 0: exact exp, 1: ExpCast-FP8 bytes (Eq 7), 2: the conventional
 *   bytes ExpCast replaces, E4M3_RNE(2^(u + 8)) (§3.3); relative to the running
 *   max over Bv-key tiles.  out[nrows*d].  With pmode 0 and r = V'-1mu^T it must
 *   equal exact attention (mean restoration, Eq 6). */
void orc_attention_recurrence(const double* q, const double* kp, const double* r,
                              const double* mu, int N, int d, int Bv, int pmode,
                              const int32_t* rows, int nrows, double* out);

/* 8-bit VC-Attention output for the listed query rows of one prepared head
 * (ExpCast-FP8 probabilities, E4M3 residual, online mean restoration).
 * out[nrows*d] bf16 bits.  Also returns the fp64 values before bf16 rounding
 * in out64 if non-NULL.  Compared with the GPU by relative L2. */
void orc_attention8(const orc_prep8_out* prep, int N, int d,
                    const int32_t* rows, int nrows, uint16_t* out, double* out64);

/* The same with the conventional probability bytes, E4M3_RNE(2^(u + 8)): the
 * exponential then the cast that ExpCast-FP8 replaces (§3.3; the "Naive FP8"
 * kernel of §4.5 Table 4 on a naive preparation, V-Smooth without ExpCast on a
 * V-Smooth one).  Pinned: the recurrence (pmode 2) on the dequantised
 * operands; the recurrence's bytes against torch's exp-then-cast. */
void orc_attention8_exp(const orc_prep8_out* prep, int N, int d,
                        const int32_t* rows, int nrows, uint16_t* out, double* out64);

/* 4-bit variant: NVFP4 operands, conventional exp, NVFP4 P, means unscaled.
 * Pinned: the value path with flat scores; one pass over all keys at the
 * row maximum when key block 0 holds it; and the unrolled recurrence
 * (each block quantised at its prefix maximum, weighted by 2^(m_j - M)) on
 * general inputs, with the formats restated from their definitions. */
void orc_attention4(const orc_prep4_out* prep, int N, int d,
                    const int32_t* rows, int nrows, uint16_t* out, double* out64);

#ifdef __cplusplus
}
#endif
#endif
