/*
 * vca.h — C ABI of the VC-Attention library for GB300 (sm_103a).
 *
 * VC-Attention ("VC-Attention: Value Smoothing and Softmax Casting for
 * Low-bit Attention", arXiv 2609.15810) computes non-causal attention
 * O = softmax(Q K^T / sqrt(d)) V with low-bit operands:
 *   - V-Smooth (§3.2): per (batch, head) a k-means over value tokens gives
 *     labels z and the stable permutation pi = argsort(z) (Eq 3); keys and
 *     values are gathered by pi, each 128-row block mean mu_j is subtracted
 *     (Eq 4) and only the residual is quantised.  Q and K are quantised to
 *     E4M3 with one scale per 128-token block.
 *   - The fused attention (§3.3, Eq 1, Eq 6, Eq 7): FP8 QK^T and PV on the
 *     tensor cores, ExpCast-FP8 probability bytes, online mean restoration.
 *
 * Conventions for every function below
 *   - Tensors Q, K, V, O are bf16, shape [B, H, N, d], contiguous row-major,
 *     d fastest.  Device pointers must be 16-byte aligned.
 *   - All device memory is caller-owned.  The library never allocates, frees
 *     or synchronises, except vca_get_status, which synchronises `stream`, and
 *     the host-buffer pipeline (vca_pipeline_*), which owns its streams and
 *     events and blocks in vca_pipeline_wait / _flush.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Argument errors are returned synchronously, before any
 *     launch; a launch failure returns VCA_ERR_CUDA.  Data-dependent failures
 *     (a cached permutation that does not match, a device-side wait that
 *     expired) are recorded in the state blob's status word and reported by
 *     vca_get_status.
 *   - d must be 128.  1 <= k_clusters <= min(N, 256).  N >= 1.
 */
#ifndef VCA_H
#define VCA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* vca_stream_t; /* same type as cudaStream_t */

typedef enum {
  VCA_OK = 0,
  VCA_ERR_INVALID_ARG = -1,      /* null pointer, bad shape, misaligned pointer */
  VCA_ERR_UNSUPPORTED = -2,      /* d != 128, bits not 8 or 4, k out of range */
  VCA_ERR_CUDA = -3,             /* a CUDA call or launch failed */
  VCA_ERR_BUFFER_TOO_SMALL = -4, /* state_bytes < vca_state_bytes(...) */
  VCA_ERR_NO_CACHED_PERM = -5,   /* reuse_perm=1 but the blob holds no matching permutation */
  VCA_ERR_TIMEOUT = -6,          /* a device-side pipeline wait gave up (no hang) */
  VCA_ERR_STATE_MISMATCH = -7    /* the blob was prepared for another shape or bit width */
} vca_status;

#define VCA_DEFAULT_ITERS 10
#define VCA_DEFAULT_SEED 0ull
/* reuse_perm modes of vca_vsmooth_prepare */
#define VCA_PERM_FRESH 0
#define VCA_PERM_REUSE 1
#define VCA_PERM_WARM 2
#define VCA_PERM_PLAIN 3
#define VCA_PERM_NAIVE 4
#define VCA_BLOCK_ROWS 128 /* B_v: the hardware block of the block means (paper §3.2, Eq 4) */

/* Offsets (bytes from the start of the state blob) of every array the
 * preparation writes, for inspection and tests.  nb = ceil(N/128) blocks,
 * Npad = 128*nb, BH = B*H.  An offset of 0 means "absent for this bit width". */
typedef struct {
  uint64_t total_bytes;
  uint64_t header;    /* 256 B: shape, bit width, flags */
  uint64_t status;    /* int32 status word (device side) */
  uint64_t labels;    /* int32 [BH][N]  k-means label z of each token (last assignment) */
  uint64_t perm;      /* int32 [BH][N]  pi: permuted row i holds source token perm[i] */
  uint64_t centroids; /* int8  [BH][k][d] centroids on the int8 feature grid */
  uint64_t grid;      /* fp32  [BH] per-head feature grid scale (and scratch) */
  uint64_t features;  /* fp16 (k <= 128) or int8 [BH][N][d] k-means features (scratch) */
  uint64_t sums;      /* int32 [BH][k][d] + counts int32 [BH][k] (scratch) */
  uint64_t qhat;      /* e4m3  [BH][Npad][d] */
  uint64_t sq;        /* fp32  [BH][nb]    Q block scales */
  uint64_t khat;      /* e4m3  [BH][Npad][d] permuted, centred keys */
  uint64_t sk;        /* fp32  [BH][nb]    K' block scales */
  uint64_t kbar;      /* bf16  [BH][d]     key channel mean */
  uint64_t ksum;      /* fp32  [BH][nb][d] per-block key sums (scratch) */
  uint64_t rhatT;     /* e4m3  [BH][d][Npad] residual codes, tokens fastest */
  uint64_t sv;        /* fp32  [BH][d]     per-channel residual scales */
  uint64_t mu;        /* bf16  [BH][nb][d] block means (unscaled) */
  uint64_t mutilde;   /* fp32  [BH][nb][d] mu / sv */
  uint64_t mside;     /* bf16 mean operand of the restoration MMA: 8-bit
                       * [BH][ceil(nb/8)][2][128*16]; 4-bit [BH][ceil(nb/4)][128*16] */
  uint64_t vamax;     /* fp32  [BH][nb][d] per-block residual channel maxima (scratch) */
  /* 4-bit (NVFP4) path.  E2M1 codes are packed two per byte, element 2i in the
   * low nibble.  Scale tiles (UE4M3, one per 16 elements along the product's
   * reduction dimension) cover 128 rows x 8 blocks in 1024 bytes: the scale
   * of row m, block kb sits at (kb/4)*512 + (m%32)*16 + (m/32)*4 + kb%4, the
   * order the tensor core reads scale factors in. */
  uint64_t q4;        /* e2m1 packed [BH][Npad][d/2] */
  uint64_t q4s;       /* ue4m3 [BH][nb][1024] scale tile per 128 query rows (blocks along d) */
  uint64_t k4;        /* e2m1 packed [BH][Npad][d/2] permuted, centred keys */
  uint64_t kr4s;      /* ue4m3 [BH][nb][2][1024] per key block: the K' scale tile (rows =
                       * keys, blocks along d), then the R scale tile (rows = channels,
                       * blocks of 16 tokens) */
  uint64_t r4T;       /* e2m1 packed [BH][d][Npad/2] residual codes, tokens fastest */
  uint64_t g4;        /* fp32 [BH][4] global scales gq, gk, gr, 0 */
} vca_state_layout;

/* Size in bytes of the state blob for this problem (0 if the arguments are
 * invalid or unsupported: d != 128, bits not 8 or 4, k outside 1..min(256, N),
 * B*H > 65535, N > 2^24, or B*H*Npad >= 2^31).  The caller allocates it (any device allocation,
 * 256-byte aligned). */
size_t vca_state_bytes(int B, int H, int N, int d, int k_clusters, int bits);

/* Fill `out` with the offsets of the state blob's arrays.  Returns VCA_OK or
 * an argument error. */
int vca_state_layout_get(int B, int H, int N, int d, int k_clusters, int bits,
                         vca_state_layout* out);

/* V-Smooth preprocessing (paper §3.2 Eq 3-4, §3.4 "Fused preprocessing",
 * Appx B).  Reads q, k, v (bf16 [B,H,N,d], device) and writes every operand of
 * the attention kernels into `state` (device, state_bytes >= vca_state_bytes).
 *   k_clusters  k-means clusters per (b, h)
 *   reuse_perm  VCA_PERM_FRESH (0): run k-means (iters Lloyd iterations,
 *               seeded by `seed`) and cache pi, the centroids and the feature
 *               grid scale in the blob;
 *               VCA_PERM_REUSE (1): skip grouping and reuse the cached pi
 *               (paper §3.4 "Amortized grouping schedule");
 *               VCA_PERM_WARM (2): run iters Lloyd iterations started from
 *               the cached centroids (paper §3.2 "Unbalanced clusters cost
 *               little": warm-starting each step from the previous step's
 *               centroids), moved to this call's feature grid at the same
 *               value-space position, c = clamp(RNE(c * (s_cached / s)),
 *               -127, 127) in fp32; `seed` is unused; the new pi, centroids
 *               and scale replace the cached ones;
 *               VCA_PERM_PLAIN (3): a step after the grouping window (paper
 *               §3.4: the remaining steps run the plain low-bit kernel on the
 *               permutation the window left behind): the cached pi, no block
 *               demeaning, so every mean is 0 and the value operand is V[pi]
 *               quantised per channel; the attention calls are unchanged;
 *               VCA_PERM_NAIVE (4): the naive comparison preparation (paper
 *               §4.1 "Baselines", §4.5 Table 4 "Naive FP8"): sequence order
 *               (pi = identity, no grouping), no key centring, no block
 *               demeaning; Q and K per block and V per channel as usual.  It
 *               leaves no grouping behind for modes 1-3.
 *               Modes 1-3 need a blob grouped by a call with the same
 *               B, H, N, d, k_clusters and bits, else the status word gets
 *               VCA_ERR_NO_CACHED_PERM and no operand is written.
 *   bits        8 (E4M3 path) or 4 (NVFP4 path)
 *   iters       >= 1 Lloyd iterations (VCA_DEFAULT_ITERS)
 *   seed        k-means seed (VCA_DEFAULT_SEED); the initial centroids of head
 *               (b,h) are k distinct tokens drawn by SplitMix64 from the state
 *               seed ^ (0x9E3779B97F4A7C15 * (b*H + h + 1)).
 * Clears the status word unless reuse fails. */
int vca_vsmooth_prepare(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                        int k_clusters, int reuse_perm, int bits, int iters, uint64_t seed,
                        void* state, size_t state_bytes, vca_stream_t stream);

/* Options of vca_vsmooth_prepare_ex. */
/* The QK Hadamard rotation (paper Appx B: the Q kernel fuses the rotation
 * before quantisation; the K kernel fuses it after the gather and before the
 * mean subtraction is quantised): every row of Q and of K' = K[pi] - kbar is
 * multiplied by H / sqrt(128) (H the 128 x 128 Sylvester-Hadamard matrix)
 * before its block scale and codes are taken, so QK^T is unchanged in exact
 * arithmetic.  The rotation is the fast transform in fp32: butterflies
 * (a, b) -> (a + b, a - b) on channel pairs (i, i + s), i & s = 0, for
 * s = 1, 2, ..., 64 in that order, then one multiply by fp32(1/sqrt(128)).
 * The attention calls are unchanged; V is not rotated. */
#define VCA_PREP_QK_HADAMARD 1u

/* vca_vsmooth_prepare with options: flags is 0 or VCA_PREP_QK_HADAMARD (any
 * other bit: VCA_ERR_INVALID_ARG).  vca_vsmooth_prepare is this call with
 * flags = 0; every other argument is the same. */
int vca_vsmooth_prepare_ex(const void* q, const void* k, const void* v, int B, int H, int N,
                           int d, int k_clusters, int reuse_perm, int bits, int iters,
                           uint64_t seed, unsigned flags, void* state, size_t state_bytes,
                           vca_stream_t stream);

/* 8-bit fused attention (paper §3.1 Eq 1, §3.2 Eq 6, §3.3 Eq 7): FP8 QK'^T
 * and P R on tcgen05 tensor cores, ExpCast-FP8 probability bytes relative to
 * the running row maximum, block means restored from the row sums in the same
 * accumulator.  `state` must hold a bits=8 preparation of the same shape.
 * Writes o (bf16 [B,H,N,d], device) in the original query order. */
int vca_attention_fp8(void* state, size_t state_bytes, int B, int H, int N, int d, void* o,
                      vca_stream_t stream);

/* The same product with the conventional probability bytes that ExpCast-FP8
 * replaces (paper §3.3): E4M3_RNE(2^(u + 8)) from the fp32 exponential (MUFU)
 * and the hardware E4M3 cast, u the log2-domain score minus the running row
 * maximum.  On a VCA_PERM_NAIVE preparation this is the "Naive FP8" kernel the
 * pages compare against (§4.5 Table 4); on a V-Smooth preparation it is
 * V-Smooth without ExpCast.  Same arguments, layout and errors as
 * vca_attention_fp8. */
int vca_attention_fp8_exp(void* state, size_t state_bytes, int B, int H, int N, int d, void* o,
                          vca_stream_t stream);

/* 4-bit variant (paper §4.1 "Implementation", Appx A, Appx B): NVFP4 Q, K'
 * and residual with E4M3 scales per 16 elements along each product's
 * reduction dimension, conventional exponential, NVFP4 probabilities, means
 * added unscaled.  `state` must hold a bits=4 preparation. */
int vca_attention_nvfp4(void* state, size_t state_bytes, int B, int H, int N, int d, void* o,
                        vca_stream_t stream);

/* BF16 reference attention on tcgen05 (the role BF16 FlashAttention-4 plays in
 * paper §4.1 "Baselines"): exact-max online softmax with an fp32 exponential,
 * bf16 probabilities.  q, k, v, o bf16 [B,H,N,d], device, 16-byte aligned;
 * d = 128, B*H <= 65535, N <= 2^24 (else VCA_ERR_UNSUPPORTED).  `status` is a
 * device int32 that receives kernel-side failures (may be NULL). */
int vca_attention_bf16_ref(const void* q, const void* k, const void* v, int B, int H, int N,
                           int d, void* o, int* status, vca_stream_t stream);

/* Synchronise `stream`, then read and clear the status word of `state`
 * (or of the int32 at `status_word` when state is NULL; or, when both are
 * NULL, the status word of vca_kmeans_permutation_noalloc's scratch on the
 * current device, VCA_OK if that call has not run there).  Returns VCA_OK or
 * the first recorded error. */
int vca_get_status(void* state, int* status_word, vca_stream_t stream);

/* Human-readable name of a vca_status value. */
const char* vca_status_string(int status);

/* Largest N accepted by vca_kmeans_permutation_noalloc. */
#define VCA_NOALLOC_MAX_TOKENS 32768

/* The grouping step (k-means labels and the stable permutation) for one
 * (batch, head) of V, for callers that cannot allocate device memory: code
 * whose device memory is handed out by a host framework's own pool, or loops
 * that must not pay cudaMalloc's implicit synchronisation.  This entry point
 * has no counterpart in the paper; it computes exactly what
 * vca_vsmooth_prepare stores as `labels` and `perm` for head (b, h) of an
 * H-head problem (same seed rule), without a state blob.
 *   v       bf16 [N, 128] device pointer (16-byte aligned), one head
 *   labels  int32 [N] device output, perm int32 [N] device output (each at
 *           least N entries: the kernels write N of each)
 *   N <= VCA_NOALLOC_MAX_TOKENS, else VCA_ERR_UNSUPPORTED (nothing launched).
 * Its scratch (about 4.3 MB) is a fixed array inside this library's device
 * image; every GPU that loads the library holds it until the process exits.
 * It allocates and frees nothing.  The first call on a device looks up the
 * array's device address once (cudaGetSymbolAddress), so make that first
 * call before capturing any stream.  All calls share the one array: calls
 * whose execution overlaps on the GPU (other streams, other host threads)
 * race and must be serialised by the caller.
 * Device-side failures (for example, k distinct initial tokens that cannot be
 * drawn) are recorded in a status word at the start of the array, which each
 * call clears first; the call's later kernels then skip their work and labels
 * and perm keep stale contents.  vca_get_status(NULL, NULL, stream) reads and
 * clears that word on the current device. */
int vca_kmeans_permutation_noalloc(const void* v, int N, int d, int k_clusters, int iters,
                                   uint64_t seed, int b, int h, int H, int32_t* labels,
                                   int32_t* perm, vca_stream_t stream);

/* ---- host-buffer pipeline: the end-to-end call of a serving loop ----
 *
 * Host-memory plumbing around the paper's operation (no counterpart in the
 * paper): one call per denoising step of a video model's attention layer.
 * Each step takes Q, K, V from host memory and returns O to host memory:
 *   Q, K, V (host) -> the step's staging slot (device)    the pipeline's H2D stream
 *   vca_vsmooth_prepare_ex, then vca_attention_fp8 (bits 8) or
 *   vca_attention_nvfp4 (bits 4) on the slot             `stream`
 *   O (slot) -> o_host                                    the pipeline's D2H stream
 * Step i uses slot i % slots.  Its input copies start once step i - slots has
 * finished reading that slot, and its compute once they have landed and step
 * i - slots's O has been read back.  Copies of later steps and read-backs of
 * earlier ones therefore overlap the compute.  With slots >= 3 a copy that
 * stalls is absorbed by the compute of the steps in between.  Page-locked host
 * memory that sat idle for a while can make the first large copy after the
 * pause several times slower.  All steps share one state blob, and the compute
 * runs them in submission order, so a reuse_perm step sees the grouping of the
 * step before it.
 *
 * Memory and resources: `workspace` (device, caller-owned, 256-byte aligned,
 * at least vca_pipeline_workspace_bytes(...)) holds the state blob, then
 * `slots` staging sets of Q, K, V and O.  vca_pipeline_create allocates the
 * pipeline object (host memory), two non-blocking CUDA streams and 3 x slots
 * events; vca_pipeline_destroy releases them.  These are the only resources
 * this library creates, and vca_pipeline_wait / vca_pipeline_flush are the
 * only calls besides vca_get_status that block the host.
 * Host buffers (bf16 [B,H,N,d] each) should be page-locked; pageable memory
 * works, but its copies do not overlap.  The step's q/k/v_host must stay
 * unchanged, and o_host unread, until vca_pipeline_wait(step) (or
 * vca_pipeline_flush) has returned.
 * Errors: argument errors are returned before anything is enqueued; a failed
 * CUDA call returns VCA_ERR_CUDA; device-side failures go to the state blob's
 * status word, which vca_pipeline_flush reads and clears (vca_get_status
 * semantics).
 * Threads: a pipeline object is not thread-safe; one host thread at a time
 * calls submit, wait and flush on it.  Separate pipelines (separate
 * workspaces) may run from separate threads. */
typedef struct vca_pipeline vca_pipeline;

#define VCA_PIPELINE_MAX_SLOTS 8

/* Workspace bytes for a pipeline of this shape: the state blob rounded up to
 * 256 bytes, plus `slots` (1..VCA_PIPELINE_MAX_SLOTS) x 4 tensors of
 * B*H*N*d*2 bytes, each rounded up to 256.  0 for an invalid shape. */
size_t vca_pipeline_workspace_bytes(int B, int H, int N, int d, int k_clusters, int bits,
                                    int slots);

/* Create a pipeline over `workspace`.  `stream` carries the compute. */
int vca_pipeline_create(int B, int H, int N, int d, int k_clusters, int bits, int slots,
                        void* workspace, size_t workspace_bytes, vca_stream_t stream,
                        vca_pipeline** out);

/* Option bit of vca_pipeline_submit's flags: run vca_attention_fp8_exp (the
 * conventional exp-then-cast probability bytes) instead of vca_attention_fp8.
 * Only for bits = 8. */
#define VCA_PIPELINE_FP8_EXP 0x100u

/* Enqueue one step.  reuse_perm, iters and seed as for vca_vsmooth_prepare_ex;
 * flags is VCA_PREP_QK_HADAMARD and/or VCA_PIPELINE_FP8_EXP.  On success *step
 * (may be NULL) receives the step number, 0, 1, 2, ... in submission order.
 * Does not block on the GPU, except when a CUDA call fails after the step's
 * copies were enqueued: then it waits for the pipeline's streams before
 * returning the error, so the host buffers are free to reuse at once and the
 * step's slot holds no work in flight (the step is not counted). */
int vca_pipeline_submit(vca_pipeline* p, const void* q_host, const void* k_host,
                        const void* v_host, void* o_host, int reuse_perm, int iters,
                        uint64_t seed, unsigned flags, int64_t* step);

/* Block until step `step` (< the number of submitted steps) has written
 * o_host.  This implies its inputs were read. */
int vca_pipeline_wait(vca_pipeline* p, int64_t step);

/* Block until every submitted step has finished, then read and clear the
 * status word of the state blob. */
int vca_pipeline_flush(vca_pipeline* p);

/* The state blob inside the workspace (device pointer), e.g. for inspection
 * of the last step's preparation once flushed. */
void* vca_pipeline_state(vca_pipeline* p);

/* Wait for the pipeline's work, then release its streams, events and the
 * pipeline object (not the workspace).  NULL is accepted. */
int vca_pipeline_destroy(vca_pipeline* p);

/* ---- test entry points (device buffers) ---- */

/* ExpCast-FP8 device function on n inputs: out[i] = clip_[0,120](RNE(fma(a[i],
 * acc[i], b[i]))) (paper §3.3 Eq 7 in the single-FMA form). */
int vca_debug_expcast(const float* acc, const float* a, const float* b, uint8_t* out, size_t n,
                      vca_stream_t stream);

/* The per-row byte step of vca_attention_fp8's softmax, through the same
 * device code (paper §3.3 Eq 7 and the running maximum of Eq 1): for each of
 * `rows` rows of 128 fp32 scores s (raw QK^T accumulators, row-major), keys
 * at and past valid[r] (1..128) are masked to -inf, Mn[r] = max(M[r],
 * a[r] * max_c s[r][c]) (NaN scores ignored), and codes[r][c] is the ExpCast
 * byte clip_[0,120](RNE(fma(a[r], s[r][c], 119.65f - Mn[r]))), evaluated in
 * the kernel's paired form (FMA, a multiply by 2^-149 that rounds onto the
 * subnormal grid, a saturating byte pack) where that is exact and in the
 * single-FMA form otherwise.  a[r] >= 0 as in the kernel (a product of
 * positive scales).  codes: device, 16-byte aligned, rows x 128 bytes. */
int vca_debug_expcast_rows(const float* s, const float* a, const float* M, const int* valid,
                           uint8_t* codes, float* Mn, size_t rows, vca_stream_t stream);

/* The failure path of the kernels' bounded waits, without a fault: one CTA
 * whose barriers are never arrived at.  Its first warp waits with a limit of
 * limit_ns (1 ns .. 100 ms; mode 0 the suspending wait, mode 1 the spinning
 * wait of the MMA issuers, mode 2 the polled wait of the 4-bit S issuer), then
 * records VCA_ERR_TIMEOUT's bit in the device
 * int32 *status and raises the CTA's abort flag; its second warp waits with
 * the kernels' own one-second limit and leaves through that flag.  out
 * (device, 4 x uint64): per warp 1 if its wait gave up, then per warp the
 * nanoseconds it waited.  vca_get_status(NULL, status, stream) then returns
 * VCA_ERR_TIMEOUT. */
int vca_debug_wait_timeout(int mode, uint64_t limit_ns, int* status, uint64_t* out,
                           vca_stream_t stream);

/* The device E4M3 and E2M1 encoders on n fp32 inputs (out_e2m1: one code per
 * byte, low nibble). */
int vca_debug_encode(const float* x, uint8_t* out_e4m3, uint8_t* out_e2m1, size_t n,
                     vca_stream_t stream);

/* One 128 x N tcgen05 product with the operand layouts the kernels use, for
 * layout tests.  mode: 0 FP8 K-major 128B-swizzle (K=128); 1 BF16 K-major
 * 128B-swizzle (K=128); 2 BF16 with B MN-major 128B-swizzle (K=64);
 * 3 BF16 K-major no-swizzle (K=16); 4 BF16 with A in tensor memory (K=128);
 * 5 FP8 with A in tensor memory (K=128); 6 mode 0 followed by mode 3 into the
 * same accumulator; 7 NVFP4 block-scaled (K=128, 64-byte swizzle, scale
 * factors copied to tensor memory).  a: [128][K] row-major (bytes per element
 * as the mode's type; for mode 6, a holds the 128x128 FP8 A then the 128x16
 * BF16 A; for mode 7, [128][64] packed E2M1 bytes, element 2i in the low
 * nibble, then [128][8] UE4M3 scales, one per 16 elements along K), b: [N][K]
 * row-major likewise, d: fp32 [128][N]; N = 128. */
int vca_debug_mma(int mode, const void* a, const void* b, float* d, vca_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* VCA_H */
