// The C ABI (include/vca.h): argument validation, state-blob layout and the
// launch of the preparation and attention kernels.  No allocation, no
// synchronisation except in vca_get_status.
#include <cstring>

#include "common.cuh"
#include "prep.h"

namespace vca {

int compute_layout(int B, int H, int N, int d, int k, int bits, vca_state_layout* L) {
  if (B < 1 || H < 1 || N < 1 || !L) return VCA_ERR_INVALID_ARG;
  if (d != 128 || (bits != 8 && bits != 4)) return VCA_ERR_UNSUPPORTED;
  if (k < 1 || k > 256 || k > N) return VCA_ERR_UNSUPPORTED;
  // B*H is the y extent of the preparation's grids (at most 65535); the TMA
  // row coordinates and the token indices are 32-bit (B*H*Npad < 2^31)
  if ((int64_t)B * H > 65535 || N > (1 << 24)) return VCA_ERR_UNSUPPORTED;
  if ((int64_t)B * H * ((N + 127) / 128 * 128) >= (int64_t)1 << 31) return VCA_ERR_UNSUPPORTED;
  std::memset(L, 0, sizeof(*L));
  const uint64_t BH = (uint64_t)B * H, nb = (N + 127) / 128, Npad = nb * 128;
  uint64_t off = 0;
  auto take = [&](uint64_t bytes) {
    off = (off + 1023) & ~uint64_t(1023);
    const uint64_t o = off;
    off += bytes;
    return o;
  };
  // Everything the attention kernels read depends only on (B, H, N, bits) and
  // comes first, so the attention calls can locate it without k.
  L->header = take(256);
  L->status = take(4);
  if (bits == 8) {
    L->qhat = take(BH * Npad * d);
    L->sq = take(BH * nb * 4);
    L->khat = take(BH * Npad * d);
    L->sk = take(BH * nb * 4);
    L->rhatT = take(BH * d * Npad);
    L->sv = take(BH * d * 4);
    L->mutilde = take(BH * nb * d * 4);
  } else {
    L->q4 = take(BH * Npad * d / 2);
    L->q4s = take(BH * nb * kScaleTileBytes);
    L->k4 = take(BH * Npad * d / 2);
    L->kr4s = take(BH * nb * 2 * kScaleTileBytes);
    L->r4T = take(BH * d * Npad / 2);
    L->g4 = take(BH * 16);
  }
  L->mside = bits == 8 ? take(BH * ((nb + kGroup - 1) / kGroup) * kGroupBytes)
                       : take(BH * ((nb + kGroup4 - 1) / kGroup4) * kGroup4Bytes);
  L->mu = take(BH * nb * d * 2);
  L->kbar = take(BH * d * 2);
  L->perm = take(BH * N * 4);
  L->labels = take(BH * N * 4);
  L->ksum = take(BH * nb * d * 4);
  L->vamax = take(BH * nb * d * 4);
  L->grid = take(BH * 8);
  L->features = take(BH * N * d * 2);  // fp16 (k <= 128) or int8
  L->centroids = take(BH * k * d);
  L->sums = take(BH * k * d * 4 + BH * k * 4);
  L->total_bytes = (off + 1023) & ~uint64_t(1023);
  return VCA_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t dim0,
                  uint64_t dim1, uint64_t row_bytes, uint32_t box0, uint32_t box1,
                  int swizzle) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return false;
    fn = (EncodeTiledFn)p;
  }
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle == 64    ? CU_TENSOR_MAP_SWIZZLE_64B
            : swizzle == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                             : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace vca

using namespace vca;

namespace {
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
}  // namespace

extern "C" {

size_t vca_state_bytes(int B, int H, int N, int d, int k_clusters, int bits) {
  vca_state_layout L;
  return compute_layout(B, H, N, d, k_clusters, bits, &L) == VCA_OK ? (size_t)L.total_bytes : 0;
}

int vca_state_layout_get(int B, int H, int N, int d, int k_clusters, int bits,
                         vca_state_layout* out) {
  return compute_layout(B, H, N, d, k_clusters, bits, out);
}

int vca_vsmooth_prepare(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                        int k_clusters, int reuse_perm, int bits, int iters, uint64_t seed,
                        void* state, size_t state_bytes, vca_stream_t stream) {
  return vca_vsmooth_prepare_ex(q, k, v, B, H, N, d, k_clusters, reuse_perm, bits, iters, seed,
                                0u, state, state_bytes, stream);
}

int vca_vsmooth_prepare_ex(const void* q, const void* k, const void* v, int B, int H, int N,
                           int d, int k_clusters, int reuse_perm, int bits, int iters,
                           uint64_t seed, unsigned flags, void* state, size_t state_bytes,
                           vca_stream_t stream) {
  vca_state_layout L;
  const int rc = compute_layout(B, H, N, d, k_clusters, bits, &L);
  if (rc != VCA_OK) return rc;
  if (!q || !k || !v || !state) return VCA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || ((uintptr_t)state & 255u))
    return VCA_ERR_INVALID_ARG;
  if (reuse_perm != VCA_PERM_FRESH && reuse_perm != VCA_PERM_REUSE &&
      reuse_perm != VCA_PERM_WARM && reuse_perm != VCA_PERM_PLAIN && reuse_perm != VCA_PERM_NAIVE)
    return VCA_ERR_INVALID_ARG;
  if (iters < 1 || iters > 1000) return VCA_ERR_INVALID_ARG;
  if (flags & ~VCA_PREP_QK_HADAMARD) return VCA_ERR_INVALID_ARG;
  if (state_bytes < L.total_bytes) return VCA_ERR_BUFFER_TOO_SMALL;
  PrepArgs a;
  a.q = (const uint16_t*)q;
  a.k_in = (const uint16_t*)k;
  a.v = (const uint16_t*)v;
  a.B = B; a.H = H; a.N = N; a.nb = (N + 127) / 128; a.Npad = a.nb * 128;
  a.k = k_clusters; a.iters = iters; a.reuse = reuse_perm; a.seed = seed;
  a.flags = flags;
  a.state = (uint8_t*)state;
  a.L = L;
  return bits == 8 ? launch_prepare8(a, (cudaStream_t)stream)
                   : launch_prepare4(a, (cudaStream_t)stream);
}

// Layout of the operands an attention call reads (independent of k).
static int attention_common(void* state, size_t state_bytes, int B, int H, int N, int d, void* o,
                            int bits, vca_state_layout* L) {
  const int rc = compute_layout(B, H, N, d, 1, bits, L);
  if (rc != VCA_OK) return rc;
  if (!state || !o) return VCA_ERR_INVALID_ARG;
  if (((uintptr_t)state & 255u) || !aligned16(o)) return VCA_ERR_INVALID_ARG;
  if (state_bytes < L->labels) return VCA_ERR_BUFFER_TOO_SMALL;
  return VCA_OK;
}

int vca_attention_fp8(void* state, size_t state_bytes, int B, int H, int N, int d, void* o,
                      vca_stream_t stream) {
  vca_state_layout L;
  const int rc = attention_common(state, state_bytes, B, H, N, d, o, 8, &L);
  if (rc != VCA_OK) return rc;
  return launch_attention_fp8((uint8_t*)state, L, B, H, N, o, true, (cudaStream_t)stream);
}

int vca_attention_fp8_exp(void* state, size_t state_bytes, int B, int H, int N, int d, void* o,
                          vca_stream_t stream) {
  vca_state_layout L;
  const int rc = attention_common(state, state_bytes, B, H, N, d, o, 8, &L);
  if (rc != VCA_OK) return rc;
  return launch_attention_fp8((uint8_t*)state, L, B, H, N, o, false, (cudaStream_t)stream);
}

int vca_attention_nvfp4(void* state, size_t state_bytes, int B, int H, int N, int d, void* o,
                        vca_stream_t stream) {
  vca_state_layout L;
  const int rc = attention_common(state, state_bytes, B, H, N, d, o, 4, &L);
  if (rc != VCA_OK) return rc;
  return launch_attention_nvfp4((uint8_t*)state, L, B, H, N, o, (cudaStream_t)stream);
}

int vca_attention_bf16_ref(const void* q, const void* k, const void* v, int B, int H, int N,
                           int d, void* o, int* status, vca_stream_t stream) {
  if (B < 1 || H < 1 || N < 1) return VCA_ERR_INVALID_ARG;
  if (d != 128 || (int64_t)B * H > 65535 || N > (1 << 24)) return VCA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o) return VCA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return VCA_ERR_INVALID_ARG;
  return launch_attention_bf16(q, k, v, B, H, N, o, status, (cudaStream_t)stream);
}

int vca_get_status(void* state, int* status_word, vca_stream_t stream) {
  int* dev = status_word;
  if (state) {
    vca_state_layout L;
    compute_layout(1, 1, 1, 128, 1, 8, &L);  // the status offset does not depend on the shape
    dev = reinterpret_cast<int*>((uint8_t*)state + L.status);
  } else if (!status_word) {
    dev = noalloc_status_word();  // the allocation-free grouping call's word
  }
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return VCA_ERR_CUDA;
  if (!dev) return VCA_OK;  // that call has not run on this device
  int h = 0;
  if (cudaMemcpy(&h, dev, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return VCA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(dev, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return VCA_ERR_CUDA;
  if (h == 0) return VCA_OK;
  if (h & kStatNoPerm) return VCA_ERR_NO_CACHED_PERM;
  if (h & kStatStateMismatch) return VCA_ERR_STATE_MISMATCH;
  if (h & kStatTimeout) return VCA_ERR_TIMEOUT;
  return VCA_ERR_INVALID_ARG;
}

const char* vca_status_string(int s) {
  switch (s) {
    case VCA_OK: return "ok";
    case VCA_ERR_INVALID_ARG: return "invalid argument";
    case VCA_ERR_UNSUPPORTED: return "unsupported shape or bit width";
    case VCA_ERR_CUDA: return "CUDA error";
    case VCA_ERR_BUFFER_TOO_SMALL: return "state buffer too small";
    case VCA_ERR_NO_CACHED_PERM: return "no cached permutation for this shape";
    case VCA_ERR_TIMEOUT: return "device pipeline wait timed out";
    case VCA_ERR_STATE_MISMATCH: return "state prepared for another shape or bit width";
    default: return "unknown status";
  }
}

}  // extern "C"
