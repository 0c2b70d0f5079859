// Host-buffer pipeline of the C ABI (include/vca.h, vca_pipeline_*): staging
// slots in a caller-owned device workspace, one non-blocking stream per copy
// direction and per-slot events that order each step's copies against the
// compute of the steps around it.  Host code only; the compute is the
// library's preparation and attention entry points.
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>

#include "../../include/vca.h"

struct vca_pipeline {
  int B, H, N, d, k, bits, slots;
  size_t tensor_bytes, state_bytes, slot_stride;
  uint8_t* ws;
  cudaStream_t compute, h2d, d2h;
  cudaEvent_t in_ready[VCA_PIPELINE_MAX_SLOTS];  // the slot's inputs have landed
  cudaEvent_t consumed[VCA_PIPELINE_MAX_SLOTS];  // the slot's compute is done
  cudaEvent_t d2h_done[VCA_PIPELINE_MAX_SLOTS];  // the slot's O is in host memory
  int64_t submitted;
};

namespace {

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// 0 on an invalid shape (vca_state_bytes's checks) or slot count
bool pipeline_sizes(int B, int H, int N, int d, int k, int bits, int slots, size_t* tensor,
                    size_t* state, size_t* total) {
  if (slots < 1 || slots > VCA_PIPELINE_MAX_SLOTS) return false;
  const size_t sb = vca_state_bytes(B, H, N, d, k, bits);
  if (sb == 0) return false;
  *tensor = round256((size_t)B * H * N * d * 2);
  *state = round256(sb);
  *total = *state + (size_t)slots * 4 * *tensor;
  return true;
}

uint8_t* slot_ptr(const vca_pipeline* p, int slot, int which) {  // which: 0 q, 1 k, 2 v, 3 o
  return p->ws + p->state_bytes + (size_t)slot * p->slot_stride + (size_t)which * p->tensor_bytes;
}

void release(vca_pipeline* p) {
  for (int s = 0; s < VCA_PIPELINE_MAX_SLOTS; ++s) {
    if (p->in_ready[s]) cudaEventDestroy(p->in_ready[s]);
    if (p->consumed[s]) cudaEventDestroy(p->consumed[s]);
    if (p->d2h_done[s]) cudaEventDestroy(p->d2h_done[s]);
  }
  if (p->h2d) cudaStreamDestroy(p->h2d);
  if (p->d2h) cudaStreamDestroy(p->d2h);
  std::free(p);
}

}  // namespace

extern "C" {

size_t vca_pipeline_workspace_bytes(int B, int H, int N, int d, int k_clusters, int bits,
                                    int slots) {
  size_t t, s, total;
  return pipeline_sizes(B, H, N, d, k_clusters, bits, slots, &t, &s, &total) ? total : 0;
}

int vca_pipeline_create(int B, int H, int N, int d, int k_clusters, int bits, int slots,
                        void* workspace, size_t workspace_bytes, vca_stream_t stream,
                        vca_pipeline** out) {
  if (!out) return VCA_ERR_INVALID_ARG;
  *out = nullptr;
  size_t t, s, total;
  if (!pipeline_sizes(B, H, N, d, k_clusters, bits, slots, &t, &s, &total))
    return (slots < 1 || slots > VCA_PIPELINE_MAX_SLOTS) ? VCA_ERR_INVALID_ARG
                                                         : VCA_ERR_UNSUPPORTED;
  if (!workspace || ((uintptr_t)workspace & 255u)) return VCA_ERR_INVALID_ARG;
  if (workspace_bytes < total) return VCA_ERR_BUFFER_TOO_SMALL;
  vca_pipeline* p = static_cast<vca_pipeline*>(std::calloc(1, sizeof(vca_pipeline)));
  if (!p) return VCA_ERR_CUDA;
  p->B = B; p->H = H; p->N = N; p->d = d; p->k = k_clusters; p->bits = bits; p->slots = slots;
  p->tensor_bytes = t;
  p->state_bytes = s;
  p->slot_stride = 4 * t;
  p->ws = static_cast<uint8_t*>(workspace);
  p->compute = (cudaStream_t)stream;
  bool ok = cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; ok && i < slots; ++i)
    ok = cudaEventCreateWithFlags(&p->in_ready[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->consumed[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->d2h_done[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    release(p);
    return VCA_ERR_CUDA;
  }
  *out = p;
  return VCA_OK;
}

int vca_pipeline_submit(vca_pipeline* p, const void* q_host, const void* k_host,
                        const void* v_host, void* o_host, int reuse_perm, int iters,
                        uint64_t seed, unsigned flags, int64_t* step) {
  if (!p || !q_host || !k_host || !v_host || !o_host) return VCA_ERR_INVALID_ARG;
  // the preparation's own argument checks, here so that nothing is enqueued
  // for a step that would be refused
  if (reuse_perm < VCA_PERM_FRESH || reuse_perm > VCA_PERM_NAIVE) return VCA_ERR_INVALID_ARG;
  if (iters < 1 || iters > 1000) return VCA_ERR_INVALID_ARG;
  if (flags & ~(VCA_PREP_QK_HADAMARD | VCA_PIPELINE_FP8_EXP)) return VCA_ERR_INVALID_ARG;
  const bool exp_bytes = (flags & VCA_PIPELINE_FP8_EXP) != 0;
  if (exp_bytes && p->bits != 8) return VCA_ERR_INVALID_ARG;
  const int64_t i = p->submitted;
  const int s = (int)(i % p->slots);
  const size_t nbytes = (size_t)p->B * p->H * p->N * p->d * 2;
  uint8_t* dq = slot_ptr(p, s, 0);
  uint8_t* dk = slot_ptr(p, s, 1);
  uint8_t* dv = slot_ptr(p, s, 2);
  uint8_t* dout = slot_ptr(p, s, 3);
  const bool reused = i >= p->slots;
  // inputs: after step i - slots has finished reading the slot
  if (reused && cudaStreamWaitEvent(p->h2d, p->consumed[s], 0) != cudaSuccess) return VCA_ERR_CUDA;
  // From the first copy on, a failure must not leave work in flight that
  // still reads the caller's host buffers or the slot: wait for all of it.
  auto fail = [&](int rc) {
    cudaStreamSynchronize(p->h2d);
    cudaStreamSynchronize(p->compute);
    cudaStreamSynchronize(p->d2h);
    return rc;
  };
  const void* src[3] = {q_host, k_host, v_host};
  uint8_t* dst[3] = {dq, dk, dv};
  for (int t = 0; t < 3; ++t)
    if (cudaMemcpyAsync(dst[t], src[t], nbytes, cudaMemcpyHostToDevice, p->h2d) != cudaSuccess)
      return fail(VCA_ERR_CUDA);
  if (cudaEventRecord(p->in_ready[s], p->h2d) != cudaSuccess) return fail(VCA_ERR_CUDA);
  // compute: once the inputs landed and step i - slots's O was read back
  if (cudaStreamWaitEvent(p->compute, p->in_ready[s], 0) != cudaSuccess) return fail(VCA_ERR_CUDA);
  if (reused && cudaStreamWaitEvent(p->compute, p->d2h_done[s], 0) != cudaSuccess)
    return fail(VCA_ERR_CUDA);
  int rc = vca_vsmooth_prepare_ex(dq, dk, dv, p->B, p->H, p->N, p->d, p->k, reuse_perm, p->bits,
                                  iters, seed, flags & VCA_PREP_QK_HADAMARD, p->ws,
                                  p->state_bytes,
                                  (vca_stream_t)p->compute);
  if (rc != VCA_OK) return fail(rc);
  const vca_stream_t cs = (vca_stream_t)p->compute;
  if (p->bits == 4)
    rc = vca_attention_nvfp4(p->ws, p->state_bytes, p->B, p->H, p->N, p->d, dout, cs);
  else if (exp_bytes)
    rc = vca_attention_fp8_exp(p->ws, p->state_bytes, p->B, p->H, p->N, p->d, dout, cs);
  else
    rc = vca_attention_fp8(p->ws, p->state_bytes, p->B, p->H, p->N, p->d, dout, cs);
  if (rc != VCA_OK) return fail(rc);
  if (cudaEventRecord(p->consumed[s], p->compute) != cudaSuccess) return fail(VCA_ERR_CUDA);
  // read-back
  if (cudaStreamWaitEvent(p->d2h, p->consumed[s], 0) != cudaSuccess) return fail(VCA_ERR_CUDA);
  if (cudaMemcpyAsync(o_host, dout, nbytes, cudaMemcpyDeviceToHost, p->d2h) != cudaSuccess)
    return fail(VCA_ERR_CUDA);
  if (cudaEventRecord(p->d2h_done[s], p->d2h) != cudaSuccess) return fail(VCA_ERR_CUDA);
  p->submitted = i + 1;
  if (step) *step = i;
  return VCA_OK;
}

int vca_pipeline_wait(vca_pipeline* p, int64_t step) {
  if (!p || step < 0 || step >= p->submitted) return VCA_ERR_INVALID_ARG;
  // the slot's event marks its latest read-back, which comes after this step's
  return cudaEventSynchronize(p->d2h_done[step % p->slots]) == cudaSuccess ? VCA_OK
                                                                          : VCA_ERR_CUDA;
}

int vca_pipeline_flush(vca_pipeline* p) {
  if (!p) return VCA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(p->h2d) != cudaSuccess || cudaStreamSynchronize(p->d2h) != cudaSuccess)
    return VCA_ERR_CUDA;
  return vca_get_status(p->ws, nullptr, (vca_stream_t)p->compute);
}

void* vca_pipeline_state(vca_pipeline* p) { return p ? p->ws : nullptr; }

int vca_pipeline_destroy(vca_pipeline* p) {
  if (!p) return VCA_OK;
  const bool ok = cudaStreamSynchronize(p->h2d) == cudaSuccess &&
                  cudaStreamSynchronize(p->d2h) == cudaSuccess &&
                  cudaStreamSynchronize(p->compute) == cudaSuccess;
  release(p);
  return ok ? VCA_OK : VCA_ERR_CUDA;
}

}  // extern "C"
