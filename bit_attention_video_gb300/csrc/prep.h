// Internal interfaces of the VC-Attention library: state-blob layout, the
// arguments of the preparation chain and the kernel launchers.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/vca.h"

namespace vca {

constexpr uint32_t kStateMagic = 0x31414356u;  // "VCA1"
constexpr uint32_t kTileBytes = 128 * 128;         // one 128 x 128 E4M3 tile
// Mean operand of the restoration MMA for a group of kGroup key blocks: two
// 128 (channel) x 16 (K) bf16 K-major chunks without swizzle (hi, lo); slot k
// of the group is K column k, columns kGroup..15 are zero.
constexpr int kGroup = 8;
constexpr uint32_t kGroupBytes = 2 * 128 * 16 * 2;
// 4-bit path: groups of kGroup4 blocks share one 128 (channel) x 16 (K) bf16
// K-major chunk without swizzle; K row k holds the block mean of slot
// (k % 8) / 2, so that each softmax thread's row-sum pair (hi, lo) of every
// slot meets its block's mean.
constexpr int kGroup4 = 4;
constexpr uint32_t kGroup4Bytes = 128 * 16 * 2;
constexpr uint32_t kTile4Bytes = 128 * 64;         // one 128 x 128 E2M1 tile
constexpr uint32_t kScaleTileBytes = 1024;         // UE4M3 scales of a 128 x 128 tile

// Header words (uint32): magic, B, H, N, d, k, bits, perm cached, operands ready.

// Computes the blob layout; returns VCA_OK or an argument error.
int compute_layout(int B, int H, int N, int d, int k, int bits, vca_state_layout* L);

struct PrepArgs {
  const uint16_t* q;
  const uint16_t* k_in;
  const uint16_t* v;
  int B, H, N, nb, Npad, k, iters, reuse;
  unsigned flags;  // VCA_PREP_* options
  uint64_t seed;
  uint8_t* state;
  vca_state_layout L;
};

int launch_prepare8(const PrepArgs& a, cudaStream_t st);
int launch_prepare4(const PrepArgs& a, cudaStream_t st);
// expcast = false: the conventional exponential-then-E4M3 bytes
int launch_attention_fp8(uint8_t* state, const vca_state_layout& L, int B, int H, int N, void* o,
                         bool expcast, cudaStream_t st);
int launch_attention_nvfp4(uint8_t* state, const vca_state_layout& L, int B, int H, int N,
                           void* o, cudaStream_t st);
int launch_attention_bf16(const void* q, const void* k, const void* v, int B, int H, int N,
                          void* o, int* status, cudaStream_t st);

// The status word of vca_kmeans_permutation_noalloc's fixed scratch on the
// current device, or nullptr if that entry point has not run on it yet.
int* noalloc_status_word();

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
// 2-D tensor of `elem_bytes`-byte elements: inner extent `dim0`, `dim1` rows of
// `row_bytes` bytes, box (box0, box1); `swizzle` = 128, 64 (bytes) or 0 (none).
bool make_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t dim0,
                  uint64_t dim1, uint64_t row_bytes, uint32_t box0, uint32_t box1,
                  int swizzle = 128);

}  // namespace vca
