// 4-bit (NVFP4) VC-Attention: preparation and attention.
#include "common.cuh"
#include "prep.h"

namespace vca {

int launch_prepare4(const PrepArgs&, cudaStream_t) { return VCA_ERR_UNSUPPORTED; }

int launch_attention_nvfp4(uint8_t*, const vca_state_layout&, int, int, int, void*,
                           cudaStream_t) {
  return VCA_ERR_UNSUPPORTED;
}

}  // namespace vca
