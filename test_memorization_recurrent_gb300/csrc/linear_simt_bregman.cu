// linear_simt_bregman.cu -- the CUDA-core linear kernel's instantiation for the
// Bregman (sigmoid link) retention gate (token-serial walk); the kernel itself is in
// linear_simt_body.cuh.
#include "linear_simt_body.cuh"

namespace atlas {

cudaError_t linear_simt_bregman_launch(const cudaLaunchConfig_t* cfg, const LinArgs& a,
                                       const LinSimtSmem& s, const int* flags) {
  return linear_simt_launch_gate<ATLAS_RET_BREGMAN>(cfg, a, s, flags);
}

}  // namespace atlas
