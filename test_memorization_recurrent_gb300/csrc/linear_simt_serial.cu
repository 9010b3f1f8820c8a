// linear_simt_serial.cu -- the CUDA-core linear kernel's token-serial
// instantiation (elastic-net, Bregman and KL retention gates); the kernel itself
// is in linear_simt_body.cuh.
#include "linear_simt_body.cuh"

namespace atlas {

cudaError_t linear_simt_serial_launch(const cudaLaunchConfig_t* cfg, const LinArgs& a,
                                      const LinSimtSmem& s, const int* flags) {
  const cudaError_t e = cudaFuncSetAttribute(
      linear_simt_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)cfg->dynamicSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(cfg, linear_simt_kernel<true>, a, s, flags);
}

}  // namespace atlas
