// noalloc.cu -- atlas_mem_forward_noalloc: the chunked update for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run the update: code inside a custom allocator or memory-pool
// callback, host code that must not grow the device footprint after start-up,
// or hosts whose device memory is fully reserved in advance.  For them this
// entry point takes its scratch from one file-scope device array instead of
// the caller's workspace.  The array exists once per device that loads the
// library and stays allocated until the process exits.
#include <mutex>

#include "atlas_mem.h"

// Scratch shared by every call of atlas_mem_forward_noalloc on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATLAS_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device.  In host code the array's name is only a host-side stand-in, so
// the address has to come from cudaGetSymbolAddress.
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATLAS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ATLAS_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ATLAS_OK;
}

}  // namespace

extern "C" int atlas_mem_forward_noalloc(const void* K, const void* Q, const void* V,
                                         const float* alpha, const float* eta,
                                         const float* theta, const float* gamma,
                                         const atlas_mem_cfg* cfg, float* Y, float* M_final,
                                         void* stream) {
  if (!cfg) return ATLAS_ERR_INVALID;
  const size_t need = atlas_mem_workspace_bytes(cfg);
  if (need == (size_t)-1) return ATLAS_ERR_INVALID;
  if (need > (size_t)ATLAS_NOALLOC_SCRATCH_BYTES) return ATLAS_ERR_WORKSPACE;
  atlas_mem_cfg c = *cfg;
  c.workspace = nullptr;
  c.workspace_bytes = 0;
  if (need > 0) {
    void* p = nullptr;
    const int rc = scratch_for_current_device(&p);
    if (rc != ATLAS_OK) return rc;
    c.workspace = p;
    c.workspace_bytes = (size_t)ATLAS_NOALLOC_SCRATCH_BYTES;
  }
  return atlas_mem_forward(K, Q, V, alpha, eta, theta, gamma, &c, Y, M_final, stream);
}
