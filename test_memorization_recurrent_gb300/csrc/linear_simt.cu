// linear_simt.cu -- the CUDA-core linear kernel's chunk-table instantiation,
// its plan (rows per CTA, clusters for the robust bias) and the launch of
// either instantiation; the kernel itself is in linear_simt_body.cuh.
#include "linear_simt_body.cuh"

namespace atlas {

// Rows per CTA (RV) and CTAs per cluster (robust bias only; a head's row blocks
// form one cluster of ncl <= 8 CTAs, so RV = ceil(d_v / ncl)).
static int plan(const LinArgs& a, int heads, LinSimtSmem* out) {
  const int Lmax = a.b + a.c - 1;
  const size_t limit = 200 * 1024;
  const bool robust = a.lk == ATLAS_LOSS_ROBUST;
  int RV = a.d_v, ncl = 1;
  while (RV > 1) {
    LinSimtSmem s = lin_simt_layout(RV, a.D, Lmax, a.b, a.d_k, a.pgen);
    const long ctas = (long)heads * ((a.d_v + RV - 1) / RV);
    if (s.bytes() <= limit && (ctas >= 152 || RV <= 4)) break;
    if (robust) {
      if (ncl == 8) break;
      ncl *= 2;
      RV = (a.d_v + ncl - 1) / ncl;
    } else {
      RV = (RV + 1) / 2;
    }
  }
  LinSimtSmem s = lin_simt_layout(RV, a.D, Lmax, a.b, a.d_k, a.pgen);
  if (s.bytes() > limit) return ATLAS_ERR_UNSUPPORTED;
  s.ncl = robust ? ncl : 1;
  *out = s;
  return ATLAS_OK;
}

int linear_simt_plan(const LinArgs& a, int heads, int* RV_out, size_t* smem_out) {
  LinSimtSmem s;
  const int rc = plan(a, heads, &s);
  if (rc) return rc;
  *RV_out = s.RV;
  *smem_out = s.bytes();
  return ATLAS_OK;
}

static int launch(const LinArgs& a, int heads, const int* flags, cudaStream_t st) {
  LinSimtSmem s;
  int rc = plan(a, heads, &s);
  if (rc) return rc;
  if (flags && s.ncl > 1) return ATLAS_ERR_UNSUPPORTED;
  const size_t smem = s.bytes();
  const int rows = flags ? 1 : (s.ncl > 1 ? s.ncl : (a.d_v + s.RV - 1) / s.RV);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(heads, rows);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (s.ncl > 1) {  // one cluster per head: its ncl row blocks
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = s.ncl;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  } else if (flags) {  // after the tensor-core kernel: launch overlaps its tail
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaError_t e;
  switch (a.ret) {
    case ATLAS_RET_ELASTIC: e = linear_simt_elastic_launch(&cfg, a, s, flags); break;
    case ATLAS_RET_BREGMAN: e = linear_simt_bregman_launch(&cfg, a, s, flags); break;
    case ATLAS_RET_KL: e = linear_simt_kl_launch(&cfg, a, s, flags); break;
    default: e = linear_simt_launch_gate<ATLAS_RET_L2>(&cfg, a, s, flags); break;
  }
  if (e != cudaSuccess) return ATLAS_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ATLAS_OK : ATLAS_ERR_CUDA;
}

int linear_simt_launch(const LinArgs& a, int heads, cudaStream_t st) {
  return launch(a, heads, nullptr, st);
}

int linear_simt_launch_flagged(const LinArgs& a, int heads, const int* flags, cudaStream_t st) {
  return launch(a, heads, flags, st);
}

}  // namespace atlas
