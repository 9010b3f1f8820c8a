// atlas_mem.cu -- C-ABI entry points: argument validation, path choice,
// workspace sizing and launch.  Every computation happens in the kernels of
// linear_*.cu and mlp_*.cu; this file only plans.
#include <string.h>

#include "atlas_mem.h"
#include "kernels.h"

using namespace atlas;

namespace {

enum Path {
  PATH_INVALID = 0, PATH_LINEAR_SIMT, PATH_LINEAR_TC, PATH_LINEAR_SEQ, PATH_LINEAR_CHUNK,
  PATH_MLP_SIMT, PATH_MLP_TC, PATH_LINEAR_WIDE
};

// Monomials of degree exactly e in d variables: C(d + e - 1, e).
long monomials(long d, int e) {
  long c = 1;
  for (int i = 1; i <= e; ++i) c = c * (d + i - 1) / i;
  return c;
}

long feature_dim_long(const atlas_mem_cfg* c) {
  if (c->mem == ATLAS_MEM_LINEAR && c->phi == ATLAS_PHI_POLY2)
    return (long)c->d_k + (long)c->d_k * (c->d_k + 1) / 2;
  if (c->mem == ATLAS_MEM_LINEAR && c->phi == ATLAS_PHI_POLY) {
    long D = 0;
    for (int e = 0; e <= c->phi_degree; ++e)
      if (c->phi_coef[e] != 0.f) D += monomials(c->d_k, e);
    return D;
  }
  return c->d_k;
}

int feature_dim(const atlas_mem_cfg* c) { return (int)feature_dim_long(c); }

// Structural validation (no pointers).  Returns ATLAS_OK, INVALID or UNSUPPORTED.
int check_cfg(const atlas_mem_cfg* c) {
  if (!c) return ATLAS_ERR_INVALID;
  if (c->B < 0 || c->H < 0 || c->N < 0) return ATLAS_ERR_INVALID;
  if (c->d_k <= 0 || c->d_v <= 0 || c->c < 1 || c->b < 1) return ATLAS_ERR_INVALID;
  if (c->mem < ATLAS_MEM_LINEAR || c->mem > ATLAS_MEM_MLP_GATED) return ATLAS_ERR_INVALID;
  if (c->phi != ATLAS_PHI_IDENTITY && c->phi != ATLAS_PHI_POLY2 && c->phi != ATLAS_PHI_POLY)
    return ATLAS_ERR_INVALID;
  if (c->phi == ATLAS_PHI_POLY) {
    if (c->phi_degree < 1 || c->phi_degree > ATLAS_PHI_MAX_DEGREE) return ATLAS_ERR_INVALID;
    for (int e = 0; e <= c->phi_degree; ++e)
      if (!(c->phi_coef[e] == c->phi_coef[e]) || c->phi_coef[e] > 3e38f || c->phi_coef[e] < -3e38f)
        return ATLAS_ERR_INVALID;  // NaN or infinite
    if (c->d_k > 255) return ATLAS_ERR_UNSUPPORTED;
    const long D = feature_dim_long(c);
    if (D < 1) return ATLAS_ERR_INVALID;
    if (D > 16384) return ATLAS_ERR_UNSUPPORTED;
  }
  if (c->loss < ATLAS_LOSS_L2 || c->loss > ATLAS_LOSS_ROBUST) return ATLAS_ERR_INVALID;
  if (c->loss == ATLAS_LOSS_ROBUST && !(c->loss_param >= 0.f && c->loss_param < 3e38f))
    return ATLAS_ERR_INVALID;
  if (c->retention < ATLAS_RET_L2 || c->retention > ATLAS_RET_LQ) return ATLAS_ERR_INVALID;
  if (c->retention == ATLAS_RET_ELASTIC && !(c->ret_param >= 0.f && c->ret_param < 3e38f))
    return ATLAS_ERR_INVALID;
  if (c->retention == ATLAS_RET_KL && !(c->ret_param > 0.f && c->ret_param < 3e38f))
    return ATLAS_ERR_INVALID;
  if (c->retention == ATLAS_RET_LQ && !(c->ret_param >= 1.f && c->ret_param < 1e6f))
    return ATLAS_ERR_INVALID;
  if (c->loss == ATLAS_LOSS_LP && !(c->loss_param >= 1.f && c->loss_param < 1e6f))
    return ATLAS_ERR_INVALID;
  if (c->loss == ATLAS_LOSS_HUBER && !(c->loss_param > 0.f && c->loss_param < 3e38f))
    return ATLAS_ERR_INVALID;
  if (c->in_dtype != ATLAS_F32 && c->in_dtype != ATLAS_BF16) return ATLAS_ERR_INVALID;
  if (c->ns_steps < 0 || c->n_history < 0) return ATLAS_ERR_INVALID;
  if ((long)c->B * c->H > 65535L * 1024) return ATLAS_ERR_UNSUPPORTED;
  if (c->mem != ATLAS_MEM_LINEAR) {
    if (c->d_h <= 0 || c->d_k != c->d_v) return ATLAS_ERR_INVALID;
    if (c->phi != ATLAS_PHI_IDENTITY) return ATLAS_ERR_INVALID;
    if (c->loss == ATLAS_LOSS_DOT) return ATLAS_ERR_UNSUPPORTED;
    if (c->retention != ATLAS_RET_L2) return ATLAS_ERR_UNSUPPORTED;
  } else {
    if (c->ns_steps > 0) return ATLAS_ERR_UNSUPPORTED;
    if (c->phi == ATLAS_PHI_POLY2 && c->d_k > 64) return ATLAS_ERR_UNSUPPORTED;
  }
  return ATLAS_OK;
}

LinArgs lin_args(const void* K, const void* Q, const void* V, const float* alpha,
                 const float* eta, const float* theta, const float* gamma,
                 const atlas_mem_cfg* c, float* Y, float* M) {
  LinArgs a;
  a.K = K; a.Q = Q; a.V = V;
  a.alpha = alpha; a.eta = eta; a.theta = theta; a.gamma = gamma;
  a.Y = Y; a.M = M; a.S = c->S_state;
  a.N = c->N; a.d_k = c->d_k; a.d_v = c->d_v; a.D = feature_dim(c);
  a.c = c->c; a.b = c->b;
  a.poly = c->phi == ATLAS_PHI_POLY2;
  a.dot = c->loss == ATLAS_LOSS_DOT;
  a.lk = c->loss;
  a.lp = c->loss_param;
  a.bf16 = c->in_dtype == ATLAS_BF16;
  a.nh = c->n_history;
  a.pgen = c->phi == ATLAS_PHI_POLY;
  a.pdeg = a.pgen ? c->phi_degree : 0;
  for (int e = 0; e < 5; ++e) a.pcoef[e] = (a.pgen && e <= c->phi_degree) ? c->phi_coef[e] : 0.f;
  a.ret = c->retention;
  a.rp = c->ret_param;
  return a;
}

MlpArgs mlp_args(const void* K, const void* Q, const void* V, const float* alpha,
                 const float* eta, const float* theta, const float* gamma,
                 const atlas_mem_cfg* c, float* Y, float* M) {
  MlpArgs a;
  a.K = K; a.Q = Q; a.V = V;
  a.alpha = alpha; a.eta = eta; a.theta = theta; a.gamma = gamma;
  a.Y = Y; a.M = M; a.S = c->S_state;
  a.heads = c->B * c->H; a.N = c->N; a.d = c->d_k; a.dh = c->d_h; a.c = c->c; a.b = c->b;
  a.nh = c->n_history;
  a.bf16 = c->in_dtype == ATLAS_BF16;
  a.lk = c->loss;
  a.lp = c->loss_param;
  a.ns_steps = c->ns_steps;
  a.ns_a = c->ns_a; a.ns_b = c->ns_b; a.ns_c = c->ns_c; a.ns_eps = c->ns_eps;
  a.s_is_zero = c->S_state == nullptr;
  a.status = c->status_dev;
  a.ln = c->mem == ATLAS_MEM_MLP_LN;
  a.gated = c->mem == ATLAS_MEM_MLP_GATED;
  return a;
}

Path choose_path(const atlas_mem_cfg* c) {
  if (check_cfg(c) != ATLAS_OK) return PATH_INVALID;
  if (c->mem != ATLAS_MEM_LINEAR) {
    MlpArgs m = mlp_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, c,
                         nullptr, nullptr);
    // the tensor-core kernels take no history rows (with c = 1 they would not matter,
    // but the K / V strides would): such calls go to the CUDA-core path
    return (m.nh == 0 && mlp_tc_supported(m)) ? PATH_MLP_TC : PATH_MLP_SIMT;
  }
  LinArgs a = lin_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, c,
                       nullptr, nullptr);
  const int heads = c->B * c->H;
  // wide feature maps (the degree-2 map, the gated map): the fused cluster kernel
  if (linear_wide_supported(a, heads) && !(a.nh == 0 && linear_tc_supported(a)) &&
      !linear_seq_supported(a))
    return PATH_LINEAR_WIDE;
  // the gated polynomial map, the retention gates and the robust bias: CUDA-core kernel only
  if (a.pgen || a.ret != ATLAS_RET_L2 || a.lk == ATLAS_LOSS_ROBUST) {
    int RV;
    size_t smem;
    return linear_simt_plan(a, c->B * c->H, &RV, &smem) == ATLAS_OK ? PATH_LINEAR_SIMT
                                                                      : PATH_INVALID;
  }
  if (a.nh == 0 && linear_tc_supported(a)) return PATH_LINEAR_TC;
  if (linear_seq_supported(a)) return PATH_LINEAR_SEQ;
  if (linear_chunk_supported(a)) return PATH_LINEAR_CHUNK;
  int RV;
  size_t smem;
  if (linear_simt_plan(a, c->B * c->H, &RV, &smem) != ATLAS_OK) return PATH_INVALID;
  return PATH_LINEAR_SIMT;
}

}  // namespace

extern "C" {

size_t atlas_mem_state_size(const atlas_mem_cfg* cfg) {
  if (check_cfg(cfg) != ATLAS_OK) return 0;
  if (cfg->mem == ATLAS_MEM_MLP_GATED) return (size_t)3 * cfg->d_k * cfg->d_h;
  if (cfg->mem != ATLAS_MEM_LINEAR) return (size_t)2 * cfg->d_k * cfg->d_h;
  return (size_t)cfg->d_v * feature_dim(cfg);
}

size_t atlas_mem_workspace_bytes(const atlas_mem_cfg* cfg) {
  if (check_cfg(cfg) != ATLAS_OK) return (size_t)-1;
  if (cfg->mem != ATLAS_MEM_LINEAR) {
    MlpArgs a = mlp_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, cfg,
                         nullptr, nullptr);
    return choose_path(cfg) == PATH_MLP_TC ? mlp_tc_workspace_bytes(a)
                                           : mlp_simt_workspace_bytes(a);
  }
  if (choose_path(cfg) == PATH_LINEAR_TC) return linear_tc_workspace_bytes(cfg->B * cfg->H);
  if (choose_path(cfg) == PATH_LINEAR_CHUNK) {
    LinArgs a = lin_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, cfg,
                         nullptr, nullptr);
    return linear_chunk_workspace_bytes(a, cfg->B * cfg->H);
  }
  return 0;
}

const char* atlas_mem_path(const atlas_mem_cfg* cfg) {
  switch (choose_path(cfg)) {
    case PATH_LINEAR_SIMT: return "linear_simt";
    case PATH_LINEAR_TC: return "linear_tc";
    case PATH_LINEAR_SEQ: return "linear_seq";
    case PATH_LINEAR_CHUNK: return "linear_chunk";
    case PATH_LINEAR_WIDE: return "linear_wide";
    case PATH_MLP_SIMT: return "mlp_simt";
    case PATH_MLP_TC: return "mlp_tc";
    default: return "";
  }
}

long atlas_mem_launch_count(const atlas_mem_cfg* cfg) {
  switch (choose_path(cfg)) {
    case PATH_LINEAR_SIMT:
    case PATH_LINEAR_SEQ:
    case PATH_LINEAR_WIDE:
    case PATH_MLP_TC:
      return (long)cfg->B * cfg->H > 0 ? 1 : 0;
    case PATH_LINEAR_TC:
      return (long)cfg->B * cfg->H > 0 ? 2 : 0;
    case PATH_LINEAR_CHUNK: {
      LinArgs a = lin_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, cfg,
                           nullptr, nullptr);
      return linear_chunk_launch_count(a, cfg->B * cfg->H);
    }
    case PATH_MLP_SIMT: {
      if ((long)cfg->B * cfg->H == 0) return 0;
      MlpArgs a = mlp_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, cfg,
                           nullptr, nullptr);
      return mlp_simt_launch_count(a);
    }
    default: return 0;
  }
}

int atlas_mem_forward(const void* K, const void* Q, const void* V, const float* alpha,
                      const float* eta, const float* theta, const float* gamma,
                      const atlas_mem_cfg* cfg, float* Y, float* M_final, void* stream) {
  int rc = check_cfg(cfg);
  if (rc != ATLAS_OK) return rc;
  const long heads = (long)cfg->B * cfg->H;
  if (heads == 0) return ATLAS_OK;
  if (!M_final || !gamma) return ATLAS_ERR_INVALID;
  if (cfg->N > 0 && (!K || !Q || !V || !alpha || !eta || !theta || !Y)) return ATLAS_ERR_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Path path = choose_path(cfg);
  if (path == PATH_INVALID) return ATLAS_ERR_UNSUPPORTED;
  if (path == PATH_MLP_TC) {
    MlpArgs a = mlp_args(K, Q, V, alpha, eta, theta, gamma, cfg, Y, M_final);
    const size_t need = mlp_tc_workspace_bytes(a);
    if (!cfg->workspace || cfg->workspace_bytes < need) return ATLAS_ERR_WORKSPACE;
    if (cfg->N == 0) return ATLAS_OK;
    return mlp_tc_launch(a, cfg->workspace, st);
  }
  if (path == PATH_MLP_SIMT) {
    MlpArgs a = mlp_args(K, Q, V, alpha, eta, theta, gamma, cfg, Y, M_final);
    const size_t need = mlp_simt_workspace_bytes(a);
    if (need > 0 && (!cfg->workspace || cfg->workspace_bytes < need)) return ATLAS_ERR_WORKSPACE;
    if (cfg->N == 0) return ATLAS_OK;
    return mlp_simt_forward(a, cfg->workspace, st);
  }
  LinArgs a = lin_args(K, Q, V, alpha, eta, theta, gamma, cfg, Y, M_final);
  if (path == PATH_LINEAR_TC) {
    const size_t need = linear_tc_workspace_bytes((int)heads);
    if (!cfg->workspace || cfg->workspace_bytes < need) return ATLAS_ERR_WORKSPACE;
    return linear_tc_launch(a, (int)heads, cfg->status_dev, cfg->workspace, st);
  }
  if (path == PATH_LINEAR_SEQ) return linear_seq_launch(a, (int)heads, st);
  if (path == PATH_LINEAR_WIDE) return linear_wide_launch(a, (int)heads, st);
  if (path == PATH_LINEAR_CHUNK) {
    const size_t need = linear_chunk_workspace_bytes(a, (int)heads);
    if (!cfg->workspace || cfg->workspace_bytes < need) return ATLAS_ERR_WORKSPACE;
    return linear_chunk_forward(a, (int)heads, cfg->workspace, st);
  }
  return linear_simt_launch(a, (int)heads, st);
}

namespace {

// Structural checks of a backward description (no pointers).
int backward_plan(const atlas_mem_cfg* cfg, LinArgs* out) {
  const int rc = check_cfg(cfg);
  if (rc != ATLAS_OK) return rc;
  if (cfg->mem != ATLAS_MEM_LINEAR || cfg->ns_steps > 0) return ATLAS_ERR_UNSUPPORTED;
  if (cfg->loss != ATLAS_LOSS_L2 && cfg->loss != ATLAS_LOSS_LP && cfg->loss != ATLAS_LOSS_HUBER)
    return ATLAS_ERR_UNSUPPORTED;
  if (cfg->retention != ATLAS_RET_L2) return ATLAS_ERR_UNSUPPORTED;
  *out = lin_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, cfg, nullptr,
                  nullptr);
  return linear_bwd_supported(*out) ? ATLAS_OK : ATLAS_ERR_UNSUPPORTED;
}

}  // namespace

size_t atlas_mem_backward_workspace_bytes(const atlas_mem_cfg* cfg) {
  LinArgs a;
  if (backward_plan(cfg, &a) != ATLAS_OK) return (size_t)-1;
  return linear_bwd_workspace_bytes(a, cfg->B * cfg->H);
}

int atlas_mem_backward(const void* K, const void* Q, const void* V, const float* alpha,
                       const float* eta, const float* theta, const float* gamma,
                       const atlas_mem_cfg* cfg, const float* M0, const float* dY, float* dM,
                       float* dK, float* dQ, float* dV, float* dalpha, float* deta,
                       float* dtheta, void* stream) {
  LinArgs a;
  const int rc = backward_plan(cfg, &a);
  if (rc != ATLAS_OK) return rc;
  const long heads = (long)cfg->B * cfg->H;
  if (heads == 0) return ATLAS_OK;
  if (!M0 || !dM || !gamma) return ATLAS_ERR_INVALID;
  if (cfg->N > 0 && (!K || !Q || !V || !alpha || !eta || !theta || !dY || !dK || !dQ || !dV ||
                     !dalpha || !deta || !dtheta))
    return ATLAS_ERR_INVALID;
  const size_t need = linear_bwd_workspace_bytes(a, (int)heads);
  if (!cfg->workspace || cfg->workspace_bytes < need) return ATLAS_ERR_WORKSPACE;
  a = lin_args(K, Q, V, alpha, eta, theta, gamma, cfg, nullptr, nullptr);
  return linear_bwd_launch(a, (int)heads, M0, dY, dM, dK, dQ, dV, dalpha, deta, dtheta,
                           cfg->status_dev, cfg->workspace, reinterpret_cast<cudaStream_t>(stream));
}

const char* atlas_mem_strerror(int status) {
  switch (status) {
    case ATLAS_OK: return "ok";
    case ATLAS_ERR_INVALID: return "invalid argument";
    case ATLAS_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATLAS_ERR_WORKSPACE: return "workspace missing or too small";
    case ATLAS_ERR_CUDA: return "CUDA runtime error";
    case ATLAS_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

}  // extern "C"
