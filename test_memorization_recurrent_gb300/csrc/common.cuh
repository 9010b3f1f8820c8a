// common.cuh -- small device helpers shared by the memory-update kernels.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "atlas_mem.h"

#define ATLAS_HD __host__ __device__ __forceinline__

// Programmatic dependent launch.  pdl_launch_dependents lets the next kernel on
// the stream, when it was launched with programmatic stream serialisation, be
// scheduled before this grid ends; pdl_wait returns once the grid this one
// depends on has completed and its writes are visible (at once when there is
// none), so everything before it may only touch on-chip state and parameters.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Element t of a K/Q/V tensor stored as fp32 or bf16.
__device__ __forceinline__ float ld_in(const void* p, long idx, int bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[idx]);
  return reinterpret_cast<const float*>(p)[idx];
}

// Attentional bias, per output coordinate with error e = y - v, in units of the
// l2 bias's derivative 2e ("It's All Connected: ...", #1 Alternative Attentional
// Biases): l2 (and the dot product, whose "error" is already -v): e; l_p,
// sum |e|^p: (p/2) |e|^(p-1) sign(e); Huber with threshold delta (per
// coordinate, e^2 inside): e clamped to [-delta, delta].
__device__ __forceinline__ float lp_grad(float e, float p) {
  const float a = fabsf(e);
  float m;  // |e|^(p-1); p is uniform, so the branches cost nothing
  if (p == 3.f)
    m = a * a;
  else if (p == 2.f)
    m = a;
  else
    m = exp2f((p - 1.f) * log2f(a));
  return a == 0.f ? 0.f : copysignf(0.5f * p * m, e);
}
__device__ __forceinline__ float huber_grad(float e, float delta) {
  return fminf(fmaxf(e, -delta), delta);
}
// Half the bias's derivative per coordinate (l2: e).  The robust bias returns e
// here and is finished per token by robust_scale, since it needs ||e||.
__device__ __forceinline__ float bias_grad(float e, int kind, float prm) {
  if (kind == ATLAS_LOSS_LP) return lp_grad(e, prm);
  if (kind == ATLAS_LOSS_HUBER) return huber_grad(e, prm);
  return e;
}
// Robust bias ("It's All Connected (Miras)", #1 Alternative Attentional Biases,
// read as (||e|| + Delta)^2): half its gradient is e (1 + Delta / ||e||), 0 at e = 0.
__device__ __forceinline__ float robust_scale(float norm, float delta) {
  return norm > 0.f ? 1.f + delta / norm : 0.f;
}

// Feature j of Phi(x) for x in shared memory.  Degree-2 map (ATLAS review
// §3.1, constant dropped): j < d -> x_j; otherwise the product x_p x_q of the
// pair (p <= q) in i-major order, looked up in the pair table.
__device__ __forceinline__ float phi_at(const float* x, int j, int d, const uint8_t* pp,
                                        const uint8_t* pq, int poly) {
  if (!poly || j < d) return x[j];
  return x[pp[j - d]] * x[pq[j - d]];
}

// Per-chunk scalar tables of the unrolled momentum / decay recursion.
// Within a chunk with start state (M0, S0) and window gradients G_i taken at
// M0 (i over the L window tokens), for the chunk's n-th token:
//   S_n = eps_n S0 - sum_i U[n,i] G_i,   M_n = a_n M0 + beta_n S0 - sum_i W[n,i] G_i
// with a_n = prod(1-alpha), eps_n = prod(eta), beta_n = (1-alpha_n) beta_{n-1} + eps_n,
// U[n,i] = eta_n U[n-1,i] + theta_n gamma[t_n - t_i] (lag inside the window),
// W[n,i] = (1-alpha_n) W[n-1,i] + U[n,i].
// Threads tid = 0 .. nthr - 1 (whole warps) share the window columns: each column's
// recursion over n belongs to one thread, and every warp loads the gates of 32
// tokens at a time and broadcasts them from lane to lane.  Urun/Wrun are running
// rows of length L; Wt (nb x ldw) receives every W row, Ut every U row (either may
// be null); thread 0 writes a_n, eps_n, beta_n.  The caller synchronises after.
__device__ __forceinline__ void chunk_tables(const float* alpha, const float* eta,
                                             const float* theta, const float* gamma, int t0,
                                             int nb, int i0, int L, int c, float* Urun,
                                             float* Wrun, float* Wt, int ldw, float* Ut,
                                             float* a_out, float* e_out, float* b_out, int tid,
                                             int nthr) {
  const int lane = tid & 31;
  for (int i = tid; i < L; i += nthr) {
    Urun[i] = 0.f;
    Wrun[i] = 0.f;
  }
  float pa = 1.f, pe = 1.f, pb = 0.f;
  float g_keep = 1.f, g_eta = 0.f, g_theta = 0.f;
  for (int n = 0; n < nb; ++n) {
    const int tn = t0 + n;
    if ((n & 31) == 0) {
      const int mine = tn + lane;
      g_keep = mine < t0 + nb ? 1.f - alpha[mine] : 1.f;
      g_eta = mine < t0 + nb ? eta[mine] : 0.f;
      g_theta = mine < t0 + nb ? theta[mine] : 0.f;
    }
    const float keep = __shfl_sync(0xFFFFFFFFu, g_keep, n & 31);
    const float et = __shfl_sync(0xFFFFFFFFu, g_eta, n & 31);
    const float th = __shfl_sync(0xFFFFFFFFu, g_theta, n & 31);
    pa *= keep;
    pe *= et;
    pb = keep * pb + pe;
    for (int i = tid; i < L; i += nthr) {
      const int lag = tn - (i0 + i);
      const float g = (lag >= 0 && lag < c) ? gamma[lag] : 0.f;
      const float u = et * Urun[i] + th * g;
      const float w = keep * Wrun[i] + u;
      Urun[i] = u;
      Wrun[i] = w;
      if (Wt) Wt[n * ldw + i] = w;
      if (Ut) Ut[n * ldw + i] = u;
    }
    if (tid == 0) {
      a_out[n] = pa;
      e_out[n] = pe;
      b_out[n] = pb;
    }
  }
}

// The same tables built by one warp (the caller's lanes).
__device__ __forceinline__ void chunk_tables_warp(const float* alpha, const float* eta,
                                                  const float* theta, const float* gamma,
                                                  int t0, int nb, int i0, int L, int c,
                                                  float* Urun, float* Wrun, float* Wt, int ldw,
                                                  float* Ut, float* a_out, float* e_out,
                                                  float* b_out) {
  chunk_tables(alpha, eta, theta, gamma, t0, nb, i0, L, c, Urun, Wrun, Wt, ldw, Ut, a_out, e_out,
               b_out, threadIdx.x & 31, 32);
  __syncwarp();
}
