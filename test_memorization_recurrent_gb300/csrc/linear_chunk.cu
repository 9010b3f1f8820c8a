// linear_chunk.cu -- chunked update of a linear memory with a wide feature map
// (the degree-2 polynomial map, D = d_k + d_k (d_k + 1) / 2), host-driven per
// chunk, every launch over all heads; the contractions run as batched tcgen05
// GEMMs with bf16 hi/lo operands (tc_gemm.cu).
//
// Per chunk of nb tokens starting at t0, window tokens i0..t1-1 (L of them,
// i0 = max(-n_history, t0-c+1)); "논문 리뷰 Google ATLAS" §3.1 (feature map),
// §3.2 (Omega rule), §3.3 (gradients at the chunk-start state);
// "[Paper Review] Titans 논문 이해하기" (momentum, decay, readout after the write):
//   Phi = [phi(k_i)] (L x D),  E = Phi M0^T - V_w   (dot loss: E = -V_w)
//   P[n,i] = W[n,i] phi(q_n).phi(k_i),   phi(q).phi(k) = s + (s^2 + sum_j (q_j k_j)^2) / 2
//            for the degree-2 map (s = q.k; identity map: s)
//   y_n = a_n M0 phi(q_n) + beta_n S0 phi(q_n) - 2 sum_i P[n,i] e_i
//   M_b = a_b M0 + beta_b S0 - 2 sum_i W[b,i] e_i phi(k_i)^T,  S_b = eps_b S0 - 2 sum_i U[b,i] e_i phi(k_i)^T
// with the scalar tables of the unrolled momentum / decay recursion
// (chunk_tables_warp).
#include <string.h>

#include "common.cuh"
#include "kernels.h"

namespace atlas {

namespace {

struct LcWs {
  long Phi, Vw, E, PhiQ, P, W, U, ta, te, tb, Urun, Wrun, per_head;
  size_t bytes;
  int Lmax;
};

LcWs lc_layout(const LinArgs& a, int heads) {
  LcWs w;
  const long L = a.b + a.c - 1, D = a.D, b = a.b;
  long o = 0;
  w.Lmax = (int)L;
  w.Phi = o; o += L * D;
  w.Vw = o; o += L * a.d_v;
  w.E = o; o += L * a.d_v;
  w.PhiQ = o; o += b * D;
  w.P = o; o += b * L;
  w.W = o; o += b * L;
  w.U = o; o += b * L;
  w.ta = o; o += b;
  w.te = o; o += b;
  w.tb = o; o += b;
  w.Urun = o; o += L;
  w.Wrun = o; o += L;
  o = (o + 63) & ~63L;
  w.per_head = o;
  w.bytes = (size_t)o * heads * sizeof(float);
  return w;
}

constexpr int kMaxPairs = 64 * 65 / 2;  // d_k <= 64

// Feature j of the key / query row x (d_k values): x_j, or x_p x_q for the
// pair (p <= q) number j - d_k in i-major order (pair tables pp, pq).
__device__ __forceinline__ float phi_feature(const float* x, int j, int dk, int poly,
                                             const uint8_t* pp, const uint8_t* pq) {
  if (!poly || j < dk) return x[j];
  return x[pp[j - dk]] * x[pq[j - dk]];
}

// One CTA per (head, slice of the window): features of the window keys and the
// chunk queries, V rows, the tables (first CTA of the head) and the masked
// query-key products.
__global__ void lc_gather_kernel(LinArgs p, LcWs w, float* ws, int t0, int nb, int i0, int L) {
  extern __shared__ float lc_sm[];  // keys of the window [L][d_k], queries [nb][d_k]
  __shared__ uint8_t pp[kMaxPairs], pq[kMaxPairs];
  const int h = blockIdx.y;
  float* base = ws + (long)h * w.per_head;
  const int dk = p.d_k, D = p.D, dv = p.d_v;
  const long kb = ((long)h * (p.N + p.nh) + p.nh) * dk, vb = ((long)h * (p.N + p.nh) + p.nh) * dv;
  const long qb = (long)h * p.N * dk;
  float* Ks = lc_sm;
  float* Qs = Ks + L * dk;
  float* run = Qs + nb * dk;  // running U and W rows of the table recursion [2][L]
  for (int x = threadIdx.x; x < L * dk; x += blockDim.x)
    Ks[x] = ld_in(p.K, kb + (long)i0 * dk + x, p.bf16);
  for (int x = threadIdx.x; x < nb * dk; x += blockDim.x)
    Qs[x] = ld_in(p.Q, qb + (long)t0 * dk + x, p.bf16);
  if (p.poly && threadIdx.x == 32) {
    int o = 0;
    for (int i = 0; i < dk; ++i)
      for (int j = i; j < dk; ++j) {
        pp[o] = (uint8_t)i;
        pq[o] = (uint8_t)j;
        ++o;
      }
  }
  if (blockIdx.x == 0 && threadIdx.x < 32) {  // running rows in shared memory
    const long gb = (long)h * p.N;
    chunk_tables_warp(p.alpha + gb, p.eta + gb, p.theta + gb, p.gamma, t0, nb, i0, L, p.c,
                      run, run + L, base + w.W, L, base + w.U, base + w.ta, base + w.te,
                      base + w.tb);
    for (int i = threadIdx.x; i < L; i += 32) {  // the last rows (for the state update)
      base[w.Urun + i] = run[i];
      base[w.Wrun + i] = run[L + i];
    }
  }
  __syncthreads();
  const long tid = (long)blockIdx.x * blockDim.x + threadIdx.x, nt = (long)gridDim.x * blockDim.x;
  for (long x = tid; x < (long)L * D; x += nt) {
    const int i = (int)(x / D), j = (int)(x % D);
    base[w.Phi + x] = phi_feature(Ks + i * dk, j, dk, p.poly, pp, pq);
  }
  for (long x = tid; x < (long)nb * D; x += nt) {
    const int n = (int)(x / D), j = (int)(x % D);
    base[w.PhiQ + x] = phi_feature(Qs + n * dk, j, dk, p.poly, pp, pq);
  }
  for (long x = tid; x < (long)L * dv; x += nt)
    base[w.Vw + x] = ld_in(p.V, vb + (long)i0 * dv + x, p.bf16);
}

// P[n,i] = W[n,i] phi(q_n).phi(k_i) (after the tables are in place).
__global__ void lc_qk_kernel(LinArgs p, LcWs w, float* ws, int t0, int nb, int i0, int L) {
  const int h = blockIdx.y;
  float* base = ws + (long)h * w.per_head;
  const int dk = p.d_k;
  const long kb = ((long)h * (p.N + p.nh) + p.nh) * dk, qb = (long)h * p.N * dk;
  for (long x = (long)blockIdx.x * blockDim.x + threadIdx.x; x < (long)nb * L;
       x += (long)gridDim.x * blockDim.x) {
    const int n = (int)(x / L), i = (int)(x % L);
    const float wt = base[w.W + n * L + i];
    float v = 0.f;
    if (wt != 0.f) {
      float s = 0.f, s2 = 0.f;
      for (int j = 0; j < dk; ++j) {
        const float qk = ld_in(p.Q, qb + (long)(t0 + n) * dk + j, p.bf16) *
                         ld_in(p.K, kb + (long)(i0 + i) * dk + j, p.bf16);
        s += qk;
        s2 += qk * qk;
      }
      v = wt * (p.poly ? s + 0.5f * (s * s + s2) : s);
    }
    base[w.P + n * L + i] = v;
  }
}

// The chunk's rows of Y set to zero before the split-K readout products add up.
__global__ void lc_zero_rows_kernel(float* Y, long head_stride, long n) {
  float* y = Y + blockIdx.y * head_stride;
  for (long x = blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x)
    y[x] = 0.f;
}

// E = -V_w (the state term is added by the product; the dot loss has none).
__global__ void lc_neg_kernel(float* ws, long per_head, long E, long Vw, long n) {
  float* base = ws + blockIdx.y * per_head;
  for (long x = blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x)
    base[E + x] = -base[Vw + x];
}

// E <- the attentional bias's derivative of E (l_p, Huber), elementwise.
__global__ void lc_bias_kernel(float* ws, long per_head, long E, long n, int kind, float prm) {
  float* e = ws + blockIdx.y * per_head + E;
  for (long x = blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x)
    e[x] = bias_grad(e[x], kind, prm);
}

// M = a_b M + beta_b S, S = eps_b S (the S0 terms of the chunk's last token).
__global__ void lc_carry_kernel(float* M, float* S, long state, const float* ws, long per_head,
                                long ta, long te, long tb, int last) {
  const int h = blockIdx.y;
  const float* base = ws + (long)h * per_head;
  const float a = base[ta + last], e = base[te + last], b = base[tb + last];
  for (long x = blockIdx.x * blockDim.x + threadIdx.x; x < state;
       x += (long)gridDim.x * blockDim.x) {
    const float s0 = S[h * state + x];
    M[h * state + x] = a * M[h * state + x] + b * s0;
    S[h * state + x] = e * s0;
  }
}

TcGemm tc0() {
  TcGemm g;
  memset(&g, 0, sizeof(g));
  g.alpha = 1.f;
  return g;
}

dim3 ew_grid(long n, int heads) {
  long blocks = (n + 255) / 256;
  if (blocks > 128) blocks = 128;
  return dim3((unsigned)blocks, heads);
}

}  // namespace

bool linear_chunk_supported(const LinArgs& a) {
  return !a.pgen && a.ret == ATLAS_RET_L2 && a.lk != ATLAS_LOSS_ROBUST && a.D >= 256 &&
         a.d_v <= 512;
}

size_t linear_chunk_workspace_bytes(const LinArgs& a, int heads) {
  const size_t s = (size_t)heads * a.d_v * a.D * sizeof(float);  // S when none is given
  return lc_layout(a, heads).bytes + (a.S ? 0 : s);
}

long linear_chunk_launch_count(const LinArgs& a, int heads) {
  if (heads <= 0 || a.N <= 0) return 0;
  const long chunks = (a.N + a.b - 1) / a.b;
  const long bias = (a.lk == ATLAS_LOSS_LP || a.lk == ATLAS_LOSS_HUBER) ? 1 : 0;
  return (a.S ? 0 : 1) + chunks * (11 + bias);
}

int linear_chunk_forward(const LinArgs& a0, int heads, void* wsv, cudaStream_t st) {
  LinArgs p = a0;
  const LcWs w = lc_layout(p, heads);
  float* ws = reinterpret_cast<float*>(wsv);
  const int H = heads, D = p.D, dv = p.d_v, dk = p.d_k;
  const long state = (long)dv * D, PH = w.per_head;
  if (!p.S) {
    p.S = ws + PH * H;
    if (cudaMemsetAsync(p.S, 0, sizeof(float) * state * H, st) != cudaSuccess)
      return ATLAS_ERR_CUDA;
  }
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(lc_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             96 * 1024) != cudaSuccess)
      return ATLAS_ERR_CUDA;
    attr = true;
  }
#define LC_CK(x)                       \
  do {                                 \
    int rc_ = (x);                     \
    if (rc_ != ATLAS_OK) return rc_;   \
  } while (0)
#define LC_CL()                                                    \
  do {                                                             \
    if (cudaGetLastError() != cudaSuccess) return ATLAS_ERR_CUDA;  \
  } while (0)
  for (int t0 = 0; t0 < p.N; t0 += p.b) {
    const int t1 = min(p.N, t0 + p.b), nb = t1 - t0;
    const int i0 = max(-p.nh, t0 - p.c + 1), L = t1 - i0;
    const size_t gsm = sizeof(float) * ((size_t)(L + nb) * dk + 2 * L);
    if (gsm > 96 * 1024) return ATLAS_ERR_UNSUPPORTED;
    lc_gather_kernel<<<dim3(8, H), 256, gsm, st>>>(p, w, ws, t0, nb, i0, L);
    LC_CL();
    lc_qk_kernel<<<dim3(8, H), 256, 0, st>>>(p, w, ws, t0, nb, i0, L);
    LC_CL();
    // E = Phi M0^T - V_w: -V_w, then the product over K = D split across CTAs
    const int ks = (D + 127) / 128;
    lc_neg_kernel<<<ew_grid((long)L * dv, H), 256, 0, st>>>(ws, PH, w.E, w.Vw, (long)L * dv);
    LC_CL();
    if (!p.dot) {
      TcGemm g = tc0();
      g.batch = H; g.M = L; g.N = dv; g.K = D; g.ksplit = ks; g.accumulate = 1;
      g.A = ws + w.Phi; g.sAb = PH; g.sAm = D; g.sAk = 1;
      g.B = p.M; g.sBb = state; g.sBk = 1; g.sBn = D;
      g.C = ws + w.E; g.sCb = PH; g.sCm = dv; g.sCn = 1;
      LC_CK(tc_gemm_launch(g, st));
    }
    if (p.lk == ATLAS_LOSS_LP || p.lk == ATLAS_LOSS_HUBER) {
      lc_bias_kernel<<<ew_grid((long)L * dv, H), 256, 0, st>>>(ws, PH, w.E, (long)L * dv, p.lk,
                                                               p.lp);
      LC_CL();
    }
    // y = a (PhiQ M0^T) + beta (PhiQ S0^T) - 2 P E (split K, added onto zeros)
    float* Y = p.Y + (long)t0 * dv;
    lc_zero_rows_kernel<<<ew_grid((long)nb * dv, H), 256, 0, st>>>(Y, (long)p.N * dv,
                                                                    (long)nb * dv);
    LC_CL();
    TcGemm g = tc0();
    g.batch = H; g.M = nb; g.N = dv; g.K = D; g.ksplit = ks; g.accumulate = 1;
    g.A = ws + w.PhiQ; g.sAb = PH; g.sAm = D; g.sAk = 1;
    g.B = p.M; g.sBb = state; g.sBk = 1; g.sBn = D;
    g.rowscale = ws + w.ta; g.sRb = PH;
    g.C = Y; g.sCb = (long)p.N * dv; g.sCm = dv; g.sCn = 1;
    LC_CK(tc_gemm_launch(g, st));
    g.B = p.S; g.rowscale = ws + w.tb;
    LC_CK(tc_gemm_launch(g, st));
    g = tc0();
    g.batch = H; g.M = nb; g.N = dv; g.K = L;
    g.A = ws + w.P; g.sAb = PH; g.sAm = L; g.sAk = 1;
    g.B = ws + w.E; g.sBb = PH; g.sBk = dv; g.sBn = 1;
    g.C = Y; g.sCb = (long)p.N * dv; g.sCm = dv; g.sCn = 1;
    g.alpha = -2.f; g.accumulate = 1;
    LC_CK(tc_gemm_launch(g, st));
    // state at the chunk end: the S0 terms, then the window products
    lc_carry_kernel<<<ew_grid(state, H), 256, 0, st>>>(p.M, p.S, state, ws, PH, w.ta, w.te, w.tb,
                                                      nb - 1);
    LC_CL();
    g = tc0();
    g.batch = H; g.M = dv; g.N = D; g.K = L;
    g.A = ws + w.E; g.sAb = PH; g.sAm = 1; g.sAk = dv;
    g.kscale = ws + w.Wrun; g.sKb = PH;
    g.B = ws + w.Phi; g.sBb = PH; g.sBk = D; g.sBn = 1;
    g.C = p.M; g.sCb = state; g.sCm = D; g.sCn = 1;
    g.alpha = -2.f; g.accumulate = 1;
    LC_CK(tc_gemm_launch(g, st));
    g.kscale = ws + w.Urun;
    g.C = p.S;
    LC_CK(tc_gemm_launch(g, st));
  }
  return ATLAS_OK;
#undef LC_CK
#undef LC_CL
}

}  // namespace atlas
