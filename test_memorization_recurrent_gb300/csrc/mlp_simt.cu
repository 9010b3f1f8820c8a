// mlp_simt.cu -- chunked update of the residual MLP memory
// M(x) = x + W1 GELU(W2 x) on CUDA cores (fp32), host-driven per chunk, every
// launch batched over all heads.  Handles any window c, chunk b, momentum and
// the Newton-Schulz-orthogonalised momentum.
//
// Per chunk (window tokens i0..t1-1, L of them; "논문 리뷰 Google ATLAS" §3.3
// and "It's All Connected (Miras)" Training: gradients at the chunk-start
// state; "ATLAS ... (paperlayer)" App. E: residual 2-layer GELU MLP memory):
//   Z = K_w W2^T, H = GELU(Z), E = K_w + H W1^T - V_w,  Delta = (E W1) * GELU'(Z)
//   (so grad_W1 l_i = 2 e_i h_i^T and grad_W2 l_i = 2 delta_i k_i^T at M0).
// Without Newton-Schulz the whole chunk follows from the scalar tables
// (a, eps, beta, U, W of chunk_tables_warp):
//   z_q = a W2_0 q + beta S2_0 q - 2 sum_i W[n,i] (k_i.q) delta_i,   h_q = GELU(z_q)
//   y   = q + a W1_0 h_q + beta S1_0 h_q - 2 sum_i W[n,i] (h_i.h_q) e_i
//   W1  = a_b W1_0 + beta_b S1_0 - 2 sum_i W[b,i] e_i h_i^T,  S1 = eps_b S1_0 - 2 sum_i U[b,i] e_i h_i^T
//   (W2, S2 likewise with delta_i k_i^T).
// With Newton-Schulz ("ATLAS ... (paperlayer)" §5) the update of M is not
// linear in S, so every token of the chunk is stepped in turn:
//   S = eta S - theta g_n, g_n = 2 sum_j gamma_j [e h^T | delta k^T]_{n-j};
//   W = (1 - alpha) W + NS(S) per weight matrix; y = q + W1 GELU(W2 q).
// NS uses the Gram matrix of the short side: (X X^T) X = X (X^T X).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace atlas {

// ------------------------------------------------------------- batched GEMM

struct Gemm {
  int M, N, K, batch;
  const float* A; long sAb, sAm, sAk;
  const float* B; long sBb, sBk, sBn;
  float* C; long sCb, sCm, sCn;
  float alpha;
  const float* rowscale; long sRb;          // optional per-row factor of the product
  const float* emul; long sEb, sEm, sEn;    // optional elementwise factor of the product
  int accumulate;                           // C += term (else C = term)
  int epi;                                  // 1: C = GELU(C), C2 = GELU'(pre)
  float* C2; long sC2b, sC2m, sC2n;
};

__device__ __forceinline__ float gelu_f(float x) {
  return 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
}
__device__ __forceinline__ float gelu_prime_f(float x) {
  return 0.5f * (1.f + erff(x * 0.70710678118654752f)) +
         x * 0.39894228040143268f * expf(-0.5f * x * x);
}

constexpr int GT = 64, GK = 16;

__global__ void __launch_bounds__(256) gemm_kernel(Gemm g) {
  __shared__ float As[GK][GT + 1];
  __shared__ float Bs[GK][GT + 1];
  const int bz = blockIdx.z;
  const int m0 = blockIdx.y * GT, n0 = blockIdx.x * GT;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const float* A = g.A + bz * g.sAb;
  const float* B = g.B + bz * g.sBb;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < g.K; k0 += GK) {
    for (int x = threadIdx.x; x < GK * GT; x += 256) {
      const int kk = x / GT, mm = x % GT;
      const int m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < g.M && k < g.K) ? A[m * g.sAm + k * g.sAk] : 0.f;
      const int n = n0 + mm;
      Bs[kk][mm] = (n < g.N && k < g.K) ? B[k * g.sBk + n * g.sBn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < GK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        a[u] = As[kk][ty + 16 * u];
        b[u] = Bs[kk][tx + 16 * u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] += a[u] * b[v];
    }
    __syncthreads();
  }
  float* C = g.C + bz * g.sCb;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int m = m0 + ty + 16 * u;
    if (m >= g.M) continue;
    const float rs = g.rowscale ? g.rowscale[bz * g.sRb + m] : 1.f;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int n = n0 + tx + 16 * v;
      if (n >= g.N) continue;
      float t = g.alpha * rs * acc[u][v];
      if (g.emul) t *= g.emul[bz * g.sEb + m * g.sEm + n * g.sEn];
      float* c = C + m * g.sCm + n * g.sCn;
      const float pre = g.accumulate ? *c + t : t;
      if (g.epi == 1) {
        *c = gelu_f(pre);
        if (g.C2) g.C2[bz * g.sC2b + m * g.sC2m + n * g.sC2n] = gelu_prime_f(pre);
      } else {
        *c = pre;
      }
    }
  }
}

static Gemm gemm0() {
  Gemm g;
  memset(&g, 0, sizeof(g));
  g.alpha = 1.f;
  return g;
}

static int run_gemm(const Gemm& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0 || g.batch <= 0) return ATLAS_OK;
  dim3 grid((g.N + GT - 1) / GT, (g.M + GT - 1) / GT, g.batch);
  gemm_kernel<<<grid, 256, 0, st>>>(g);
  return cudaGetLastError() == cudaSuccess ? ATLAS_OK : ATLAS_ERR_CUDA;
}

// --------------------------------------------------------------- workspace

struct MlpWs {
  long Kw, Vw, E, Qc, H, Gp, Dl, ta, te, tb, U, W, P1, P2, Zq, Gq, Ew, Eu, Dw, Du, X, T1, T2,
      A, nrm, per_head;
  long S;  // S buffer (all heads), when the caller gives none
  size_t bytes;
};

static MlpWs mlp_layout(const MlpArgs& a) {
  MlpWs w;
  const long L = a.b + a.c - 1, d = a.d, dh = a.dh, b = a.b;
  const long big = d > dh ? d : dh, small = d < dh ? d : dh;
  long o = 0;
  w.Kw = o; o += L * d;
  w.Vw = o; o += L * d;
  w.E = o; o += L * d;
  w.Qc = o; o += b * d;
  w.H = o; o += L * dh;
  w.Gp = o; o += L * dh;
  w.Dl = o; o += L * dh;
  w.ta = o; o += b;
  w.te = o; o += b;
  w.tb = o; o += b;
  w.U = o; o += b * L;
  w.W = o; o += b * L;
  w.P1 = o; o += b * L;
  w.P2 = o; o += b * L;
  w.Zq = o; o += b * dh;
  w.Gq = o; o += b * dh;
  w.Ew = o; o += L * d;
  w.Eu = o; o += L * d;
  w.Dw = o; o += L * dh;
  w.Du = o; o += L * dh;
  w.X = o; o += big * small;
  w.T1 = o; o += big * small;
  w.T2 = o; o += big * small;
  w.A = o; o += small * small;
  w.nrm = o; o += 4;
  o = (o + 63) & ~63L;
  w.per_head = o;
  w.S = o * a.heads;
  long total = w.S + (a.S ? 0 : (long)a.heads * 2 * d * dh);
  w.bytes = (size_t)total * sizeof(float);
  return w;
}

size_t mlp_simt_workspace_bytes(const MlpArgs& a) { return mlp_layout(a).bytes; }

// ---------------------------------------------------------- small kernels

// Window and chunk inputs as fp32, E preset to K - V, and the scalar tables.
__global__ void mlp_gather_kernel(MlpArgs p, MlpWs w, float* ws, int t0, int nb, int i0, int L) {
  const int h = blockIdx.x;
  float* base = ws + h * w.per_head;
  const int d = p.d;
  const long kb = (long)h * p.N * d;
  for (int x = threadIdx.x; x < L * d; x += blockDim.x) {
    const float k = ld_in(p.K, kb + (long)i0 * d + x, p.bf16);
    const float v = ld_in(p.V, kb + (long)i0 * d + x, p.bf16);
    base[w.Kw + x] = k;
    base[w.Vw + x] = v;
    base[w.E + x] = k - v;
  }
  for (int x = threadIdx.x; x < nb * d; x += blockDim.x)
    base[w.Qc + x] = ld_in(p.Q, kb + (long)t0 * d + x, p.bf16);
  if (threadIdx.x < 32) {
    const long gb = (long)h * p.N;
    // U and W rows go to their tables; the running rows reuse P1/P2 scratch.
    chunk_tables_warp(p.alpha + gb, p.eta + gb, p.theta + gb, p.gamma, t0, nb, i0, L, p.c,
                      base + w.P1, base + w.P2, base + w.W, L, base + w.U, base + w.ta,
                      base + w.te, base + w.tb);
  }
}

// dst[i, :] = s[i] * src[i, :] for the rows of the window (s = last table row).
__global__ void scale_rows_kernel(float* ws, long per_head, long dst, long src, long svec,
                                  int rows, int cols) {
  float* base = ws + blockIdx.y * per_head;
  for (long x = blockIdx.x * blockDim.x + threadIdx.x; x < (long)rows * cols;
       x += (long)gridDim.x * blockDim.x) {
    const int i = (int)(x / cols);
    base[dst + x] = base[svec + i] * base[src + x];
  }
}

// M = a_b M + beta_b S; S = eps_b S (the S0 terms of the chunk's last token).
__global__ void state_carry_kernel(float* M, float* S, long state, const float* ws,
                                   long per_head, long ta, long te, long tb, int last) {
  const int h = blockIdx.y;
  const float* base = ws + h * per_head;
  const float a = base[ta + last], e = base[te + last], b = base[tb + last];
  float* m = M + h * state;
  float* s = S + h * state;
  for (long x = blockIdx.x * blockDim.x + threadIdx.x; x < state;
       x += (long)gridDim.x * blockDim.x) {
    const float s0 = s[x];
    m[x] = a * m[x] + b * s0;
    s[x] = e * s0;
  }
}

// Y rows of the chunk start as the residual q.
__global__ void copy_q_kernel(const float* ws, long per_head, long Qc, float* Y, long N, int d,
                              int t0, int n_lo, int n_hi) {
  const int h = blockIdx.x;
  const float* q = ws + h * per_head + Qc;
  for (int x = threadIdx.x; x < (n_hi - n_lo) * d; x += blockDim.x)
    Y[(long)h * N * d + (long)(t0 + n_lo) * d + x] = q[n_lo * d + x];
}

// S = eta_t S - theta_t g_t with g_t = 2 sum_j gamma_j grad_{t-j} at the
// chunk-start state: [e h^T] on the W1 block, [delta k^T] on the W2 block.
__global__ void ns_momentum_kernel(MlpArgs p, MlpWs w, const float* ws, int t, int i0) {
  const int h = blockIdx.y;
  const float* base = ws + h * w.per_head;
  const long d = p.d, dh = p.dh, half = d * dh;
  const float et = p.eta[(long)h * p.N + t], th = p.theta[(long)h * p.N + t];
  float* S = p.S + h * 2 * half;
  const int j_lo = max(i0, t - p.c + 1);
  for (long x = blockIdx.x * blockDim.x + threadIdx.x; x < 2 * half;
       x += (long)gridDim.x * blockDim.x) {
    float g = 0.f;
    if (x < half) {
      const int r = (int)(x / dh), col = (int)(x % dh);
      for (int i = j_lo; i <= t; ++i)
        g += p.gamma[t - i] * base[w.E + (i - i0) * d + r] * base[w.H + (i - i0) * dh + col];
    } else {
      const long y = x - half;
      const int row = (int)(y / d), col = (int)(y % d);
      for (int i = j_lo; i <= t; ++i)
        g += p.gamma[t - i] * base[w.Dl + (i - i0) * dh + row] * base[w.Kw + (i - i0) * d + col];
    }
    S[x] = et * S[x] - th * 2.f * g;
  }
}

// X = S / (||S||_F + eps) for one weight block of every head.
__global__ void ns_init_kernel(const float* S, long state, long off, long n, float eps, float* ws,
                               long per_head, long X) {
  const int h = blockIdx.x;
  const float* s = S + h * state + off;
  __shared__ float red[256];
  float acc = 0.f;
  for (long x = threadIdx.x; x < n; x += blockDim.x) acc += s[x] * s[x];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  const float inv = 1.f / (sqrtf(red[0]) + eps);
  float* xo = ws + h * per_head + X;
  for (long x = threadIdx.x; x < n; x += blockDim.x) xo[x] = s[x] * inv;
}

// X = a X + b T1 + c T2.
__global__ void ns_combine_kernel(float* ws, long per_head, long X, long T1, long T2, long n,
                                  float a, float b, float c) {
  float* base = ws + blockIdx.y * per_head;
  for (long x = blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x)
    base[X + x] = a * base[X + x] + b * base[T1 + x] + c * base[T2 + x];
}

// W_block = (1 - alpha_t) W_block + X.
__global__ void ns_apply_kernel(float* M, long state, long off, long n, const float* alpha,
                                long N, int t, const float* ws, long per_head, long X) {
  const int h = blockIdx.y;
  const float keep = 1.f - alpha[(long)h * N + t];
  float* m = M + h * state + off;
  const float* xs = ws + h * per_head + X;
  for (long x = blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x)
    m[x] = keep * m[x] + xs[x];
}

// ------------------------------------------------------------- host driver

static dim3 ew_grid(long n, int heads) {
  long blocks = (n + 255) / 256;
  if (blocks > 256) blocks = 256;
  return dim3((unsigned)blocks, heads);
}

#define CK(x)                    \
  do {                           \
    int rc_ = (x);               \
    if (rc_ != ATLAS_OK) return rc_; \
  } while (0)
#define CL()                                                          \
  do {                                                                \
    if (cudaGetLastError() != cudaSuccess) return ATLAS_ERR_CUDA;     \
  } while (0)

long mlp_simt_launch_count(const MlpArgs& a) {
  const long chunks = (a.N + a.b - 1) / a.b;
  if (a.ns_steps > 0) {
    const long per_tok = 1 + 2 * (1 + 3L * a.ns_steps + a.ns_steps + 1) + 1 + 1 + 1;
    return 1 + chunks * 4 + (long)a.N * per_tok;
  }
  return 1 + chunks * (4 + 1 + 3 + 1 + 4 + 4 + 1 + 4);
}

int mlp_simt_forward(const MlpArgs& p0, void* wsv, cudaStream_t st) {
  MlpArgs p = p0;
  MlpWs w = mlp_layout(p);
  float* ws = reinterpret_cast<float*>(wsv);
  const long d = p.d, dh = p.dh, half = d * dh, state = 2 * half;
  const int H = p.heads;
  if (!p.S) {
    p.S = ws + w.S;
    if (cudaMemsetAsync(p.S, 0, sizeof(float) * state * H, st) != cudaSuccess)
      return ATLAS_ERR_CUDA;
  }
  float* W1 = p.M;
  float* W2 = p.M + half;
  float* S1 = p.S;
  float* S2 = p.S + half;
  const long PH = w.per_head;
  for (int t0 = 0; t0 < p.N; t0 += p.b) {
    const int t1 = min(p.N, t0 + p.b), nb = t1 - t0;
    const int i0 = max(0, t0 - p.c + 1), L = t1 - i0;
    mlp_gather_kernel<<<H, 256, 0, st>>>(p, w, ws, t0, nb, i0, L);
    CL();
    // Z = K_w W2^T ; H = GELU(Z), Gp = GELU'(Z)
    Gemm g = gemm0();
    g.batch = H; g.M = L; g.N = (int)dh; g.K = (int)d;
    g.A = ws + w.Kw; g.sAb = PH; g.sAm = d; g.sAk = 1;
    g.B = W2; g.sBb = state; g.sBk = 1; g.sBn = d;
    g.C = ws + w.H; g.sCb = PH; g.sCm = dh; g.sCn = 1;
    g.epi = 1; g.C2 = ws + w.Gp; g.sC2b = PH; g.sC2m = dh; g.sC2n = 1;
    CK(run_gemm(g, st));
    // E = (K_w - V_w) + H W1^T
    g = gemm0();
    g.batch = H; g.M = L; g.N = (int)d; g.K = (int)dh;
    g.A = ws + w.H; g.sAb = PH; g.sAm = dh; g.sAk = 1;
    g.B = W1; g.sBb = state; g.sBk = 1; g.sBn = dh;
    g.C = ws + w.E; g.sCb = PH; g.sCm = d; g.sCn = 1;
    g.accumulate = 1;
    CK(run_gemm(g, st));
    // Delta = (E W1) * GELU'(Z)
    g = gemm0();
    g.batch = H; g.M = L; g.N = (int)dh; g.K = (int)d;
    g.A = ws + w.E; g.sAb = PH; g.sAm = d; g.sAk = 1;
    g.B = W1; g.sBb = state; g.sBk = dh; g.sBn = 1;
    g.emul = ws + w.Gp; g.sEb = PH; g.sEm = dh; g.sEn = 1;
    g.C = ws + w.Dl; g.sCb = PH; g.sCm = dh; g.sCn = 1;
    CK(run_gemm(g, st));

    if (p.ns_steps <= 0) {
      // P1 = W * (Q K_w^T)
      g = gemm0();
      g.batch = H; g.M = nb; g.N = L; g.K = (int)d;
      g.A = ws + w.Qc; g.sAb = PH; g.sAm = d; g.sAk = 1;
      g.B = ws + w.Kw; g.sBb = PH; g.sBk = 1; g.sBn = d;
      g.emul = ws + w.W; g.sEb = PH; g.sEm = L; g.sEn = 1;
      g.C = ws + w.P1; g.sCb = PH; g.sCm = L; g.sCn = 1;
      CK(run_gemm(g, st));
      // Zq = a (Q W2^T) + beta (Q S2^T) - 2 P1 Delta ; Hq = GELU(Zq)
      g = gemm0();
      g.batch = H; g.M = nb; g.N = (int)dh; g.K = (int)d;
      g.A = ws + w.Qc; g.sAb = PH; g.sAm = d; g.sAk = 1;
      g.B = W2; g.sBb = state; g.sBk = 1; g.sBn = d;
      g.rowscale = ws + w.ta; g.sRb = PH;
      g.C = ws + w.Zq; g.sCb = PH; g.sCm = dh; g.sCn = 1;
      CK(run_gemm(g, st));
      g.B = S2; g.rowscale = ws + w.tb; g.accumulate = 1;
      CK(run_gemm(g, st));
      g = gemm0();
      g.batch = H; g.M = nb; g.N = (int)dh; g.K = L;
      g.A = ws + w.P1; g.sAb = PH; g.sAm = L; g.sAk = 1;
      g.B = ws + w.Dl; g.sBb = PH; g.sBk = dh; g.sBn = 1;
      g.C = ws + w.Zq; g.sCb = PH; g.sCm = dh; g.sCn = 1;
      g.alpha = -2.f; g.accumulate = 1; g.epi = 1;
      g.C2 = ws + w.Gq; g.sC2b = PH; g.sC2m = dh; g.sC2n = 1;
      CK(run_gemm(g, st));
      // P2 = W * (Hq H^T)
      g = gemm0();
      g.batch = H; g.M = nb; g.N = L; g.K = (int)dh;
      g.A = ws + w.Zq; g.sAb = PH; g.sAm = dh; g.sAk = 1;
      g.B = ws + w.H; g.sBb = PH; g.sBk = 1; g.sBn = dh;
      g.emul = ws + w.W; g.sEb = PH; g.sEm = L; g.sEn = 1;
      g.C = ws + w.P2; g.sCb = PH; g.sCm = L; g.sCn = 1;
      CK(run_gemm(g, st));
      // Y = q + a (Hq W1^T) + beta (Hq S1^T) - 2 P2 E
      copy_q_kernel<<<H, 256, 0, st>>>(ws, PH, w.Qc, p.Y, p.N, (int)d, t0, 0, nb);
      CL();
      g = gemm0();
      g.batch = H; g.M = nb; g.N = (int)d; g.K = (int)dh;
      g.A = ws + w.Zq; g.sAb = PH; g.sAm = dh; g.sAk = 1;
      g.B = W1; g.sBb = state; g.sBk = 1; g.sBn = dh;
      g.rowscale = ws + w.ta; g.sRb = PH;
      g.C = p.Y + (long)t0 * d; g.sCb = (long)p.N * d; g.sCm = d; g.sCn = 1;
      g.accumulate = 1;
      CK(run_gemm(g, st));
      g.B = S1; g.rowscale = ws + w.tb;
      CK(run_gemm(g, st));
      g = gemm0();
      g.batch = H; g.M = nb; g.N = (int)d; g.K = L;
      g.A = ws + w.P2; g.sAb = PH; g.sAm = L; g.sAk = 1;
      g.B = ws + w.E; g.sBb = PH; g.sBk = d; g.sBn = 1;
      g.C = p.Y + (long)t0 * d; g.sCb = (long)p.N * d; g.sCm = d; g.sCn = 1;
      g.alpha = -2.f; g.accumulate = 1;
      CK(run_gemm(g, st));
      // state carry: rows of E and Delta weighted by the last W / U rows
      const long lastW = w.W + (long)(nb - 1) * L, lastU = w.U + (long)(nb - 1) * L;
      dim3 eg = ew_grid((long)L * dh, H);
      scale_rows_kernel<<<eg, 256, 0, st>>>(ws, PH, w.Ew, w.E, lastW, L, (int)d);
      scale_rows_kernel<<<eg, 256, 0, st>>>(ws, PH, w.Eu, w.E, lastU, L, (int)d);
      scale_rows_kernel<<<eg, 256, 0, st>>>(ws, PH, w.Dw, w.Dl, lastW, L, (int)dh);
      scale_rows_kernel<<<eg, 256, 0, st>>>(ws, PH, w.Du, w.Dl, lastU, L, (int)dh);
      CL();
      state_carry_kernel<<<ew_grid(state, H), 256, 0, st>>>(p.M, p.S, state, ws, PH, w.ta, w.te,
                                                            w.tb, nb - 1);
      CL();
      // W1 += -2 Ew^T H ; S1 += -2 Eu^T H
      g = gemm0();
      g.batch = H; g.M = (int)d; g.N = (int)dh; g.K = L;
      g.A = ws + w.Ew; g.sAb = PH; g.sAm = 1; g.sAk = d;
      g.B = ws + w.H; g.sBb = PH; g.sBk = dh; g.sBn = 1;
      g.C = W1; g.sCb = state; g.sCm = dh; g.sCn = 1;
      g.alpha = -2.f; g.accumulate = 1;
      CK(run_gemm(g, st));
      g.A = ws + w.Eu; g.C = S1;
      CK(run_gemm(g, st));
      // W2 += -2 Dw^T K_w ; S2 += -2 Du^T K_w
      g = gemm0();
      g.batch = H; g.M = (int)dh; g.N = (int)d; g.K = L;
      g.A = ws + w.Dw; g.sAb = PH; g.sAm = 1; g.sAk = dh;
      g.B = ws + w.Kw; g.sBb = PH; g.sBk = d; g.sBn = 1;
      g.C = W2; g.sCb = state; g.sCm = d; g.sCn = 1;
      g.alpha = -2.f; g.accumulate = 1;
      CK(run_gemm(g, st));
      g.A = ws + w.Du; g.C = S2;
      CK(run_gemm(g, st));
      continue;
    }

    // Newton-Schulz momentum: token by token inside the chunk
    for (int n = 0; n < nb; ++n) {
      const int t = t0 + n;
      ns_momentum_kernel<<<ew_grid(state, H), 256, 0, st>>>(p, w, ws, t, i0);
      CL();
      for (int blk = 0; blk < 2; ++blk) {
        const int rows = blk == 0 ? (int)d : (int)dh;
        const int cols = blk == 0 ? (int)dh : (int)d;
        const long off = blk == 0 ? 0 : half;
        const long nel = (long)rows * cols;
        ns_init_kernel<<<H, 256, 0, st>>>(p.S, state, off, nel, p.ns_eps, ws, PH, w.X);
        CL();
        for (int it = 0; it < p.ns_steps; ++it) {
          const bool wide = rows <= cols;
          const int sm = wide ? rows : cols;
          // Gram of the short side
          g = gemm0();
          g.batch = H; g.M = sm; g.N = sm; g.K = wide ? cols : rows;
          g.A = ws + w.X; g.sAb = PH;
          g.B = ws + w.X; g.sBb = PH;
          if (wide) { g.sAm = cols; g.sAk = 1; g.sBk = 1; g.sBn = cols; }
          else { g.sAm = 1; g.sAk = cols; g.sBk = cols; g.sBn = 1; }
          g.C = ws + w.A; g.sCb = PH; g.sCm = sm; g.sCn = 1;
          CK(run_gemm(g, st));
          // T1 = A X (wide) or X A (tall); T2 = A T1 or T1 A
          for (int pass = 0; pass < 2; ++pass) {
            const long src = pass == 0 ? w.X : w.T1;
            const long dst = pass == 0 ? w.T1 : w.T2;
            g = gemm0();
            g.batch = H; g.M = rows; g.N = cols; g.K = sm;
            if (wide) {
              g.A = ws + w.A; g.sAb = PH; g.sAm = sm; g.sAk = 1;
              g.B = ws + src; g.sBb = PH; g.sBk = cols; g.sBn = 1;
            } else {
              g.A = ws + src; g.sAb = PH; g.sAm = cols; g.sAk = 1;
              g.B = ws + w.A; g.sBb = PH; g.sBk = sm; g.sBn = 1;
            }
            g.C = ws + dst; g.sCb = PH; g.sCm = cols; g.sCn = 1;
            CK(run_gemm(g, st));
          }
          ns_combine_kernel<<<ew_grid(nel, H), 256, 0, st>>>(ws, PH, w.X, w.T1, w.T2, nel,
                                                              p.ns_a, p.ns_b, p.ns_c);
          CL();
        }
        ns_apply_kernel<<<ew_grid(nel, H), 256, 0, st>>>(p.M, state, off, nel, p.alpha, p.N, t,
                                                           ws, PH, w.X);
        CL();
      }
      // y_t = q_t + W1 GELU(W2 q_t)
      g = gemm0();
      g.batch = H; g.M = 1; g.N = (int)dh; g.K = (int)d;
      g.A = ws + w.Qc + (long)n * d; g.sAb = PH; g.sAm = d; g.sAk = 1;
      g.B = W2; g.sBb = state; g.sBk = 1; g.sBn = d;
      g.C = ws + w.Zq; g.sCb = PH; g.sCm = dh; g.sCn = 1;
      g.epi = 1;
      CK(run_gemm(g, st));
      copy_q_kernel<<<H, 256, 0, st>>>(ws, PH, w.Qc, p.Y, p.N, (int)d, t0, n, n + 1);
      CL();
      g = gemm0();
      g.batch = H; g.M = 1; g.N = (int)d; g.K = (int)dh;
      g.A = ws + w.Zq; g.sAb = PH; g.sAm = dh; g.sAk = 1;
      g.B = W1; g.sBb = state; g.sBk = 1; g.sBn = dh;
      g.C = p.Y + (long)t * d; g.sCb = (long)p.N * d; g.sCm = d; g.sCn = 1;
      g.accumulate = 1;
      CK(run_gemm(g, st));
    }
  }
  return ATLAS_OK;
}

}  // namespace atlas
