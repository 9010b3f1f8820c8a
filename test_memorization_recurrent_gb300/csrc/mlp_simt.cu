// mlp_simt.cu -- chunked update of the residual MLP memory
// M(x) = x + W1 GELU(W2 x), host-driven per chunk, every launch batched over
// all heads: the products as batched tensor-core GEMMs (tc_gemm.cu, bf16 hi/lo
// operands, fp32 accumulation, with the GELU / GELU' and elementwise-factor
// epilogues), the elementwise steps and tables on CUDA cores.  Handles any
// window c, chunk b, momentum and the Newton-Schulz-orthogonalised momentum.
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
// linear in S, but S itself still is: within a chunk
//   S_n = eps_n S0 - sum_i U[n,i] G_i,   G_i = 2 [e_i h_i^T | delta_i k_i^T] at M0,
// so every S_n of the chunk is built at once (one product per head and weight
// block, batched over n), N_n = NS(S_n) runs for all (head, n) instances
// together, and with r[n,m] = prod_{l=m+1..n} (1 - alpha_l)
//   M_n = a_n M0 + sum_{m<=n} r[n,m] N_m,
//   zq_n = a_n W2_0 q_n + sum_{m<=n} r[n,m] N2_m q_n,   hq_n = GELU(zq_n),
//   y_n  = q_n + a_n W1_0 hq_n + sum_{m<=n} r[n,m] N1_m hq_n.
// NS uses the Gram matrix of the short side: (X X^T) X = X (X^T X).  These
// batched products run on the tensor cores (tc_gemm.cu, bf16 hi/lo operands).
//
// The layer-normalised memory M(x) = x + LN(W1 GELU(W2 x)) ("It's All Connected
// (Miras)", the Moneta / Yaad / Memora memory; plain LN over the d outputs, no
// scale or shift, 1e-5 under the square root) changes two places.  At the
// chunk-start state the branch output u_i = W1 h_i is normalised per token,
// e_i = k_i + LN(u_i) - v_i, and the error rows are replaced by the gradient
// with respect to u: is (dy - mean(dy) - n mean(dy n)) with n = LN(u), is the
// inverse standard deviation and dy the bias derivative of e; everything after
// that (Delta, the state updates, the readout's intra-chunk terms) uses those rows
// as the plain memory uses its errors.  The readout accumulates u_q for every
// query (no residual) and finishes with y = q + LN(u_q).
//
// The gated memory M(x) = x + W1 (GELU(W2 x) * (W3 x)) ("ATLAS ... (paperlayer)"
// §5, Atlas++: a gated MLP with three linear maps; W3 is d_h x d like W2 and is
// stored after it) has the hidden activation h = GELU(z) * w with z = W2 x,
// w = W3 x, and with dh = E W1 the gradient factors delta = dh * w * GELU'(z) of
// W2 and delta3 = dh * GELU(z) of W3.  W3 is carried like W2 (its readout
// wq = W3_n q decomposes the same way), and Newton-Schulz treats it as a third
// weight block (batched products; the fused kernel takes two blocks).
//
// The robust bias ("It's All Connected (Miras)", #1 Alternative Attentional
// Biases) scales each token's error row e by 1 + Delta / ||e|| (one warp per row;
// for the layer-normalised memory inside the LN error kernel, on e = k + LN(u) - v).
#include <math.h>
#include <string.h>

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

static Gemm gemm0() {
  Gemm g;
  memset(&g, 0, sizeof(g));
  g.alpha = 1.f;
  return g;
}

static TcGemm tc0() {
  TcGemm g;
  memset(&g, 0, sizeof(g));
  g.alpha = 1.f;
  return g;
}

// Every product of the path runs on the tensor cores (tc_gemm.cu, bf16 hi/lo
// operands, fp32 accumulation) with the same epilogue: the elementwise factor,
// accumulation and the GELU / GELU' pair.
static int run_gemm(const Gemm& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0 || g.batch <= 0) return ATLAS_OK;
  TcGemm t = tc0();
  t.M = g.M; t.N = g.N; t.K = g.K; t.batch = g.batch;
  t.A = g.A; t.sAb = g.sAb; t.sAm = g.sAm; t.sAk = g.sAk;
  t.B = g.B; t.sBb = g.sBb; t.sBk = g.sBk; t.sBn = g.sBn;
  t.C = g.C; t.sCb = g.sCb; t.sCm = g.sCm; t.sCn = g.sCn;
  t.alpha = g.alpha;
  t.rowscale = g.rowscale; t.sRb = g.sRb;
  t.emul = g.emul; t.sMb = g.sEb; t.sMm = g.sEm; t.sMn = g.sEn;
  t.accumulate = g.accumulate;
  t.epi = g.epi;
  t.C2 = g.C2; t.sC2b = g.sC2b; t.sC2m = g.sC2m; t.sC2n = g.sC2n;
  return tc_gemm_launch(t, st);
}

// --------------------------------------------------------------- workspace

struct MlpWs {
  long Kw, Vw, E, Qc, H, Gp, Dl, ta, te, tb, U, W, P1, P2, Zq, Gq, Ew, Eu, Dw, Du, X, T1, T2,
      A, nrm, per_head;
  // gated memory: gate w = K W3^T, gated hidden h, E W1, delta3 and its weighted
  // rows, the readout's gate wq (zero-sized otherwise)
  long Wg, Hg, Dh, D3, D3w, D3u, Wq;
  long S;  // S buffer (all heads), when the caller gives none
  // Newton-Schulz, all (head, token) instances of a chunk: S_n / NS iterate,
  // the second iterate, Gram and its square, and the readout products.
  long nsX, nsT, nsA, nsA2, nsP, nsR;
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
  const long gl = a.gated ? L * dh : 0, gb = a.gated ? b * dh : 0;
  w.Wg = o; o += gl;
  w.Hg = o; o += gl;
  w.Dh = o; o += gl;
  w.D3 = o; o += gl;
  w.D3w = o; o += gl;
  w.D3u = o; o += gl;
  w.Wq = o; o += gb;
  o = (o + 63) & ~63L;
  w.per_head = o;
  w.S = o * a.heads;
  const long nblk = a.gated ? 3 : 2;
  long total = w.S + (a.S ? 0 : (long)a.heads * nblk * d * dh);
  w.nsX = w.nsT = w.nsA = w.nsA2 = w.nsP = w.nsR = 0;
  if (a.ns_steps > 0) {
    const long inst = (long)a.heads * b, state = nblk * d * dh;
    w.nsX = total; total += inst * state;
    w.nsT = total; total += inst * state;
    w.nsA = total; total += inst * nblk * small * small;
    w.nsA2 = total; total += inst * nblk * small * small;
    w.nsP = total; total += inst * dh * b * (a.gated ? 2 : 1);
    w.nsR = total; total += inst * d * b;
  }
  w.bytes = (size_t)total * sizeof(float);
  return w;
}

size_t mlp_simt_workspace_bytes(const MlpArgs& a) { return mlp_layout(a).bytes; }

// ---------------------------------------------------------- small kernels

// Window lengths whose two running table rows fit in 48 KB of shared memory.
constexpr int kRunSmem = 6144;

// Window and chunk inputs as fp32, E preset to K - V (CTAs (h, y) share head h's
// elements), and the scalar tables (CTA (h, 0), after its share).
__global__ void mlp_gather_kernel(MlpArgs p, MlpWs w, float* ws, int t0, int nb, int i0, int L) {
  const int h = blockIdx.x;
  float* base = ws + h * w.per_head;
  const int d = p.d;
  // K, V: head stride (nh + N) rows, token 0 at row nh (i0 may be negative)
  const long kb = ((long)h * (p.N + p.nh) + p.nh) * d;
  const long qb = (long)h * p.N * d;
  const int g = blockIdx.y * blockDim.x + threadIdx.x, ng = gridDim.y * blockDim.x;
  for (int x = g; x < L * d; x += ng) {
    const float k = ld_in(p.K, kb + (long)i0 * d + x, p.bf16);
    const float v = ld_in(p.V, kb + (long)i0 * d + x, p.bf16);
    base[w.Kw + x] = k;
    base[w.Vw + x] = v;
    base[w.E + x] = k - v;
  }
  for (int x = g; x < nb * d; x += ng)
    base[w.Qc + x] = ld_in(p.Q, qb + (long)t0 * d + x, p.bf16);
  if (blockIdx.y != 0) return;
  {  // every thread of the CTA takes window columns of the tables
    const long gb = (long)h * p.N;
    // U and W rows go to their tables; the running rows live in shared memory
    // when they fit (dynamic size 2 L floats), else in the P1/P2 scratch
    extern __shared__ float run_sm[];
    float* run_u = L <= kRunSmem ? run_sm : base + w.P1;
    float* run_w = L <= kRunSmem ? run_sm + L : base + w.P2;
    chunk_tables(p.alpha + gb, p.eta + gb, p.theta + gb, p.gamma, t0, nb, i0, L, p.c, run_u,
                 run_w, base + w.W, L, base + w.U, base + w.ta, base + w.te, base + w.tb,
                 threadIdx.x, blockDim.x);
  }
}

// Gated memory, window rows: Hg = H * Wg (H = GELU(Z)), in all heads.
__global__ void gate_hidden_kernel(float* ws, long per_head, long Hg, long H, long Wg, long n) {
  float* base = ws + (long)blockIdx.y * per_head;
  for (long x = blockIdx.x * (long)blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x)
    base[Hg + x] = base[H + x] * base[Wg + x];
}

// Gated memory, window rows: from dh = E W1 (in Dh), Delta = dh * w * GELU'(z) and
// Delta3 = dh * GELU(z).
__global__ void gate_grad_kernel(float* ws, long per_head, long Dl, long D3, long Dh, long Wg,
                                 long Gp, long H, long n) {
  float* base = ws + (long)blockIdx.y * per_head;
  for (long x = blockIdx.x * (long)blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x) {
    const float dh = base[Dh + x];
    base[Dl + x] = dh * base[Wg + x] * base[Gp + x];
    base[D3 + x] = dh * base[H + x];
  }
}

// Gated memory, query rows: Zq (holding GELU(zq)) <- GELU(zq) * wq.
__global__ void gate_query_kernel(float* ws, long per_head, long Zq, long Wq, long n) {
  float* base = ws + (long)blockIdx.y * per_head;
  for (long x = blockIdx.x * (long)blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x)
    base[Zq + x] *= base[Wq + x];
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

// Y rows of the chunk start as the residual q (or 0 when the branch output is
// normalised before the residual is added).
__global__ void copy_q_kernel(const float* ws, long per_head, long Qc, float* Y, long N, int d,
                              int t0, int n_lo, int n_hi, int zero) {
  const int h = blockIdx.x;
  const float* q = ws + h * per_head + Qc;
  for (int x = threadIdx.x; x < (n_hi - n_lo) * d; x += blockDim.x)
    Y[(long)h * N * d + (long)(t0 + n_lo) * d + x] = zero ? 0.f : q[n_lo * d + x];
}

__device__ __forceinline__ float warp_allsum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}

constexpr float kLnEps = 1e-5f;

// Layer-normalised memory, window rows (one warp per row): U holds the branch
// output u = h W1^T at the chunk-start state, E holds k - v.  Leaves in E the
// gradient factor of u, in units of the l2 bias's 2e:
//   n = (u - mean u) is,  is = 1 / sqrt(var u + eps),  e = (k - v) + n,
//   dy = bias'(e),  E <- is (dy - mean(dy) - n mean(dy n)).
__global__ void ln_error_kernel(float* ws, long per_head, long Eo, long Uo, int rows, int d,
                                int kind, float prm) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  float* base = ws + (long)blockIdx.y * per_head;
  float* u = base + Uo + (long)row * d;
  float* e = base + Eo + (long)row * d;
  float s = 0.f;
  for (int j = lane; j < d; j += 32) s += u[j];
  const float mu = warp_allsum(s) / d;
  float v = 0.f;
  for (int j = lane; j < d; j += 32) v += (u[j] - mu) * (u[j] - mu);
  const float is = rsqrtf(warp_allsum(v) / d + kLnEps);
  float rs = 1.f;  // robust bias: the row's scale 1 + Delta / ||e||
  if (kind == ATLAS_LOSS_ROBUST) {
    float ss = 0.f;
    for (int j = lane; j < d; j += 32) {
      const float r = e[j] + (u[j] - mu) * is;
      ss += r * r;
    }
    rs = robust_scale(sqrtf(warp_allsum(ss)), prm);
  }
  float s1 = 0.f, s2 = 0.f;
  for (int j = lane; j < d; j += 32) {
    const float n = (u[j] - mu) * is;
    const float dy = bias_grad(e[j] + n, kind, prm) * rs;
    u[j] = n;
    e[j] = dy;
    s1 += dy;
    s2 += dy * n;
  }
  const float m1 = warp_allsum(s1) / d, m2 = warp_allsum(s2) / d;
  for (int j = lane; j < d; j += 32) e[j] = is * (e[j] - m1 - u[j] * m2);
}

// Layer-normalised memory, query rows of the chunk (one warp per row): Y holds
// the branch output u_q; y = q + LN(u_q).
__global__ void ln_readout_kernel(const float* ws, long per_head, long Qc, float* Y, long N,
                                  int d, int t0, int nb) {
  const int lane = threadIdx.x & 31;
  const int n = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (n >= nb) return;
  const float* q = ws + (long)blockIdx.y * per_head + Qc + (long)n * d;
  float* y = Y + (long)blockIdx.y * N * d + (long)(t0 + n) * d;
  float s = 0.f;
  for (int j = lane; j < d; j += 32) s += y[j];
  const float mu = warp_allsum(s) / d;
  float v = 0.f;
  for (int j = lane; j < d; j += 32) v += (y[j] - mu) * (y[j] - mu);
  const float is = rsqrtf(warp_allsum(v) / d + kLnEps);
  for (int j = lane; j < d; j += 32) y[j] = q[j] + (y[j] - mu) * is;
}

// E <- the attentional bias's derivative of E (in units of the l2 bias's 2e),
// rows of every head.
__global__ void bias_rows_kernel(float* ws, long per_head, long n, int kind, float prm) {
  float* e = ws + (long)blockIdx.y * per_head;
  for (long x = blockIdx.x * (long)blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x)
    e[x] = bias_grad(e[x], kind, prm);
}

// Robust bias: each E row (one token's d coordinates, every head) times
// 1 + Delta / ||row|| (0 for a zero row); one warp per row.
__global__ void robust_rows_kernel(float* ws, long per_head, long Eo, int rows, int d,
                                   float delta) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  float* e = ws + (long)blockIdx.y * per_head + Eo + (long)row * d;
  float ss = 0.f;
  for (int j = lane; j < d; j += 32) ss += e[j] * e[j];
  const float f = robust_scale(sqrtf(warp_allsum(ss)), delta);
  for (int j = lane; j < d; j += 32) e[j] *= f;
}

// X[inst][block] = S[inst][block] / (||S[inst][block]||_F + eps), in place; one
// CTA per (instance, block).
__global__ void ns_normalize_kernel(float* X, long state, long half, float eps) {
  float* x = X + (long)blockIdx.x * state + (long)blockIdx.y * half;
  __shared__ float red[256];
  float acc = 0.f;
  for (long i = threadIdx.x; i < half; i += blockDim.x) acc += x[i] * x[i];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  const float inv = 1.f / (sqrtf(red[0]) + eps);
  for (long i = threadIdx.x; i < half; i += blockDim.x) x[i] *= inv;
}

// Every momentum S_n of a chunk, streamed token by token (the Newton-Schulz
// path needs each one): S_n = eta_n S_{n-1} - theta_n g_n with the window
// gradient g_n = sum_{lag < c} gamma[lag] G_{n-lag}, G_i = 2 a_i b_i^T taken at
// the chunk-start state (a, b: the two factor rows of weight block blk, E and the
// hidden activation for W1, Delta (Delta3) and K for W2 (W3)).  With gamma
// constant over the window, g_{n+1} = g_n + 2 gamma (G_{n+1} - G_{n+1-c}): two
// rank-1 terms per token; otherwise the window is summed afresh for each token.
// One CTA per (128 x 128 tile of a weight block, head); thread (ty, tx) of a
// 16 x 16 grid holds rows ty + 16 u (u < 8) and columns 4 tx + 64 w .. + 3
// (w < 2) of S and g in registers and writes S_n with 16-byte stores.
struct MomStream {
  int ra, cb;              // block shape: rows (the a factor's width), columns (b's)
  long a_off, b_off;       // workspace offsets of the window rows [L][ra], [L][cb]
  long blk_off;            // offset of the block in the state
};

__global__ void __launch_bounds__(256) mom_stream_kernel(MlpArgs p, MlpWs w, const float* ws,
                                                         float* X, MomStream m0, MomStream m1,
                                                         MomStream m2, int nblk, int t0, int nb,
                                                         int i0) {
  const int tiles_per_blk = 4;  // 128 x 512 blocks in 128 x 128 tiles
  const int blk = blockIdx.x / tiles_per_blk, tile = blockIdx.x % tiles_per_blk;
  if (blk >= nblk) return;
  // field by field: a reference to a selected parameter would copy all three to local memory
  MomStream ms;
  ms.ra = blk == 0 ? m0.ra : blk == 1 ? m1.ra : m2.ra;
  ms.cb = blk == 0 ? m0.cb : blk == 1 ? m1.cb : m2.cb;
  ms.a_off = blk == 0 ? m0.a_off : blk == 1 ? m1.a_off : m2.a_off;
  ms.b_off = blk == 0 ? m0.b_off : blk == 1 ? m1.b_off : m2.b_off;
  ms.blk_off = blk == 0 ? m0.blk_off : blk == 1 ? m1.blk_off : m2.blk_off;
  const int h = blockIdx.y;
  const float* base = ws + (long)h * w.per_head;
  const float* A = base + ms.a_off;  // [L][ra]
  const float* B = base + ms.b_off;  // [L][cb]
  const long state = (long)(p.gated ? 3 : 2) * p.d * p.dh;
  // the tile: rows [r0, r0 + 128) of a (ra) and columns [c0, c0 + 128) of b (cb)
  const int r0 = ms.ra > 128 ? 128 * tile : 0, c0 = ms.ra > 128 ? 0 : 128 * tile;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int c = p.c;
  const float* eta = p.eta + (long)h * p.N;
  const float* theta = p.theta + (long)h * p.N;
  bool gconst = true;
  const float g0 = p.gamma[0];
  for (int l = 1; l < c; ++l) gconst &= p.gamma[l] == g0;
  float sv[8][8], gv[8][8];
  const float* S0 = p.S + (long)h * state + ms.blk_off;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int r = r0 + ty + 16 * u;
#pragma unroll
    for (int wq = 0; wq < 2; ++wq) {
      const float4 x = *reinterpret_cast<const float4*>(S0 + (long)r * ms.cb + c0 + 4 * tx + 64 * wq);
      sv[u][4 * wq] = x.x; sv[u][4 * wq + 1] = x.y; sv[u][4 * wq + 2] = x.z; sv[u][4 * wq + 3] = x.w;
    }
  }
  // this thread's parts of the window row li: a (times f) and b
  auto load_row = [&](int li, float f, float* a, float* b) {
#pragma unroll
    for (int u = 0; u < 8; ++u) a[u] = f * A[(long)li * ms.ra + r0 + ty + 16 * u];
#pragma unroll
    for (int wq = 0; wq < 2; ++wq) {
      const float4 x = *reinterpret_cast<const float4*>(B + (long)li * ms.cb + c0 + 4 * tx + 64 * wq);
      b[4 * wq] = x.x; b[4 * wq + 1] = x.y; b[4 * wq + 2] = x.z; b[4 * wq + 3] = x.w;
    }
  };
  auto add_row = [&](const float* a, const float* b) {  // g += a b^T
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int v = 0; v < 8; ++v) gv[u][v] = fmaf(a[u], b[v], gv[u][v]);
  };
  auto window = [&](int t) {  // g = 2 sum over the window of token t
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int v = 0; v < 8; ++v) gv[u][v] = 0.f;
    int i = max(i0, t - c + 1);
    for (; i + 3 <= t; i += 4) {  // four rows' loads in flight before their products
      float a[4][8], b[4][8];
#pragma unroll
      for (int q = 0; q < 4; ++q) load_row(i + q - i0, 2.f * p.gamma[t - i - q], a[q], b[q]);
#pragma unroll
      for (int q = 0; q < 4; ++q) add_row(a[q], b[q]);
    }
    for (; i <= t; ++i) {
      float a[8], b[8];
      load_row(i - i0, 2.f * p.gamma[t - i], a, b);
      add_row(a, b);
    }
  };
  // constant gamma: the rows entering (token t) and leaving (token t - c) the
  // window of token t, loaded one token ahead
  float ain[8], bin[8], aout[8], bout[8];
  bool out_row = false;
  for (int n = 0; n < nb; ++n) {
    const int t = t0 + n;
    if (n == 0 || !gconst) {
      window(t);
    } else {  // slide: token t enters, token t - c leaves (if it was in the window)
      add_row(ain, bin);
      if (out_row) add_row(aout, bout);
    }
    if (gconst && n + 1 < nb) {
      load_row(t + 1 - i0, 2.f * g0, ain, bin);
      out_row = t + 1 - c >= i0;
      if (out_row) load_row(t + 1 - c - i0, -2.f * g0, aout, bout);
    }
    const float et = eta[t], th = theta[t];
    float* Xn = X + ((long)h * nb + n) * state + ms.blk_off;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = r0 + ty + 16 * u;
#pragma unroll
      for (int v = 0; v < 8; ++v) sv[u][v] = et * sv[u][v] - th * gv[u][v];
#pragma unroll
      for (int wq = 0; wq < 2; ++wq)
        *reinterpret_cast<float4*>(Xn + (long)r * ms.cb + c0 + 4 * tx + 64 * wq) =
            make_float4(sv[u][4 * wq], sv[u][4 * wq + 1], sv[u][4 * wq + 2], sv[u][4 * wq + 3]);
    }
  }
}

// out[h][row][col] = S_{nb-1} of head h (the momentum carried to the next chunk).
__global__ void ns_copy_last_kernel(float* S, const float* Sn, long state, int nb) {
  const int h = blockIdx.y;
  const float* src = Sn + ((long)h * nb + nb - 1) * state;
  for (long x = blockIdx.x * blockDim.x + threadIdx.x; x < state;
       x += (long)gridDim.x * blockDim.x)
    S[h * state + x] = src[x];
}

// out[h][n][j] (row stride ld) += sum_{m<=n} r[n,m] Pm[h][m][j][n] with
// r[n,m] = prod_{l=m+1..n} (1 - alpha_l); then optionally GELU.
__global__ void ns_readout_add_kernel(float* out, long out_head, long ld, const float* P,
                                      int rows, int nb, const float* alpha, long N, int t0,
                                      int gelu) {
  const int h = blockIdx.y;
  const long per = (long)rows * nb;
  for (long x = blockIdx.x * blockDim.x + threadIdx.x; x < per;
       x += (long)gridDim.x * blockDim.x) {
    // n fastest: a warp reads consecutive n of one row j of each P_m
    const int n = (int)(x % nb), j = (int)(x / nb);
    const float* ph = P + (long)h * nb * per + (long)j * nb + n;
    // acc_k = (1 - alpha_k) acc_{k-1} + P_k, so acc_n = sum_{m<=n} r[n,m] P_m
    float acc = 0.f;
    for (int k = 0; k <= n; ++k)
      acc = fmaf(1.f - alpha[(long)h * N + t0 + k], acc, ph[(long)k * per]);
    float* o = out + h * out_head + (long)n * ld + j;
    float v = *o + acc;
    if (gelu) v = 0.5f * v * (1.f + erff(v * 0.70710678118654752f));
    *o = v;
  }
}

// M[h] = a_L M[h] + sum_m r[L,m] N_m (L = nb - 1), both weight blocks.
__global__ void ns_state_kernel(float* M, long state, const float* X, int nb, const float* ws,
                                long per_head, long ta, const float* alpha, long N, int t0) {
  const int h = blockIdx.y;
  const float aL = ws[h * per_head + ta + nb - 1];
  for (long x = blockIdx.x * blockDim.x + threadIdx.x; x < state;
       x += (long)gridDim.x * blockDim.x) {
    float acc = 0.f, r = 1.f;
    for (int m = nb - 1; m >= 0; --m) {
      acc += r * X[((long)h * nb + m) * state + x];
      r *= 1.f - alpha[(long)h * N + t0 + m];
    }
    M[h * state + x] = aL * M[h * state + x] + acc;
  }
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
  // the bias kernel on E; the layer-normalised memory instead adds the LN of the
  // error rows and the LN of the readout rows
  long extra = a.ln ? 2 : (a.lk != ATLAS_LOSS_L2 ? 1 : 0);
  // the gated memory: the gate's product, the gated hidden, the gate gradients;
  // without Newton-Schulz the gate's three readout products, its product with
  // GELU(zq), two weighted-row kernels and two state products; with it, the third
  // block's momentum product, its readout product, the add and the product with
  // GELU(zq), three more products per block and step (unfused), and no fusion
  if (a.gated) extra += 3 + (a.ns_steps > 0 ? 5 + 3L * a.ns_steps : 3 + 1 + 2 + 2);
  const bool fused = ns_fused_supported(a.d, a.dh) && !a.gated;
  // the momenta: one streamed launch for 128 x 512 blocks instead of one product per block
  const long mom = (a.d == 128 && a.dh == 512) ? 1 - (a.gated ? 3 : 2) : 0;
  if (a.ns_steps > 0) return 1 + chunks * (extra + mom + (fused ? 16 : 16 + 6L * a.ns_steps));
  return 1 + chunks * (extra + 4 + 1 + 3 + 1 + 4 + 4 + 1 + 4);
}

int mlp_simt_forward(const MlpArgs& p0, void* wsv, cudaStream_t st) {
  MlpArgs p = p0;
  MlpWs w = mlp_layout(p);
  float* ws = reinterpret_cast<float*>(wsv);
  const long d = p.d, dh = p.dh, half = d * dh;
  const long nblk = p.gated ? 3 : 2, state = nblk * half;
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
  float* W3 = p.M + 2 * half;  // gated memory only
  float* S3 = p.S + 2 * half;
  const long PH = w.per_head;
  // the streamed momenta cover the 128 x 512 / 512 x 128 blocks in 128 x 128 tiles
  const bool mom_stream_ok = d == 128 && dh == 512;
  for (int t0 = 0; t0 < p.N; t0 += p.b) {
    const int t1 = min(p.N, t0 + p.b), nb = t1 - t0;
    const int i0 = max(-p.nh, t0 - p.c + 1), L = t1 - i0;  // history rows enter windows
    mlp_gather_kernel<<<dim3(H, 8), 256, L <= kRunSmem ? 2 * L * sizeof(float) : 0, st>>>(
        p, w, ws, t0, nb, i0, L);
    CL();
    // Z = K_w W2^T ; H = GELU(Z), Gp = GELU'(Z)
    Gemm g = gemm0();
    g.batch = H; g.M = L; g.N = (int)dh; g.K = (int)d;
    g.A = ws + w.Kw; g.sAb = PH; g.sAm = d; g.sAk = 1;
    g.B = W2; g.sBb = state; g.sBk = 1; g.sBn = d;
    g.C = ws + w.H; g.sCb = PH; g.sCm = dh; g.sCn = 1;
    g.epi = 1; g.C2 = ws + w.Gp; g.sC2b = PH; g.sC2m = dh; g.sC2n = 1;
    CK(run_gemm(g, st));
    // the hidden activation the rest uses: H, or for the gated memory Hg = H * (K_w W3^T)
    const long hid = p.gated ? w.Hg : w.H;
    if (p.gated) {
      g = gemm0();
      g.batch = H; g.M = L; g.N = (int)dh; g.K = (int)d;
      g.A = ws + w.Kw; g.sAb = PH; g.sAm = d; g.sAk = 1;
      g.B = W3; g.sBb = state; g.sBk = 1; g.sBn = d;
      g.C = ws + w.Wg; g.sCb = PH; g.sCm = dh; g.sCn = 1;
      CK(run_gemm(g, st));
      gate_hidden_kernel<<<ew_grid((long)L * dh, H), 256, 0, st>>>(ws, PH, w.Hg, w.H, w.Wg,
                                                                   (long)L * dh);
      CL();
    }
    // E = (K_w - V_w) + H W1^T  (layer-normalised memory: U = H W1^T into the Ew
    // scratch, which is free until the state carry, then E from U)
    g = gemm0();
    g.batch = H; g.M = L; g.N = (int)d; g.K = (int)dh;
    g.A = ws + hid; g.sAb = PH; g.sAm = dh; g.sAk = 1;
    g.B = W1; g.sBb = state; g.sBk = 1; g.sBn = dh;
    g.C = ws + (p.ln ? w.Ew : w.E); g.sCb = PH; g.sCm = d; g.sCn = 1;
    g.accumulate = p.ln ? 0 : 1;
    CK(run_gemm(g, st));
    if (p.ln) {
      ln_error_kernel<<<dim3((unsigned)((L + 7) / 8), H), 256, 0, st>>>(ws, PH, w.E, w.Ew, L,
                                                                         (int)d, p.lk, p.lp);
      CL();
    } else if (p.lk == ATLAS_LOSS_ROBUST) {  // the robust bias scales whole E rows
      robust_rows_kernel<<<dim3((unsigned)((L + 7) / 8), H), 256, 0, st>>>(ws, PH, w.E, L, (int)d,
                                                                           p.lp);
      CL();
    } else if (p.lk != ATLAS_LOSS_L2) {  // the attentional bias acts on E elementwise
      bias_rows_kernel<<<ew_grid((long)L * d, H), 256, 0, st>>>(ws + w.E, PH, (long)L * d, p.lk,
                                                               p.lp);
      CL();
    }
    // Delta = (E W1) * GELU'(Z)  (gated: dh = E W1, then Delta and Delta3)
    g = gemm0();
    g.batch = H; g.M = L; g.N = (int)dh; g.K = (int)d;
    g.A = ws + w.E; g.sAb = PH; g.sAm = d; g.sAk = 1;
    g.B = W1; g.sBb = state; g.sBk = dh; g.sBn = 1;
    if (!p.gated) {
      g.emul = ws + w.Gp; g.sEb = PH; g.sEm = dh; g.sEn = 1;
    }
    g.C = ws + (p.gated ? w.Dh : w.Dl); g.sCb = PH; g.sCm = dh; g.sCn = 1;
    CK(run_gemm(g, st));
    if (p.gated) {
      gate_grad_kernel<<<ew_grid((long)L * dh, H), 256, 0, st>>>(ws, PH, w.Dl, w.D3, w.Dh, w.Wg,
                                                                 w.Gp, w.H, (long)L * dh);
      CL();
    }

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
      if (p.gated) {  // wq = a (Q W3^T) + beta (Q S3^T) - 2 P1 Delta3 ; Hq = GELU(zq) * wq
        g = gemm0();
        g.batch = H; g.M = nb; g.N = (int)dh; g.K = (int)d;
        g.A = ws + w.Qc; g.sAb = PH; g.sAm = d; g.sAk = 1;
        g.B = W3; g.sBb = state; g.sBk = 1; g.sBn = d;
        g.rowscale = ws + w.ta; g.sRb = PH;
        g.C = ws + w.Wq; g.sCb = PH; g.sCm = dh; g.sCn = 1;
        CK(run_gemm(g, st));
        g.B = S3; g.rowscale = ws + w.tb; g.accumulate = 1;
        CK(run_gemm(g, st));
        g = gemm0();
        g.batch = H; g.M = nb; g.N = (int)dh; g.K = L;
        g.A = ws + w.P1; g.sAb = PH; g.sAm = L; g.sAk = 1;
        g.B = ws + w.D3; g.sBb = PH; g.sBk = dh; g.sBn = 1;
        g.C = ws + w.Wq; g.sCb = PH; g.sCm = dh; g.sCn = 1;
        g.alpha = -2.f; g.accumulate = 1;
        CK(run_gemm(g, st));
        gate_query_kernel<<<ew_grid((long)nb * dh, H), 256, 0, st>>>(ws, PH, w.Zq, w.Wq,
                                                                     (long)nb * dh);
        CL();
      }
      // P2 = W * (Hq H^T)
      g = gemm0();
      g.batch = H; g.M = nb; g.N = L; g.K = (int)dh;
      g.A = ws + w.Zq; g.sAb = PH; g.sAm = dh; g.sAk = 1;
      g.B = ws + hid; g.sBb = PH; g.sBk = 1; g.sBn = dh;
      g.emul = ws + w.W; g.sEb = PH; g.sEm = L; g.sEn = 1;
      g.C = ws + w.P2; g.sCb = PH; g.sCm = L; g.sCn = 1;
      CK(run_gemm(g, st));
      // Y = q + a (Hq W1^T) + beta (Hq S1^T) - 2 P2 E
      copy_q_kernel<<<H, 256, 0, st>>>(ws, PH, w.Qc, p.Y, p.N, (int)d, t0, 0, nb, p.ln);
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
      if (p.ln) {
        ln_readout_kernel<<<dim3((unsigned)((nb + 7) / 8), H), 256, 0, st>>>(ws, PH, w.Qc, p.Y,
                                                                            p.N, (int)d, t0, nb);
        CL();
      }
      // state carry: rows of E and Delta weighted by the last W / U rows
      const long lastW = w.W + (long)(nb - 1) * L, lastU = w.U + (long)(nb - 1) * L;
      dim3 eg = ew_grid((long)L * dh, H);
      scale_rows_kernel<<<eg, 256, 0, st>>>(ws, PH, w.Ew, w.E, lastW, L, (int)d);
      scale_rows_kernel<<<eg, 256, 0, st>>>(ws, PH, w.Eu, w.E, lastU, L, (int)d);
      scale_rows_kernel<<<eg, 256, 0, st>>>(ws, PH, w.Dw, w.Dl, lastW, L, (int)dh);
      scale_rows_kernel<<<eg, 256, 0, st>>>(ws, PH, w.Du, w.Dl, lastU, L, (int)dh);
      if (p.gated) {
        scale_rows_kernel<<<eg, 256, 0, st>>>(ws, PH, w.D3w, w.D3, lastW, L, (int)dh);
        scale_rows_kernel<<<eg, 256, 0, st>>>(ws, PH, w.D3u, w.D3, lastU, L, (int)dh);
      }
      CL();
      state_carry_kernel<<<ew_grid(state, H), 256, 0, st>>>(p.M, p.S, state, ws, PH, w.ta, w.te,
                                                            w.tb, nb - 1);
      CL();
      // W1 += -2 Ew^T H ; S1 += -2 Eu^T H
      g = gemm0();
      g.batch = H; g.M = (int)d; g.N = (int)dh; g.K = L;
      g.A = ws + w.Ew; g.sAb = PH; g.sAm = 1; g.sAk = d;
      g.B = ws + hid; g.sBb = PH; g.sBk = dh; g.sBn = 1;
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
      if (p.gated) {  // W3 += -2 D3w^T K_w ; S3 += -2 D3u^T K_w
        g.A = ws + w.D3w; g.C = W3;
        CK(run_gemm(g, st));
        g.A = ws + w.D3u; g.C = S3;
        CK(run_gemm(g, st));
      }
      continue;
    }

    // Newton-Schulz momentum: every S_n of the chunk, then NS on all of them
    {
      const long sq = d < dh ? (long)d * d : (long)dh * dh;  // Gram of the short side
      const long inst = (long)H * nb;
      float* X = ws + w.nsX;
      float* T = ws + w.nsT;
      float* Ag = ws + w.nsA;
      float* A2 = ws + w.nsA2;
      // S_n = eps_n S0 - 2 sum_i U[n,i] [e_i h_i^T | delta_i k_i^T]: eps_n S0 enters as
      // the products' addend (per-instance factor eps_n of the head's S0)
      if (mom_stream_ok) {  // streamed token by token
        MomStream m[3];
        m[0] = MomStream{(int)d, (int)dh, w.E, hid, 0};
        m[1] = MomStream{(int)dh, (int)d, w.Dl, w.Kw, half};
        m[2] = MomStream{(int)dh, (int)d, w.D3, w.Kw, 2 * half};
        mom_stream_kernel<<<dim3((unsigned)(4 * nblk), (unsigned)H), 256, 0, st>>>(
            p, w, ws, X, m[0], m[1], m[2], (int)nblk, t0, nb, i0);
        CL();
      } else {  // instances (h, n): batch h * nb + n, per-head operands shared over n
        TcGemm t = tc0();
        t.batch = (int)inst; t.bdiv = nb; t.M = (int)d; t.N = (int)dh; t.K = L;
        t.A = ws + w.E; t.sAb = PH; t.sAm = 1; t.sAk = d;
        t.B = ws + hid; t.sBb = PH; t.sBk = dh; t.sBn = 1;
        t.kscale = ws + w.U; t.sKb = PH; t.sKb2 = L;
        t.C = X; t.sCb = (long)nb * state; t.sCb2 = state; t.sCm = dh; t.sCn = 1;
        t.alpha = -2.f;
        t.D = p.S; t.sDb = state; t.sDb2 = 0; t.sDm = dh; t.sDn = 1; t.beta = 1.f;
        t.dscale = ws + w.te; t.sEb = PH; t.sEb2 = 1;
        CK(tc_gemm_launch(t, st));
        t.M = (int)dh; t.N = (int)d;
        t.A = ws + w.Dl; t.sAm = 1; t.sAk = dh;
        t.B = ws + w.Kw; t.sBk = d; t.sBn = 1;
        t.C = X + half; t.sCm = d;
        t.D = p.S + half; t.sDm = d;
        CK(tc_gemm_launch(t, st));
        if (p.gated) {  // the W3 block, from Delta3 like W2 from Delta
          t.A = ws + w.D3;
          t.C = X + 2 * half;
          t.D = p.S + 2 * half;
          CK(tc_gemm_launch(t, st));
        }
      }
      ns_copy_last_kernel<<<ew_grid(state, H), 256, 0, st>>>(p.S, X, state, nb);
      CL();
      // N_n = NS(S_n), per weight block; X0 = S / (||S|| + eps)
      if (ns_fused_supported((int)d, (int)dh) && !p.gated) {  // every instance on chip
        NsArgs n;
        n.X = X; n.inst_stride = state; n.half = half; n.n_inst = (int)inst;
        n.steps = p.ns_steps; n.a = p.ns_a; n.b = p.ns_b; n.c = p.ns_c; n.eps = p.ns_eps;
        n.status = p.status;
        CK(ns_fused_launch(n, st));
      } else {
      ns_normalize_kernel<<<dim3((unsigned)inst, (unsigned)nblk), 256, 0, st>>>(X, state, half,
                                                                                p.ns_eps);
      CL();
      for (int it = 0; it < p.ns_steps; ++it) {
        for (int blk = 0; blk < nblk; ++blk) {
          // block 0: W1 (d x dh); block 1: W2 (dh x d); block 2 (gated): W3 (dh x d);
          // Gram of the short side
          const long rows = blk == 0 ? d : dh, cols = blk == 0 ? dh : d;
          const bool wide = rows <= cols;
          const long sm = wide ? rows : cols;
          const long off = blk * half, aoff = blk * sq;
          TcGemm g1 = tc0();  // G = X X^T (wide) or X^T X (tall)
          g1.batch = (int)inst; g1.M = (int)sm; g1.N = (int)sm; g1.K = (int)(wide ? cols : rows);
          g1.A = X + off; g1.sAb = state;
          g1.B = X + off; g1.sBb = state;
          if (wide) { g1.sAm = cols; g1.sAk = 1; g1.sBk = 1; g1.sBn = cols; }
          else { g1.sAm = 1; g1.sAk = cols; g1.sBk = cols; g1.sBn = 1; }
          g1.C = Ag + aoff; g1.sCb = nblk * sq; g1.sCm = sm; g1.sCn = 1;
          g1.symmetric = sm == 128;  // both operands are the same tile of X
          CK(tc_gemm_launch(g1, st));
          TcGemm g2 = tc0();  // b G + c G^2
          g2.batch = (int)inst; g2.M = (int)sm; g2.N = (int)sm; g2.K = (int)sm;  // G^2
          g2.A = Ag + aoff; g2.sAb = nblk * sq; g2.sAm = sm; g2.sAk = 1;
          g2.B = Ag + aoff; g2.sBb = nblk * sq; g2.sBk = sm; g2.sBn = 1;
          g2.C = A2 + aoff; g2.sCb = nblk * sq; g2.sCm = sm; g2.sCn = 1;
          g2.alpha = p.ns_c;  // b G + c G^2
          g2.D = Ag + aoff; g2.sDb = nblk * sq; g2.sDm = sm; g2.sDn = 1; g2.beta = p.ns_b;
          CK(tc_gemm_launch(g2, st));
          // T = a X + (b G + c G^2) X  (wide)  or  a X + X (b G + c G^2)  (tall)
          TcGemm g3 = tc0();
          g3.batch = (int)inst; g3.M = (int)rows; g3.N = (int)cols;
          g3.C = T + off; g3.sCb = state; g3.sCm = cols; g3.sCn = 1;
          g3.D = X + off; g3.sDb = state; g3.sDm = cols; g3.sDn = 1; g3.beta = p.ns_a;
          if (wide) {
            g3.K = (int)rows;
            g3.A = A2 + aoff; g3.sAb = nblk * sq; g3.sAm = sm; g3.sAk = 1;
            g3.B = X + off; g3.sBb = state; g3.sBk = cols; g3.sBn = 1;
          } else {
            g3.K = (int)cols;
            g3.A = X + off; g3.sAb = state; g3.sAm = cols; g3.sAk = 1;
            g3.B = A2 + aoff; g3.sBb = nblk * sq; g3.sBk = sm; g3.sBn = 1;
          }
          CK(tc_gemm_launch(g3, st));
        }
        float* tmp = X; X = T; T = tmp;
      }
      }
      // readout: zq_n = a_n W2_0 q_n + sum_{m<=n} r[n,m] N2_m q_n -> GELU
      g = gemm0();
      g.batch = H; g.M = nb; g.N = (int)dh; g.K = (int)d;
      g.A = ws + w.Qc; g.sAb = PH; g.sAm = d; g.sAk = 1;
      g.B = W2; g.sBb = state; g.sBk = 1; g.sBn = d;
      g.rowscale = ws + w.ta; g.sRb = PH;
      g.C = ws + w.Zq; g.sCb = PH; g.sCm = dh; g.sCn = 1;
      CK(run_gemm(g, st));
      float* P = ws + w.nsP;
      float* R = ws + w.nsR;
      {
        TcGemm t = tc0();
        t.batch = (int)inst; t.bdiv = nb; t.M = (int)dh; t.N = nb; t.K = (int)d;
        t.A = X + half; t.sAb = (long)nb * state; t.sAb2 = state; t.sAm = d; t.sAk = 1;
        t.B = ws + w.Qc; t.sBb = PH; t.sBk = 1; t.sBn = d;
        t.C = P; t.sCb = (long)nb * dh * nb; t.sCb2 = dh * nb; t.sCm = nb; t.sCn = 1;
        CK(tc_gemm_launch(t, st));
      }
      ns_readout_add_kernel<<<ew_grid((long)nb * dh, H), 256, 0, st>>>(
          ws + w.Zq, PH, dh, P, (int)dh, nb, p.alpha, p.N, t0, 1);
      CL();
      if (p.gated) {  // wq_n = a_n W3_0 q_n + sum_{m<=n} r[n,m] N3_m q_n ; hq = GELU(zq) * wq
        g = gemm0();
        g.batch = H; g.M = nb; g.N = (int)dh; g.K = (int)d;
        g.A = ws + w.Qc; g.sAb = PH; g.sAm = d; g.sAk = 1;
        g.B = W3; g.sBb = state; g.sBk = 1; g.sBn = d;
        g.rowscale = ws + w.ta; g.sRb = PH;
        g.C = ws + w.Wq; g.sCb = PH; g.sCm = dh; g.sCn = 1;
        CK(run_gemm(g, st));
        float* P3 = P + inst * dh * nb;
        TcGemm t = tc0();
        t.batch = (int)inst; t.bdiv = nb; t.M = (int)dh; t.N = nb; t.K = (int)d;
        t.A = X + 2 * half; t.sAb = (long)nb * state; t.sAb2 = state; t.sAm = d; t.sAk = 1;
        t.B = ws + w.Qc; t.sBb = PH; t.sBk = 1; t.sBn = d;
        t.C = P3; t.sCb = (long)nb * dh * nb; t.sCb2 = dh * nb; t.sCm = nb; t.sCn = 1;
        CK(tc_gemm_launch(t, st));
        ns_readout_add_kernel<<<ew_grid((long)nb * dh, H), 256, 0, st>>>(
            ws + w.Wq, PH, dh, P3, (int)dh, nb, p.alpha, p.N, t0, 0);
        CL();
        gate_query_kernel<<<ew_grid((long)nb * dh, H), 256, 0, st>>>(ws, PH, w.Zq, w.Wq,
                                                                     (long)nb * dh);
        CL();
      }
      // y_n = q_n + a_n W1_0 hq_n + sum_{m<=n} r[n,m] N1_m hq_n
      copy_q_kernel<<<H, 256, 0, st>>>(ws, PH, w.Qc, p.Y, p.N, (int)d, t0, 0, nb, p.ln);
      CL();
      g = gemm0();
      g.batch = H; g.M = nb; g.N = (int)d; g.K = (int)dh;
      g.A = ws + w.Zq; g.sAb = PH; g.sAm = dh; g.sAk = 1;
      g.B = W1; g.sBb = state; g.sBk = 1; g.sBn = dh;
      g.rowscale = ws + w.ta; g.sRb = PH;
      g.C = p.Y + (long)t0 * d; g.sCb = (long)p.N * d; g.sCm = d; g.sCn = 1;
      g.accumulate = 1;
      CK(run_gemm(g, st));
      {
        TcGemm t = tc0();
        t.batch = (int)inst; t.bdiv = nb; t.M = (int)d; t.N = nb; t.K = (int)dh;
        t.A = X; t.sAb = (long)nb * state; t.sAb2 = state; t.sAm = dh; t.sAk = 1;
        t.B = ws + w.Zq; t.sBb = PH; t.sBk = 1; t.sBn = dh;
        t.C = R; t.sCb = (long)nb * d * nb; t.sCb2 = d * nb; t.sCm = nb; t.sCn = 1;
        CK(tc_gemm_launch(t, st));
      }
      ns_readout_add_kernel<<<ew_grid((long)nb * d, H), 256, 0, st>>>(
          p.Y + (long)t0 * d, (long)p.N * d, d, R, (int)d, nb, p.alpha, p.N, t0, 0);
      CL();
      if (p.ln) {
        ln_readout_kernel<<<dim3((unsigned)((nb + 7) / 8), H), 256, 0, st>>>(ws, PH, w.Qc, p.Y,
                                                                            p.N, (int)d, t0, nb);
        CL();
      }
      // M = a_L M0 + sum_m r[L,m] N_m (after the readout, which used M0)
      ns_state_kernel<<<ew_grid(state, H), 256, 0, st>>>(p.M, state, X, nb, ws, PH, w.ta,
                                                          p.alpha, p.N, t0);
      CL();
    }
  }
  return ATLAS_OK;
}

}  // namespace atlas
