// linear_bwd.cu -- backward pass of the chunked update of a linear memory
// (the outer-loop gradients: "논문 리뷰 Google ATLAS", Deep Memory Module --
// the memory is fitted at test time inside, everything that produces k, q, v and
// the gates is trained outside; "It's All Connected (Miras)", Associative Memory
// & Attentional Bias, Remark 2), on CUDA cores in fp32.
//
// Scope: identity feature map, d_k = d_v = 128, chunk b = 64, window c = 1, a
// forward without momentum (eta = 0; the gradient with respect to eta is still
// returned), the l2, l_p or Huber bias.  Loss L = sum_t <dY_t, y_t> + <dM_N, M_N>.
//
// Forward of one chunk from its start state M0 (value row v, feature f; tokens
// n, i = 0..63), as in the tensor-core forward kernel:
//   E[i][v] = bias(T[i][v] - V[i][v]),  T = K M0^T          (the errors)
//   Y[n][v] = a_n (M0 q_n)[v] - 2 sum_{i<=n} C[n][i] E[i][v],  C = W (.) P, P = Q K^T
//   M_end   = a_63 M0 - 2 sum_i wb_i E[i][:]^T k_i,             wb_i = W[63][i]
// with a_n = prod_{l<=n} (1 - alpha_l), W[n][i] = gamma_0 theta_i prod_{l=i+1..n}
// (1 - alpha_l) ("[Paper Review] Titans 논문 이해하기": S_t = -theta_t grad,
// M_t = (1 - alpha_t) M_{t-1} + S_t, y_t = M_t q_t; gradients at the chunk-start
// state, ATLAS review §3.3).  Reverse, given dY and dMe = dL/dM_end:
//   dE = -2 C^T dY - 2 diag(wb) Z,  Z = K dMe^T;   dT = dE (.) bias'(T - V);  dV = -dT
//   dM0 = a_63 dMe + dY^T diag(a) Q + dT^T K                    (becomes the previous dMe)
//   dK  = dT M0 - 2 diag(wb) E dMe + dP^T Q,   dQ = diag(a) dY M0 + dP K
//   dC  = -2 dY E^T,  dP = W (.) dC,  dW = P (.) dC (+ dwb on row 63),
//   dwb_i = -2 sum_v E[i][v] Z[i][v],   da_n = <dY_n, M0 q_n> (+ <dMe, M0> for n = 63)
// and the gate gradients from (da, dW) by scans over the table definitions:
//   U[l][i] = sum_{n>=l} dW[n][i] prod_{m=l+1..n} (1 - alpha_m),   R_l = the same for da,
//   dtheta_i = gamma_0 U[i][i],   dalpha_l = -a_{l-1} R_l - sum_{i<l} W[l-1][i] U[l][i],
//   deta_n = gamma_0 theta_{n-1} U[n][n-1]  (the momentum S_{n-1} = -2 gamma_0
//   theta_{n-1} e_{n-1} k_{n-1}^T that eta_n would carry), and for a chunk's first
//   token the same term with the previous chunk's last token.
//
// The recursion dMe -> dM0 and everything it needs are separable over the value
// rows v; only the outputs dK, dQ, dC, dwb, da sum over v.  So:
//   bwd_tables_kernel  (head x chunk): W, a, P, C and the first-token factors;
//   bwd_rows_kernel    (head x 32-row block): the forward once, keeping every
//                      chunk-start state, then the reverse over the chunks; writes
//                      dV, dM_0 and per-row-block partial sums;
//   bwd_finish_kernel  (head x chunk): sums the partials, dP, the gate scans, dK, dQ.
#include "common.cuh"
#include "kernels.h"
#include "simt_tiles.cuh"

namespace atlas {

namespace {

constexpr int kD = 128;           // d_k = d_v
constexpr int kB = 64;            // chunk
constexpr int kRB = 32;           // value rows per CTA of the recursion kernel
constexpr int kR = kD / kRB;      // row blocks per head
constexpr int kPad = kD + 1;      // padded row stride: state rows, K rows
constexpr int kPadB = kRB + 1;    // padded stride of [token][row] tiles
constexpr int kThreads = 256;

struct BwdArgs {
  const void* K;
  const void* Q;
  const void* V;
  const float* alpha;
  const float* eta;
  const float* theta;
  const float* gamma;
  const float* M0;
  const float* dY;
  float* dM;
  float* dK;
  float* dQ;
  float* dV;
  float* dalpha;
  float* deta;
  float* dtheta;
  int heads, N, nch, bf16, lk;
  float lp;
  int* status;
  // workspace
  float* Mck;  // [heads][nch][kD][kD] chunk-start states
  float* tW;   // [heads][nch][kB][kB] W[n][i]
  float* tP;   // [heads][nch][kB][kB] q_n . k_i
  float* tC;   // [heads][nch][kB][kB] W (.) P
  float* tA;   // [heads][nch][kB] a_n
  float* tR;   // [heads][nch][kB + 1]: r[m][0] (q_m . k_{t0-1}), then r[63][0]
  float* pK;   // [kR][heads][N][kD] partial dK
  float* pQ;   // [kR][heads][N][kD] partial dQ
  float* pC;   // [kR][heads][nch][kB][kB] partial dC
  float* pWb;  // [kR][heads][nch][kB] partial dwb
  float* pA;   // [kR][heads][nch][kB] partial da
  float* pE0;  // [kR][heads][nch] partial <dM_{t0} k_{t0-1}, e_{t0-1}>
};

struct BwdLayout {
  size_t Mck, tW, tP, tC, tA, tR, pK, pQ, pC, pWb, pA, pE0, total;  // float offsets
};

BwdLayout bwd_layout(long heads, long N) {
  const long nch = (N + kB - 1) / kB;
  BwdLayout L;
  size_t o = 0;
  auto take = [&](size_t n) {
    size_t at = o;
    o += (n + 63) & ~(size_t)63;  // 256-byte aligned blocks
    return at;
  };
  L.Mck = take((size_t)heads * nch * kD * kD);
  L.tW = take((size_t)heads * nch * kB * kB);
  L.tP = take((size_t)heads * nch * kB * kB);
  L.tC = take((size_t)heads * nch * kB * kB);
  L.tA = take((size_t)heads * nch * kB);
  L.tR = take((size_t)heads * nch * (kB + 1));
  L.pK = take((size_t)kR * heads * N * kD);
  L.pQ = take((size_t)kR * heads * N * kD);
  L.pC = take((size_t)kR * heads * nch * kB * kB);
  L.pWb = take((size_t)kR * heads * nch * kB);
  L.pA = take((size_t)kR * heads * nch * kB);
  L.pE0 = take((size_t)kR * heads * nch);
  L.total = o;
  return L;
}

// The attentional bias's derivative (in units of the l2 bias's 2e) and its
// derivative: l2 e -> 1; Huber clamp(e, -delta, delta) -> [|e| <= delta];
// l_p (p/2)|e|^(p-1) sign e -> (p/2)(p-1)|e|^(p-2) (0 at e = 0).
__device__ __forceinline__ float bias_grad2(float e, int kind, float prm) {
  if (kind == ATLAS_LOSS_HUBER) return fabsf(e) <= prm ? 1.f : 0.f;
  if (kind == ATLAS_LOSS_LP) {
    if (prm == 2.f) return 1.f;
    const float a = fabsf(e);
    if (a == 0.f) return 0.f;
    const float m = prm == 3.f ? a : exp2f((prm - 2.f) * log2f(a));
    return 0.5f * prm * (prm - 1.f) * m;
  }
  return 1.f;
}

// K, Q rows of chunk j (tokens t0.., zero past N) into fp32 shared memory with
// row strides ldk, ldq.
__device__ __forceinline__ void load_kq(const BwdArgs& p, int h, int t0, int nb, float* sK,
                                        int ldk, float* sQ, int ldq) {
  const long base = ((long)h * p.N + t0) * kD;
  for (int x = threadIdx.x; x < kB * kD; x += kThreads) {
    const int i = x / kD, f = x % kD;
    const bool ok = i < nb;
    sK[i * ldk + f] = ok ? ld_in(p.K, base + x, p.bf16) : 0.f;
    if (sQ) sQ[i * ldq + f] = ok ? ld_in(p.Q, base + x, p.bf16) : 0.f;
  }
}

}  // namespace

// ------------------------------------------------------------ gate tables

__global__ void __launch_bounds__(kThreads) bwd_tables_kernel(BwdArgs p) {
  extern __shared__ float sm[];
  float* sK = sm;                  // [kB][kPad]
  float* sQ = sK + kB * kPad;      // [kB][kD]
  float* sKp = sQ + kB * kD;       // [kD] k_{t0-1}
  float* sAl = sKp + kD;           // [kB] alpha (0 past N)
  float* sTh = sAl + kB;           // [kB] theta (0 past N)
  float* sW = sTh + kB;            // [kB][kB]
  float* sR = sW + kB * kB;        // [kB] r[m][0]
  const int h = blockIdx.x / p.nch, j = blockIdx.x % p.nch;
  const int t0 = j * kB, nb = min(kB, p.N - t0);
  const int tid = threadIdx.x;
  const long g = (long)h * p.N + t0;  // gate index of token t0
  const long cb = (long)h * p.nch + j;
  load_kq(p, h, t0, nb, sK, kPad, sQ, kD);
  if (tid < kD) sKp[tid] = j > 0 ? ld_in(p.K, (g - 1) * kD + tid, p.bf16) : 0.f;
  if (tid < kB) {
    const bool ok = tid < nb;
    sAl[tid] = ok ? p.alpha[g + tid] : 0.f;
    sTh[tid] = ok ? p.theta[g + tid] : 0.f;
    if (ok && p.eta[g + tid] != 0.f && p.status) atomicExch(p.status, ATLAS_ERR_UNSUPPORTED);
  }
  __syncthreads();
  const float g0 = p.gamma[0];
  if (tid < kB) {  // column i of W: W[i][i] = g0 theta_i, then (1 - alpha_n) per step
    const int i = tid;
    float w = 0.f;
    for (int n = 0; n < kB; ++n) {
      if (n == i) w = g0 * sTh[i];
      else if (n > i) w *= 1.f - sAl[n];
      sW[n * kB + i] = n >= i ? w : 0.f;
    }
  } else if (tid == kB) {  // a_n and r[m][0] = prod_{l=1..m} (1 - alpha_l)
    float a = 1.f, r = 1.f;
    for (int n = 0; n < kB; ++n) {
      a *= 1.f - sAl[n];
      if (n > 0) r *= 1.f - sAl[n];
      p.tA[cb * kB + n] = a;
      sR[n] = r;
    }
    p.tR[cb * (kB + 1) + kB] = r;
  }
  __syncthreads();
  {  // P[n][i] = q_n . k_i and C = W (.) P; thread: i = tid % 64, n = tid / 64 + 4 r
    const int i = tid & 63, ng = tid >> 6;
    float acc[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) acc[r] = 0.f;
    for (int f = 0; f < kD; ++f) {
      const float kv = sK[i * kPad + f];
#pragma unroll
      for (int r = 0; r < 16; ++r) acc[r] += sQ[(ng + 4 * r) * kD + f] * kv;
    }
    const long o = cb * kB * kB;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int n = ng + 4 * r;
      const float w = sW[n * kB + i];
      p.tP[o + n * kB + i] = acc[r];
      p.tW[o + n * kB + i] = w;
      p.tC[o + n * kB + i] = w * acc[r];
    }
  }
  if (tid < kB) {  // r[m][0] (q_m . k_{t0-1})
    float s = 0.f;
    for (int f = 0; f < kD; ++f) s += sQ[tid * kD + f] * sKp[f];
    p.tR[cb * (kB + 1) + tid] = sR[tid] * s;
  }
}

// ------------------------------------------------- row-block recursion
//
// Every product of the recursion is a small dense contraction over shared
// memory, computed by register tiles (simt_tiles.cuh): 256 threads as a 16 x 16
// grid, each accumulating a few outputs spaced 16 apart, so a k-step loads a
// handful of operands for several FMAs.  The three phases that share operands
// accumulate their products together.

// t = K M0^T, z = K dMe^T, mq = Q M0^T for the chunk's 64 tokens x 32 rows
// (thread: tokens ty + 16 u, rows tx + 16 v).
template <class FE>
__device__ __forceinline__ void bwd_tile_tzq(const float* sK, const float* sQ, const float* sM0,
                                             const float* sDM, const FE& fe) {
  constexpr int TM = 4, TN = 2;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float at[TM][TN], az[TM][TN], aq[TM][TN];
#pragma unroll
  for (int u = 0; u < TM; ++u)
#pragma unroll
    for (int v = 0; v < TN; ++v) at[u][v] = az[u][v] = aq[u][v] = 0.f;
  for (int f = 0; f < kD; ++f) {
    float k[TM], q[TM], m[TN], d[TN];
#pragma unroll
    for (int u = 0; u < TM; ++u) {
      k[u] = sK[(ty + 16 * u) * kPad + f];
      q[u] = sQ[(ty + 16 * u) * kPad + f];
    }
#pragma unroll
    for (int v = 0; v < TN; ++v) {
      m[v] = sM0[(tx + 16 * v) * kPad + f];
      d[v] = sDM[(tx + 16 * v) * kPad + f];
    }
#pragma unroll
    for (int u = 0; u < TM; ++u)
#pragma unroll
      for (int v = 0; v < TN; ++v) {
        at[u][v] = fmaf(k[u], m[v], at[u][v]);
        az[u][v] = fmaf(k[u], d[v], az[u][v]);
        aq[u][v] = fmaf(q[u], m[v], aq[u][v]);
      }
  }
#pragma unroll
  for (int u = 0; u < TM; ++u)
#pragma unroll
    for (int v = 0; v < TN; ++v) fe(ty + 16 * u, tx + 16 * v, at[u][v], az[u][v], aq[u][v]);
}

// s1 = dT M0, s2 = E dMe, s3 = dY M0 for 64 tokens x 128 features (two column
// blocks of 64; thread: tokens ty + 16 u, features tx + 16 v).
template <class FE>
__device__ __forceinline__ void bwd_tile_kq(const float* sDT, const float* sE, const float* sDY,
                                            const float* sM0, const float* sDM, const FE& fe) {
  constexpr int TM = 4, TN = 4;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int f0 = 0; f0 < kD; f0 += 16 * TN) {
    float s1[TM][TN], s2[TM][TN], s3[TM][TN];
#pragma unroll
    for (int u = 0; u < TM; ++u)
#pragma unroll
      for (int v = 0; v < TN; ++v) s1[u][v] = s2[u][v] = s3[u][v] = 0.f;
    for (int r = 0; r < kRB; ++r) {
      float dt[TM], e[TM], dy[TM], m[TN], d[TN];
#pragma unroll
      for (int u = 0; u < TM; ++u) {
        const int i = ty + 16 * u;
        dt[u] = sDT[i * kPadB + r];
        e[u] = sE[i * kPadB + r];
        dy[u] = sDY[i * kPadB + r];
      }
#pragma unroll
      for (int v = 0; v < TN; ++v) {
        m[v] = sM0[r * kPad + f0 + tx + 16 * v];
        d[v] = sDM[r * kPad + f0 + tx + 16 * v];
      }
#pragma unroll
      for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) {
          s1[u][v] = fmaf(dt[u], m[v], s1[u][v]);
          s2[u][v] = fmaf(e[u], d[v], s2[u][v]);
          s3[u][v] = fmaf(dy[u], m[v], s3[u][v]);
        }
    }
#pragma unroll
    for (int u = 0; u < TM; ++u)
#pragma unroll
      for (int v = 0; v < TN; ++v)
        fe(ty + 16 * u, f0 + tx + 16 * v, s1[u][v], s2[u][v], s3[u][v]);
  }
}

// dMe[v][f] <- a_63 dMe[v][f] + sum_n (a_n dY[n][v] Q[n][f] + dT[n][v] K[n][f])
// (thread: rows ty + 16 u, features tx + 16 v).
__device__ __forceinline__ void bwd_tile_dm(const float* sA, const float* sDY, const float* sDT,
                                            const float* sQ, const float* sK, float* sDM) {
  constexpr int TM = 2, TN = 8;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[TM][TN];
#pragma unroll
  for (int u = 0; u < TM; ++u)
#pragma unroll
    for (int v = 0; v < TN; ++v) acc[u][v] = 0.f;
  for (int n = 0; n < kB; ++n) {
    const float an = sA[n];
    float ay[TM], dt[TM], q[TN], k[TN];
#pragma unroll
    for (int u = 0; u < TM; ++u) {
      ay[u] = an * sDY[n * kPadB + ty + 16 * u];
      dt[u] = sDT[n * kPadB + ty + 16 * u];
    }
#pragma unroll
    for (int v = 0; v < TN; ++v) {
      q[v] = sQ[n * kPad + tx + 16 * v];
      k[v] = sK[n * kPad + tx + 16 * v];
    }
#pragma unroll
    for (int u = 0; u < TM; ++u)
#pragma unroll
      for (int v = 0; v < TN; ++v) acc[u][v] = fmaf(ay[u], q[v], fmaf(dt[u], k[v], acc[u][v]));
  }
  const float a63 = sA[kB - 1];
#pragma unroll
  for (int u = 0; u < TM; ++u)
#pragma unroll
    for (int v = 0; v < TN; ++v) {
      float* x = sDM + (ty + 16 * u) * kPad + tx + 16 * v;
      *x = a63 * *x + acc[u][v];
    }
}

__global__ void __launch_bounds__(kThreads, 1) bwd_rows_kernel(BwdArgs p) {
  extern __shared__ float sm[];
  float* sM0 = sm;                    // [kRB][kPad] state rows
  float* sDM = sM0 + kRB * kPad;      // [kRB][kPad] dMe rows
  float* sK = sDM + kRB * kPad;       // [kB][kPad]
  float* sQ = sK + kB * kPad;         // [kB][kPad]
  float* sV = sQ + kB * kPad;         // [kB][kPadB] V[i][v]
  float* sDY = sV + kB * kPadB;       // [kB][kPadB]
  float* sE = sDY + kB * kPadB;       // [kB][kPadB]
  float* sBP = sE + kB * kPadB;       // [kB][kPadB] bias'
  float* sDT = sBP + kB * kPadB;      // [kB][kPadB]
  float* sZ = sDT + kB * kPadB;       // [kB][kPadB] (K dMe^T)[i][v]
  float* sMq = sZ + kB * kPadB;       // [kB][kPadB] (M0 q_n)[v]
  float* sC = sMq + kB * kPadB;       // [kB][kB]
  float* sA = sC + kB * kB;           // [kB]
  float* sWb = sA + kB;               // [kB]
  float* sRp = sWb + kB;              // [kB + 1]
  float* sKp = sRp + kB + 1;          // [kD]
  float* sX = sKp + kD;               // [kRB]

  const int h = blockIdx.x / kR, rb = blockIdx.x % kR, v0 = rb * kRB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.N, nch = p.nch;
  const long hN = (long)h * N;
  const size_t MS = (size_t)kD * kD;

  for (int x = tid; x < kRB * kD; x += kThreads) {
    const int v = x / kD, f = x % kD;
    sM0[v * kPad + f] = p.M0[(size_t)h * MS + (size_t)(v0 + v) * kD + f];
  }
  // ------------------------------------------------------------ forward
  for (int j = 0; j < nch; ++j) {
    const int t0 = j * kB, nb = min(kB, N - t0);
    const long cb = (long)h * nch + j;
    __syncthreads();
    float* ck = p.Mck + (size_t)cb * MS;
    for (int x = tid; x < kRB * kD; x += kThreads) {
      const int v = x / kD, f = x % kD;
      ck[(size_t)(v0 + v) * kD + f] = sM0[v * kPad + f];
    }
    load_kq(p, h, t0, nb, sK, kPad, nullptr, 0);
    for (int x = tid; x < kB * kRB; x += kThreads) {
      const int i = x / kRB, v = x % kRB;
      sV[i * kPadB + v] = i < nb ? ld_in(p.V, (hN + t0 + i) * kD + v0 + v, p.bf16) : 0.f;
    }
    if (tid < kB) {
      sA[tid] = p.tA[cb * kB + tid];
      sWb[tid] = p.tW[cb * kB * kB + (kB - 1) * kB + tid];
    }
    __syncthreads();
    {  // E[i][v] = wb_i bias(K M0^T - V)
      auto fa = [&](int i, int f) { return sK[i * kPad + f]; };
      auto fb = [&](int f, int v) { return sM0[v * kPad + f]; };
      auto fe = [&](int i, int v, float t) {
        sE[i * kPadB + v] = sWb[i] * bias_grad(t - sV[i * kPadB + v], p.lk, p.lp);
      };
      tile_gemm<16, 4, 2>(kB, kRB, kD, fa, fb, fe);
    }
    __syncthreads();
    {  // M_end[v][f] = a_63 M0[v][f] - 2 sum_i (wb E)[i][v] k_i[f]
      const float a63 = sA[kB - 1];
      auto fa = [&](int v, int i) { return sE[i * kPadB + v]; };
      auto fb = [&](int i, int f) { return sK[i * kPad + f]; };
      auto fe = [&](int v, int f, float s) {
        sM0[v * kPad + f] = a63 * sM0[v * kPad + f] - 2.f * s;
      };
      tile_gemm<16, 2, 8>(kRB, kD, kB, fa, fb, fe);
    }
  }
  // ------------------------------------------------------------ reverse
  __syncthreads();
  for (int x = tid; x < kRB * kD; x += kThreads) {
    const int v = x / kD, f = x % kD;
    sDM[v * kPad + f] = p.dM[(size_t)h * MS + (size_t)(v0 + v) * kD + f];
  }
  bool have_x = false;
  for (int j = nch - 1; j >= 0; --j) {
    const int t0 = j * kB, nb = min(kB, N - t0);
    const long cb = (long)h * nch + j;
    __syncthreads();
    const float* ck = p.Mck + (size_t)cb * MS;
    for (int x = tid; x < kRB * kD; x += kThreads) {
      const int v = x / kD, f = x % kD;
      sM0[v * kPad + f] = ck[(size_t)(v0 + v) * kD + f];
    }
    load_kq(p, h, t0, nb, sK, kPad, sQ, kPad);
    for (int x = tid; x < kB * kRB; x += kThreads) {
      const int i = x / kRB, v = x % kRB;
      const bool ok = i < nb;
      sV[i * kPadB + v] = ok ? ld_in(p.V, (hN + t0 + i) * kD + v0 + v, p.bf16) : 0.f;
      sDY[i * kPadB + v] = ok ? p.dY[(hN + t0 + i) * kD + v0 + v] : 0.f;
    }
    for (int x = tid; x < kB * kB; x += kThreads) sC[x] = p.tC[cb * kB * kB + x];
    if (tid < kB) {
      sA[tid] = p.tA[cb * kB + tid];
      sWb[tid] = p.tW[cb * kB * kB + (kB - 1) * kB + tid];
    }
    if (tid <= kB) sRp[tid] = p.tR[cb * (kB + 1) + tid];
    if (tid < kD) sKp[tid] = j > 0 ? ld_in(p.K, (hN + t0 - 1) * kD + tid, p.bf16) : 0.f;
    __syncthreads();
    // -- T, E, bias'; Z = K dMe^T; Mq = M0 q
    bwd_tile_tzq(sK, sQ, sM0, sDM, [&](int i, int v, float t, float z, float mq) {
      const float e = t - sV[i * kPadB + v];
      sE[i * kPadB + v] = bias_grad(e, p.lk, p.lp);
      sBP[i * kPadB + v] = bias_grad2(e, p.lk, p.lp);
      sZ[i * kPadB + v] = z;
      sMq[i * kPadB + v] = mq;
    });
    __syncthreads();
    if (warp == 0 && have_x) {
      // <dM_{t0'} k_{t0'-1}, e_{t0'-1}> of the chunk after this one (its first
      // token's momentum term), with e_{t0'-1} = this chunk's last error
      const float s = warp_sum(sX[lane] * sE[(kB - 1) * kPadB + lane]);
      if (lane == 0) p.pE0[((size_t)rb * p.heads + h) * nch + j + 1] = s;
    }
    // -- dE, dT, dV (dE = -2 C^T dY - 2 wb Z)
    {
      auto fa = [&](int i, int n) { return sC[n * kB + i]; };
      auto fb = [&](int n, int v) { return sDY[n * kPadB + v]; };
      auto fe = [&](int i, int v, float s) {
        const float dE = -2.f * s - 2.f * sWb[i] * sZ[i * kPadB + v];
        const float dT = dE * sBP[i * kPadB + v];
        sDT[i * kPadB + v] = dT;
        if (i < nb) p.dV[(hN + t0 + i) * kD + v0 + v] = -dT;
      };
      tile_gemm<16, 4, 2>(kB, kRB, kB, fa, fb, fe);
    }
    // -- dwb and da partials (warp: tokens warp + 8 r; lane: row v)
    {
      const size_t pb = ((size_t)rb * p.heads + h) * nch + j;
#pragma unroll 2
      for (int r = 0; r < 8; ++r) {
        const int i = warp + 8 * r;
        const float wbp = warp_sum(sE[i * kPadB + lane] * sZ[i * kPadB + lane]);
        float ap = sDY[i * kPadB + lane] * sMq[i * kPadB + lane];
        if (i == kB - 1) {  // a_63 also scales M0 in M_end
          for (int f = 0; f < kD; ++f) ap += sDM[lane * kPad + f] * sM0[lane * kPad + f];
        }
        ap = warp_sum(ap);
        if (lane == 0) {
          p.pWb[pb * kB + i] = -2.f * wbp;
          p.pA[pb * kB + i] = ap;
        }
      }
    }
    __syncthreads();
    // -- dK, dQ, dC partials; the first token's momentum vector x
    {
      const size_t ob = ((size_t)rb * p.heads + h) * N;
      bwd_tile_kq(sDT, sE, sDY, sM0, sDM, [&](int i, int f, float s1, float s2, float s3) {
        if (i < nb) {
          p.pK[(ob + t0 + i) * kD + f] = s1 - 2.f * sWb[i] * s2;
          p.pQ[(ob + t0 + i) * kD + f] = sA[i] * s3;
        }
      });
      const size_t cbo = (((size_t)rb * p.heads + h) * nch + j) * kB * kB;
      auto fa = [&](int n, int v) { return sDY[n * kPadB + v]; };
      auto fb = [&](int v, int i) { return sE[i * kPadB + v]; };
      auto fe = [&](int n, int i, float s) { p.pC[cbo + n * kB + i] = -2.f * s; };
      tile_gemm<16, 4, 4>(kB, kB, kRB, fa, fb, fe);
      if (warp == 0) {
        // x[v] = (dM_{t0} k_{t0-1})[v]: dM_{t0} = sum_m r[m][0] dy_m q_m^T + r[63][0] dMe
        float s = 0.f;
        for (int m = 0; m < kB; ++m) s += sRp[m] * sDY[m * kPadB + lane];
        float z = 0.f;
        for (int f2 = 0; f2 < kD; ++f2) z += sDM[lane * kPad + f2] * sKp[f2];
        sX[lane] = s + sRp[kB] * z;
      }
    }
    have_x = j > 0;
    __syncthreads();
    // -- dMe <- a_63 dMe + dY^T diag(a) Q + dT^T K
    bwd_tile_dm(sA, sDY, sDT, sQ, sK, sDM);
  }
  __syncthreads();
  for (int x = tid; x < kRB * kD; x += kThreads) {
    const int v = x / kD, f = x % kD;
    p.dM[(size_t)h * MS + (size_t)(v0 + v) * kD + f] = sDM[v * kPad + f];
  }
}

// ------------------------------------------------------------- finish

__global__ void __launch_bounds__(kThreads) bwd_finish_kernel(BwdArgs p) {
  extern __shared__ float sm[];
  float* sK = sm;                 // [kB][kD]
  float* sQ = sK + kB * kD;       // [kB][kD]
  float* sW = sQ + kB * kD;       // [kB][kB]
  float* sU = sW + kB * kB;       // [kB][kB]  dW, then U
  float* sDP = sU + kB * kB;      // [kB][kB]
  float* sAl = sDP + kB * kB;     // [kB]
  float* sTh = sAl + kB;          // [kB]
  float* sA = sTh + kB;           // [kB]
  float* sDa = sA + kB;           // [kB]
  float* sRs = sDa + kB;          // [kB]
  const int h = blockIdx.x / p.nch, j = blockIdx.x % p.nch;
  const int t0 = j * kB, nb = min(kB, p.N - t0);
  const int tid = threadIdx.x;
  const long g = (long)h * p.N + t0;
  const long cb = (long)h * p.nch + j;
  const size_t cbo = (size_t)cb * kB * kB;
  load_kq(p, h, t0, nb, sK, kD, sQ, kD);
  for (int x = tid; x < kB * kB; x += kThreads) {
    const int n = x / kB, i = x % kB;
    float dc = 0.f;
#pragma unroll
    for (int rb = 0; rb < kR; ++rb)
      dc += p.pC[(((size_t)rb * p.heads + h) * p.nch + j) * kB * kB + x];
    const float w = p.tW[cbo + x];
    sW[x] = w;
    const bool low = i <= n;
    sDP[x] = low ? w * dc : 0.f;
    sU[x] = low ? p.tP[cbo + x] * dc : 0.f;
  }
  if (tid < kB) {
    const bool ok = tid < nb;
    sAl[tid] = ok ? p.alpha[g + tid] : 0.f;
    sTh[tid] = ok ? p.theta[g + tid] : 0.f;
    sA[tid] = p.tA[cb * kB + tid];
    float da = 0.f;
    for (int rb = 0; rb < kR; ++rb) da += p.pA[(((size_t)rb * p.heads + h) * p.nch + j) * kB + tid];
    sDa[tid] = da;
  }
  __syncthreads();
  if (tid < kB) {  // wb is row 63 of W
    float dwb = 0.f;
    for (int rb = 0; rb < kR; ++rb)
      dwb += p.pWb[(((size_t)rb * p.heads + h) * p.nch + j) * kB + tid];
    sU[(kB - 1) * kB + tid] += dwb;
  }
  __syncthreads();
  if (tid < kB) {  // column scans: U[n][i] = dW[n][i] + (1 - alpha_{n+1}) U[n+1][i]
    const int i = tid;
    float acc = sU[(kB - 1) * kB + i];
    for (int n = kB - 2; n >= i; --n) {
      acc = sU[n * kB + i] + (1.f - sAl[n + 1]) * acc;
      sU[n * kB + i] = acc;
    }
  } else if (tid == kB) {  // R_l = da_l + (1 - alpha_{l+1}) R_{l+1}
    float acc = sDa[kB - 1];
    sRs[kB - 1] = acc;
    for (int l = kB - 2; l >= 0; --l) {
      acc = sDa[l] + (1.f - sAl[l + 1]) * acc;
      sRs[l] = acc;
    }
  }
  __syncthreads();
  const float g0 = p.gamma[0];
  if (tid < nb) {
    const int l = tid;
    p.dtheta[g + l] = g0 * sU[l * kB + l];
    float de;
    if (l > 0) {
      de = g0 * sTh[l - 1] * sU[l * kB + l - 1];
    } else if (j > 0) {
      float s = 0.f;
      for (int rb = 0; rb < kR; ++rb) s += p.pE0[((size_t)rb * p.heads + h) * p.nch + j];
      de = -2.f * g0 * p.theta[g - 1] * s;
    } else {
      de = 0.f;  // the momentum before the first token is zero
    }
    p.deta[g + l] = de;
    float da = -(l > 0 ? sA[l - 1] : 1.f) * sRs[l];
    for (int i = 0; i < l; ++i) da -= sW[(l - 1) * kB + i] * sU[l * kB + i];
    p.dalpha[g + l] = da;
  }
  {  // dK[i] = sum of partials + sum_n dP[n][i] q_n; dQ[n] = ... + sum_i dP[n][i] k_i
    const int f = tid & (kD - 1), ig = tid >> 7;
    for (int r = 0; r < kB / 2; ++r) {
      const int i = ig + 2 * r;
      if (i >= nb) continue;
      float sk = 0.f, sq = 0.f;
      for (int n = 0; n < kB; ++n) {
        sk += sDP[n * kB + i] * sQ[n * kD + f];
        sq += sDP[i * kB + n] * sK[n * kD + f];
      }
      for (int rb = 0; rb < kR; ++rb) {
        const size_t o = (((size_t)rb * p.heads + h) * p.N + t0 + i) * kD + f;
        sk += p.pK[o];
        sq += p.pQ[o];
      }
      p.dK[(g + i) * kD + f] = sk;
      p.dQ[(g + i) * kD + f] = sq;
    }
  }
}

// ---------------------------------------------------------------- host

namespace {

constexpr size_t kTablesSmem = sizeof(float) * ((size_t)kB * kPad + kB * kD + kD + 2 * kB +
                                                kB * kB + kB);
constexpr size_t kRowsSmem = sizeof(float) * ((size_t)2 * kRB * kPad + 2 * kB * kPad +
                                              7 * kB * kPadB + kB * kB + 3 * kB + 1 + kD + kRB);
constexpr size_t kFinishSmem = sizeof(float) * ((size_t)2 * kB * kD + 3 * kB * kB + 5 * kB);

}  // namespace

bool linear_bwd_supported(const LinArgs& a) {
  return a.d_k == kD && a.d_v == kD && a.D == kD && a.b == kB && a.c == 1 && !a.poly && !a.dot &&
         !a.pgen && a.ret == ATLAS_RET_L2 && a.lk != ATLAS_LOSS_ROBUST &&
         a.nh == 0 && a.S == nullptr;
}

size_t linear_bwd_workspace_bytes(const LinArgs& a, int heads) {
  return bwd_layout(heads, a.N).total * sizeof(float);
}

int linear_bwd_launch(const LinArgs& a, int heads, const float* M0, const float* dY, float* dM,
                      float* dK, float* dQ, float* dV, float* dalpha, float* deta, float* dtheta,
                      int* status, void* ws, cudaStream_t st) {
  if (!linear_bwd_supported(a)) return ATLAS_ERR_UNSUPPORTED;
  if (heads == 0 || a.N == 0) return ATLAS_OK;
  const BwdLayout L = bwd_layout(heads, a.N);
  float* w = reinterpret_cast<float*>(ws);
  BwdArgs p;
  p.K = a.K; p.Q = a.Q; p.V = a.V;
  p.alpha = a.alpha; p.eta = a.eta; p.theta = a.theta; p.gamma = a.gamma;
  p.M0 = M0; p.dY = dY; p.dM = dM; p.dK = dK; p.dQ = dQ; p.dV = dV;
  p.dalpha = dalpha; p.deta = deta; p.dtheta = dtheta;
  p.heads = heads; p.N = a.N; p.nch = (a.N + kB - 1) / kB; p.bf16 = a.bf16;
  p.lk = a.lk; p.lp = a.lp; p.status = status;
  p.Mck = w + L.Mck; p.tW = w + L.tW; p.tP = w + L.tP; p.tC = w + L.tC; p.tA = w + L.tA;
  p.tR = w + L.tR; p.pK = w + L.pK; p.pQ = w + L.pQ; p.pC = w + L.pC; p.pWb = w + L.pWb;
  p.pA = w + L.pA; p.pE0 = w + L.pE0;
  if (cudaFuncSetAttribute(bwd_tables_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kTablesSmem) != cudaSuccess ||
      cudaFuncSetAttribute(bwd_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kRowsSmem) != cudaSuccess ||
      cudaFuncSetAttribute(bwd_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kFinishSmem) != cudaSuccess)
    return ATLAS_ERR_CUDA;
  const int cells = heads * p.nch;
  bwd_tables_kernel<<<cells, kThreads, kTablesSmem, st>>>(p);
  bwd_rows_kernel<<<heads * kR, kThreads, kRowsSmem, st>>>(p);
  bwd_finish_kernel<<<cells, kThreads, kFinishSmem, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? ATLAS_OK : ATLAS_ERR_CUDA;
}

}  // namespace atlas
