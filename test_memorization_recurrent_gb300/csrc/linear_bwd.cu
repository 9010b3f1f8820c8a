// linear_bwd.cu -- backward pass of the chunked update of a linear memory
// (the outer-loop gradients: "논문 리뷰 Google ATLAS", Deep Memory Module --
// the memory is fitted at test time inside, everything that produces k, q, v and
// the gates is trained outside; "It's All Connected (Miras)", Associative Memory
// & Attentional Bias, Remark 2), on CUDA cores in fp32.
//
// Scope: identity feature map, d_k = d_v = 128, chunk b = 64, window c = 1,
// momentum and decay (any eta, alpha, theta), the momentum starting at zero, the
// l2, l_p or Huber bias.  Loss L = sum_t <dY_t, y_t> + <dM_N, M_N>.
//
// Forward of one chunk from its start state (M0, S0) (value row v, feature f;
// tokens n, i = 0..63), as in the forward kernels ("[Paper Review] Titans 논문
// 이해하기": S_t = eta_t S_{t-1} - theta_t grad, M_t = (1 - alpha_t) M_{t-1} + S_t,
// y_t = M_t q_t; gradients at the chunk-start state, ATLAS review §3.3):
//   E[i][v] = bias(T[i][v] - V[i][v]),  T = K M0^T                       (the errors)
//   Y[n][v] = a_n (M0 q_n)[v] + b_n (S0 q_n)[v] - 2 sum_{i<=n} C[n][i] E[i][v],
//             C = W (.) P, P = Q K^T
//   M_end   = a_63 M0 + b_63 S0 - 2 sum_i wb_i E[i]^T k_i,   wb_i = W[63][i]
//   S_end   = e_63 S0 - 2 sum_i ub_i E[i]^T k_i,             ub_i = U[63][i]
// with the tables a_n = prod_{l<=n} (1 - alpha_l), e_n = prod_{l<=n} eta_l,
// b_n = (1 - alpha_n) b_{n-1} + e_n, U[n][i] = eta_n U[n-1][i] + gamma_0 theta_n [n = i],
// W[n][i] = (1 - alpha_n) W[n-1][i] + U[n][i].  Reverse, given dY, dMe = dL/dM_end and
// dSe = dL/dS_end:
//   dE = -2 C^T dY - 2 diag(wb) Z - 2 diag(ub) Zs,  Z = K dMe^T, Zs = K dSe^T;
//   dT = dE (.) bias'(T - V);  dV = -dT
//   dM0 = a_63 dMe + dY^T diag(a) Q + dT^T K                   (the previous chunk's dMe)
//   dS0 = b_63 dMe + e_63 dSe + dY^T diag(b) Q                 (the previous chunk's dSe)
//   dK  = dT M0 - 2 diag(wb) E dMe - 2 diag(ub) E dSe + dP^T Q
//   dQ  = diag(a) dY M0 + diag(b) dY S0 + dP K
//   dC  = -2 dY E^T,  dP = W (.) dC,  dW = P (.) dC (+ dwb on row 63),  dU = dub on row 63,
//   dwb_i = -2 <E_i, Z_i>,  dub_i = -2 <E_i, Zs_i>,  da_n = <dY_n, M0 q_n>,
//   db_n = <dY_n, S0 q_n> (+ <dMe, M0>, <dMe, S0> on n = 63),  de_63 = <dSe, S0>,
// and the gate gradients from (da, db, de, dW, dU) by one reverse scan over each
// table's recursion.  Tokens past N in the last chunk act with alpha = theta =
// eta = 0, which leaves M unchanged (the momentum after the last token is not
// an output).
//
// The recursion (dMe, dSe) -> (dM0, dS0) and everything it needs are separable
// over the value rows v; only dK, dQ, dC and the table gradients sum over v.  So:
//   bwd_tables_kernel  (head x chunk): the tables, P and C;
//   bwd_rows_kernel    (head x 32-row block): the forward once, keeping every
//                      chunk-start state, then the reverse over the chunks;
//                      writes dV, dM_0 and per-row-block partial sums;
//   bwd_finish_kernel  (head x chunk): sums the gate-term partials, dP, the gate
//                      scans, the dP products of dK and dQ;
//   bwd_partials_kernel (streaming): adds the row-block partials of dK and dQ.
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
  float* Mck;  // [heads][nch][kD][kD] chunk-start M
  float* Sck;  // [heads][nch][kD][kD] chunk-start S
  float* tW;   // [heads][nch][kB][kB] W[n][i]
  float* tU;   // [heads][nch][kB][kB] U[n][i]
  float* tP;   // [heads][nch][kB][kB] q_n . k_i
  float* tC;   // [heads][nch][kB][kB] W (.) P
  float* tA;   // [heads][nch][kB] a_n
  float* tBe;  // [heads][nch][kB] b_n
  float* tEp;  // [heads][nch][kB] e_n
  float* pK;   // [kR][heads][N][kD] partial dK
  float* pQ;   // [kR][heads][N][kD] partial dQ
  float* pC;   // [kR][heads][nch][kB][kB] partial dC
  float* pWb;  // [kR][heads][nch][kB] partial dwb
  float* pUb;  // [kR][heads][nch][kB] partial dub
  float* pA;   // [kR][heads][nch][kB] partial da
  float* pB;   // [kR][heads][nch][kB] partial db
  float* pE;   // [kR][heads][nch] partial de_63
  int* mom;    // [heads] 1 when some eta of the head is non-zero (set by the tables kernel)
};

struct BwdLayout {
  size_t Mck, Sck, tW, tU, tP, tC, tA, tBe, tEp, pK, pQ, pC, pWb, pUb, pA, pB, pE, mom, total;
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
  L.Sck = take((size_t)heads * nch * kD * kD);
  L.tW = take((size_t)heads * nch * kB * kB);
  L.tU = take((size_t)heads * nch * kB * kB);
  L.tP = take((size_t)heads * nch * kB * kB);
  L.tC = take((size_t)heads * nch * kB * kB);
  L.tA = take((size_t)heads * nch * kB);
  L.tBe = take((size_t)heads * nch * kB);
  L.tEp = take((size_t)heads * nch * kB);
  L.pK = take((size_t)kR * heads * N * kD);
  L.pQ = take((size_t)kR * heads * N * kD);
  L.pC = take((size_t)kR * heads * nch * kB * kB);
  L.pWb = take((size_t)kR * heads * nch * kB);
  L.pUb = take((size_t)kR * heads * nch * kB);
  L.pA = take((size_t)kR * heads * nch * kB);
  L.pB = take((size_t)kR * heads * nch * kB);
  L.pE = take((size_t)kR * heads * nch);
  L.mom = take((size_t)heads);  // ints
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

__device__ __forceinline__ void prefetch_l2(const void* a) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
}

// Into L2, ahead of their loads: the inputs of chunk j of head h that this CTA
// (value rows [v0, v0 + kRB)) reads -- K, V and, in the reverse pass (rev), Q,
// dY, the chunk-start state and momentum rows and C.  One 128-byte line each.
__device__ __forceinline__ void prefetch_chunk(const BwdArgs& p, int h, int j, int v0, bool rev) {
  const int t0 = j * kB, nb = min(kB, p.N - t0);
  const int es = p.bf16 ? 2 : 4;
  const long row0 = (long)h * p.N + t0;
  const char* K = reinterpret_cast<const char*>(p.K) + row0 * kD * es;
  const char* Q = reinterpret_cast<const char*>(p.Q) + row0 * kD * es;
  const int lines = nb * kD * es / 128;
  for (int x = threadIdx.x; x < lines; x += kThreads) {
    prefetch_l2(K + 128 * (long)x);
    if (rev) prefetch_l2(Q + 128 * (long)x);
  }
  for (int i = threadIdx.x; i < nb; i += kThreads) {
    prefetch_l2(reinterpret_cast<const char*>(p.V) + ((row0 + i) * kD + v0) * es);
    if (rev) prefetch_l2(p.dY + (row0 + i) * kD + v0);
  }
  if (!rev) return;
  const long cb = (long)h * p.nch + j;
  const size_t MS = (size_t)kD * kD;
  for (int x = threadIdx.x; x < kRB * kD / 32; x += kThreads) {  // 32 floats a line
    const size_t o = cb * MS + (size_t)v0 * kD + 32 * (size_t)x;
    prefetch_l2(p.Mck + o);
    prefetch_l2(p.Sck + o);
  }
  for (int x = threadIdx.x; x < kB * kB / 32; x += kThreads) prefetch_l2(p.tC + cb * kB * kB + 32 * x);
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
  float* sAl = sQ + kB * kD;       // [kB] alpha (0 past N)
  float* sEt = sAl + kB;           // [kB] eta (0 past N)
  float* sTh = sEt + kB;           // [kB] theta (0 past N)
  float* sW = sTh + kB;            // [kB][kB]
  const int h = blockIdx.x / p.nch, j = blockIdx.x % p.nch;
  const int t0 = j * kB, nb = min(kB, p.N - t0);
  const int tid = threadIdx.x;
  const long g = (long)h * p.N + t0;  // gate index of token t0
  const long cb = (long)h * p.nch + j;
  load_kq(p, h, t0, nb, sK, kPad, sQ, kD);
  if (tid < kB) {
    const bool ok = tid < nb;
    sAl[tid] = ok ? p.alpha[g + tid] : 0.f;
    sEt[tid] = ok ? p.eta[g + tid] : 0.f;
    sTh[tid] = ok ? p.theta[g + tid] : 0.f;
    if (sEt[tid] != 0.f) p.mom[h] = 1;
  }
  __syncthreads();
  const float g0 = p.gamma[0];
  if (tid < kB) {  // column i of U and W
    const int i = tid;
    float u = 0.f, w = 0.f;
    const long o = cb * kB * kB;
    for (int n = 0; n < kB; ++n) {
      u = sEt[n] * u + (n == i ? g0 * sTh[n] : 0.f);
      w = (1.f - sAl[n]) * w + u;
      sW[n * kB + i] = w;
      p.tU[o + n * kB + i] = u;
    }
  } else if (tid == kB) {  // a_n, e_n, b_n
    float a = 1.f, e = 1.f, b = 0.f;
    for (int n = 0; n < kB; ++n) {
      a *= 1.f - sAl[n];
      e *= sEt[n];
      b = (1.f - sAl[n]) * b + e;
      p.tA[cb * kB + n] = a;
      p.tEp[cb * kB + n] = e;
      p.tBe[cb * kB + n] = b;
    }
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
      const float w = n >= i ? sW[n * kB + i] : 0.f;
      p.tP[o + n * kB + i] = acc[r];
      p.tW[o + n * kB + i] = w;
      p.tC[o + n * kB + i] = w * acc[r];
    }
  }
}

// ------------------------------------------------- row-block recursion
//
// Every product of the recursion is a small dense contraction over shared
// memory, computed by register tiles (simt_tiles.cuh): 256 threads as a 16 x 16
// grid, each accumulating a few outputs spaced 16 apart, so a k-step loads a
// handful of operands for several FMAs.  Products that share operands
// accumulate together.

// t = K M0^T, z = K dMe^T, zs = K dSe^T, mq = Q M0^T, sq = Q S0^T for the chunk's
// 64 tokens x 32 rows (thread: tokens ty + 16 u, rows tx + 16 v).
template <bool MOM, class FE>
__device__ __forceinline__ void bwd_tile_r1(const float* sK, const float* sQ, const float* sM0,
                                            const float* sS0, const float* sDM, const float* sDS,
                                            const FE& fe) {
  constexpr int TM = 4, TN = 2;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float at[TM][TN], az[TM][TN], azs[TM][TN], aq[TM][TN], asq[TM][TN];
#pragma unroll
  for (int u = 0; u < TM; ++u)
#pragma unroll
    for (int v = 0; v < TN; ++v) at[u][v] = az[u][v] = azs[u][v] = aq[u][v] = asq[u][v] = 0.f;
  for (int f = 0; f < kD; ++f) {
    float k[TM], q[TM], m[TN], s[TN], d[TN], ds[TN];
#pragma unroll
    for (int u = 0; u < TM; ++u) {
      k[u] = sK[(ty + 16 * u) * kPad + f];
      q[u] = sQ[(ty + 16 * u) * kPad + f];
    }
#pragma unroll
    for (int v = 0; v < TN; ++v) {
      const int r = (tx + 16 * v) * kPad + f;
      m[v] = sM0[r];
      d[v] = sDM[r];
      s[v] = sS0[r];
      if (MOM) ds[v] = sDS[r];
    }
#pragma unroll
    for (int u = 0; u < TM; ++u)
#pragma unroll
      for (int v = 0; v < TN; ++v) {
        at[u][v] = fmaf(k[u], m[v], at[u][v]);
        az[u][v] = fmaf(k[u], d[v], az[u][v]);
        aq[u][v] = fmaf(q[u], m[v], aq[u][v]);
        asq[u][v] = fmaf(q[u], s[v], asq[u][v]);
        if (MOM) azs[u][v] = fmaf(k[u], ds[v], azs[u][v]);
      }
  }
#pragma unroll
  for (int u = 0; u < TM; ++u)
#pragma unroll
    for (int v = 0; v < TN; ++v)
      fe(ty + 16 * u, tx + 16 * v, at[u][v], az[u][v], azs[u][v], aq[u][v], asq[u][v]);
}

// For 64 tokens x 128 features (two column blocks of 64; thread: tokens
// ty + 16 u, features tx + 16 v): the products dT M0, E dMe, E dSe, dY M0, dY S0
// that the dK and dQ partials combine.
template <bool MOM, class FE>
__device__ __forceinline__ void bwd_tile_kq(const float* sDT, const float* sE, const float* sDY,
                                            const float* sM0, const float* sS0, const float* sDM,
                                            const float* sDS, const FE& fe) {
  constexpr int TM = 4, TN = 4;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int f0 = 0; f0 < kD; f0 += 16 * TN) {
    float s1[TM][TN], s2[TM][TN], s2s[TM][TN], s3[TM][TN], s3s[TM][TN];
#pragma unroll
    for (int u = 0; u < TM; ++u)
#pragma unroll
      for (int v = 0; v < TN; ++v) s1[u][v] = s2[u][v] = s2s[u][v] = s3[u][v] = s3s[u][v] = 0.f;
    for (int r = 0; r < kRB; ++r) {
      float dt[TM], e[TM], dy[TM], m[TN], s[TN], d[TN], ds[TN];
#pragma unroll
      for (int u = 0; u < TM; ++u) {
        const int i = ty + 16 * u;
        dt[u] = sDT[i * kPadB + r];
        e[u] = sE[i * kPadB + r];
        dy[u] = sDY[i * kPadB + r];
      }
#pragma unroll
      for (int v = 0; v < TN; ++v) {
        const int x = r * kPad + f0 + tx + 16 * v;
        m[v] = sM0[x];
        d[v] = sDM[x];
        if (MOM) {
          s[v] = sS0[x];
          ds[v] = sDS[x];
        }
      }
#pragma unroll
      for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) {
          s1[u][v] = fmaf(dt[u], m[v], s1[u][v]);
          s2[u][v] = fmaf(e[u], d[v], s2[u][v]);
          s3[u][v] = fmaf(dy[u], m[v], s3[u][v]);
          if (MOM) {
            s2s[u][v] = fmaf(e[u], ds[v], s2s[u][v]);
            s3s[u][v] = fmaf(dy[u], s[v], s3s[u][v]);
          }
        }
    }
#pragma unroll
    for (int u = 0; u < TM; ++u)
#pragma unroll
      for (int v = 0; v < TN; ++v)
        fe(ty + 16 * u, f0 + tx + 16 * v, s1[u][v], s2[u][v], s2s[u][v], s3[u][v], s3s[u][v]);
  }
}

// The forward replay's chunk end (thread: rows ty + 16 u, features tx + 16 v):
// M_end = a_63 M0 + b_63 S0 - 2 sum_i wb_i E[i] k_i, S_end = e_63 S0 - 2 sum_i ub_i E[i] k_i.
__device__ __forceinline__ void bwd_tile_fwd_end(const float* sE, const float* sK,
                                                 const float* sWb, const float* sUb, float a63,
                                                 float b63, float e63, float* sM0, float* sS0) {
  constexpr int TM = 2, TN = 8;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float gw[TM][TN], gu[TM][TN];
#pragma unroll
  for (int u = 0; u < TM; ++u)
#pragma unroll
    for (int v = 0; v < TN; ++v) gw[u][v] = gu[u][v] = 0.f;
  for (int i = 0; i < kB; ++i) {
    const float wb = sWb[i], ub = sUb[i];
    float ew[TM], eu[TM], k[TN];
#pragma unroll
    for (int u = 0; u < TM; ++u) {
      const float e = sE[i * kPadB + ty + 16 * u];
      ew[u] = wb * e;
      eu[u] = ub * e;
    }
#pragma unroll
    for (int v = 0; v < TN; ++v) k[v] = sK[i * kPad + tx + 16 * v];
#pragma unroll
    for (int u = 0; u < TM; ++u)
#pragma unroll
      for (int v = 0; v < TN; ++v) {
        gw[u][v] = fmaf(ew[u], k[v], gw[u][v]);
        gu[u][v] = fmaf(eu[u], k[v], gu[u][v]);
      }
  }
#pragma unroll
  for (int u = 0; u < TM; ++u)
#pragma unroll
    for (int v = 0; v < TN; ++v) {
      const int x = (ty + 16 * u) * kPad + tx + 16 * v;
      const float m0 = sM0[x], s0 = sS0[x];
      sM0[x] = a63 * m0 + b63 * s0 - 2.f * gw[u][v];
      sS0[x] = e63 * s0 - 2.f * gu[u][v];
    }
}

// (dMe, dSe) <- (a_63 dMe + dY^T diag(a) Q + dT^T K, b_63 dMe + e_63 dSe + dY^T diag(b) Q)
// (thread: rows ty + 16 u, features tx + 16 v).
template <bool MOM>
__device__ __forceinline__ void bwd_tile_dm(const float* sA, const float* sBe, float e63,
                                            const float* sDY, const float* sDT, const float* sQ,
                                            const float* sK, float* sDM, float* sDS) {
  constexpr int TM = 2, TN = 8;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float am[TM][TN], as[TM][TN];
#pragma unroll
  for (int u = 0; u < TM; ++u)
#pragma unroll
    for (int v = 0; v < TN; ++v) am[u][v] = as[u][v] = 0.f;
  for (int n = 0; n < kB; ++n) {
    const float an = sA[n], bn = sBe[n];
    float ay[TM], by[TM], dt[TM], q[TN], k[TN];
#pragma unroll
    for (int u = 0; u < TM; ++u) {
      const float dy = sDY[n * kPadB + ty + 16 * u];
      ay[u] = an * dy;
      by[u] = bn * dy;
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
      for (int v = 0; v < TN; ++v) {
        am[u][v] = fmaf(ay[u], q[v], fmaf(dt[u], k[v], am[u][v]));
        if (MOM) as[u][v] = fmaf(by[u], q[v], as[u][v]);
      }
  }
  const float a63 = sA[kB - 1], b63 = sBe[kB - 1];
#pragma unroll
  for (int u = 0; u < TM; ++u)
#pragma unroll
    for (int v = 0; v < TN; ++v) {
      const int x = (ty + 16 * u) * kPad + tx + 16 * v;
      const float dm = sDM[x];
      if (MOM) sDS[x] = b63 * dm + e63 * sDS[x] + as[u][v];
      sDM[x] = a63 * dm + am[u][v];
    }
}

// MOM: the head has momentum somewhere.  Without it b = e = 0 and dSe stays
// zero, so the products with dSe and the b-weighted readout terms are skipped;
// S0 (the previous chunk's last step) is still tracked, because the gradient of
// the b table, which eta's gradient at eta = 0 needs, reads it.
template <bool MOM>
__device__ __forceinline__ void bwd_rows_body(const BwdArgs& p) {
  extern __shared__ float sm[];
  float* sM0 = sm;                    // [kRB][kPad] state rows M
  float* sS0 = sM0 + kRB * kPad;      // [kRB][kPad] momentum rows S
  float* sDM = sS0 + kRB * kPad;      // [kRB][kPad] dMe rows
  float* sDS = sDM + kRB * kPad;      // [kRB][kPad] dSe rows
  float* sK = sDS + kRB * kPad;       // [kB][kPad]
  float* sQ = sK + kB * kPad;         // [kB][kPad]
  float* sV = sQ + kB * kPad;         // [kB][kPadB] V[i][v]
  float* sDY = sV + kB * kPadB;       // [kB][kPadB]
  float* sE = sDY + kB * kPadB;       // [kB][kPadB] bias(e)
  float* sBP = sE + kB * kPadB;       // [kB][kPadB] bias'(e)
  float* sDT = sBP + kB * kPadB;      // [kB][kPadB]
  float* sZC = sDT + kB * kPadB;      // [kB][kPadB] wb Z + ub Zs
  float* sC = sZC + kB * kPadB;       // [kB][kB]
  float* sA = sC + kB * kB;           // [kB] a_n
  float* sBe = sA + kB;               // [kB] b_n
  float* sWb = sBe + kB;              // [kB] W[63][i]
  float* sUb = sWb + kB;              // [kB] U[63][i]
  float* sAcc = sUb + kB;             // [4][kB] da, db, dwb, dub; then 3 scalars

  const int h = blockIdx.x / kR, rb = blockIdx.x % kR, v0 = rb * kRB;
  const int tid = threadIdx.x, lane = tid & 31;
  const int N = p.N, nch = p.nch;
  const long hN = (long)h * N;
  const size_t MS = (size_t)kD * kD;

  for (int x = tid; x < kRB * kD; x += kThreads) {
    const int v = x / kD, f = x % kD;
    sM0[v * kPad + f] = p.M0[(size_t)h * MS + (size_t)(v0 + v) * kD + f];
    sS0[v * kPad + f] = 0.f;  // the momentum starts at zero
  }
  // ------------------------------------------------------------ forward
  for (int j = 0; j < nch; ++j) {
    const int t0 = j * kB, nb = min(kB, N - t0);
    const long cb = (long)h * nch + j;
    __syncthreads();
    float* ck = p.Mck + (size_t)cb * MS;
    float* cs = p.Sck + (size_t)cb * MS;
    for (int x = tid; x < kRB * kD; x += kThreads) {
      const int v = x / kD, f = x % kD;
      ck[(size_t)(v0 + v) * kD + f] = sM0[v * kPad + f];
      cs[(size_t)(v0 + v) * kD + f] = sS0[v * kPad + f];
    }
    load_kq(p, h, t0, nb, sK, kPad, nullptr, 0);
    for (int x = tid; x < kB * kRB; x += kThreads) {
      const int i = x / kRB, v = x % kRB;
      sV[i * kPadB + v] = i < nb ? ld_in(p.V, (hN + t0 + i) * kD + v0 + v, p.bf16) : 0.f;
    }
    if (tid < kB) {
      sA[tid] = p.tA[cb * kB + tid];
      sBe[tid] = p.tBe[cb * kB + tid];
      sWb[tid] = p.tW[cb * kB * kB + (kB - 1) * kB + tid];
      sUb[tid] = p.tU[cb * kB * kB + (kB - 1) * kB + tid];
    }
    __syncthreads();
    if (j + 1 < nch) prefetch_chunk(p, h, j + 1, v0, false);
    {  // E[i][v] = bias(K M0^T - V)
      auto fa = [&](int i, int f) { return sK[i * kPad + f]; };
      auto fb = [&](int f, int v) { return sM0[v * kPad + f]; };
      auto fe = [&](int i, int v, float t) {
        sE[i * kPadB + v] = bias_grad(t - sV[i * kPadB + v], p.lk, p.lp);
      };
      tile_gemm<16, 4, 2>(kB, kRB, kD, fa, fb, fe);
    }
    __syncthreads();
    bwd_tile_fwd_end(sE, sK, sWb, sUb, sA[kB - 1], sBe[kB - 1], p.tEp[cb * kB + kB - 1], sM0,
                     sS0);
  }
  // ------------------------------------------------------------ reverse
  __syncthreads();
  for (int x = tid; x < kRB * kD; x += kThreads) {
    const int v = x / kD, f = x % kD;
    sDM[v * kPad + f] = p.dM[(size_t)h * MS + (size_t)(v0 + v) * kD + f];
    sDS[v * kPad + f] = 0.f;  // the momentum after the last token is not an output
  }
  for (int j = nch - 1; j >= 0; --j) {
    const int t0 = j * kB, nb = min(kB, N - t0);
    const long cb = (long)h * nch + j;
    const size_t pb = ((size_t)rb * p.heads + h) * nch + j;
    __syncthreads();
    const float* ck = p.Mck + (size_t)cb * MS;
    const float* cs = p.Sck + (size_t)cb * MS;
    for (int x = tid; x < kRB * kD; x += kThreads) {
      const int v = x / kD, f = x % kD;
      sM0[v * kPad + f] = ck[(size_t)(v0 + v) * kD + f];
      sS0[v * kPad + f] = cs[(size_t)(v0 + v) * kD + f];
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
      sBe[tid] = p.tBe[cb * kB + tid];
      sWb[tid] = p.tW[cb * kB * kB + (kB - 1) * kB + tid];
      sUb[tid] = p.tU[cb * kB * kB + (kB - 1) * kB + tid];
    }
    for (int x = tid; x < 4 * kB + 3; x += kThreads) sAcc[x] = 0.f;
    const float e63 = p.tEp[cb * kB + kB - 1];
    __syncthreads();
    if (j > 0) prefetch_chunk(p, h, j - 1, v0, true);
    // -- errors, bias', the weighted Z; da, db, dwb, dub summed over this block's rows
    bwd_tile_r1<MOM>(sK, sQ, sM0, sS0, sDM, sDS,
                [&](int i, int v, float t, float z, float zs, float mq, float sq) {
      const float e = t - sV[i * kPadB + v];
      const float E = bias_grad(e, p.lk, p.lp);
      const float dy = sDY[i * kPadB + v];
      sE[i * kPadB + v] = E;
      sBP[i * kPadB + v] = bias_grad2(e, p.lk, p.lp);
      sZC[i * kPadB + v] = MOM ? sWb[i] * z + sUb[i] * zs : sWb[i] * z;
      atomicAdd(&sAcc[i], dy * mq);
      atomicAdd(&sAcc[kB + i], dy * sq);
      atomicAdd(&sAcc[2 * kB + i], E * z);
      if (MOM) atomicAdd(&sAcc[3 * kB + i], E * zs);
    });
    {  // <dMe, M0>, <dMe, S0>, <dSe, S0> over this block's rows
      float x0 = 0.f, x1 = 0.f, x2 = 0.f;
      for (int x = tid; x < kRB * kD; x += kThreads) {
        const int o = (x / kD) * kPad + x % kD;
        x0 += sDM[o] * sM0[o];
        x1 += sDM[o] * sS0[o];
        if (MOM) x2 += sDS[o] * sS0[o];
      }
      x0 = warp_sum(x0);
      x1 = warp_sum(x1);
      x2 = warp_sum(x2);
      if (lane == 0) {
        atomicAdd(&sAcc[4 * kB], x0);
        atomicAdd(&sAcc[4 * kB + 1], x1);
        atomicAdd(&sAcc[4 * kB + 2], x2);
      }
    }
    __syncthreads();
    if (tid < kB) {
      const bool last = tid == kB - 1;
      p.pA[pb * kB + tid] = sAcc[tid] + (last ? sAcc[4 * kB] : 0.f);
      p.pB[pb * kB + tid] = sAcc[kB + tid] + (last ? sAcc[4 * kB + 1] : 0.f);
      p.pWb[pb * kB + tid] = -2.f * sAcc[2 * kB + tid];
      p.pUb[pb * kB + tid] = -2.f * sAcc[3 * kB + tid];
    } else if (tid == kB) {
      p.pE[pb] = sAcc[4 * kB + 2];
    }
    // -- dE, dT, dV (dE = -2 C^T dY - 2 (wb Z + ub Zs))
    {
      auto fa = [&](int i, int n) { return sC[n * kB + i]; };
      auto fb = [&](int n, int v) { return sDY[n * kPadB + v]; };
      auto fe = [&](int i, int v, float s) {
        const float dE = -2.f * s - 2.f * sZC[i * kPadB + v];
        const float dT = dE * sBP[i * kPadB + v];
        sDT[i * kPadB + v] = dT;
        if (i < nb) p.dV[(hN + t0 + i) * kD + v0 + v] = -dT;
      };
      tile_gemm<16, 4, 2>(kB, kRB, kB, fa, fb, fe);
    }
    __syncthreads();
    // -- dK, dQ, dC partials
    {
      const size_t ob = ((size_t)rb * p.heads + h) * N;
      bwd_tile_kq<MOM>(sDT, sE, sDY, sM0, sS0, sDM, sDS,
                       [&](int i, int f, float s1, float s2, float s2s, float s3, float s3s) {
        if (i < nb) {
          p.pK[(ob + t0 + i) * kD + f] =
              MOM ? s1 - 2.f * sWb[i] * s2 - 2.f * sUb[i] * s2s : s1 - 2.f * sWb[i] * s2;
          p.pQ[(ob + t0 + i) * kD + f] = MOM ? sA[i] * s3 + sBe[i] * s3s : sA[i] * s3;
        }
      });
      const size_t cbo = pb * kB * kB;
      auto fa = [&](int n, int v) { return sDY[n * kPadB + v]; };
      auto fb = [&](int v, int i) { return sE[i * kPadB + v]; };
      auto fe = [&](int n, int i, float s) { p.pC[cbo + n * kB + i] = -2.f * s; };
      tile_gemm<16, 4, 4>(kB, kB, kRB, fa, fb, fe);
    }
    __syncthreads();
    // -- (dMe, dSe) <- (dM0, dS0)
    bwd_tile_dm<MOM>(sA, sBe, e63, sDY, sDT, sQ, sK, sDM, sDS);
  }
  __syncthreads();
  for (int x = tid; x < kRB * kD; x += kThreads) {
    const int v = x / kD, f = x % kD;
    p.dM[(size_t)h * MS + (size_t)(v0 + v) * kD + f] = sDM[v * kPad + f];
  }
}

__global__ void __launch_bounds__(kThreads, 1) bwd_rows_kernel(BwdArgs p) {
  if (p.mom[blockIdx.x / kR])
    bwd_rows_body<true>(p);
  else
    bwd_rows_body<false>(p);
}

// ------------------------------------------------------------- finish

__global__ void __launch_bounds__(kThreads) bwd_finish_kernel(BwdArgs p) {
  extern __shared__ float sm[];
  float* sW = sm;                 // [kB][kB] W, then the dalpha terms
  float* sU = sW + kB * kB;       // [kB][kB] U, then the deta terms
  float* sDW = sU + kB * kB;      // [kB][kB] dW
  float* sDP = sDW + kB * kB;     // [kB][kB]
  float* sAl = sDP + kB * kB;     // [kB]
  float* sEt = sAl + kB;          // [kB]
  float* sA = sEt + kB;           // [kB]
  float* sBe = sA + kB;           // [kB]
  float* sEp = sBe + kB;          // [kB]
  float* sDa = sEp + kB;          // [kB]
  float* sDb = sDa + kB;          // [kB]
  float* sDub = sDb + kB;         // [kB]
  float* sSa = sDub + kB;         // [kB] the scalar tables' dalpha terms
  float* sSe = sSa + kB;          // [kB] the scalar tables' deta terms
  float* sTh = sSe + kB;          // [kB] dtheta
  const int h = blockIdx.x / p.nch, j = blockIdx.x % p.nch;
  const int t0 = j * kB, nb = min(kB, p.N - t0);
  const int tid = threadIdx.x;
  const long g = (long)h * p.N + t0;
  const long cb = (long)h * p.nch + j;
  const size_t cbo = (size_t)cb * kB * kB;
  for (int x = tid; x < kB * kB; x += kThreads) {
    const int n = x / kB, i = x % kB;
    float dc = 0.f;
#pragma unroll
    for (int rb = 0; rb < kR; ++rb)
      dc += p.pC[(((size_t)rb * p.heads + h) * p.nch + j) * kB * kB + x];
    const float w = p.tW[cbo + x];
    sW[x] = w;
    sU[x] = p.tU[cbo + x];
    const bool low = i <= n;
    sDP[x] = low ? w * dc : 0.f;
    sDW[x] = low ? p.tP[cbo + x] * dc : 0.f;
  }
  float dE63 = 0.f;
  if (tid < kB) {
    const bool ok = tid < nb;
    sAl[tid] = ok ? p.alpha[g + tid] : 0.f;
    sEt[tid] = ok ? p.eta[g + tid] : 0.f;
    sA[tid] = p.tA[cb * kB + tid];
    sBe[tid] = p.tBe[cb * kB + tid];
    sEp[tid] = p.tEp[cb * kB + tid];
    float da = 0.f, db = 0.f, dub = 0.f;
    for (int rb = 0; rb < kR; ++rb) {
      const size_t o = (((size_t)rb * p.heads + h) * p.nch + j) * kB + tid;
      da += p.pA[o];
      db += p.pB[o];
      dub += p.pUb[o];
    }
    sDa[tid] = da;
    sDb[tid] = db;
    sDub[tid] = dub;
  } else if (tid == kB) {
    for (int rb = 0; rb < kR; ++rb) dE63 += p.pE[((size_t)rb * p.heads + h) * p.nch + j];
  }
  __syncthreads();
  if (tid < kB) {  // wb is row 63 of W
    float dwb = 0.f;
    for (int rb = 0; rb < kR; ++rb)
      dwb += p.pWb[(((size_t)rb * p.heads + h) * p.nch + j) * kB + tid];
    sDW[(kB - 1) * kB + tid] += dwb;
  }
  __syncthreads();
  const float g0 = p.gamma[0];
  if (tid < kB) {
    // column i of the W / U recursions, n = 63 .. 0: Wb, Ub are the adjoints of
    // W[n][i], U[n][i]; the dalpha and deta terms replace W and U in place
    const int i = tid;
    float Wb = 0.f, Ub = 0.f;
    for (int n = kB - 1; n >= 0; --n) {
      Wb += sDW[n * kB + i];
      Ub += (n == kB - 1 ? sDub[i] : 0.f) + Wb;  // W[n] = (1 - alpha_n) W[n-1] + U[n]
      const float wp = n > 0 ? sW[(n - 1) * kB + i] : 0.f;
      const float up = n > 0 ? sU[(n - 1) * kB + i] : 0.f;
      if (n == i) sTh[i] = g0 * Ub;          // U[n][n] = eta_n U[n-1][n] + g0 theta_n
      sW[n * kB + i] = -Wb * wp;             // dalpha_n term
      sU[n * kB + i] = Ub * up;              // deta_n term
      Wb *= 1.f - sAl[n];
      Ub *= sEt[n];
    }
  } else if (tid == kB) {
    // the scalar tables a, b, e, n = 63 .. 0
    float Ab = 0.f, Bb = 0.f, Eb = 0.f;
    for (int n = kB - 1; n >= 0; --n) {
      Ab += sDa[n];
      Bb += sDb[n];
      Eb += (n == kB - 1 ? dE63 : 0.f) + Bb;  // b_n = (1 - alpha_n) b_{n-1} + e_n
      const float ap = n > 0 ? sA[n - 1] : 1.f;
      const float bp = n > 0 ? sBe[n - 1] : 0.f;
      const float ep = n > 0 ? sEp[n - 1] : 1.f;
      sSa[n] = -Ab * ap - Bb * bp;
      sSe[n] = Eb * ep;
      Ab *= 1.f - sAl[n];
      Bb *= 1.f - sAl[n];
      Eb *= sEt[n];
    }
  }
  __syncthreads();
  if (tid < nb) {
    const int n = tid;
    float da = sSa[n], de = sSe[n];
    for (int i = 0; i < kB; ++i) {
      da += sW[n * kB + i];
      de += sU[n * kB + i];
    }
    p.dalpha[g + n] = da;
    p.deta[g + n] = de;
    p.dtheta[g + n] = sTh[n];
  }
  {  // dK[i] = sum_n dP[n][i] q_n, dQ[i] = sum_n dP[i][n] k_n (register-tiled: an 8 x 4
     // block of (i, f) a thread; q_n and k_n straight from global memory, a warp reading
     // 128 consecutive bytes, so that three CTAs fit an SM); the row-block partials are
     // added by bwd_partials_kernel
    auto row = [&](const void* X, int n, int f) {
      return n < nb ? ld_in(X, (g + n) * kD + f, p.bf16) : 0.f;
    };
    tile_gemm<32, 8, 4>(nb, kD, kB, [&](int i, int n) { return sDP[n * kB + i]; },
                        [&](int n, int f) { return row(p.Q, n, f); },
                        [&](int i, int f, float s) { p.dK[(g + i) * kD + f] = s; });
    tile_gemm<32, 8, 4>(nb, kD, kB, [&](int i, int n) { return sDP[i * kB + n]; },
                        [&](int n, int f) { return row(p.K, n, f); },
                        [&](int i, int f, float s) { p.dQ[(g + i) * kD + f] = s; });
  }
}

// dK += the kR row-block partials of dK, dQ likewise, in row-block order: a
// streaming pass over every head and token (the finish kernel, one large CTA
// per SM, left too few loads in flight for it).
__global__ void __launch_bounds__(kThreads) bwd_partials_kernel(BwdArgs p) {
  const size_t T = (size_t)p.heads * p.N * kD;
  for (size_t x = (size_t)blockIdx.x * kThreads + threadIdx.x; x < T;
       x += (size_t)gridDim.x * kThreads) {
    float sk = p.dK[x], sq = p.dQ[x];
#pragma unroll
    for (int rb = 0; rb < kR; ++rb) {
      sk += p.pK[rb * T + x];
      sq += p.pQ[rb * T + x];
    }
    p.dK[x] = sk;
    p.dQ[x] = sq;
  }
}

// ---------------------------------------------------------------- host

namespace {

constexpr size_t kTablesSmem = sizeof(float) * ((size_t)kB * kPad + kB * kD + 3 * kB + kB * kB);
constexpr size_t kRowsSmem = sizeof(float) * ((size_t)4 * kRB * kPad + 2 * kB * kPad +
                                              6 * kB * kPadB + kB * kB + 4 * kB + 4 * kB + 3);
constexpr size_t kFinishSmem = sizeof(float) * ((size_t)4 * kB * kB + 11 * kB);

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
  p.Mck = w + L.Mck; p.Sck = w + L.Sck; p.tW = w + L.tW; p.tU = w + L.tU; p.tP = w + L.tP;
  p.tC = w + L.tC; p.tA = w + L.tA; p.tBe = w + L.tBe; p.tEp = w + L.tEp; p.pK = w + L.pK;
  p.pQ = w + L.pQ; p.pC = w + L.pC; p.pWb = w + L.pWb; p.pUb = w + L.pUb; p.pA = w + L.pA;
  p.pB = w + L.pB; p.pE = w + L.pE;
  p.mom = reinterpret_cast<int*>(w + L.mom);
  if (cudaMemsetAsync(p.mom, 0, sizeof(int) * heads, st) != cudaSuccess) return ATLAS_ERR_CUDA;
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
  bwd_partials_kernel<<<152 * 8, kThreads, 0, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? ATLAS_OK : ATLAS_ERR_CUDA;
}

}  // namespace atlas
