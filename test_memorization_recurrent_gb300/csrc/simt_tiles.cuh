// simt_tiles.cuh -- register-tiled block products over shared memory for the
// CUDA-core chunk kernels (256 threads), and the feature maps they read.
#pragma once

#include "common.cuh"

namespace atlas {

// Feature j of the gated polynomial map: a_e times the product of the e indexed
// entries of x (entry t of the monomial table; 0xFF marks unused index bytes).
__device__ __forceinline__ float phi_gated(const float* x, uint32_t t, const float* a) {
  float v = 1.f;
  int e = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const uint32_t i = (t >> (8 * r)) & 0xFFu;
    if (i != 0xFFu) {
      v *= x[i];
      ++e;
    }
  }
  return a[e] * v;
}

// Phi of the rows of x (shared memory, row stride ld): identity, the degree-2
// map (pair table pp, pq) or the gated map (monomial table ftab, coefficients a).
struct Feat {
  const float* x;
  int ld, dk, poly, pgen;
  const uint8_t* pp;
  const uint8_t* pq;
  const uint32_t* ftab;
  const float* a;
  __device__ __forceinline__ float operator()(int row, int j) const {
    const float* r = x + row * ld;
    if (pgen) return phi_gated(r, ftab[j], a);
    if (!poly || j < dk) return r[j];
    return r[pp[j - dk]] * r[pq[j - dk]];
  }
};

// The identity map read straight from the rows of x (row stride ld).
struct FeatId {
  const float* x;
  int ld;
  __device__ __forceinline__ float operator()(int row, int j) const { return x[row * ld + j]; }
};

// C = A B over k < K for an m x n output: thread (ty, tx) of a TY x TX grid
// (TY TX = 256) owns rows ty + TY u and columns tx + TX v of each block; fe
// receives each finished output.  Operand indices are clamped into range, so
// the loads stay in bounds and only in-range outputs are delivered.
template <int TX, int TM, int TN, class FA, class FB, class FE>
__device__ __forceinline__ void tile_gemm(int m, int n, int K, const FA& fa, const FB& fb,
                                          const FE& fe) {
  constexpr int TY = 256 / TX;
  const int tx = threadIdx.x % TX, ty = threadIdx.x / TX;
  for (int m0 = 0; m0 < m; m0 += TY * TM)
    for (int n0 = 0; n0 < n; n0 += TX * TN) {
      int mi[TM], nj[TN];
#pragma unroll
      for (int u = 0; u < TM; ++u) mi[u] = min(m0 + ty + TY * u, m - 1);
#pragma unroll
      for (int v = 0; v < TN; ++v) nj[v] = min(n0 + tx + TX * v, n - 1);
      float acc[TM][TN];
#pragma unroll
      for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) acc[u][v] = 0.f;
      for (int k = 0; k < K; ++k) {
        float a[TM], b[TN];
#pragma unroll
        for (int u = 0; u < TM; ++u) a[u] = fa(mi[u], k);
#pragma unroll
        for (int v = 0; v < TN; ++v) b[v] = fb(k, nj[v]);
#pragma unroll
        for (int u = 0; u < TM; ++u)
#pragma unroll
          for (int v = 0; v < TN; ++v) acc[u][v] = fmaf(a[u], b[v], acc[u][v]);
      }
#pragma unroll
      for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) {
          const int r = m0 + ty + TY * u, c = n0 + tx + TX * v;
          if (r < m && c < n) fe(r, c, acc[u][v]);
        }
    }
}

// State carry to the chunk end: with gw[r, j] = sum_i W_b[i] E[i, r] Phi(k_i)[j]
// and gu likewise with U_b,  M = a_b M + beta_b S - 2 gw,  S = eps_b S - 2 gu.
template <int TX, int TM, int TN, class FK>
__device__ __forceinline__ void carry_tile(int rv, int D, int Lw, const FK& fk, const float* E,
                                           const float* Wrun, const float* Urun, float* Ms,
                                           float* Ss, int Dp, float a_b, float b_b, float e_b) {
  constexpr int TY = 256 / TX;
  const int tx = threadIdx.x % TX, ty = threadIdx.x / TX;
  for (int m0 = 0; m0 < rv; m0 += TY * TM)
    for (int n0 = 0; n0 < D; n0 += TX * TN) {
      int mi[TM], nj[TN];
#pragma unroll
      for (int u = 0; u < TM; ++u) mi[u] = min(m0 + ty + TY * u, rv - 1);
#pragma unroll
      for (int v = 0; v < TN; ++v) nj[v] = min(n0 + tx + TX * v, D - 1);
      float gw[TM][TN], gu[TM][TN];
#pragma unroll
      for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) gw[u][v] = gu[u][v] = 0.f;
      for (int i = 0; i < Lw; ++i) {
        const float w = Wrun[i], uu = Urun[i];
        float ew[TM], eu[TM], f[TN];
#pragma unroll
        for (int u = 0; u < TM; ++u) {
          const float e = E[i * rv + mi[u]];
          ew[u] = e * w;
          eu[u] = e * uu;
        }
#pragma unroll
        for (int v = 0; v < TN; ++v) f[v] = fk(i, nj[v]);
#pragma unroll
        for (int u = 0; u < TM; ++u)
#pragma unroll
          for (int v = 0; v < TN; ++v) {
            gw[u][v] = fmaf(ew[u], f[v], gw[u][v]);
            gu[u][v] = fmaf(eu[u], f[v], gu[u][v]);
          }
      }
#pragma unroll
      for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) {
          const int r = m0 + ty + TY * u, j = n0 + tx + TX * v;
          if (r < rv && j < D) {
            const long x = (long)r * Dp + j;
            const float m0v = Ms[x], s0v = Ss[x];
            Ms[x] = a_b * m0v + b_b * s0v - 2.f * gw[u][v];
            Ss[x] = e_b * s0v - 2.f * gu[u][v];
          }
        }
    }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}

}  // namespace atlas
