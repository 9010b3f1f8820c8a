// linear_simt_body.cuh -- chunked Omega-rule update of a linear matrix memory on
// CUDA cores (fp32), for any feature map, window, chunk and gate setting: the
// kernel body, instantiated once per gate family -- the chunk tables (l2, l_q;
// linear_simt.cu) and each token-serial gate (linear_simt_elastic.cu,
// linear_simt_bregman.cu, linear_simt_kl.cu) -- so that they compile in parallel.
//
// The memory y = M Phi(x) decomposes over the rows of M: the error
// e_i[r] = M[r,:] . Phi(k_i) - v_i[r] and the readout y_n[r] = M_n[r,:] . Phi(q_n)
// only involve row r.  Each CTA therefore owns RV rows of M and of the momentum
// S of one head, keeps them in shared memory for the whole sequence and walks
// the chunks in order; no CTA ever waits on another.
//
// Per chunk of nb tokens starting at t0, with window tokens i0..t1-1 (L of them,
// i0 = max(-n_history, t0-c+1): history rows of K, V enter windows too) -- "논문 리뷰 Google ATLAS" §3.3 (gradients at the
// chunk-start state), "[Paper Review] Titans 논문 이해하기" (momentum, decay,
// readout after the write):
//   E[i,r]  = M0[r,:] . Phi(k_i) - v_i[r]              (dot bias: -v_i[r])
//   y_n[r]  = a_n M0[r,:].Phi(q_n) + beta_n S0[r,:].Phi(q_n)
//             - 2 sum_i W[n,i] (Phi(k_i).Phi(q_n)) E[i,r]
//   M[r,:]  = a_b M0 + beta_b S0 - 2 sum_i W[b,i] E[i,r] Phi(k_i)
//   S[r,:]  = eps_b S0 - 2 sum_i U[b,i] E[i,r] Phi(k_i)
// with the scalar tables of chunk_tables.  Phi(q).Phi(k) for the degree-2
// map is evaluated as s + (s^2 + sum_j q_j^2 k_j^2)/2 with s = q.k, which is the
// same sum regrouped.  The gated polynomial map of any degree ("논문 리뷰 Google
// ATLAS" §3.1, Input gating) keeps one 32-bit entry per feature (its sorted
// monomial indices, 0xFF past its degree) in shared memory, and its lifted inner
// product is sum_e a_e^2 h_e(z), z_j = q_j k_j, with the complete homogeneous
// symmetric polynomials h_e from the power sums of z (Newton's identities).
//
// Retention gates other than l2 ("It's All Connected (Miras)", #2 Alternative
// Retention Gates).  The l_q memory keeps the tables: its state is the plain
// accumulator A, and the memory A_r / z_r with the per-row normaliser
// z_r = ||A_r||_q^(q-2) taken at the chunk start enters the errors and the
// readout as one scale per row.  Elastic net, Bregman (sigmoid link) and KL map
// the decayed step through a non-linear function at every token, so their chunk
// walks the tokens one by one after the errors E: per token, one warp per row r
// forms the window gradient sum_i gamma[t-i] E[i,r] Phi(k_i), steps S and the
// state, and reads the row out.  The Bregman state is kept as logits and the KL
// state as log M (the same maps, without a log per step); both are converted at
// load and store.
//
// Every product of a chunk is a small dense contraction over shared memory,
// computed by register tiles: 256 threads form a TY x TX grid and each thread
// accumulates TM x TN outputs spaced TY and TX apart, so a k-step loads TM + TN
// operands for TM TN FMAs.  Rows of M, S, K and Q are stored with odd strides,
// which keeps the column walks free of bank conflicts.  The token-serial walk
// has a fast form for D <= 128 and at most 64 rows: four lanes share a row and
// keep its M and S in registers for the whole chunk (32 columns each), so each
// row's sums take two shuffle steps.
//
// The robust bias scales each window token's error row by 1 + Delta/||e||, which
// needs the norm over all d_v rows of the head.  Its row blocks therefore form
// one thread-block cluster per head (at most 8 CTAs): each CTA writes the partial
// squared norms of its rows to shared memory, and after a cluster barrier every
// CTA adds the partials of all ranks through distributed shared memory; a second
// barrier keeps them until every rank has read them.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "simt_tiles.cuh"

namespace atlas {

struct LinSimtSmem {
  int RV, D, Lmax, b, d_k, pgen;
  int Dp, dkp;  // odd row strides of M / S and of K / Q (conflict-free column walks)
  int ncl;      // CTAs per head in one cluster (robust bias), else 1
  // float offsets
  long Ms, Ss, Kw, Qc, Vw, E, P, Urun, Wrun, sa, se, sb, Z, NR, coef, total_floats;
  long pairs_bytes;
  size_t bytes() const { return total_floats * sizeof(float) + pairs_bytes; }
};

static LinSimtSmem lin_simt_layout(int RV, int D, int Lmax, int b, int d_k, int pgen) {
  LinSimtSmem s;
  s.RV = RV; s.D = D; s.Lmax = Lmax; s.b = b; s.d_k = d_k; s.pgen = pgen; s.ncl = 1;
  s.Dp = D | 1;
  s.dkp = d_k | 1;
  long o = 0;
  s.Ms = o; o += (long)RV * s.Dp;
  s.Ss = o; o += (long)RV * s.Dp;
  s.Kw = o; o += (long)Lmax * s.dkp;
  s.Qc = o; o += (long)b * s.dkp;
  s.Vw = o; o += (long)Lmax * RV;
  s.E = o; o += (long)Lmax * RV;
  s.P = o; o += (long)b * Lmax;
  s.Urun = o; o += Lmax;
  s.Wrun = o; o += Lmax;
  s.sa = o; o += b;
  s.se = o; o += b;
  s.sb = o; o += b;
  s.Z = o; o += RV;
  s.NR = o; o += Lmax;
  s.coef = o; o += 8;
  s.total_floats = o;
  s.pairs_bytes = pgen ? 4L * D : 2L * (D - d_k > 0 ? D - d_k : 0);
  return s;
}

// Tile shapes by the number of rows a CTA owns: class 1..4 for rv <= 16, 32, 64
// and beyond.
__device__ __forceinline__ int rows_class(int rv) {
  return rv <= 16 ? 1 : rv <= 32 ? 2 : rv <= 64 ? 3 : 4;
}

// m x rv outputs with the rows r as columns (errors, readout operands).
template <class FA, class FB, class FE>
__device__ __forceinline__ void gemm_by_rows(int cls, int m, int rv, int K, const FA& fa,
                                             const FB& fb, const FE& fe) {
  switch (cls) {
    case 1: tile_gemm<16, 4, 1>(m, rv, K, fa, fb, fe); break;
    case 2: tile_gemm<16, 4, 2>(m, rv, K, fa, fb, fe); break;
    case 3: tile_gemm<16, 4, 4>(m, rv, K, fa, fb, fe); break;
    default: tile_gemm<16, 4, 8>(m, rv, K, fa, fb, fe); break;
  }
}

// Readout of the chunk's queries: y[n, r] = z_r (sa_n Phi(q_n).M[r] + sb_n
// Phi(q_n).S[r] - 2 sum_i P[n, i] E[i, r]); the S term is skipped when every
// sb_n of the chunk is 0.
template <int TX, int TM, int TN>
__device__ __forceinline__ void readout_tile(int nb, int rv, int D, int Lw, const Feat& fq,
                                             const float* Ms, const float* Ss, int Dp,
                                             const float* P, int ldp, const float* E,
                                             const float* sa, const float* sb, bool with_s,
                                             const float* Z, float* Y, int dv) {
  constexpr int TY = 256 / TX;
  const int tx = threadIdx.x % TX, ty = threadIdx.x / TX;
  for (int m0 = 0; m0 < nb; m0 += TY * TM)
    for (int n0 = 0; n0 < rv; n0 += TX * TN) {
      int mi[TM], nj[TN];
#pragma unroll
      for (int u = 0; u < TM; ++u) mi[u] = min(m0 + ty + TY * u, nb - 1);
#pragma unroll
      for (int v = 0; v < TN; ++v) nj[v] = min(n0 + tx + TX * v, rv - 1);
      float am[TM][TN], as[TM][TN];
#pragma unroll
      for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) am[u][v] = as[u][v] = 0.f;
      for (int j = 0; j < D; ++j) {
        float a[TM], bm[TN];
#pragma unroll
        for (int u = 0; u < TM; ++u) a[u] = fq(mi[u], j);
#pragma unroll
        for (int v = 0; v < TN; ++v) bm[v] = Ms[nj[v] * Dp + j];
#pragma unroll
        for (int u = 0; u < TM; ++u)
#pragma unroll
          for (int v = 0; v < TN; ++v) am[u][v] = fmaf(a[u], bm[v], am[u][v]);
        if (with_s) {
          float bs[TN];
#pragma unroll
          for (int v = 0; v < TN; ++v) bs[v] = Ss[nj[v] * Dp + j];
#pragma unroll
          for (int u = 0; u < TM; ++u)
#pragma unroll
            for (int v = 0; v < TN; ++v) as[u][v] = fmaf(a[u], bs[v], as[u][v]);
        }
      }
#pragma unroll
      for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) am[u][v] = sa[mi[u]] * am[u][v] + sb[mi[u]] * as[u][v];
      for (int i = 0; i < Lw; ++i) {
        float a[TM], be[TN];
#pragma unroll
        for (int u = 0; u < TM; ++u) a[u] = -2.f * P[mi[u] * ldp + i];
#pragma unroll
        for (int v = 0; v < TN; ++v) be[v] = E[i * rv + nj[v]];
#pragma unroll
        for (int u = 0; u < TM; ++u)
#pragma unroll
          for (int v = 0; v < TN; ++v) am[u][v] = fmaf(a[u], be[v], am[u][v]);
      }
#pragma unroll
      for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) {
          const int n = m0 + ty + TY * u, r = n0 + tx + TX * v;
          if (n < nb && r < rv) Y[(long)n * dv + r] = Z ? am[u][v] * Z[r] : am[u][v];
        }
    }
}

// P[n, i] <- P[n, i] (the W table on entry) times Phi(q_n).Phi(k_i), from the
// power sums p_m = sum_j (q_j k_j)^m, m <= NP, of 64 x 64 blocks (thread tile
// 4 x 4): kind 0 the identity map (p_1), 1 the degree-2 map, p_1 + (p_1^2 + p_2)/2,
// 2 the gated map, sum_e a_e^2 h_e with the complete homogeneous symmetric
// polynomials h_e from the power sums (Newton's identities).
template <int NP>
__device__ __forceinline__ void qk_tile(int nb, int Lw, int dk, const float* Qc, const float* Kw,
                                        int dkp, float* P, int ldp, int kind, const float* a,
                                        int deg) {
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  for (int m0 = 0; m0 < nb; m0 += 64)
    for (int n0 = 0; n0 < Lw; n0 += 64) {
      int mi[4], nj[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        mi[u] = min(m0 + ty + 16 * u, nb - 1);
        nj[u] = min(n0 + tx + 16 * u, Lw - 1);
      }
      float ps[NP][4][4];
#pragma unroll
      for (int e = 0; e < NP; ++e)
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) ps[e][u][v] = 0.f;
      for (int j = 0; j < dk; ++j) {
        float q[4], k[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          q[u] = Qc[mi[u] * dkp + j];
          k[u] = Kw[nj[u] * dkp + j];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const float z = q[u] * k[v];
            float zz = z;
#pragma unroll
            for (int e = 0; e < NP; ++e) {
              ps[e][u][v] += zz;
              zz *= z;
            }
          }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int n = m0 + ty + 16 * u, i = n0 + tx + 16 * v;
          if (n >= nb || i >= Lw) continue;
          float val;
          if (kind == 0) {
            val = ps[0][u][v];
          } else if (kind == 1) {
            val = ps[0][u][v] + 0.5f * (ps[0][u][v] * ps[0][u][v] + ps[NP > 1 ? 1 : 0][u][v]);
          } else {
            float h[5];
            h[0] = 1.f;
            val = a[0] * a[0];
#pragma unroll
            for (int m = 1; m <= 4; ++m) {
              float acc = 0.f;
#pragma unroll
              for (int l = 1; l <= m; ++l) acc += (l <= NP ? ps[l <= NP ? l - 1 : 0][u][v] : 0.f) * h[m - l];
              h[m] = acc / (float)m;
              if (m <= deg) val += a[m] * a[m] * h[m];
            }
          }
          P[n * ldp + i] *= val;
        }
    }
}

// The memory entry a state entry stands for: the state itself (MK 0), the
// sigmoid of a logit (MK 1, Bregman) or the exponential of log M (MK 2, KL).
template <int MK>
__device__ __forceinline__ float mem_entry(float m) {
  if (MK == 1) return 1.f / (1.f + expf(-m));
  if (MK == 2) return expf(m);
  return m;
}

// Running (max, sum of exp) pairs of a softmax, combined across the warp.
__device__ __forceinline__ void warp_lse(float& mx, float& den) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xFFFFFFFFu, mx, o);
    const float od = __shfl_xor_sync(0xFFFFFFFFu, den, o);
    const float nm = fmaxf(mx, om);
    den = (den > 0.f ? den * expf(mx - nm) : 0.f) + (od > 0.f ? od * expf(om - nm) : 0.f);
    mx = nm;
  }
}

// Token-serial walk of one chunk for a non-linear gate (RK: ATLAS_RET_*), D <= 128,
// at most 64 rows.  Four lanes share a row (warp w holds rows 8 w .. 8 w + 7), each
// keeping 32 of its columns (sub + 4 u) of M and S in registers for the whole
// chunk, so a row's sums take two shuffle steps.  Per token: the window gradient
// from the chunk-start errors (the current key's features in registers, earlier
// window keys read from shared memory), the momentum and state steps, the gate
// and the row readout; the rows go back to shared memory at the chunk end.
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xFFFFFFFFu, x, 1);
  return x + __shfl_xor_sync(0xFFFFFFFFu, x, 2);
}

template <int RK, class FT>
__device__ __forceinline__ void serial_chunk_quad(int nb, int t0, int i0, int c, int rv, int D,
                                                  int Dp, float* Ms, float* Ss, const float* E,
                                                  const FT& fq, const FT& fk,
                                                  const float* sa, const float* se,
                                                  const float* sb, const float* gam, float lam,
                                                  float logc, float* Y, int dv) {
  constexpr int CPL = 32;  // columns per lane
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane & 3, row = warp * 8 + (lane >> 2);
  const bool live = row < rv;
  const int rr = live ? row : 0;  // a valid row index for the loads of idle lanes
  float m[CPL], sv[CPL];
#pragma unroll
  for (int u = 0; u < CPL; ++u) {
    const int j = sub + 4 * u;
    const bool ok = live && j < D;
    m[u] = ok ? Ms[rr * Dp + j] : 0.f;
    sv[u] = ok ? Ss[rr * Dp + j] : 0.f;
  }
  for (int n = 0; n < nb; ++n) {
    const int t = t0 + n;
    const int hi = t - i0, nwin = min(c, hi + 1);  // window rows hi, hi - 1, ... of token t
    const float keep = 1.f - sa[n], et = se[n], th2 = 2.f * sb[n];
    const float e0 = gam[0] * E[hi * rv + rr];
    float acc = 0.f, mx = -INFINITY, den = 0.f;
#pragma unroll
    for (int h = 0; h < CPL; h += CPL / 2) {  // two halves of the lane's columns
      float g[CPL / 2];
#pragma unroll
      for (int u = 0; u < CPL / 2; ++u) g[u] = e0 * fk(hi, min(sub + 4 * (h + u), D - 1));
      for (int w = 1; w < nwin; ++w) {
        const float ew = gam[w] * E[(hi - w) * rv + rr];
#pragma unroll
        for (int u = 0; u < CPL / 2; ++u)
          g[u] = fmaf(ew, fk(hi - w, min(sub + 4 * (h + u), D - 1)), g[u]);
      }
#pragma unroll
      for (int u = 0; u < CPL / 2; ++u) {
        const int j = sub + 4 * (h + u);
        if (j >= D) continue;
        const float s1 = et * sv[h + u] - th2 * g[u];
        sv[h + u] = s1;
        float v = fmaf(keep, m[h + u], s1);
        if (RK == ATLAS_RET_ELASTIC) {
          const float a = fabsf(v) - lam;
          v = a > 0.f ? copysignf(a, v) : 0.f;
          acc = fmaf(v, fq(n, j), acc);
        } else if (RK == ATLAS_RET_BREGMAN) {
          acc = fmaf(fq(n, j), __fdividef(1.f, 1.f + __expf(-v)), acc);
        } else {  // KL: the row's maximum first
          mx = fmaxf(mx, v);
        }
        m[h + u] = v;
      }
    }
    if (RK == ATLAS_RET_KL) {
      // M = c softmax(u): with the row maximum mx, den = sum exp(u - mx) and
      // num = sum exp(u - mx) q, the readout is c num / den and log M = u - shift
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
      float num = 0.f;
#pragma unroll
      for (int u = 0; u < CPL; ++u) {
        const int j = sub + 4 * u;
        if (j >= D) continue;
        const float e = __expf(m[u] - mx);
        den += e;
        num = fmaf(e, fq(n, j), num);
      }
      den = quad_sum(den);
      num = quad_sum(num);
      const float shift = mx + __logf(den) - logc;
#pragma unroll
      for (int u = 0; u < CPL; ++u) m[u] -= shift;
      acc = lam * num / den;  // lam carries the gate's parameter, here the row mass c
    } else {
      acc = quad_sum(acc);
    }
    if (sub == 0 && live) Y[(long)t * dv + row] = acc;
  }
#pragma unroll
  for (int u = 0; u < CPL; ++u) {
    const int j = sub + 4 * u;
    if (live && j < D) {
      Ms[row * Dp + j] = m[u];
      Ss[row * Dp + j] = sv[u];
    }
  }
}

__device__ __forceinline__ void lin_prefetch_l2(const void* a) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
}

// One CTA: rows [r0, r0 + RV) of one head, the whole sequence.  GATE: ATLAS_RET_L2
// for the chunk tables (the l2 and l_q gates), else the token-serial gate it names.
template <int GATE>
__device__ __forceinline__ void linear_simt_rows(const LinArgs& p, const LinSimtSmem& L, int head,
                                                 int r0);

// flags != nullptr: only the heads whose flag is set (the heads the tensor-core
// kernel leaves, which it marks); every other head returns at once, and each
// CTA walks all row blocks of its head so that the grid stays one CTA per head.
// Launched with programmatic stream serialisation when it follows the tensor-core
// kernel: it lets its own successor be scheduled, then waits for its predecessor.
template <int GATE>
__global__ void __launch_bounds__(256) linear_simt_kernel(LinArgs p, LinSimtSmem L,
                                                          const int* flags) {
  const int head = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  if (flags) {
    if (flags[head] == 0) return;
    for (int r0 = 0; r0 < p.d_v; r0 += L.RV) {
      linear_simt_rows<GATE>(p, L, head, r0);
      __syncthreads();
    }
    return;
  }
  linear_simt_rows<GATE>(p, L, head, blockIdx.y * L.RV);
}

template <int GATE>
__device__ __forceinline__ void linear_simt_rows(const LinArgs& p, const LinSimtSmem& L, int head,
                                                 int r0) {
  constexpr bool SERIAL = GATE != ATLAS_RET_L2;
  extern __shared__ float sm[];
  float* Ms = sm + L.Ms;
  float* Ss = sm + L.Ss;
  float* Kw = sm + L.Kw;
  float* Qc = sm + L.Qc;
  float* Vw = sm + L.Vw;
  float* E = sm + L.E;
  float* P = sm + L.P;
  float* Urun = sm + L.Urun;
  float* Wrun = sm + L.Wrun;
  float* sa = sm + L.sa;
  float* se = sm + L.se;
  float* sb = sm + L.sb;
  float* Z = sm + L.Z;
  float* coef = sm + L.coef;
  uint8_t* pp = reinterpret_cast<uint8_t*>(sm + L.total_floats);
  uint8_t* pq = pp + (L.D - p.d_k > 0 ? L.D - p.d_k : 0);
  uint32_t* ftab = reinterpret_cast<uint32_t*>(sm + L.total_floats);  // gated map

  const int rv = max(0, min(L.RV, p.d_v - r0));  // a cluster's last CTA may hold none
  const int D = L.D, dk = p.d_k, dv = p.d_v;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  const long state = (long)dv * D;
  const int Dp = L.Dp, dkp = L.dkp;

  if (tid < 5) coef[tid] = p.pcoef[tid];
  // pair table of the degree-2 map
  if (p.poly && tid == 0) {
    int o = 0;
    for (int i = 0; i < dk; ++i)
      for (int j = i; j < dk; ++j) { pp[o] = (uint8_t)i; pq[o] = (uint8_t)j; ++o; }
  }
  // monomial table of the gated map: degrees with a non-zero coefficient, each
  // degree's sorted index tuples in lexicographic order (the next tuple raises
  // the last entry that can still grow and resets the entries after it)
  if (p.pgen && tid == 0) {
    int o = 0;
    for (int e = 0; e <= p.pdeg; ++e) {
      if (p.pcoef[e] == 0.f) continue;
      int idx[4] = {0, 0, 0, 0};
      while (true) {
        uint32_t t = 0xFFFFFFFFu;
        for (int r = 0; r < e; ++r) t = (t & ~(0xFFu << (8 * r))) | ((uint32_t)idx[r] << (8 * r));
        ftab[o++] = t;
        int r = e - 1;
        while (r >= 0 && idx[r] == dk - 1) --r;
        if (r < 0) break;
        ++idx[r];
        for (int s2 = r + 1; s2 < e; ++s2) idx[s2] = idx[r];
      }
    }
  }
  const Feat fk{Kw, dkp, dk, p.poly, p.pgen, pp, pq, ftab, coef};
  const Feat fq{Qc, dkp, dk, p.poly, p.pgen, pp, pq, ftab, coef};
  float* Mg = p.M + head * state + (long)r0 * D;
  float* Sg = p.S ? p.S + head * state + (long)r0 * D : nullptr;
  const int ret = p.ret;
  constexpr bool serial = SERIAL;
  const int mk = ret == ATLAS_RET_BREGMAN ? 1 : ret == ATLAS_RET_KL ? 2 : 0;
  for (long x = tid; x < (long)rv * D; x += nt) {
    float m = Mg[x];
    if (ret == ATLAS_RET_BREGMAN) m = logf(m / (1.f - m));  // state as logits
    if (ret == ATLAS_RET_KL) m = logf(m);                   // state as log M
    const long xs = (x / D) * Dp + x % D;
    Ms[xs] = m;
    Ss[xs] = Sg ? Sg[x] : 0.f;
  }
  const float* alpha = p.alpha + (long)head * p.N;
  const float* eta = p.eta + (long)head * p.N;
  const float* theta = p.theta + (long)head * p.N;
  // K, V: head stride (nh + N) rows, token 0 at row nh; Q, Y: head stride N rows
  const long kbase = ((long)head * (p.N + p.nh) + p.nh) * dk;
  const long vbase = ((long)head * (p.N + p.nh) + p.nh) * dv;
  const long qbase = (long)head * p.N * dk;
  float* Yh = p.Y + (long)head * p.N * dv + r0;
  const float logc = ret == ATLAS_RET_KL ? logf(p.rp) : 0.f;
  const int cls = rows_class(rv);

  for (int t0 = 0; t0 < p.N; t0 += p.b) {
    const int t1 = min(p.N, t0 + p.b);
    const int nb = t1 - t0;
    const int i0 = max(-p.nh, t0 - p.c + 1);
    const int Lw = t1 - i0;
    __syncthreads();
    for (int x = tid; x < Lw * dk; x += nt)
      Kw[(x / dk) * dkp + x % dk] = ld_in(p.K, kbase + (long)i0 * dk + x, p.bf16);
    for (int x = tid; x < nb * dk; x += nt)
      Qc[(x / dk) * dkp + x % dk] = ld_in(p.Q, qbase + (long)t0 * dk + x, p.bf16);
    for (int x = tid; x < Lw * rv; x += nt) {
      const int i = x / rv, r = x % rv;
      Vw[x] = ld_in(p.V, vbase + (long)(i0 + i) * dv + r0 + r, p.bf16);
    }
    if (serial) {  // the gates of the chunk's tokens, and gamma by lag
      for (int n = tid; n < nb; n += nt) {
        sa[n] = alpha[t0 + n];
        se[n] = eta[t0 + n];
        sb[n] = theta[t0 + n];
      }
      for (int l = tid; l < p.c; l += nt) Urun[l] = p.gamma[l];
    } else {
      chunk_tables(alpha, eta, theta, p.gamma, t0, nb, i0, Lw, p.c, Urun, Wrun, P, L.Lmax,
                   nullptr, sa, se, sb, tid, nt);
    }
    // l_q: Z[r] = 1 / ||A_r||_q^(q-2) of the chunk-start accumulator (1 for a zero row)
    if (ret == ATLAS_RET_LQ) {
      for (int r = warp; r < rv; r += nw) {
        const float* m = Ms + (long)r * Dp;
        float acc = 0.f;
        for (int j = lane; j < D; j += 32) acc += powf(fabsf(m[j]), p.rp);
        acc = warp_sum(acc);
        if (lane == 0) Z[r] = acc > 0.f ? 1.f / powf(acc, (p.rp - 2.f) / p.rp) : 1.f;
      }
    }
    __syncthreads();
    if (t1 < p.N) {  // the next chunk's own K, Q and V rows into L2 ahead of their loads
      const int n1 = min(p.N, t1 + p.b), es = p.bf16 ? 2 : 4;
      const char* Kn = reinterpret_cast<const char*>(p.K) + (kbase + (long)t1 * dk) * es;
      const char* Qn = reinterpret_cast<const char*>(p.Q) + (qbase + (long)t1 * dk) * es;
      const int kl = ((n1 - t1) * dk * es + 127) / 128;
      for (int x = tid; x < kl; x += nt) {
        lin_prefetch_l2(Kn + 128 * (long)x);
        lin_prefetch_l2(Qn + 128 * (long)x);
      }
      const int segl = (rv * es + 127) / 128;  // lines of one V row segment
      for (int x = tid; x < (n1 - t1) * segl; x += nt)
        lin_prefetch_l2(reinterpret_cast<const char*>(p.V) +
                        (vbase + (long)(t1 + x / segl) * dv + r0) * es + 128 * (x % segl));
    }
    // errors at the chunk-start memory
    if (p.dot) {
      for (int x = tid; x < Lw * rv; x += nt) E[x] = -Vw[x];
    } else {
      const bool lq = ret == ATLAS_RET_LQ;
      auto fe = [&](int i, int r, float acc) {
        const float s = lq ? acc * Z[r] : acc;
        E[i * rv + r] = bias_grad(s - Vw[i * rv + r], p.lk, p.lp);
      };
      if constexpr (!SERIAL) {
        auto fb = [&](int j, int r) { return Ms[r * Dp + j]; };
        gemm_by_rows(cls, Lw, rv, D, fk, fb, fe);
      } else {
        auto fb = [&](int j, int r) {
          const float m = Ms[r * Dp + j];
          return mk == 1 ? mem_entry<1>(m) : mk == 2 ? mem_entry<2>(m) : m;
        };
        gemm_by_rows(cls, Lw, rv, D, fk, fb, fe);
      }
    }
    if (p.lk == ATLAS_LOSS_ROBUST) {
      float* NR = sm + L.NR;
      __syncthreads();
      for (int i = warp; i < Lw; i += nw) {  // this CTA's part of ||e_i||^2
        const float* e = E + i * rv;
        float ss = 0.f;
        for (int r = lane; r < rv; r += 32) ss += e[r] * e[r];
        ss = warp_sum(ss);
        if (lane == 0) NR[i] = ss;
      }
      namespace cg = cooperative_groups;
      if (L.ncl > 1)
        cg::this_cluster().sync();
      else
        __syncthreads();
      for (int i = warp; i < Lw; i += nw) {
        float part = 0.f;
        if (L.ncl > 1) {
          if (lane < L.ncl) part = *cg::this_cluster().map_shared_rank(NR + i, lane);
        } else if (lane == 0) {
          part = NR[i];
        }
        const float f = robust_scale(sqrtf(warp_sum(part)), p.lp);
        float* e = E + i * rv;
        for (int r = lane; r < rv; r += 32) e[r] *= f;
      }
      if (L.ncl > 1) cg::this_cluster().sync();  // every rank has read NR
    }
    if constexpr (SERIAL) {
      __syncthreads();
      if (D <= 128 && rv <= 64) {
        if (!p.poly && !p.pgen)  // the identity map: features are the key and query entries
          serial_chunk_quad<GATE>(nb, t0, i0, p.c, rv, D, Dp, Ms, Ss, E, FeatId{Qc, dkp},
                                  FeatId{Kw, dkp}, sa, se, sb, Urun, p.rp, logc, Yh, dv);
        else
          serial_chunk_quad<GATE>(nb, t0, i0, p.c, rv, D, Dp, Ms, Ss, E, fq, fk, sa, se, sb, Urun,
                                  p.rp, logc, Yh, dv);
        continue;
      }
      // wide feature maps: one warp per row, lanes over the columns
      for (int n = 0; n < nb; ++n) {
        const int t = t0 + n;
        const float keep = 1.f - sa[n], et = se[n], th2 = 2.f * sb[n];
        const int hi = t - i0, lo = max(0, hi - p.c + 1);  // window rows of token t
        for (int r = warp; r < rv; r += nw) {
          float* m = Ms + (long)r * Dp;
          float* sr = Ss + (long)r * Dp;
          float acc = 0.f, mx = -INFINITY, den = 0.f;
          for (int j = lane; j < D; j += 32) {
            float g = 0.f;
            for (int i = lo; i <= hi; ++i) g += Urun[hi - i] * E[i * rv + r] * fk(i, j);
            const float sv = et * sr[j] - th2 * g;
            sr[j] = sv;
            float u = keep * m[j] + sv;
            if (ret == ATLAS_RET_ELASTIC) {
              const float a = fabsf(u) - p.rp;
              u = a > 0.f ? copysignf(a, u) : 0.f;
              acc += u * fq(n, j);
            } else if (ret == ATLAS_RET_BREGMAN) {
              acc += fq(n, j) / (1.f + expf(-u));
            } else {  // KL: running max and sum of exp for the row's softmax
              if (u > mx) {
                den = den * expf(mx - u) + 1.f;
                mx = u;
              } else {
                den += expf(u - mx);
              }
            }
            m[j] = u;
          }
          if (ret == ATLAS_RET_KL) {
            warp_lse(mx, den);
            const float shift = mx + logf(den) - logc;  // log M = u - lse(u) + log c
            for (int j = lane; j < D; j += 32) {
              const float lm = m[j] - shift;
              m[j] = lm;
              acc += expf(lm) * fq(n, j);
            }
          }
          acc = warp_sum(acc);
          if (lane == 0) Yh[(long)t * dv + r] = acc;
        }
      }
      continue;
    }
    if constexpr (!SERIAL) {
      // masked query-key products P[n,i] = W[n,i] * Phi(q_n).Phi(k_i)
      if (p.pgen)
        qk_tile<4>(nb, Lw, dk, Qc, Kw, dkp, P, L.Lmax, 2, coef, p.pdeg);
      else if (p.poly)
        qk_tile<2>(nb, Lw, dk, Qc, Kw, dkp, P, L.Lmax, 1, coef, 0);
      else
        qk_tile<1>(nb, Lw, dk, Qc, Kw, dkp, P, L.Lmax, 0, coef, 0);
      __syncthreads();
      // readout y_n = M_n Phi(q_n) (l_q: the accumulator's row times Z)
      {
        bool with_s = false;
        for (int n = 0; n < nb; ++n) with_s |= sb[n] != 0.f;
        const float* zr = ret == ATLAS_RET_LQ ? Z : nullptr;
        float* Yc = Yh + (long)t0 * dv;
        switch (cls) {
          case 1: readout_tile<16, 4, 1>(nb, rv, D, Lw, fq, Ms, Ss, Dp, P, L.Lmax, E, sa, sb, with_s, zr, Yc, dv); break;
          case 2: readout_tile<16, 4, 2>(nb, rv, D, Lw, fq, Ms, Ss, Dp, P, L.Lmax, E, sa, sb, with_s, zr, Yc, dv); break;
          case 3: readout_tile<16, 4, 4>(nb, rv, D, Lw, fq, Ms, Ss, Dp, P, L.Lmax, E, sa, sb, with_s, zr, Yc, dv); break;
          default: readout_tile<16, 4, 8>(nb, rv, D, Lw, fq, Ms, Ss, Dp, P, L.Lmax, E, sa, sb, with_s, zr, Yc, dv); break;
        }
      }
      __syncthreads();
      // carry the state to the end of the chunk
      {
        const float a_b = sa[nb - 1], e_b = se[nb - 1], b_b = sb[nb - 1];
        switch (cls) {
          case 1: carry_tile<16, 1, 8>(rv, D, Lw, fk, E, Wrun, Urun, Ms, Ss, Dp, a_b, b_b, e_b); break;
          case 2: carry_tile<16, 2, 8>(rv, D, Lw, fk, E, Wrun, Urun, Ms, Ss, Dp, a_b, b_b, e_b); break;
          case 3: carry_tile<16, 4, 8>(rv, D, Lw, fk, E, Wrun, Urun, Ms, Ss, Dp, a_b, b_b, e_b); break;
          default: carry_tile<16, 8, 4>(rv, D, Lw, fk, E, Wrun, Urun, Ms, Ss, Dp, a_b, b_b, e_b); break;
        }
      }
    }
  }
  __syncthreads();
  for (long x = tid; x < (long)rv * D; x += nt) {
    const long xs = (x / D) * Dp + x % D;
    float m = Ms[xs];
    if (mk == 1) m = mem_entry<1>(m);
    if (mk == 2) m = mem_entry<2>(m);
    Mg[x] = m;
    if (Sg) Sg[x] = Ss[xs];
  }
}

// Launches of the token-serial instantiations (one translation unit each).
cudaError_t linear_simt_elastic_launch(const cudaLaunchConfig_t* cfg, const LinArgs& a,
                                       const LinSimtSmem& s, const int* flags);
cudaError_t linear_simt_bregman_launch(const cudaLaunchConfig_t* cfg, const LinArgs& a,
                                       const LinSimtSmem& s, const int* flags);
cudaError_t linear_simt_kl_launch(const cudaLaunchConfig_t* cfg, const LinArgs& a,
                                  const LinSimtSmem& s, const int* flags);

// Sets the kernel's shared-memory limit and launches it.
template <int GATE>
cudaError_t linear_simt_launch_gate(const cudaLaunchConfig_t* cfg, const LinArgs& a,
                                    const LinSimtSmem& s, const int* flags) {
  const cudaError_t e = cudaFuncSetAttribute(linear_simt_kernel<GATE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)cfg->dynamicSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(cfg, linear_simt_kernel<GATE>, a, s, flags);
}

}  // namespace atlas
