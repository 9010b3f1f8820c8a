// linear_simt.cu -- chunked Omega-rule update of a linear matrix memory on
// CUDA cores (fp32), for any feature map, window, chunk and gate setting.
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
// with the scalar tables of chunk_tables_warp.  Phi(q).Phi(k) for the degree-2
// map is evaluated as s + (s^2 + sum_j q_j^2 k_j^2)/2 with s = q.k, which is the
// same sum regrouped.  The gated polynomial map of any degree ("논문 리뷰 Google
// ATLAS" §3.1, Input gating) keeps one 32-bit entry per feature (its sorted
// monomial indices, 0xFF past its degree) in shared memory, and its lifted inner
// product is sum_e a_e^2 h_e(z), z_j = q_j k_j, with the complete homogeneous
// symmetric polynomials h_e from the power sums of z (Newton's identities).
#include "common.cuh"
#include "kernels.h"

namespace atlas {

struct LinSimtSmem {
  int RV, D, Lmax, b, d_k, pgen;
  // float offsets
  long Ms, Ss, Kw, Qc, Vw, E, P, Urun, Wrun, sa, se, sb, total_floats;
  long pairs_bytes;
  size_t bytes() const { return total_floats * sizeof(float) + pairs_bytes; }
};

static LinSimtSmem lin_simt_layout(int RV, int D, int Lmax, int b, int d_k, int pgen) {
  LinSimtSmem s;
  s.RV = RV; s.D = D; s.Lmax = Lmax; s.b = b; s.d_k = d_k; s.pgen = pgen;
  long o = 0;
  s.Ms = o; o += (long)RV * D;
  s.Ss = o; o += (long)RV * D;
  s.Kw = o; o += (long)Lmax * d_k;
  s.Qc = o; o += (long)b * d_k;
  s.Vw = o; o += (long)Lmax * RV;
  s.E = o; o += (long)Lmax * RV;
  s.P = o; o += (long)b * Lmax;
  s.Urun = o; o += Lmax;
  s.Wrun = o; o += Lmax;
  s.sa = o; o += b;
  s.se = o; o += b;
  s.sb = o; o += b;
  s.total_floats = o;
  s.pairs_bytes = pgen ? 4L * D : 2L * (D - d_k > 0 ? D - d_k : 0);
  return s;
}

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

// Phi(q).Phi(k) of the gated map: sum_e a_e^2 h_e(z), z_j = q_j k_j.
__device__ __forceinline__ float phi_gated_dot(const float* q, const float* k, int dk,
                                               const float* a, int deg) {
  float pw[5] = {0.f, 0.f, 0.f, 0.f, 0.f};  // power sums p_1 .. p_4
  for (int j = 0; j < dk; ++j) {
    const float z = q[j] * k[j];
    float zz = z;
#pragma unroll
    for (int m = 1; m <= 4; ++m) {
      if (m <= deg) pw[m] += zz;
      zz *= z;
    }
  }
  float h[5];
  h[0] = 1.f;
  float v = a[0] * a[0];
#pragma unroll
  for (int m = 1; m <= 4; ++m) {
    float s = 0.f;
#pragma unroll
    for (int i = 1; i <= m; ++i) s += pw[i] * h[m - i];
    h[m] = s / (float)m;
    if (m <= deg) v += a[m] * a[m] * h[m];
  }
  return v;
}

// One CTA: rows [r0, r0 + RV) of one head, the whole sequence.
__device__ __forceinline__ void linear_simt_rows(const LinArgs& p, const LinSimtSmem& L, int head,
                                                 int r0);

// flags != nullptr: only the heads whose flag is set (the heads the tensor-core
// kernel leaves, which it marks); every other head returns at once, and each
// CTA walks all row blocks of its head so that the grid stays one CTA per head.
__global__ void __launch_bounds__(256) linear_simt_kernel(LinArgs p, LinSimtSmem L,
                                                          const int* flags) {
  const int head = blockIdx.x;
  if (flags) {
    if (flags[head] == 0) return;
    for (int r0 = 0; r0 < p.d_v; r0 += L.RV) {
      linear_simt_rows(p, L, head, r0);
      __syncthreads();
    }
    return;
  }
  linear_simt_rows(p, L, head, blockIdx.y * L.RV);
}

__device__ __forceinline__ void linear_simt_rows(const LinArgs& p, const LinSimtSmem& L, int head,
                                                 int r0) {
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
  uint8_t* pp = reinterpret_cast<uint8_t*>(sm + L.total_floats);
  uint8_t* pq = pp + (L.D - p.d_k > 0 ? L.D - p.d_k : 0);
  uint32_t* ftab = reinterpret_cast<uint32_t*>(sm + L.total_floats);  // gated map


  const int rv = min(L.RV, p.d_v - r0);
  const int D = L.D, dk = p.d_k, dv = p.d_v;
  const int tid = threadIdx.x, nt = blockDim.x;
  const long state = (long)dv * D;

  // pair table of the degree-2 map
  if (p.poly) {
    if (tid == 0) {
      int o = 0;
      for (int i = 0; i < dk; ++i)
        for (int j = i; j < dk; ++j) { pp[o] = (uint8_t)i; pq[o] = (uint8_t)j; ++o; }
    }
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
  auto feat = [&](const float* x, int j) -> float {
    return p.pgen ? phi_gated(x, ftab[j], p.pcoef) : phi_at(x, j, dk, pp, pq, p.poly);
  };
  float* Mg = p.M + head * state + (long)r0 * D;
  float* Sg = p.S ? p.S + head * state + (long)r0 * D : nullptr;
  for (long x = tid; x < (long)rv * D; x += nt) {
    Ms[x] = Mg[x];
    Ss[x] = Sg ? Sg[x] : 0.f;
  }
  const float* alpha = p.alpha + (long)head * p.N;
  const float* eta = p.eta + (long)head * p.N;
  const float* theta = p.theta + (long)head * p.N;
  // K, V: head stride (nh + N) rows, token 0 at row nh; Q, Y: head stride N rows
  const long kbase = ((long)head * (p.N + p.nh) + p.nh) * dk;
  const long vbase = ((long)head * (p.N + p.nh) + p.nh) * dv;
  const long qbase = (long)head * p.N * dk;
  const long ybase = (long)head * p.N * dv;

  for (int t0 = 0; t0 < p.N; t0 += p.b) {
    const int t1 = min(p.N, t0 + p.b);
    const int nb = t1 - t0;
    const int i0 = max(-p.nh, t0 - p.c + 1);
    const int Lw = t1 - i0;
    __syncthreads();
    for (int x = tid; x < Lw * dk; x += nt) Kw[x] = ld_in(p.K, kbase + (long)i0 * dk + x, p.bf16);
    for (int x = tid; x < nb * dk; x += nt) Qc[x] = ld_in(p.Q, qbase + (long)t0 * dk + x, p.bf16);
    for (int x = tid; x < Lw * rv; x += nt) {
      const int i = x / rv, r = x % rv;
      Vw[x] = ld_in(p.V, vbase + (long)(i0 + i) * dv + r0 + r, p.bf16);
    }
    if (tid < 32)
      chunk_tables_warp(alpha, eta, theta, p.gamma, t0, nb, i0, Lw, p.c, Urun, Wrun, P, L.Lmax,
                        nullptr, sa, se, sb);
    __syncthreads();
    // errors at the chunk-start state
    for (int x = tid; x < Lw * rv; x += nt) {
      const int i = x / rv, r = x % rv;
      float e;
      if (p.dot) {
        e = -Vw[x];
      } else {
        const float* m = Ms + (long)r * D;
        const float* k = Kw + i * dk;
        float s = 0.f;
        for (int j = 0; j < D; ++j) s += m[j] * feat(k, j);
        e = bias_grad(s - Vw[x], p.lk, p.lp);
      }
      E[x] = e;
    }
    // masked query-key products P[n,i] = W[n,i] * Phi(q_n).Phi(k_i)
    for (int x = tid; x < nb * Lw; x += nt) {
      const int n = x / Lw, i = x % Lw;
      const float w = P[n * L.Lmax + i];
      float v = 0.f;
      if (w != 0.f) {
        const float* q = Qc + n * dk;
        const float* k = Kw + i * dk;
        if (p.pgen) {
          v = phi_gated_dot(q, k, dk, p.pcoef, p.pdeg);
        } else {
          float s = 0.f, s2 = 0.f;
          for (int j = 0; j < dk; ++j) {
            const float qk = q[j] * k[j];
            s += qk;
            s2 += qk * qk;
          }
          v = p.poly ? s + 0.5f * (s * s + s2) : s;
        }
        v *= w;
      }
      P[n * L.Lmax + i] = v;
    }
    __syncthreads();
    // readout y_n = M_n Phi(q_n)
    for (int x = tid; x < nb * rv; x += nt) {
      const int n = x / rv, r = x % rv;
      const float* q = Qc + n * dk;
      const float* m = Ms + (long)r * D;
      const float* s = Ss + (long)r * D;
      float ym = 0.f, ys = 0.f;
      for (int j = 0; j < D; ++j) {
        const float f = feat(q, j);
        ym += m[j] * f;
        ys += s[j] * f;
      }
      float acc = 0.f;
      for (int i = 0; i < Lw; ++i) acc += P[n * L.Lmax + i] * E[i * rv + r];
      p.Y[ybase + (long)(t0 + n) * dv + r0 + r] = sa[n] * ym + sb[n] * ys - 2.f * acc;
    }
    __syncthreads();
    // carry the state to the end of the chunk
    const float a_b = sa[nb - 1], e_b = se[nb - 1], b_b = sb[nb - 1];
    for (long x = tid; x < (long)rv * D; x += nt) {
      const int r = (int)(x / D), j = (int)(x % D);
      float gw = 0.f, gu = 0.f;
      for (int i = 0; i < Lw; ++i) {
        const float f = E[i * rv + r] * feat(Kw + i * dk, j);
        gw += Wrun[i] * f;
        gu += Urun[i] * f;
      }
      const float m0 = Ms[x], s0 = Ss[x];
      Ms[x] = a_b * m0 + b_b * s0 - 2.f * gw;
      Ss[x] = e_b * s0 - 2.f * gu;
    }
  }
  __syncthreads();
  for (long x = tid; x < (long)rv * D; x += nt) {
    Mg[x] = Ms[x];
    if (Sg) Sg[x] = Ss[x];
  }
}

int linear_simt_plan(const LinArgs& a, int heads, int* RV_out, size_t* smem_out) {
  const int Lmax = a.b + a.c - 1;
  const size_t limit = 200 * 1024;
  int RV = a.d_v;
  while (RV > 1) {
    LinSimtSmem s = lin_simt_layout(RV, a.D, Lmax, a.b, a.d_k, a.pgen);
    const long ctas = (long)heads * ((a.d_v + RV - 1) / RV);
    if (s.bytes() <= limit && (ctas >= 152 || RV <= 4)) break;
    RV = (RV + 1) / 2;
  }
  LinSimtSmem s = lin_simt_layout(RV, a.D, Lmax, a.b, a.d_k, a.pgen);
  if (s.bytes() > limit) return ATLAS_ERR_UNSUPPORTED;
  *RV_out = RV;
  *smem_out = s.bytes();
  return ATLAS_OK;
}

static int launch(const LinArgs& a, int heads, const int* flags, cudaStream_t st) {
  int RV;
  size_t smem;
  int rc = linear_simt_plan(a, heads, &RV, &smem);
  if (rc) return rc;
  LinSimtSmem s = lin_simt_layout(RV, a.D, a.b + a.c - 1, a.b, a.d_k, a.pgen);
  if (cudaFuncSetAttribute(linear_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return ATLAS_ERR_CUDA;
  dim3 grid(heads, flags ? 1 : (a.d_v + RV - 1) / RV);
  linear_simt_kernel<<<grid, 256, smem, st>>>(a, s, flags);
  return cudaGetLastError() == cudaSuccess ? ATLAS_OK : ATLAS_ERR_CUDA;
}

int linear_simt_launch(const LinArgs& a, int heads, cudaStream_t st) {
  return launch(a, heads, nullptr, st);
}

int linear_simt_launch_flagged(const LinArgs& a, int heads, const int* flags, cudaStream_t st) {
  return launch(a, heads, flags, st);
}

}  // namespace atlas
