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
// The robust bias scales each window token's error row by 1 + Delta/||e||, which
// needs the norm over all d_v rows of the head.  Its row blocks therefore form
// one thread-block cluster per head (at most 8 CTAs): each CTA writes the partial
// squared norms of its rows to shared memory, and after a cluster barrier every
// CTA adds the partials of all ranks through distributed shared memory; a second
// barrier keeps them until every rank has read them.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace atlas {

struct LinSimtSmem {
  int RV, D, Lmax, b, d_k, pgen;
  int ncl;  // CTAs per head in one cluster (robust bias), else 1
  // float offsets
  long Ms, Ss, Kw, Qc, Vw, E, P, Urun, Wrun, sa, se, sb, Z, NR, total_floats;
  long pairs_bytes;
  size_t bytes() const { return total_floats * sizeof(float) + pairs_bytes; }
};

static LinSimtSmem lin_simt_layout(int RV, int D, int Lmax, int b, int d_k, int pgen) {
  LinSimtSmem s;
  s.RV = RV; s.D = D; s.Lmax = Lmax; s.b = b; s.d_k = d_k; s.pgen = pgen; s.ncl = 1;
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
  s.Z = o; o += RV;
  s.NR = o; o += Lmax;
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


  const int rv = max(0, min(L.RV, p.d_v - r0));  // a cluster's last CTA may hold none
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
  const int ret = p.ret;
  const bool serial = ret == ATLAS_RET_ELASTIC || ret == ATLAS_RET_BREGMAN || ret == ATLAS_RET_KL;
  for (long x = tid; x < (long)rv * D; x += nt) {
    float m = Mg[x];
    if (ret == ATLAS_RET_BREGMAN) m = logf(m / (1.f - m));  // state as logits
    if (ret == ATLAS_RET_KL) m = logf(m);                   // state as log M
    Ms[x] = m;
    Ss[x] = Sg ? Sg[x] : 0.f;
  }
  // the memory entry a state entry stands for at a chunk start (l_q: before the
  // row scale Z)
  auto mem_of = [&](float m) -> float {
    if (ret == ATLAS_RET_BREGMAN) return 1.f / (1.f + expf(-m));
    if (ret == ATLAS_RET_KL) return expf(m);
    return m;
  };
  const float* alpha = p.alpha + (long)head * p.N;
  const float* eta = p.eta + (long)head * p.N;
  const float* theta = p.theta + (long)head * p.N;
  // K, V: head stride (nh + N) rows, token 0 at row nh; Q, Y: head stride N rows
  const long kbase = ((long)head * (p.N + p.nh) + p.nh) * dk;
  const long vbase = ((long)head * (p.N + p.nh) + p.nh) * dv;
  const long qbase = (long)head * p.N * dk;
  const long ybase = (long)head * p.N * dv;
  const int lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  float* Z = sm + L.Z;
  const float logc = ret == ATLAS_RET_KL ? logf(p.rp) : 0.f;

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
    if (serial) {  // the gates of the chunk's tokens, and gamma by lag
      for (int n = tid; n < nb; n += nt) {
        sa[n] = alpha[t0 + n];
        se[n] = eta[t0 + n];
        sb[n] = theta[t0 + n];
      }
      for (int l = tid; l < p.c; l += nt) Urun[l] = p.gamma[l];
    } else if (tid < 32) {
      chunk_tables_warp(alpha, eta, theta, p.gamma, t0, nb, i0, Lw, p.c, Urun, Wrun, P, L.Lmax,
                        nullptr, sa, se, sb);
    }
    // l_q: Z[r] = 1 / ||A_r||_q^(q-2) of the chunk-start accumulator (1 for a zero row)
    if (ret == ATLAS_RET_LQ) {
      for (int r = warp; r < rv; r += nw) {
        const float* m = Ms + (long)r * D;
        float acc = 0.f;
        for (int j = lane; j < D; j += 32) acc += powf(fabsf(m[j]), p.rp);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        if (lane == 0) Z[r] = acc > 0.f ? 1.f / powf(acc, (p.rp - 2.f) / p.rp) : 1.f;
      }
    }
    __syncthreads();
    // errors at the chunk-start memory
    for (int x = tid; x < Lw * rv; x += nt) {
      const int i = x / rv, r = x % rv;
      float e;
      if (p.dot) {
        e = -Vw[x];
      } else {
        const float* m = Ms + (long)r * D;
        const float* k = Kw + i * dk;
        float s = 0.f;
        for (int j = 0; j < D; ++j) s += mem_of(m[j]) * feat(k, j);
        if (ret == ATLAS_RET_LQ) s *= Z[r];
        e = bias_grad(s - Vw[x], p.lk, p.lp);
      }
      E[x] = e;
    }
    if (p.lk == ATLAS_LOSS_ROBUST) {
      float* NR = sm + L.NR;
      __syncthreads();
      for (int i = warp; i < Lw; i += nw) {  // this CTA's part of ||e_i||^2
        const float* e = E + i * rv;
        float ss = 0.f;
        for (int r = lane; r < rv; r += 32) ss += e[r] * e[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
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
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
        const float f = robust_scale(sqrtf(part), p.lp);
        float* e = E + i * rv;
        for (int r = lane; r < rv; r += 32) e[r] *= f;
      }
      if (L.ncl > 1) cg::this_cluster().sync();  // every rank has read NR
    }
    if (serial) {
      __syncthreads();
      // token by token; warp w owns rows w, w + nw, ... for the whole chunk
      for (int n = 0; n < nb; ++n) {
        const int t = t0 + n;
        const float keep = 1.f - sa[n], et = se[n], th2 = 2.f * sb[n];
        const int hi = t - i0, lo = max(0, hi - p.c + 1);  // window rows of token t
        const float* q = Qc + n * dk;
        for (int r = warp; r < rv; r += nw) {
          float* m = Ms + (long)r * D;
          float* sr = Ss + (long)r * D;
          float acc = 0.f, mx = -INFINITY, den = 0.f;
          for (int j = lane; j < D; j += 32) {
            float g = 0.f;
            for (int i = lo; i <= hi; ++i) g += Urun[hi - i] * E[i * rv + r] * feat(Kw + i * dk, j);
            const float sv = et * sr[j] - th2 * g;
            sr[j] = sv;
            float u = keep * m[j] + sv;
            if (ret == ATLAS_RET_ELASTIC) {
              const float a = fabsf(u) - p.rp;
              u = a > 0.f ? copysignf(a, u) : 0.f;
              acc += u * feat(q, j);
            } else if (ret == ATLAS_RET_BREGMAN) {
              acc += feat(q, j) / (1.f + expf(-u));
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
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              const float om = __shfl_xor_sync(0xFFFFFFFFu, mx, o);
              const float od = __shfl_xor_sync(0xFFFFFFFFu, den, o);
              const float nm = fmaxf(mx, om);
              den = (den > 0.f ? den * expf(mx - nm) : 0.f) + (od > 0.f ? od * expf(om - nm) : 0.f);
              mx = nm;
            }
            // log M = u - logsumexp(u) + log c
            const float shift = mx + logf(den) - logc;
            for (int j = lane; j < D; j += 32) {
              const float lm = m[j] - shift;
              m[j] = lm;
              acc += expf(lm) * feat(q, j);
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
          if (lane == 0) p.Y[ybase + (long)t * dv + r0 + r] = acc;
        }
      }
      continue;
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
    // readout y_n = M_n Phi(q_n) (l_q: the accumulator's row times Z)
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
      float y = sa[n] * ym + sb[n] * ys - 2.f * acc;
      if (ret == ATLAS_RET_LQ) y *= Z[r];
      p.Y[ybase + (long)(t0 + n) * dv + r0 + r] = y;
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
    Mg[x] = serial ? mem_of(Ms[x]) : Ms[x];
    if (Sg) Sg[x] = Ss[x];
  }
}

// Rows per CTA (RV) and CTAs per cluster (robust bias only; a head's row blocks
// form one cluster of ncl <= 8 CTAs, so RV = ceil(d_v / ncl)).
static int plan(const LinArgs& a, int heads, LinSimtSmem* out) {
  const int Lmax = a.b + a.c - 1;
  const size_t limit = 200 * 1024;
  const bool robust = a.lk == ATLAS_LOSS_ROBUST;
  int RV = a.d_v, ncl = 1;
  while (RV > 1) {
    LinSimtSmem s = lin_simt_layout(RV, a.D, Lmax, a.b, a.d_k, a.pgen);
    const long ctas = (long)heads * ((a.d_v + RV - 1) / RV);
    if (s.bytes() <= limit && (ctas >= 152 || RV <= 4)) break;
    if (robust) {
      if (ncl == 8) break;
      ncl *= 2;
      RV = (a.d_v + ncl - 1) / ncl;
    } else {
      RV = (RV + 1) / 2;
    }
  }
  LinSimtSmem s = lin_simt_layout(RV, a.D, Lmax, a.b, a.d_k, a.pgen);
  if (s.bytes() > limit) return ATLAS_ERR_UNSUPPORTED;
  s.ncl = robust ? ncl : 1;
  *out = s;
  return ATLAS_OK;
}

int linear_simt_plan(const LinArgs& a, int heads, int* RV_out, size_t* smem_out) {
  LinSimtSmem s;
  const int rc = plan(a, heads, &s);
  if (rc) return rc;
  *RV_out = s.RV;
  *smem_out = s.bytes();
  return ATLAS_OK;
}

static int launch(const LinArgs& a, int heads, const int* flags, cudaStream_t st) {
  LinSimtSmem s;
  int rc = plan(a, heads, &s);
  if (rc) return rc;
  if (flags && s.ncl > 1) return ATLAS_ERR_UNSUPPORTED;
  const size_t smem = s.bytes();
  if (cudaFuncSetAttribute(linear_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return ATLAS_ERR_CUDA;
  const int rows = flags ? 1 : (s.ncl > 1 ? s.ncl : (a.d_v + s.RV - 1) / s.RV);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(heads, rows);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (s.ncl > 1) {  // one cluster per head: its ncl row blocks
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = s.ncl;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if (cudaLaunchKernelEx(&cfg, linear_simt_kernel, a, s, flags) != cudaSuccess)
    return ATLAS_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ATLAS_OK : ATLAS_ERR_CUDA;
}

int linear_simt_launch(const LinArgs& a, int heads, cudaStream_t st) {
  return launch(a, heads, nullptr, st);
}

int linear_simt_launch_flagged(const LinArgs& a, int heads, const int* flags, cudaStream_t st) {
  return launch(a, heads, flags, st);
}

}  // namespace atlas
