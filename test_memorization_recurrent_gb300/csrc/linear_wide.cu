// linear_wide.cu -- chunked Omega-rule update of a linear memory with a wide
// feature map (D >= 256 features: the degree-2 map, the gated polynomial map),
// every chunk on device, the state on chip for the whole sequence.
//
// One thread-block cluster of CL CTAs per head; CTA c owns the feature columns
// [c DJ, (c + 1) DJ) of M and S (all d_v rows) in shared memory.  Per chunk of
// nb tokens starting at t0, window tokens i0..t1-1 (Lw of them) -- "논문 리뷰
// Google ATLAS" §3.1 (feature map), §3.2 (Omega rule), §3.3 (gradients at the
// chunk-start state); "[Paper Review] Titans 논문 이해하기" (momentum, decay,
// readout after the write):
//   E[i,r]  = bias(M0[r,:].Phi(k_i) - v_i[r])
//   y_n[r]  = a_n M0[r,:].Phi(q_n) + beta_n S0[r,:].Phi(q_n) - 2 sum_i W[n,i] (Phi(q_n).Phi(k_i)) E[i,r]
//   M[r,:]  = a_b M0 + beta_b S0 - 2 sum_i W[b,i] E[i,r] Phi(k_i),  S likewise with U
// (the scalar tables of chunk_tables).  The products over the feature
// dimension split by column slice: each CTA forms the partial errors and the
// partial readout of its slice, and the cluster adds them through distributed
// shared memory -- CTA c sums the partials of every rank for its share of the
// window rows (and applies the bias, which sees whole error rows, so the robust
// bias fits here too) and for its share of the chunk's queries (and adds their
// intra-chunk term, which needs the finished errors of the whole window).  Every
// CTA then copies the finished error rows of the others and carries its own
// columns of M and S.  Features are evaluated from the keys and queries in
// shared memory as the products read them; nothing of Phi is stored.
//
// Three cluster barriers per chunk: after the partial errors (A), after the
// finished error rows (B), after the partial readout (D).  Every remote read of
// a buffer happens between the barrier that publishes it and the next barrier,
// and a rank writes that buffer again only after passing that next barrier, so
// no rank overwrites what another still reads.  A last barrier keeps every
// CTA's shared memory until all ranks have read it.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "simt_tiles.cuh"

namespace atlas {

namespace cg = cooperative_groups;

struct WideSmem {
  int CL, DJ, DJp, dv, Lmax, b, dk, dkp, D;
  // float offsets
  long Ms, Ss, Kw, Qc, E, EP, YP, Wt, Wrun, Urun, sa, se, sb, coef, total_floats;
  long pairs_bytes;
  size_t bytes() const { return total_floats * sizeof(float) + pairs_bytes; }
};

static WideSmem wide_layout(const LinArgs& a, int CL) {
  WideSmem s;
  s.CL = CL;
  s.D = a.D;
  s.dv = a.d_v;
  s.b = a.b;
  s.dk = a.d_k;
  s.dkp = a.d_k | 1;
  s.Lmax = a.b + a.c - 1;
  s.DJ = ((a.D + CL - 1) / CL + 15) / 16 * 16;  // slice width, a multiple of 16
  s.DJp = s.DJ | 1;
  long o = 0;
  s.Ms = o; o += (long)s.dv * s.DJp;
  s.Ss = o; o += (long)s.dv * s.DJp;
  s.Kw = o; o += (long)s.Lmax * s.dkp;
  s.Qc = o; o += (long)s.b * s.dkp;
  s.E = o; o += (long)s.Lmax * s.dv;
  s.EP = o; o += (long)s.Lmax * s.dv;
  s.YP = o; o += (long)s.b * s.dv;
  s.Wt = o; o += (long)s.b * s.Lmax;
  s.Wrun = o; o += s.Lmax;
  s.Urun = o; o += s.Lmax;
  s.sa = o; o += s.b;
  s.se = o; o += s.b;
  s.sb = o; o += s.b;
  s.coef = o; o += 8;
  s.total_floats = o;
  s.pairs_bytes = a.pgen ? 4L * a.D : 2L * (a.D - a.d_k > 0 ? a.D - a.d_k : 0);
  return s;
}

constexpr size_t kWideSmemLimit = 225 * 1024;

// The degree-2 map alone (no gated-map branch): x_j, then the pair products.
struct FeatP2 {
  const float* x;
  int ld, dk;
  const uint8_t* pp;
  const uint8_t* pq;
  __device__ __forceinline__ float operator()(int row, int j) const {
    const float* r = x + row * ld;
    return j < dk ? r[j] : r[pp[j - dk]] * r[pq[j - dk]];
  }
};

// Features of a column slice: feature j0 + j of row `row`.
template <class F>
struct FeatSlice {
  F f;
  int j0;
  __device__ __forceinline__ float operator()(int row, int j) const { return f(row, j0 + j); }
};

// Rows [lo, hi) of `n` items split over CL ranks.
__device__ __forceinline__ int share_lo(int n, int CL, int c) { return (int)((long)n * c / CL); }

// Partial readout of the slice: YP[n, r] = sa_n Phi(q_n).M[r] + sb_n Phi(q_n).S[r]
// (slice columns only; the S term skipped when every sb_n is 0).
template <int TX, int TM, int TN, class FQ>
__device__ __forceinline__ void readout_partial(int nb, int dv, int dj, const FQ& fq,
                                                const float* Ms, const float* Ss, int DJp,
                                                const float* sa, const float* sb, bool with_s,
                                                float* YP) {
  constexpr int TY = 256 / TX;
  const int tx = threadIdx.x % TX, ty = threadIdx.x / TX;
  for (int m0 = 0; m0 < nb; m0 += TY * TM)
    for (int n0 = 0; n0 < dv; n0 += TX * TN) {
      int mi[TM], nj[TN];
#pragma unroll
      for (int u = 0; u < TM; ++u) mi[u] = min(m0 + ty + TY * u, nb - 1);
#pragma unroll
      for (int v = 0; v < TN; ++v) nj[v] = min(n0 + tx + TX * v, dv - 1);
      float am[TM][TN], as[TM][TN];
#pragma unroll
      for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) am[u][v] = as[u][v] = 0.f;
      for (int j = 0; j < dj; ++j) {
        float a[TM], bm[TN];
#pragma unroll
        for (int u = 0; u < TM; ++u) a[u] = fq(mi[u], j);
#pragma unroll
        for (int v = 0; v < TN; ++v) bm[v] = Ms[nj[v] * DJp + j];
#pragma unroll
        for (int u = 0; u < TM; ++u)
#pragma unroll
          for (int v = 0; v < TN; ++v) am[u][v] = fmaf(a[u], bm[v], am[u][v]);
        if (with_s) {
          float bs[TN];
#pragma unroll
          for (int v = 0; v < TN; ++v) bs[v] = Ss[nj[v] * DJp + j];
#pragma unroll
          for (int u = 0; u < TM; ++u)
#pragma unroll
            for (int v = 0; v < TN; ++v) as[u][v] = fmaf(a[u], bs[v], as[u][v]);
        }
      }
#pragma unroll
      for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) {
          const int n = m0 + ty + TY * u, r = n0 + tx + TX * v;
          if (n < nb && r < dv) YP[n * dv + r] = sa[n] * am[u][v] + sb[n] * as[u][v];
        }
    }
}

// FEAT: 0 the identity map, 1 the degree-2 map, 2 the gated polynomial map.
template <int FEAT>
__global__ void __launch_bounds__(256, 1) linear_wide_kernel(LinArgs p, WideSmem L) {
  extern __shared__ float sm[];
  cg::cluster_group cl = cg::this_cluster();
  const int CL = L.CL;
  const int rank = (int)cl.block_rank();  // cluster (CL, 1, 1) over grid (CL, heads)
  const int head = blockIdx.y;
  float* Ms = sm + L.Ms;
  float* Ss = sm + L.Ss;
  float* Kw = sm + L.Kw;
  float* Qc = sm + L.Qc;
  float* E = sm + L.E;
  float* EP = sm + L.EP;
  float* YP = sm + L.YP;
  float* Wt = sm + L.Wt;
  float* Wrun = sm + L.Wrun;
  float* Urun = sm + L.Urun;
  float* sa = sm + L.sa;
  float* se = sm + L.se;
  float* sb = sm + L.sb;
  float* coef = sm + L.coef;
  uint8_t* pp = reinterpret_cast<uint8_t*>(sm + L.total_floats);
  uint8_t* pq = pp + (L.D - p.d_k > 0 ? L.D - p.d_k : 0);
  uint32_t* ftab = reinterpret_cast<uint32_t*>(sm + L.total_floats);

  const int D = L.D, dk = p.d_k, dv = p.d_v, dkp = L.dkp, DJp = L.DJp, Lmax = L.Lmax;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  const int j0 = rank * L.DJ, dj = max(0, min(L.DJ, D - j0));
  const long state = (long)dv * D;

  if (tid < 5) coef[tid] = p.pcoef[tid];
  if (p.poly && tid == 0) {  // pair table of the degree-2 map
    int o = 0;
    for (int i = 0; i < dk; ++i)
      for (int j = i; j < dk; ++j) { pp[o] = (uint8_t)i; pq[o] = (uint8_t)j; ++o; }
  }
  if (p.pgen && tid == 0) {  // monomial table of the gated map (see the CUDA-core kernel)
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
  auto make = [&](const float* x) {
    if constexpr (FEAT == 0)
      return FeatSlice<FeatId>{FeatId{x, dkp}, j0};
    else if constexpr (FEAT == 1)
      return FeatSlice<FeatP2>{FeatP2{x, dkp, dk, pp, pq}, j0};
    else
      return FeatSlice<Feat>{Feat{x, dkp, dk, p.poly, p.pgen, pp, pq, ftab, coef}, j0};
  };
  const auto fk = make(Kw);
  const auto fq = make(Qc);
  float* Mg = p.M + head * state;
  float* Sg = p.S ? p.S + head * state : nullptr;
  for (long x = tid; x < (long)dv * dj; x += nt) {
    const int r = (int)(x / dj), j = (int)(x % dj);
    Ms[r * DJp + j] = Mg[(long)r * D + j0 + j];
    Ss[r * DJp + j] = Sg ? Sg[(long)r * D + j0 + j] : 0.f;
  }
  const float* alpha = p.alpha + (long)head * p.N;
  const float* eta = p.eta + (long)head * p.N;
  const float* theta = p.theta + (long)head * p.N;
  const long kbase = ((long)head * (p.N + p.nh) + p.nh) * dk;
  const long vbase = ((long)head * (p.N + p.nh) + p.nh) * dv;
  const long qbase = (long)head * p.N * dk;
  float* Yh = p.Y + (long)head * p.N * dv;
  const int cls = dv <= 8 ? 0 : dv <= 16 ? 1 : dv <= 32 ? 2 : dv <= 64 ? 3 : 4;

  for (int t0 = 0; t0 < p.N; t0 += p.b) {
    const int t1 = min(p.N, t0 + p.b);
    const int nb = t1 - t0;
    const int i0 = max(-p.nh, t0 - p.c + 1);
    const int Lw = t1 - i0;
    const int ilo = share_lo(Lw, CL, rank), ihi = share_lo(Lw, CL, rank + 1);
    const int nlo = share_lo(nb, CL, rank), nhi = share_lo(nb, CL, rank + 1);
    __syncthreads();
    for (int x = tid; x < Lw * dk; x += nt)
      Kw[(x / dk) * dkp + x % dk] = ld_in(p.K, kbase + (long)i0 * dk + x, p.bf16);
    for (int x = tid; x < nb * dk; x += nt)
      Qc[(x / dk) * dkp + x % dk] = ld_in(p.Q, qbase + (long)t0 * dk + x, p.bf16);
    chunk_tables(alpha, eta, theta, p.gamma, t0, nb, i0, Lw, p.c, Urun, Wrun, Wt, Lmax, nullptr,
                 sa, se, sb, tid, nt);
    __syncthreads();
    // 1. partial errors over this slice; P for this rank's queries (in place in Wt)
    if (!p.dot) {
      auto fb = [&](int j, int r) { return Ms[r * DJp + j]; };
      auto fe = [&](int i, int r, float acc) { EP[i * dv + r] = acc; };
      switch (cls) {
        case 0: tile_gemm<8, 4, 1>(Lw, dv, dj, fk, fb, fe); break;
        case 1: tile_gemm<16, 4, 1>(Lw, dv, dj, fk, fb, fe); break;
        case 2: tile_gemm<16, 4, 2>(Lw, dv, dj, fk, fb, fe); break;
        case 3: tile_gemm<16, 4, 4>(Lw, dv, dj, fk, fb, fe); break;
        default: tile_gemm<16, 4, 8>(Lw, dv, dj, fk, fb, fe); break;
      }
    }
    for (int x = tid; x < (nhi - nlo) * Lw; x += nt) {
      const int n = nlo + x / Lw, i = x % Lw;
      const float w = Wt[n * Lmax + i];
      float v = 0.f;
      if (w != 0.f) {  // Phi(q).Phi(k) from the power sums of q_j k_j
        const float* q = Qc + n * dkp;
        const float* k = Kw + i * dkp;
        float pw[4] = {0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < dk; ++j) {
          const float z = q[j] * k[j];
          pw[0] += z;
          pw[1] += z * z;
          if (p.pgen) {
            pw[2] += z * z * z;
            pw[3] += z * z * z * z;
          }
        }
        if (p.pgen) {
          float h[5];
          h[0] = 1.f;
          v = coef[0] * coef[0];
#pragma unroll
          for (int m = 1; m <= 4; ++m) {
            float acc = 0.f;
#pragma unroll
            for (int l = 1; l <= m; ++l) acc += pw[l - 1] * h[m - l];
            h[m] = acc / (float)m;
            if (m <= p.pdeg) v += coef[m] * coef[m] * h[m];
          }
        } else {
          v = p.poly ? pw[0] + 0.5f * (pw[0] * pw[0] + pw[1]) : pw[0];
        }
        v *= w;
      }
      Wt[n * Lmax + i] = v;
    }
    cl.sync();  // A: every rank's partial errors are in place
    // 2. this rank's window rows: the errors summed over the ranks, then the bias
    for (int i = ilo + warp; i < ihi; i += nw) {
      float ev[4];  // d_v <= 128: lane l holds r = l + 32 u
      float ss = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = lane + 32 * u;
        ev[u] = 0.f;
        if (r >= dv) continue;
        float s = 0.f;
        if (!p.dot)
          for (int c = 0; c < CL; ++c) s += *cl.map_shared_rank(EP + i * dv + r, c);
        const float v = ld_in(p.V, vbase + (long)(i0 + i) * dv + r, p.bf16);
        ev[u] = p.dot ? -v : s - v;
        ss += ev[u] * ev[u];
      }
      const float f = p.lk == ATLAS_LOSS_ROBUST ? robust_scale(sqrtf(warp_sum(ss)), p.lp) : 1.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = lane + 32 * u;
        if (r < dv) E[i * dv + r] = p.dot ? ev[u] : bias_grad(ev[u], p.lk, p.lp) * f;
      }
    }
    cl.sync();  // B: every rank's finished error rows are in place
    // 3. the other ranks' error rows
    for (int c = 0; c < CL; ++c) {
      if (c == rank) continue;
      const int lo = share_lo(Lw, CL, c), hi = share_lo(Lw, CL, c + 1);
      const float* src = cl.map_shared_rank(E, c);
      for (int x = lo * dv + tid; x < hi * dv; x += nt) E[x] = src[x];
    }
    __syncthreads();
    // 4. partial readout of the slice; this rank's queries add the intra-chunk term
    {
      bool with_s = false;
      for (int n = 0; n < nb; ++n) with_s |= sb[n] != 0.f;
      switch (cls) {
        case 0: readout_partial<8, 4, 1>(nb, dv, dj, fq, Ms, Ss, DJp, sa, sb, with_s, YP); break;
        case 1: readout_partial<16, 4, 1>(nb, dv, dj, fq, Ms, Ss, DJp, sa, sb, with_s, YP); break;
        case 2: readout_partial<16, 4, 2>(nb, dv, dj, fq, Ms, Ss, DJp, sa, sb, with_s, YP); break;
        case 3: readout_partial<16, 4, 4>(nb, dv, dj, fq, Ms, Ss, DJp, sa, sb, with_s, YP); break;
        default: readout_partial<16, 4, 8>(nb, dv, dj, fq, Ms, Ss, DJp, sa, sb, with_s, YP); break;
      }
    }
    __syncthreads();
    {
      auto fa = [&](int n, int i) { return Wt[(nlo + n) * Lmax + i]; };
      auto fb = [&](int i, int r) { return E[i * dv + r]; };
      auto fe = [&](int n, int r, float acc) { YP[(nlo + n) * dv + r] -= 2.f * acc; };
      switch (cls) {
        case 0: tile_gemm<8, 4, 1>(nhi - nlo, dv, Lw, fa, fb, fe); break;
        case 1: tile_gemm<16, 4, 1>(nhi - nlo, dv, Lw, fa, fb, fe); break;
        case 2: tile_gemm<16, 4, 2>(nhi - nlo, dv, Lw, fa, fb, fe); break;
        case 3: tile_gemm<16, 4, 4>(nhi - nlo, dv, Lw, fa, fb, fe); break;
        default: tile_gemm<16, 4, 8>(nhi - nlo, dv, Lw, fa, fb, fe); break;
      }
    }
    cl.sync();  // D: every rank's partial readout is in place
    // 5. this rank's queries: the readout summed over the ranks
    for (int x = nlo * dv + tid; x < nhi * dv; x += nt) {
      float y = 0.f;
      for (int c = 0; c < CL; ++c) y += *cl.map_shared_rank(YP + x, c);
      Yh[(long)t0 * dv + x] = y;
    }
    // 6. carry this rank's columns of M and S to the chunk end
    {
      const float a_b = sa[nb - 1], e_b = se[nb - 1], b_b = sb[nb - 1];
      switch (cls) {
        case 0: carry_tile<32, 1, 5>(dv, dj, Lw, fk, E, Wrun, Urun, Ms, Ss, DJp, a_b, b_b, e_b); break;
        case 1: carry_tile<16, 1, 9>(dv, dj, Lw, fk, E, Wrun, Urun, Ms, Ss, DJp, a_b, b_b, e_b); break;
        case 2: carry_tile<16, 2, 9>(dv, dj, Lw, fk, E, Wrun, Urun, Ms, Ss, DJp, a_b, b_b, e_b); break;
        case 3: carry_tile<16, 4, 9>(dv, dj, Lw, fk, E, Wrun, Urun, Ms, Ss, DJp, a_b, b_b, e_b); break;
        default: carry_tile<16, 8, 5>(dv, dj, Lw, fk, E, Wrun, Urun, Ms, Ss, DJp, a_b, b_b, e_b); break;
      }
    }
  }
  __syncthreads();
  for (long x = tid; x < (long)dv * dj; x += nt) {
    const int r = (int)(x / dj), j = (int)(x % dj);
    Mg[(long)r * D + j0 + j] = Ms[r * DJp + j];
    if (Sg) Sg[(long)r * D + j0 + j] = Ss[r * DJp + j];
  }
  cl.sync();  // no rank leaves while another may still read its shared memory
}

// Cluster size: the smallest of 2, 4, 8 whose slice fits, doubled while the
// clusters of all heads still fit the 152 SMs at one CTA each.
static int wide_plan(const LinArgs& a, int heads, WideSmem* out) {
  int CL = 0;
  for (int c = 2; c <= 8; c *= 2)
    if (wide_layout(a, c).bytes() <= kWideSmemLimit) {
      CL = c;
      break;
    }
  if (!CL) return ATLAS_ERR_UNSUPPORTED;
  while (CL < 8 && (long)heads * 2 * CL <= 152) CL *= 2;
  *out = wide_layout(a, CL);
  return ATLAS_OK;
}

bool linear_wide_supported(const LinArgs& a, int heads) {
  if (a.D < 256 || a.d_v > 128 || a.ret != ATLAS_RET_L2 || heads <= 0 || heads > 65535)
    return false;
  WideSmem s;
  return wide_plan(a, heads, &s) == ATLAS_OK;
}

int linear_wide_launch(const LinArgs& a, int heads, cudaStream_t st) {
  if (!linear_wide_supported(a, heads)) return ATLAS_ERR_UNSUPPORTED;
  if (a.N == 0) return ATLAS_OK;
  WideSmem s;
  wide_plan(a, heads, &s);
  const size_t smem = s.bytes();
  const int feat = a.pgen ? 2 : a.poly ? 1 : 0;
  auto kern = feat == 2 ? linear_wide_kernel<2> : feat == 1 ? linear_wide_kernel<1>
                                                            : linear_wide_kernel<0>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return ATLAS_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.CL, heads);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = s.CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, a, s) != cudaSuccess) return ATLAS_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ATLAS_OK : ATLAS_ERR_CUDA;
}

}  // namespace atlas
