// linear_seq.cu -- latency path of the update of a small linear memory
// (identity feature map, D = d_k = 32, window c <= 8, any chunk length b):
// token after token, with every state element in a register.
//
// The rows of M never mix: row r's window errors e_j[r] need only row r of the
// chunk-start state, and its gradient, momentum, decay and readout stay in row
// r.  So eight lanes own one row (four columns each), a warp owns four rows, a
// CTA of four warps sixteen rows, and the grid covers (rows / 16) x heads.
// Per token t ("논문 리뷰 Google ATLAS" §3.2 Omega rule and §3.3 chunk-start
// weights; "[Paper Review] Titans 논문 이해하기" momentum, forgetting and
// retrieval):
//   e_j[r] = M0[r,:] . k_{t-j} - v_{t-j}[r]  (dot loss: -v_{t-j}[r])   j < c
//   S[r,:] = eta_t S[r,:] - 2 theta_t sum_j gamma_j e_j[r] k_{t-j}
//   M[r,:] = (1 - alpha_t) M[r,:] + S[r,:],      y_t[r] = M[r,:] . q_t
// where M0 is the state at the start of t's chunk (M itself when b = 1) and
// window tokens before the history rows (token -n_history) are absent.  The window's row dot products are a
// four-term in-register sum plus three shuffle levels; the readout's eight
// per-lane shares go to shared memory and are summed once per tile, off the
// token-to-token dependency chain.  K, Q, the CTA's V rows and the
// gates move through shared memory in tiles of kT tokens; the next tile is
// loaded into registers while the current one is processed, and the last c-1
// rows of a tile stay on as the window history of the next.
#include "common.cuh"
#include "kernels.h"

namespace atlas {

namespace {
constexpr int kT = 64;           // tokens per tile
constexpr int kRows = 16;        // rows of M per CTA
constexpr int kThr = 128;        // 4 warps x 4 rows x 8 lanes
constexpr int kMaxC = 8;
constexpr int kKPer = kT * 32 / kThr;     // K (and Q) elements per thread per tile
constexpr int kVPer = kT * kRows / kThr;  // V elements per thread per tile
constexpr int kGPer = (3 * kT + kThr - 1) / kThr;

struct SeqSmem {
  float K[kMaxC - 1 + kT][32];
  float V[kMaxC - 1 + kT][kRows];
  float Q[kT][32];
  float G[3][kT];  // alpha, eta, theta
  float Yp[kT][kRows][8];  // per-lane shares of y
};

__device__ __forceinline__ float row_sum8(float x) {
  x += __shfl_xor_sync(0xFFFFFFFFu, x, 1);
  x += __shfl_xor_sync(0xFFFFFFFFu, x, 2);
  x += __shfl_xor_sync(0xFFFFFFFFu, x, 4);
  return x;
}
}  // namespace

// Shared-memory operands of one token for one lane.
template <int C>
struct TokOps {
  float4 k[C];   // window keys k_{t-j}, this lane's four columns
  float v[C];    // window values v_{t-j}[r]
  float4 q;
  float keep, eta, th2;
};

template <int C>
__device__ __forceinline__ void load_tok(const SeqSmem& sm, int u, int rl, int cg, TokOps<C>& o) {
#pragma unroll
  for (int j = 0; j < C; ++j) {
    o.k[j] = *reinterpret_cast<const float4*>(&sm.K[C - 1 + u - j][4 * cg]);
    o.v[j] = sm.V[C - 1 + u - j][rl];
  }
  o.q = *reinterpret_cast<const float4*>(&sm.Q[u][4 * cg]);
  o.keep = 1.f - sm.G[0][u];
  o.eta = sm.G[1][u];
  o.th2 = 2.f * sm.G[2][u];
}

template <int C>
__global__ void __launch_bounds__(kThr) linear_seq_kernel(LinArgs p) {
  extern __shared__ __align__(16) unsigned char seq_smem_raw[];
  SeqSmem& sm = *reinterpret_cast<SeqSmem*>(seq_smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int head = blockIdx.y, r0 = blockIdx.x * kRows;
  const int rl = warp * 4 + (lane >> 3);  // row inside the CTA
  const int r = r0 + rl, cg = lane & 7;   // columns 4cg .. 4cg+3
  const int dv = p.d_v, N = p.N;
  const bool row_ok = r < dv;
  // K, V: head stride (nh + N) rows with token 0 at row nh; Q, Y, gates: N rows
  const int nh = p.nh;
  const long kb = ((long)head * (N + nh) + nh) * 32, vb = ((long)head * (N + nh) + nh) * dv;
  const long qb = (long)head * N * 32, yb = (long)head * N * dv, gb = (long)head * N;
  float* Mrow = p.M + ((long)head * dv + r) * 32 + 4 * cg;
  float* Srow = p.S ? p.S + ((long)head * dv + r) * 32 + 4 * cg : nullptr;
  // the dot loss has no state term in its error: fold that into the copy of M0
  const float ldot = p.dot ? 0.f : 1.f;

  float m[4], s[4], m0[4], gam[C];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    m[x] = row_ok ? Mrow[x] : 0.f;
    s[x] = (row_ok && Srow) ? Srow[x] : 0.f;
    m0[x] = ldot * m[x];
  }
#pragma unroll
  for (int j = 0; j < C; ++j) gam[j] = p.gamma[j];

  // tile loader: registers <- tokens [t0, t0 + kT) (zero past N)
  float pk[kKPer], pq[kKPer], pv[kVPer], pg[kGPer];
  auto fetch = [&](int t0) {
#pragma unroll
    for (int x = 0; x < kKPer; ++x) {
      const int e = x * kThr + tid, t = t0 + e / 32;
      pk[x] = t < N ? ld_in(p.K, kb + (long)t * 32 + (e & 31), p.bf16) : 0.f;
      pq[x] = t < N ? ld_in(p.Q, qb + (long)t * 32 + (e & 31), p.bf16) : 0.f;
    }
#pragma unroll
    for (int x = 0; x < kVPer; ++x) {
      const int e = x * kThr + tid, t = t0 + e / kRows, rr = r0 + e % kRows;
      pv[x] = (t < N && rr < dv) ? ld_in(p.V, vb + (long)t * dv + rr, p.bf16) : 0.f;
    }
#pragma unroll
    for (int x = 0; x < kGPer; ++x) {
      const int e = x * kThr + tid, which = e / kT, t = t0 + e % kT;
      pg[x] = 0.f;
      if (which < 3 && t < N) pg[x] = (which == 0 ? p.alpha : which == 1 ? p.eta : p.theta)[gb + t];
    }
  };
  auto deposit = [&]() {
#pragma unroll
    for (int x = 0; x < kKPer; ++x) {
      const int e = x * kThr + tid;
      sm.K[C - 1 + e / 32][e & 31] = pk[x];
      sm.Q[e / 32][e & 31] = pq[x];
    }
#pragma unroll
    for (int x = 0; x < kVPer; ++x) {
      const int e = x * kThr + tid;
      sm.V[C - 1 + e / kRows][e % kRows] = pv[x];
    }
#pragma unroll
    for (int x = 0; x < kGPer; ++x) {
      const int e = x * kThr + tid;
      if (e < 3 * kT) sm.G[e / kT][e % kT] = pg[x];
    }
  };

  // window history of the first tile: the history rows, absent before -nh
  for (int e = tid; e < (C - 1) * 32; e += kThr) {
    const int t = e / 32 - (C - 1);
    sm.K[e / 32][e & 31] = t >= -nh ? ld_in(p.K, kb + (long)t * 32 + (e & 31), p.bf16) : 0.f;
  }
  for (int e = tid; e < (C - 1) * kRows; e += kThr) {
    const int t = e / kRows - (C - 1), rr = r0 + e % kRows;
    sm.V[e / kRows][e % kRows] =
        (t >= -nh && rr < dv) ? ld_in(p.V, vb + (long)t * dv + rr, p.bf16) : 0.f;
  }
  fetch(0);
  deposit();
  __syncthreads();

  int pos = 0;  // position of the token inside its chunk
  for (int t0 = 0; t0 < N; t0 += kT) {
    const int ntok = min(kT, N - t0);
    if (t0 + kT < N) fetch(t0 + kT);  // lands while this tile is processed
    TokOps<C> cur, nxt;
    load_tok<C>(sm, 0, rl, cg, cur);
    for (int u = 0; u < ntok; ++u) {
      load_tok<C>(sm, u + 1 < kT ? u + 1 : u, rl, cg, nxt);  // operands of the next token
      const bool start = pos == 0;
      pos = pos + 1 == p.b ? 0 : pos + 1;
#pragma unroll
      for (int x = 0; x < 4; ++x) m0[x] = start ? ldot * m[x] : m0[x];
      float e[C];
#pragma unroll
      for (int j = 0; j < C; ++j)
        e[j] = row_sum8(m0[0] * cur.k[j].x + m0[1] * cur.k[j].y + m0[2] * cur.k[j].z +
                        m0[3] * cur.k[j].w);
      float g[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < C; ++j) {
        const float w = gam[j] * bias_grad(e[j] - cur.v[j], p.lk, p.lp);
        g[0] += w * cur.k[j].x;
        g[1] += w * cur.k[j].y;
        g[2] += w * cur.k[j].z;
        g[3] += w * cur.k[j].w;
      }
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        s[x] = cur.eta * s[x] - cur.th2 * g[x];
        m[x] = cur.keep * m[x] + s[x];
      }
      // this lane's share of y_t[r]; the eight shares are summed after the tile
      sm.Yp[u][rl][cg] = m[0] * cur.q.x + m[1] * cur.q.y + m[2] * cur.q.z + m[3] * cur.q.w;
      cur = nxt;
    }
    // history for the next tile, readout of this one
    float hk[((kMaxC - 1) * 32 + kThr - 1) / kThr], hv[((kMaxC - 1) * kRows + kThr - 1) / kThr];
    __syncthreads();
#pragma unroll
    for (int x = 0; x < (int)(sizeof(hk) / sizeof(float)); ++x) {
      const int e = x * kThr + tid;
      if (e < (C - 1) * 32) hk[x] = sm.K[kT + e / 32][e & 31];
    }
#pragma unroll
    for (int x = 0; x < (int)(sizeof(hv) / sizeof(float)); ++x) {
      const int e = x * kThr + tid;
      if (e < (C - 1) * kRows) hv[x] = sm.V[kT + e / kRows][e % kRows];
    }
    for (int e = tid; e < ntok * kRows; e += kThr) {
      const int u = e / kRows, rr = e % kRows;
      if (r0 + rr < dv) {
        const float4 a = *reinterpret_cast<const float4*>(&sm.Yp[u][rr][0]);
        const float4 b = *reinterpret_cast<const float4*>(&sm.Yp[u][rr][4]);
        p.Y[yb + (long)(t0 + u) * dv + r0 + rr] = ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w));
      }
    }
    __syncthreads();
    if (t0 + kT < N) {
#pragma unroll
      for (int x = 0; x < (int)(sizeof(hk) / sizeof(float)); ++x) {
        const int e = x * kThr + tid;
        if (e < (C - 1) * 32) sm.K[e / 32][e & 31] = hk[x];
      }
#pragma unroll
      for (int x = 0; x < (int)(sizeof(hv) / sizeof(float)); ++x) {
        const int e = x * kThr + tid;
        if (e < (C - 1) * kRows) sm.V[e / kRows][e % kRows] = hv[x];
      }
      deposit();
    }
    __syncthreads();
  }
  if (row_ok) {
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      Mrow[x] = m[x];
      if (Srow) Srow[x] = s[x];
    }
  }
}

bool linear_seq_supported(const LinArgs& a) {
  return !a.poly && !a.pgen && a.ret == ATLAS_RET_L2 && a.lk != ATLAS_LOSS_ROBUST &&
         a.d_k == 32 && a.D == 32 && a.d_v >= 1 && a.c >= 1 && a.c <= kMaxC;
}

int linear_seq_launch(const LinArgs& a, int heads, cudaStream_t st) {
  if (!linear_seq_supported(a)) return ATLAS_ERR_UNSUPPORTED;
  if (heads <= 0) return ATLAS_OK;
  const dim3 grid((a.d_v + kRows - 1) / kRows, heads);
  const int smem = (int)sizeof(SeqSmem);
  static bool attr_set[kMaxC + 1] = {};
  if (!attr_set[a.c]) {
    cudaError_t e = cudaSuccess;
    switch (a.c) {
      case 1: e = cudaFuncSetAttribute(linear_seq_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); break;
      case 2: e = cudaFuncSetAttribute(linear_seq_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); break;
      case 3: e = cudaFuncSetAttribute(linear_seq_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); break;
      case 4: e = cudaFuncSetAttribute(linear_seq_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); break;
      case 5: e = cudaFuncSetAttribute(linear_seq_kernel<5>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); break;
      case 6: e = cudaFuncSetAttribute(linear_seq_kernel<6>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); break;
      case 7: e = cudaFuncSetAttribute(linear_seq_kernel<7>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); break;
      default: e = cudaFuncSetAttribute(linear_seq_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); break;
    }
    if (e != cudaSuccess) return ATLAS_ERR_CUDA;
    attr_set[a.c] = true;
  }
  switch (a.c) {
    case 1: linear_seq_kernel<1><<<grid, kThr, smem, st>>>(a); break;
    case 2: linear_seq_kernel<2><<<grid, kThr, smem, st>>>(a); break;
    case 3: linear_seq_kernel<3><<<grid, kThr, smem, st>>>(a); break;
    case 4: linear_seq_kernel<4><<<grid, kThr, smem, st>>>(a); break;
    case 5: linear_seq_kernel<5><<<grid, kThr, smem, st>>>(a); break;
    case 6: linear_seq_kernel<6><<<grid, kThr, smem, st>>>(a); break;
    case 7: linear_seq_kernel<7><<<grid, kThr, smem, st>>>(a); break;
    default: linear_seq_kernel<8><<<grid, kThr, smem, st>>>(a); break;
  }
  return cudaGetLastError() == cudaSuccess ? ATLAS_OK : ATLAS_ERR_CUDA;
}

}  // namespace atlas
