// linear_tc.cu -- tensor-core (tcgen05 + TMEM + TMA) path of the chunked
// update of a linear memory: identity feature map, d_k = d_v = 128, chunk
// b = 64, window c = 1, bf16 K/Q/V, fp32 state, no momentum (eta = 0).
//
// One persistent CTA per head walks the chunks in order ("논문 리뷰 Google
// ATLAS" §3.3: every gradient of a chunk at the chunk-start state).  With
// c = 1 and eta = 0 the chunk of tokens n = 0..63 starting in state M0 is
//   E      = Phi M0^T - V                         (64 x 128, the errors)
//   y_n    = a_n (M0 q_n) - 2 sum_{i<=n} W[n,i] (q_n . k_i) e_i
//   M_end  = a_63 M0 - 2 sum_i W[63,i] e_i k_i^T
// with a_n = prod_{l<=n} (1 - alpha_l) and W[n,i] = gamma_0 theta_i
// prod_{l=i+1..n} (1 - alpha_l) ("[Paper Review] Titans 논문 이해하기":
// S_t = -theta_t grad, M_t = (1 - alpha_t) M_{t-1} + S_t, y_t = M_t q_t).
//
// Four tensor-core products per chunk (M = 128 rows, fp32 accumulators in TMEM):
//   D_QP = [Phi; Q] Phi^T          (rows 64..127: q_n . k_i)
//   D1   = [Phi; Q] M0^T           (rows 0..63: Phi M0^T; rows 64..127: Q M0^T)
//   dM   = Ew^T Phi                (Ew = W[63,:] * E, the rank-64 state update)
//   D1  += [* ; P'] E              (P' = -2 W * (Q Phi^T), added onto the rows
//                                   64..127 of D1 once they are scaled by a_n:
//                                   they become y_n)
// K, Q, V are bf16 and exact; the state-derived operands (M0, E, Ew, P) are
// split into bf16 hi + lo parts (x = hi + lo to ~2^-17), so every product keeps
// fp32-level accuracy.  The fp32 master state M lives in the registers of the
// eight epilogue warps (thread = row of M, 64 columns each).
//
// Warp roles (320 threads): warp 0 issues TMA loads of chunk j+1 while chunk j
// runs (two stages); warp 1 builds the per-chunk gate tables and issues the
// MMAs from one thread; warps 2..9 are the epilogue (TMEM -> registers ->
// shared memory / global), two warps per 32-lane TMEM quadrant.
//
// Heads whose eta has any non-zero entry are left to the CUDA-core kernel,
// which is launched right after this one and takes exactly those heads (both
// kernels read eta and decide the same way).  Every wait on an mbarrier is
// bounded; on expiry the kernel records ATLAS_ERR_TIMEOUT in the status word,
// drains its in-flight copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_primitives.cuh"

namespace atlas {
using namespace tc;

namespace {

constexpr int kThreads = 320;
constexpr int kChunk = 64;
constexpr int kDim = 128;
constexpr long long kWaitLimit = 2000000000LL;  // clock cycles (~1 s)

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t STAGE_BYTES = 33792;  // Phi/Q (4 x 8 KB) + gates (3 x 256 B), padded
constexpr uint32_t OFF_STAGE0 = 0;
constexpr uint32_t OFF_MHI = 2 * STAGE_BYTES;       // 67584
constexpr uint32_t OFF_MLO = OFF_MHI + 32768;
constexpr uint32_t OFF_EHI = OFF_MLO + 32768;
constexpr uint32_t OFF_ELO = OFF_EHI + 16384;
constexpr uint32_t OFF_EWHI = OFF_ELO + 16384;
constexpr uint32_t OFF_EWLO = OFF_EWHI + 16384;
constexpr uint32_t OFF_PHI = OFF_EWLO + 16384;      // preceded by 8 KB of EWLO (A-tile rows 0..63)
constexpr uint32_t OFF_PLO = OFF_PHI + 8192;
constexpr uint32_t OFF_TAB = OFF_PLO + 8192;
constexpr uint32_t TAB_FLOATS = 5 * kChunk;          // a, pb, wb, keep, th
constexpr uint32_t OFF_ELAST = OFF_TAB + 2 * TAB_FLOATS * 4;
constexpr uint32_t OFF_BARS = OFF_ELAST + kDim * 4;
constexpr uint32_t SMEM_USED = OFF_BARS + 256;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;   // alignment slack

constexpr uint32_t STAGE_TX = 4 * 8192 + 3 * 256;

// TMEM columns: D1 is double-buffered so that the readout of chunk j can
// leave TMEM while chunk j+1's products already run.
constexpr uint32_t TM_QP = 0, TM_D1 = 64, TM_DM = 320, TM_COLS = 512;
__device__ __forceinline__ uint32_t tm_d1(int j) { return TM_D1 + 128u * (uint32_t)(j & 1); }

enum Bar {
  B_FULL0 = 0, B_FULL1, B_EMPTY0, B_EMPTY1, B_QP, B_D1, B_DM, B_Y, B_E, B_P, B_M, B_TAB0, B_TAB1,
  B_S, B_DRAIN, B_COUNT
};

struct TcParams {
  const __nv_bfloat16* K;
  const __nv_bfloat16* V;
  const float* eta;
  const float* theta;
  const float* gamma;
  float* Y;
  float* M;
  float* S;  // optional
  int* status;
  int N;
};

struct TcMaps {
  CUtensorMap k, q, alpha, eta, theta;
};

__device__ __forceinline__ void table_ptrs(unsigned char* sm, int buf, float*& a, float*& pb,
                                           float*& wb, float*& keep, float*& th) {
  float* t = reinterpret_cast<float*>(sm + OFF_TAB) + buf * TAB_FLOATS;
  a = t;
  pb = t + kChunk;
  wb = t + 2 * kChunk;
  keep = t + 3 * kChunk;
  th = t + 4 * kChunk;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    linear_tc_kernel(const __grid_constant__ TcMaps maps, TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BARS + B_COUNT * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_BARS + B_COUNT * 8 + 8);

  const int head = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.N;
  const int nchunks = (N + kChunk - 1) / kChunk;

  // ---- heads with momentum belong to the CUDA-core kernel
  {
    const float4* e4 = reinterpret_cast<const float4*>(p.eta + (long)head * N);
    int nz = 0;
    for (int x = tid; x < N / 4; x += kThreads) {
      const float4 v = e4[x];
      nz |= (v.x != 0.f) | (v.y != 0.f) | (v.z != 0.f) | (v.w != 0.f);
    }
    if (__syncthreads_or(nz)) return;
  }
  if (nchunks == 0) return;

  if (tid == 0) {
    for (int b = 0; b < B_COUNT; ++b) {
      uint32_t cnt = 1;
      if (b == B_E || b == B_P) cnt = 4;
      if (b == B_M || b == B_S) cnt = 8;
      mbar_init(&bars[b], cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&maps.k);
    prefetch_tmap(&maps.q);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_u32(sm);

  auto fail = [&]() {
    *abort_flag = 1;
    if (p.status) atomicExch(p.status, ATLAS_ERR_TIMEOUT);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < nchunks; ++j) {
        const int s = j & 1;
        if (j >= 2 && !mbar_wait(&bars[B_EMPTY0 + s], ((j - 2) >> 1) & 1, abort_flag, kWaitLimit)) {
          fail();
          break;
        }
        unsigned char* st = sm + OFF_STAGE0 + s * STAGE_BYTES;
        uint64_t* fb = &bars[B_FULL0 + s];
        mbar_arrive_expect_tx(fb, STAGE_TX);
        const int t0 = j * kChunk;
        tma_load_3d(st + 0, &maps.k, fb, 0, t0, head);
        tma_load_3d(st + 8192, &maps.q, fb, 0, t0, head);
        tma_load_3d(st + 16384, &maps.k, fb, 64, t0, head);
        tma_load_3d(st + 24576, &maps.q, fb, 64, t0, head);
        tma_load_2d(st + 32768, &maps.alpha, fb, t0, head);
        tma_load_2d(st + 32768 + 256, &maps.eta, fb, t0, head);
        tma_load_2d(st + 32768 + 512, &maps.theta, fb, t0, head);
        issued = j + 1;
      }
      // drain: every issued load must land before shared memory is released
      for (int j = issued - 2 < 0 ? 0 : issued - 2; j < issued; ++j) {
        volatile int zero = 0;
        mbar_wait(&bars[B_FULL0 + (j & 1)], (j >> 1) & 1, &zero, kWaitLimit);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------- tables + MMA issuer
    const float g0 = p.gamma[0];
    auto tables = [&](int j) -> bool {
      const int s = j & 1;
      if (!mbar_wait(&bars[B_FULL0 + s], (j >> 1) & 1, abort_flag, kWaitLimit)) return false;
      if (lane == 0) {
        const float* ga = reinterpret_cast<const float*>(sm + OFF_STAGE0 + s * STAGE_BYTES + 32768);
        const float* gt = ga + 128;
        float *a, *pb, *wb, *keep, *th;
        table_ptrs(sm, s, a, pb, wb, keep, th);
        float pa = 1.f, pbv = 1.f;
        for (int n = 0; n < kChunk; ++n) {
          const float k = 1.f - ga[n];
          keep[n] = k;
          th[n] = gt[n] * g0;
          pa *= k;
          a[n] = pa;
          if (n >= 32) pbv *= k;
          pb[n] = n >= 32 ? pbv : 1.f;
        }
        float suf = 1.f;  // prod_{l=i+1..63} keep_l
        for (int i = kChunk - 1; i >= 0; --i) {
          wb[i] = th[i] * suf;
          suf *= keep[i];
        }
        mbar_arrive(&bars[B_TAB0 + s]);
      }
      __syncwarp();
      return true;
    };
    bool ok = tables(0);
    if (!ok) fail();
    for (int j = 0; ok && j < nchunks; ++j) {
      const int s = j & 1;
      const uint32_t st = sbase + OFF_STAGE0 + s * STAGE_BYTES;
      // stage j is loaded (waited in tables(j))
      tc_fence_after();
      if (lane == 0) {
        const uint32_t id = idesc_bf16(128, 64, false, false);
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          mma_bf16(tmem + TM_QP, sdesc_sw128(st + off, 16, 1024), sdesc_sw128(st + off, 16, 1024),
                   id, k > 0);
        }
        mma_commit(&bars[B_QP]);
      }
      __syncwarp();
      if (!mbar_wait(&bars[B_M], j & 1, abort_flag, kWaitLimit)) { ok = false; break; }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t id = idesc_bf16(128, 128, false, false);
        for (int k = 0; k < 16; ++k) {
          const uint32_t off = ((k & 7) >> 2) * 16384 + (k & 3) * 32;
          const uint32_t mb = sbase + (k < 8 ? OFF_MHI : OFF_MLO);
          mma_bf16(tmem + tm_d1(j), sdesc_sw128(st + off, 16, 1024),
                   sdesc_sw128(mb + off, 16, 1024), id, k > 0);
        }
        mma_commit(&bars[B_D1]);
      }
      __syncwarp();
      if (!mbar_wait(&bars[B_E], j & 1, abort_flag, kWaitLimit)) { ok = false; break; }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t id = idesc_bf16(128, 128, true, true);
        for (int k = 0; k < 8; ++k) {
          const uint32_t ew = sbase + ((k < 4) ? OFF_EWHI : OFF_EWLO) + (k & 3) * 2048;
          mma_bf16(tmem + TM_DM, sdesc_sw128(ew, 8192, 1024),
                   sdesc_sw128(st + (k & 3) * 2048, 16384, 1024), id, k > 0);
        }
        mma_commit(&bars[B_DM]);
      }
      __syncwarp();
      if (!mbar_wait(&bars[B_P], j & 1, abort_flag, kWaitLimit)) { ok = false; break; }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t id = idesc_bf16(128, 128, false, true);
        for (int k = 0; k < 12; ++k) {
          const int part = k >> 2;  // 0: Phi*Ehi, 1: Phi*Elo, 2: Plo*Ehi
          const uint32_t pa = sbase + (part < 2 ? OFF_PHI : OFF_PLO) - 8192 + (k & 3) * 32;
          const uint32_t eb = sbase + (part == 1 ? OFF_ELO : OFF_EHI) + (k & 3) * 2048;
          mma_bf16(tmem + tm_d1(j), sdesc_sw128(pa, 16, 1024), sdesc_sw128(eb, 8192, 1024), id, 1);
        }
        mma_commit(&bars[B_Y]);
        mma_commit(&bars[B_EMPTY0 + s]);
      }
      __syncwarp();
      if (j + 1 < nchunks && !tables(j + 1)) { ok = false; break; }
    }
    if (!ok) fail();
    if (lane == 0) {
      // no MMA may outlive the TMEM: wait for everything this thread issued
      volatile int zero = 0;
      mma_commit(&bars[B_DRAIN]);
      mbar_wait(&bars[B_DRAIN], 0, &zero, kWaitLimit);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;             // TMEM lane quadrant
    const int h = (warp - 2) >> 2;      // column half
    const int r = 32 * q + lane;        // TMEM lane = row of the 128-row tiles
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
    const bool low = q < 2;
    float m[64];
    {
      const float4* src = reinterpret_cast<const float4*>(p.M + ((long)head * kDim + r) * kDim + 64 * h);
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const float4 v = src[x];
        m[4 * x] = v.x; m[4 * x + 1] = v.y; m[4 * x + 2] = v.z; m[4 * x + 3] = v.w;
      }
      const uint32_t mh = sbase + OFF_MHI + h * 16384, ml = sbase + OFF_MLO + h * 16384;
#pragma unroll
      for (int c = 0; c < 8; ++c) store_split8(mh + sw128_offset(r, c), ml + sw128_offset(r, c), m + 8 * c);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_M]);
    }
    const __nv_bfloat16* Vh = p.V + (long)head * N * kDim;
    float* Yh = p.Y + (long)head * N * kDim;
    bool ok = true;
    for (int j = 0; j < nchunks; ++j) {
      const int s = j & 1, t0 = j * kChunk;
      const uint32_t par = j & 1;
      if (!mbar_wait(&bars[B_TAB0 + s], (j >> 1) & 1, abort_flag, kWaitLimit)) { ok = false; break; }
      float *ta, *tpb, *twb, *tkeep, *tth;
      table_ptrs(sm, s, ta, tpb, twb, tkeep, tth);
      if (low) {
        // ---- errors E = Phi M0^T - V of token i = r
        const int i = r;
        uint32_t vv[32];  // 64 bf16 values of v_i, packed in pairs
        const bool valid = t0 + i < N;
        const uint4* vsrc = reinterpret_cast<const uint4*>(Vh + (long)(t0 + i) * kDim + 64 * h);
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const uint4 v = valid ? vsrc[x] : make_uint4(0, 0, 0, 0);
          vv[4 * x] = v.x; vv[4 * x + 1] = v.y; vv[4 * x + 2] = v.z; vv[4 * x + 3] = v.w;
        }
        if (!mbar_wait(&bars[B_D1], par, abort_flag, kWaitLimit)) { ok = false; break; }
        tc_fence_after();
        const float w_i = twb[i];
        const bool last_tok = p.S && j == nchunks - 1 && t0 + i == N - 1;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float d[32];
          tmem_ld32(tl + tm_d1(j) + 64 * h + 32 * cc, d);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float e[8], ew[8];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const uint32_t pk = vv[16 * cc + 4 * c + x];
              e[2 * x] = d[8 * c + 2 * x] - __uint_as_float(pk << 16);
              e[2 * x + 1] = d[8 * c + 2 * x + 1] - __uint_as_float(pk & 0xFFFF0000u);
            }
#pragma unroll
            for (int x = 0; x < 8; ++x) ew[x] = w_i * e[x];
            const uint32_t o = h * 8192 + sw128_offset(i, 4 * cc + c);
            store_split8(sbase + OFF_EHI + o, sbase + OFF_ELO + o, e);
            store_split8(sbase + OFF_EWHI + o, sbase + OFF_EWLO + o, ew);
            if (last_tok) {
              float* el = reinterpret_cast<float*>(sm + OFF_ELAST) + 64 * h + 32 * cc + 8 * c;
#pragma unroll
              for (int x = 0; x < 8; ++x) el[x] = e[x];
            }
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_E]);
      } else {
        // ---- P = W * (Q Phi^T) of query n = r - 64, keys i in [32h, 32h+32)
        const int n = r - 64;
        if (!mbar_wait(&bars[B_QP], par, abort_flag, kWaitLimit)) { ok = false; break; }
        tc_fence_after();
        float pv[32];  // q_n . k_i, then P[n,i]
        tmem_ld32(tl + TM_QP + 32 * h, pv);
        // W[n,i] = th_i prod_{l=i+1..n} keep_l, walked from i = 32h+31 down to 32h
        float da = (h == 0 && n >= 32) ? tpb[n] : 1.f;
#pragma unroll
        for (int x = 31; x >= 0; --x) {
          const int i = 32 * h + x;
          const bool in = i <= n;
          pv[x] = in ? -2.f * tth[i] * da * pv[x] : 0.f;
          da = in ? da * tkeep[i] : da;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t o = sw128_offset(n, 4 * h + c);
          store_split8(sbase + OFF_PHI + o, sbase + OFF_PLO + o, pv + 8 * c);
        }
        fence_proxy_async_smem();
        // ---- scale this query row of Q M0^T by a_n in place; the readout MMA
        //      then adds -2 (P E)_n onto it
        if (!mbar_wait(&bars[B_D1], par, abort_flag, kWaitLimit)) { ok = false; break; }
        tc_fence_after();
        {
          const float an = ta[n];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            float t[32];
            const uint32_t ad = tl + tm_d1(j) + 64 * h + 32 * cc;
            tmem_ld32(ad, t);
#pragma unroll
            for (int x = 0; x < 32; ++x) t[x] *= an;
            tmem_st32(ad, t);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_P]);
      }
      // ---- state update M = a_63 M - 2 dM; write the next chunk's M operand
      if (!mbar_wait(&bars[B_DM], par, abort_flag, kWaitLimit)) { ok = false; break; }
      tc_fence_after();
      {
        const float ab = ta[kChunk - 1];
        const uint32_t mh = sbase + OFF_MHI + h * 16384, ml = sbase + OFF_MLO + h * 16384;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float dm[32];
          tmem_ld32(tl + TM_DM + 64 * h + 32 * cc, dm);
#pragma unroll
          for (int x = 0; x < 32; ++x) m[32 * cc + x] = ab * m[32 * cc + x] - 2.f * dm[x];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            store_split8(mh + sw128_offset(r, 4 * cc + c), ml + sw128_offset(r, 4 * cc + c),
                         m + 32 * cc + 8 * c);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_M]);
      }
      if (!low) {
        // ---- readout: rows 64..127 of D1 now hold y_n = a_n (M0 q_n) - 2 (P E)_n
        const int n = r - 64;
        if (!mbar_wait(&bars[B_Y], par, abort_flag, kWaitLimit)) { ok = false; break; }
        tc_fence_after();
        const bool valid = t0 + n < N;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float y[32];
          tmem_ld32(tl + tm_d1(j) + 64 * h + 32 * cc, y);
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(Yh + (long)(t0 + n) * kDim + 64 * h + 32 * cc);
#pragma unroll
            for (int x = 0; x < 8; ++x)
              dst[x] = make_float4(y[4 * x], y[4 * x + 1], y[4 * x + 2], y[4 * x + 3]);
          }
        }
        tc_fence_before();
      }
    }
    if (!ok) fail();
    if (ok) {
      float4* dst = reinterpret_cast<float4*>(p.M + ((long)head * kDim + r) * kDim + 64 * h);
#pragma unroll
      for (int x = 0; x < 16; ++x) dst[x] = make_float4(m[4 * x], m[4 * x + 1], m[4 * x + 2], m[4 * x + 3]);
    }
    if (p.S) {
      // eta = 0: the final momentum is S_N = -gamma_0 theta_{N-1} 2 e_{N-1} k_{N-1}^T
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_S]);
      if (mbar_wait(&bars[B_S], 0, abort_flag, kWaitLimit) && ok) {
        const float* el = reinterpret_cast<const float*>(sm + OFF_ELAST);
        const float coef = -2.f * p.gamma[0] * p.theta[(long)head * N + N - 1] * el[r];
        const __nv_bfloat16* kl = p.K + ((long)head * N + N - 1) * kDim + 64 * h;
        float* dst = p.S + ((long)head * kDim + r) * kDim + 64 * h;
        for (int x = 0; x < 64; ++x) dst[x] = coef * __bfloat162float(kl[x]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

// ------------------------------------------------------------------ host

namespace {

std::mutex g_enc_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lock(g_enc_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

bool make_map_kq(CUtensorMap* m, const void* base, int N, int heads) {
  cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)N, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)kDim * 2, (cuuint64_t)N * kDim * 2};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_gate(CUtensorMap* m, const float* base, int N, int heads) {
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)heads};
  cuuint64_t strides[1] = {(cuuint64_t)N * 4};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t es[2] = {1, 1};
  return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

bool linear_tc_supported(const LinArgs& a) {
  return a.d_k == kDim && a.d_v == kDim && a.D == kDim && a.b == kChunk && a.c == 1 && !a.poly &&
         !a.dot && a.bf16 && a.N > 0 && (a.N % 4) == 0;
}

int linear_tc_launch(const LinArgs& a, int heads, int* status, cudaStream_t st) {
  if (!linear_tc_supported(a)) return ATLAS_ERR_UNSUPPORTED;
  if (!aligned16(a.K) || !aligned16(a.Q) || !aligned16(a.V) || !aligned16(a.alpha) ||
      !aligned16(a.eta) || !aligned16(a.theta) || !aligned16(a.Y) || !aligned16(a.M) ||
      (a.S && !aligned16(a.S)))
    return ATLAS_ERR_UNSUPPORTED;
  if (!encoder()) return ATLAS_ERR_CUDA;
  TcMaps maps;
  if (!make_map_kq(&maps.k, a.K, a.N, heads) || !make_map_kq(&maps.q, a.Q, a.N, heads) ||
      !make_map_gate(&maps.alpha, a.alpha, a.N, heads) ||
      !make_map_gate(&maps.eta, a.eta, a.N, heads) ||
      !make_map_gate(&maps.theta, a.theta, a.N, heads))
    return ATLAS_ERR_CUDA;
  TcParams p;
  p.K = reinterpret_cast<const __nv_bfloat16*>(a.K);
  p.V = reinterpret_cast<const __nv_bfloat16*>(a.V);
  p.eta = a.eta;
  p.theta = a.theta;
  p.gamma = a.gamma;
  p.Y = a.Y;
  p.M = a.M;
  p.S = a.S;
  p.status = status;
  p.N = a.N;
  if (cudaFuncSetAttribute(linear_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)SMEM_ALLOC) != cudaSuccess)
    return ATLAS_ERR_CUDA;
  linear_tc_kernel<<<heads, kThreads, SMEM_ALLOC, st>>>(maps, p);
  if (cudaGetLastError() != cudaSuccess) return ATLAS_ERR_CUDA;
  // heads with a non-zero eta: the CUDA-core kernel takes exactly those
  return linear_simt_launch_masked(a, heads, st);
}

}  // namespace atlas
