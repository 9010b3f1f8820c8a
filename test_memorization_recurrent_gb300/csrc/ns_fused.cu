// ns_fused.cu -- Newton-Schulz orthogonalisation ("ATLAS ... (paperlayer)" §5:
// Muon on the momentum) of many 128 x 512 matrices, each kept on chip for all
// its iterations:
//   X_0 = S / (||S||_F + eps),   X <- (a I + b G + c G^2) X,  G = X X^T   (steps times)
// A 512 x 128 matrix is handled as its transpose (NS commutes with transposition).
//
// One cluster of two CTAs per matrix at a time (persistent over the list of
// matrices); CTA c holds columns [256c, 256c + 256) of the 128 x 512 iterate Z,
// as bf16 hi/lo pairs in shared memory (the MMA operand) and, after each
// update, as the fp32 product in TMEM.  Per iteration:
//   G_c = Z_c Z_c^T            (tcgen05, hi*hi + hi*lo + lo*hi)        -> TMEM
//   G = G_0 + G_1              CTA c owns rows [64c, 64c + 64): the other CTA's
//                              partial rows arrive by a bulk copy, the finished
//                              rows go back to it the same way (bf16 hi/lo)
//   G2 = G G                   -> TMEM
//   B = a I + b G + c G2       -> shared memory (hi/lo), over G
//   Z_c <- B Z_c               -> TMEM, then the hi/lo copy of Z_c is refreshed
// 16 warps, four per 32-lane TMEM quadrant; one thread of warp 0 issues each
// product once its inputs are in place (every warp waits for that product next).
// Every wait is bounded; a timeout sets ATLAS_ERR_TIMEOUT in the status word.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_primitives.cuh"

namespace atlas {
using namespace tc;

namespace {

constexpr int kR = 128;     // rows of the wide iterate
constexpr int kCols = 512;  // its columns
constexpr int kHalf = 256;  // columns per CTA
constexpr int kDW = 16;     // data warps
constexpr int kThrN = kDW * 32;
constexpr long long kWaitN = 2000000000LL;

// shared memory (bytes from a 1024-aligned base)
//   S_Z   Z_c [128][256]: hi in 4 atoms of 64 columns (16 KB each) | lo
//   S_G   G, then B [128][128]: hi in 2 atoms | lo; the rows of the other CTA
//         first stage this CTA's outgoing partial sums (fp32)
//   S_RX  the other CTA's partial sums of this CTA's rows: 4 pieces of 8 KB,
//         piece h = columns [32h, 32h + 32) of the 64 rows
constexpr uint32_t S_Z = 0;
constexpr uint32_t S_G = 131072;
constexpr uint32_t S_RX = 196608;
constexpr uint32_t S_MISC = 229376;  // partial norms [16], the other CTA's norm
constexpr uint32_t S_BAR = S_MISC + 128;
constexpr uint32_t SMEM_N = S_BAR + 256 + 1024;

// TMEM columns
constexpr uint32_t T_Z = 0, T_G = 256, T_G2 = 384;

enum NBar {
  N_ZREADY = 0, N_G, N_RX, N_OWN0, N_OWN1, N_GFULL, N_GACK, N_G2, N_BREADY, N_UPD, N_NP,
  N_NORM, N_DRAIN, N_COUNT
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t a, uint32_t cluster_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr),
      "r"(a), "r"(cluster_bar)
      : "memory");
}
// shared memory of this CTA -> shared memory of a CTA of the cluster, counted
// as complete_tx bytes on that CTA's barrier
__device__ __forceinline__ void bulk_s2c(uint32_t dst, uint32_t src, uint32_t bytes,
                                         uint32_t dst_bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst),
      "r"(src), "r"(bytes), "r"(dst_bar)
      : "memory");
}
__device__ __forceinline__ void remote_arrive(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ bool try_wait_acq_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;"
      "\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded wait with cluster-scope acquire (barriers completed by the other CTA)
__device__ __forceinline__ bool wait_c(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const long long t0 = clock64();
  while (!try_wait_acq_cluster(bar, parity)) {
    if (*abort) return false;
    if (clock64() - t0 > kWaitN) return false;
  }
  return true;
}

__device__ __forceinline__ void ld_pair8(uint32_t ahi, uint32_t alo, float* x) {
  uint32_t h[4], l[4];
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
               : "r"(ahi));
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(l[0]), "=r"(l[1]), "=r"(l[2]), "=r"(l[3])
               : "r"(alo));
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    x[2 * p] = __uint_as_float(h[p] << 16) + __uint_as_float(l[p] << 16);
    x[2 * p + 1] = __uint_as_float(h[p] & 0xFFFF0000u) + __uint_as_float(l[p] & 0xFFFF0000u);
  }
}
// element (row, col) of a K-major tile whose rows are 64 bf16 per atom
__device__ __forceinline__ uint32_t kt_off(uint32_t row, uint32_t col) {
  return (col >> 6) * 16384u + sw128_offset(row, (col & 63) >> 3);
}
// 16-byte chunk j (0..7) of row rr in a piece of fp32 rows of 32 values (chunk
// index XOR (rr % 8) so that 8 consecutive rows cover all banks)
__device__ __forceinline__ uint32_t piece_off(uint32_t rr, uint32_t j) {
  return rr * 128u + ((j ^ (rr & 7u)) << 4);
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThrN, 1)
    ns_fused_kernel(NsArgs p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S_BAR + 8 * N_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + S_BAR + 8 * N_COUNT + 8);
  float* part = reinterpret_cast<float*>(sm + S_MISC);  // [16] warp sums, [16] the other CTA's

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t c = cluster_rank(), peer = c ^ 1u;
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  const int items = 2 * p.n_inst;

  if (tid == 0) {
    // arrivals per phase: the data warps (16), the four warps of a quadrant,
    // the two copying warps and the thread posting the expected bytes (3), or 1
#pragma unroll
    for (int b = 0; b < N_COUNT; ++b)
      mbar_init(&bars[b], (b == N_ZREADY || b == N_BREADY || b == N_NP) ? 16u
                          : (b == N_OWN0 || b == N_OWN1)                   ? 4u
                          : b == N_GFULL                                   ? 3u
                                                                           : 1u);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() {
    if (*abort_flag == 0 && p.status) atomicExch(p.status, ATLAS_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  constexpr uint32_t id128 = idesc_bf16(128, 128, false, false);
  constexpr uint32_t id256 = idesc_bf16(128, 256, false, true);
  auto dk = [&](uint32_t off) { return sdesc_sw128(sb + off, 16, 1024); };
  auto dm = [&](uint32_t off) { return sdesc_sw128(sb + off, 16384, 1024); };
  {
    // =========================== data warps
    const int q = warp & 3, h = warp >> 2;  // TMEM quadrant; column quarter
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    const int r = q * 32 + lane;               // row of Z, G (TMEM lane)
    const bool own = (uint32_t)(q >> 1) == c;  // G rows [64c, 64c + 64) are this CTA's
    const uint32_t rr = (uint32_t)(32 * (q & 1) + lane);  // row within the owner's 64
    bool ok = true;
    uint32_t ph = 0, iph = 0;  // iterations done; items done
    auto W = [&](int b, uint32_t par) {
      return __all_sync(0xFFFFFFFFu, mbar_wait(&bars[b], par, abort_flag, kWaitN)) != 0;
    };
    auto WC = [&](int b, uint32_t par) {
      return __all_sync(0xFFFFFFFFu, wait_c(&bars[b], par, abort_flag)) != 0;
    };
    auto arrive_warp = [&](int b) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[b]);
    };
    for (int w = cluster; ok && w < items; w += nclusters, ++iph) {
      const int inst = w >> 1, type = w & 1;
      float* base = p.X + (long)inst * p.inst_stride + (type ? p.half : 0);
      const int col0 = kHalf * (int)c + 64 * h;  // this thread's 64 columns of the 512
      // ---- X_0 = S / (||S|| + eps) (type 1: of S^T) -> hi / lo in shared memory;
      // the block is read twice (the second time from L2): sum of squares, then scaled
      auto load8 = [&](int j0, float* v) {
        if (type == 0) {
          const float4* src = reinterpret_cast<const float4*>(base + (long)r * kCols + col0 + j0);
          const float4 x = src[0], y = src[1];
          v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
          v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = base[(long)(col0 + j0 + e) * kR + r];
        }
      };
      {
        float ss = 0.f;
#pragma unroll 2
        for (int k = 0; k < 8; ++k) {
          float v[8];
          load8(8 * k, v);
#pragma unroll
          for (int e = 0; e < 8; ++e) ss += v[e] * v[e];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
        if (lane == 0) part[warp] = ss;
        arrive_warp(N_NP);
        if (!(ok = W(N_NP, iph & 1))) break;
        float cta = 0.f;
#pragma unroll
        for (int x = 0; x < kDW; ++x) cta += part[x];
        if (warp == 0 && lane == 0) {  // this CTA's sum to the other CTA
          mbar_arrive_expect_tx(&bars[N_NORM], 4);
          st_async_b32(mapa(sb + S_MISC + 4 * kDW, peer), __float_as_uint(cta),
                       mapa(smem_u32(&bars[N_NORM]), peer));
        }
        if (!(ok = WC(N_NORM, iph & 1))) break;
        const float inv = 1.f / (sqrtf(cta + part[kDW]) + p.eps);
#pragma unroll 2
        for (int k = 0; k < 8; ++k) {
          float v[8];
          load8(8 * k, v);
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] *= inv;
          const uint32_t off = kt_off(r, 64 * h + 8 * k);
          store_split8(sb + S_Z + off, sb + S_Z + 65536 + off, v);
        }
        fence_proxy_async_smem();
        arrive_warp(N_ZREADY);
      }

      for (int it = 0; ok && it < p.steps; ++it, ++ph) {
        const uint32_t par = ph & 1;
        if (warp == 0) {  // G_c = Z_c Z_c^T over the CTA's 256 columns
          if (!(ok = W(N_ZREADY, par))) break;
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
#pragma unroll
              for (int s = 0; s < 3; ++s) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_bf16(tmem + T_G, dk(S_Z + (s == 2 ? 65536 : 0) + off),
                         dk(S_Z + (s == 1 ? 65536 : 0) + off), id128, (kk | s) ? 1u : 0u);
              }
            mma_commit(&bars[N_G]);
          }
          __syncwarp();
        }
        // ---- G = G_0 + G_1 (this thread: row r, columns [32h, 32h + 32))
        if (!(ok = W(N_G, par))) break;
        tc_fence_after();
        float g[32];
        tmem_ld32(tl + T_G + 32 * h, g);
        if (!own) {  // partial sums of the other CTA's rows: stage, then one bulk copy per warp
          const uint32_t stage = sb + S_G + 16384 * h + 8192 * peer;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_shared_v4(stage + piece_off(rr, j), __float_as_uint(g[4 * j]),
                         __float_as_uint(g[4 * j + 1]), __float_as_uint(g[4 * j + 2]),
                         __float_as_uint(g[4 * j + 3]));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const uint32_t blk = 4096 * (q & 1);
            bulk_s2c(mapa(sb + S_RX + 8192 * h + blk, peer), stage + blk, 4096,
                     mapa(smem_u32(&bars[N_RX]), peer));
          }
        } else {
          if (h == 0 && lane == 0 && q == 2 * (int)c) {
            mbar_arrive_expect_tx(&bars[N_RX], 32768);     // the other CTA's partial sums
            mbar_arrive_expect_tx(&bars[N_GFULL], 32768);  // its finished rows (hi / lo)
          }
          if (!(ok = WC(N_RX, par))) break;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 x =
                *reinterpret_cast<const float4*>(sm + S_RX + 8192 * h + piece_off(rr, j));
            g[4 * j] += x.x; g[4 * j + 1] += x.y; g[4 * j + 2] += x.z; g[4 * j + 3] += x.w;
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t off = kt_off(r, 32 * h + 8 * k);
            store_split8(sb + S_G + off, sb + S_G + 32768 + off, g + 8 * k);
          }
          fence_proxy_async_smem();
          arrive_warp(N_OWN0 + (q & 1));
          if (h == 0) {  // the quadrant's 32 finished rows to the other CTA
            if (!(ok = W(N_OWN0 + (q & 1), par))) break;
            if (lane == 0) {
              const uint32_t bar = mapa(smem_u32(&bars[N_GFULL]), peer);
#pragma unroll
              for (int t = 0; t < 4; ++t) {  // hi atom 0, hi atom 1, lo atom 0, lo atom 1
                const uint32_t off = S_G + 16384 * t + 4096 * q;
                bulk_s2c(mapa(sb + off, peer), sb + off, 4096, bar);
              }
              mbar_arrive(&bars[N_GFULL]);
            }
            __syncwarp();
          }
        }
        if (!(ok = WC(N_GFULL, par))) break;
        if (warp == 0 && lane == 0)  // this CTA's copy of the other's rows has landed
          remote_arrive(mapa(smem_u32(&bars[N_GACK]), peer));
        if (warp == 0) {  // G2 = G G (G symmetric: one tile, both sides)
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
#pragma unroll
              for (int s = 0; s < 3; ++s) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_bf16(tmem + T_G2, dk(S_G + (s == 2 ? 32768 : 0) + off),
                         dk(S_G + (s == 1 ? 32768 : 0) + off), id128, (kk | s) ? 1u : 0u);
              }
            mma_commit(&bars[N_G2]);
          }
          __syncwarp();
        }
        // ---- B = a I + b G + c G^2 (G from shared memory, G^2 from TMEM), over G
        if (!(ok = W(N_G2, par))) break;
        if (own && !(ok = WC(N_GACK, par))) break;  // own rows no longer read by the copy
        tc_fence_after();
        float g2[32];
        tmem_ld32(tl + T_G2 + 32 * h, g2);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t off = kt_off(r, 32 * h + 8 * k);
          float gg[8];
          ld_pair8(sb + S_G + off, sb + S_G + 32768 + off, gg);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            gg[e] = p.b * gg[e] + p.c * g2[8 * k + e];
            if (32 * h + 8 * k + e == r) gg[e] += p.a;
          }
          store_split8(sb + S_G + off, sb + S_G + 32768 + off, gg);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        arrive_warp(N_BREADY);
        if (warp == 0) {  // Z_c = B Z_c
          if (!(ok = W(N_BREADY, par))) break;
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
#pragma unroll
              for (int s = 0; s < 3; ++s) {
                const uint32_t a = S_G + (s == 2 ? 32768 : 0) + (kk >> 2) * 16384 + (kk & 3) * 32;
                const uint32_t b = S_Z + (s == 1 ? 65536 : 0) + kk * 2048;
                mma_bf16(tmem + T_Z, dk(a), dm(b), id256, (kk | s) ? 1u : 0u);
              }
            mma_commit(&bars[N_UPD]);
          }
          __syncwarp();
        }
        // ---- refresh the hi / lo copy of Z_c, or write the result out
        if (!(ok = W(N_UPD, par))) break;
        tc_fence_after();
        const bool last = it + 1 == p.steps;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          float v[32];
          tmem_ld32(tl + T_Z + 64 * h + 32 * u, v);
          if (!last) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t off = kt_off(r, 64 * h + 32 * u + 8 * k);
              store_split8(sb + S_Z + off, sb + S_Z + 65536 + off, v + 8 * k);
            }
          } else if (type == 0) {
            float4* dst = reinterpret_cast<float4*>(base + (long)r * kCols + col0 + 32 * u);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) base[(long)(col0 + 32 * u + e) * kR + r] = v[e];
          }
        }
        tc_fence_before();
        if (!last) {
          fence_proxy_async_smem();
          arrive_warp(N_ZREADY);
        }
      }
    }
    if (!ok) {
      fail();
      if (warp == 0 && lane == 0) {  // no MMA may outlive the TMEM
        volatile int zero = 0;
        mma_commit(&bars[N_DRAIN]);
        mbar_wait(&bars[N_DRAIN], 0, &zero, kWaitN);
      }
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while the other may still write into it
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

bool ns_fused_supported(int d, int dh) { return d == kR && dh == kCols; }

int ns_fused_launch(const NsArgs& a, cudaStream_t st) {
  if (a.n_inst <= 0 || a.steps <= 0) return ATLAS_OK;
  if ((reinterpret_cast<uintptr_t>(a.X) & 15) || (a.inst_stride & 3) || (a.half & 3))
    return ATLAS_ERR_UNSUPPORTED;
  static bool attr = false;
  static int nsm = 0;
  if (!attr) {
    if (cudaFuncSetAttribute(ns_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_N) != cudaSuccess)
      return ATLAS_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATLAS_ERR_CUDA;
    attr = true;
  }
  int clusters = nsm / 2;
  if (clusters > 2 * a.n_inst) clusters = 2 * a.n_inst;
  if (clusters < 1) clusters = 1;
  ns_fused_kernel<<<2 * clusters, kThrN, SMEM_N, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? ATLAS_OK : ATLAS_ERR_CUDA;
}

}  // namespace atlas
