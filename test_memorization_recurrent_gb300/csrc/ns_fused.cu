// ns_fused.cu -- Newton-Schulz orthogonalisation ("ATLAS ... (paperlayer)" §5:
// Muon on the momentum) of many 128 x 512 matrices, each kept on chip for all
// its iterations:
//   X_0 = S / (||S||_F + eps),   X <- a X + b (X X^T) X + c (X X^T)^2 X   (steps times)
// A 512 x 128 matrix is handled as its transpose (NS commutes with transposition).
//
// One cluster of two CTAs per matrix at a time (persistent over the list of
// matrices); CTA c holds columns [256c, 256c + 256) of the 128 x 512 iterate Z:
// fp32 in TMEM (the accumulator of the update) and as bf16 hi/lo pairs in shared
// memory (the MMA operand).  Per iteration:
//   G_c = Z_c Z_c^T            (tcgen05, hi*hi + hi*lo + lo*hi)        -> TMEM
//   G = G_0 + G_1              CTA c owns rows [64c, 64c + 64): the other CTA's
//                              partial rows arrive by st.async, the finished
//                              rows go back to it as bf16 hi/lo pairs
//   G2 = G G                   -> TMEM
//   B = b G + c G2             -> shared memory (hi/lo)
//   Z_c <- a Z_c + B Z_c       -> TMEM (a Z_c was stored there with the hi/lo copy)
// Warps 0..7 move data (two per 32-lane TMEM quadrant), warp 8 issues the MMAs.
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
constexpr int kThrN = 288;  // 8 data warps + 1 MMA warp
constexpr long long kWaitN = 2000000000LL;

// shared memory (bytes from a 1024-aligned base)
constexpr uint32_t S_Z = 0;            // Z_c [128][256] hi (4 atoms) | lo: 128 KB
constexpr uint32_t S_G = 131072;       // G, then B [128][128] hi (2 atoms) | lo: 64 KB
constexpr uint32_t S_RX = 196608;      // the other CTA's partial rows [64][128] fp32: 32 KB
constexpr uint32_t S_MISC = 229376;    // partial norms [8], the other CTA's norm
constexpr uint32_t S_BAR = S_MISC + 64;
constexpr uint32_t SMEM_N = S_BAR + 256 + 1024;

// TMEM columns
constexpr uint32_t T_Z = 0, T_G = 256, T_G2 = 384;

enum NBar { N_ZREADY = 0, N_G, N_RX, N_GFULL, N_G2, N_BREADY, N_UPD, N_NP, N_NORM, N_DRAIN, N_COUNT };

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
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                            uint32_t d, uint32_t cluster_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::
          "r"(addr),
      "r"(a), "r"(b), "r"(c), "r"(d), "r"(cluster_bar)
      : "memory");
}
__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t a, uint32_t cluster_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr),
      "r"(a), "r"(cluster_bar)
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

__device__ __forceinline__ uint32_t bits_rn(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
// 8 values -> hi / lo pairs of bf16 packed into two uint4 (element 2p in the low half)
__device__ __forceinline__ void split8u(const float* x, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const float h0 = __bfloat162float(__float2bfloat16_rn(x[2 * p]));
    const float h1 = __bfloat162float(__float2bfloat16_rn(x[2 * p + 1]));
    h[p] = bits_rn(h0) | (bits_rn(h1) << 16);
    l[p] = bits_rn(x[2 * p] - h0) | (bits_rn(x[2 * p + 1] - h1) << 16);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
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
// 16-byte chunk q (0..31) of row rr of the receive buffer (rows of 512 bytes,
// chunk index XOR (rr % 8) so that a warp's rows spread over the banks)
__device__ __forceinline__ uint32_t rx_off(uint32_t rr, uint32_t q) {
  return rr * 512u + ((q ^ (rr & 7u)) << 4);
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
  float* part = reinterpret_cast<float*>(sm + S_MISC);  // [8] warp sums, [8] the other CTA's

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t c = cluster_rank(), peer = c ^ 1u;
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  const int items = 2 * p.n_inst;

  if (tid == 0) {
    // arrivals per phase: the data warps (8), the MMA commit (1), or the owner
    // warps and the thread posting the expected bytes (5)
#pragma unroll
    for (int b = 0; b < N_COUNT; ++b)
      mbar_init(&bars[b], (b == N_ZREADY || b == N_BREADY || b == N_NP) ? 8u : b == N_GFULL ? 5u : 1u);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8) {
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

  if (warp == 8) {
    // =========================== MMA issuer
    bool ok = true;
    if (lane == 0) {
      uint32_t ph = 0;  // completed iterations over all items
      constexpr uint32_t id128 = idesc_bf16(128, 128, false, false);
      constexpr uint32_t id256 = idesc_bf16(128, 256, false, true);
      auto dk = [&](uint32_t off) { return sdesc_sw128(sb + off, 16, 1024); };
      auto dm = [&](uint32_t off) { return sdesc_sw128(sb + off, 16384, 1024); };
      for (int w = cluster; ok && w < items; w += nclusters) {
        for (int it = 0; ok && it < p.steps; ++it, ++ph) {
          const uint32_t par = ph & 1;
          if (!(ok = mbar_wait(&bars[N_ZREADY], par, abort_flag, kWaitN))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)  // G_c = Z_c Z_c^T over the CTA's 256 columns
#pragma unroll
            for (int s = 0; s < 3; ++s) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              mma_bf16(tmem + T_G, dk(S_Z + (s == 2 ? 65536 : 0) + off),
                       dk(S_Z + (s == 1 ? 65536 : 0) + off), id128, (kk | s) ? 1u : 0u);
            }
          mma_commit(&bars[N_G]);
          if (!(ok = wait_c(&bars[N_GFULL], par, abort_flag))) break;
          fence_proxy_async_smem();  // rows stored by the other CTA -> visible to the MMA
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // G2 = G G (G symmetric: one tile, both sides)
#pragma unroll
            for (int s = 0; s < 3; ++s) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              mma_bf16(tmem + T_G2, dk(S_G + (s == 2 ? 32768 : 0) + off),
                       dk(S_G + (s == 1 ? 32768 : 0) + off), id128, (kk | s) ? 1u : 0u);
            }
          mma_commit(&bars[N_G2]);
          if (!(ok = mbar_wait(&bars[N_BREADY], par, abort_flag, kWaitN))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // Z_c (already a Z_c) += B Z_c
#pragma unroll
            for (int s = 0; s < 3; ++s) {
              const uint32_t a = S_G + (s == 2 ? 32768 : 0) + (kk >> 2) * 16384 + (kk & 3) * 32;
              const uint32_t b = S_Z + (s == 1 ? 65536 : 0) + kk * 2048;
              mma_bf16(tmem + T_Z, dk(a), dm(b), id256, 1u);
            }
          mma_commit(&bars[N_UPD]);
        }
      }
      if (!ok) {
        fail();
        volatile int zero = 0;
        mma_commit(&bars[N_DRAIN]);
        mbar_wait(&bars[N_DRAIN], 0, &zero, kWaitN);
      }
    }
    __syncwarp();
  } else {
    // =========================== data warps
    const int q = warp & 3, h = warp >> 2;
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    const int r = q * 32 + lane;                     // row of Z, G (TMEM lane)
    const bool own = (uint32_t)(q >> 1) == c;        // G rows [64c, 64c + 64) are this CTA's
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
      // ---- load the CTA's 128 x 256 block of S (type 1: of S^T), sum of squares
      float ss = 0.f;
      for (int u = 0; u < 4; ++u) {
        const int j0 = 128 * h + 32 * u, col0 = kHalf * (int)c + j0;
        float v[32];
        if (type == 0) {
          const float4* src = reinterpret_cast<const float4*>(base + (long)r * kCols + col0);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 x = src[e];
            v[4 * e] = x.x; v[4 * e + 1] = x.y; v[4 * e + 2] = x.z; v[4 * e + 3] = x.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = base[(long)(col0 + e) * kR + r];
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) ss += v[e] * v[e];
        tmem_st32(tl + T_Z + j0, v);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
      if (lane == 0) part[warp] = ss;
      arrive_warp(N_NP);
      if (!(ok = W(N_NP, iph & 1))) break;
      float cta = 0.f;
#pragma unroll
      for (int x = 0; x < 8; ++x) cta += part[x];
      if (warp == 0 && lane == 0) {  // this CTA's sum to the other CTA
        mbar_arrive_expect_tx(&bars[N_NORM], 4);
        st_async_b32(mapa(sb + S_MISC + 32, peer), __float_as_uint(cta),
                     mapa(smem_u32(&bars[N_NORM]), peer));
      }
      if (!(ok = WC(N_NORM, iph & 1))) break;
      const float inv = 1.f / (sqrtf(cta + part[8]) + p.eps);
      // ---- X_0 = S / (||S|| + eps): TMEM (fp32) and shared memory (hi / lo)
      for (int u = 0; u < 4; ++u) {
        const int j0 = 128 * h + 32 * u;
        float v[32];
        tmem_ld32(tl + T_Z + j0, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] *= inv;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t off = kt_off(r, j0 + 8 * k);
          store_split8(sb + S_Z + off, sb + S_Z + 65536 + off, v + 8 * k);
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] *= p.a;
        tmem_st32(tl + T_Z + j0, v);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      arrive_warp(N_ZREADY);

      for (int it = 0; ok && it < p.steps; ++it, ++ph) {
        const uint32_t par = ph & 1;
        // ---- G = G_0 + G_1: partial rows of the other CTA's half go to it
        if (!(ok = W(N_G, par))) break;
        tc_fence_after();
        float g[64];
        tmem_ld32(tl + T_G + 64 * h, g);
        tmem_ld32(tl + T_G + 64 * h + 32, g + 32);
        tc_fence_before();
        if (!own) {
          const uint32_t rr = (uint32_t)(r - 64 * (int)peer);
          const uint32_t bar = mapa(smem_u32(&bars[N_RX]), peer);
#pragma unroll
          for (int k = 0; k < 16; ++k)
            st_async_v4(mapa(sb + S_RX + rx_off(rr, 16 * h + k), peer), __float_as_uint(g[4 * k]),
                        __float_as_uint(g[4 * k + 1]), __float_as_uint(g[4 * k + 2]),
                        __float_as_uint(g[4 * k + 3]), bar);
        } else {
          if (h == 0 && lane == 0 && q == 2 * (int)c) {
            mbar_arrive_expect_tx(&bars[N_RX], 32768);   // the other CTA's partial rows
            mbar_arrive_expect_tx(&bars[N_GFULL], 32768);  // its finished rows (hi / lo)
          }
          if (!(ok = WC(N_RX, par))) break;
          const uint32_t rr = (uint32_t)(r - 64 * (int)c);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float4 x = *reinterpret_cast<const float4*>(sm + S_RX + rx_off(rr, 16 * h + k));
            g[4 * k] += x.x; g[4 * k + 1] += x.y; g[4 * k + 2] += x.z; g[4 * k + 3] += x.w;
          }
          const uint32_t bar = mapa(smem_u32(&bars[N_GFULL]), peer);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t off = kt_off(r, 64 * h + 8 * k);
            uint4 hi, lo;
            split8u(g + 8 * k, hi, lo);
            st_shared_v4(sb + S_G + off, hi.x, hi.y, hi.z, hi.w);
            st_shared_v4(sb + S_G + 32768 + off, lo.x, lo.y, lo.z, lo.w);
            st_async_v4(mapa(sb + S_G + off, peer), hi.x, hi.y, hi.z, hi.w, bar);
            st_async_v4(mapa(sb + S_G + 32768 + off, peer), lo.x, lo.y, lo.z, lo.w, bar);
          }
          fence_proxy_async_smem();
          arrive_warp(N_GFULL);
        }
        // ---- B = b G + c G^2 (G from shared memory, G^2 from TMEM)
        if (!(ok = W(N_G2, par))) break;
        if (!(ok = WC(N_GFULL, par))) break;
        tc_fence_after();
        float g2[64];
        tmem_ld32(tl + T_G2 + 64 * h, g2);
        tmem_ld32(tl + T_G2 + 64 * h + 32, g2 + 32);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = kt_off(r, 64 * h + 8 * k);
          float gg[8];
          ld_pair8(sb + S_G + off, sb + S_G + 32768 + off, gg);
#pragma unroll
          for (int e = 0; e < 8; ++e) gg[e] = p.b * gg[e] + p.c * g2[8 * k + e];
          store_split8(sb + S_G + off, sb + S_G + 32768 + off, gg);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        arrive_warp(N_BREADY);
        // ---- refresh the hi / lo copy of Z_c, or write the result out
        if (!(ok = W(N_UPD, par))) break;
        tc_fence_after();
        const bool last = it + 1 == p.steps;
        for (int u = 0; u < 4; ++u) {
          const int j0 = 128 * h + 32 * u, col0 = kHalf * (int)c + j0;
          float v[32];
          tmem_ld32(tl + T_Z + j0, v);
          if (!last) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t off = kt_off(r, j0 + 8 * k);
              store_split8(sb + S_Z + off, sb + S_Z + 65536 + off, v + 8 * k);
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] *= p.a;  // the update accumulates onto a Z
            tmem_st32(tl + T_Z + j0, v);
          } else if (type == 0) {
            float4* dst = reinterpret_cast<float4*>(base + (long)r * kCols + col0);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) base[(long)(col0 + e) * kR + r] = v[e];
          }
        }
        if (!last) {
          fence_proxy_async_smem();
          tc_fence_before();
          arrive_warp(N_ZREADY);
        }
      }
    }
    if (!ok) fail();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while the other may still write into it
  if (warp == 8) {
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
