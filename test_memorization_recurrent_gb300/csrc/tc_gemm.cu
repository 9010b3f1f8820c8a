// tc_gemm.cu -- batched tensor-core GEMM (tcgen05, TMEM accumulator) on fp32
// operands with arbitrary strides, used by the batched Newton-Schulz step and
// the window products of the MLP-memory path.
//
//   C[b](m, n) = alpha * rowscale[b](m) * sum_k A[b](m, k) kscale[b](k) B[b](k, n)
//                (* emul[b](m, n)) + beta * dscale[b] * D[b](m, n)  (+ C[b](m, n) when
//                accumulating), then optionally C = GELU(that), C2 = GELU'(that)
//
// Each operand element is split into bf16 hi + lo (hi = rn(x), lo = rn(x - hi));
// the product is accumulated in fp32 from hi*hi + hi*lo + lo*hi, which keeps
// ~2^-16 relative accuracy per operand from bf16 tensor-core instructions.
//
// Tile 128 x 128 per CTA, K in blocks of 64.  256 threads stage a block's fp32
// operands into shared memory as 128B-swizzled K-major bf16 tiles (hi and lo);
// the next block is loaded into registers while the tensor cores work on the
// current one.  Loads are 16-byte vectors along whichever of the two operand
// dimensions is contiguous (the host checks alignment), scalar otherwise.  One
// thread issues the 12 MMAs of a block; the epilogue reads the accumulator out
// of TMEM, two warps per 32-lane quadrant.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_primitives.cuh"

namespace atlas {
using namespace tc;

namespace {

__device__ __forceinline__ float gelu_exact(float x) {
  return 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
}
__device__ __forceinline__ float gelu_exact_prime(float x) {
  return 0.5f * (1.f + erff(x * 0.70710678118654752f)) +
         x * 0.39894228040143268f * expf(-0.5f * x * x);
}

constexpr int TB = 128;           // tile M = tile N
constexpr int TK = 64;            // K block (one 128-byte bf16 row)
constexpr int kThr = 256;
constexpr uint32_t TILE = 16384;  // 128 rows x 128 B
constexpr uint32_t OFF_AHI = 0, OFF_ALO = TILE, OFF_BHI = 2 * TILE, OFF_BLO = 3 * TILE;
constexpr uint32_t SMEM_G = 4 * TILE + 1024 + 64;
constexpr long long kWaitLimitG = 2000000000LL;

// Operand access modes (host-chosen).
enum Mode { M_SCALAR = 0, M_KVEC = 1, M_RVEC = 2 };

struct Operand {
  const float* X;
  long sR, sK;   // strides of row r and k
  int R, K;      // extents
  int mode;
  const float* ks;  // optional per-k factor
};

// Raw values of one K block of one operand for this thread: 32 floats.
//   M_KVEC:  4 chunks (row, 8 consecutive k), rows tid/8 + 32 j, chunk tid % 8
//   M_RVEC:  rows 4*(tid%32) .. +3, k = 8*(tid/32) .. +7 (4 rows x 8 k)
//   M_SCALAR: as M_KVEC, element by element
__device__ __forceinline__ void load_block(const Operand& o, int r0, int k0, float* v) {
  const int tid = threadIdx.x;
  if (o.mode == M_RVEC) {
    const int rb = 4 * (tid & 31), kb = 8 * (tid >> 5);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int k = k0 + kb + e, r = r0 + rb;
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (k < o.K) {
        if (r + 3 < o.R) {
          x = *reinterpret_cast<const float4*>(o.X + (long)k * o.sK + r);
        } else {
          if (r < o.R) x.x = o.X[(long)k * o.sK + r];
          if (r + 1 < o.R) x.y = o.X[(long)k * o.sK + r + 1];
          if (r + 2 < o.R) x.z = o.X[(long)k * o.sK + r + 2];
        }
        if (o.ks) {
          const float f = o.ks[k];
          x.x *= f; x.y *= f; x.z *= f; x.w *= f;
        }
      }
      v[e] = x.x; v[8 + e] = x.y; v[16 + e] = x.z; v[24 + e] = x.w;  // [row][k]
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = r0 + (tid >> 3) + 32 * j, k = k0 + 8 * (tid & 7);
    float* x = v + 8 * j;
    if (o.mode == M_KVEC && r < o.R && k + 7 < o.K) {
      const float4 a = *reinterpret_cast<const float4*>(o.X + (long)r * o.sR + k);
      const float4 b = *reinterpret_cast<const float4*>(o.X + (long)r * o.sR + k + 4);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        x[e] = (r < o.R && k + e < o.K) ? o.X[(long)r * o.sR + (long)(k + e) * o.sK] : 0.f;
    }
    if (o.ks) {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] *= (k + e < o.K) ? o.ks[k + e] : 0.f;
    }
  }
}

// Split the block held in v into the hi / lo tiles.  Rows at or past `rows` (the
// operand's extent inside this tile) are left as they are: a row of A or B only
// reaches the output row or column of the same index, which is never stored.
__device__ __forceinline__ void store_block(const Operand& o, const float* v, uint32_t hi,
                                            uint32_t lo, int rows) {
  const int tid = threadIdx.x;
  if (o.mode == M_RVEC) {
    // all lanes of a warp hold the same k chunk; rotating the row order by lane
    // spreads one store instruction over all eight 16-byte bank groups
    // (the row is picked by selects, not by indexing v, so that v stays in registers)
    const int l = tid & 31, rb = 4 * l, c = tid >> 5;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int qq = (q + l) & 3;
      float t[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        t[e] = (qq & 2) ? ((qq & 1) ? v[24 + e] : v[16 + e]) : ((qq & 1) ? v[8 + e] : v[e]);
      const uint32_t off = sw128_offset((uint32_t)(rb + qq), (uint32_t)c);
      if (rb + qq < rows) store_split8(hi + off, lo + off, t);
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if ((tid >> 3) + 32 * j >= rows) break;
    const uint32_t off = sw128_offset((uint32_t)((tid >> 3) + 32 * j), (uint32_t)(tid & 7));
    store_split8(hi + off, lo + off, v + 8 * j);
  }
}

}  // namespace

__global__ void __launch_bounds__(kThr, 2) tc_gemm_kernel(TcGemm g) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 4 * TILE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + 4 * TILE + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + 4 * TILE + 16);

  const int nsplit = g.ksplit > 1 ? g.ksplit : 1;
  const int bz = blockIdx.z / nsplit, split = blockIdx.z % nsplit;
  const long bo = g.bdiv > 0 ? bz / g.bdiv : bz, bi = g.bdiv > 0 ? bz % g.bdiv : 0;
  // this CTA's K range (whole blocks of TK)
  const int kchunk = ((g.K + nsplit - 1) / nsplit + TK - 1) / TK * TK;
  const int kbeg = split * kchunk, kend = min(g.K, kbeg + kchunk);
  const int m0 = blockIdx.y * TB, n0 = blockIdx.x * TB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // A(m, k) and B(k, n) seen as rows m / n over k
  Operand oa{g.A + bo * g.sAb + bi * g.sAb2, g.sAm, g.sAk, g.M, kend, g.modeA,
             g.kscale ? g.kscale + bo * g.sKb + bi * g.sKb2 : nullptr};
  Operand ob{g.B + bo * g.sBb + bi * g.sBb2, g.sBn, g.sBk, g.N, kend, g.modeB, nullptr};
  const bool sym = g.symmetric != 0;

  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, TB);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sb = smem_u32(sm);
  const uint64_t dK = sdesc_sw128(0, 16, 1024) | (uint64_t)((sb >> 4) & 0x3FFFu);
  constexpr uint32_t kId = idesc_bf16(128, 128, false, false);

  bool ok = true;
  int commits = 0;
  const int nkb = kend > kbeg ? (kend - kbeg + TK - 1) / TK : 0;
  float va[32], vb[32];
  if (nkb > 0) {
    load_block(oa, m0, kbeg, va);
    if (!sym) load_block(ob, n0, kbeg, vb);
  }
  for (int kb = 0; kb < nkb && ok; ++kb) {
    if (kb > 0) {  // the tiles are read by the previous block's MMAs until they complete
      ok = mbar_wait(bar, commits & 1, abort_flag, kWaitLimitG);
      ++commits;
      tc_fence_after();
      if (!ok) break;
    }
    store_block(oa, va, sb + OFF_AHI, sb + OFF_ALO, min(TB, g.M - m0));
    if (!sym) store_block(ob, vb, sb + OFF_BHI, sb + OFF_BLO, min(TB, g.N - n0));
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
#pragma unroll
      for (int s = 0; s < 12; ++s) {
        const int part = s >> 2, k = s & 3;  // hi*hi, hi*lo, lo*hi
        const uint32_t a = (part == 2 ? OFF_ALO : OFF_AHI) + 32 * k;
        const uint32_t b = (sym ? (part == 1 ? OFF_ALO : OFF_AHI) : (part == 1 ? OFF_BLO : OFF_BHI)) +
                           32 * k;
        mma_bf16(tmem, dK + (a >> 4), dK + (b >> 4), kId, (kb > 0 || s > 0) ? 1u : 0u);
      }
      mma_commit(bar);
    }
    __syncwarp();
    if (kb + 1 < nkb) {  // next block into registers while the MMAs run
      load_block(oa, m0, kbeg + (kb + 1) * TK, va);
      if (!sym) load_block(ob, n0, kbeg + (kb + 1) * TK, vb);
    }
  }
  if (ok && nkb > 0) {
    ok = mbar_wait(bar, commits & 1, abort_flag, kWaitLimitG);
    ++commits;
    tc_fence_after();
  }
  if (!ok) {
    if (tid == 0 && g.status) atomicExch(g.status, ATLAS_ERR_TIMEOUT);
  } else if (nkb > 0 && g.sCn == 1 && (!g.D || g.sDn == 1)) {
    // ---- epilogue through shared memory (the operand tiles are free): thread =
    // row m, columns [64 (warp / 4), +64) into an fp32 [128][128] tile in 16-byte
    // groups, group g of row m at g XOR (m % 32); then each warp writes whole rows,
    // four columns a lane
    float* tile = reinterpret_cast<float*>(sm);
    {
      const int q = warp & 3, half = warp >> 2;
      const int ml = q * 32 + lane;
      const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int c0 = 64 * half; c0 < 64 * half + 64 && n0 + c0 < g.N; c0 += 32) {
        float acc[32];
        tmem_ld32(tl + c0, acc);
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4)
          *reinterpret_cast<float4*>(tile + ml * TB + 4 * (((c0 >> 2) + g4) ^ lane)) =
              make_float4(acc[4 * g4], acc[4 * g4 + 1], acc[4 * g4 + 2], acc[4 * g4 + 3]);
      }
    }
    __syncthreads();
    float* C = g.C + bo * g.sCb + bi * g.sCb2;
    const float* D = g.D ? g.D + bo * g.sDb + bi * g.sDb2 : nullptr;
    const float db = g.beta * (g.dscale ? g.dscale[bo * g.sEb + bi * g.sEb2] : 1.f);
    const float* RS = g.rowscale ? g.rowscale + bo * g.sRb + bi * g.sRb2 : nullptr;
    // rows of C start 16-byte aligned: whole groups go out as one vector
    const bool cvec = ((reinterpret_cast<uintptr_t>(C) & 15) == 0) && (g.sCm & 3) == 0;
    const int n = n0 + 4 * lane;  // this lane's columns n .. n + 3
    for (int ml = warp; ml < TB; ml += kThr / 32) {
      const int m = m0 + ml;
      if (m >= g.M) break;
      if (n >= g.N) continue;
      const float rs = g.alpha * (RS ? RS[m] : 1.f);
      const float4 t4 = *reinterpret_cast<const float4*>(tile + ml * TB + 4 * (lane ^ (ml & 31)));
      float t[4] = {rs * t4.x, rs * t4.y, rs * t4.z, rs * t4.w};
      float* crow = C + (long)m * g.sCm;
      if (nsplit > 1) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (n + e < g.N) atomicAdd(crow + n + e, t[e]);
        continue;
      }
      const bool full = cvec && n + 3 < g.N;
      const float* drow = D ? D + (long)m * g.sDm : nullptr;
      float cur[4] = {0.f, 0.f, 0.f, 0.f};
      if (g.accumulate) {
        if (full) {
          const float4 c4 = *reinterpret_cast<const float4*>(crow + n);
          cur[0] = c4.x; cur[1] = c4.y; cur[2] = c4.z; cur[3] = c4.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (n + e < g.N) cur[e] = crow[n + e];
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (n + e >= g.N) break;
        float x = t[e];
        if (g.emul) x *= g.emul[bo * g.sMb + bi * g.sMb2 + (long)m * g.sMm + (long)(n + e) * g.sMn];
        if (drow) x += db * drow[n + e];
        float pre = g.accumulate ? cur[e] + x : x;
        if (g.epi) {
          if (g.C2)
            g.C2[bo * g.sC2b + bi * g.sC2b2 + (long)m * g.sC2m + (long)(n + e) * g.sC2n] =
                gelu_exact_prime(pre);
          pre = gelu_exact(pre);
        }
        t[e] = pre;
      }
      if (full) {
        *reinterpret_cast<float4*>(crow + n) = make_float4(t[0], t[1], t[2], t[3]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (n + e < g.N) crow[n + e] = t[e];
      }
    }
  } else if (nkb > 0) {
    // ---- general strides: thread = row m of the tile, columns [64 (warp / 4), +64)
    const int q = warp & 3, half = warp >> 2;
    const int m = m0 + q * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    const float rs =
        (g.rowscale && m < g.M) ? g.rowscale[bo * g.sRb + bi * g.sRb2 + m] : 1.f;
    float* C = g.C + bo * g.sCb + bi * g.sCb2;
    const float* D = g.D ? g.D + bo * g.sDb + bi * g.sDb2 : nullptr;
    const float db = g.beta * (g.dscale ? g.dscale[bo * g.sEb + bi * g.sEb2] : 1.f);
#pragma unroll 1
    for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 32) {
      float acc[32];
      tmem_ld32(tl + c0, acc);
      if (m < g.M) {
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const int n = n0 + c0 + x;
          if (n >= g.N) continue;
          float t = g.alpha * rs * acc[x];
          if (g.emul) t *= g.emul[bo * g.sMb + bi * g.sMb2 + (long)m * g.sMm + (long)n * g.sMn];
          if (D) t += db * D[(long)m * g.sDm + (long)n * g.sDn];
          float* c = C + (long)m * g.sCm + (long)n * g.sCn;
          const float pre = g.accumulate ? *c + t : t;
          if (g.epi) {
            *c = gelu_exact(pre);
            if (g.C2)
              g.C2[bo * g.sC2b + bi * g.sC2b2 + (long)m * g.sC2m + (long)n * g.sC2n] =
                  gelu_exact_prime(pre);
          } else {
            *c = pre;
          }
        }
      }
    }
  }
  // no MMA may outlive the TMEM (on a timeout, wait once more without abort)
  if (!ok && tid == 0) {
    volatile int zero = 0;
    mma_commit(bar);
    mbar_wait(bar, commits & 1, &zero, kWaitLimitG);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TB);
  }
}

namespace {

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Vector mode for an operand X(r, k) = X[r * sR + k * sK] with rows / k extents.
int pick_mode(const float* X, long sR, long sK, long sb, long sb2, int batch) {
  const bool base_ok = al16(X) && (batch <= 1 || (sb % 4 == 0 && sb2 % 4 == 0));
  if (sK == 1 && sR % 4 == 0 && base_ok) return M_KVEC;
  if (sR == 1 && sK % 4 == 0 && base_ok) return M_RVEC;
  return M_SCALAR;
}

}  // namespace

int tc_gemm_launch(const TcGemm& g0, cudaStream_t st) {
  if (g0.M <= 0 || g0.N <= 0 || g0.batch <= 0) return ATLAS_OK;
  TcGemm g = g0;
  if (g.symmetric && (g.M != TB || g.N != TB)) return ATLAS_ERR_UNSUPPORTED;
  const int nsplit = g.ksplit > 1 ? g.ksplit : 1;
  if (nsplit > 1 && (g.D || g.sCn != 1 || g.emul || g.epi)) return ATLAS_ERR_UNSUPPORTED;
  g.modeA = pick_mode(g.A, g.sAm, g.sAk, g.sAb, g.sAb2, g.batch);
  g.modeB = pick_mode(g.B, g.sBn, g.sBk, g.sBb, g.sBb2, g.batch);
  // a per-k factor is applied elementwise: the vector paths handle it too
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_G) != cudaSuccess)
      return ATLAS_ERR_CUDA;
    attr_set = true;
  }
  dim3 grid((g.N + TB - 1) / TB, (g.M + TB - 1) / TB, g.batch * nsplit);
  tc_gemm_kernel<<<grid, kThr, SMEM_G, st>>>(g);
  return cudaGetLastError() == cudaSuccess ? ATLAS_OK : ATLAS_ERR_CUDA;
}

}  // namespace atlas
