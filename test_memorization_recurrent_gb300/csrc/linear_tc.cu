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
// With s_n = prod_{l=n+1..63} (1 - alpha_l), W[n,i] = gamma_0 theta_i s_i / s_n for
// i <= n (s_i / s_n is the product over l = i+1..n), so both the state update and the
// intra-chunk readout use the same weighted errors Ew_i = gamma_0 theta_i s_i e_i:
//   M_end = a_63 M0 - 2 Ew^T Phi,   y_n = a_n (M0 q_n) + sum_{i<=n} (-2 q_n.k_i / s_n) Ew_i.
// A chunk whose s_0 falls below 1e-30 (a decay gate at or near 1), or whose
// eta has a non-zero entry (momentum), is not handled here: the head is flagged
// and recomputed from scratch by the CUDA-core kernel.
//
// Products per chunk, with the value index v on the TMEM lanes (fp32 accumulators):
//   [Qy | T]   = M0 [Q; Phi]^T           (128 x 128)  T -> Ew^T = s.theta.(T - V^T)
//   QP         = [Phi; Phi] Q^T, rows i, 64+i: k_i . q_n -> P'' = -2 [i<=n] k_i.q_n / s_n
//   [dM | Yi]  = Ew^T [Phi | P'']        (128 x 192)  one MMA chain for both
//   y^T        = a_n Qy + Yi,            M_end = a_63 M0 - 2 dM
// M0 and Ew are A operands held in TMEM (bf16 hi + lo halves, x = hi + lo to
// ~2^-16); Phi, Q (bf16, exact) come from shared memory by TMA; P'' is split
// the same way into shared memory.  The fp32 master state M lives in the
// registers of the epilogue warps (thread = row v, 64 columns).  Y leaves
// through a shared-memory tile and one TMA store per chunk.
//
// Warp roles (320 threads): warp 0 issues TMA loads two chunks deep; warp 1
// builds the gate tables (warp-wide scans) and issues every MMA from one
// thread; warps 2..9 are the epilogue, two per 32-lane TMEM quadrant.
//
// The CUDA-core kernel is launched right after this one: this kernel writes
// one flag per head to the workspace and that kernel takes exactly the flagged
// heads.  Every
// mbarrier wait is bounded; on expiry the kernel records ATLAS_ERR_TIMEOUT in
// the status word, drains its in-flight copies and MMAs, frees TMEM and returns.
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

constexpr int kThreads = 352;
constexpr int kTablesWarp = 10;
constexpr int kChunk = 64;
constexpr int kDim = 128;
constexpr long long kWaitLimit = 2000000000LL;  // clock cycles (~1 s)
constexpr float kMinSuffix = 1e-30f;            // smallest s_0 handled here

// Test builds only: with ATLAS_TEST_WITHHOLD_LOADS defined, the producer of
// head 0 never issues the loads of chunk 1, so the consumers' bounded wait on
// that stage runs out and the abort path (status word, drain, TMEM release)
// runs.  Every access stays in bounds and every wait still ends.  The library
// the package builds never defines it.
#ifdef ATLAS_TEST_WITHHOLD_LOADS
constexpr bool kWithholdChunk1OfHead0 = true;
#else
constexpr bool kWithholdChunk1OfHead0 = false;
#endif

// shared-memory map (bytes from a 1024-aligned base)
//   stage, per 64-feature half kb (KB_STRIDE apart): Q | Phi | Phi again (8 KB
//   each, 128B-swizzled, loaded by TMA; [Q; Phi] is the state product's B
//   operand, [Phi; Phi] the M = 128 A operand of QP, which so puts the k.q block
//   in both lane halves) | P''hi | P''lo ([i][n], 128B-swizzled, written by the
//   epilogue) | V (64 x 128 bf16, row-major) | alpha | eta | theta
constexpr uint32_t KB_STRIDE = 24576;
constexpr uint32_t ST_K = 8192;                      // Phi kb0 (kb1 at + KB_STRIDE)
constexpr uint32_t ST_PHI = ST_K + 2 * KB_STRIDE;    // third MN-major atom after Phi kb0, kb1
constexpr uint32_t ST_PLO = ST_PHI + 8192;
constexpr uint32_t ST_V = ST_PLO + 8192;
constexpr uint32_t ST_GATES = ST_V + 16384;
constexpr uint32_t STAGE_BYTES = ST_GATES + 1024;  // 91136 = 89 x 1024
constexpr int kStages = 2;
constexpr uint32_t OFF_STAGE0 = 0;
constexpr uint32_t OFF_Y = kStages * STAGE_BYTES;     // y tile [64 n][128 v] fp32, 32 KB
constexpr uint32_t OFF_TAB = OFF_Y + 32768;
constexpr uint32_t TAB_FLOATS = 3 * kChunk;           // a, wb, cn
constexpr uint32_t OFF_ELAST = OFF_TAB + 2 * TAB_FLOATS * 4;
constexpr uint32_t OFF_BARS = OFF_ELAST + kDim * 4;
constexpr uint32_t SMEM_USED = OFF_BARS + 256;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;    // alignment slack

constexpr uint32_t STAGE_TX = 6 * 8192 + 16384 + 3 * 256;  // with the gates (N % 4 == 0)
constexpr uint32_t STAGE_TX_NOGATES = 6 * 8192 + 16384;

// TMEM columns
constexpr uint32_t TM_QY = 0;      // [Qy | T]            (128)
constexpr uint32_t TM_T = 64;
constexpr uint32_t TM_QP = 128;    // k_i . q_n (64 queries), token i in lanes i and 64 + i
constexpr uint32_t TM_DM = 192;    // [dM | Yi]           (192)
constexpr uint32_t TM_YI = 320;
constexpr uint32_t TM_MHI = 384;   // A operand M0: hi (64 cols = 128 bf16), lo
constexpr uint32_t TM_MLO = 448;
constexpr uint32_t TM_EWHI = 384;  // A operand Ew (reuses the M0 columns once T is done)
constexpr uint32_t TM_EWLO = 416;
constexpr uint32_t TM_COLS = 512;

enum Bar {
  B_FULL0 = 0, B_FULL1, B_EMPTY0, B_EMPTY1, B_QP, B_D1, B_DM, B_E, B_P, B_M, B_TAB0, B_TAB1,
  B_TFREE0, B_TFREE1, B_S, B_DRAIN, B_YS, B_YF, B_COUNT
};

// abort_flag values
constexpr int kRun = 0, kTimeout = 1, kHandOff = 2;

struct TcParams {
  const __nv_bfloat16* K;
  const float* alpha;
  const float* eta;
  const float* theta;
  const float* gamma;
  float* Y;
  float* M;
  float* S;     // optional
  int* status;  // optional
  int* flags;   // [heads]: 1 = left to the CUDA-core kernel
  int N;
  int gate_tma;  // gates loaded by TMA (N % 4 == 0, aligned rows), else with plain loads
  int lk;        // attentional bias (ATLAS_LOSS_L2, _LP or _HUBER)
  float lp;      // its parameter
};

struct TcMaps {
  CUtensorMap k, q, v, alpha, eta, theta, y;
};

__device__ __forceinline__ float* table(unsigned char* sm, int buf) {
  return reinterpret_cast<float*>(sm + OFF_TAB) + buf * TAB_FLOATS;
}

// Split 8 fp32 values x = hi + lo into two bf16x8 chunks: hi keeps the top 16
// bits (truncation), lo = rn(x - hi), so |x - hi - lo| <= 2^-16 |x|.
__device__ __forceinline__ void split8(const float* x, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t a = __float_as_uint(x[2 * p]), b = __float_as_uint(x[2 * p + 1]);
    h[p] = __byte_perm(a, b, 0x7632);  // top halves of a (low) and b (high)
    const float ra = x[2 * p] - __uint_as_float(a & 0xFFFF0000u);
    const float rb = x[2 * p + 1] - __uint_as_float(b & 0xFFFF0000u);
    const __nv_bfloat162 r = __floats2bfloat162_rn(ra, rb);
    l[p] = *reinterpret_cast<const uint32_t*>(&r);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void st_shared_u4(uint32_t addr, const uint4& v) {
  st_shared_v4(addr, v.x, v.y, v.z, v.w);
}

// Load 16 consecutive fp32 columns of this thread's lane (load and wait in one
// statement, like tmem_ld32).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Pack 32 fp32 values into hi / lo bf16 pairs (element 2c in the low half of
// column c), the TMEM A-operand layout.
__device__ __forceinline__ void pack_split32(const float* x, uint32_t* hi, uint32_t* lo) {
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const uint32_t a = __float_as_uint(x[2 * c]), b = __float_as_uint(x[2 * c + 1]);
    hi[c] = __byte_perm(a, b, 0x7632);
    const __nv_bfloat162 r = __floats2bfloat162_rn(x[2 * c] - __uint_as_float(a & 0xFFFF0000u),
                                                   x[2 * c + 1] - __uint_as_float(b & 0xFFFF0000u));
    lo[c] = *reinterpret_cast<const uint32_t*>(&r);
  }
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

  // the next launch (the CUDA-core kernel for handed-off heads) may be scheduled
  // now: it waits for this grid's completion before it reads anything
  pdl_launch_dependents();
  if (nchunks == 0) {
    pdl_wait();
    if (tid == 0) p.flags[head] = 0;
    return;
  }

  if (tid == 0) {
    for (int b = 0; b < B_COUNT; ++b) {
      uint32_t cnt = 1;
      if (b == B_P || b == B_E || b == B_M || b == B_S || b == B_YS || b == B_TFREE0 ||
          b == B_TFREE1)
        cnt = 8;
      mbar_init(&bars[b], cnt);
    }
    *abort_flag = kRun;
    fence_barrier_init();
    prefetch_tmap(&maps.k);
    prefetch_tmap(&maps.q);
    prefetch_tmap(&maps.v);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TM_COLS);
    tmem_relinquish();
  }
  // the set-up above touched only on-chip state; the preceding launch's outputs
  // (inputs, state, flags of this call) are complete from here
  pdl_wait();
  // the head is this kernel's unless a chunk hands it off (momentum, reset gate)
  if (tid == 0) p.flags[head] = 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_u32(sm);

  auto timeout = [&]() {
    if (*abort_flag == kRun) {
      *abort_flag = kTimeout;
      if (p.status) atomicExch(p.status, ATLAS_ERR_TIMEOUT);
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < nchunks; ++j) {
        const int s = j % kStages;
        if (j >= kStages &&
            !mbar_wait(&bars[B_EMPTY0 + s], ((j - kStages) / kStages) & 1, abort_flag, kWaitLimit)) {
          timeout();
          break;
        }
        if (kWithholdChunk1OfHead0 && head == 0 && j == 1) continue;  // test builds only
        unsigned char* st = sm + OFF_STAGE0 + s * STAGE_BYTES;
        uint64_t* fb = &bars[B_FULL0 + s];
        mbar_arrive_expect_tx(fb, p.gate_tma ? STAGE_TX : STAGE_TX_NOGATES);
        const int t0 = j * kChunk;
        for (int kb = 0; kb < 2; ++kb) {
          unsigned char* sk = st + kb * KB_STRIDE;
          tma_load_3d(sk, &maps.q, fb, 64 * kb, t0, head);
          tma_load_3d(sk + 8192, &maps.k, fb, 64 * kb, t0, head);
          tma_load_3d(sk + 16384, &maps.k, fb, 64 * kb, t0, head);
        }
        tma_load_3d(st + ST_V, &maps.v, fb, 0, t0, head);
        if (p.gate_tma) {  // gate rows of N floats start 16-byte aligned
          tma_load_2d(st + ST_GATES, &maps.alpha, fb, t0, head);
          tma_load_2d(st + ST_GATES + 256, &maps.eta, fb, t0, head);
          tma_load_2d(st + ST_GATES + 512, &maps.theta, fb, t0, head);
        }
        issued = j + 1;
      }
      // drain: every issued load must land before shared memory is released
      for (int j = issued - kStages < 0 ? 0 : issued - kStages; j < issued; ++j) {
        volatile int zero = 0;
        mbar_wait(&bars[B_FULL0 + j % kStages], (j / kStages) & 1, &zero, kWaitLimit);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    // descriptor constants: address bits are added per use
    const uint64_t dK = sdesc_sw128(0, 16, 1024);       // K-major, 128-byte rows
    const uint64_t dMN = sdesc_sw128(0, KB_STRIDE, 1024);  // MN-major, atoms KB_STRIDE apart
    constexpr uint32_t kId128 = idesc_bf16(128, 128, false, false);
    constexpr uint32_t kId64 = idesc_bf16(128, 64, false, false);
    constexpr uint32_t kId192mn = idesc_bf16(128, 192, false, true);
    constexpr uint32_t kId64mn = idesc_bf16(128, 64, false, true);
    // QP = [Phi; Phi] Q^T: rows i and 64 + i both hold k_i . q_n for the 64
    // queries, so every TMEM lane quadrant can read the block for its tokens
    auto issue_qp = [&](int j) {
      const uint32_t st = sbase + OFF_STAGE0 + (j % kStages) * STAGE_BYTES;
      const uint64_t dst = dK | (uint64_t)((st >> 4) & 0x3FFFu);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t off = (k >> 2) * KB_STRIDE + (k & 3) * 32;
        mma_bf16(tmem + TM_QP, dst + ((off + ST_K) >> 4), dst + (off >> 4), kId64, k > 0);
      }
      mma_commit(&bars[B_QP]);
    };
    // tables(0) published: its stage has landed
    bool ok = mbar_wait(&bars[B_TAB0], 0, abort_flag, kWaitLimit);
    if (ok && lane == 0) issue_qp(0);
    __syncwarp();
    for (int j = 0; ok && j < nchunks; ++j) {
      const int s = j % kStages;
      const uint32_t st = sbase + OFF_STAGE0 + s * STAGE_BYTES;
      // M0 in TMEM and the previous chunk's [Qy | T] read out
      if (!mbar_wait(&bars[B_M], j & 1, abort_flag, kWaitLimit)) { ok = false; break; }
      tc_fence_after();
      if (lane == 0) {  // [Qy | T] = M0 [Q; Phi]^T; hi then lo halves of M0
        const uint64_t dst = dK | (uint64_t)((st >> 4) & 0x3FFFu);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint32_t am = tmem + (k < 8 ? TM_MHI : TM_MLO) + 8 * (k & 7);
          const uint32_t off = ((k & 7) >> 2) * KB_STRIDE + (k & 3) * 32;
          mma_bf16_ta(tmem + TM_QY, am, dst + (off >> 4), kId128, k > 0);  // [Qy | T]
        }
        mma_commit(&bars[B_D1]);
      }
      __syncwarp();
      if (!mbar_wait(&bars[B_E], j & 1, abort_flag, kWaitLimit)) { ok = false; break; }
      if (!mbar_wait(&bars[B_P], j & 1, abort_flag, kWaitLimit)) { ok = false; break; }
      tc_fence_after();
      if (lane == 0) {
        // [dM | Yi] = Ew^T [Phi | P''hi] (Ew hi, then lo), then Yi += Ew_hi^T P''lo
        const uint64_t dph = dMN | (uint64_t)(((st + ST_K) >> 4) & 0x3FFFu);
        const uint64_t dpl = dMN | (uint64_t)(((st + ST_PLO) >> 4) & 0x3FFFu);
#pragma unroll
        for (int k = 0; k < 12; ++k) {
          const uint32_t ae = tmem + ((k >> 2) == 1 ? TM_EWLO : TM_EWHI) + 8 * (k & 3);
          const uint64_t b = ((k >> 2) == 2 ? dpl : dph) + (((k & 3) * 2048) >> 4);
          if (k < 8)
            mma_bf16_ta(tmem + TM_DM, ae, b, kId192mn, k > 0);
          else
            mma_bf16_ta(tmem + TM_YI, ae, b, kId64mn, 1);
        }
        mma_commit(&bars[B_DM]);
        mma_commit(&bars[B_EMPTY0 + s]);
      }
      __syncwarp();
      // the next chunk's QP once its tables (and so its stage) are in place; the
      // P-epilogue of j is done, so its QP was read
      if (j + 1 < nchunks) {
        if (!mbar_wait(&bars[B_TAB0 + ((j + 1) & 1)], ((j + 1) >> 1) & 1, abort_flag,
                       kWaitLimit)) { ok = false; break; }
        if (lane == 0) issue_qp(j + 1);
        __syncwarp();
      }
    }
    if (!ok) timeout();
    if (lane == 0) {
      // no MMA may outlive the TMEM: wait for everything this thread issued
      volatile int zero = 0;
      mma_commit(&bars[B_DRAIN]);
      mbar_wait(&bars[B_DRAIN], 0, &zero, kWaitLimit);
    }
    __syncwarp();
  } else if (warp == kTablesWarp) {
    // -------------------------------------------------------- gate tables
    const float g0 = p.gamma[0];
    // Gate tables of chunk j (warp-wide scans, lane l owns tokens 2l, 2l+1):
    // a_n = prod_{l<=n}(1-alpha_l), wb_i = gamma_0 theta_i s_i, cn_n = -2 / s_n.
    // Returns false on a timeout, or if s_0 is too small (hand the head off).
    auto tables = [&](int j) -> bool {
      const int s = j % kStages;
      if (!mbar_wait(&bars[B_FULL0 + s], (j / kStages) & 1, abort_flag, kWaitLimit)) {
        timeout();
        return false;
      }
      float* ga = reinterpret_cast<float*>(sm + OFF_STAGE0 + s * STAGE_BYTES + ST_GATES);
      float* ge = ga + 64;
      float* gt = ga + 128;
      if (!p.gate_tma) {  // plain loads into the stage (zero past the end, as TMA fills)
        const long gb = (long)head * N + (long)j * kChunk;
        const int nb = min(kChunk, N - j * kChunk);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int n = 2 * lane + x;
          ga[n] = n < nb ? p.alpha[gb + n] : 0.f;
          ge[n] = n < nb ? p.eta[gb + n] : 0.f;
          gt[n] = n < nb ? p.theta[gb + n] : 0.f;
        }
        __syncwarp();
      }
      float* tb = table(sm, j & 1);
      float *a = tb, *wb = tb + kChunk, *cn = tb + 2 * kChunk;
      const unsigned full = 0xFFFFFFFFu;
      const int n0 = 2 * lane, n1 = n0 + 1;
      const float k0 = 1.f - ga[n0], k1 = 1.f - ga[n1];
      float pa = k0 * k1;  // inclusive prefix product over lanes
      float sf = pa;       // inclusive suffix product over lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float ua = __shfl_up_sync(full, pa, o);
        const float ds = __shfl_down_sync(full, sf, o);
        if (lane >= o) pa *= ua;
        if (lane + o < 32) sf *= ds;
      }
      float ea = __shfl_up_sync(full, pa, 1);    // product over tokens < n0
      float es = __shfl_down_sync(full, sf, 1);  // product over tokens > n1 (= s_{n1})
      if (lane == 0) ea = 1.f;
      if (lane == 31) es = 1.f;
      const float s1 = es, s0 = es * k1;          // s_{n1}, s_{n0}
      a[n0] = ea * k0;
      a[n1] = ea * k0 * k1;
      wb[n0] = gt[n0] * g0 * s0;
      wb[n1] = gt[n1] * g0 * s1;
      cn[n0] = -2.f / s0;
      cn[n1] = -2.f / s1;
      const bool handled = __shfl_sync(full, s0, 0) >= kMinSuffix &&  // s_0 is the smallest
                           !__any_sync(full, ge[n0] != 0.f || ge[n1] != 0.f);
      __syncwarp();
      if (!handled) {
        if (lane == 0 && *abort_flag == kRun) {
          *abort_flag = kHandOff;
          p.flags[head] = 1;
        }
        return false;
      }
      if (lane == 0) mbar_arrive(&bars[B_TAB0 + (j & 1)]);
      return true;
    };
    // chunk j's tables go into buffer j & 1 once the epilogue is done with
    // chunk j - 2's (B_TFREE); the MMA issuer and the epilogue wait on B_TAB
    for (int j = 0; j < nchunks; ++j) {
      if (j >= 2 && !mbar_wait(&bars[B_TFREE0 + (j & 1)], ((j - 2) >> 1) & 1, abort_flag,
                               kWaitLimit)) {
        timeout();
        break;
      }
      if (!tables(j)) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;             // TMEM lane quadrant
    const int h = (warp - 2) >> 2;      // half: columns / tokens / queries
    const int v = 32 * q + lane;        // TMEM lane = value index v (or token i)
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
    const bool elected = warp == 2 && lane == 0;
    float m[64];                        // M0[v][64h .. 64h+63]
    {
      const float4* src = reinterpret_cast<const float4*>(p.M + ((long)head * kDim + v) * kDim + 64 * h);
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const float4 t = src[x];
        m[4 * x] = t.x; m[4 * x + 1] = t.y; m[4 * x + 2] = t.z; m[4 * x + 3] = t.w;
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t hi[16], lo[16];
        pack_split32(m + 32 * cc, hi, lo);
        tmem_st16(tl + TM_MHI + 32 * h + 16 * cc, hi);
        tmem_st16(tl + TM_MLO + 32 * h + 16 * cc, lo);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_M]);
    }
    bool ok = true;
    for (int j = 0; j < nchunks; ++j) {
      const int t0 = j * kChunk;
      const uint32_t par = j & 1;
      unsigned char* stg = sm + OFF_STAGE0 + (j % kStages) * STAGE_BYTES;
      if (!mbar_wait(&bars[B_TAB0 + (j & 1)], (j >> 1) & 1, abort_flag, kWaitLimit)) { ok = false; break; }
      const float* tb = table(sm, j & 1);
      const float *ta = tb, *twb = tb + kChunk, *tcn = tb + 2 * kChunk;
      // V^T[v][i] of this thread's tokens, read before the products are done
      float vt[32];
      {
        const __nv_bfloat16* Vs = reinterpret_cast<const __nv_bfloat16*>(stg + ST_V);
#pragma unroll
        for (int x = 0; x < 32; ++x) vt[x] = __bfloat162float(Vs[(32 * h + x) * kDim + v]);
      }
      {
        // ---- P''[i][n] = -2 [i <= n] (k_i . q_n) / s_n for token i and 16 queries:
        // the low lane quadrants take the queries n < 32, the high ones n >= 32
        const int i = 32 * (q & 1) + lane;
        const int n0 = (q >= 2 ? 32 : 0) + 16 * h;
        if (!mbar_wait(&bars[B_QP], par, abort_flag, kWaitLimit)) { ok = false; break; }
        tc_fence_after();
        float pv[16];
        tmem_ld16(tl + TM_QP + n0, pv);  // column = query: n0 .. n0 + 15
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const float4 c4 = reinterpret_cast<const float4*>(tcn + n0)[x];
          const int n = n0 + 4 * x;
          pv[4 * x] = n >= i ? c4.x * pv[4 * x] : 0.f;
          pv[4 * x + 1] = n + 1 >= i ? c4.y * pv[4 * x + 1] : 0.f;
          pv[4 * x + 2] = n + 2 >= i ? c4.z * pv[4 * x + 2] : 0.f;
          pv[4 * x + 3] = n + 3 >= i ? c4.w * pv[4 * x + 3] : 0.f;
        }
        const uint32_t ph = smem_u32(stg + ST_PHI), pl = smem_u32(stg + ST_PLO);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint4 hi, lo;
          split8(pv + 8 * c, hi, lo);
          const uint32_t o = sw128_offset(i, n0 / 8 + c);
          st_shared_u4(ph + o, hi);
          st_shared_u4(pl + o, lo);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_P]);
      }
      if (!mbar_wait(&bars[B_D1], par, abort_flag, kWaitLimit)) { ok = false; break; }
      tc_fence_after();
      {
        // ---- Ew^T[v][i] = wb_i (T[v][i] - V[i][v]) for tokens i in [32h, 32h+32)
        float e[32];
        tmem_ld32(tl + TM_T + 32 * h, e);
#pragma unroll
        for (int x = 0; x < 32; ++x) e[x] -= vt[x];
        if (p.lk == ATLAS_LOSS_HUBER) {  // attentional bias, one loop per kind
#pragma unroll
          for (int x = 0; x < 32; ++x) e[x] = huber_grad(e[x], p.lp);
        } else if (p.lk == ATLAS_LOSS_LP) {
#pragma unroll
          for (int x = 0; x < 32; ++x) e[x] = lp_grad(e[x], p.lp);
        }
        if (p.S && j == nchunks - 1) {
          const int il = N - 1 - t0 - 32 * h;
          if (il >= 0 && il < 32) {
            float* el = reinterpret_cast<float*>(sm + OFF_ELAST);
#pragma unroll
            for (int x = 0; x < 32; ++x)
              if (x == il) el[v] = e[x];
          }
        }
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const float4 w4 = reinterpret_cast<const float4*>(twb + 32 * h)[x];
          e[4 * x] *= w4.x; e[4 * x + 1] *= w4.y; e[4 * x + 2] *= w4.z; e[4 * x + 3] *= w4.w;
        }
        uint32_t hi[16], lo[16];
        pack_split32(e, hi, lo);
        tmem_st16(tl + TM_EWHI + 16 * h, hi);
        tmem_st16(tl + TM_EWLO + 16 * h, lo);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_E]);
      }
      // ---- [dM | Yi] done: readout first (frees [Qy | T]), then the state update
      if (!mbar_wait(&bars[B_DM], par, abort_flag, kWaitLimit)) { ok = false; break; }
      tc_fence_after();
      {
        if (elected) {  // the previous chunk's store has finished reading the tile
          bulk_wait_read0();
          mbar_arrive(&bars[B_YF]);
        }
        float y[32], yi[32];
        tmem_ld32(tl + TM_QY + 32 * h, y);
        tmem_ld32(tl + TM_YI + 32 * h, yi);
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const float4 a4 = reinterpret_cast<const float4*>(ta + 32 * h)[x];
          y[4 * x] = a4.x * y[4 * x] + yi[4 * x];
          y[4 * x + 1] = a4.y * y[4 * x + 1] + yi[4 * x + 1];
          y[4 * x + 2] = a4.z * y[4 * x + 2] + yi[4 * x + 2];
          y[4 * x + 3] = a4.w * y[4 * x + 3] + yi[4 * x + 3];
        }
        if (!mbar_wait(&bars[B_YF], par, abort_flag, kWaitLimit)) { ok = false; break; }
        float* yt = reinterpret_cast<float*>(sm + OFF_Y) + 32 * h * kDim + v;
#pragma unroll
        for (int x = 0; x < 32; ++x) yt[x * kDim] = y[x];
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_YS]);
      }
      {
        const float ab = ta[kChunk - 1];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float dm[32];
          tmem_ld32(tl + TM_DM + 64 * h + 32 * cc, dm);
#pragma unroll
          for (int x = 0; x < 32; ++x) m[32 * cc + x] = ab * m[32 * cc + x] - 2.f * dm[x];
          uint32_t hi[16], lo[16];
          pack_split32(m + 32 * cc, hi, lo);
          tmem_st16(tl + TM_MHI + 32 * h + 16 * cc, hi);
          tmem_st16(tl + TM_MLO + 32 * h + 16 * cc, lo);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars[B_M]);
          mbar_arrive(&bars[B_TFREE0 + (j & 1)]);  // table j is no longer read
        }
      }
      if (elected) {
        if (!mbar_wait(&bars[B_YS], par, abort_flag, kWaitLimit)) { ok = false; break; }
        tma_store_3d(&maps.y, sm + OFF_Y, 0, t0, head);  // rows past N are clipped
        bulk_commit();
      }
    }
    if (!ok && *abort_flag != kHandOff) timeout();
    if (elected) bulk_wait0();  // Y stores complete before exit
    const bool done = *abort_flag == kRun;
    if (done) {
      float4* dst = reinterpret_cast<float4*>(p.M + ((long)head * kDim + v) * kDim + 64 * h);
#pragma unroll
      for (int x = 0; x < 16; ++x) dst[x] = make_float4(m[4 * x], m[4 * x + 1], m[4 * x + 2], m[4 * x + 3]);
    }
    if (p.S && done) {
      // eta = 0: the final momentum is S_N = -gamma_0 theta_{N-1} 2 e_{N-1} k_{N-1}^T
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_S]);
      if (mbar_wait(&bars[B_S], 0, abort_flag, kWaitLimit)) {
        const float* el = reinterpret_cast<const float*>(sm + OFF_ELAST);
        const float coef = -2.f * p.gamma[0] * p.theta[(long)head * N + N - 1] * el[v];
        const __nv_bfloat16* kl = p.K + ((long)head * N + N - 1) * kDim + 64 * h;
        float* dst = p.S + ((long)head * kDim + v) * kDim + 64 * h;
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

// [heads, N, 128] bf16, boxes of 64 tokens x `cols` features.
bool make_map_tokens(CUtensorMap* m, const void* base, int N, int heads, int cols, bool swz) {
  cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)N, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)kDim * 2, (cuuint64_t)N * kDim * 2};
  cuuint32_t box[3] = {(cuuint32_t)cols, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
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

// [heads, N, 128] fp32 outputs, boxes of 64 tokens x 128 values.
bool make_map_y(CUtensorMap* m, float* base, int N, int heads) {
  cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)N, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)kDim * 4, (cuuint64_t)N * kDim * 4};
  cuuint32_t box[3] = {(cuuint32_t)kDim, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

bool linear_tc_supported(const LinArgs& a) {
  return a.d_k == kDim && a.d_v == kDim && a.D == kDim && a.b == kChunk && a.c == 1 && !a.poly &&
         !a.pgen && a.ret == ATLAS_RET_L2 && a.lk != ATLAS_LOSS_ROBUST &&
         !a.dot && a.bf16 && a.N > 0;
}

size_t linear_tc_workspace_bytes(int heads) { return (size_t)heads * sizeof(int); }

int linear_tc_launch(const LinArgs& a, int heads, int* status, void* workspace, cudaStream_t st) {
  if (!linear_tc_supported(a)) return ATLAS_ERR_UNSUPPORTED;
  if (!aligned16(a.K) || !aligned16(a.Q) || !aligned16(a.V) || !aligned16(a.Y) ||
      !aligned16(a.M) || (a.S && !aligned16(a.S)))
    return ATLAS_ERR_UNSUPPORTED;
  if (!workspace) return ATLAS_ERR_WORKSPACE;
  if (!encoder()) return ATLAS_ERR_CUDA;
  TcMaps maps;
  if (!make_map_tokens(&maps.k, a.K, a.N, heads, 64, true) ||
      !make_map_tokens(&maps.q, a.Q, a.N, heads, 64, true) ||
      !make_map_tokens(&maps.v, a.V, a.N, heads, 128, false) ||
      !make_map_y(&maps.y, a.Y, a.N, heads))
    return ATLAS_ERR_CUDA;
  const bool gate_tma =
      (a.N % 4) == 0 && aligned16(a.alpha) && aligned16(a.eta) && aligned16(a.theta);
  memset(&maps.alpha, 0, sizeof(maps.alpha));
  memset(&maps.eta, 0, sizeof(maps.eta));
  memset(&maps.theta, 0, sizeof(maps.theta));
  if (gate_tma && (!make_map_gate(&maps.alpha, a.alpha, a.N, heads) ||
                   !make_map_gate(&maps.eta, a.eta, a.N, heads) ||
                   !make_map_gate(&maps.theta, a.theta, a.N, heads)))
    return ATLAS_ERR_CUDA;
  TcParams p;
  p.K = reinterpret_cast<const __nv_bfloat16*>(a.K);
  p.alpha = a.alpha;
  p.eta = a.eta;
  p.theta = a.theta;
  p.gamma = a.gamma;
  p.Y = a.Y;
  p.M = a.M;
  p.S = a.S;
  p.status = status;
  p.flags = reinterpret_cast<int*>(workspace);
  p.N = a.N;
  p.gate_tma = gate_tma ? 1 : 0;
  p.lk = a.lk;
  p.lp = a.lp;
  if (cudaFuncSetAttribute(linear_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)SMEM_ALLOC) != cudaSuccess)
    return ATLAS_ERR_CUDA;
  // launched with programmatic stream serialisation: its launch and set-up overlap
  // the tail of the preceding kernel, and it waits for that kernel before any
  // global access
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(heads);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SMEM_ALLOC;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, linear_tc_kernel, maps, p) != cudaSuccess ||
      cudaGetLastError() != cudaSuccess)
    return ATLAS_ERR_CUDA;
  // heads with a non-zero eta: the CUDA-core kernel takes exactly the flagged ones
  return linear_simt_launch_flagged(a, heads, p.flags, st);
}

}  // namespace atlas
