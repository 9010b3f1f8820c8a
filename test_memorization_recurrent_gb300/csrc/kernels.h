// kernels.h -- internal interface between the C-ABI host layer and the kernels.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

namespace atlas {

// Arguments of every linear-memory kernel (one head = one [N, .] slice).
struct LinArgs {
  const void* K;
  const void* Q;
  const void* V;
  const float* alpha;
  const float* eta;
  const float* theta;
  const float* gamma;
  float* Y;
  float* M;  // [heads, d_v, D] in/out
  float* S;  // [heads, d_v, D] in/out, or nullptr (start at zero, not returned)
  int N, d_k, d_v, D, c, b;
  int poly, dot, bf16;
  int lk;    // attentional bias: 0 l2, 1 dot, 2 l_p, 3 Huber, 4 robust (ATLAS_LOSS_*)
  float lp;  // its parameter (p, delta)
  int nh;  // history rows ahead of token 0 in K and V (head stride (nh + N) rows)
  int pgen;        // gated polynomial map of degree pdeg (poly is 0 then)
  int pdeg;
  float pcoef[5];  // a_0 .. a_pdeg
  int ret;         // retention gate (ATLAS_RET_*)
  float rp;        // its parameter (lambda, c, q)
};

int linear_simt_launch(const LinArgs& a, int heads, cudaStream_t st);
// Same kernel, restricted to the heads whose flag (device int per head) is set.
int linear_simt_launch_flagged(const LinArgs& a, int heads, const int* flags, cudaStream_t st);
int linear_simt_plan(const LinArgs& a, int heads, int* RV_out, size_t* smem_out);

// Token-serial path for small linear memories (identity map, d_k = 32,
// window c <= 8, any chunk length): state in registers, rows split over CTAs.
bool linear_seq_supported(const LinArgs& a);
int linear_seq_launch(const LinArgs& a, int heads, cudaStream_t st);

// Fused path for linear memories with a wide feature map (D >= 256): one
// thread-block cluster per head, feature columns split over its CTAs.
bool linear_wide_supported(const LinArgs& a, int heads);
int linear_wide_launch(const LinArgs& a, int heads, cudaStream_t st);

// Host-driven path for linear memories with a wide feature map (D >= 256, the
// degree-2 map): per chunk, batched tensor-core GEMMs over all heads.
bool linear_chunk_supported(const LinArgs& a);
size_t linear_chunk_workspace_bytes(const LinArgs& a, int heads);
long linear_chunk_launch_count(const LinArgs& a, int heads);
int linear_chunk_forward(const LinArgs& a, int heads, void* ws, cudaStream_t st);

// Tensor-core path: linear memory, identity map, d_k = d_v = 128, bf16 inputs,
// b = 64, c = 1, N % 4 == 0.  Launches the tensor-core kernel (heads with
// eta == 0; it flags the others in the workspace) and the CUDA-core kernel on
// the flagged heads.  Workspace: one int per head.
bool linear_tc_supported(const LinArgs& a);
size_t linear_tc_workspace_bytes(int heads);
int linear_tc_launch(const LinArgs& a, int heads, int* status, void* workspace, cudaStream_t st);

// Backward pass (linear_bwd.cu): identity map, d_k = d_v = 128, b = 64, c = 1,
// eta = 0 in the forward, no history rows, no momentum state in or out.
// Three launches; the workspace holds the chunk-start states, the gate tables
// and the per-row-block partial sums.
bool linear_bwd_supported(const LinArgs& a);
size_t linear_bwd_workspace_bytes(const LinArgs& a, int heads);
int linear_bwd_launch(const LinArgs& a, int heads, const float* M0, const float* dY, float* dM,
                      float* dK, float* dQ, float* dV, float* dalpha, float* deta, float* dtheta,
                      int* status, void* ws, cudaStream_t st);

// Batched strided GEMM on fp32 operands (tc_gemm.cu, tensor cores with bf16
// hi/lo operand splitting), used by the MLP-memory path:
//   C[b](m,n) = alpha rowscale[b](m) sum_k A[b](m,k) kscale[b](k) B[b](k,n) + beta D[b](m,n)
//               (+ C[b](m,n) when accumulate is set)
// Batch index b splits as (b / bdiv, b % bdiv) when bdiv > 0; every batched
// pointer then moves by s?b per outer and s?b2 per inner step (bdiv = 0: only
// the outer strides, over b).  symmetric: B(k, n) = A(n, k) and M = N = 128
// (a Gram tile): the operand is staged once and serves both sides.
struct TcGemm {
  int M, N, K, batch, bdiv;
  const float* A; long sAb, sAb2, sAm, sAk;
  const float* B; long sBb, sBb2, sBk, sBn;
  float* C; long sCb, sCb2, sCm, sCn;
  float alpha;
  const float* rowscale; long sRb, sRb2;    // optional per-row factor of the product
  const float* kscale; long sKb, sKb2;      // optional per-k factor of A
  const float* D; long sDb, sDb2, sDm, sDn; // optional addend beta * D
  const float* dscale; long sEb, sEb2;      // optional per-batch factor of the addend
  float beta;
  int accumulate;                           // C += term (else C = term)
  int ksplit;                               // > 1: K split over that many CTAs, their
                                            // terms added to C atomically (no D)
  int symmetric;
  const float* emul; long sMb, sMb2, sMm, sMn;  // optional elementwise factor of the product
  int epi;                                  // 1: C = GELU(pre), C2 = GELU'(pre), pre the
  float* C2; long sC2b, sC2b2, sC2m, sC2n;  // value C would otherwise take
  int* status;                              // optional device status word (timeouts)
  int modeA, modeB;                         // set by tc_gemm_launch (operand load paths)
};

int tc_gemm_launch(const TcGemm& g, cudaStream_t st);

// Arguments of the MLP-memory path.
struct MlpArgs {
  const void* K;
  const void* Q;
  const void* V;
  const float* alpha;
  const float* eta;
  const float* theta;
  const float* gamma;
  float* Y;
  float* M;  // [heads, W1 (d x dh) | W2 (dh x d)] in/out
  float* S;  // same layout, in/out (caller's or workspace)
  int heads, N, d, dh, c, b;
  int nh;  // history rows ahead of token 0 in K and V
  int bf16;
  int lk;    // attentional bias: 0 l2, 2 l_p, 3 Huber, 4 robust (ATLAS_LOSS_*)
  float lp;  // its parameter (p, delta)
  int ns_steps;
  float ns_a, ns_b, ns_c, ns_eps;
  int s_is_zero;  // S must be cleared before the first chunk
  int* status;    // optional device status word (timeouts)
  int ln;         // layer-normalised memory x + LN(W1 GELU(W2 x)) (CUDA-core path only)
  int gated;      // gated memory x + W1 (GELU(W2 x) * (W3 x)), W3 after W2 (CUDA-core path only)
};

size_t mlp_simt_workspace_bytes(const MlpArgs& a);

// Tensor-core path (mlp_tc.cu): d = 128, d_h = 512, c = 1, b = 64, bf16 inputs,
// no Newton-Schulz.  One 4-CTA cluster per head; the workspace holds the W2,
// S2, S1 slices of every head as bf16 hi/lo pairs.
bool mlp_tc_supported(const MlpArgs& a);
size_t mlp_tc_workspace_bytes(const MlpArgs& a);
int mlp_tc_launch(const MlpArgs& a, void* ws, cudaStream_t st);
int mlp_simt_forward(const MlpArgs& a, void* ws, cudaStream_t st);
long mlp_simt_launch_count(const MlpArgs& a);

// Fused Newton-Schulz (ns_fused.cu): n_inst instances, each two blocks of one
// MLP state (W1 part d x dh at X + i * inst_stride, W2 part dh x d at + half),
// every block normalised by its own Frobenius norm and iterated `steps` times
// in place.  Supported for d = 128, dh = 512; X 16-byte aligned.
struct NsArgs {
  float* X;
  long inst_stride, half;
  int n_inst, steps;
  float a, b, c, eps;
  int* status;  // optional device status word (timeouts)
};
bool ns_fused_supported(int d, int dh);
int ns_fused_launch(const NsArgs& a, cudaStream_t st);

}  // namespace atlas
