/*
 * atlas_mem.h -- C ABI of the GB300 test-time memory update library
 * (libatlasmem.so, built for sm_103a).
 *
 * The operation (Titans / Miras / ATLAS family).  For every head, a memory M
 * (a d_v x D matrix over features Phi(k), or a residual MLP
 * M(x) = x + W1 GELU(W2 x)) takes, per token t, one momentum step on the
 * sliding-window ("Omega rule") loss
 *     l_t(M) = sum_{j=0..c-1} gamma[j] * || M(Phi(k_{t-j})) - v_{t-j} ||^2
 *   S_t = eta_t S_{t-1} - theta_t grad l_t,      M_t = (1 - alpha_t) M_{t-1} + S_t
 * (or + NS(S_t), a Newton-Schulz orthogonalised momentum), and is read out as
 *     y_t = M_t(Phi(q_t)).
 * In the chunked form every gradient of the tokens of a chunk of b tokens is
 * taken at the state the previous chunk ended with; b = 1 is the recurrence.
 *
 * Sources (page title, section):
 *   "[Paper Review] Titans 논문 이해하기": Learning Process and Surprise
 *     Metric (S_t), Objective (l2 loss), Forgetting Mechanism (M_t),
 *     Retrieving a Memory (y = M*(q), no update while reading), 3.2 (chunked
 *     mini-batch GD as matmuls).
 *   "논문 리뷰 Google ATLAS": 3.1 (polynomial feature map Phi_p), 3.2 (Omega
 *     rule), 3.3 (chunked Omega rule, gradients at the chunk-start state).
 *   "ATLAS: Learning to Optimally Memorize the Context at Test Time"
 *     (paperlayer summary): 5 Memory Optimization (Muon / Newton-Schulz),
 *     App. E (2-layer residual MLP memory, GELU).
 *   "It's All Connected: ... (Miras)": Associative Memory & Attentional Bias
 *     (dot-product bias = linear attention), #1 Alternative Attentional Biases
 *     (l_p, Huber, robust), #2 Alternative Retention Gates, Training
 *     (chunk-wise parallelisation; the layer outputs M(q_t)).
 *
 * Conventions shared by every entry point:
 *   - All tensor arguments are DEVICE pointers owned by the caller, contiguous,
 *     head-major: index [b][h][token][feature].  The library never frees them.
 *   - Calls only enqueue work on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream) and return without synchronising.
 *   - Argument errors are reported before anything is launched; the output
 *     buffers are then untouched.
 *   - The library allocates no device memory: scratch comes from the
 *     caller's `workspace`.
 */
#ifndef ATLAS_MEM_H
#define ATLAS_MEM_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* memory architecture */
#define ATLAS_MEM_LINEAR 0 /* M: d_v x D matrix, y = M Phi(x) */
#define ATLAS_MEM_MLP 1    /* M(x) = x + W1 GELU(W2 x), d_k = d_v = d */
/* MLP memory variants ("It's All Connected (Miras)": the Moneta / Yaad / Memora
 * memory with LN; paperlayer ATLAS summary §5: the Atlas++ gated MLP), any window,
 * chunk, momentum and Newton-Schulz, on the CUDA-core MLP path: */
#define ATLAS_MEM_MLP_LN 2    /* x + LN(W1 GELU(W2 x)), plain LN over the d outputs (no
                                 scale or shift, variance over d, 1e-5 under the root) */
#define ATLAS_MEM_MLP_GATED 3 /* x + W1 (GELU(W2 x) * (W3 x)), W3 d_h x d after W2; state
                                 and momentum 3 d d_h; Newton-Schulz on all three blocks */
/* feature map (linear memory only; the MLP takes x itself) */
#define ATLAS_PHI_IDENTITY 0 /* D = d_k */
#define ATLAS_PHI_POLY2 1    /* D = d_k + d_k(d_k+1)/2: [x_i] then [x_i x_j, i<=j, i-major] */
/* Gated polynomial map of degree p = cfg->phi_degree ("논문 리뷰 Google ATLAS",
 * §3.1 Polynomial Feature Mapping and Input gating):
 *   Phi(x) = [a_0; a_1 x; a_2 (x_i x_j)_{i<=j}; ...; a_p (degree-p monomials)]
 * with a_e = cfg->phi_coef[e]; each degree's monomials appear once (no
 * multinomial weights), in lexicographic order of their sorted index tuples; a
 * degree whose a_e is 0 is left out, so D = sum over kept e of C(d_k + e - 1, e).
 * a = (0, 1, 1) is ATLAS_PHI_POLY2.  Runs on the CUDA-core linear kernels (the
 * fused cluster kernel once D >= 256 and d_v <= 128); d_k <= 255, D <= 16384. */
#define ATLAS_PHI_POLY 2
#define ATLAS_PHI_MAX_DEGREE 4
/* attentional bias */
#define ATLAS_LOSS_L2 0  /* ||M(Phi(k)) - v||^2 (gradient carries the factor 2) */
#define ATLAS_LOSS_DOT 1 /* -2 <M(Phi(k)), v> (linear memory only: linear attention) */
/* Miras alternative attentional biases ("It's All Connected: ...", #1 Alternative
 * Attentional Biases), e = M(Phi(k)) - v per output coordinate: */
#define ATLAS_LOSS_LP 2    /* sum |e|^p, p = loss_param >= 1 (gradient p |e|^(p-1) sign e) */
#define ATLAS_LOSS_HUBER 3 /* sum e^2 for |e| <= delta, 2 delta |e| - delta^2 beyond, with
                              delta = loss_param > 0 (gradient 2 clamp(e, -delta, delta)) */
/* Robust bias against a value shift of norm at most Delta = loss_param >= 0,
 * read as its worst case (||e|| + Delta)^2 over the whole value vector e:
 * gradient 2 e (1 + Delta / ||e||), 0 at e = 0.  Delta = 0 is ATLAS_LOSS_L2.
 * Couples the d_v coordinates of a token, so the CUDA-core kernels run it (linear
 * memory: a head's row blocks form one thread-block cluster and add their
 * partial norms; wide feature maps: the fused cluster kernel, whose error rows
 * are whole; MLP memories: the CUDA-core MLP path). */
#define ATLAS_LOSS_ROBUST 4
/* Retention gate of the linear memory ("It's All Connected: ... (Miras)", #2
 * Alternative Retention Gates), the map from (M_{t-1}, alpha_t, U_t), U_t the
 * momentum's contribution S_t, to M_t.  Every gate other than ATLAS_RET_L2
 * takes the identity or degree-2 map or the gated polynomial map, no
 * Newton-Schulz, and runs on the CUDA-core linear kernel; elastic net, Bregman
 * and KL walk the tokens of a chunk one by one (the map is not linear in the
 * gradients), l_q keeps the chunk tables.  ret_param is the gate's parameter. */
#define ATLAS_RET_L2 0      /* M = (1 - alpha) M + U */
#define ATLAS_RET_ELASTIC 1 /* then soft thresholding: M = sign(u) max(|u| - lambda, 0),
                               lambda = ret_param >= 0 (the proximal step of an l1 term) */
#define ATLAS_RET_BREGMAN 2 /* Bregman retention with the sigmoid link: M = sigmoid(
                               (1 - alpha) logit(M) + U), entries in (0, 1); M_0 must lie
                               in (0, 1) (entries outside give NaN); ret_param unused */
#define ATLAS_RET_KL 3      /* per row: M = c softmax((1 - alpha) log M + U), c = ret_param
                               > 0 the row mass; M_0 entries must be > 0 */
#define ATLAS_RET_LQ 4      /* l_q memory (Moneta): A = (1 - alpha) A + U is the state
                               (M_final holds A), the memory reads A_r / ||A_r||_q^(q-2)
                               per row r (a zero row stays zero), q = ret_param in
                               [1, 1e6); the normaliser is taken at each chunk start and
                               held over the chunk (every token when b = 1) */
/* K, Q, V element type */
#define ATLAS_F32 0
#define ATLAS_BF16 1

/* status codes */
#define ATLAS_OK 0
#define ATLAS_ERR_INVALID -1     /* null pointer, bad size, bad enum value */
#define ATLAS_ERR_UNSUPPORTED -2 /* valid description that no kernel here handles */
#define ATLAS_ERR_WORKSPACE -3   /* workspace missing or smaller than required */
#define ATLAS_ERR_CUDA -4        /* a CUDA runtime call or launch failed */
#define ATLAS_ERR_TIMEOUT -5     /* a bounded device-side wait ran out (status word) */

typedef struct atlas_mem_cfg {
  int B, H, N;        /* batch, heads, tokens per head (N >= 0) */
  int d_k, d_v, d_h;  /* key width, value width, MLP hidden width (0 for linear) */
  int mem;            /* ATLAS_MEM_* */
  int phi;            /* ATLAS_PHI_* */
  int loss;           /* ATLAS_LOSS_* */
  float loss_param;   /* p of ATLAS_LOSS_LP, delta of ATLAS_LOSS_HUBER, Delta of
                         ATLAS_LOSS_ROBUST; unused otherwise */
  int c;              /* Omega window length (>= 1); gamma has c entries */
  int b;              /* chunk length (>= 1); 1 = token recurrence */
  int ns_steps;       /* Newton-Schulz iterations on the momentum, 0 = plain momentum */
  float ns_a, ns_b, ns_c; /* X <- a X + b (X X^T) X + c (X X^T)^2 X */
  float ns_eps;       /* X_0 = S / (||S||_F + ns_eps) */
  int in_dtype;       /* ATLAS_F32 or ATLAS_BF16 for K, Q, V */
  float* S_state;     /* optional device momentum [B,H,state] in/out; NULL = start
                         from zero and do not return it */
  int n_history;      /* >= 0: K and V hold n_history + N rows per head, history
                         first.  History rows only enter the windows of the N
                         processed tokens (they update nothing and have no output),
                         so a sequence split on a chunk boundary into two calls --
                         the second given the first part's last c - 1 keys and
                         values as history, and its M and S -- equals one call. */
  void* workspace;    /* device scratch of at least atlas_mem_workspace_bytes() */
  size_t workspace_bytes;
  int* status_dev;    /* optional device int; set to ATLAS_ERR_TIMEOUT by a kernel
                         whose bounded wait ran out (never cleared by the library) */
  int phi_degree;     /* ATLAS_PHI_POLY: p, 1..ATLAS_PHI_MAX_DEGREE (ignored otherwise) */
  float phi_coef[ATLAS_PHI_MAX_DEGREE + 1]; /* ATLAS_PHI_POLY: a_0 .. a_p */
  int retention;      /* ATLAS_RET_* (linear memory; ATLAS_RET_L2 otherwise) */
  float ret_param;    /* lambda, c or q of the gate (see ATLAS_RET_*) */
} atlas_mem_cfg;

/* Number of fp32 entries in one head's memory state (and momentum):
 * linear d_v * D; MLP and LN MLP 2 * d * d_h; gated MLP 3 * d * d_h.  0 for an
 * invalid description. */
size_t atlas_mem_state_size(const atlas_mem_cfg* cfg);

/* Bytes of device workspace atlas_mem_forward needs for this description
 * (may be 0).  (size_t)-1 for an invalid description. */
size_t atlas_mem_workspace_bytes(const atlas_mem_cfg* cfg);

/* The chunked memory update over all B*H heads (nh = cfg->n_history).
 *   K      [B,H,nh+N,d_k] keys (fp32 or bf16 per cfg->in_dtype), history rows first
 *   Q      [B,H,N,d_k]  queries (same type)
 *   V      [B,H,nh+N,d_v] values (same type), history rows first
 *   alpha, eta, theta [B,H,N] fp32 per-token decay, momentum and step gates
 *   gamma  [c] fp32     window weight by lag: gamma[j] weighs token t-j in l_t
 *   Y      [B,H,N,d_v]  fp32 out: y_t = M_t(Phi(q_t))
 *   M_final [B,H,state] fp32 in/out: M_0 on entry, M_N on return.  Linear
 *          layout d_v x D row-major; MLP layout W1 (d x d_h) then W2
 *          (d_h x d), both row-major (gated: then W3, d_h x d).
 * Returns ATLAS_OK or a negative ATLAS_ERR_* code. */
int atlas_mem_forward(const void* K, const void* Q, const void* V, const float* alpha,
                      const float* eta, const float* theta, const float* gamma,
                      const atlas_mem_cfg* cfg, float* Y, float* M_final, void* stream);

/* Bytes of device workspace atlas_mem_backward needs for this description;
 * (size_t)-1 if the description is invalid or not covered (see below). */
size_t atlas_mem_backward_workspace_bytes(const atlas_mem_cfg* cfg);

/* Backward pass: the gradients that train everything outside the memory (the
 * outer loop of "논문 리뷰 Google ATLAS", Deep Memory Module; "It's All
 * Connected (Miras)", Associative Memory & Attentional Bias, Remark 2).  For
 * the forward atlas_mem_forward computes from the same inputs and initial
 * state M0, with the scalar loss
 *     L = sum_t <dY_t, y_t> + <dM_N, M_N>
 * it returns dL/dK, dL/dQ, dL/dV, dL/dalpha, dL/deta, dL/dtheta and dL/dM_0.
 * Covered: linear memory, identity map, d_k = d_v = 128, b = 64, c = 1, the
 * l2, l_p or Huber bias, momentum and decay with any gates, no history rows,
 * cfg->S_state = NULL (the forward starts from zero momentum; its final
 * momentum gets no gradient).  Anything else returns ATLAS_ERR_UNSUPPORTED
 * before any launch.  The window weight gamma[0] is an input but gets no
 * gradient.
 *   K, Q, V, alpha, eta, theta, gamma: as for atlas_mem_forward
 *   M0     [B,H,d_v,d_k] fp32 in: the forward's initial state
 *   dY     [B,H,N,d_v]   fp32 in: dL/dY
 *   dM     [B,H,d_v,d_k] fp32 in/out: dL/dM_N on entry, dL/dM_0 on return
 *   dK, dQ [B,H,N,d_k], dV [B,H,N,d_v], dalpha, deta, dtheta [B,H,N]: fp32 out
 * Workspace: cfg->workspace of at least atlas_mem_backward_workspace_bytes()
 * (the chunk-start states and momenta, gate tables and partial sums; ~8.2 KB
 * per token).
 * Four kernel launches on `stream`; returns ATLAS_OK or an ATLAS_ERR_* code. */
int atlas_mem_backward(const void* K, const void* Q, const void* V, const float* alpha,
                       const float* eta, const float* theta, const float* gamma,
                       const atlas_mem_cfg* cfg, const float* M0, const float* dY, float* dM,
                       float* dK, float* dQ, float* dV, float* dalpha, float* deta,
                       float* dtheta, void* stream);

/* Size of the device scratch array that atlas_mem_forward_noalloc uses:
 * 32 MiB, held by every GPU that loads the library until the process exits. */
#define ATLAS_NOALLOC_SCRATCH_BYTES (32u << 20)

/* atlas_mem_forward for callers that cannot allocate device memory.
 * (No counterpart in the method's description: a library convenience.)
 * Code that runs where allocation is not allowed -- inside an allocator or
 * memory-pool callback, or in a process whose device memory is reserved up
 * front -- cannot create the workspace atlas_mem_forward asks for.  This entry
 * point takes the same arguments, ignores cfg->workspace and
 * cfg->workspace_bytes, and uses a fixed scratch array built into the library
 * instead; it calls no cudaMalloc, cudaFree or allocating routine.
 * - Limit: a description whose atlas_mem_workspace_bytes() exceeds
 *   ATLAS_NOALLOC_SCRATCH_BYTES returns ATLAS_ERR_WORKSPACE and launches
 *   nothing (split the heads over several calls instead).
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 * - Start-up: the CUDA runtime loads a library's device code lazily by
 *   default, on first use, and loading it is what places the scratch array
 *   (and each kernel family's code) in device memory.  So the first call on
 *   a device can take device memory, and a first call of another kernel
 *   family can too.  A caller that must not allocate later makes one call
 *   per problem description it will use at start-up, before it reserves or
 *   hands out its memory, or runs with CUDA_MODULE_LOADING=EAGER so that
 *   everything is loaded with the library.
 * - All calls on a device share the one array and each call overwrites it:
 *   calls whose work overlaps on the GPU (different streams, or threads)
 *   race and give wrong results.  Serialise them, e.g. on one stream.
 * - The array's address is cached per device for the life of the process;
 *   cudaDeviceReset (or any teardown of the device's primary context)
 *   invalidates it, so do not call this entry point after one.
 * Returns what atlas_mem_forward returns. */
int atlas_mem_forward_noalloc(const void* K, const void* Q, const void* V, const float* alpha,
                              const float* eta, const float* theta, const float* gamma,
                              const atlas_mem_cfg* cfg, float* Y, float* M_final, void* stream);

/* Static description of a status code. */
const char* atlas_mem_strerror(int status);

/* Name of the kernel family atlas_mem_forward would launch for cfg (for
 * reports): "linear_tc", "linear_seq", "linear_wide", "linear_chunk",
 * "linear_simt", "mlp_tc", "mlp_simt", or "" if invalid. */
const char* atlas_mem_path(const atlas_mem_cfg* cfg);

/* Number of kernel launches atlas_mem_forward makes for cfg (for reports). */
long atlas_mem_launch_count(const atlas_mem_cfg* cfg);

#ifdef __cplusplus
}
#endif

#endif /* ATLAS_MEM_H */
