/*
 * atlas_oracle.c -- plain, slow, fp64 CPU oracle of the test-time memory update
 * (Titans / Miras / ATLAS family).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the package's smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * library: every formula here is written out again from the pages.
 *
 * Sources (page title, section):
 *   [Titans]  "[Paper Review] Titans 논문 이해하기" (rahites.tistory.com),
 *             "Learning Process and Surprise Metric" (momentum S_t),
 *             "Objective" (l2 attentional bias), "Forgetting Mechanism"
 *             (M_t = (1-alpha_t) M_{t-1} + S_t), "Retrieving a Memory"
 *             (y_t = M*(q_t), a forward pass without update).
 *   [ATLAS]   "논문 리뷰 Google ATLAS" (velog.io), §3.1 (polynomial feature
 *             map Phi_p, l2 bias on Phi(k)), §3.2 (Omega rule: sliding-window
 *             loss sum_{i=t-c+1..t} gamma_i ||M(Phi(k_i)) - v_i||^2),
 *             §3.3 (chunked form: gradients inside a chunk taken at the state
 *             the previous chunk ended with).
 *   [ATLAS-s] "ATLAS: Learning to Optimally Memorize the Context at Test
 *             Time" (paperlayer.ai summary), §5 Memory Optimization (Muon /
 *             Newton-Schulz in place of plain GD; Atlas++: a gated MLP memory
 *             with three linear maps), App. E (2-layer residual MLP memory,
 *             expansion 4, GELU), §6 (residual connections and layer
 *             normalisation in the memory).
 *   [Miras]   "It's All Connected: A Journey Through Test-Time Memorization,
 *             ..." (still-with-you.github.io), Associative Memory & Attentional
 *             Bias (linear attention = GD on -2<Mk, v>), #1 Alternative
 *             Attentional Biases (l_p loss ||M(k) - v||_p^p, Huber loss),
 *             Training (chunk-wise parallelisation at the chunk-start state,
 *             Miras layer outputs M(q_t); the memory x + LN(W1 sigma(W2 x))).
 *
 * Readings taken where the pages are silent or disagree (each one is listed
 * in the design notes of the repository):
 *   - gate names follow [Titans]/[Miras]: S_t = eta_t S_{t-1} - theta_t g_t,
 *     M_t = (1 - alpha_t) M_{t-1} + S_t;
 *   - the loss is ||.||^2 with no 1/2, so the gradient carries the factor 2;
 *   - the chunk-start state is the state after the last token of the
 *     previous chunk, so b = 1 is the token recurrence;
 *   - gamma is fixed per lag j = t - i (gamma[0] weighs the current token),
 *     not renormalised, and the window is clipped at the first token;
 *   - readout is after the write: y_t = M_t(Phi(q_t));
 *   - Phi_2(x) = [x_1..x_d, x_i x_j for i <= j, i-major], no constant term and
 *     no multinomial weights (d = 32 gives 560 features);
 *   - the general map with input gating ([ATLAS] §3.1, "Input gating": a_i
 *     switches the features of degree i on or off) is
 *     Phi(x) = [a_0; a_1 x; a_2 (x_i x_j)_{i<=j}; ...; a_p (degree-p monomials)],
 *     every degree's monomials once, without multinomial weights, in
 *     lexicographic order of their sorted index tuples; a degree whose a_d is 0
 *     is left out of the feature vector (so a = (0, 1, 1) is Phi_2 above);
 *   - MLP memory M(x) = x + W1 GELU(W2 x) without LayerNorm, exact (erf) GELU;
 *   - Newton-Schulz (when enabled) acts on the momentum of each weight matrix
 *     separately, per token: M_t = (1 - alpha_t) M_{t-1} + NS(S_t), with
 *     X_0 = S / (||S||_F + eps) and the literal X X^T Gram;
 *   - the layer-normalised MLP memory is x + LN(W1 GELU(W2 x)) with a plain
 *     LN (no learned scale or shift; variance over the d outputs, divided by
 *     d, plus 1e-5 under the square root);
 *   - the gated (Atlas++) memory is x + W1 (GELU(W2 x) * (W3 x)), with W2 and
 *     W3 both d_h x d, and Newton-Schulz (when enabled) applied to W3 as to W2;
 *   - the Huber bias is taken per coordinate with one threshold delta for all
 *     tokens, scaled to agree with the l2 bias inside the threshold:
 *     h(e) = e^2 for |e| <= delta, 2 delta |e| - delta^2 beyond (the pages let
 *     delta vary per token and channel; a constant is the plainest case);
 *   - the value-shift robust bias ([Miras] #1: the worst case over a shift of v
 *     within radius Delta, closed form 1/2 ||e||^2 + Delta ||e|| + 1/2 Delta^2)
 *     is scaled by 2 like the Huber bias, ||e||^2 + 2 Delta ||e|| + Delta^2, so
 *     Delta = 0 is the l2 bias; its gradient 2 e (1 + Delta / ||e||) is 0 at e = 0;
 *   - retention gates ([Miras] #2 Alternative Retention Gates, linear memory):
 *     the l2 gate's step U = (1 - alpha_t) M_{t-1} + S_t becomes
 *       elastic net: M_t = sign(U) max(|U| - gamma, 0) (soft thresholding);
 *       Bregman with a sigmoid link: M_t = sigmoid((1 - alpha_t) logit(M_{t-1}) + S_t);
 *       KL: each row of M a distribution of mass c,
 *           M_t = c softmax((1 - alpha_t) log M_{t-1} + S_t) per row;
 *       l_q (Moneta): the state is the accumulator A_t = (1 - alpha_t) A_{t-1} + S_t
 *           and the memory is A / ||A||_q^(q-2) per row, the normaliser taken at
 *           each chunk start ("Moneta applies the l_q normalisation at the chunk
 *           end"; b = 1 renormalises every token);
 *     alpha_t keeps its role of retention strength and S_t the (momentum) step;
 *     the rows are the memory's output rows (one per value coordinate);
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORC_MEM_LINEAR 0
#define ORC_MEM_MLP 1
#define ORC_MEM_MLP_LN 2     /* x + LN(W1 GELU(W2 x)) */
#define ORC_MEM_MLP_GATED 3  /* x + W1 (GELU(W2 x) * (W3 x)) */
#define ORC_LN_EPS 1e-5
#define ORC_PHI_IDENTITY 0
#define ORC_PHI_POLY2 1
#define ORC_PHI_POLY 2       /* degree phi_degree, input-gating coefficients phi_coef */
#define ORC_PHI_MAX_DEGREE 4
#define ORC_LOSS_L2 0
#define ORC_LOSS_DOT 1
#define ORC_LOSS_LP 2
#define ORC_LOSS_HUBER 3
#define ORC_LOSS_ROBUST 4   /* value-shift robust bias, radius loss_param */
/* retention gates (linear memory): the map from the decayed step to the new state */
#define ORC_RET_L2 0        /* M = (1 - alpha) M + S */
#define ORC_RET_ELASTIC 1   /* then soft thresholding by ret_param */
#define ORC_RET_BREGMAN 2   /* M = sigmoid((1 - alpha) logit(M) + S) */
#define ORC_RET_KL 3        /* per row: M = c softmax((1 - alpha) log M + S), c = ret_param */
#define ORC_RET_LQ 4        /* A = (1 - alpha) A + S, memory A / ||A||_q^(q-2) per row, q = ret_param */

/* Per-head problem description.  All tensors handed to the oracle are fp64,
 * one head after another. */
typedef struct {
  int N;        /* tokens */
  int d_k;      /* key / query width before the feature map */
  int d_v;      /* value width */
  int d_h;      /* MLP hidden width (MLP memory only) */
  int mem;      /* ORC_MEM_LINEAR, ORC_MEM_MLP, ORC_MEM_MLP_LN or ORC_MEM_MLP_GATED */
  int phi;      /* ORC_PHI_IDENTITY or ORC_PHI_POLY2 (linear memory only) */
  int loss;     /* ORC_LOSS_L2, _DOT, _LP or _HUBER */
  int c;        /* Omega window length, >= 1 */
  int b;        /* chunk length, >= 1 (1 = token recurrence) */
  int ns_steps; /* Newton-Schulz iterations on the momentum, 0 = none */
  double ns_a, ns_b, ns_c, ns_eps;
  int n_history; /* tokens before the first processed one: K, V rows that only
                    enter the windows of processed tokens (they update nothing) */
  double loss_param; /* p of the l_p bias (>= 1), delta of the Huber bias (> 0) */
  int phi_degree;    /* ORC_PHI_POLY: highest degree p (1..ORC_PHI_MAX_DEGREE) */
  double phi_coef[ORC_PHI_MAX_DEGREE + 1]; /* ORC_PHI_POLY: a_0 .. a_p */
  int retention;     /* ORC_RET_* (linear memory; ORC_RET_L2 for the MLP memories) */
  double ret_param;  /* gamma of ELASTIC, c of KL, q of LQ */
} orc_cfg;

/* ------------------------------------------------------------------ sizes */

/* Number of monomials of degree exactly e in d variables: C(d + e - 1, e). */
static long orc_monomials(int d, int e) {
  long c = 1;
  for (int i = 1; i <= e; ++i) c = c * (d + i - 1) / i;
  return c;
}

/* Width of Phi(x).  [ATLAS] §3.1: Phi_p(x) = [x^beta]_{|beta| <= p}; with the
 * constant dropped and p = 2 that is d linear terms and d(d+1)/2 products; the
 * gated map keeps the degrees whose coefficient is non-zero. */
int orc_feature_dim(const orc_cfg* g) {
  if (g->mem != ORC_MEM_LINEAR) return g->d_k;
  if (g->phi == ORC_PHI_POLY2) return g->d_k + g->d_k * (g->d_k + 1) / 2;
  if (g->phi == ORC_PHI_POLY) {
    long D = 0;
    for (int e = 0; e <= g->phi_degree; ++e)
      if (g->phi_coef[e] != 0.0) D += orc_monomials(g->d_k, e);
    return (int)D;
  }
  return g->d_k;
}

/* Number of fp64 entries in one head's memory state (and in its momentum). */
long orc_state_size(const orc_cfg* g) {
  if (g->mem == ORC_MEM_MLP || g->mem == ORC_MEM_MLP_LN) return 2L * g->d_k * g->d_h;
  if (g->mem == ORC_MEM_MLP_GATED) return 3L * g->d_k * g->d_h;
  return (long)g->d_v * orc_feature_dim(g);
}

/* --------------------------------------------------------- feature map Phi */

/* Visit the sorted index tuples i_1 <= ... <= i_e over [0, d) in lexicographic
 * order: the first tuple is all zeros, the next raises the last entry that can
 * still grow and resets the entries after it to that value.  Returns 0 after
 * the last tuple. */
static int orc_next_tuple(int* idx, int e, int d) {
  int r = e - 1;
  while (r >= 0 && idx[r] == d - 1) --r;
  if (r < 0) return 0;
  ++idx[r];
  for (int s = r + 1; s < e; ++s) idx[s] = idx[r];
  return 1;
}

/* Apply fn(ctx, feature, degree, idx) to every feature of the gated map in order. */
static void orc_poly_features(const orc_cfg* g, void (*fn)(void*, int, int, const int*),
                              void* ctx) {
  int j = 0, idx[ORC_PHI_MAX_DEGREE];
  for (int e = 0; e <= g->phi_degree; ++e) {
    if (g->phi_coef[e] == 0.0) continue;
    for (int r = 0; r < e; ++r) idx[r] = 0;
    do {
      fn(ctx, j++, e, idx);
    } while (e > 0 && orc_next_tuple(idx, e, g->d_k));
  }
}

typedef struct {
  const orc_cfg* g;
  const double* x;
  double* out;
} orc_phi_ctx;

static void orc_phi_one(void* c, int j, int e, const int* idx) {
  orc_phi_ctx* p = (orc_phi_ctx*)c;
  double v = p->g->phi_coef[e];
  for (int r = 0; r < e; ++r) v *= p->x[idx[r]];
  p->out[j] = v;
}

/* [ATLAS] §3.1 polynomial map (degree 2, or general with input gating), read as
 * described above. */
void orc_phi(const orc_cfg* g, const double* x, double* out) {
  int d = g->d_k;
  if (g->mem == ORC_MEM_LINEAR && g->phi == ORC_PHI_POLY) {
    orc_phi_ctx c = {g, x, out};
    orc_poly_features(g, orc_phi_one, &c);
    return;
  }
  for (int i = 0; i < d; ++i) out[i] = x[i];
  if (g->mem != ORC_MEM_LINEAR || g->phi == ORC_PHI_IDENTITY) return;
  int p = d;
  for (int i = 0; i < d; ++i)
    for (int j = i; j < d; ++j) out[p++] = x[i] * x[j];
}

/* ------------------------------------------------------------------- GELU */

/* GELU(x) = x * P(X <= x), X ~ N(0,1), written with erf. */
double orc_gelu(double x) { return 0.5 * x * (1.0 + erf(x / sqrt(2.0))); }

/* d/dx GELU(x) = P(X <= x) + x * pdf(x). */
double orc_gelu_prime(double x) {
  const double inv_sqrt_2pi = 0.39894228040143267794;
  return 0.5 * (1.0 + erf(x / sqrt(2.0))) + x * inv_sqrt_2pi * exp(-0.5 * x * x);
}

/* ------------------------------------------------------- memory forward */

/* The MLP memories' branch, M(x) = x + out:
 *   plain:  z = W2 x, h = GELU(z),                 out = W1 h
 *   LN:     the same, then out = LN(W1 h) = (u - mean u) / sqrt(var u + 1e-5)
 *   gated:  z = W2 x, w = W3 x, h = GELU(z) * w,   out = W1 h
 * Intermediates (each may be NULL): z, w [d_h]; h [d_h]; the branch output
 * [d] (after LN for the LN memory); the normalised values' 1 / sqrt(var + eps)
 * (LN memory only, one value). */
static void orc_mlp_forward(const orc_cfg* g, const double* state, const double* x, double* z_out,
                            double* w_out, double* h_out, double* out, double* inv_sd) {
  int d = g->d_k, dh = g->d_h;
  const double* W1 = state;                  /* d  x dh */
  const double* W2 = state + (long)d * dh;   /* dh x d  */
  const double* W3 = state + 2L * d * dh;    /* dh x d  (gated memory) */
  double* h = (double*)malloc(sizeof(double) * dh);
  for (int j = 0; j < dh; ++j) {
    double z = 0.0;
    for (int i = 0; i < d; ++i) z += W2[(long)j * d + i] * x[i];
    double w = 1.0;
    if (g->mem == ORC_MEM_MLP_GATED) {
      w = 0.0;
      for (int i = 0; i < d; ++i) w += W3[(long)j * d + i] * x[i];
    }
    if (z_out) z_out[j] = z;
    if (w_out) w_out[j] = w;
    h[j] = orc_gelu(z) * w;
    if (h_out) h_out[j] = h[j];
  }
  for (int r = 0; r < d; ++r) {
    double s = 0.0;
    for (int j = 0; j < dh; ++j) s += W1[(long)r * dh + j] * h[j];
    out[r] = s;
  }
  if (g->mem == ORC_MEM_MLP_LN) {
    double mu = 0.0, var = 0.0;
    for (int r = 0; r < d; ++r) mu += out[r];
    mu /= d;
    for (int r = 0; r < d; ++r) var += (out[r] - mu) * (out[r] - mu);
    var /= d;
    const double is = 1.0 / sqrt(var + ORC_LN_EPS);
    for (int r = 0; r < d; ++r) out[r] = (out[r] - mu) * is;
    if (inv_sd) *inv_sd = is;
  }
  free(h);
}

/* Memory output M(x) for a key/query x (before Phi).
 * Linear: M Phi(x).  MLP: x + W1 GELU(W2 x)  ([ATLAS-s] App. E; [Titans]
 * Memory Architecture); LN: x + LN(W1 GELU(W2 x)) ([Miras] Moneta, Yaad,
 * Memora memory; [ATLAS-s] §6); gated: x + W1 (GELU(W2 x) * (W3 x))
 * ([ATLAS-s] §5, Atlas++).  `out` has d_v entries. */
void orc_memory_apply(const orc_cfg* g, const double* state, const double* x, double* out) {
  if (g->mem == ORC_MEM_LINEAR) {
    int D = orc_feature_dim(g);
    double* f = (double*)malloc(sizeof(double) * D);
    orc_phi(g, x, f);
    for (int r = 0; r < g->d_v; ++r) {
      double s = 0.0;
      for (int j = 0; j < D; ++j) s += state[(long)r * D + j] * f[j];
      out[r] = s;
    }
    free(f);
    return;
  }
  int d = g->d_k;
  double* u = (double*)malloc(sizeof(double) * d);
  orc_mlp_forward(g, state, x, NULL, NULL, NULL, u, NULL);
  for (int r = 0; r < d; ++r) out[r] = x[r] + u[r];
  free(u);
}

/* ------------------------------------------------------- loss gradient */

/* Derivative of the bias with respect to one output coordinate y, with
 * e = y - v.  [Titans] Objective: l2, sum e^2 -> 2 e.  [Miras] #1 Alternative
 * Attentional Biases: l_p, sum |e|^p -> p |e|^(p-1) sign(e); Huber (per
 * coordinate, see the readings above) -> 2 e inside the threshold,
 * 2 delta sign(e) beyond. */
static double orc_bias_dy(const orc_cfg* g, double e) {
  if (g->loss == ORC_LOSS_LP) {
    if (e == 0.0) return 0.0;
    const double s = e > 0.0 ? 1.0 : -1.0;
    return g->loss_param * pow(fabs(e), g->loss_param - 1.0) * s;
  }
  if (g->loss == ORC_LOSS_HUBER) {
    const double d = g->loss_param;
    if (fabs(e) <= d) return 2.0 * e;
    return e > 0.0 ? 2.0 * d : -2.0 * d;
  }
  return 2.0 * e;
}

/* Derivative of the bias with respect to the whole output vector y (n entries),
 * e = y - v: orc_bias_dy per coordinate, or the robust bias
 * 2 e (1 + Delta / ||e||) (0 at e = 0). */
static void orc_bias_vec(const orc_cfg* g, const double* e, int n, double* out) {
  if (g->loss == ORC_LOSS_ROBUST) {
    double ne = 0.0;
    for (int r = 0; r < n; ++r) ne += e[r] * e[r];
    ne = sqrt(ne);
    for (int r = 0; r < n; ++r) out[r] = ne > 0.0 ? 2.0 * e[r] * (1.0 + g->loss_param / ne) : 0.0;
    return;
  }
  for (int r = 0; r < n; ++r) out[r] = orc_bias_dy(g, e[r]);
}

/* Gradient of the attentional bias with respect to the memory state, written
 * into G (state layout).
 *   l2  ([Titans] Objective; [ATLAS] §3.1):  l = ||M(Phi(k)) - v||^2.
 *   dot ([Miras] Associative Memory & Attentional Bias): l = -2 <M(Phi(k)), v>.
 *   l_p, Huber ([Miras] #1 Alternative Attentional Biases): orc_bias_dy.
 * For the MLP memories the gradient is plain backpropagation through the
 * branch of orc_mlp_forward (and LN's mean and variance for the LN memory). */
void orc_grad(const orc_cfg* g, const double* state, const double* k, const double* v, double* G) {
  if (g->mem == ORC_MEM_LINEAR) {
    int D = orc_feature_dim(g), dv = g->d_v;
    double* f = (double*)malloc(sizeof(double) * D);
    double* e = (double*)malloc(sizeof(double) * dv);
    orc_phi(g, k, f);
    for (int r = 0; r < dv; ++r) {
      if (g->loss == ORC_LOSS_DOT) {
        e[r] = -2.0 * v[r];         /* dl/d(M Phi) = -2 v */
      } else {
        double s = 0.0;
        for (int j = 0; j < D; ++j) s += state[(long)r * D + j] * f[j];
        e[r] = s - v[r];
      }
    }
    if (g->loss != ORC_LOSS_DOT) orc_bias_vec(g, e, dv, e);  /* l2: 2 (M Phi - v) */
    for (int r = 0; r < dv; ++r)
      for (int j = 0; j < D; ++j) G[(long)r * D + j] = e[r] * f[j];
    free(f);
    free(e);
    return;
  }
  int d = g->d_k, dh = g->d_h;
  const double* W1 = state;
  double* G1 = G;
  double* G2 = G + (long)d * dh;
  double* G3 = G + 2L * d * dh;
  double* z = (double*)malloc(sizeof(double) * dh);
  double* w = (double*)malloc(sizeof(double) * dh);
  double* h = (double*)malloc(sizeof(double) * dh);
  double* o = (double*)malloc(sizeof(double) * d);
  double* dy = (double*)malloc(sizeof(double) * d);
  double* du = (double*)malloc(sizeof(double) * d);
  double is = 1.0;
  orc_mlp_forward(g, state, k, z, w, h, o, &is);
  for (int r = 0; r < d; ++r) dy[r] = g->loss == ORC_LOSS_DOT ? -2.0 * v[r] : k[r] + o[r] - v[r];
  if (g->loss != ORC_LOSS_DOT) orc_bias_vec(g, dy, d, dy);
  /* through LN: du = is (dy - mean(dy) - n mean(dy * n)), n = the normalised values */
  if (g->mem == ORC_MEM_MLP_LN) {
    double m1 = 0.0, m2 = 0.0;
    for (int r = 0; r < d; ++r) {
      m1 += dy[r];
      m2 += dy[r] * o[r];
    }
    m1 /= d;
    m2 /= d;
    for (int r = 0; r < d; ++r) du[r] = is * (dy[r] - m1 - o[r] * m2);
  } else {
    for (int r = 0; r < d; ++r) du[r] = dy[r];
  }
  /* dl/dW1 = du h^T */
  for (int r = 0; r < d; ++r)
    for (int j = 0; j < dh; ++j) G1[(long)r * dh + j] = du[r] * h[j];
  /* dl/dh = W1^T du; h = GELU(z) w: dl/dz = dl/dh w GELU'(z), dl/dw = dl/dh GELU(z) */
  for (int j = 0; j < dh; ++j) {
    double s = 0.0;
    for (int r = 0; r < d; ++r) s += W1[(long)r * dh + j] * du[r];
    const double dz = s * w[j] * orc_gelu_prime(z[j]);
    for (int i = 0; i < d; ++i) G2[(long)j * d + i] = dz * k[i];
    if (g->mem == ORC_MEM_MLP_GATED) {
      const double dw = s * orc_gelu(z[j]);
      for (int i = 0; i < d; ++i) G3[(long)j * d + i] = dw * k[i];
    }
  }
  free(z);
  free(w);
  free(h);
  free(o);
  free(dy);
  free(du);
}

/* ------------------------------------------------------ Newton-Schulz */

/* C (m x n) = A (m x p) * B (p x n), all row-major. */
static void orc_matmul(int m, int p, int n, const double* A, const double* B, double* C) {
  for (int i = 0; i < m; ++i) {
    for (int j = 0; j < n; ++j) C[(long)i * n + j] = 0.0;
    for (int l = 0; l < p; ++l) {
      double a = A[(long)i * p + l];
      for (int j = 0; j < n; ++j) C[(long)i * n + j] += a * B[(long)l * n + j];
    }
  }
}

/* Newton-Schulz orthogonalisation of one rows x cols matrix ([ATLAS-s] §5,
 * Muon): X_0 = S / (||S||_F + eps); repeat X <- a X + b (X X^T) X +
 * c (X X^T)^2 X, where (X X^T)^2 X is evaluated as (X X^T)((X X^T) X). */
void orc_newton_schulz(int rows, int cols, const double* S, int steps, double a, double b,
                       double c, double eps, double* out) {
  long n = (long)rows * cols;
  double nrm = 0.0;
  for (long i = 0; i < n; ++i) nrm += S[i] * S[i];
  nrm = sqrt(nrm);
  double* X = out;
  for (long i = 0; i < n; ++i) X[i] = S[i] / (nrm + eps);
  double* Xt = (double*)malloc(sizeof(double) * n);
  double* A = (double*)malloc(sizeof(double) * (long)rows * rows);
  double* AX = (double*)malloc(sizeof(double) * n);
  double* AAX = (double*)malloc(sizeof(double) * n);
  for (int it = 0; it < steps; ++it) {
    for (int i = 0; i < rows; ++i)
      for (int j = 0; j < cols; ++j) Xt[(long)j * rows + i] = X[(long)i * cols + j];
    orc_matmul(rows, cols, rows, X, Xt, A);     /* A = X X^T */
    orc_matmul(rows, rows, cols, A, X, AX);     /* A X */
    orc_matmul(rows, rows, cols, A, AX, AAX);   /* A (A X) */
    for (long i = 0; i < n; ++i) X[i] = a * X[i] + b * AX[i] + c * AAX[i];
  }
  free(Xt);
  free(A);
  free(AX);
  free(AAX);
}

/* The update a momentum contributes to the memory: S itself, or NS(S) applied
 * to each weight matrix of the state on its own. */
static void orc_momentum_update(const orc_cfg* g, const double* S, double* out) {
  long n = orc_state_size(g);
  if (g->ns_steps <= 0) {
    memcpy(out, S, sizeof(double) * n);
    return;
  }
  if (g->mem == ORC_MEM_LINEAR) {
    orc_newton_schulz(g->d_v, orc_feature_dim(g), S, g->ns_steps, g->ns_a, g->ns_b, g->ns_c,
                      g->ns_eps, out);
    return;
  }
  long half = (long)g->d_k * g->d_h;
  orc_newton_schulz(g->d_k, g->d_h, S, g->ns_steps, g->ns_a, g->ns_b, g->ns_c, g->ns_eps, out);
  orc_newton_schulz(g->d_h, g->d_k, S + half, g->ns_steps, g->ns_a, g->ns_b, g->ns_c, g->ns_eps,
                    out + half);
  if (g->mem == ORC_MEM_MLP_GATED)  /* W3, like W2 */
    orc_newton_schulz(g->d_h, g->d_k, S + 2 * half, g->ns_steps, g->ns_a, g->ns_b, g->ns_c,
                      g->ns_eps, out + 2 * half);
}

/* ------------------------------------------------------- one head, one token */

/* l_q gate: per-row normalisers z_r = ||A_r||_q^(q-2) of the accumulator A. */
static void orc_lq_norms(const orc_cfg* g, const double* A, double* z) {
  int D = orc_feature_dim(g);
  double q = g->ret_param;
  for (int r = 0; r < g->d_v; ++r) {
    double s = 0.0;
    for (int j = 0; j < D; ++j) s += pow(fabs(A[(long)r * D + j]), q);
    z[r] = s > 0.0 ? pow(s, (q - 2.0) / q) : 0.0;
  }
}

/* The memory a state describes: the state itself, or for the l_q gate the
 * accumulator divided per row by its normalisers (a zero row stays zero). */
static void orc_memory_of(const orc_cfg* g, const double* M, const double* z, double* W) {
  long n = orc_state_size(g);
  if (g->retention != ORC_RET_LQ) {
    memcpy(W, M, sizeof(double) * n);
    return;
  }
  int D = orc_feature_dim(g);
  for (int r = 0; r < g->d_v; ++r)
    for (int j = 0; j < D; ++j) {
      long x = (long)r * D + j;
      W[x] = z[r] > 0.0 ? M[x] / z[r] : M[x];
    }
}

/* The retention gate's map from the state and the step to the new state
 * ([Titans] Forgetting Mechanism for the l2 gate; [Miras] #2 Alternative
 * Retention Gates for the others, read as described at the top). */
static void orc_retain(const orc_cfg* g, double alpha, const double* upd, double* M) {
  long n = orc_state_size(g);
  switch (g->retention) {
    case ORC_RET_ELASTIC:
      for (long j = 0; j < n; ++j) {
        double u = (1.0 - alpha) * M[j] + upd[j];
        double m = fabs(u) - g->ret_param;
        M[j] = m > 0.0 ? (u > 0.0 ? m : -m) : 0.0;
      }
      return;
    case ORC_RET_BREGMAN:
      for (long j = 0; j < n; ++j) {
        double u = (1.0 - alpha) * log(M[j] / (1.0 - M[j])) + upd[j];
        M[j] = 1.0 / (1.0 + exp(-u));
      }
      return;
    case ORC_RET_KL: {
      int D = orc_feature_dim(g);
      for (int r = 0; r < g->d_v; ++r) {
        double* m = M + (long)r * D;
        const double* u = upd + (long)r * D;
        double mx = -INFINITY;
        for (int j = 0; j < D; ++j) {
          m[j] = (1.0 - alpha) * log(m[j]) + u[j];
          if (m[j] > mx) mx = m[j];
        }
        double s = 0.0;
        for (int j = 0; j < D; ++j) {
          m[j] = exp(m[j] - mx);
          s += m[j];
        }
        for (int j = 0; j < D; ++j) m[j] *= g->ret_param / s;
      }
      return;
    }
    default:  /* l2 and the l_q accumulator */
      for (long j = 0; j < n; ++j) M[j] = (1.0 - alpha) * M[j] + upd[j];
  }
}

/* Shared token step: S = eta S - theta g; M = retain(M, U(S)); y = memory(M)(Phi(q)).
 * ([Titans] Surprise Metric, Forgetting Mechanism, Retrieving.)  z: the l_q
 * gate's normalisers of the current chunk (else unused); W: scratch. */
static void orc_token_step(const orc_cfg* g, double alpha, double eta, double theta,
                           const double* grad, const double* q, double* M, double* S,
                           double* upd, double* y, const double* z, double* W) {
  long n = orc_state_size(g);
  for (long j = 0; j < n; ++j) S[j] = eta * S[j] - theta * grad[j];
  orc_momentum_update(g, S, upd);
  orc_retain(g, alpha, upd, M);
  orc_memory_of(g, M, z, W);
  orc_memory_apply(g, W, q, y);
}

/* Chunked Omega rule for one head ([ATLAS] §3.3, [Miras] Training): for every
 * chunk of b tokens, M0 is the state the previous chunk ended with, and every
 * token n of the chunk uses g_n = sum_{i=n-c+1..n, i>=0} gamma[n-i] grad(M0; k_i, v_i).
 * b = 1 makes M0 the state right before each token. */
static void orc_head_chunked(const orc_cfg* g, const double* K, const double* Q, const double* V,
                             const double* alpha, const double* eta, const double* theta,
                             const double* gamma, double* M, double* S, double* Y) {
  long n = orc_state_size(g);
  double* M0 = (double*)malloc(sizeof(double) * n);
  double* gsum = (double*)malloc(sizeof(double) * n);
  double* Gi = (double*)malloc(sizeof(double) * n);
  double* upd = (double*)malloc(sizeof(double) * n);
  double* W = (double*)malloc(sizeof(double) * n);
  double* z = (double*)malloc(sizeof(double) * (g->d_v > 0 ? g->d_v : 1));
  int dk = g->d_k, dv = g->d_v, nh = g->n_history;
  /* K, V rows: token i (from -nh) is row i + nh */
  for (int t0 = 0; t0 < g->N; t0 += g->b) {
    /* the chunk-start memory (the l_q gate renormalises here only) */
    if (g->retention == ORC_RET_LQ) orc_lq_norms(g, M, z);
    orc_memory_of(g, M, z, M0);
    int t1 = t0 + g->b < g->N ? t0 + g->b : g->N;
    for (int t = t0; t < t1; ++t) {
      for (long j = 0; j < n; ++j) gsum[j] = 0.0;
      int i0 = t - g->c + 1 < -nh ? -nh : t - g->c + 1;
      for (int i = i0; i <= t; ++i) {
        orc_grad(g, M0, K + (long)(i + nh) * dk, V + (long)(i + nh) * dv, Gi);
        double w = gamma[t - i];
        for (long j = 0; j < n; ++j) gsum[j] += w * Gi[j];
      }
      orc_token_step(g, alpha[t], eta[t], theta[t], gsum, Q + (long)t * dk, M, S, upd,
                     Y + (long)t * dv, z, W);
    }
  }
  free(M0);
  free(gsum);
  free(Gi);
  free(upd);
  free(W);
  free(z);
}

/* Token recurrence for one head, written separately from the chunked loop:
 * the gradient of every window term is taken at M_{t-1}
 * ([ATLAS] §3.3, the b = 1 case; [Titans] Surprise Metric). */
static void orc_head_recurrent(const orc_cfg* g, const double* K, const double* Q,
                               const double* V, const double* alpha, const double* eta,
                               const double* theta, const double* gamma, double* M, double* S,
                               double* Y) {
  long n = orc_state_size(g);
  double* gsum = (double*)malloc(sizeof(double) * n);
  double* Gi = (double*)malloc(sizeof(double) * n);
  double* upd = (double*)malloc(sizeof(double) * n);
  double* W = (double*)malloc(sizeof(double) * n);
  double* Wt = (double*)malloc(sizeof(double) * n);
  double* z = (double*)malloc(sizeof(double) * (g->d_v > 0 ? g->d_v : 1));
  int dk = g->d_k, dv = g->d_v, nh = g->n_history;
  for (int t = 0; t < g->N; ++t) {
    /* the memory before the token (the l_q gate renormalises every token) */
    if (g->retention == ORC_RET_LQ) orc_lq_norms(g, M, z);
    orc_memory_of(g, M, z, Wt);
    for (long j = 0; j < n; ++j) gsum[j] = 0.0;
    for (int lag = 0; lag < g->c && t - lag >= -nh; ++lag) {
      int i = t - lag;
      orc_grad(g, Wt, K + (long)(i + nh) * dk, V + (long)(i + nh) * dv, Gi);
      for (long j = 0; j < n; ++j) gsum[j] += gamma[lag] * Gi[j];
    }
    orc_token_step(g, alpha[t], eta[t], theta[t], gsum, Q + (long)t * dk, M, S, upd,
                   Y + (long)t * dv, z, W);
  }
  free(gsum);
  free(Gi);
  free(upd);
  free(W);
  free(Wt);
  free(z);
}

/* ----------------------------------------------------- threads over heads */

typedef struct {
  const orc_cfg* g;
  int recurrent;
  int h0, h1;
  const double *K, *Q, *V, *alpha, *eta, *theta, *gamma;
  double *M, *S, *Y;
} orc_job;

static void* orc_worker(void* p) {
  orc_job* j = (orc_job*)p;
  const orc_cfg* g = j->g;
  long ns = orc_state_size(g);
  for (int h = j->h0; h < j->h1; ++h) {
    const long nkv = (long)g->N + g->n_history;
    const double* K = j->K + (long)h * nkv * g->d_k;
    const double* Q = j->Q + (long)h * g->N * g->d_k;
    const double* V = j->V + (long)h * nkv * g->d_v;
    const double* a = j->alpha + (long)h * g->N;
    const double* e = j->eta + (long)h * g->N;
    const double* th = j->theta + (long)h * g->N;
    double* M = j->M + (long)h * ns;
    double* S = j->S + (long)h * ns;
    double* Y = j->Y + (long)h * g->N * g->d_v;
    if (j->recurrent)
      orc_head_recurrent(g, K, Q, V, a, e, th, j->gamma, M, S, Y);
    else
      orc_head_chunked(g, K, Q, V, a, e, th, j->gamma, M, S, Y);
  }
  return NULL;
}

static int orc_check(const orc_cfg* g) {
  if (g->N < 0 || g->d_k <= 0 || g->d_v <= 0 || g->c < 1 || g->b < 1) return -1;
  if (g->n_history < 0) return -1;
  if (g->mem < ORC_MEM_LINEAR || g->mem > ORC_MEM_MLP_GATED) return -1;
  if (g->mem != ORC_MEM_LINEAR && (g->d_h <= 0 || g->d_k != g->d_v)) return -1;
  if (g->loss < ORC_LOSS_L2 || g->loss > ORC_LOSS_ROBUST) return -1;
  if (g->loss == ORC_LOSS_ROBUST && !(g->loss_param >= 0.0)) return -1;
  if (g->retention < ORC_RET_L2 || g->retention > ORC_RET_LQ) return -1;
  if (g->retention != ORC_RET_L2) {
    if (g->mem != ORC_MEM_LINEAR || g->ns_steps > 0) return -1;
    if (g->retention == ORC_RET_ELASTIC && !(g->ret_param >= 0.0)) return -1;
    if (g->retention == ORC_RET_KL && !(g->ret_param > 0.0)) return -1;
    if (g->retention == ORC_RET_LQ && !(g->ret_param >= 1.0)) return -1;
  }
  if (g->loss == ORC_LOSS_LP && !(g->loss_param >= 1.0 && g->loss_param < 1e6)) return -1;
  if (g->loss == ORC_LOSS_HUBER && !(g->loss_param > 0.0)) return -1;
  if (g->phi == ORC_PHI_POLY) {
    if (g->phi_degree < 1 || g->phi_degree > ORC_PHI_MAX_DEGREE) return -1;
    if (orc_feature_dim(g) < 1) return -1;
  }
  return 0;
}

static int orc_run(const orc_cfg* g, int recurrent, int n_heads, const double* K,
                   const double* Q, const double* V, const double* alpha, const double* eta,
                   const double* theta, const double* gamma, double* M, double* S, double* Y,
                   int n_threads) {
  if (orc_check(g) != 0 || n_heads < 0) return -1;
  if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (n_threads > n_heads) n_threads = n_heads;
  if (n_threads < 1) n_threads = 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * n_threads);
  orc_job* jobs = (orc_job*)malloc(sizeof(orc_job) * n_threads);
  for (int w = 0; w < n_threads; ++w) {
    orc_job j = {g, recurrent, (int)((long)n_heads * w / n_threads),
                 (int)((long)n_heads * (w + 1) / n_threads), K, Q, V, alpha, eta, theta,
                 gamma, M, S, Y};
    jobs[w] = j;
    pthread_create(&th[w], NULL, orc_worker, &jobs[w]);
  }
  for (int w = 0; w < n_threads; ++w) pthread_join(th[w], NULL);
  free(th);
  free(jobs);
  return 0;
}

/* Chunked forward over n_heads independent heads.  K: [heads, n_history + N, d_k]
 * and V: [heads, n_history + N, d_v] (history rows first); Q: [heads, N, d_k];
 * alpha, eta, theta: [heads, N]; gamma: [c] by lag;
 * M, S: [heads, state] in/out (state layout: linear M is d_v x D row-major;
 * MLP is W1 (d x d_h) then W2 (d_h x d)); Y: [heads, N, d_v] out.
 * Returns 0, or -1 on an invalid description. */
int orc_forward_chunked(const orc_cfg* g, int n_heads, const double* K, const double* Q,
                        const double* V, const double* alpha, const double* eta,
                        const double* theta, const double* gamma, double* M, double* S,
                        double* Y, int n_threads) {
  return orc_run(g, 0, n_heads, K, Q, V, alpha, eta, theta, gamma, M, S, Y, n_threads);
}

/* Token-recurrent forward, same arguments (b is ignored). */
int orc_forward_recurrent(const orc_cfg* g, int n_heads, const double* K, const double* Q,
                          const double* V, const double* alpha, const double* eta,
                          const double* theta, const double* gamma, double* M, double* S,
                          double* Y, int n_threads) {
  return orc_run(g, 1, n_heads, K, Q, V, alpha, eta, theta, gamma, M, S, Y, n_threads);
}

/* ============================================================== backward
 *
 * Gradients of a scalar loss on the outputs with respect to every input of
 * the chunked update: the outer loop that trains what the inner loop does not
 * ([ATLAS] "Deep Memory Module": the memory is optimised at test time inside,
 * the projections producing k, q, v and the gates by an outer loop; [Miras]
 * Associative Memory & Attentional Bias, Remark 2).  The loss is
 *     L = sum_t <dY_t, y_t> + <dM_N, M_N> + <dS_N, S_N>
 * for given upstream gradients dY, dM_N, dS_N.  This is the literal reverse of
 * orc_head_chunked for a linear memory (any feature map, bias, window, chunk,
 * momentum; no Newton-Schulz): the chunk-start states are kept, each chunk's
 * token states are recomputed from them, and every step of the forward loop
 * is differentiated in reverse order. */

/* d/de of orc_bias_dy (the second derivative of the bias). */
static double orc_bias_d2(const orc_cfg* g, double e) {
  if (g->loss == ORC_LOSS_LP) {
    const double p = g->loss_param;
    if (p == 2.0) return 2.0;
    if (e == 0.0) return 0.0;  /* the limit for p > 2; undefined for p < 2 */
    return p * (p - 1.0) * pow(fabs(e), p - 2.0);
  }
  if (g->loss == ORC_LOSS_HUBER) return fabs(e) <= g->loss_param ? 2.0 : 0.0;
  return 2.0;
}

typedef struct {
  const orc_cfg* g;
  const double* x;
  const double* dphi;
  double* dx;
} orc_phib_ctx;

/* d(a_e x_{i_1} ... x_{i_e}) / dx_{i_r}: the product of the other factors. */
static void orc_phib_one(void* c, int j, int e, const int* idx) {
  orc_phib_ctx* p = (orc_phib_ctx*)c;
  for (int r = 0; r < e; ++r) {
    double v = p->g->phi_coef[e] * p->dphi[j];
    for (int s = 0; s < e; ++s)
      if (s != r) v *= p->x[idx[s]];
    p->dx[idx[r]] += v;
  }
}

/* dx += (dPhi/dx)^T dphi for the map of orc_phi. */
static void orc_phi_backward(const orc_cfg* g, const double* x, const double* dphi, double* dx) {
  int d = g->d_k;
  if (g->phi == ORC_PHI_POLY) {
    orc_phib_ctx c = {g, x, dphi, dx};
    orc_poly_features(g, orc_phib_one, &c);
    return;
  }
  for (int i = 0; i < d; ++i) dx[i] += dphi[i];
  if (g->phi == ORC_PHI_IDENTITY) return;
  int p = d;
  for (int i = 0; i < d; ++i)
    for (int j = i; j < d; ++j) {
      dx[i] += dphi[p] * x[j];
      dx[j] += dphi[p] * x[i];
      ++p;
    }
}

/* Reverse of orc_grad for a linear memory: given dG (state layout), add the
 * gradients with respect to the state M0 (dM0), the key k (dk) and the value
 * v (dv).  G = psi Phi(k)^T with psi = bias_dy(M0 Phi(k) - v) (dot: -2 v). */
static void orc_grad_backward(const orc_cfg* g, const double* M0, const double* k,
                              const double* v, const double* dG, double* dM0, double* dk,
                              double* dv) {
  int D = orc_feature_dim(g), nv = g->d_v;
  double* f = (double*)malloc(sizeof(double) * D);
  double* df = (double*)calloc(D, sizeof(double));
  orc_phi(g, k, f);
  for (int r = 0; r < nv; ++r) {
    double s = 0.0, dpsi = 0.0;
    for (int j = 0; j < D; ++j) {
      s += M0[(long)r * D + j] * f[j];
      dpsi += dG[(long)r * D + j] * f[j];
    }
    if (g->loss == ORC_LOSS_DOT) {
      for (int j = 0; j < D; ++j) df[j] += dG[(long)r * D + j] * (-2.0 * v[r]);
      dv[r] += -2.0 * dpsi;
      continue;
    }
    const double e = s - v[r];
    const double psi = orc_bias_dy(g, e);
    const double ds = dpsi * orc_bias_d2(g, e);
    dv[r] -= ds;
    for (int j = 0; j < D; ++j) {
      df[j] += dG[(long)r * D + j] * psi + M0[(long)r * D + j] * ds;
      dM0[(long)r * D + j] += ds * f[j];
    }
  }
  orc_phi_backward(g, k, df, dk);
  free(f);
  free(df);
}

static double orc_dot(long n, const double* a, const double* b) {
  double s = 0.0;
  for (long i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}

/* One chunk [t0, t1) forward from (M, S), as orc_head_chunked; with the
 * recording arrays given, the state before each token (Mb, Sb) and its
 * windowed gradient (Gs) are kept, b entries of the state size each. */
static void orc_chunk_forward(const orc_cfg* g, int t0, int t1, const double* K, const double* Q,
                              const double* V, const double* alpha, const double* eta,
                              const double* theta, const double* gamma, double* M, double* S,
                              double* Mb, double* Sb, double* Gs) {
  long n = orc_state_size(g);
  int dk = g->d_k, dv = g->d_v, nh = g->n_history;
  double* M0 = (double*)malloc(sizeof(double) * n);
  double* gsum = (double*)malloc(sizeof(double) * n);
  double* Gi = (double*)malloc(sizeof(double) * n);
  double* upd = (double*)malloc(sizeof(double) * n);
  double* y = (double*)malloc(sizeof(double) * dv);
  double* W = (double*)malloc(sizeof(double) * n);
  memcpy(M0, M, sizeof(double) * n);
  for (int t = t0; t < t1; ++t) {
    for (long j = 0; j < n; ++j) gsum[j] = 0.0;
    int i0 = t - g->c + 1 < -nh ? -nh : t - g->c + 1;
    for (int i = i0; i <= t; ++i) {
      orc_grad(g, M0, K + (long)(i + nh) * dk, V + (long)(i + nh) * dv, Gi);
      for (long j = 0; j < n; ++j) gsum[j] += gamma[t - i] * Gi[j];
    }
    if (Mb) {
      memcpy(Mb + (long)(t - t0) * n, M, sizeof(double) * n);
      memcpy(Sb + (long)(t - t0) * n, S, sizeof(double) * n);
      memcpy(Gs + (long)(t - t0) * n, gsum, sizeof(double) * n);
    }
    orc_token_step(g, alpha[t], eta[t], theta[t], gsum, Q + (long)t * dk, M, S, upd, y, NULL, W);
  }
  free(M0);
  free(gsum);
  free(Gi);
  free(upd);
  free(y);
  free(W);
}

/* Reverse pass of one head.  In: the forward inputs, M and S at the start
 * (M_in, S_in), dY [N, d_v], and dM, dS holding dL/dM_N, dL/dS_N.  Out: dM, dS
 * overwritten with dL/dM_0, dL/dS_0; dK, dV [n_history + N, .], dQ [N, d_k],
 * dalpha, deta, dtheta [N], dgamma [c] (all overwritten). */
static void orc_head_backward(const orc_cfg* g, const double* K, const double* Q,
                              const double* V, const double* alpha, const double* eta,
                              const double* theta, const double* gamma, const double* M_in,
                              const double* S_in, const double* dY, double* dM, double* dS,
                              double* dK, double* dQ, double* dV, double* dalpha, double* deta,
                              double* dtheta, double* dgamma) {
  long n = orc_state_size(g);
  int D = orc_feature_dim(g), dk = g->d_k, dv = g->d_v, nh = g->n_history, b = g->b;
  int nchunks = (g->N + b - 1) / b;
  memset(dK, 0, sizeof(double) * (long)(nh + g->N) * dk);
  memset(dV, 0, sizeof(double) * (long)(nh + g->N) * dv);
  memset(dQ, 0, sizeof(double) * (long)g->N * dk);
  memset(dgamma, 0, sizeof(double) * g->c);
  /* forward once: the state at every chunk start */
  double* Mc = (double*)malloc(sizeof(double) * n * (nchunks > 0 ? nchunks : 1));
  double* Sc = (double*)malloc(sizeof(double) * n * (nchunks > 0 ? nchunks : 1));
  double* M = (double*)malloc(sizeof(double) * n);
  double* S = (double*)malloc(sizeof(double) * n);
  memcpy(M, M_in, sizeof(double) * n);
  memcpy(S, S_in, sizeof(double) * n);
  for (int c = 0; c < nchunks; ++c) {
    int t0 = c * b, t1 = t0 + b < g->N ? t0 + b : g->N;
    memcpy(Mc + (long)c * n, M, sizeof(double) * n);
    memcpy(Sc + (long)c * n, S, sizeof(double) * n);
    orc_chunk_forward(g, t0, t1, K, Q, V, alpha, eta, theta, gamma, M, S, NULL, NULL, NULL);
  }
  double* Mb = (double*)malloc(sizeof(double) * n * b);
  double* Sb = (double*)malloc(sizeof(double) * n * b);
  double* Gs = (double*)malloc(sizeof(double) * n * b);
  double* Mt = (double*)malloc(sizeof(double) * n);
  double* St = (double*)malloc(sizeof(double) * n);
  double* dg = (double*)malloc(sizeof(double) * n);
  double* dG = (double*)malloc(sizeof(double) * n);
  double* Gi = (double*)malloc(sizeof(double) * n);
  double* dMc = (double*)malloc(sizeof(double) * n);
  double* fq = (double*)malloc(sizeof(double) * D);
  double* dfq = (double*)malloc(sizeof(double) * D);
  for (int c = nchunks - 1; c >= 0; --c) {
    int t0 = c * b, t1 = t0 + b < g->N ? t0 + b : g->N;
    const double* M0 = Mc + (long)c * n;
    memcpy(M, M0, sizeof(double) * n);
    memcpy(S, Sc + (long)c * n, sizeof(double) * n);
    orc_chunk_forward(g, t0, t1, K, Q, V, alpha, eta, theta, gamma, M, S, Mb, Sb, Gs);
    for (long j = 0; j < n; ++j) dMc[j] = 0.0;
    for (int t = t1 - 1; t >= t0; --t) {
      const double* Mp = Mb + (long)(t - t0) * n;  /* M_{t-1} */
      const double* Sp = Sb + (long)(t - t0) * n;  /* S_{t-1} */
      const double* gt = Gs + (long)(t - t0) * n;  /* g_t */
      /* the token's states: S_t = eta S_{t-1} - theta g_t, M_t = (1-alpha) M_{t-1} + S_t */
      for (long j = 0; j < n; ++j) {
        St[j] = eta[t] * Sp[j] - theta[t] * gt[j];
        Mt[j] = (1.0 - alpha[t]) * Mp[j] + St[j];
      }
      /* y_t = M_t Phi(q_t) */
      orc_phi(g, Q + (long)t * dk, fq);
      for (int j = 0; j < D; ++j) dfq[j] = 0.0;
      for (int r = 0; r < dv; ++r) {
        const double dy = dY[(long)t * dv + r];
        for (int j = 0; j < D; ++j) {
          dM[(long)r * D + j] += dy * fq[j];
          dfq[j] += Mt[(long)r * D + j] * dy;
        }
      }
      orc_phi_backward(g, Q + (long)t * dk, dfq, dQ + (long)t * dk);
      /* M_t = (1 - alpha_t) M_{t-1} + S_t */
      dalpha[t] = -orc_dot(n, dM, Mp);
      for (long j = 0; j < n; ++j) {
        dS[j] += dM[j];
        dM[j] *= 1.0 - alpha[t];
      }
      /* S_t = eta_t S_{t-1} - theta_t g_t */
      deta[t] = orc_dot(n, dS, Sp);
      dtheta[t] = -orc_dot(n, dS, gt);
      for (long j = 0; j < n; ++j) {
        dg[j] = -theta[t] * dS[j];
        dS[j] *= eta[t];
      }
      /* g_t = sum over the window of gamma[t - i] grad(M0; k_i, v_i) */
      int i0 = t - g->c + 1 < -nh ? -nh : t - g->c + 1;
      for (int i = i0; i <= t; ++i) {
        const double* ki = K + (long)(i + nh) * dk;
        const double* vi = V + (long)(i + nh) * dv;
        orc_grad(g, M0, ki, vi, Gi);
        dgamma[t - i] += orc_dot(n, dg, Gi);
        for (long j = 0; j < n; ++j) dG[j] = gamma[t - i] * dg[j];
        orc_grad_backward(g, M0, ki, vi, dG, dMc, dK + (long)(i + nh) * dk,
                          dV + (long)(i + nh) * dv);
      }
    }
    /* the chunk-start state M0 is the state the previous chunk ended with */
    for (long j = 0; j < n; ++j) dM[j] += dMc[j];
  }
  free(Mc); free(Sc); free(M); free(S); free(Mb); free(Sb); free(Gs); free(Mt); free(St);
  free(dg); free(dG); free(Gi); free(dMc); free(fq); free(dfq);
}

typedef struct {
  const orc_cfg* g;
  int h0, h1;
  const double *K, *Q, *V, *alpha, *eta, *theta, *gamma, *M, *S, *dY;
  double *dM, *dS, *dK, *dQ, *dV, *dalpha, *deta, *dtheta, *dgamma;
} orc_bjob;

static void* orc_bworker(void* p) {
  orc_bjob* j = (orc_bjob*)p;
  const orc_cfg* g = j->g;
  long ns = orc_state_size(g);
  const long nkv = (long)g->N + g->n_history;
  for (int h = j->h0; h < j->h1; ++h) {
    orc_head_backward(g, j->K + h * nkv * g->d_k, j->Q + (long)h * g->N * g->d_k,
                      j->V + h * nkv * g->d_v, j->alpha + (long)h * g->N,
                      j->eta + (long)h * g->N, j->theta + (long)h * g->N, j->gamma,
                      j->M + h * ns, j->S + h * ns, j->dY + (long)h * g->N * g->d_v,
                      j->dM + h * ns, j->dS + h * ns, j->dK + h * nkv * g->d_k,
                      j->dQ + (long)h * g->N * g->d_k, j->dV + h * nkv * g->d_v,
                      j->dalpha + (long)h * g->N, j->deta + (long)h * g->N,
                      j->dtheta + (long)h * g->N, j->dgamma + (long)h * g->c);
  }
  return NULL;
}

/* Backward of orc_forward_chunked over n_heads heads (linear memory without
 * Newton-Schulz; -1 otherwise).  M, S: [heads, state] at the start of the
 * forward; dY: [heads, N, d_v]; dM, dS: [heads, state], in: dL/dM_N, dL/dS_N,
 * out: dL/dM_0, dL/dS_0; dK, dV: [heads, n_history + N, .]; dQ: [heads, N, d_k];
 * dalpha, deta, dtheta: [heads, N]; dgamma: [heads, c] (per head: gamma is
 * shared, so its gradient is the sum over heads). */
int orc_backward_chunked(const orc_cfg* g, int n_heads, const double* K, const double* Q,
                         const double* V, const double* alpha, const double* eta,
                         const double* theta, const double* gamma, const double* M,
                         const double* S, const double* dY, double* dM, double* dS, double* dK,
                         double* dQ, double* dV, double* dalpha, double* deta, double* dtheta,
                         double* dgamma, int n_threads) {
  if (orc_check(g) != 0 || n_heads < 0) return -1;
  if (g->mem != ORC_MEM_LINEAR || g->ns_steps > 0) return -1;
  if (g->retention != ORC_RET_L2 || g->loss == ORC_LOSS_ROBUST) return -1;
  if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (n_threads > n_heads) n_threads = n_heads;
  if (n_threads < 1) n_threads = 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * n_threads);
  orc_bjob* jobs = (orc_bjob*)malloc(sizeof(orc_bjob) * n_threads);
  for (int w = 0; w < n_threads; ++w) {
    orc_bjob j = {g, (int)((long)n_heads * w / n_threads),
                  (int)((long)n_heads * (w + 1) / n_threads), K, Q, V, alpha, eta, theta,
                  gamma, M, S, dY, dM, dS, dK, dQ, dV, dalpha, deta, dtheta, dgamma};
    jobs[w] = j;
    pthread_create(&th[w], NULL, orc_bworker, &jobs[w]);
  }
  for (int w = 0; w < n_threads; ++w) pthread_join(th[w], NULL);
  free(th);
  free(jobs);
  return 0;
}
