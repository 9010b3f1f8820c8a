"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a closed
form the pages state (DeltaNet, linear attention, the chunk equation of the
ATLAS review §3.3, the OmegaNet linear update), an invariant (exact recall of
orthonormal keys, chunk size irrelevant for a state-independent gradient), a
library routine (numpy SVD for Newton-Schulz, scipy's normal CDF for GELU),
finite differences (every gradient) or a brute-force enumeration (the feature
map).  They are chosen so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
from scipy.stats import norm

import oracle

RNG = np.random.default_rng(12345)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_inputs(rng, H, N, d_k, d_v, alpha_hi=0.1, eta=(0.5, 0.9), theta=(0.05, 0.3)):
    K = unit_rows(rng.standard_normal((H, N, d_k)))
    Q = unit_rows(rng.standard_normal((H, N, d_k)))
    V = rng.standard_normal((H, N, d_v))
    a = rng.uniform(0, alpha_hi, (H, N))
    e = rng.uniform(*eta, (H, N)) if eta is not None else np.zeros((H, N))
    t = rng.uniform(*theta, (H, N))
    return K, Q, V, a, e, t


def poly2(x):
    """Brute-force degree-2 feature map from exponent vectors."""
    d = x.shape[-1]
    feats = [x[..., i] for i in range(d)]
    feats += [x[..., i] * x[..., j] for i, j in itertools.combinations_with_replacement(range(d), 2)]
    return np.stack(feats, axis=-1)


# ------------------------------------------------------------------ feature map


def test_phi_poly2_matches_golden_enumeration():
    rows = [list(map(int, l.split())) for l in open(os.path.join(GOLDEN, "phi_poly2_d3.txt"))
            if l.strip() and not l.startswith("#")]
    cfg = oracle.make_cfg(1, 3, 1, phi=oracle.PHI_POLY2)
    assert oracle.feature_dim(cfg) == len(rows) == 9
    x = np.array([2.0, 3.0, 5.0])  # distinct primes: each monomial has a unique value
    f = oracle.phi(cfg, x)
    for idx, *expo in rows:
        assert f[idx] == np.prod(x ** np.array(expo))


def test_phi_poly2_count_and_order_d32():
    cfg = oracle.make_cfg(1, 32, 1, phi=oracle.PHI_POLY2)
    assert oracle.feature_dim(cfg) == 560  # 32 + 32*33/2
    x = RNG.standard_normal(32)
    np.testing.assert_array_equal(oracle.phi(cfg, x), poly2(x))


def test_phi_identity():
    cfg = oracle.make_cfg(1, 5, 2)
    x = RNG.standard_normal(5)
    np.testing.assert_array_equal(oracle.phi(cfg, x), x)


# ------------------------------------------------------------------------ GELU


@pytest.mark.parametrize("x", [-6.0, -2.5, -1.0, -0.3, 0.0, 0.2, 0.7, 1.5, 4.0])
def test_gelu_is_x_times_normal_cdf(x):
    assert abs(oracle.gelu(x) - x * norm.cdf(x)) < 1e-15 * max(1.0, abs(x))


@pytest.mark.parametrize("x", [-3.0, -1.2, -0.1, 0.0, 0.4, 1.1, 2.7])
def test_gelu_prime_by_finite_differences(x):
    h = 1e-5
    fd = ((x + h) * norm.cdf(x + h) - (x - h) * norm.cdf(x - h)) / (2 * h)
    assert abs(oracle.gelu_prime(x) - fd) < 1e-9


# ---------------------------------------------------------------- gradients


def _loss(cfg, state, k, v):
    """The attentional biases written out: l2 and dot (Titans Objective, Miras
    Associative Memory), l_p and Huber (Miras #1 Alternative Attentional Biases;
    Huber per coordinate, equal to e^2 inside the threshold)."""
    y = oracle.memory_apply(cfg, state, k)
    e = y - v
    if cfg.loss == oracle.LOSS_DOT:
        return -2.0 * float(np.dot(y, v))
    if cfg.loss == oracle.LOSS_LP:
        return float(np.sum(np.abs(e) ** cfg.loss_param))
    if cfg.loss == oracle.LOSS_HUBER:
        d = cfg.loss_param
        a = np.abs(e)
        return float(np.sum(np.where(a <= d, e ** 2, 2 * d * a - d * d)))
    return float(np.sum(e ** 2))


def _fd_grad(cfg, state, k, v, h=1e-6):
    g = np.zeros_like(state)
    for j in range(state.size):
        sp, sm = state.copy(), state.copy()
        sp[j] += h
        sm[j] -= h
        g[j] = (_loss(cfg, sp, k, v) - _loss(cfg, sm, k, v)) / (2 * h)
    return g


BIASES = [(oracle.LOSS_L2, 0.0), (oracle.LOSS_DOT, 0.0), (oracle.LOSS_LP, 3.0),
          (oracle.LOSS_LP, 1.5), (oracle.LOSS_HUBER, 0.4)]


MLPS = [oracle.MEM_MLP, oracle.MEM_MLP_LN, oracle.MEM_MLP_GATED]


@pytest.mark.parametrize("mem", MLPS)
@pytest.mark.parametrize("loss,prm", BIASES)
def test_mlp_gradient_by_finite_differences(mem, loss, prm):
    """Every MLP memory (plain, layer-normalised, gated) and every bias: the
    backpropagated gradient against central differences of the written-out loss."""
    d, dh = 4, 6
    cfg = oracle.make_cfg(1, d, d, dh, mem=mem, loss=loss, loss_param=prm)
    state = RNG.standard_normal(oracle.state_size(cfg)) * 0.7
    k, v = RNG.standard_normal(d), RNG.standard_normal(d)
    np.testing.assert_allclose(oracle.grad(cfg, state, k, v), _fd_grad(cfg, state, k, v),
                               rtol=1e-7, atol=1e-8)


@pytest.mark.parametrize("phi", [oracle.PHI_IDENTITY, oracle.PHI_POLY2])
@pytest.mark.parametrize("loss,prm", BIASES)
def test_linear_gradient_by_finite_differences(phi, loss, prm):
    d_k, d_v = 3, 4
    cfg = oracle.make_cfg(1, d_k, d_v, phi=phi, loss=loss, loss_param=prm)
    D = oracle.feature_dim(cfg)
    state = RNG.standard_normal(d_v * D)
    k, v = RNG.standard_normal(d_k), RNG.standard_normal(d_v)
    np.testing.assert_allclose(oracle.grad(cfg, state, k, v), _fd_grad(cfg, state, k, v),
                               rtol=1e-7, atol=1e-8)


@pytest.mark.parametrize("mem", [oracle.MEM_LINEAR, oracle.MEM_MLP])
def test_lp_with_p2_and_huber_with_a_huge_threshold_are_the_l2_bias(mem):
    """|e|^2 is e^2, and a Huber threshold above every error never clips: both
    runs must equal the l2 run to the last bit (the gradient 2 |e| sign(e) and
    2 e are the same number)."""
    H, N, d, dh = 2, 37, 4, 8
    rng = np.random.default_rng(5)
    K, Q, V, a, e, t = rand_inputs(rng, H, N, d, d, theta=(0.005, 0.03))  # bounded trajectory
    kw = dict(c=3, b=4, d_h=dh if mem == oracle.MEM_MLP else 0, mem=mem)
    M0 = None if mem == oracle.MEM_LINEAR else rng.standard_normal((H, 2 * d * dh)) * 0.1
    base = run(oracle.make_cfg(N, d, d, **kw), K, Q, V, a, e, t, np.ones(3), M0)
    for loss, prm in ((oracle.LOSS_LP, 2.0), (oracle.LOSS_HUBER, 1e300)):
        out = run(oracle.make_cfg(N, d, d, loss=loss, loss_param=prm, **kw), K, Q, V, a, e, t,
                  np.ones(3), M0)
        for x, y in zip(out, base):
            assert np.isfinite(y).all() and np.array_equal(x, y)


@pytest.mark.parametrize("loss,prm,step", [
    (oracle.LOSS_HUBER, 0.05, lambda v, prm: 2 * prm * np.sign(v)),  # every |v| > delta: clipped
    (oracle.LOSS_LP, 1.0, lambda v, prm: np.sign(v)),                # sign of the error only
    (oracle.LOSS_LP, 3.0, lambda v, prm: 3 * v * np.abs(v)),
])
def test_first_token_under_the_alternative_biases(loss, prm, step):
    """From M_0 = 0, S_0 = 0 the first error is e = -v, so
    S_1 = -theta_1 dl/dM = theta_1 psi(v) k^T with psi the bias derivative, and
    y_1 = (1 - alpha_1) 0 + S_1 q = theta_1 (k . q) psi(v): Huber's
    2 delta sign(v) beyond the threshold, l_1's sign(v) (the pages' value-less
    +-1 memory), l_3's 3 v |v|."""
    H, N, d = 3, 1, 5
    rng = np.random.default_rng(9)
    K, Q, _, a, e, t = rand_inputs(rng, H, N, d, d)
    V = np.sign(rng.standard_normal((H, N, d))) * rng.uniform(0.2, 1.5, (H, N, d))
    cfg = oracle.make_cfg(N, d, d, loss=loss, loss_param=prm)
    Y, M, S = run(cfg, K, Q, V, a, e, t, np.ones(1))
    for h in range(H):
        k, q, v = K[h, 0], Q[h, 0], V[h, 0]
        ref = t[h, 0] * np.dot(k, q) * step(v, prm)
        np.testing.assert_allclose(Y[h, 0], ref, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(M[h].reshape(d, d), t[h, 0] * np.outer(step(v, prm), k),
                                   rtol=1e-13, atol=1e-15)


def test_invalid_bias_parameters_are_rejected():
    K, Q, V, a, e, t = rand_inputs(RNG, 1, 4, 3, 3)
    for loss, prm in ((oracle.LOSS_LP, 0.5), (oracle.LOSS_HUBER, 0.0), (7, 1.0)):
        with pytest.raises(Exception):
            run(oracle.make_cfg(4, 3, 3, loss=loss, loss_param=prm), K, Q, V, a, e, t, np.ones(1))


def test_mlp_memory_apply_residual_form():
    """With W1 = 0 the residual MLP memory is the identity map."""
    d, dh = 5, 7
    cfg = oracle.make_cfg(1, d, d, dh, mem=oracle.MEM_MLP)
    state = np.concatenate([np.zeros(d * dh), RNG.standard_normal(dh * d)])
    x = RNG.standard_normal(d)
    np.testing.assert_array_equal(oracle.memory_apply(cfg, state, x), x)
    # and with W2 = I-like rows and W1 = [I 0], the output is x + GELU(x)
    dh = d
    W1 = np.eye(d)
    W2 = np.eye(d)
    cfg = oracle.make_cfg(1, d, d, dh, mem=oracle.MEM_MLP)
    y = oracle.memory_apply(cfg, np.concatenate([W1.ravel(), W2.ravel()]), x)
    np.testing.assert_allclose(y, x + x * norm.cdf(x), rtol=0, atol=1e-15)


def test_layer_normalised_memory_is_ln_of_the_plain_branch():
    """M_LN(x) - x is the plain branch M(x) - x = W1 GELU(W2 x) normalised to zero
    mean and unit variance (biased variance over the d outputs, eps 1e-5 inside
    the square root), with the same W1, W2."""
    d, dh = 6, 9
    state = RNG.standard_normal(2 * d * dh) * 0.6
    x = RNG.standard_normal(d)
    u = oracle.memory_apply(oracle.make_cfg(1, d, d, dh, mem=oracle.MEM_MLP), state, x) - x
    y = oracle.memory_apply(oracle.make_cfg(1, d, d, dh, mem=oracle.MEM_MLP_LN), state, x)
    ref = (u - u.mean()) / np.sqrt(u.var() + 1e-5)
    np.testing.assert_allclose(y - x, ref, rtol=0, atol=1e-13)
    assert abs((y - x).mean()) < 1e-13


def test_gated_memory_reduces_to_the_plain_one_when_the_gate_is_one():
    """x = e_0 and W3 with a first column of ones give W3 x = 1 for every hidden
    unit: the gated memory x + W1 (GELU(W2 x) * (W3 x)) equals the plain one.  With
    W3 = 0 it is the identity, and only W3's gradient is non-zero."""
    d, dh = 5, 7
    W12 = RNG.standard_normal(2 * d * dh) * 0.6
    W3 = RNG.standard_normal((dh, d))
    W3[:, 0] = 1.0
    x = np.zeros(d)
    x[0] = 1.0
    plain = oracle.memory_apply(oracle.make_cfg(1, d, d, dh, mem=oracle.MEM_MLP), W12, x)
    cfg = oracle.make_cfg(1, d, d, dh, mem=oracle.MEM_MLP_GATED)
    gated = oracle.memory_apply(cfg, np.concatenate([W12, W3.ravel()]), x)
    np.testing.assert_allclose(gated, plain, rtol=0, atol=1e-15)
    state = np.concatenate([W12, np.zeros(dh * d)])
    k, v = RNG.standard_normal(d), RNG.standard_normal(d)
    np.testing.assert_array_equal(oracle.memory_apply(cfg, state, k), k)
    G = oracle.grad(cfg, state, k, v)
    assert not G[:2 * d * dh].any() and G[2 * d * dh:].any()


# ------------------------------------------------------------- Newton-Schulz

NS = (3.4445, -4.7750, 2.0315)


@pytest.mark.parametrize("shape", [(6, 10), (10, 6), (8, 8)])
def test_newton_schulz_acts_on_singular_values(shape):
    """NS commutes with the SVD: NS(S) = U p^(5)(Sigma / (||S||_F + eps)) V^T for
    the scalar quintic p(s) = a s + b s^3 + c s^5."""
    S = RNG.standard_normal(shape)
    eps = 1e-7
    out = oracle.newton_schulz(S, 5, *NS, eps)
    U, s, Vt = np.linalg.svd(S, full_matrices=False)
    x = s / (np.linalg.norm(S) + eps)
    for _ in range(5):
        x = NS[0] * x + NS[1] * x ** 3 + NS[2] * x ** 5
    np.testing.assert_allclose(out, (U * x) @ Vt, rtol=0, atol=1e-12)


def test_newton_schulz_zero_input_is_zero():
    out = oracle.newton_schulz(np.zeros((4, 6)), 5, *NS, 1e-7)
    assert np.all(out == 0.0)


# ---------------------------------------------------------- forward: closed forms


def run(cfg, K, Q, V, a, e, t, gamma, M0=None, S0=None, recurrent=False):
    return oracle.forward(cfg, K, Q, V, a, e, t, gamma, M0, S0, recurrent=recurrent)


@pytest.mark.parametrize("b", [1, 3])
def test_deltanet_reduction(b):
    """Linear memory, c = 1, eta = 0: M_t = (1 - alpha_t) M_{t-1} + beta_t (v_t - M_{t-1} k_t) k_t^T
    with beta_t = 2 theta_t (DeltaNet with a forget gate; the ATLAS review's
    Introduction and the Miras post's Background state the rule).  Only b = 1
    is the delta rule; for b = 3 the check is on the first token of each
    chunk only, where M_{t-1} is the chunk-start state."""
    H, N, d = 2, 12, 6
    K, Q, V, a, _, t = rand_inputs(RNG, H, N, d, d)
    e = np.zeros((H, N))
    cfg = oracle.make_cfg(N, d, d, c=1, b=b)
    Y, M, _ = run(cfg, K, Q, V, a, e, t, np.ones(1))
    for h in range(H):
        Mr = np.zeros((d, d))
        for i in range(N):
            k, v = K[h, i], V[h, i]
            Mr = (1 - a[h, i]) * Mr + 2 * t[h, i] * np.outer(v - Mr @ k, k)
            if b == 1 or i % b == 0:
                np.testing.assert_allclose(Y[h, i], Mr @ Q[h, i], rtol=0, atol=1e-12)
            if b != 1 and i % b == 0:
                break
        if b == 1:
            np.testing.assert_allclose(M[h].reshape(d, d), Mr, rtol=0, atol=1e-12)


@pytest.mark.parametrize("b", [1, 4, 16])
def test_linear_attention_reduction(b):
    """Dot-product bias, c = 1, alpha = eta = 0, theta = 1/2: one GD step on
    -2<M k, v> adds v k^T, so y_t = sum_{i<=t} (k_i . q_t) v_i -- causal linear
    attention (Miras post, Background and Associative Memory) -- for any b."""
    H, N, d_k, d_v = 2, 16, 5, 3
    K, Q, V, _, _, _ = rand_inputs(RNG, H, N, d_k, d_v)
    z = np.zeros((H, N))
    cfg = oracle.make_cfg(N, d_k, d_v, c=1, b=b, loss=oracle.LOSS_DOT)
    Y, M, _ = run(cfg, K, Q, V, z, z, z + 0.5, np.ones(1))
    for h in range(H):
        ref = np.tril(Q[h] @ K[h].T) @ V[h]
        np.testing.assert_allclose(Y[h], ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(M[h].reshape(d_v, d_k), V[h].T @ K[h], rtol=0, atol=1e-12)


def gated_window_matrix(a, e, t, gamma, N):
    """A[t, i]: weight of v_i phi_i^T in M_t when every gradient is -2 v phi^T:
    M_t = sum_m Pa(t,m) S_m, S_m = sum_{m'} Pe(m,m') theta_{m'} g_{m'},
    g_{m'} = -2 sum_j gamma_j v_{m'-j} phi_{m'-j}^T."""
    c = len(gamma)
    Pa = np.zeros((N, N))
    Pe = np.zeros((N, N))
    for i in range(N):
        for j in range(i + 1):
            Pa[i, j] = np.prod(1 - a[j + 1:i + 1])
            Pe[i, j] = np.prod(e[j + 1:i + 1])
    G = np.zeros((N, N))
    for m in range(N):
        for lag in range(c):
            if m - lag >= 0:
                G[m, m - lag] = gamma[lag]
    return 2.0 * Pa @ Pe @ np.diag(t) @ G


@pytest.mark.parametrize("b", [1, 5, 32])
@pytest.mark.parametrize("phi", [oracle.PHI_IDENTITY, oracle.PHI_POLY2])
def test_dot_loss_gated_attention_closed_form(b, phi):
    """With a state-independent gradient the momentum, decay and window unroll
    into a masked attention: y_t = sum_i A[t,i] (phi(k_i) . phi(q_t)) v_i.
    Pins the momentum recursion, the (1 - alpha) decay, the lag indexing of
    gamma and the window clipping at the first token, for any chunk size."""
    H, N, d_k, d_v, c = 2, 21, 3, 4, 4
    K, Q, V, a, e, t = rand_inputs(RNG, H, N, d_k, d_v)
    gamma = RNG.uniform(0.2, 1.0, c)
    cfg = oracle.make_cfg(N, d_k, d_v, c=c, b=b, phi=phi, loss=oracle.LOSS_DOT)
    Y, _, _ = run(cfg, K, Q, V, a, e, t, gamma)
    f = (lambda x: poly2(x)) if phi == oracle.PHI_POLY2 else (lambda x: x)
    for h in range(H):
        A = gated_window_matrix(a[h], e[h], t[h], gamma, N)
        ref = (A * (f(Q[h]) @ f(K[h]).T)) @ V[h]
        np.testing.assert_allclose(Y[h], ref, rtol=0, atol=1e-11)


@pytest.mark.parametrize("b,c", [(4, 3), (5, 1), (7, 8)])
def test_chunk_equation_without_momentum(b, c):
    """ATLAS review §3.3 chunk equation (eta = 0), read with the chunk-start
    state t' and gamma by lag:
        M_t = prod_{j=t'+1..t}(1-alpha_j) M_{t'}
              - sum_{n=t'+1..t} prod_{j=n+1..t}(1-alpha_j) theta_n
                  sum_{i=n-c+1..n} gamma_{n-i} grad l(M_{t'}; k_i, v_i),
    grad l(M; k, v) = 2 (M k - v) k^T.  Checked on Y and the final state, with a
    ragged last chunk."""
    H, N, d_k, d_v = 2, 23, 5, 4
    K, Q, V, a, _, t = rand_inputs(RNG, H, N, d_k, d_v)
    e = np.zeros((H, N))
    gamma = RNG.uniform(0.3, 1.0, c)
    cfg = oracle.make_cfg(N, d_k, d_v, c=c, b=b)
    M0 = RNG.standard_normal((H, d_v * d_k)) * 0.3
    Y, M, _ = run(cfg, K, Q, V, a, e, t, gamma, M0=M0)
    for h in range(H):
        Ms = M0[h].reshape(d_v, d_k).copy()
        for t0 in range(0, N, b):
            Mc = Ms.copy()
            t1 = min(N, t0 + b)
            for tt in range(t0, t1):
                Mt = np.prod(1 - a[h, t0:tt + 1]) * Mc
                for n in range(t0, tt + 1):
                    gs = sum(gamma[n - i] * 2 * np.outer(Mc @ K[h, i] - V[h, i], K[h, i])
                             for i in range(max(0, n - c + 1), n + 1))
                    Mt = Mt - np.prod(1 - a[h, n + 1:tt + 1]) * t[h, n] * gs
                np.testing.assert_allclose(Y[h, tt], Mt @ Q[h, tt], rtol=0, atol=1e-11)
                Ms = Mt
        np.testing.assert_allclose(M[h].reshape(d_v, d_k), Ms, rtol=0, atol=1e-11)


@pytest.mark.parametrize("b,c", [(6, 3), (4, 1), (1, 5)])
@pytest.mark.parametrize("phi", [oracle.PHI_IDENTITY, oracle.PHI_POLY2])
def test_chunk_momentum_sum_form(b, c, phi):
    """With momentum the chunk unrolls to sums over the chunk's tokens:
        S_n = (prod_{m<=n} eta_m) S0 - sum_{m<=n} prod_{m<l<=n} eta_l theta_m g_m,
        M_n = (prod_{m<=n}(1-alpha_m)) M0 + sum_{m<=n} prod_{m<l<=n}(1-alpha_l) S_m,
    g_m = sum_j gamma_j 2 (M0 phi_{m-j} - v_{m-j}) phi_{m-j}^T at the chunk-start
    M0 (Titans review, Surprise Metric and Forgetting Mechanism; ATLAS review
    §3.3).  The oracle applies the recursion token by token; this sums it."""
    H, N, d_k, d_v = 2, 19, 3, 4
    K, Q, V, a, e, t = rand_inputs(RNG, H, N, d_k, d_v)
    gamma = RNG.uniform(0.3, 1.0, c)
    cfg = oracle.make_cfg(N, d_k, d_v, c=c, b=b, phi=phi)
    D = oracle.feature_dim(cfg)
    M0 = RNG.standard_normal((H, d_v * D)) * 0.2
    S0 = RNG.standard_normal((H, d_v * D)) * 0.2
    Y, M, S = run(cfg, K, Q, V, a, e, t, gamma, M0=M0, S0=S0)
    f = (lambda x: poly2(x)) if phi == oracle.PHI_POLY2 else (lambda x: x)
    for h in range(H):
        Mc, Sc = M0[h].reshape(d_v, D).copy(), S0[h].reshape(d_v, D).copy()
        P = f(K[h])
        for t0 in range(0, N, b):
            t1 = min(N, t0 + b)
            g = {}
            for m in range(t0, t1):
                g[m] = sum(gamma[m - i] * 2 * np.outer(Mc @ P[i] - V[h, i], P[i])
                           for i in range(max(0, m - c + 1), m + 1))
            Sn = {}
            for n in range(t0, t1):
                Sn[n] = np.prod(e[h, t0:n + 1]) * Sc - sum(
                    np.prod(e[h, m + 1:n + 1]) * t[h, m] * g[m] for m in range(t0, n + 1))
                Mn = np.prod(1 - a[h, t0:n + 1]) * Mc + sum(
                    np.prod(1 - a[h, m + 1:n + 1]) * Sn[m] for m in range(t0, n + 1))
                np.testing.assert_allclose(Y[h, n], Mn @ f(Q[h, n]), rtol=0, atol=1e-11)
            Mc, Sc = Mn, Sn[t1 - 1]
        np.testing.assert_allclose(M[h].reshape(d_v, D), Mc, rtol=0, atol=1e-11)
        np.testing.assert_allclose(S[h].reshape(d_v, D), Sc, rtol=0, atol=1e-11)


def test_omeganet_linear_update_reading():
    """ATLAS review §3.2 OmegaNet linear update, read as (see design notes):
    M_t = M_{t-1} ((1-alpha_t) I - 2 theta_t sum_i gamma phi_i phi_i^T)
          + 2 theta_t sum_i gamma v_i phi_i^T   (b = 1, eta = 0)."""
    H, N, d_k, d_v, c = 1, 15, 4, 3, 3
    K, Q, V, a, _, t = rand_inputs(RNG, H, N, d_k, d_v)
    e = np.zeros((H, N))
    gamma = RNG.uniform(0.3, 1.0, c)
    cfg = oracle.make_cfg(N, d_k, d_v, c=c, b=1, phi=oracle.PHI_POLY2)
    Y, _, _ = run(cfg, K, Q, V, a, e, t, gamma)
    P = poly2(K[0])
    D = P.shape[1]
    Mr = np.zeros((d_v, D))
    for n in range(N):
        win = range(max(0, n - c + 1), n + 1)
        A = sum(gamma[n - i] * np.outer(P[i], P[i]) for i in win)
        B = sum(gamma[n - i] * np.outer(V[0, i], P[i]) for i in win)
        Mr = Mr @ ((1 - a[0, n]) * np.eye(D) - 2 * t[0, n] * A) + 2 * t[0, n] * B
        np.testing.assert_allclose(Y[0, n], Mr @ poly2(Q[0, n]), rtol=0, atol=1e-12)


@pytest.mark.parametrize("c,b", [(1, 1), (4, 1), (1, 16)])
def test_orthonormal_keys_recalled_exactly(c, b):
    """A d_v x d_k matrix memory stores d_k pairs with orthonormal keys exactly
    (ATLAS review §3.1, capacity of the l2 bias): theta = 1/2, alpha = eta = 0.
    With b = 1 earlier window terms have zero gradient once stored, so any c
    recalls; with c = 1 every gradient at M0 = 0 adds v k^T, so any b does."""
    d_k, d_v = 16, 7
    Qm, _ = np.linalg.qr(RNG.standard_normal((d_k, d_k)))
    K = Qm.T[None]  # rows orthonormal
    V = RNG.standard_normal((1, d_k, d_v))
    z = np.zeros((1, d_k))
    gamma = np.concatenate([[1.0], RNG.uniform(0.2, 1.0, c - 1)])  # gamma_0 = 1
    cfg = oracle.make_cfg(d_k, d_k, d_v, c=c, b=b)
    _, M, _ = run(cfg, K, K, V, z, z, z + 0.5, gamma)
    np.testing.assert_allclose(K[0] @ M[0].reshape(d_v, d_k).T, V[0], rtol=0, atol=1e-12)


def _ns_scalar(s, steps=5):
    for _ in range(steps):
        s = NS[0] * s + NS[1] * s ** 3 + NS[2] * s ** 5
    return s


@pytest.mark.parametrize("mem", [oracle.MEM_LINEAR, oracle.MEM_MLP, oracle.MEM_MLP_LN,
                                 oracle.MEM_MLP_GATED])
def test_first_step_with_newton_schulz(mem):
    """First token from S0 = 0: S_1 = -theta_1 grad, a rank-1 matrix per weight,
    whose Newton-Schulz image is p^(5)(s/(s+eps)) times its direction; so
    M_1 = (1 - alpha_1) M_0 - p5 grad/||grad||_F per weight matrix (ATLAS
    summary §5, Muon in place of GD, as read in the design notes)."""
    d, dh, eps = 4, 6, 1e-7
    if mem != oracle.MEM_LINEAR:
        cfg = oracle.make_cfg(1, d, d, dh, mem=mem, c=1, b=1, ns_steps=5, ns_a=NS[0],
                              ns_b=NS[1], ns_c=NS[2], ns_eps=eps)
        nb = 3 if mem == oracle.MEM_MLP_GATED else 2
        M0 = RNG.standard_normal((1, nb * d * dh)) * 0.5
        blocks = [slice(i * d * dh, (i + 1) * d * dh) for i in range(nb)]
    else:
        cfg = oracle.make_cfg(1, d, 3, c=1, b=1, ns_steps=5, ns_a=NS[0], ns_b=NS[1],
                              ns_c=NS[2], ns_eps=eps)
        M0 = RNG.standard_normal((1, 3 * d)) * 0.5
        blocks = [slice(0, 3 * d)]
    k = unit_rows(RNG.standard_normal((1, 1, d)))
    q = unit_rows(RNG.standard_normal((1, 1, d)))
    v = RNG.standard_normal((1, 1, cfg.d_v))
    a, e, t = np.array([[0.07]]), np.array([[0.6]]), np.array([[0.3]])
    Y, M, _ = run(cfg, k, q, v, a, e, t, np.ones(1), M0=M0)
    G = oracle.grad(cfg, M0[0], k[0, 0], v[0, 0])
    ref = (1 - 0.07) * M0[0]
    for sl in blocks:
        s = 0.3 * np.linalg.norm(G[sl])
        ref[sl] -= _ns_scalar(s / (s + eps)) * G[sl] / np.linalg.norm(G[sl])
    np.testing.assert_allclose(M[0], ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Y[0, 0], oracle.memory_apply(cfg, ref, q[0, 0]), rtol=0,
                               atol=1e-12)


# ------------------------------------------------- cross-checks of the two loops


@pytest.mark.parametrize("kind", ["linear", "poly2", "mlp", "mlp_ns", "linear_ns"])
def test_chunk_size_one_equals_token_recurrence(kind):
    """b = 1 in the chunked loop is the token recurrence (the chunk-start state
    is then the state right before each token)."""
    H, N, c = 2, 9, 3
    kw = dict(c=c, b=1)
    d_k, d_v, dh = 4, 4, 0
    if kind == "poly2":
        kw["phi"] = oracle.PHI_POLY2
        d_v = 3
    if kind.startswith("mlp"):
        dh = 6
        kw.update(mem=oracle.MEM_MLP)
    if kind.endswith("_ns"):
        kw.update(ns_steps=5, ns_a=NS[0], ns_b=NS[1], ns_c=NS[2], ns_eps=1e-7)
    cfg = oracle.make_cfg(N, d_k, d_v, dh, **kw)
    K, Q, V, a, e, t = rand_inputs(RNG, H, N, d_k, d_v)
    gamma = RNG.uniform(0.3, 1.0, c)
    M0 = RNG.standard_normal((H, oracle.state_size(cfg))) * 0.1
    Yc, Mc, Sc = run(cfg, K, Q, V, a, e, t, gamma, M0=M0)
    Yr, Mr, Sr = run(cfg, K, Q, V, a, e, t, gamma, M0=M0, recurrent=True)
    np.testing.assert_allclose(Yc, Yr, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Mc, Mr, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Sc, Sr, rtol=0, atol=1e-12)


def test_chunked_differs_from_recurrence_for_l2():
    """Sanity: for the l2 bias a chunk of b > 1 is an approximation, so the two
    loops must differ (catches a chunked loop that silently re-reads M)."""
    H, N, d = 1, 16, 4
    cfg = oracle.make_cfg(N, d, d, c=2, b=8)
    K, Q, V, a, e, t = rand_inputs(RNG, H, N, d, d)
    Yc, _, _ = run(cfg, K, Q, V, a, e, t, np.ones(2))
    Yr, _, _ = run(cfg, K, Q, V, a, e, t, np.ones(2), recurrent=True)
    assert np.abs(Yc - Yr).max() > 1e-6
    np.testing.assert_allclose(Yc[0, 0], Yr[0, 0], rtol=0, atol=1e-14)


def test_heads_are_independent_and_threading_is_deterministic():
    H, N, d = 5, 10, 3
    cfg = oracle.make_cfg(N, d, d, c=2, b=4)
    K, Q, V, a, e, t = rand_inputs(RNG, H, N, d, d)
    Y1, M1, _ = oracle.forward(cfg, K, Q, V, a, e, t, np.ones(2), n_threads=1)
    Y3, M3, _ = oracle.forward(cfg, K, Q, V, a, e, t, np.ones(2), n_threads=3)
    np.testing.assert_array_equal(Y1, Y3)
    Ys, _, _ = oracle.forward(cfg, K[2:3], Q[2:3], V[2:3], a[2:3], e[2:3], t[2:3], np.ones(2))
    np.testing.assert_array_equal(Ys[0], Y1[2])


def test_empty_sequence():
    cfg = oracle.make_cfg(0, 3, 3, c=2, b=4)
    z3 = np.zeros((2, 0, 3))
    z = np.zeros((2, 0))
    M0 = RNG.standard_normal((2, 9))
    Y, M, S = run(cfg, z3, z3, z3, z, z, z, np.ones(2), M0=M0)
    assert Y.shape == (2, 0, 3)
    np.testing.assert_array_equal(M, M0)


# ---------------------------------------------------------------- history rows

def _split_run(cfg_kw, K, Q, V, a, e, t, gamma, T, M0=None):
    """One call over tokens [0, T) and a second over [T, N) whose K, V carry the
    last c - 1 tokens of the first part as history, M and S handed over."""
    N, c = K.shape[1], cfg_kw["c"]
    d_k, d_v = K.shape[2], V.shape[2]
    c1 = oracle.make_cfg(T, d_k, d_v, **cfg_kw)
    Y1, M1, S1 = oracle.forward(c1, K[:, :T], Q[:, :T], V[:, :T], a[:, :T], e[:, :T], t[:, :T],
                                gamma, M0=M0)
    nh = min(c - 1, T)
    c2 = oracle.make_cfg(N - T, d_k, d_v, n_history=nh, **cfg_kw)
    Y2, M2, S2 = oracle.forward(c2, K[:, T - nh:], Q[:, T:], V[:, T - nh:], a[:, T:], e[:, T:],
                                t[:, T:], gamma, M0=M1, S0=S1)
    return np.concatenate([Y1, Y2], axis=1), M2, S2


@pytest.mark.parametrize("kw,T", [
    (dict(c=4, b=1), 7),                                          # exact recurrence
    (dict(c=5, b=8), 16),                                         # chunked, split on a chunk edge
    (dict(c=12, b=4, phi=oracle.PHI_POLY2), 8),                   # window longer than both parts' chunk
    (dict(c=3, b=4, mem=oracle.MEM_MLP, d_h=6), 8),               # MLP memory
    (dict(c=3, b=2, mem=oracle.MEM_MLP, d_h=6, ns_steps=3, ns_a=3.4445, ns_b=-4.775,
          ns_c=2.0315, ns_eps=1e-7), 6),                          # Newton-Schulz momentum
])
def test_history_rows_make_a_split_call_exact(kw, T):
    """Tokens only enter later windows through history rows: a sequence split on a
    chunk boundary into two calls, the second carrying the first part's last c - 1
    keys and values as history and its state, reproduces one call over all of it."""
    rng = np.random.default_rng(3)
    d_k = 3 if kw.get("phi") == oracle.PHI_POLY2 else 4
    d_v = d_k if kw.get("mem") == oracle.MEM_MLP else 3
    N = T + 9
    K, Q, V, a, e, t = rand_inputs(rng, 2, N, d_k, d_v)
    gamma = np.exp(-np.arange(kw["c"]) / 3.0)
    M0 = None
    if kw.get("mem") == oracle.MEM_MLP:
        M0 = rng.standard_normal((2, 2 * d_k * kw["d_h"])) * 0.3
    Yf, Mf, Sf = oracle.forward(oracle.make_cfg(N, d_k, d_v, **kw), K, Q, V, a, e, t, gamma, M0=M0)
    Ys, Ms, Ss = _split_run(kw, K, Q, V, a, e, t, gamma, T, M0=M0)
    np.testing.assert_allclose(Ys, Yf, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(Ms, Mf, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(Ss, Sf, rtol=1e-10, atol=1e-12)


def test_history_beyond_the_window_is_ignored():
    rng = np.random.default_rng(4)
    K, Q, V, a, e, t = rand_inputs(rng, 1, 20, 4, 3)
    gamma = np.ones(4)
    kw = dict(c=4, b=2)
    c3 = oracle.make_cfg(10, 4, 3, n_history=3, **kw)
    c9 = oracle.make_cfg(10, 4, 3, n_history=9, **kw)
    Y3, M3, S3 = oracle.forward(c3, K[:, 7:], Q[:, 10:], V[:, 7:], a[:, 10:], e[:, 10:], t[:, 10:],
                                gamma)
    Y9, M9, S9 = oracle.forward(c9, K[:, 1:], Q[:, 10:], V[:, 1:], a[:, 10:], e[:, 10:], t[:, 10:],
                                gamma)
    np.testing.assert_array_equal(Y3, Y9)
    np.testing.assert_array_equal(M3, M9)
    # and a history row inside the window does change the result
    c0 = oracle.make_cfg(10, 4, 3, **kw)
    Y0, _, _ = oracle.forward(c0, K[:, 10:], Q[:, 10:], V[:, 10:], a[:, 10:], e[:, 10:], t[:, 10:],
                              gamma)
    assert np.abs(Y0 - Y3).max() > 1e-3
