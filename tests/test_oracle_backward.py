"""Pins of the backward oracle (the outer-loop gradients through the chunked
update of a linear memory).

Two independent checks:
- central finite differences of the forward oracle's scalar loss
  L = sum <dY, Y> + <dM_N, M_N> + <dS_N, S_N> with respect to every input
  (K, Q, V, alpha, eta, theta, gamma, M_0, S_0), on cases that cover the
  recurrence (b = 1), chunks with windows longer than one token, history rows,
  momentum, the degree-2 feature map, the l_p, Huber and dot-product biases;
- the closed-form gradients of causal linear attention: with the dot-product
  bias, alpha = eta = 0, theta = 1/2 and a one-token window the update is
  y_n = sum_{i<=n} (k_i . q_n) v_i ("It's All Connected (Miras)", Associative
  Memory & Attentional Bias), whose gradients with respect to K, Q, V and the
  three gates follow from the masked products written out below.
"""
import zlib

import numpy as np
import pytest

import oracle

H = 2


def _inputs(cfg, seed):
    r = np.random.default_rng(seed)
    nkv = cfg.N + cfg.n_history
    K = r.standard_normal((H, nkv, cfg.d_k))
    K /= np.linalg.norm(K, axis=-1, keepdims=True)
    Q = r.standard_normal((H, cfg.N, cfg.d_k))
    Q /= np.linalg.norm(Q, axis=-1, keepdims=True)
    ns = oracle.state_size(cfg)
    return dict(K=K, Q=Q, V=r.standard_normal((H, nkv, cfg.d_v)),
                alpha=r.uniform(0.0, 0.1, (H, cfg.N)), eta=r.uniform(0.3, 0.9, (H, cfg.N)),
                theta=r.uniform(0.05, 0.3, (H, cfg.N)), gamma=r.uniform(0.5, 1.5, cfg.c),
                M0=r.standard_normal((H, ns)) * 0.1, S0=r.standard_normal((H, ns)) * 0.1)


def _loss(cfg, x, dY, dM, dS):
    Y, M, S = oracle.forward(cfg, x["K"], x["Q"], x["V"], x["alpha"], x["eta"], x["theta"],
                             x["gamma"], x["M0"], x["S0"])
    return float(np.sum(dY * Y) + np.sum(dM * M) + np.sum(dS * S))


GRAD_OF = dict(K="dK", Q="dQ", V="dV", alpha="dalpha", eta="deta", theta="dtheta",
               gamma="dgamma", M0="dM0", S0="dS0")

CASES = {
    "recurrence": dict(N=7, d_k=4, d_v=3, c=1, b=1),
    "window-chunk-history": dict(N=11, d_k=4, d_v=3, c=3, b=4, n_history=2),
    "poly2": dict(N=10, d_k=3, d_v=2, c=2, b=3, phi=oracle.PHI_POLY2),
    "lp3": dict(N=8, d_k=4, d_v=3, c=2, b=2, loss=oracle.LOSS_LP, loss_param=3.0),
    "huber": dict(N=9, d_k=4, d_v=3, c=2, b=3, loss=oracle.LOSS_HUBER, loss_param=0.3),
    "dot": dict(N=8, d_k=4, d_v=3, c=2, b=2, loss=oracle.LOSS_DOT),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_matches_finite_differences(case):
    cfg = oracle.make_cfg(**CASES[case])
    x = _inputs(cfg, seed=zlib.crc32(case.encode()) % 1000)  # fixed across processes
    r = np.random.default_rng(5)
    ns = oracle.state_size(cfg)
    dY = r.standard_normal((H, cfg.N, cfg.d_v))
    dM = r.standard_normal((H, ns))
    dS = r.standard_normal((H, ns))
    g = oracle.backward(cfg, x["K"], x["Q"], x["V"], x["alpha"], x["eta"], x["theta"],
                        x["gamma"], x["M0"], x["S0"], dY, dM, dS)
    h = 1e-6
    for name, gname in GRAD_OF.items():
        arr = x[name]
        picks = r.choice(arr.size, size=min(6, arr.size), replace=False)
        for flat in picks:
            idx = np.unravel_index(flat, arr.shape)
            old = arr[idx]
            arr[idx] = old + h
            lp = _loss(cfg, x, dY, dM, dS)
            arr[idx] = old - h
            lm = _loss(cfg, x, dY, dM, dS)
            arr[idx] = old
            fd = (lp - lm) / (2 * h)
            an = g[gname][idx]
            # central differences with h = 1e-6; the l_p and Huber biases are not
            # smooth to third order at e = 0 / |e| = delta, hence 1e-5, still far
            # below the O(1) relative error of a dropped or mis-signed term
            assert abs(fd - an) <= 1e-5 * max(1.0, abs(fd)), (case, name, idx, fd, an)


@pytest.mark.parametrize("b", [1, 5])
def test_backward_of_linear_attention_closed_form(b):
    N, d, dv = 13, 5, 4
    cfg = oracle.make_cfg(N, d, dv, loss=oracle.LOSS_DOT, c=1, b=b)
    r = np.random.default_rng(11)
    K = r.standard_normal((1, N, d))
    Q = r.standard_normal((1, N, d))
    V = r.standard_normal((1, N, dv))
    dY = r.standard_normal((1, N, dv))
    z = np.zeros((1, N))
    g = oracle.backward(cfg, K, Q, V, z, z, z + 0.5, np.ones(1), None, None, dY)
    k, q, v, dy = K[0], Q[0], V[0], dY[0]
    mask = np.tril(np.ones((N, N)))           # [n, i]: i <= n
    A = mask * (q @ k.T)                      # k_i . q_n
    Bm = mask * (dy @ v.T)                    # dy_n . v_i
    np.testing.assert_allclose(g["dV"][0], A.T @ dy, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dQ"][0], Bm @ k, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dK"][0], Bm.T @ q, rtol=1e-10, atol=1e-12)
    full_A, full_B = q @ k.T, dy @ v.T         # unmasked [n, i]
    later = np.triu(np.ones((N, N))).T        # [n, t]: n >= t
    # S_t = v_t k_t^T (theta = 1/2 times the -2 v k^T gradient) feeds every y_n, n >= t
    np.testing.assert_allclose(g["dtheta"][0], 2 * np.sum(later * full_A * full_B, axis=0),
                               rtol=1e-10, atol=1e-12)
    # M_{t-1} = sum_{i<t} v_i k_i^T is scaled by (1 - alpha_t) for every y_n, n >= t
    dalpha = np.array([-sum(full_A[n, i] * full_B[n, i] for n in range(t, N) for i in range(t))
                       for t in range(N)])
    np.testing.assert_allclose(g["dalpha"][0], dalpha, rtol=1e-10, atol=1e-12)
    # S_{t-1} = v_{t-1} k_{t-1}^T carried into S_t by eta_t
    deta = np.array([0.0] + [sum(full_A[n, t - 1] * full_B[n, t - 1] for n in range(t, N))
                             for t in range(1, N)])
    np.testing.assert_allclose(g["deta"][0], deta, rtol=1e-10, atol=1e-12)
    # with M_0 = 0 the start state's gradient is sum_n dy_n q_n^T
    np.testing.assert_allclose(g["dM0"][0].reshape(dv, d), dy.T @ q, rtol=1e-10, atol=1e-12)


def test_backward_rejects_what_it_does_not_cover():
    cfg = oracle.make_cfg(4, 4, 4, d_h=8, mem=oracle.MEM_MLP)
    z = np.zeros((1, 4))
    with pytest.raises(ValueError):
        oracle.backward(cfg, np.zeros((1, 4, 4)), np.zeros((1, 4, 4)), np.zeros((1, 4, 4)), z, z,
                        z, np.ones(1), None, None, np.zeros((1, 4, 4)))
