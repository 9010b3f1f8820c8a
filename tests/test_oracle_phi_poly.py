"""Pins of the gated polynomial feature map ("논문 리뷰 Google ATLAS", §3.1:
Polynomial Feature Mapping, and Input gating: a_i switches the features of
degree i on or off) as the oracle computes it:
Phi(x) = [a_0; a_1 x; a_2 (x_i x_j)_{i<=j}; ...; a_p (degree-p monomials)].

- Every feature against a brute-force enumeration of the monomials
  (itertools.combinations_with_replacement) for several widths, degrees and
  gatings; a zero coefficient drops its degree from the vector.
- a = (0, 1, 1) is the degree-2 map bit for bit.
- The lifted inner product has the closed form
  Phi(q).Phi(k) = sum_e a_e^2 h_e(q * k), h_e the complete homogeneous symmetric
  polynomial of the elementwise products, evaluated by Newton's identities.
- With the dot-product bias, alpha = eta = 0 and theta = 1/2, the update is
  linear attention over the lifted features: y_n = sum_{i<=n} (Phi(k_i).Phi(q_n)) v_i.
- The backward pass through the map: finite differences of the forward oracle.
"""
import itertools

import numpy as np
import pytest

import oracle


def brute_phi(x, coef):
    out = []
    for e, a in enumerate(coef):
        if a == 0.0:
            continue
        for tup in itertools.combinations_with_replacement(range(len(x)), e):
            out.append(a * np.prod([x[i] for i in tup]) if e else a)
    return np.array(out)


def h_sym(z, e):
    """Complete homogeneous symmetric polynomial h_e(z) by Newton's identities."""
    p = [None] + [np.sum(z ** i) for i in range(1, e + 1)]
    h = [1.0]
    for m in range(1, e + 1):
        h.append(sum(p[i] * h[m - i] for i in range(1, m + 1)) / m)
    return h[e]


@pytest.mark.parametrize("d,coef", [
    (1, (0.0, 1.0, 1.0, 1.0)),
    (3, (0.5, 1.0, -2.0, 3.0)),
    (4, (0.0, 1.0, 0.0, 0.7)),       # degree 2 switched off
    (5, (1.0, 0.0, 0.0, 0.0, 0.25)),  # constant and degree 4 only
    (6, (0.0, 1.0, 1.0)),
])
def test_features_match_brute_force_enumeration(d, coef):
    cfg = oracle.make_cfg(1, d, 1, phi=oracle.PHI_POLY, phi_coef=coef)
    x = np.random.default_rng(d).standard_normal(d)
    ref = brute_phi(x, coef)
    assert oracle.feature_dim(cfg) == len(ref)
    np.testing.assert_allclose(oracle.phi(cfg, x), ref, rtol=1e-14, atol=0)


def test_degree_two_gating_is_the_degree_two_map():
    d = 7
    g = oracle.make_cfg(1, d, 1, phi=oracle.PHI_POLY, phi_coef=(0.0, 1.0, 1.0))
    p2 = oracle.make_cfg(1, d, 1, phi=oracle.PHI_POLY2)
    x = np.random.default_rng(1).standard_normal(d)
    assert oracle.feature_dim(g) == oracle.feature_dim(p2) == d + d * (d + 1) // 2
    assert np.array_equal(oracle.phi(g, x), oracle.phi(p2, x))


@pytest.mark.parametrize("coef", [(0.0, 1.0, 1.0, 1.0), (0.3, 0.5, 0.0, 2.0, 1.5)])
def test_lifted_inner_product_closed_form(coef):
    d = 6
    cfg = oracle.make_cfg(1, d, 1, phi=oracle.PHI_POLY, phi_coef=coef)
    r = np.random.default_rng(2)
    for _ in range(5):
        q, k = r.standard_normal(d), r.standard_normal(d)
        lhs = oracle.phi(cfg, q) @ oracle.phi(cfg, k)
        rhs = sum(a * a * h_sym(q * k, e) for e, a in enumerate(coef))
        assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(rhs))


@pytest.mark.parametrize("b", [1, 4])
def test_linear_attention_over_lifted_features(b):
    N, d, dv = 11, 4, 3
    coef = (0.5, 1.0, 0.8, 0.6)
    cfg = oracle.make_cfg(N, d, dv, phi=oracle.PHI_POLY, phi_coef=coef, loss=oracle.LOSS_DOT,
                          c=1, b=b)
    r = np.random.default_rng(4)
    K = r.standard_normal((1, N, d)) * 0.5
    Q = r.standard_normal((1, N, d)) * 0.5
    V = r.standard_normal((1, N, dv))
    z = np.zeros((1, N))
    Y, _, _ = oracle.forward(cfg, K, Q, V, z, z, z + 0.5, np.ones(1))
    for n in range(N):
        kern = [sum(a * a * h_sym(K[0, i] * Q[0, n], e) for e, a in enumerate(coef))
                for i in range(n + 1)]
        np.testing.assert_allclose(Y[0, n], np.asarray(kern) @ V[0, :n + 1], rtol=1e-10,
                                   atol=1e-12)


def test_backward_through_the_gated_map_matches_finite_differences():
    N, d, dv = 7, 3, 2
    cfg = oracle.make_cfg(N, d, dv, phi=oracle.PHI_POLY, phi_coef=(0.2, 1.0, -0.7, 0.5), c=2,
                          b=3)
    r = np.random.default_rng(9)
    ns = oracle.state_size(cfg)
    x = dict(K=r.standard_normal((1, N, d)) * 0.5, Q=r.standard_normal((1, N, d)) * 0.5,
             V=r.standard_normal((1, N, dv)), alpha=r.uniform(0, 0.1, (1, N)),
             eta=r.uniform(0.3, 0.9, (1, N)), theta=r.uniform(0.05, 0.3, (1, N)),
             gamma=r.uniform(0.5, 1.5, 2), M0=r.standard_normal((1, ns)) * 0.1,
             S0=r.standard_normal((1, ns)) * 0.1)
    dY = r.standard_normal((1, N, dv))
    dM = r.standard_normal((1, ns))

    def loss():
        Y, M, _ = oracle.forward(cfg, x["K"], x["Q"], x["V"], x["alpha"], x["eta"], x["theta"],
                                 x["gamma"], x["M0"], x["S0"])
        return float(np.sum(dY * Y) + np.sum(dM * M))

    g = oracle.backward(cfg, x["K"], x["Q"], x["V"], x["alpha"], x["eta"], x["theta"],
                        x["gamma"], x["M0"], x["S0"], dY, dM)
    h = 1e-6
    for name, gname in (("K", "dK"), ("Q", "dQ")):
        for flat in range(x[name].size):
            idx = np.unravel_index(flat, x[name].shape)
            old = x[name][idx]
            x[name][idx] = old + h
            lp = loss()
            x[name][idx] = old - h
            lm = loss()
            x[name][idx] = old
            fd = (lp - lm) / (2 * h)
            assert abs(fd - g[gname][idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx)
