"""Pins of the retention gates and of the value-shift robust bias as the oracle
computes them ("It's All Connected (Miras)", #2 Alternative Retention Gates and
#1 Alternative Attentional Biases).

Each gate is pinned by what its definition fixes without re-running its formula:
- every gate: the chunked loop at b = 1 equals the separately written token
  recurrence, and the gate's neutral parameter reduces it to the l2 gate;
- elastic net: each new state is the proximal point of gamma ||.||_1 at the l2
  step (checked through its optimality conditions), and a threshold above every
  step leaves the memory at zero;
- Bregman (sigmoid link): entries stay in (0, 1); with no gradient the logits
  decay by prod (1 - alpha);
- KL: every row keeps mass c with positive entries; with no gradient the rows
  follow c softmax(prod (1 - alpha) log M_0);
- l_q (Moneta): q = 2 is the plain accumulation; with no gradient the readout is
  the accumulator's rows over ||A_r||_q^(q-2), and the normaliser refreshed only
  at chunk starts differs from the per-token one once b > 1;
- robust bias: Delta = 0 is the l2 bias, and the memory gradient matches central
  differences of ||e||^2 + 2 Delta ||e|| + Delta^2.
"""
import numpy as np
import pytest

import oracle

D, DV, N = 4, 3, 9


def _inputs(seed, positive=False, H=2, n=N):
    r = np.random.default_rng(seed)
    K = r.standard_normal((H, n, D))
    K /= np.linalg.norm(K, axis=-1, keepdims=True)
    Q = r.standard_normal((H, n, D))
    Q /= np.linalg.norm(Q, axis=-1, keepdims=True)
    M0 = r.uniform(0.2, 0.8, (H, DV * D)) if positive else r.standard_normal((H, DV * D)) * 0.3
    return dict(K=K, Q=Q, V=r.standard_normal((H, n, DV)), alpha=r.uniform(0, 0.1, (H, n)),
                eta=r.uniform(0.3, 0.8, (H, n)), theta=r.uniform(0.05, 0.2, (H, n)),
                gamma=r.uniform(0.5, 1.5, 2), M0=M0)


def _run(cfg, x, recurrent=False, S0=None):
    return oracle.forward(cfg, x["K"], x["Q"], x["V"], x["alpha"], x["eta"], x["theta"],
                          x["gamma"], x["M0"], S0, recurrent=recurrent)


GATES = [
    (oracle.RET_ELASTIC, 0.05, False),
    (oracle.RET_BREGMAN, 0.0, True),
    (oracle.RET_KL, 1.5, True),
    (oracle.RET_LQ, 4.0, False),
]


@pytest.mark.parametrize("ret,prm,positive", GATES)
def test_chunk_of_one_equals_the_token_recurrence(ret, prm, positive):
    x = _inputs(1, positive)
    cfg = oracle.make_cfg(N, D, DV, c=2, b=1, retention=ret, ret_param=prm)
    Yc, Mc, Sc = _run(cfg, x)
    Yr, Mr, Sr = _run(cfg, x, recurrent=True)
    np.testing.assert_allclose(Yc, Yr, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(Mc, Mr, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("ret,prm", [(oracle.RET_ELASTIC, 0.0), (oracle.RET_LQ, 2.0)])
def test_neutral_parameter_is_the_l2_gate(ret, prm):
    x = _inputs(2)
    base = oracle.make_cfg(N, D, DV, c=2, b=4)
    cfg = oracle.make_cfg(N, D, DV, c=2, b=4, retention=ret, ret_param=prm)
    Y0, M0, _ = _run(base, x)
    Y1, M1, _ = _run(cfg, x)
    assert np.array_equal(Y0, Y1) and np.array_equal(M0, M1)


def test_elastic_net_state_is_the_proximal_point_of_the_l2_step():
    x = _inputs(3)
    gam = 0.08
    cfg2 = oracle.make_cfg(1, D, DV, c=2, b=1)
    cfge = oracle.make_cfg(1, D, DV, c=2, b=1, retention=oracle.RET_ELASTIC, ret_param=gam)
    for t in range(1, 5):  # token t from the elastic state after t tokens
        sub = {k: (v[:, :t] if k in ("K", "Q", "V", "alpha", "eta", "theta") else v)
               for k, v in x.items()}
        cfg_t = oracle.make_cfg(t, D, DV, c=2, b=1, retention=oracle.RET_ELASTIC, ret_param=gam)
        _, Mt, St = _run(cfg_t, sub)
        nxt = {k: (v[:, t:t + 1] if k in ("K", "Q", "V", "alpha", "eta", "theta") else v)
               for k, v in x.items()}
        nxt["M0"] = Mt
        nxt["K"] = x["K"][:, t - 1:t + 1]
        nxt["V"] = x["V"][:, t - 1:t + 1]
        cfg2h = oracle.make_cfg(1, D, DV, c=2, b=1, n_history=1)
        cfgeh = oracle.make_cfg(1, D, DV, c=2, b=1, n_history=1, retention=oracle.RET_ELASTIC,
                                ret_param=gam)
        _, U, _ = oracle.forward(cfg2h, nxt["K"], nxt["Q"], nxt["V"], nxt["alpha"], nxt["eta"],
                                 nxt["theta"], nxt["gamma"], Mt, St)
        _, Mn, _ = oracle.forward(cfgeh, nxt["K"], nxt["Q"], nxt["V"], nxt["alpha"], nxt["eta"],
                                  nxt["theta"], nxt["gamma"], Mt, St)
        # optimality of min_W 1/2 ||W - U||^2 + gamma ||W||_1
        nz = Mn != 0
        np.testing.assert_allclose(Mn[nz] - U[nz] + gam * np.sign(Mn[nz]), 0.0, atol=1e-12)
        assert np.all(np.abs(U[~nz]) <= gam + 1e-12)
    assert cfg2.retention == 0 and cfge.retention == oracle.RET_ELASTIC


def test_elastic_net_threshold_above_every_step_keeps_the_memory_at_zero():
    x = _inputs(4)
    x["M0"][:] = 0.0
    cfg = oracle.make_cfg(N, D, DV, c=2, b=3, retention=oracle.RET_ELASTIC, ret_param=1e6)
    Y, M, _ = _run(cfg, x)
    assert np.all(M == 0.0) and np.all(Y == 0.0)


def test_bregman_without_gradient_decays_the_logits():
    x = _inputs(5, positive=True)
    x["theta"][:] = 0.0
    cfg = oracle.make_cfg(N, D, DV, c=2, b=3, retention=oracle.RET_BREGMAN)
    Y, M, _ = _run(cfg, x)
    lg0 = np.log(x["M0"] / (1 - x["M0"]))
    keep = np.prod(1 - x["alpha"], axis=1, keepdims=True)
    np.testing.assert_allclose(M, 1 / (1 + np.exp(-keep * lg0)), rtol=1e-12)
    x = _inputs(6, positive=True)
    Y, M, _ = _run(cfg, x)
    assert np.all((M > 0) & (M < 1))


def test_kl_rows_keep_their_mass_and_follow_the_tempered_softmax():
    c = 1.5
    x = _inputs(7, positive=True)
    cfg = oracle.make_cfg(N, D, DV, c=2, b=3, retention=oracle.RET_KL, ret_param=c)
    _, M, _ = _run(cfg, x)
    rows = M.reshape(2, DV, D)
    np.testing.assert_allclose(rows.sum(axis=-1), c, rtol=1e-12)
    assert np.all(rows > 0)
    x["theta"][:] = 0.0
    _, M, _ = _run(cfg, x)
    keep = np.prod(1 - x["alpha"], axis=1)[:, None, None]
    z = keep * np.log(x["M0"].reshape(2, DV, D))
    ref = c * np.exp(z) / np.exp(z).sum(axis=-1, keepdims=True)
    np.testing.assert_allclose(M.reshape(2, DV, D), ref, rtol=1e-12)


def test_lq_readout_without_gradient_and_chunk_start_normaliser():
    q = 4.0
    x = _inputs(8)
    x["theta"][:] = 0.0
    x["alpha"][:] = 0.0
    cfg = oracle.make_cfg(N, D, DV, c=2, b=3, retention=oracle.RET_LQ, ret_param=q)
    Y, M, _ = _run(cfg, x)
    A = x["M0"].reshape(2, DV, D)
    z = np.sum(np.abs(A) ** q, axis=-1) ** ((q - 2) / q)
    Wm = A / z[..., None]
    ref = np.einsum("hrj,hnj->hnr", Wm, x["Q"])
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(M, x["M0"])  # the state is the accumulator
    # with gradients, refreshing the normaliser per chunk is not per token
    x = _inputs(9)
    Yb, _, _ = _run(oracle.make_cfg(N, D, DV, c=2, b=3, retention=oracle.RET_LQ, ret_param=q), x)
    Y1, _, _ = _run(oracle.make_cfg(N, D, DV, c=2, b=1, retention=oracle.RET_LQ, ret_param=q), x)
    assert not np.allclose(Yb[:, 1:], Y1[:, 1:])


def test_robust_bias():
    x = _inputs(10)
    Y0, M0, _ = _run(oracle.make_cfg(N, D, DV, c=2, b=3), x)
    Y1, M1, _ = _run(oracle.make_cfg(N, D, DV, c=2, b=3, loss=oracle.LOSS_ROBUST,
                                     loss_param=0.0), x)
    assert np.array_equal(Y0, Y1) and np.array_equal(M0, M1)
    Dl = 0.4
    cfg = oracle.make_cfg(1, D, DV, loss=oracle.LOSS_ROBUST, loss_param=Dl)
    r = np.random.default_rng(11)
    M = r.standard_normal(DV * D)
    k, v = r.standard_normal(D), r.standard_normal(DV)
    G = oracle.grad(cfg, M, k, v)

    def loss(m):
        e = m.reshape(DV, D) @ k - v
        ne = np.linalg.norm(e)
        return ne ** 2 + 2 * Dl * ne + Dl ** 2

    h = 1e-6
    for j in range(M.size):
        mp, mm = M.copy(), M.copy()
        mp[j] += h
        mm[j] -= h
        assert abs((loss(mp) - loss(mm)) / (2 * h) - G[j]) <= 1e-6 * max(1.0, abs(G[j]))
    x = _inputs(12)
    cfg = oracle.make_cfg(N, D, DV, c=2, b=1, loss=oracle.LOSS_ROBUST, loss_param=Dl)
    Yc, _, _ = _run(cfg, x)
    Yr, _, _ = _run(cfg, x, recurrent=True)
    np.testing.assert_allclose(Yc, Yr, rtol=1e-12, atol=1e-14)
