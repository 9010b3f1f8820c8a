"""Parity of the backward pass (atlas_mem_backward, called through the C ABI)
with the fp64 backward oracle on the same seeded inputs and upstream gradients,
with and without momentum in the forward:
dK, dQ, dV, dalpha, deta, dtheta and dM_0, each within the bf16-input tolerance
(max |x - y| / RMS(y) <= 2e-2).  Small cases span several chunks and a ragged
tail; the full-size case runs every head of the DeltaNet-like workload in one
call and compares sampled heads over their whole sequence."""
import numpy as np
import pytest

import oracle
import workloads as W
from parity_util import oracle_cfg, rel_err, tol

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from test_memorization_recurrent_gb300 import build
    build.build()


def upstream(w, heads, N, seed=3):
    r = np.random.default_rng(seed)
    dY = r.standard_normal((heads, N, w.d_v)).astype(np.float32)
    dM = (r.standard_normal((heads, w.state_size)) * 0.1).astype(np.float32)
    return dY, dM


def run_both(w, inp, dY, dMN, sample=None):
    from test_memorization_recurrent_gb300.harness import BackwardRunner, to_device
    N = inp["K"].shape[1]
    d = to_device(w, inp)
    r = BackwardRunner(w, inp["K"].shape[0], N)
    g = r(d, torch.from_numpy(dY).cuda(), torch.from_numpy(dMN).cuda())
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    got = {k: v.cpu().numpy() for k, v in g.items()}
    sel = slice(None) if sample is None else sample
    sub = {k: (v[sel] if k != "gamma" else v) for k, v in inp.items()}
    ref = oracle.backward(oracle_cfg(w, N), sub["K"], sub["Q"], sub["V"], sub["alpha"],
                          sub["eta"], sub["theta"], sub["gamma"], sub["M0"], None, dY[sel],
                          dMN[sel])
    return {k: v[sel] for k, v in got.items()}, ref


def check(w, got, ref, what):
    for k in ("dK", "dQ", "dV", "dalpha", "deta", "dtheta", "dM0"):
        assert np.isfinite(got[k]).all(), (what, k)
        e = rel_err(got[k], ref[k], True)
        assert e <= tol(w), f"{what}: {k} err {e:.3e}"


@pytest.mark.parametrize("N", [1, 64, 64 * 2 + 17])
@pytest.mark.parametrize("loss,prm", [(W.LOSS_L2, 0.0), (W.LOSS_HUBER, 0.3), (W.LOSS_LP, 3.0)])
def test_backward_small(N, loss, prm):
    w = W.workload(2, N=N, loss=loss, loss_param=prm)
    inp = W.generate(w, heads=[0, 5, 9])
    inp["M0"] = (np.random.default_rng(N).standard_normal(inp["M0"].shape) * 0.05).astype(np.float32)
    dY, dMN = upstream(w, 3, N)
    got, ref = run_both(w, inp, dY, dMN)
    check(w, got, ref, f"N={N} loss={loss}")


def test_backward_full_size_sampled():
    """Every head of the DeltaNet-like workload (128 x 4096) in one call; three
    heads compared with the oracle over their whole sequence."""
    w = W.workload(2)
    inp = W.generate(w)
    dY, dMN = upstream(w, w.heads, w.N)
    got, ref = run_both(w, inp, dY, dMN, sample=[0, 77, 127])
    check(w, got, ref, "full size")


@pytest.mark.parametrize("N", [64 + 9, 64 * 3])
@pytest.mark.parametrize("loss,prm", [(W.LOSS_L2, 0.0), (W.LOSS_HUBER, 0.3)])
def test_backward_with_momentum(N, loss, prm):
    """Momentum in the forward (eta ~ U(0.5, 0.9), as the other workloads draw it):
    the momentum's own tables and their gradients, the chunk-start momentum carried
    through the reverse, and eta's gradient against the oracle."""
    w = W.workload(2, N=N, loss=loss, loss_param=prm, eta=(0.5, 0.9))
    inp = W.generate(w, heads=[0, 5, 9])
    inp["M0"] = (np.random.default_rng(N).standard_normal(inp["M0"].shape) * 0.05).astype(np.float32)
    dY, dMN = upstream(w, 3, N)
    got, ref = run_both(w, inp, dY, dMN)
    check(w, got, ref, f"momentum N={N} loss={loss}")


def test_backward_momentum_on_some_tokens_only():
    """eta non-zero on a few tokens of one head, zero elsewhere (the DeltaNet gates
    with a momentum burst), including the first token of a chunk."""
    w = W.workload(2, N=64 * 2 + 30)
    inp = W.generate(w, heads=[0, 1])
    inp["eta"][1, [5, 63, 64, 65, 100]] = 0.7
    dY, dMN = upstream(w, 2, w.N)
    got, ref = run_both(w, inp, dY, dMN)
    check(w, got, ref, "momentum burst")
