"""Parity of the CUDA path (called through the C ABI) with the fp64 oracle on
the same seeded inputs.

Small cases span several chunks and a ragged tail; full-size cases run every
head of a workload in the launch configuration the benchmark times and compare
sampled heads (whole sequences where the oracle is quick, a token prefix
otherwise -- the update is causal, so a prefix of the outputs is exact).
Tolerances: fp32 inputs max|x-y|/max|y| <= 1e-4; bf16 inputs max|x-y|/RMS(y)
<= 2e-2, on Y and on M_final separately.
"""
import numpy as np
import pytest

import workloads as W
from parity_util import oracle_cfg, rel_err, run_oracle, tol

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from test_memorization_recurrent_gb300 import build
    build.build()


def gpu_run(w, inp, N=None, S0=None, with_S=False):
    from test_memorization_recurrent_gb300.harness import Runner, to_device
    N = inp["K"].shape[1] if N is None else N
    sub = {k: (v[:, :N] if k in ("K", "Q", "V", "alpha", "eta", "theta") else v)
           for k, v in inp.items()}
    d = to_device(w, sub)
    r = Runner(w, sub["K"].shape[0], N, with_S=with_S or S0 is not None)
    S0d = None if S0 is None else torch.from_numpy(np.asarray(S0, np.float32)).cuda()
    Y, M = r(d, S0=S0d)
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    S = None if r.S is None else r.S.cpu().numpy()
    return Y.cpu().numpy(), M.cpu().numpy(), S


def check(w, Yg, Mg, Yo, Mo, what=""):
    ey, em = rel_err(Yg, Yo, w.bf16), rel_err(Mg, Mo, w.bf16)
    assert np.isfinite(Yg).all() and np.isfinite(Mg).all(), what
    assert ey <= tol(w), f"{what} Y err {ey:.3e} > {tol(w)}"
    assert em <= tol(w), f"{what} M err {em:.3e} > {tol(w)}"
    return ey, em


# ------------------------------------------------------------------ small cases

SMALL = {
    1: dict(heads=[0], N=512),
    2: dict(heads=[0, 5, 9], N=64 * 3 + 17),
    3: dict(heads=[0, 3], N=64 * 2 + 37),
    4: dict(heads=[0, 7], N=64 * 2 + 19),
    5: dict(heads=[0, 11], N=64 + 21),
}


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_small_parity(wid):
    w = W.workload(wid, bounded=True)
    s = SMALL[wid]
    inp = W.generate(w, heads=s["heads"], n_tokens=s["N"])
    Yo, Mo, _ = run_oracle(w, inp)
    Yg, Mg, _ = gpu_run(w, inp)
    check(w, Yg, Mg, Yo, Mo, f"workload {wid}")


@pytest.mark.parametrize("wid", [3, 4])
def test_small_parity_verbatim_gates_finite_prefix(wid):
    """The literal gates of the poly2 and MLP workloads overflow after a few
    chunks; parity is checked on the prefix where the oracle stays finite and
    moderate, with the error taken relative to the RMS of each chunk."""
    w = W.workload(wid)
    N = 2 * w.b
    inp = W.generate(w, heads=[1], n_tokens=N)
    Yo, Mo, _ = run_oracle(w, inp)
    Yg, Mg, _ = gpu_run(w, inp)
    for c0 in range(0, N, w.b):
        yo, yg = Yo[:, c0:c0 + w.b], Yg[:, c0:c0 + w.b]
        if not np.isfinite(yo).all() or np.abs(yo).max() > 1e6:
            break
        assert rel_err(yg, yo, True) <= tol(w), f"chunk {c0 // w.b}"


@pytest.mark.parametrize("b", [1, 5, 64])
def test_linear_attention_mode(b):
    """Dot-product bias, alpha = eta = 0, theta = 1/2: the GPU path reproduces
    causal linear attention for any chunk size (checked against the oracle,
    itself pinned to (Q K^T * mask) V)."""
    w = W.workload(2, loss=W.LOSS_DOT, b=b, N=150)
    inp = W.generate(w, heads=[0, 1])
    inp["alpha"][:] = 0
    inp["eta"][:] = 0
    inp["theta"][:] = 0.5
    Yo, Mo, _ = run_oracle(w, inp)
    Yg, Mg, _ = gpu_run(w, inp)
    check(w, Yg, Mg, Yo, Mo)


@pytest.mark.parametrize("wid", [1, 2, 4])
def test_momentum_state_round_trip(wid):
    """Two calls over halves of the sequence (split on a chunk boundary, c = 1
    or handled by the caller) carrying M and S equal one call over all of it."""
    w = W.workload(wid, bounded=True, c=1)
    N = 4 * w.b if w.b > 1 else 64
    inp = W.generate(w, heads=[0, 2], n_tokens=N)
    Yo, Mo, So = run_oracle(w, inp)
    half = N // 2
    first = {k: (v[:, :half] if k in ("K", "Q", "V", "alpha", "eta", "theta") else v)
             for k, v in inp.items()}
    second = {k: (v[:, half:] if k in ("K", "Q", "V", "alpha", "eta", "theta") else v)
              for k, v in inp.items()}
    Y1, M1, S1 = gpu_run(w, first, with_S=True)
    second["M0"] = M1
    Y2, M2, S2 = gpu_run(w, second, S0=S1)
    check(w, np.concatenate([Y1, Y2], axis=1), M2, Yo, Mo, "split")
    assert rel_err(S2, So, w.bf16) <= tol(w)


@pytest.mark.parametrize("N", [0, 1, 63, 65])
def test_edge_lengths(N):
    w = W.workload(3, bounded=True, N=max(N, 1))
    inp = W.generate(w, heads=[0], n_tokens=N)
    Yo, Mo, _ = run_oracle(w, inp)
    Yg, Mg, _ = gpu_run(w, inp)
    if N:
        check(w, Yg, Mg, Yo, Mo)
    else:
        np.testing.assert_array_equal(Mg, inp["M0"])


def test_chunk_longer_than_sequence_and_window_longer_than_chunk():
    w = W.workload(1, b=16, c=40, N=30)
    inp = W.generate(w)
    Yo, Mo, _ = run_oracle(w, inp)
    Yg, Mg, _ = gpu_run(w, inp)
    check(w, Yg, Mg, Yo, Mo)


# ------------------------------------------------- token-serial linear path

def test_token_serial_path_selected_for_the_exact_recurrence_workload():
    from test_memorization_recurrent_gb300.harness import cfg_for
    import test_memorization_recurrent_gb300 as A
    w = W.workload(1)
    assert A.atlas_mem_path(cfg_for(w, w.heads, w.N)) == "linear_seq"
    assert A.atlas_mem_path(cfg_for(w.with_(c=9), 1, 64)) == "linear_simt"
    assert A.atlas_mem_path(cfg_for(w.with_(d_k=16, d_v=16), 1, 64)) == "linear_simt"


@pytest.mark.parametrize("c,b,d_v,H,N,loss,bf16", [
    (1, 1, 32, 1, 64, W.LOSS_L2, False),
    (4, 1, 32, 2, 513, W.LOSS_L2, False),     # several tiles, ragged tail
    (8, 16, 32, 1, 200, W.LOSS_L2, False),    # widest window, chunked
    (3, 5, 20, 3, 131, W.LOSS_L2, False),     # ragged rows, chunk not a power of 2
    (2, 64, 48, 1, 300, W.LOSS_L2, True),     # two CTAs of rows, bf16 inputs
    (5, 1, 7, 2, 66, W.LOSS_DOT, False),      # dot loss
    (4, 8, 32, 1, 1, W.LOSS_L2, False),       # one token
])
def test_token_serial_path(c, b, d_v, H, N, loss, bf16):
    w = W.workload(1, c=c, b=b, d_v=d_v, H=H, N=N, loss=loss, bf16=bf16)
    inp = W.generate(w)
    Yo, Mo, So = run_oracle(w, inp)
    Yg, Mg, Sg = gpu_run(w, inp, with_S=True)
    check(w, Yg, Mg, Yo, Mo, f"c={c} b={b} d_v={d_v}")
    assert rel_err(Sg, So, w.bf16) <= tol(w)


# ------------------------------------------------------ tensor-core MLP path

def test_mlp_tensor_core_path_selected():
    from test_memorization_recurrent_gb300.harness import cfg_for
    import test_memorization_recurrent_gb300 as A
    w = W.workload(4)
    assert A.atlas_mem_path(cfg_for(w, w.heads, w.N)) == "mlp_tc"
    assert A.atlas_mem_path(cfg_for(w.with_(c=2), 2, 64)) == "mlp_simt"
    assert A.atlas_mem_path(cfg_for(w.with_(d_h=256), 2, 64)) == "mlp_simt"
    assert A.atlas_mem_path(cfg_for(W.workload(5), 16, 64)) == "mlp_simt"  # Newton-Schulz


@pytest.mark.parametrize("N,heads", [(1, [5]), (64, [0, 1, 2]), (200, [3, 30]), (517, [9])])
def test_mlp_tensor_core_path(N, heads):
    """Chunk-aligned, ragged and single-token lengths; momentum S in and out."""
    w = W.workload(4, bounded=True, N=N)
    inp = W.generate(w, heads=heads, n_tokens=N)
    Yo, Mo, So = run_oracle(w, inp)
    Yg, Mg, Sg = gpu_run(w, inp, with_S=True)
    check(w, Yg, Mg, Yo, Mo, f"N={N}")
    assert rel_err(Sg, So, w.bf16) <= tol(w)


@pytest.mark.parametrize("wid,N,heads", [(4, 147, [0, 7]), (5, 85, [0, 11])])
def test_repeated_runs_are_bit_identical(wid, N, heads):
    """The cluster kernels (MLP tensor-core path, fused Newton-Schulz) hand data
    between warps and CTAs through TMEM and shared memory; a missing ordering
    shows up as run-to-run differences long before it breaks a tolerance.  Eight
    runs of the same inputs must agree to the bit."""
    w = W.workload(wid, bounded=True)
    inp = W.generate(w, heads=heads, n_tokens=N)
    Y0, M0, S0 = gpu_run(w, inp, with_S=True)
    for _ in range(7):
        Y, M, S = gpu_run(w, inp, with_S=True)
        assert np.array_equal(Y, Y0) and np.array_equal(M, M0) and np.array_equal(S, S0)


def test_mlp_tensor_core_path_with_initial_momentum():
    """A non-zero S_0 (state handed over from a previous call) enters both the
    decay of M and the momentum; compared with the oracle started from the same S_0."""
    w = W.workload(4, bounded=True, N=130)
    inp = W.generate(w, heads=[4, 11], n_tokens=130)
    rng = np.random.default_rng(7)
    S0 = (rng.standard_normal(inp["M0"].shape) * 0.01).astype(np.float32)
    Yo, Mo, So = run_oracle(w, inp, S0=S0)
    Yg, Mg, Sg = gpu_run(w, inp, S0=S0)
    check(w, Yg, Mg, Yo, Mo, "S0")
    assert rel_err(Sg, So, w.bf16) <= tol(w)


# ------------------------------------------------------------- history rows

@pytest.mark.parametrize("wid,kw,N,nh,heads", [
    (1, dict(), 100, 3, [0]),                 # token-serial kernel, window 4, b = 1
    (1, dict(b=16, c=6, H=2), 70, 9, [0, 1]),  # token-serial, chunked; history > window
    (1, dict(c=12), 50, 11, [0]),             # linear CUDA-core kernel (window > 8)
    (3, {}, 80, 63, [0, 5]),                  # poly2, window 64
    (4, dict(c=3), 100, 2, [0, 3]),           # MLP CUDA-core path
    (5, {}, 70, 255, [2]),                    # Newton-Schulz, window 256
])
def test_history_rows(wid, kw, N, nh, heads):
    """K and V carry n_history rows ahead of the processed tokens; they enter the
    windows of the first tokens only.  Same history given to the oracle."""
    from test_memorization_recurrent_gb300.harness import Runner, to_device
    import oracle
    w = W.workload(wid, bounded=True, **kw)
    full = W.generate(w.with_(N=N + nh), heads=heads, n_tokens=N + nh)
    inp = dict(full)
    for k in ("Q", "alpha", "eta", "theta"):
        inp[k] = full[k][:, nh:]
    ho = {k: inp[k] for k in ("K", "Q", "V", "alpha", "eta", "theta")}
    Yo, Mo, So = oracle.forward(oracle_cfg(w, N, nh), ho["K"], ho["Q"], ho["V"], ho["alpha"],
                                ho["eta"], ho["theta"], inp["gamma"], inp["M0"])
    d = to_device(w, inp)
    r = Runner(w, len(heads), N, with_S=True, n_history=nh)
    Yg, Mg = r(d)
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    check(w, Yg.cpu().numpy(), Mg.cpu().numpy(), Yo, Mo, f"history {nh}")
    assert rel_err(r.S.cpu().numpy(), So, w.bf16) <= tol(w)


# -------------------------------------------------------------- full sizes

@pytest.mark.parametrize("wid,sample,prefix", [
    (2, [0, 77, 127], None),     # all 128 heads x 4096; sampled heads in full
    (3, [0, 31], None),          # all 32 heads x 8192; sampled heads in full
    (4, [0, 19], None),          # all 32 heads x 16384; sampled heads in full
])
def test_full_size_sampled(wid, sample, prefix):
    """The launch the benchmark times (every head, full length); sampled heads are
    compared with the oracle over their whole sequence, Y and M_final."""
    w = W.workload(wid, bounded=True)
    inp = W.generate(w)
    Yg, Mg, _ = gpu_run(w, inp)
    assert np.isfinite(Yg).all() and np.isfinite(Mg).all()
    sub = {k: (v[sample] if k not in ("gamma",) else v) for k, v in inp.items()}
    Yo, Mo, _ = run_oracle(w, sub, N=prefix)
    if prefix is None:
        check(w, Yg[sample], Mg[sample], Yo, Mo, f"workload {wid}")
    else:
        ey = rel_err(Yg[sample, :prefix], Yo, w.bf16)
        assert ey <= tol(w), f"workload {wid} Y prefix err {ey:.3e}"


def test_newton_schulz_workload_all_heads():
    """The ATLAS workload (MLP memory, window 256, five Newton-Schulz steps) with
    all 16 heads in one launch, over 320 tokens: five chunks, so the 256-token
    window fills and slides.  Every head is compared with the oracle on Y, M_final
    and the momentum S."""
    w = W.workload(5, bounded=True)
    N = 5 * w.b
    inp = W.generate(w, n_tokens=N)
    Yg, Mg, Sg = gpu_run(w, inp, with_S=True)
    Yo, Mo, So = run_oracle(w, inp)
    check(w, Yg, Mg, Yo, Mo, "ATLAS workload, 16 heads")
    assert rel_err(Sg, So, w.bf16) <= tol(w)


# ------------------------------------------------- tensor-core linear path

def test_tensor_core_path_selected_for_the_deltanet_workload():
    import test_memorization_recurrent_gb300 as A
    from test_memorization_recurrent_gb300.harness import cfg_for
    w = W.workload(2)
    assert A.atlas_mem_path(cfg_for(w, w.heads, w.N)) == "linear_tc"
    assert A.atlas_mem_path(cfg_for(w, 3, 212)) == "linear_tc"
    assert A.atlas_mem_path(cfg_for(w, 3, 209)) == "linear_tc"  # gates by plain loads


@pytest.mark.parametrize("N", [64, 212, 64 * 5, 209, 1, 63])
def test_tensor_core_path_small(N):
    """Several chunks and a ragged tail (N = 212) through the tcgen05 kernel; lengths
    that are not a multiple of 4 (gate rows not 16-byte aligned: plain gate loads)."""
    w = W.workload(2, N=N)
    inp = W.generate(w, heads=[0, 3, 8, 13])
    inp["M0"] = (np.random.default_rng(N).standard_normal(inp["M0"].shape) * 0.1).astype(np.float32)
    Yo, Mo, _ = run_oracle(w, inp)
    Yg, Mg, _ = gpu_run(w, inp)
    check(w, Yg, Mg, Yo, Mo, f"N={N}")


def test_tensor_core_path_mixed_momentum_heads_and_state_out():
    """Heads with a non-zero eta go to the CUDA-core kernel in the same call;
    the momentum returned through S_state matches for both kinds of head."""
    w = W.workload(2, N=256)
    inp = W.generate(w, heads=[0, 1, 2, 3])
    rng = np.random.default_rng(7)
    inp["eta"][1] = rng.uniform(0.5, 0.9, w.N).astype(np.float32)
    inp["eta"][3, 100] = 0.25
    Yo, Mo, So = run_oracle(w, inp)
    Yg, Mg, Sg = gpu_run(w, inp, with_S=True)
    check(w, Yg, Mg, Yo, Mo, "mixed")
    assert rel_err(Sg, So, True) <= tol(w)


def test_tensor_core_path_hands_off_a_full_reset_gate():
    """alpha = 1 (a full reset) makes the tensor-core kernel's rescaled readout
    weights undefined; that head is recomputed by the CUDA-core kernel in the
    same call and still matches the oracle."""
    w = W.workload(2, N=256)
    inp = W.generate(w, heads=[0, 1, 2])
    inp["alpha"][1, 70] = 1.0
    inp["alpha"][2, 130:140] = 0.9999
    Yo, Mo, _ = run_oracle(w, inp)
    Yg, Mg, _ = gpu_run(w, inp)
    check(w, Yg, Mg, Yo, Mo, "reset gate")


# ------------------------------------------------- alternative attentional biases

@pytest.mark.parametrize("loss,prm", [(W.LOSS_LP, 3.0), (W.LOSS_LP, 1.5), (W.LOSS_HUBER, 0.3)])
@pytest.mark.parametrize("wid,N,heads", [
    (1, 100, [0]),          # token-serial kernel
    (2, 64 + 13, [0, 5]),   # tensor-core linear kernel (ragged tail)
    (3, 64 + 9, [0]),       # wide-feature path (batched tensor-core GEMMs)
    (4, 64 + 19, [0, 7]),   # tensor-core MLP kernel
    (5, 12, [0]),           # CUDA-core MLP path with Newton-Schulz
])
def test_alternative_biases(wid, N, heads, loss, prm):
    """l_p and Huber biases (Miras alternative attentional biases) through every
    path that applies them, against the oracle on the same inputs."""
    w = W.workload(wid, bounded=True, loss=loss, loss_param=prm)
    inp = W.generate(w, heads=heads, n_tokens=N)
    Yo, Mo, _ = run_oracle(w, inp)
    Yg, Mg, _ = gpu_run(w, inp)
    check(w, Yg, Mg, Yo, Mo, f"workload {wid} loss {loss} ({prm})")


# ------------------------------------------- gated polynomial feature map

@pytest.mark.parametrize("d_k,coef,c,b,N,heads", [
    (8, (0.0, 1.0, 1.0, 1.0), 4, 16, 70, [0, 3]),         # degree 3, D = 164
    (6, (0.5, 1.0, 0.0, 0.8, 0.4), 2, 8, 41, [1]),        # constant, degree 2 gated off, degree 4
    (16, (0.0, 1.0, 0.7, 0.3), 1, 64, 130, [0, 2]),       # degree 3, D = 968, one-token window
])
def test_gated_polynomial_map(d_k, coef, c, b, N, heads):
    """The gated polynomial map of degree 3 and 4 ("논문 리뷰 Google ATLAS" §3.1,
    Polynomial Feature Mapping and Input gating) on the CUDA-core linear kernels,
    against the oracle; momentum and decay as in the poly2 workload (bounded step)."""
    from test_memorization_recurrent_gb300.harness import cfg_for
    import test_memorization_recurrent_gb300 as A
    w = W.workload(3, bounded=True, d_k=d_k, phi=W.PHI_POLY, phi_coef=coef, c=c, b=b, N=N,
                   theta_scale=0.002)
    path = "linear_wide" if w.D >= 256 else "linear_simt"  # the fused cluster kernel when wide
    assert A.atlas_mem_path(cfg_for(w, len(heads), N)) == path
    inp = W.generate(w, heads=heads, n_tokens=N)
    Yo, Mo, So = run_oracle(w, inp)
    Yg, Mg, Sg = gpu_run(w, inp, with_S=True)
    check(w, Yg, Mg, Yo, Mo, f"gated map {coef}")
    assert rel_err(Sg, So, w.bf16) <= tol(w)


# ------------------------------------------- layer-normalised MLP memory

@pytest.mark.parametrize("wid,kw,N,heads", [
    (4, dict(), 64 + 19, [0, 7]),                        # MLP shape, c = 1, momentum
    (4, dict(c=3, b=16, d_k=32, d_v=32, d_h=64), 70, [1, 2]),   # window, smaller widths
    (5, dict(), 64 + 11, [0]),                           # Newton-Schulz, window 256
    (4, dict(loss=W.LOSS_HUBER, loss_param=0.3), 64 + 5, [3]),  # Huber bias through LN
])
def test_layer_normalised_mlp_memory(wid, kw, N, heads):
    """x + LN(W1 GELU(W2 x)) ("It's All Connected (Miras)": the Moneta / Yaad /
    Memora memory) on the CUDA-core MLP path against the oracle."""
    w = W.workload(wid, bounded=True, mem=W.MEM_MLP_LN, **kw)
    inp = W.generate(w, heads=heads, n_tokens=N)
    Yo, Mo, So = run_oracle(w, inp)
    Yg, Mg, Sg = gpu_run(w, inp, with_S=True)
    check(w, Yg, Mg, Yo, Mo, f"LN memory {kw}")
    assert rel_err(Sg, So, w.bf16) <= tol(w)


def test_layer_normalised_mlp_memory_history_rows():
    from test_memorization_recurrent_gb300.harness import Runner, to_device
    import oracle
    w = W.workload(4, bounded=True, mem=W.MEM_MLP_LN, c=3)
    N, nh, heads = 60, 2, [0, 5]
    full = W.generate(w.with_(N=N + nh), heads=heads, n_tokens=N + nh)
    inp = dict(full)
    for k in ("Q", "alpha", "eta", "theta"):
        inp[k] = full[k][:, nh:]
    Yo, Mo, So = oracle.forward(oracle_cfg(w, N, nh), inp["K"], inp["Q"], inp["V"],
                                inp["alpha"], inp["eta"], inp["theta"], inp["gamma"], inp["M0"])
    r = Runner(w, len(heads), N, with_S=True, n_history=nh)
    Yg, Mg = r(to_device(w, inp))
    torch.cuda.synchronize()
    check(w, Yg.cpu().numpy(), Mg.cpu().numpy(), Yo, Mo, "LN history")


# ------------------------------------------------ gated (Atlas++) MLP memory

@pytest.mark.parametrize("wid,kw,N,heads", [
    (4, dict(), 64 + 19, [0, 7]),                               # MLP shape, momentum
    (4, dict(w_std=0.2), 64 + 19, [4]),                         # a gate far from zero
    (4, dict(c=3, b=16, d_k=32, d_v=32, d_h=64, w_std=0.2), 70, [1, 2]),  # window
    (5, dict(), 64 + 11, [0]),                                  # Newton-Schulz on all three blocks
    (4, dict(loss=W.LOSS_LP, loss_param=3.0), 64 + 5, [3]),     # l_p bias
])
def test_gated_mlp_memory(wid, kw, N, heads):
    """x + W1 (GELU(W2 x) * (W3 x)) (the paperlayer ATLAS summary §5, Atlas++) on the
    CUDA-core MLP path against the oracle, momentum S included."""
    w = W.workload(wid, bounded=True, mem=W.MEM_MLP_GATED, **kw)
    inp = W.generate(w, heads=heads, n_tokens=N)
    Yo, Mo, So = run_oracle(w, inp)
    Yg, Mg, Sg = gpu_run(w, inp, with_S=True)
    check(w, Yg, Mg, Yo, Mo, f"gated memory {kw}")
    assert rel_err(Sg, So, w.bf16) <= tol(w)


# ------------------------------------------------- retention gates, robust bias

RET_GATES = [(W.RET_ELASTIC, 0.01), (W.RET_BREGMAN, 0.0), (W.RET_KL, 1.0), (W.RET_LQ, 3.0),
             (W.RET_LQ, 2.5)]
RET_CASES = {
    2: (dict(eta=(0.5, 0.9)), 64 * 2 + 17, [0, 9]),  # d = 128, b = 64, momentum, ragged tail
    1: (dict(), 150, [0]),                            # fp32, c = 4, b = 1: the recurrence
    3: (dict(), 64 + 9, [2]),                         # degree-2 map, window 64
}


# q = 4 reads A / ||A||_4^2, which grows as the accumulator shrinks: in the
# recurrence from a zero state it has no well-conditioned trajectory (and q < 2
# feeds the memory's growth back into itself), so q = 4 runs with chunk-start
# normalisers only (b = 64).  The degree-2 workload's steps are
# small (theta scaled down), hence its smaller elastic threshold.
@pytest.mark.parametrize("wid,ret,prm", [(wid, r, p) for wid in (2, 1, 3) for r, p in RET_GATES]
                         + [(2, W.RET_LQ, 4.0), (3, W.RET_LQ, 4.0)])
def test_retention_gates(wid, ret, prm):
    """The Miras retention gates (elastic net, Bregman with a sigmoid link, KL,
    l_q) on the CUDA-core linear kernel against the oracle, from the gate's
    neutral memory, momentum S included."""
    from test_memorization_recurrent_gb300.harness import cfg_for
    import test_memorization_recurrent_gb300 as A
    kw, N, heads = RET_CASES[wid]
    if wid == 3 and ret == W.RET_ELASTIC:
        prm = 1e-4
    w = W.workload(wid, bounded=True, retention=ret, ret_param=prm, **kw)
    assert A.atlas_mem_path(cfg_for(w, len(heads), N)) == "linear_simt"
    inp = W.generate(w, heads=heads, n_tokens=N)
    Yo, Mo, So = run_oracle(w, inp)
    Yg, Mg, Sg = gpu_run(w, inp, with_S=True)
    check(w, Yg, Mg, Yo, Mo, f"workload {wid} retention {ret} ({prm})")
    assert rel_err(Sg, So, w.bf16) <= tol(w)
    if ret == W.RET_ELASTIC:  # the thresholded memory is sparse: zeros land on zeros
        assert np.mean((Mg == 0) == (Mo == 0)) > 0.99


@pytest.mark.parametrize("ret,prm", RET_GATES[:4])
def test_retention_gates_from_a_random_state(ret, prm):
    """A random start memory (in (0.2, 0.8) for Bregman, positive rows of any mass
    for KL, Gaussian otherwise) and a random start momentum."""
    w = W.workload(2, bounded=True, retention=ret, ret_param=prm, eta=(0.5, 0.9), N=64 + 30)
    heads = [1, 4]
    inp = W.generate(w, heads=heads)
    r = np.random.default_rng(7)
    shape = inp["M0"].shape
    if ret in (W.RET_BREGMAN, W.RET_KL):
        inp["M0"] = r.uniform(0.2, 0.8, shape).astype(np.float32)
    else:
        inp["M0"] = (r.standard_normal(shape) * 0.05).astype(np.float32)
    S0 = (r.standard_normal(shape) * 0.02).astype(np.float32)
    Yo, Mo, So = run_oracle(w, inp, S0=S0.astype(np.float64))
    Yg, Mg, Sg = gpu_run(w, inp, S0=S0)
    check(w, Yg, Mg, Yo, Mo, f"retention {ret} from a random state")
    assert rel_err(Sg, So, w.bf16) <= tol(w)


@pytest.mark.parametrize("wid,kw,N,heads,path", [
    (2, dict(eta=(0.5, 0.9)), 64 + 13, [0, 5], "linear_simt"),    # 8-CTA clusters per head
    (1, dict(), 120, [0], "linear_simt"),                          # fp32 recurrence, c = 4
    (3, dict(), 64 + 9, [0], "linear_wide"),                       # degree-2 map, d_v = 64
    (2, dict(retention=W.RET_ELASTIC, ret_param=0.01), 64 + 5, [3], "linear_simt"),
    (4, dict(), 64 + 19, [0, 7], "mlp_simt"),                      # MLP memory, momentum
    (4, dict(mem=W.MEM_MLP_LN), 64 + 5, [1], "mlp_simt"),          # through LN
    (5, dict(), 12, [0], "mlp_simt"),                              # Newton-Schulz, window 256
])
def test_robust_bias(wid, kw, N, heads, path):
    """The value-shift robust bias (Miras alternative attentional biases, read as
    (||e|| + Delta)^2) against the oracle; it couples a token's coordinates, so
    the linear memory's row blocks exchange partial norms within a cluster."""
    from test_memorization_recurrent_gb300.harness import cfg_for
    import test_memorization_recurrent_gb300 as A
    w = W.workload(wid, bounded=True, loss=W.LOSS_ROBUST, loss_param=0.5, **kw)
    assert A.atlas_mem_path(cfg_for(w, len(heads), N)) == path
    inp = W.generate(w, heads=heads, n_tokens=N)
    Yo, Mo, _ = run_oracle(w, inp)
    Yg, Mg, _ = gpu_run(w, inp)
    check(w, Yg, Mg, Yo, Mo, f"workload {wid} robust {kw}")


@pytest.mark.parametrize("kw,N,heads,path", [
    (dict(d_v=160), 64 + 9, [0, 1], "linear_chunk"),   # too many value rows for the cluster
    (dict(), 64 * 2 + 5, [0, 31], "linear_wide"),       # 4-CTA clusters, momentum, window 64
    (dict(d_v=24, c=3, b=16), 70, [2], "linear_wide"),  # other widths, window, chunk
    (dict(loss=W.LOSS_DOT), 64 + 3, [4], "linear_wide"),  # dot-product bias (E = -V)
    (dict(), 1, [7], "linear_wide"),                     # one token
    (dict(d_k=24, d_v=128, c=8), 64 + 2, [0], "linear_wide"),  # 128 value rows, D = 324
])
def test_wide_feature_map_paths(kw, N, heads, path):
    """The degree-2 map (D = 560) on the fused cluster kernel and, beyond its row
    limit, on the host-driven batched path, against the oracle with momentum S."""
    from test_memorization_recurrent_gb300.harness import cfg_for
    import test_memorization_recurrent_gb300 as A
    w = W.workload(3, bounded=True, **kw)
    assert A.atlas_mem_path(cfg_for(w, len(heads), N)) == path
    inp = W.generate(w, heads=heads, n_tokens=N)
    Yo, Mo, So = run_oracle(w, inp)
    Yg, Mg, Sg = gpu_run(w, inp, with_S=True)
    check(w, Yg, Mg, Yo, Mo, f"wide map {kw}")
    assert rel_err(Sg, So, w.bf16) <= tol(w)
