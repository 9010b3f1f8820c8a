"""fp64 CPU oracle of the test-time memory update (Titans / Miras / ATLAS family).

TEST INFRASTRUCTURE ONLY.  The tests, the package smoke check and the
benchmark's CPU-baseline leg are the only callers; the CUDA library never
imports, loads or links anything here, and nothing here imports the CUDA
library.  The arithmetic lives in ``atlas_oracle.c`` (plain C, fp64, literal
token loops, threads over heads); this module only compiles it with gcc and
marshals numpy arrays through ctypes.

What each C function follows (page title, section) is stated in the C file.
Every function here is pinned by a ``-m "not gpu"`` test against a closed form,
an invariant, a library routine or brute force; see ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "atlas_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libatlas_oracle.so")

MEM_LINEAR, MEM_MLP, MEM_MLP_LN, MEM_MLP_GATED = 0, 1, 2, 3
PHI_IDENTITY, PHI_POLY2, PHI_POLY = 0, 1, 2
PHI_MAX_DEGREE = 4
LOSS_L2, LOSS_DOT, LOSS_LP, LOSS_HUBER, LOSS_ROBUST = 0, 1, 2, 3, 4
RET_L2, RET_ELASTIC, RET_BREGMAN, RET_KL, RET_LQ = 0, 1, 2, 3, 4


class OrcCfg(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int), ("d_k", ctypes.c_int), ("d_v", ctypes.c_int),
        ("d_h", ctypes.c_int), ("mem", ctypes.c_int), ("phi", ctypes.c_int),
        ("loss", ctypes.c_int), ("c", ctypes.c_int), ("b", ctypes.c_int),
        ("ns_steps", ctypes.c_int), ("ns_a", ctypes.c_double),
        ("ns_b", ctypes.c_double), ("ns_c", ctypes.c_double),
        ("ns_eps", ctypes.c_double), ("n_history", ctypes.c_int),
        ("loss_param", ctypes.c_double),
        ("phi_degree", ctypes.c_int), ("phi_coef", ctypes.c_double * (PHI_MAX_DEGREE + 1)),
        ("retention", ctypes.c_int), ("ret_param", ctypes.c_double),
    ]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags: no -march, no intrinsics)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
                           "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            cp = ctypes.POINTER(OrcCfg)
            lib.orc_feature_dim.argtypes = [cp]
            lib.orc_feature_dim.restype = ctypes.c_int
            lib.orc_state_size.argtypes = [cp]
            lib.orc_state_size.restype = ctypes.c_long
            lib.orc_phi.argtypes = [cp, dp, dp]
            lib.orc_gelu.argtypes = [ctypes.c_double]
            lib.orc_gelu.restype = ctypes.c_double
            lib.orc_gelu_prime.argtypes = [ctypes.c_double]
            lib.orc_gelu_prime.restype = ctypes.c_double
            lib.orc_memory_apply.argtypes = [cp, dp, dp, dp]
            lib.orc_grad.argtypes = [cp, dp, dp, dp, dp]
            lib.orc_newton_schulz.argtypes = [ctypes.c_int, ctypes.c_int, dp, ctypes.c_int,
                                              ctypes.c_double, ctypes.c_double,
                                              ctypes.c_double, ctypes.c_double, dp]
            fwd = [cp, ctypes.c_int] + [dp] * 10 + [ctypes.c_int]
            lib.orc_forward_chunked.argtypes = fwd
            lib.orc_forward_chunked.restype = ctypes.c_int
            lib.orc_forward_recurrent.argtypes = fwd
            lib.orc_forward_recurrent.restype = ctypes.c_int
            lib.orc_backward_chunked.argtypes = [cp, ctypes.c_int] + [dp] * 19 + [ctypes.c_int]
            lib.orc_backward_chunked.restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def make_cfg(N, d_k, d_v, d_h=0, mem=MEM_LINEAR, phi=PHI_IDENTITY, loss=LOSS_L2, c=1, b=1,
             ns_steps=0, ns_a=0.0, ns_b=0.0, ns_c=0.0, ns_eps=0.0, n_history=0,
             loss_param=0.0, phi_coef=None, retention=RET_L2, ret_param=0.0) -> OrcCfg:
    """loss_param: p of the l_p bias, delta of the Huber bias, Delta of the robust
    bias (unused otherwise).  phi_coef: a_0 .. a_p of the gated polynomial map
    (phi = PHI_POLY); p = len - 1.  retention / ret_param: the retention gate and
    its parameter (gamma of RET_ELASTIC, c of RET_KL, q of RET_LQ)."""
    coef = list(phi_coef or [])
    arr = (ctypes.c_double * (PHI_MAX_DEGREE + 1))(*([float(a) for a in coef] +
                                                     [0.0] * (PHI_MAX_DEGREE + 1 - len(coef))))
    return OrcCfg(int(N), int(d_k), int(d_v), int(d_h), int(mem), int(phi), int(loss),
                  int(c), int(b), int(ns_steps), float(ns_a), float(ns_b), float(ns_c),
                  float(ns_eps), int(n_history), float(loss_param),
                  max(0, len(coef) - 1), arr, int(retention), float(ret_param))


def feature_dim(cfg: OrcCfg) -> int:
    return _load().orc_feature_dim(ctypes.byref(cfg))


def state_size(cfg: OrcCfg) -> int:
    return _load().orc_state_size(ctypes.byref(cfg))


def phi(cfg: OrcCfg, x) -> np.ndarray:
    x = _f64(x)
    out = np.zeros(feature_dim(cfg))
    _load().orc_phi(ctypes.byref(cfg), _p(x), _p(out))
    return out


def gelu(x: float) -> float:
    return _load().orc_gelu(float(x))


def gelu_prime(x: float) -> float:
    return _load().orc_gelu_prime(float(x))


def memory_apply(cfg: OrcCfg, state, x) -> np.ndarray:
    state, x = _f64(state), _f64(x)
    out = np.zeros(cfg.d_v)
    _load().orc_memory_apply(ctypes.byref(cfg), _p(state), _p(x), _p(out))
    return out


def grad(cfg: OrcCfg, state, k, v) -> np.ndarray:
    state, k, v = _f64(state), _f64(k), _f64(v)
    G = np.zeros(state_size(cfg))
    _load().orc_grad(ctypes.byref(cfg), _p(state), _p(k), _p(v), _p(G))
    return G


def newton_schulz(S, steps, a, b, c, eps) -> np.ndarray:
    S = _f64(S)
    rows, cols = S.shape
    out = np.zeros_like(S)
    _load().orc_newton_schulz(rows, cols, _p(S), int(steps), float(a), float(b), float(c),
                              float(eps), _p(out))
    return out


def forward(cfg: OrcCfg, K, Q, V, alpha, eta, theta, gamma, M0=None, S0=None,
            recurrent: bool = False, n_threads: int = 0):
    """Run the oracle over H independent heads.

    K: [H, n_history + N, d_k] and V: [H, n_history + N, d_v] (the history rows
    first: they only enter windows); Q: [H, N, d_k]; alpha, eta, theta: [H, N];
    gamma: [c]; M0, S0: [H, state] or None (zeros).  Returns (Y [H, N, d_v],
    M [H, state], S [H, state]), all fp64.
    """
    K, Q, V = _f64(K), _f64(Q), _f64(V)
    H = K.shape[0]
    nkv = cfg.N + cfg.n_history
    assert K.shape == (H, nkv, cfg.d_k) and Q.shape == (H, cfg.N, cfg.d_k)
    assert V.shape == (H, nkv, cfg.d_v)
    alpha, eta, theta = _f64(alpha), _f64(eta), _f64(theta)
    assert alpha.shape == (H, cfg.N) and eta.shape == alpha.shape and theta.shape == alpha.shape
    gamma = _f64(gamma)
    assert gamma.shape == (cfg.c,)
    ns = state_size(cfg)
    M = np.zeros((H, ns)) if M0 is None else _f64(M0).reshape(H, ns).copy()
    S = np.zeros((H, ns)) if S0 is None else _f64(S0).reshape(H, ns).copy()
    Y = np.zeros((H, cfg.N, cfg.d_v))
    fn = _load().orc_forward_recurrent if recurrent else _load().orc_forward_chunked
    rc = fn(ctypes.byref(cfg), H, _p(K), _p(Q), _p(V), _p(alpha), _p(eta), _p(theta),
            _p(gamma), _p(M), _p(S), _p(Y), int(n_threads))
    if rc != 0:
        raise ValueError("oracle rejected the problem description")
    return Y, M, S


def backward(cfg: OrcCfg, K, Q, V, alpha, eta, theta, gamma, M0, S0, dY, dM_N=None, dS_N=None,
             n_threads: int = 0) -> dict:
    """Gradients of L = sum <dY, Y> + <dM_N, M_N> + <dS_N, S_N> through the chunked
    forward (linear memory, no Newton-Schulz) with respect to every input.

    Shapes as in ``forward``; dY: [H, N, d_v]; dM_N, dS_N: [H, state] or None (zero).
    Returns a dict of fp64 arrays: dK, dV [H, n_history + N, .], dQ [H, N, d_k],
    dalpha, deta, dtheta [H, N], dgamma [c] (summed over heads), dM0, dS0 [H, state].
    """
    K, Q, V = _f64(K), _f64(Q), _f64(V)
    H = K.shape[0]
    nkv = cfg.N + cfg.n_history
    ns = state_size(cfg)
    alpha, eta, theta, gamma = _f64(alpha), _f64(eta), _f64(theta), _f64(gamma)
    M = np.zeros((H, ns)) if M0 is None else _f64(M0).reshape(H, ns).copy()
    S = np.zeros((H, ns)) if S0 is None else _f64(S0).reshape(H, ns).copy()
    dY = _f64(dY)
    assert dY.shape == (H, cfg.N, cfg.d_v)
    dM = np.zeros((H, ns)) if dM_N is None else _f64(dM_N).reshape(H, ns).copy()
    dS = np.zeros((H, ns)) if dS_N is None else _f64(dS_N).reshape(H, ns).copy()
    out = dict(dK=np.zeros((H, nkv, cfg.d_k)), dQ=np.zeros((H, cfg.N, cfg.d_k)),
               dV=np.zeros((H, nkv, cfg.d_v)), dalpha=np.zeros((H, cfg.N)),
               deta=np.zeros((H, cfg.N)), dtheta=np.zeros((H, cfg.N)),
               dgamma=np.zeros((H, cfg.c)))
    rc = _load().orc_backward_chunked(
        ctypes.byref(cfg), H, _p(K), _p(Q), _p(V), _p(alpha), _p(eta), _p(theta), _p(gamma),
        _p(M), _p(S), _p(dY), _p(dM), _p(dS), _p(out["dK"]), _p(out["dQ"]), _p(out["dV"]),
        _p(out["dalpha"]), _p(out["deta"]), _p(out["dtheta"]), _p(out["dgamma"]),
        int(n_threads))
    if rc != 0:
        raise ValueError("backward oracle: unsupported or invalid problem description")
    out["dgamma"] = out["dgamma"].sum(axis=0)
    out["dM0"], out["dS0"] = dM, dS
    return out
