"""Seeded synthetic workloads for the test-time memory update.

This module only draws inputs; it holds none of the update's arithmetic and
imports neither the CUDA package nor the oracle, so both sides can share it.

Every random number comes from numpy's PCG64 generator seeded with the tuple
(seed, workload id, flat head index, token block), so that any subset of heads
or any token prefix is regenerated bit for bit without drawing the rest.  Keys
and queries are Gaussian rows L2-normalised in fp64, then rounded to the input
dtype (bf16 round-to-nearest-even, or fp32); values are N(0, 1) rounded the same
way.  Gates are fp32.  The five workloads follow the memory-update benchmark's
configurations: sizes, gate distributions and window weights as listed in
``WORKLOADS``; see the design notes for the readings where a distribution is
not stated.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Iterable, Optional

import numpy as np

BLOCK = 256  # tokens per independently seeded block

MEM_LINEAR, MEM_MLP, MEM_MLP_LN, MEM_MLP_GATED = 0, 1, 2, 3
PHI_IDENTITY, PHI_POLY2, PHI_POLY = 0, 1, 2
LOSS_L2, LOSS_DOT, LOSS_LP, LOSS_HUBER, LOSS_ROBUST = 0, 1, 2, 3, 4
RET_L2, RET_ELASTIC, RET_BREGMAN, RET_KL, RET_LQ = 0, 1, 2, 3, 4


@dataclasses.dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    B: int
    H: int
    N: int
    d_k: int
    d_v: int
    d_h: int = 0
    mem: int = MEM_LINEAR
    phi: int = PHI_IDENTITY
    loss: int = LOSS_L2
    loss_param: float = 0.0        # p of LOSS_LP, delta of LOSS_HUBER
    c: int = 1
    b: int = 1
    gamma: str = "ones"            # "ones" or "exp32": gamma_j = exp(-j/32)
    bf16: bool = True              # K, Q, V dtype (False: fp32)
    alpha_hi: float = 0.05         # alpha ~ U(0, alpha_hi)
    eta: tuple = (0.0, 0.0)        # eta ~ U(lo, hi); (0, 0) = identically 0
    theta: str = "sigmoid"         # "sigmoid": sigmoid(N(0,1)); "uniform": U(lo, hi)
    theta_range: tuple = (0.0, 0.0)
    theta_scale: float = 1.0
    w_std: float = 0.0             # MLP weight init std (0 for linear: M0 = 0)
    ns_steps: int = 0
    ns_coef: tuple = (0.0, 0.0, 0.0)
    ns_eps: float = 1e-7
    phi_coef: tuple = ()           # PHI_POLY: input-gating coefficients a_0 .. a_p
    retention: int = RET_L2        # retention gate of the linear memory
    ret_param: float = 0.0         # its parameter (lambda, c, q)

    @property
    def heads(self) -> int:
        return self.B * self.H

    @property
    def D(self) -> int:
        if self.mem == MEM_LINEAR and self.phi == PHI_POLY2:
            return self.d_k + self.d_k * (self.d_k + 1) // 2
        if self.mem == MEM_LINEAR and self.phi == PHI_POLY:
            return sum(math.comb(self.d_k + e - 1, e) for e, a in enumerate(self.phi_coef)
                       if a != 0.0)
        return self.d_k

    @property
    def state_size(self) -> int:
        if self.mem in (MEM_MLP, MEM_MLP_LN):
            return 2 * self.d_k * self.d_h
        if self.mem == MEM_MLP_GATED:
            return 3 * self.d_k * self.d_h
        return self.d_v * self.D

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.N

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


NS_COEF = (3.4445, -4.7750, 2.0315)

WORKLOADS = {
    1: Workload(1, "linear-omega-c4-fp32", B=1, H=1, N=512, d_k=32, d_v=32, c=4, b=1,
                bf16=False, alpha_hi=0.1, eta=(0.5, 0.9), theta="uniform",
                theta_range=(0.01, 0.1)),
    2: Workload(2, "linear-deltanet-b64-bf16", B=8, H=16, N=4096, d_k=128, d_v=128, c=1,
                b=64, alpha_hi=0.05),
    3: Workload(3, "poly2-omega-c64-bf16", B=4, H=8, N=8192, d_k=32, d_v=64,
                phi=PHI_POLY2, c=64, b=64, gamma="exp32", alpha_hi=0.05, eta=(0.5, 0.9)),
    4: Workload(4, "mlp-momentum-b64-bf16", B=4, H=8, N=16384, d_k=128, d_v=128, d_h=512,
                mem=MEM_MLP, c=1, b=64, alpha_hi=0.05, eta=(0.5, 0.9), w_std=0.02),
    5: Workload(5, "atlas-mlp-omega-c256-ns5-bf16", B=1, H=16, N=1048576, d_k=128,
                d_v=128, d_h=512, mem=MEM_MLP, c=256, b=64, alpha_hi=0.05, eta=(0.5, 0.9),
                w_std=0.02, ns_steps=5, ns_coef=NS_COEF),
}

# Bounded variants of the workloads whose literal trajectory overflows fp32
# (the step scale times the window mass and the momentum gain exceeds the
# stable range): same shapes, smaller theta (and alpha for the MLP).
BOUNDED = {
    3: dict(theta_scale=0.003),
    4: dict(theta_scale=0.03, alpha_hi=0.003),
}


def workload(wid: int, bounded: bool = False, **overrides) -> Workload:
    w = WORKLOADS[wid]
    if bounded and wid in BOUNDED:
        w = w.with_(**BOUNDED[wid])
    return w.with_(**overrides) if overrides else w


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32/fp64 values to the nearest bf16 (ties to even); returns fp32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32)


def gamma_of(w: Workload) -> np.ndarray:
    j = np.arange(w.c, dtype=np.float64)
    g = np.exp(-j / 32.0) if w.gamma == "exp32" else np.ones(w.c)
    return g.astype(np.float32)


def _rng(seed: int, w: Workload, head: int, block: int) -> np.random.Generator:
    return np.random.default_rng([seed, w.wid, head, block])


def _unit_rows(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float64)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _to_dtype(w: Workload, x: np.ndarray) -> np.ndarray:
    return round_bf16(x) if w.bf16 else np.asarray(x, dtype=np.float32)


def _block(w: Workload, seed: int, head: int, blk: int):
    r = _rng(seed, w, head, blk)
    n = BLOCK
    k = _to_dtype(w, _unit_rows(r.standard_normal((n, w.d_k), dtype=np.float32)))
    q = _to_dtype(w, _unit_rows(r.standard_normal((n, w.d_k), dtype=np.float32)))
    v = _to_dtype(w, r.standard_normal((n, w.d_v), dtype=np.float32))
    alpha = r.uniform(0.0, w.alpha_hi, n)
    if w.eta[1] > 0:
        eta = r.uniform(w.eta[0], w.eta[1], n)
    else:
        eta = np.zeros(n)
    if w.theta == "sigmoid":
        theta = 1.0 / (1.0 + np.exp(-r.standard_normal(n)))
    else:
        theta = r.uniform(w.theta_range[0], w.theta_range[1], n)
    theta = theta * w.theta_scale
    return (k, q, v, alpha.astype(np.float32), eta.astype(np.float32),
            theta.astype(np.float32))


def init_state(w: Workload, seed: int, head: int) -> np.ndarray:
    """Initial memory M_0 of one head (fp32): the gate's neutral memory for a
    linear memory (zeros; 1/2, logit 0, for the Bregman gate; rows of mass c
    spread evenly, c / D, for the KL gate); the MLP weights W1 (d x d_h) then W2
    (d_h x d), each N(0, w_std^2)."""
    if w.mem == MEM_LINEAR:
        if w.retention == RET_BREGMAN:
            return np.full(w.state_size, 0.5, dtype=np.float32)
        if w.retention == RET_KL:
            return np.full(w.state_size, w.ret_param / w.D, dtype=np.float32)
        return np.zeros(w.state_size, dtype=np.float32)
    r = _rng(seed, w, head, 1 << 30)
    return (r.standard_normal(w.state_size) * w.w_std).astype(np.float32)


def generate(w: Workload, seed: int = 0, heads: Optional[Iterable[int]] = None,
             n_tokens: Optional[int] = None) -> dict:
    """Inputs for the flat heads `heads` (default: all B*H) and the first
    `n_tokens` tokens (default: N).  Arrays are fp32 holding values exactly
    representable in the input dtype:
      K, Q [h, n, d_k]; V [h, n, d_v]; alpha, eta, theta [h, n]; gamma [c];
      M0 [h, state]."""
    heads = list(range(w.heads)) if heads is None else list(heads)
    n = w.N if n_tokens is None else int(n_tokens)
    nb = (n + BLOCK - 1) // BLOCK
    H = len(heads)
    K = np.empty((H, n, w.d_k), np.float32)
    Q = np.empty((H, n, w.d_k), np.float32)
    V = np.empty((H, n, w.d_v), np.float32)
    A = np.empty((H, n), np.float32)
    E = np.empty((H, n), np.float32)
    T = np.empty((H, n), np.float32)
    M0 = np.empty((H, w.state_size), np.float32)
    for i, h in enumerate(heads):
        for blk in range(nb):
            lo, hi = blk * BLOCK, min(n, (blk + 1) * BLOCK)
            k, q, v, a, e, t = _block(w, seed, h, blk)
            m = hi - lo
            K[i, lo:hi], Q[i, lo:hi], V[i, lo:hi] = k[:m], q[:m], v[:m]
            A[i, lo:hi], E[i, lo:hi], T[i, lo:hi] = a[:m], e[:m], t[:m]
        M0[i] = init_state(w, seed, h)
    return dict(K=K, Q=Q, V=V, alpha=A, eta=E, theta=T, gamma=gamma_of(w), M0=M0)


def flop_per_token(w: Workload) -> float:
    """Algorithmic FLOPs per token of the chunked update (the contractions the
    chunked method has to do; see the design notes for the derivation)."""
    D, dv, b = w.D, w.d_v, w.b
    L = b + w.c - 1
    momentum = w.eta[1] > 0
    if w.mem == MEM_LINEAR and w.retention in (RET_ELASTIC, RET_BREGMAN, RET_KL):
        # the token-serial chunk: errors at the chunk-start memory over the window,
        # then per token the window gradient sum (c rank-1 terms), the momentum and
        # state steps and the readout, 2 D d_v each
        return 2.0 * L * D * dv / b + 2.0 * w.c * D * dv + 6.0 * D * dv
    if w.mem == MEM_LINEAR:
        per_chunk = (2.0 * L * D * dv            # errors Phi M0^T over the window
                     + 2.0 * b * D * dv          # Q M0^T
                     + 2.0 * b * L * D           # Q Phi^T
                     + 2.0 * b * L * dv          # masked (Q Phi^T) E
                     + 2.0 * dv * L * D)         # state update E^T diag(w) Phi
        if momentum:
            per_chunk += 2.0 * b * D * dv + 2.0 * dv * L * D   # Q S0^T, S update
        return per_chunk / b
    d, dh = w.d_k, w.d_h
    fwd_bwd = 6.0 * L * d * dh            # W2 k, W1 h, W1^T e over the window
    gate = w.mem == MEM_MLP_GATED         # W3 k over the window, W3 / S3 updates and readouts
    if gate:
        fwd_bwd += 2.0 * L * d * dh
    if w.ns_steps:
        # per token: the Newton-Schulz iterations on both momenta (short-side
        # Gram, its square, one apply GEMM each), plus the readout matvecs
        ns = w.ns_steps * 2 * (2.0 * d * d * dh + 2.0 * d * d * d + 2.0 * d * d * dh)
        return fwd_bwd / b + ns + 4.0 * d * dh
    update = 8.0 * L * d * dh             # rank-L updates of W1, W2, S1, S2
    readout = 8.0 * b * d * dh + 2.0 * b * L * (2 * d + 2 * dh)
    if gate:
        update += 4.0 * L * d * dh
        readout += 4.0 * b * d * dh + 2.0 * b * L * dh
    return (fwd_bwd + update + readout) / b


def bytes_per_token(w: Workload) -> float:
    """Algorithmic HBM bytes per token: K, Q, V in, three fp32 gates in, Y (fp32) out."""
    e = 2 if w.bf16 else 4
    return (2 * w.d_k + w.d_v) * e + 3 * 4 + w.d_v * 4


def bwd_flop_per_token(w: Workload) -> float:
    """Algorithmic FLOPs per token of the backward pass of a linear memory with a
    one-token window (d = d_k = d_v, chunk b): per chunk, the forward replayed
    once to recover the chunk-start states (errors, state update), then the
    errors, K dM^T and M0 q again, C^T dY, the two terms of dM_0, the two of dK,
    dQ, dC = dY E^T, the tables' Q K^T and the finishing dP^T Q, dP K."""
    d, b = w.d_k, w.b
    X = 2.0 * b * d * d      # a (b x d) by (d x d) product
    Y = 2.0 * b * b * d      # a (b x b) by (b x d) product
    # with momentum: S_end in the replay, K dSe^T, Q S0^T, E dSe, dY S0 and the dS_0 term
    mom = 6 * X if w.eta[1] > 0 else 0.0
    return (10 * X + 5 * Y + mom) / b


def bwd_bytes_per_token(w: Workload) -> float:
    """Algorithmic HBM bytes per token of the backward pass: K, Q, V in their
    dtype, dY fp32 and three fp32 gates in; dK, dQ, dV and three gate gradients
    (fp32) out."""
    e = 2 if w.bf16 else 4
    return (2 * w.d_k + w.d_v) * e + w.d_v * 4 + 3 * 4 + (2 * w.d_k + w.d_v) * 4 + 3 * 4
