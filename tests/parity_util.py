"""Shared helpers of the parity tests: the tolerance metrics and runners of
both sides on the same seeded inputs."""
import numpy as np

import oracle

# fp32-input workloads: max |x - y| / max |y| <= 1e-4 on Y and M_final.
# bf16-input / fp32-state workloads: max |x - y| / RMS(y) <= 2e-2.
TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def rel_err(x, ref, bf16: bool) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    den = np.sqrt(np.mean(ref ** 2)) if bf16 else np.max(np.abs(ref))
    return float(np.max(np.abs(x - ref)) / max(den, 1e-300))


def tol(w) -> float:
    return TOL_BF16 if w.bf16 else TOL_F32


def oracle_cfg(w, N, n_history=0):
    a, b, c = w.ns_coef
    return oracle.make_cfg(N, w.d_k, w.d_v, w.d_h, w.mem, w.phi, w.loss, w.c, w.b,
                           w.ns_steps, a, b, c, w.ns_eps, n_history=n_history,
                           loss_param=w.loss_param, phi_coef=w.phi_coef,
                           retention=w.retention, ret_param=w.ret_param)


def run_oracle(w, inp, N=None, recurrent=False, S0=None, n_threads=0):
    N = inp["K"].shape[1] if N is None else N
    return oracle.forward(oracle_cfg(w, N), inp["K"][:, :N], inp["Q"][:, :N], inp["V"][:, :N],
                          inp["alpha"][:, :N], inp["eta"][:, :N], inp["theta"][:, :N],
                          inp["gamma"], inp["M0"], S0, recurrent=recurrent,
                          n_threads=n_threads)
