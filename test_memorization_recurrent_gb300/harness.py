"""Marshalling helpers around ``atlas_mem_forward`` for tests and benchmarks.

Turns a workload description (``workloads.Workload``) and its host arrays into
device tensors, an ``AtlasMemCfg`` and a workspace, then calls the C entry
point.  Nothing here computes any part of the update.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (BF16, F32, AtlasMemCfg, atlas_mem_forward, atlas_mem_workspace_bytes,
               make_cfg)


def cfg_for(w, heads: int, N: int, S_state=None, workspace=None, workspace_bytes=0,
            status_dev=None, n_history: int = 0) -> AtlasMemCfg:
    """Config of workload ``w`` with ``heads`` heads (as B = 1, H = heads) and N tokens."""
    a, b_, c_ = w.ns_coef
    return make_cfg(1, heads, N, w.d_k, w.d_v, w.d_h, mem=w.mem, phi=w.phi, loss=w.loss,
                    loss_param=w.loss_param, c=w.c,
                    b=w.b, ns_steps=w.ns_steps, ns_a=a, ns_b=b_, ns_c=c_, ns_eps=w.ns_eps,
                    in_dtype=BF16 if w.bf16 else F32, S_state=S_state, workspace=workspace,
                    workspace_bytes=workspace_bytes, status_dev=status_dev, n_history=n_history,
                    phi_coef=w.phi_coef, retention=w.retention, ret_param=w.ret_param)


def to_device(w, inp: dict, device="cuda") -> dict:
    """Host arrays of ``workloads.generate`` -> device tensors in the ABI's types."""
    dt = torch.bfloat16 if w.bf16 else torch.float32
    out = {}
    for k in ("K", "Q", "V"):
        out[k] = torch.from_numpy(np.ascontiguousarray(inp[k])).to(device=device, dtype=dt)
    for k in ("alpha", "eta", "theta", "gamma", "M0"):
        out[k] = torch.from_numpy(np.ascontiguousarray(inp[k], dtype=np.float32)).to(device)
    return out


class Runner:
    """Owns the output, state and workspace buffers for repeated calls."""

    def __init__(self, w, heads: int, N: int, device="cuda", with_S: bool = False,
                 n_history: int = 0):
        self.w, self.heads, self.N = w, heads, N
        self.device = device
        self.Y = torch.empty((heads, N, w.d_v), device=device, dtype=torch.float32)
        self.M = torch.empty((heads, w.state_size), device=device, dtype=torch.float32)
        self.S = (torch.zeros((heads, w.state_size), device=device, dtype=torch.float32)
                  if with_S else None)
        self.status = torch.zeros(1, device=device, dtype=torch.int32)
        probe = cfg_for(w, heads, N, S_state=self.S, n_history=n_history)
        nbytes = atlas_mem_workspace_bytes(probe)
        self.ws = (torch.empty(max(nbytes, 1), device=device, dtype=torch.uint8)
                   if nbytes else None)
        self.cfg = cfg_for(w, heads, N, S_state=self.S, workspace=self.ws,
                           workspace_bytes=nbytes, status_dev=self.status, n_history=n_history)

    def __call__(self, d: dict, M0=None, S0=None, stream=None):
        """One forward over device inputs ``d``; M0/S0 (device) reset the state first."""
        self.M.copy_(d["M0"] if M0 is None else M0)
        if self.S is not None:
            if S0 is None:
                self.S.zero_()
            else:
                self.S.copy_(S0)
        atlas_mem_forward(d["K"], d["Q"], d["V"], d["alpha"], d["eta"], d["theta"], d["gamma"],
                          self.cfg, self.Y, self.M, stream)
        return self.Y, self.M


class BackwardRunner:
    """Owns the gradient buffers and the workspace of ``atlas_mem_backward``."""

    def __init__(self, w, heads: int, N: int, device="cuda"):
        from . import atlas_mem_backward_workspace_bytes
        self.w, self.heads, self.N = w, heads, N
        f32 = dict(device=device, dtype=torch.float32)
        self.dK = torch.empty((heads, N, w.d_k), **f32)
        self.dQ = torch.empty((heads, N, w.d_k), **f32)
        self.dV = torch.empty((heads, N, w.d_v), **f32)
        self.dalpha = torch.empty((heads, N), **f32)
        self.deta = torch.empty((heads, N), **f32)
        self.dtheta = torch.empty((heads, N), **f32)
        self.dM = torch.empty((heads, w.state_size), **f32)
        self.status = torch.zeros(1, device=device, dtype=torch.int32)
        nbytes = atlas_mem_backward_workspace_bytes(cfg_for(w, heads, N))
        self.ws = torch.empty(max(nbytes, 1), device=device, dtype=torch.uint8)
        self.cfg = cfg_for(w, heads, N, workspace=self.ws, workspace_bytes=nbytes,
                           status_dev=self.status)

    def __call__(self, d: dict, dY, dM_N, stream=None):
        """Gradients for device inputs ``d`` (its "M0" is the forward's initial state),
        upstream dY [heads, N, d_v] and dM_N [heads, state] (device fp32)."""
        from . import atlas_mem_backward
        self.dM.copy_(dM_N)
        atlas_mem_backward(d["K"], d["Q"], d["V"], d["alpha"], d["eta"], d["theta"], d["gamma"],
                           self.cfg, d["M0"], dY, self.dM, self.dK, self.dQ, self.dV,
                           self.dalpha, self.deta, self.dtheta, stream)
        return dict(dK=self.dK, dQ=self.dQ, dV=self.dV, dalpha=self.dalpha, deta=self.deta,
                    dtheta=self.dtheta, dM0=self.dM)
