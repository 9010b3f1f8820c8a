"""atlas_mem_forward_noalloc: the entry point for callers that cannot allocate
device memory (code running inside an allocator callback, or with its device
memory reserved up front) gives the same results as atlas_mem_forward with a
caller-provided workspace.

It runs the MLP-memory path, whose kernels need scratch, out of the library's
built-in array.  Two calls in a row on different inputs check that nothing
left in the shared array by one call leaks into the next.  This file is named
to be collected last.
"""
import ctypes

import numpy as np
import pytest

import workloads as W
from parity_util import rel_err, tol


@pytest.fixture(scope="module")
def lib():
    from test_memorization_recurrent_gb300 import build
    build.build()
    import test_memorization_recurrent_gb300 as A
    return A


def test_oversized_problem_is_rejected_before_launch(lib):
    w = W.workload(5)  # Newton-Schulz MLP workload: far more scratch than the array holds
    from test_memorization_recurrent_gb300.harness import cfg_for
    cfg = cfg_for(w, w.heads, w.N)
    assert lib.atlas_mem_workspace_bytes(cfg) > lib.NOALLOC_SCRATCH_BYTES
    rc = lib.load_library().atlas_mem_forward_noalloc(1, 1, 1, 1, 1, 1, 1, ctypes.byref(cfg), 1,
                                                      1, None)
    assert rc == lib.ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls(lib):
    import torch
    from test_memorization_recurrent_gb300.harness import Runner, cfg_for, to_device

    w = W.workload(4, bounded=True)
    N = 2 * w.b + 19
    for seed, heads in ((0, [0, 3]), (1, [5, 6])):
        inp = W.generate(w, seed=seed, heads=heads, n_tokens=N)
        d = to_device(w, inp)
        # reference: the existing entry point with a workspace the caller allocated
        ref = Runner(w, len(heads), N)
        Y_ref, M_ref = ref(d)
        # no-alloc entry point: no workspace in the description at all
        cfg = cfg_for(w, len(heads), N)
        assert lib.atlas_mem_workspace_bytes(cfg) <= lib.NOALLOC_SCRATCH_BYTES
        Y = torch.full_like(Y_ref, float("nan"))
        M = d["M0"].clone()
        lib.atlas_mem_forward_noalloc(d["K"], d["Q"], d["V"], d["alpha"], d["eta"], d["theta"],
                                      d["gamma"], cfg, Y, M)
        torch.cuda.synchronize()
        Yn, Mn = Y.cpu().numpy(), M.cpu().numpy()
        assert np.isfinite(Yn).all()
        assert rel_err(Yn, Y_ref.cpu().numpy(), w.bf16) <= tol(w)
        assert rel_err(Mn, M_ref.cpu().numpy(), w.bf16) <= tol(w)
