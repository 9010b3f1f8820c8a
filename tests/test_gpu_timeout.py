"""A bounded device-side wait that runs out reports ATLAS_ERR_TIMEOUT through the
status word, stops the head at a chunk boundary (nothing after it is written, nor
the final state), and leaves the CUDA context usable.

Every mbarrier wait in the tensor-core kernels gives up after about a second.
To make one run out without faulting anything, the test builds a separate copy
of the library with ATLAS_TEST_WITHHOLD_LOADS defined: there the producer warp
of head 0 in the tensor-core linear kernel never issues chunk 1's tile loads,
so the gate-table wait on that stage expires after chunk 0 is done.  That head's CTA then records the
timeout, drains the MMAs it issued, frees its TMEM and returns; the other heads
of the same launch run to completion.  Nothing is read or written out of
bounds, and every wait in the kernel still ends.
"""
import ctypes

import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_withheld_loads_time_out_and_the_context_stays_usable():
    import test_memorization_recurrent_gb300 as A
    from test_memorization_recurrent_gb300 import build
    from test_memorization_recurrent_gb300.harness import Runner, cfg_for, to_device

    build.build()
    test_lib = A.open_library(build.build_variant("atlasmem_withhold",
                                                  ["ATLAS_TEST_WITHHOLD_LOADS"]))
    w = W.workload(2, N=64 * 3)  # three chunks per head
    heads = 3
    inp = W.generate(w, heads=[0, 1, 2])
    d = to_device(w, inp)

    ref = Runner(w, heads, w.N)  # the library the package builds
    assert A.atlas_mem_path(ref.cfg) == "linear_tc"
    Y_ref, M_ref = (t.clone() for t in ref(d))
    torch.cuda.synchronize()
    assert int(ref.status.item()) == 0

    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cfg = cfg_for(w, heads, w.N, workspace=ref.ws, workspace_bytes=ref.ws.numel(),
                  status_dev=status)
    Y = torch.full((heads, w.N, w.d_v), float("nan"), device="cuda")
    M = d["M0"].clone()
    stream = torch.cuda.current_stream().cuda_stream
    rc = test_lib.atlas_mem_forward(d["K"].data_ptr(), d["Q"].data_ptr(), d["V"].data_ptr(),
                                    d["alpha"].data_ptr(), d["eta"].data_ptr(),
                                    d["theta"].data_ptr(), d["gamma"].data_ptr(),
                                    ctypes.byref(cfg), Y.data_ptr(), M.data_ptr(),
                                    ctypes.c_void_p(stream))
    assert rc == A.OK  # the launch itself succeeded; the expiry is reported on the device
    torch.cuda.synchronize()
    assert int(status.item()) == A.ERR_TIMEOUT

    # head 0 finished chunk 0 (its loads were issued), then gave up at the chunk
    # boundary: chunk 0's outputs are those of a normal run, nothing after them was
    # written, and M was not written back
    y0, y0_ref = Y[0, :64].cpu().numpy(), Y_ref[0, :64].cpu().numpy()
    assert np.max(np.abs(y0 - y0_ref)) <= 1e-6 * np.sqrt(np.mean(y0_ref.astype(np.float64) ** 2))
    assert torch.isnan(Y[0, 64:]).all()
    assert torch.equal(M[0], d["M0"][0])
    # the other heads of the same launch ran to completion
    Yr, Mr = Y_ref.cpu().numpy(), M_ref.cpu().numpy()
    for h in (1, 2):
        scale = np.sqrt(np.mean(Yr[h].astype(np.float64) ** 2))
        assert np.max(np.abs(Y[h].cpu().numpy() - Yr[h])) <= 1e-6 * scale
        assert np.max(np.abs(M[h].cpu().numpy() - Mr[h])) <= 1e-6 * max(np.abs(Mr[h]).max(), 1e-30)

    # the context is still usable: the next normal call on the same stream gives
    # the same bits as before the timeout
    Y2, M2 = ref(d)
    torch.cuda.synchronize()
    assert int(ref.status.item()) == 0
    assert torch.equal(Y2, Y_ref) and torch.equal(M2, M_ref)
