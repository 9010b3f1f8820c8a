"""The C-ABI library builds, loads and exports every entry point its header
declares; host-side validation rejects bad descriptions before any launch.
No test here touches a GPU."""
import ctypes
import os
import re

import pytest

import workloads as W
from test_memorization_recurrent_gb300 import build as B
import test_memorization_recurrent_gb300 as A
from test_memorization_recurrent_gb300.harness import cfg_for

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "atlas_mem.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return A.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(atlas_mem_\w+)\s*\(", text,
                                 flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert "atlas_mem_forward" in names and "atlas_mem_workspace_bytes" in names
    assert set(A.EXPORTS) <= set(names) | set()


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        ctypes.cast(getattr(lib, name), ctypes.c_void_p)


def test_strerror_codes(lib):
    assert A.atlas_mem_strerror(0) == "ok"
    for code in (-1, -2, -3, -4, -5):
        assert A.atlas_mem_strerror(code) not in ("ok", "unknown status")
    assert A.atlas_mem_strerror(-99) == "unknown status"


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_state_size_and_path(lib, wid):
    w = W.workload(wid)
    cfg = cfg_for(w, w.heads, w.N)
    assert A.atlas_mem_state_size(cfg) == w.state_size
    assert A.atlas_mem_path(cfg) in ("linear_simt", "linear_seq", "linear_chunk", "linear_tc",
                                      "linear_wide", "mlp_simt", "mlp_tc")
    assert A.atlas_mem_launch_count(cfg) >= 1
    nbytes = A.atlas_mem_workspace_bytes(cfg)
    assert nbytes >= 0
    if w.mem == W.MEM_MLP:
        assert nbytes > 0


def _bad(**kw):
    base = dict(B=1, H=2, N=16, d_k=8, d_v=8)
    base.update(kw)
    return A.make_cfg(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(N=-1), A.ERR_INVALID),
    (dict(d_k=0), A.ERR_INVALID),
    (dict(c=0), A.ERR_INVALID),
    (dict(b=0), A.ERR_INVALID),
    (dict(mem=7), A.ERR_INVALID),
    (dict(phi=3), A.ERR_INVALID),
    (dict(loss=5), A.ERR_INVALID),
    (dict(loss=A.LOSS_ROBUST, loss_param=-0.1), A.ERR_INVALID),  # Delta >= 0
    (dict(retention=5), A.ERR_INVALID),
    (dict(retention=A.RET_ELASTIC, ret_param=-1e-3), A.ERR_INVALID),  # lambda >= 0
    (dict(retention=A.RET_KL, ret_param=0.0), A.ERR_INVALID),         # mass c > 0
    (dict(retention=A.RET_LQ, ret_param=0.5), A.ERR_INVALID),         # q >= 1
    (dict(retention=A.RET_BREGMAN, mem=A.MEM_MLP, d_h=16), A.ERR_UNSUPPORTED),
    (dict(retention=A.RET_ELASTIC, ns_steps=5), A.ERR_UNSUPPORTED),
    (dict(loss=A.LOSS_LP, loss_param=0.5), A.ERR_INVALID),      # p < 1
    (dict(loss=A.LOSS_HUBER, loss_param=0.0), A.ERR_INVALID),   # delta must be > 0
    (dict(in_dtype=5), A.ERR_INVALID),
    (dict(mem=A.MEM_MLP, d_h=0), A.ERR_INVALID),
    (dict(mem=A.MEM_MLP, d_h=16, d_v=4), A.ERR_INVALID),
    (dict(mem=A.MEM_MLP, d_h=16, loss=A.LOSS_DOT), A.ERR_UNSUPPORTED),
    (dict(mem=4, d_h=16), A.ERR_INVALID),
    (dict(mem=A.MEM_MLP_GATED, d_h=0), A.ERR_INVALID),
    (dict(ns_steps=5), A.ERR_UNSUPPORTED),
    (dict(phi=A.PHI_POLY2, d_k=80), A.ERR_UNSUPPORTED),
    (dict(phi=A.PHI_POLY), A.ERR_INVALID),                             # degree 0
    (dict(phi=A.PHI_POLY, phi_coef=(0.0, 0.0)), A.ERR_INVALID),        # no feature left
    (dict(phi=A.PHI_POLY, phi_coef=(0, 1, 1, 1, 1), d_k=40), A.ERR_UNSUPPORTED),  # D > 16384
    (dict(phi=A.PHI_POLY, phi_coef=(0, 1), mem=A.MEM_MLP, d_h=16), A.ERR_INVALID),
])
def test_invalid_descriptions_rejected_before_launch(lib, kw, code):
    cfg = _bad(**kw)
    rc = lib.atlas_mem_forward(1, 1, 1, 1, 1, 1, 1, ctypes.byref(cfg), 1, 1, None)
    assert rc == code


def test_null_pointers_rejected(lib):
    cfg = _bad()
    rc = lib.atlas_mem_forward(None, None, None, None, None, None, None, ctypes.byref(cfg), None,
                               None, None)
    assert rc == A.ERR_INVALID


def test_missing_workspace_rejected(lib):
    cfg = _bad(mem=A.MEM_MLP, d_h=16)
    assert A.atlas_mem_workspace_bytes(cfg) > 0
    rc = lib.atlas_mem_forward(1, 1, 1, 1, 1, 1, 1, ctypes.byref(cfg), 1, 1, None)
    assert rc == A.ERR_WORKSPACE


def test_zero_heads_is_a_no_op(lib):
    cfg = _bad(H=0)
    rc = lib.atlas_mem_forward(None, None, None, None, None, None, None, ctypes.byref(cfg), None,
                               None, None)
    assert rc == A.OK


def test_invalid_workspace_query():
    with pytest.raises(A.AtlasError):
        A.atlas_mem_workspace_bytes(_bad(b=0))


def test_alternative_biases_choose_paths_that_apply_them(lib):
    """l_p and Huber act on the error elementwise in every path: the workloads keep
    their l2 paths."""
    from test_memorization_recurrent_gb300.harness import cfg_for
    for loss, prm in ((A.LOSS_LP, 3.0), (A.LOSS_HUBER, 0.5)):
        for wid, path in ((1, "linear_seq"), (2, "linear_tc"), (3, "linear_wide"),
                          (4, "mlp_tc"), (5, "mlp_simt")):
            w = W.workload(wid)
            w = w.__class__(**{**w.__dict__, "loss": loss, "loss_param": prm})
            cfg = cfg_for(w, 2, 256)
            assert A.atlas_mem_path(cfg) == path, (wid, loss)


def test_bias_launches_are_counted():
    """The host-driven wide-feature and CUDA-core MLP paths add one elementwise launch
    per chunk for an l_p or Huber bias; the other paths apply it inside their kernels."""
    from test_memorization_recurrent_gb300.harness import cfg_for
    N = 64 * 3 + 5  # four chunks
    for wid, extra in ((1, 0), (2, 0), (3, 0), (4, 0), (5, 4)):
        w = W.workload(wid)
        base = A.atlas_mem_launch_count(cfg_for(w, 2, N))
        wb = w.__class__(**{**w.__dict__, "loss": A.LOSS_HUBER, "loss_param": 0.3})
        assert A.atlas_mem_launch_count(cfg_for(wb, 2, N)) == base + extra, wid


@pytest.mark.parametrize("kw", [
    dict(mem=A.MEM_MLP, d_h=512),              # MLP memory
    dict(c=2),                                 # window longer than one token
    dict(b=32),                                # another chunk length
    dict(d_k=64, d_v=64),                      # another width
    dict(loss=A.LOSS_DOT),                     # dot-product bias
    dict(n_history=3),                         # history rows
    dict(phi=A.PHI_POLY2, d_k=16, d_v=128),    # feature map
    dict(loss=A.LOSS_ROBUST, loss_param=0.5),  # robust bias
    dict(retention=A.RET_LQ, ret_param=3.0),   # a retention gate
])
def test_backward_rejects_uncovered_descriptions(lib, kw):
    base = dict(B=1, H=2, N=100, d_k=128, d_v=128, c=1, b=64)
    base.update(kw)
    cfg = A.make_cfg(**base)
    with pytest.raises(A.AtlasError):
        A.atlas_mem_backward_workspace_bytes(cfg)
    rc = lib.atlas_mem_backward(*([1] * 7), ctypes.byref(cfg), *([1] * 10))
    assert rc == A.ERR_UNSUPPORTED


def test_backward_workspace_and_missing_workspace(lib):
    cfg = A.make_cfg(B=2, H=3, N=130, d_k=128, d_v=128, c=1, b=64)
    n = A.atlas_mem_backward_workspace_bytes(cfg)
    assert n >= 6 * 130 * 128 * 4 * 4  # at least the four row blocks' dK, dQ partials
    rc = lib.atlas_mem_backward(*([1] * 7), ctypes.byref(cfg), *([1] * 10))
    assert rc == A.ERR_WORKSPACE


def test_gated_polynomial_map_sizes(lib):
    """D counts the monomials of every degree whose coefficient is non-zero; the
    gated map runs on the CUDA-core linear kernels (the fused cluster kernel once
    D >= 256)."""
    import math
    for d, coef in ((8, (0, 1, 1, 1)), (6, (0.5, 1, 0, 0.8, 0.4)), (32, (0, 1, 1))):
        cfg = A.make_cfg(B=1, H=2, N=64, d_k=d, d_v=16, phi=A.PHI_POLY, phi_coef=coef, c=2, b=8)
        D = sum(math.comb(d + e - 1, e) for e, a in enumerate(coef) if a != 0)
        assert A.atlas_mem_state_size(cfg) == 16 * D
        assert A.atlas_mem_path(cfg) == ("linear_wide" if D >= 256 else "linear_simt")
    # a = (0, 1, 1) describes the same features as the degree-2 map
    g = A.make_cfg(B=1, H=1, N=8, d_k=32, d_v=64, phi=A.PHI_POLY, phi_coef=(0, 1, 1))
    p2 = A.make_cfg(B=1, H=1, N=8, d_k=32, d_v=64, phi=A.PHI_POLY2)
    assert A.atlas_mem_state_size(g) == A.atlas_mem_state_size(p2) == 64 * 560


def test_gated_map_degree_beyond_the_maximum_is_rejected(lib):
    cfg = _bad(phi=A.PHI_POLY, phi_coef=(0, 1, 1, 1, 1))
    cfg.phi_degree = A.PHI_MAX_DEGREE + 1
    rc = lib.atlas_mem_forward(1, 1, 1, 1, 1, 1, 1, ctypes.byref(cfg), 1, 1, None)
    assert rc == A.ERR_INVALID
    with pytest.raises(ValueError):
        A.make_cfg(1, 1, 8, 4, 4, phi=A.PHI_POLY, phi_coef=(0, 1, 1, 1, 1, 1))


def test_layer_normalised_memory_runs_on_the_cuda_core_mlp_path(lib):
    from test_memorization_recurrent_gb300.harness import cfg_for
    w = W.workload(4).with_(mem=W.MEM_MLP_LN)
    cfg = cfg_for(w, 4, 256)
    assert A.atlas_mem_path(cfg) == "mlp_simt"
    assert A.atlas_mem_state_size(cfg) == 2 * 128 * 512
    assert A.atlas_mem_workspace_bytes(cfg) > 0


def test_gated_memory_runs_on_the_cuda_core_mlp_path(lib):
    from test_memorization_recurrent_gb300.harness import cfg_for
    for wid in (4, 5):
        w = W.workload(wid).with_(mem=W.MEM_MLP_GATED)
        cfg = cfg_for(w, 2, 130)
        assert A.atlas_mem_path(cfg) == "mlp_simt"
        assert A.atlas_mem_state_size(cfg) == 3 * 128 * 512
        assert A.atlas_mem_workspace_bytes(cfg) > 0


def test_retention_gates_and_robust_bias_run_on_the_cuda_core_kernels(lib):
    """Every retention gate other than l2 selects the CUDA-core linear kernel (one
    launch), as does the robust bias on a narrow map (a wide one keeps the fused
    cluster kernel, whose error rows are whole); on an MLP memory the robust bias
    takes the CUDA-core MLP path, one row-scaling launch per chunk."""
    from test_memorization_recurrent_gb300.harness import cfg_for
    for ret, prm in ((A.RET_ELASTIC, 0.01), (A.RET_BREGMAN, 0.0), (A.RET_KL, 1.0),
                     (A.RET_LQ, 3.0)):
        for wid in (1, 2, 3):
            w = W.workload(wid, retention=ret, ret_param=prm)
            cfg = cfg_for(w, 2, 256)
            assert A.atlas_mem_path(cfg) == "linear_simt", (wid, ret)
            assert A.atlas_mem_launch_count(cfg) == 1
            assert A.atlas_mem_state_size(cfg) == w.state_size
    for wid, path in ((1, "linear_simt"), (2, "linear_simt"), (3, "linear_wide")):
        w = W.workload(wid, loss=A.LOSS_ROBUST, loss_param=0.5)
        assert A.atlas_mem_path(cfg_for(w, 2, 256)) == path
    N = 64 * 3 + 5  # four chunks
    for wid, extra in ((4, 4), (5, 4)):
        w = W.workload(wid)
        base = A.atlas_mem_launch_count(cfg_for(w, 2, N))
        wr = w.with_(loss=A.LOSS_ROBUST, loss_param=0.5)
        assert A.atlas_mem_path(cfg_for(wr, 2, N)) == "mlp_simt"
        if A.atlas_mem_path(cfg_for(w, 2, N)) == "mlp_simt":
            assert A.atlas_mem_launch_count(cfg_for(wr, 2, N)) == base + extra, wid


def test_robust_bias_on_wide_memories_is_planned_in_clusters(lib):
    """The robust bias needs every row of a head; d_v = 128 rows of D = 128 do not
    fit one CTA's shared memory, so the plan splits them over a cluster (the
    call is supported, the state size unchanged)."""
    cfg = A.make_cfg(B=1, H=2, N=300, d_k=128, d_v=128, c=1, b=64, loss=A.LOSS_ROBUST,
                     loss_param=0.5)
    assert A.atlas_mem_path(cfg) == "linear_simt"
    assert A.atlas_mem_workspace_bytes(cfg) == 0


def test_wide_maps_choose_the_fused_cluster_kernel(lib):
    """The degree-2 workload and the gated degree-3 map (D = 968) run as one launch
    of the fused kernel; more than 128 value rows fall back to the host-driven path."""
    from test_memorization_recurrent_gb300.harness import cfg_for
    w = W.workload(3)
    cfg = cfg_for(w, w.heads, w.N)
    assert A.atlas_mem_path(cfg) == "linear_wide"
    assert A.atlas_mem_launch_count(cfg) == 1
    assert A.atlas_mem_workspace_bytes(cfg) == 0
    g = w.with_(d_k=16, phi=A.PHI_POLY, phi_coef=(0.0, 1.0, 1.0, 1.0))
    assert A.atlas_mem_path(cfg_for(g, 32, 2048)) == "linear_wide"
    assert A.atlas_mem_path(cfg_for(w.with_(d_v=160), 2, 256)) == "linear_chunk"
