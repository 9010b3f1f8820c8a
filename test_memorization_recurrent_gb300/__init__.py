"""GB300 (sm_103a) test-time memory update: Python binding of libatlasmem.so.

The binding only marshals arguments: it turns torch tensors into device
pointers, fills the ``atlas_mem_cfg`` struct and calls the C entry points of
``include/atlas_mem.h`` with the same names.  Every step of the update runs
in the library's CUDA kernels; if the library is missing or cannot be loaded,
importing a function here raises -- there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libatlasmem.so")

MEM_LINEAR, MEM_MLP, MEM_MLP_LN, MEM_MLP_GATED = 0, 1, 2, 3
PHI_IDENTITY, PHI_POLY2, PHI_POLY = 0, 1, 2
PHI_MAX_DEGREE = 4
LOSS_L2, LOSS_DOT, LOSS_LP, LOSS_HUBER, LOSS_ROBUST = 0, 1, 2, 3, 4
RET_L2, RET_ELASTIC, RET_BREGMAN, RET_KL, RET_LQ = 0, 1, 2, 3, 4
F32, BF16 = 0, 1

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = 0, -1, -2, -3, -4, -5

EXPORTS = ("atlas_mem_state_size", "atlas_mem_workspace_bytes", "atlas_mem_forward",
           "atlas_mem_forward_noalloc", "atlas_mem_backward", "atlas_mem_backward_workspace_bytes",
           "atlas_mem_strerror", "atlas_mem_path", "atlas_mem_launch_count")


class AtlasMemCfg(ctypes.Structure):
    """Mirror of ``atlas_mem_cfg`` in include/atlas_mem.h."""
    _fields_ = [
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int),
        ("d_k", ctypes.c_int), ("d_v", ctypes.c_int), ("d_h", ctypes.c_int),
        ("mem", ctypes.c_int), ("phi", ctypes.c_int), ("loss", ctypes.c_int),
        ("loss_param", ctypes.c_float), ("c", ctypes.c_int), ("b", ctypes.c_int),
        ("ns_steps", ctypes.c_int), ("ns_a", ctypes.c_float), ("ns_b", ctypes.c_float),
        ("ns_c", ctypes.c_float), ("ns_eps", ctypes.c_float),
        ("in_dtype", ctypes.c_int),
        ("S_state", ctypes.c_void_p), ("n_history", ctypes.c_int),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("status_dev", ctypes.c_void_p),
        ("phi_degree", ctypes.c_int), ("phi_coef", ctypes.c_float * (PHI_MAX_DEGREE + 1)),
        ("retention", ctypes.c_int), ("ret_param", ctypes.c_float),
    ]


class AtlasError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"atlas_mem error {code}: {msg}")
        self.code = code


_lock = threading.Lock()
_lib = None


def open_library(path: str):
    """Open a build of the library at ``path`` with the entry points' argument
    types set (tests also open separately built copies this way)."""
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "test_memorization_recurrent_gb300.build.build()")
    lib = ctypes.CDLL(path)
    cp = ctypes.POINTER(AtlasMemCfg)
    vp = ctypes.c_void_p
    lib.atlas_mem_state_size.argtypes = [cp]
    lib.atlas_mem_state_size.restype = ctypes.c_size_t
    lib.atlas_mem_workspace_bytes.argtypes = [cp]
    lib.atlas_mem_workspace_bytes.restype = ctypes.c_size_t
    lib.atlas_mem_forward.argtypes = [vp, vp, vp, vp, vp, vp, vp, cp, vp, vp, vp]
    lib.atlas_mem_forward.restype = ctypes.c_int
    lib.atlas_mem_strerror.argtypes = [ctypes.c_int]
    lib.atlas_mem_strerror.restype = ctypes.c_char_p
    lib.atlas_mem_path.argtypes = [cp]
    lib.atlas_mem_path.restype = ctypes.c_char_p
    lib.atlas_mem_launch_count.argtypes = [cp]
    lib.atlas_mem_launch_count.restype = ctypes.c_long
    lib.atlas_mem_forward_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, cp, vp, vp, vp]
    lib.atlas_mem_forward_noalloc.restype = ctypes.c_int
    lib.atlas_mem_backward_workspace_bytes.argtypes = [cp]
    lib.atlas_mem_backward_workspace_bytes.restype = ctypes.c_size_t
    lib.atlas_mem_backward.argtypes = [vp] * 7 + [cp] + [vp] * 10
    lib.atlas_mem_backward.restype = ctypes.c_int
    return lib


def load_library(path: str = LIB_PATH):
    """Load libatlasmem.so (built by ``build.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(path)
    return _lib


def make_cfg(B, H, N, d_k, d_v, d_h=0, mem=MEM_LINEAR, phi=PHI_IDENTITY, loss=LOSS_L2, c=1,
             b=1, ns_steps=0, ns_a=0.0, ns_b=0.0, ns_c=0.0, ns_eps=0.0, in_dtype=BF16,
             S_state=None, workspace=None, workspace_bytes=0, status_dev=None,
             n_history=0, loss_param=0.0, phi_coef=None, retention=RET_L2,
             ret_param=0.0) -> AtlasMemCfg:
    """loss_param: p of LOSS_LP, delta of LOSS_HUBER, Delta of LOSS_ROBUST (unused
    otherwise).  phi_coef: a_0 .. a_p of the gated polynomial map (phi = PHI_POLY);
    p = len - 1.  retention / ret_param: the linear memory's retention gate and its
    parameter (lambda of RET_ELASTIC, c of RET_KL, q of RET_LQ)."""
    coef = [float(a) for a in (phi_coef or [])]
    if len(coef) > PHI_MAX_DEGREE + 1:
        raise ValueError(f"at most {PHI_MAX_DEGREE + 1} coefficients (degree {PHI_MAX_DEGREE})")
    arr = (ctypes.c_float * (PHI_MAX_DEGREE + 1))(*(coef + [0.0] * (PHI_MAX_DEGREE + 1 - len(coef))))
    return AtlasMemCfg(int(B), int(H), int(N), int(d_k), int(d_v), int(d_h), int(mem), int(phi),
                       int(loss), float(loss_param), int(c), int(b), int(ns_steps), float(ns_a),
                       float(ns_b),
                       float(ns_c), float(ns_eps), int(in_dtype), _ptr(S_state), int(n_history),
                       _ptr(workspace), int(workspace_bytes), _ptr(status_dev),
                       max(0, len(coef) - 1), arr, int(retention), float(ret_param))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def atlas_mem_strerror(code: int) -> str:
    return load_library().atlas_mem_strerror(int(code)).decode()


def atlas_mem_state_size(cfg: AtlasMemCfg) -> int:
    return int(load_library().atlas_mem_state_size(ctypes.byref(cfg)))


def atlas_mem_workspace_bytes(cfg: AtlasMemCfg) -> int:
    n = int(load_library().atlas_mem_workspace_bytes(ctypes.byref(cfg)))
    if n == 2 ** 64 - 1:
        raise AtlasError(ERR_INVALID, "invalid configuration")
    return n


def atlas_mem_path(cfg: AtlasMemCfg) -> str:
    return load_library().atlas_mem_path(ctypes.byref(cfg)).decode()


def atlas_mem_launch_count(cfg: AtlasMemCfg) -> int:
    return int(load_library().atlas_mem_launch_count(ctypes.byref(cfg)))


def atlas_mem_forward(K, Q, V, alpha, eta, theta, gamma, cfg: AtlasMemCfg, Y, M_final,
                      stream=None) -> None:
    """Enqueue the chunked memory update on ``stream`` (a torch.cuda.Stream, a raw
    cudaStream_t as int, or None for torch's current stream).  Raises AtlasError
    on a non-zero status."""
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = load_library().atlas_mem_forward(
        _ptr(K), _ptr(Q), _ptr(V), _ptr(alpha), _ptr(eta), _ptr(theta), _ptr(gamma),
        ctypes.byref(cfg), _ptr(Y), _ptr(M_final), ctypes.c_void_p(stream))
    if rc != OK:
        raise AtlasError(rc, atlas_mem_strerror(rc))


NOALLOC_SCRATCH_BYTES = 32 << 20  # ATLAS_NOALLOC_SCRATCH_BYTES in include/atlas_mem.h


def atlas_mem_forward_noalloc(K, Q, V, alpha, eta, theta, gamma, cfg: AtlasMemCfg, Y, M_final,
                              stream=None) -> None:
    """``atlas_mem_forward`` for callers that cannot allocate device memory: the
    library's built-in scratch array (NOALLOC_SCRATCH_BYTES per device, shared by
    all calls on that device) replaces ``cfg.workspace``.  Calls that overlap on
    the GPU race on that array; make the first call on a device before any
    stream capture.  Raises AtlasError if the problem needs more scratch than
    the array holds."""
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = load_library().atlas_mem_forward_noalloc(
        _ptr(K), _ptr(Q), _ptr(V), _ptr(alpha), _ptr(eta), _ptr(theta), _ptr(gamma),
        ctypes.byref(cfg), _ptr(Y), _ptr(M_final), ctypes.c_void_p(stream))
    if rc == ERR_WORKSPACE:
        need = atlas_mem_workspace_bytes(cfg)
        raise AtlasError(rc, f"problem needs {need} bytes of scratch; the built-in array holds "
                             f"{NOALLOC_SCRATCH_BYTES} (split the heads over several calls)")
    if rc != OK:
        raise AtlasError(rc, atlas_mem_strerror(rc))


def atlas_mem_backward_workspace_bytes(cfg: AtlasMemCfg) -> int:
    n = int(load_library().atlas_mem_backward_workspace_bytes(ctypes.byref(cfg)))
    if n == 2 ** 64 - 1:
        raise AtlasError(ERR_UNSUPPORTED, "description not covered by the backward pass")
    return n


def atlas_mem_backward(K, Q, V, alpha, eta, theta, gamma, cfg: AtlasMemCfg, M0, dY, dM, dK, dQ,
                       dV, dalpha, deta, dtheta, stream=None) -> None:
    """Enqueue the backward pass (see include/atlas_mem.h): dM holds dL/dM_N on
    entry and dL/dM_0 on return; dK, dQ, dV, dalpha, deta, dtheta are written.
    Raises AtlasError on a non-zero status."""
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = load_library().atlas_mem_backward(
        _ptr(K), _ptr(Q), _ptr(V), _ptr(alpha), _ptr(eta), _ptr(theta), _ptr(gamma),
        ctypes.byref(cfg), _ptr(M0), _ptr(dY), _ptr(dM), _ptr(dK), _ptr(dQ), _ptr(dV),
        _ptr(dalpha), _ptr(deta), _ptr(dtheta), ctypes.c_void_p(stream))
    if rc != OK:
        raise AtlasError(rc, atlas_mem_strerror(rc))
