"""Thin ctypes binding over libgla.so, with the C ABI's names.

Argument marshalling only: tensors become device pointers, results are
returned as status codes (or raised as GlaError). Every step of the forward
pass runs in the library's CUDA kernels; there is no fallback of any kind,
and a missing or unloadable library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

GLA_OK, GLA_ERR_INVALID_ARG, GLA_ERR_UNSUPPORTED, GLA_ERR_CUDA, GLA_ERR_WORKSPACE, GLA_ERR_TIMEOUT = range(6)
GLA_BF16, GLA_FP32 = 0, 1
GLA_GATE_NONE, GLA_GATE_HEAD_SCALAR, GLA_GATE_PER_KEY, GLA_GATE_TOKEN_SCALAR, GLA_GATE_BILINEAR = 0, 1, 2, 3, 4
GLA_PATH_AUTO, GLA_PATH_TENSOR, GLA_PATH_SIMT, GLA_PATH_STAGED, GLA_PATH_FUSED, GLA_PATH_SPLIT = 0, 1, 2, 3, 4, 5

# Every symbol include/gla.h declares.
EXPORTED = ("gla_fwd", "gla_fwd_ex", "gla_fwd_workspace_size", "gla_fwd_num_stages",
            "gla_fwd_stage", "gla_fwd_stage_name", "gla_device_status", "gla_status_string",
            "gla_version", "gla_fwd_noalloc", "gla_fwd_host", "gla_host_release", "gla_bwd",
            "gla_bwd_workspace_size", "gla_bwd_num_stages", "gla_bwd_stage", "gla_bwd_stage_name",
            "gla_segment_pair_workspace_size", "gla_segment_pair",
            "gla_pair_scan", "gla_pair_combine", "gla_selftest_bounded_wait")


class GlaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}" if what else status_string(status))


class gla_fwd_params(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("log_g", ctypes.c_void_p), ("S0", ctypes.c_void_p),
        ("O", ctypes.c_void_p), ("ST", ctypes.c_void_p),
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("T", ctypes.c_int),
        ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("chunk", ctypes.c_int),
        ("dtype", ctypes.c_int), ("gate", ctypes.c_int),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("force_segments", ctypes.c_int), ("path", ctypes.c_int),
        ("log_b", ctypes.c_void_p), ("window_chunks", ctypes.c_int),
    ]


class gla_bwd_params(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("log_g", ctypes.c_void_p), ("S0", ctypes.c_void_p),
        ("grad_O", ctypes.c_void_p), ("grad_ST", ctypes.c_void_p),
        ("grad_q", ctypes.c_void_p), ("grad_k", ctypes.c_void_p), ("grad_v", ctypes.c_void_p),
        ("grad_log_g", ctypes.c_void_p), ("grad_S0", ctypes.c_void_p),
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("T", ctypes.c_int),
        ("dk", ctypes.c_int), ("dv", ctypes.c_int),
        ("dtype", ctypes.c_int), ("gate", ctypes.c_int),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("path", ctypes.c_int),
        ("log_b", ctypes.c_void_p), ("grad_log_b", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libgla.so. Raises if it is missing (unless build_if_missing) or unloadable."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"libgla.so not built ({path}); run __graft_entry__.build() "
                                   "or python -m chunkwise_gated_linear_gla_gb300.build")
            _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(gla_fwd_params)
        vp, i, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
        lib.gla_fwd.restype = st
        lib.gla_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
        lib.gla_fwd_noalloc.restype = st
        lib.gla_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
        lib.gla_fwd_ex.restype = st
        lib.gla_fwd_ex.argtypes = [P, vp]
        lib.gla_fwd_workspace_size.restype = ctypes.c_size_t
        lib.gla_fwd_workspace_size.argtypes = [P]
        lib.gla_fwd_num_stages.restype = i
        lib.gla_fwd_num_stages.argtypes = [P]
        lib.gla_fwd_stage.restype = st
        lib.gla_fwd_stage.argtypes = [P, i, vp]
        lib.gla_fwd_stage_name.restype = ctypes.c_char_p
        lib.gla_fwd_stage_name.argtypes = [P, i]
        lib.gla_bwd.restype = st
        lib.gla_bwd.argtypes = [ctypes.POINTER(gla_bwd_params), vp]
        lib.gla_bwd_workspace_size.restype = ctypes.c_size_t
        lib.gla_bwd_workspace_size.argtypes = [ctypes.POINTER(gla_bwd_params)]
        lib.gla_bwd_num_stages.restype = i
        lib.gla_bwd_num_stages.argtypes = [ctypes.POINTER(gla_bwd_params)]
        lib.gla_bwd_stage.restype = st
        lib.gla_bwd_stage.argtypes = [ctypes.POINTER(gla_bwd_params), i, vp]
        lib.gla_bwd_stage_name.restype = ctypes.c_char_p
        lib.gla_bwd_stage_name.argtypes = [ctypes.POINTER(gla_bwd_params), i]
        lib.gla_fwd_host.restype = st
        lib.gla_fwd_host.argtypes = [P, ctypes.c_size_t, vp]
        lib.gla_host_release.restype = st
        lib.gla_host_release.argtypes = []
        lib.gla_device_status.restype = st
        lib.gla_device_status.argtypes = [vp]
        lib.gla_status_string.restype = ctypes.c_char_p
        lib.gla_status_string.argtypes = [st]
        lib.gla_version.restype = i
        lib.gla_version.argtypes = []
        lib.gla_segment_pair_workspace_size.restype = ctypes.c_size_t
        lib.gla_segment_pair_workspace_size.argtypes = [P]
        lib.gla_segment_pair.restype = st
        lib.gla_segment_pair.argtypes = [P, vp, vp, vp]
        lib.gla_pair_scan.restype = st
        lib.gla_pair_scan.argtypes = [i, vp, vp, vp, vp, vp, i, i, i, i, vp]
        lib.gla_selftest_bounded_wait.restype = st
        lib.gla_selftest_bounded_wait.argtypes = [ctypes.c_uint, i, vp]
        lib.gla_pair_combine.restype = st
        lib.gla_pair_combine.argtypes = [vp, vp, vp, vp, i, i, i, i, vp]
        _lib = lib
        return lib


def status_string(s: int) -> str:
    try:
        return load().gla_status_string(int(s)).decode()
    except Exception:  # pragma: no cover - library missing
        return f"gla_status {s}"


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr() if t.numel() > 0 else None


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(s: int, what: str):
    if s != GLA_OK:
        raise GlaError(s, what)


# ---------------------------------------------------------------- C names

def gla_fwd(q, k, v, log_g, S0, O, ST, B, H, T, dk, dv, chunk=64, stream=None, check=True) -> int:
    s = load().gla_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_g), _ptr(S0), _ptr(O), _ptr(ST),
                       B, H, T, dk, dv, chunk, _stream(stream))
    if check:
        _check(s, "gla_fwd")
    return s


def gla_fwd_noalloc(q, k, v, log_g, S0, O, ST, B, H, T, dk, dv, chunk=64, stream=None, check=True) -> int:
    """gla_fwd without any device allocation (library-owned fixed scratch); see include/gla.h."""
    s = load().gla_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_g), _ptr(S0), _ptr(O), _ptr(ST),
                               B, H, T, dk, dv, chunk, _stream(stream))
    if check:
        _check(s, "gla_fwd_noalloc")
    return s


def gla_fwd_ex(p: gla_fwd_params, stream=None, check=True) -> int:
    s = load().gla_fwd_ex(ctypes.byref(p), _stream(stream))
    if check:
        _check(s, "gla_fwd_ex")
    return s


def gla_fwd_host(p: gla_fwd_params, slice_bytes=0, stream=None, check=True) -> int:
    """gla_fwd_ex with host tensors (see include/gla.h); returns once O and S_T are on the host."""
    s = load().gla_fwd_host(ctypes.byref(p), slice_bytes, _stream(stream))
    if check:
        _check(s, "gla_fwd_host")
    return s


def gla_host_release(check=True) -> int:
    s = load().gla_host_release()
    if check:
        _check(s, "gla_host_release")
    return s


def gla_bwd(p: gla_bwd_params, stream=None, check=True) -> int:
    s = load().gla_bwd(ctypes.byref(p), _stream(stream))
    if check:
        _check(s, "gla_bwd")
    return s


def gla_bwd_workspace_size(p: gla_bwd_params) -> int:
    return int(load().gla_bwd_workspace_size(ctypes.byref(p)))


def gla_bwd_num_stages(p: gla_bwd_params) -> int:
    return int(load().gla_bwd_num_stages(ctypes.byref(p)))


def gla_bwd_stage(p: gla_bwd_params, stage: int, stream=None, check=True) -> int:
    s = load().gla_bwd_stage(ctypes.byref(p), stage, _stream(stream))
    if check:
        _check(s, f"gla_bwd_stage({stage})")
    return s


def gla_bwd_stage_name(p: gla_bwd_params, stage: int) -> str:
    return load().gla_bwd_stage_name(ctypes.byref(p), stage).decode()


def make_bwd_params(q, k, v, log_g, S0, dO, dST, dq, dk, dv, dlog_g, dS0, gate=None,
                    workspace=None, path=GLA_PATH_AUTO, log_b=None, dlog_b=None) -> gla_bwd_params:
    """Fill gla_bwd_params from torch tensors (shapes read from q and v).
    log_b (the bilinear gate's log beta) selects GLA_GATE_BILINEAR; dlog_b receives its gradient."""
    import torch
    B, H, T, dk_ = q.shape
    if gate is None and log_b is not None:
        gate = GLA_GATE_BILINEAR
    if gate is None:
        if log_g is None:
            gate = GLA_GATE_NONE
        else:
            gate = {1: GLA_GATE_HEAD_SCALAR, 3: GLA_GATE_TOKEN_SCALAR}.get(log_g.dim(), GLA_GATE_PER_KEY)
    p = gla_bwd_params()
    p.q, p.k, p.v, p.log_g, p.S0 = _ptr(q), _ptr(k), _ptr(v), _ptr(log_g), _ptr(S0)
    p.grad_O, p.grad_ST = _ptr(dO), _ptr(dST)
    p.grad_q, p.grad_k, p.grad_v, p.grad_log_g, p.grad_S0 = _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dlog_g), _ptr(dS0)
    p.B, p.H, p.T, p.dk, p.dv = B, H, T, dk_, v.shape[-1]
    p.dtype = GLA_BF16 if q.dtype == torch.bfloat16 else GLA_FP32
    p.gate = gate
    p.workspace = _ptr(workspace)
    p.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    p.path = path
    p.log_b, p.grad_log_b = _ptr(log_b), _ptr(dlog_b)
    return p


def backward(q, k, v, log_g, S0, dO, dST=None, gate=None, want_dS0=True, stream=None, path=GLA_PATH_AUTO,
             log_b=None):
    """Allocate the gradients and the workspace with torch, then call gla_bwd.

    Returns (dq, dk, dv, dlog_g, dS0), fp32; dlog_g is None without a gate and
    dS0 None unless wanted. With the bilinear gate (log_b given) dlog_b is
    appended.
    """
    import torch
    B, H, T, dk_ = q.shape
    dv_ = v.shape[-1]
    dev = q.device
    dq = torch.empty((B, H, T, dk_), dtype=torch.float32, device=dev)
    dk = torch.empty((B, H, T, dk_), dtype=torch.float32, device=dev)
    dv = torch.empty((B, H, T, dv_), dtype=torch.float32, device=dev)
    dg = None if log_g is None else torch.empty(log_g.shape, dtype=torch.float32, device=dev)
    dS0 = torch.empty((B, H, dk_, dv_), dtype=torch.float32, device=dev) if want_dS0 else None
    db = None if log_b is None else torch.empty(log_b.shape, dtype=torch.float32, device=dev)
    p = make_bwd_params(q, k, v, log_g, S0, dO, dST, dq, dk, dv, dg, dS0, gate, path=path, log_b=log_b, dlog_b=db)
    n = gla_bwd_workspace_size(p)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
    p.workspace, p.workspace_bytes = ws.data_ptr(), n
    gla_bwd(p, stream)
    if log_b is not None:
        return dq, dk, dv, dg, dS0, db
    return dq, dk, dv, dg, dS0


def gla_fwd_workspace_size(p: gla_fwd_params) -> int:
    return int(load().gla_fwd_workspace_size(ctypes.byref(p)))


def gla_fwd_num_stages(p: gla_fwd_params) -> int:
    return int(load().gla_fwd_num_stages(ctypes.byref(p)))


def gla_fwd_stage(p: gla_fwd_params, stage: int, stream=None, check=True) -> int:
    s = load().gla_fwd_stage(ctypes.byref(p), stage, _stream(stream))
    if check:
        _check(s, f"gla_fwd_stage({stage})")
    return s


def gla_fwd_stage_name(p: gla_fwd_params, stage: int) -> str:
    return load().gla_fwd_stage_name(ctypes.byref(p), stage).decode()


def gla_device_status(stream=None) -> int:
    return int(load().gla_device_status(_stream(stream)))


def gla_status_string(s: int) -> str:
    return load().gla_status_string(int(s)).decode()


def gla_version() -> int:
    return int(load().gla_version())


def gla_segment_pair_workspace_size(p: gla_fwd_params) -> int:
    return int(load().gla_segment_pair_workspace_size(ctypes.byref(p)))


def gla_segment_pair(p: gla_fwd_params, log_Gamma, S_star, stream=None, check=True) -> int:
    s = load().gla_segment_pair(ctypes.byref(p), _ptr(log_Gamma), _ptr(S_star), _stream(stream))
    if check:
        _check(s, "gla_segment_pair")
    return s


def gla_pair_scan(P, log_Gamma, S_star, S0, S_in, S_T, B, H, dk, dv, stream=None, check=True) -> int:
    s = load().gla_pair_scan(P, _ptr(log_Gamma), _ptr(S_star), _ptr(S0), _ptr(S_in), _ptr(S_T),
                             B, H, dk, dv, _stream(stream))
    if check:
        _check(s, "gla_pair_scan")
    return s


def gla_pair_combine(log_Gamma2, S2, log_Gamma1, S1, B, H, dk, dv, stream=None, check=True) -> int:
    s = load().gla_pair_combine(_ptr(log_Gamma2), _ptr(S2), _ptr(log_Gamma1), _ptr(S1), B, H, dk, dv,
                                _stream(stream))
    if check:
        _check(s, "gla_pair_combine")
    return s


def gla_selftest_bounded_wait(limit_us: int, arrive: bool = False, stream=None, check=True) -> int:
    s = load().gla_selftest_bounded_wait(int(limit_us), 1 if arrive else 0, _stream(stream))
    if check:
        _check(s, "gla_selftest_bounded_wait")
    return s


# ---------------------------------------------------------------- marshalling helpers

def make_params(q, k, v, log_g, S0, O, ST, gate=None, path=GLA_PATH_AUTO, force_segments=0,
                workspace=None, chunk=64, log_b=None, window_chunks=0) -> gla_fwd_params:
    """Fill gla_fwd_params from torch tensors (shapes read from q and v).
    log_b (the bilinear gate's log beta, [B,H,T,dv]) selects GLA_GATE_BILINEAR."""
    import torch
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if gate is None and log_b is not None:
        gate = GLA_GATE_BILINEAR
    if gate is None:
        if log_g is None:
            gate = GLA_GATE_NONE
        else:
            gate = {1: GLA_GATE_HEAD_SCALAR, 3: GLA_GATE_TOKEN_SCALAR}.get(log_g.dim(), GLA_GATE_PER_KEY)
    p = gla_fwd_params()
    p.q, p.k, p.v = _ptr(q), _ptr(k), _ptr(v)
    p.log_g, p.S0, p.O, p.ST = _ptr(log_g), _ptr(S0), _ptr(O), _ptr(ST)
    p.B, p.H, p.T, p.dk, p.dv, p.chunk = B, H, T, dk, dv, chunk
    p.dtype = GLA_BF16 if q.dtype == torch.bfloat16 else GLA_FP32
    p.gate = gate
    p.workspace = _ptr(workspace)
    p.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    p.force_segments = force_segments
    p.path = path
    p.log_b = _ptr(log_b)
    p.window_chunks = window_chunks
    return p


def forward(q, k, v, log_g=None, S0=None, gate=None, want_state=True, path=GLA_PATH_AUTO,
            force_segments=0, stream=None, O=None, ST=None, log_b=None, window_chunks=0):
    """Allocate O (and ST) and the workspace with torch, then call gla_fwd_ex.

    q, k: [B,H,T,dk]; v: [B,H,T,dv] (bf16 or fp32, on the GPU); log_g fp32
    [B,H,T,dk] (per key) or [H] (per-head scalar) or None; S0 fp32 [B,H,dk,dv]
    or None. Returns (O, ST).
    """
    import torch
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if O is None:
        O = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    if ST is None and want_state:
        ST = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    p = make_params(q, k, v, log_g, S0, O, ST, gate, path, force_segments, log_b=log_b,
                    window_chunks=window_chunks)
    nbytes = gla_fwd_workspace_size(p)
    ws = None
    if nbytes > 0:
        ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=q.device)
        off = (-ws.data_ptr()) % 256
        ws = ws[off:off + nbytes]
        p.workspace = ws.data_ptr()
        p.workspace_bytes = nbytes
    gla_fwd_ex(p, stream)
    return O, ST


def _aligned_workspace(nbytes, device):
    import torch
    if nbytes == 0:
        return None
    ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + nbytes]


def segment_pair(k, v, log_g=None, gate=None, q=None, path=GLA_PATH_AUTO, stream=None):
    """The exchange pair (log Gamma [B,H,dk], S* [B,H,dk,dv], both fp32) of the segment
    whose k, v, gate are given, from a zero start (gla_segment_pair)."""
    import torch
    B, H, T, dk = k.shape
    dv = v.shape[-1]
    log_G = torch.empty((B, H, dk), dtype=torch.float32, device=k.device)
    S_star = torch.empty((B, H, dk, dv), dtype=torch.float32, device=k.device)
    p = make_params(k, k, v, log_g, None, None, None, gate, path)
    p.q = _ptr(q)
    ws = _aligned_workspace(gla_segment_pair_workspace_size(p), k.device)
    if ws is not None:
        p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    gla_segment_pair(p, log_G, S_star, stream)
    return log_G, S_star


def pair_scan(log_Gamma, S_star, S0=None, want_S_in=True, stream=None):
    """States entering each of P segments and after the last, from pairs stacked in
    sequence order (log_Gamma [P,B,H,dk], S_star [P,B,H,dk,dv]): (S_in [P,...] or None, S_T)."""
    import torch
    P, B, H, dk = log_Gamma.shape
    dv = S_star.shape[-1]
    S_in = torch.empty_like(S_star) if want_S_in else None
    S_T = torch.empty((B, H, dk, dv), dtype=torch.float32, device=S_star.device)
    gla_pair_scan(P, log_Gamma, S_star, S0, S_in, S_T, B, H, dk, dv, stream)
    return S_in, S_T


def pair_combine(log_Gamma2, S2, log_Gamma1, S1, stream=None):
    """In place: (log_Gamma1, S1) <- (log_Gamma2, S2) o (log_Gamma1, S1); pair 1 is the earlier segment."""
    B, H, dk, dv = S1.shape
    gla_pair_combine(log_Gamma2, S2, log_Gamma1, S1, B, H, dk, dv, stream)
    return log_Gamma1, S1
