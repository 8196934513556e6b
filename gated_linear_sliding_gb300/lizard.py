"""Python binding of liblizard.so: argument marshalling only.

Every function here checks tensor shapes, dtypes and contiguity, then calls the
C entry point of the same name with raw device pointers and the current CUDA
stream.  All arithmetic runs in the library's CUDA kernels; there is no CPU
path.  If the library has not been built, loading it raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

import torch

from . import _build

LIZARD_OK = 0
LIZARD_ERR_INVALID_ARG = 1
LIZARD_ERR_UNSUPPORTED = 2
LIZARD_ERR_WORKSPACE = 3
LIZARD_ERR_CUDA = 4
LIZARD_ERR_TIMEOUT = 5
LIZARD_F32 = 0
LIZARD_BF16 = 1
# decay readings (include/lizard.h, lizard_decay)
LIZARD_DECAY_DELAYED = 0
LIZARD_DECAY_MASKED = 1
LIZARD_DECAY_LAGGED = 2

EXPORTED = ["lizard_attn_fwd_workspace", "lizard_workspace_init", "lizard_attn_fwd",
            "lizard_attn_bwd_workspace", "lizard_attn_bwd", "lizard_decode_workspace",
            "lizard_decode_step", "lizard_decode_step_positions", "lizard_read_device_status",
            "lizard_status_string",
            "lizard_profile_events", "lizard_version", "lizard_attn_fwd_noalloc",
            "lizard_attn_fwd_kernel", "lizard_selftest_wait_timeout", "lizard_attn_fwd_varlen",
            "lizard_attn_fwd_varlen_workspace",
            "lizard_attn_bwd_varlen_workspace", "lizard_attn_bwd_varlen",
            "lizard_attn_fwd_noalloc_scratch", "lizard_read_noalloc_status",
            "lizard_qkvg_proj", "lizard_qkvg_proj_bwd", "lizard_gate_cache_fill"]


class lizard_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("L", ctypes.c_int64), ("Hq", ctypes.c_int64),
                ("Hkv", ctypes.c_int64), ("d", ctypes.c_int64), ("D", ctypes.c_int64),
                ("w", ctypes.c_int64), ("M", ctypes.c_int64), ("chunk", ctypes.c_int64),
                ("scale", ctypes.c_float), ("dtype", ctypes.c_int32), ("decay", ctypes.c_int32)]


class LizardError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib = None
_VP = ctypes.c_void_p
_DP = ctypes.POINTER(lizard_dims)


def load(path: str | None = None) -> ctypes.CDLL:
    """Load liblizard.so; raises if it is missing (build it with __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: the CUDA library must be built first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    lib.lizard_attn_fwd_workspace.argtypes = [_DP]
    lib.lizard_attn_fwd_workspace.restype = ctypes.c_size_t
    lib.lizard_attn_bwd_workspace.argtypes = [_DP]
    lib.lizard_attn_bwd_workspace.restype = ctypes.c_size_t
    lib.lizard_decode_workspace.argtypes = [_DP]
    lib.lizard_decode_workspace.restype = ctypes.c_size_t
    lib.lizard_selftest_wait_timeout.argtypes = [_VP, ctypes.c_size_t, ctypes.c_longlong, _VP]
    lib.lizard_selftest_wait_timeout.restype = ctypes.c_int
    lib.lizard_attn_fwd_kernel.argtypes = [_DP]
    lib.lizard_attn_fwd_kernel.restype = ctypes.c_int
    lib.lizard_workspace_init.argtypes = [_VP, ctypes.c_size_t, _VP]
    lib.lizard_workspace_init.restype = ctypes.c_int
    lib.lizard_attn_fwd.argtypes = [_DP] + [_VP] * 13 + [ctypes.c_size_t, _VP]
    lib.lizard_attn_fwd.restype = ctypes.c_int
    lib.lizard_attn_fwd_varlen_workspace.argtypes = [_DP, _VP]
    lib.lizard_attn_fwd_varlen_workspace.restype = ctypes.c_size_t
    lib.lizard_attn_fwd_varlen.argtypes = [_DP, _VP] + [_VP] * 13 + [ctypes.c_size_t, _VP]
    lib.lizard_attn_fwd_varlen.restype = ctypes.c_int
    lib.lizard_attn_bwd_varlen_workspace.argtypes = [_DP, _VP]
    lib.lizard_attn_bwd_varlen_workspace.restype = ctypes.c_size_t
    lib.lizard_attn_bwd_varlen.argtypes = [_DP, _VP] + [_VP] * 16 + [ctypes.c_size_t, _VP]
    lib.lizard_attn_bwd_varlen.restype = ctypes.c_int
    lib.lizard_attn_fwd_noalloc.argtypes = [_DP] + [_VP] * 13
    lib.lizard_attn_fwd_noalloc.restype = ctypes.c_int
    lib.lizard_attn_fwd_noalloc_scratch.argtypes = [_DP]
    lib.lizard_attn_fwd_noalloc_scratch.restype = ctypes.c_size_t
    lib.lizard_read_noalloc_status.argtypes = [_VP]
    lib.lizard_read_noalloc_status.restype = ctypes.c_int
    lib.lizard_qkvg_proj.argtypes = [_DP, ctypes.c_int64] + [_VP] * 7 + [ctypes.c_size_t, _VP]
    lib.lizard_qkvg_proj.restype = ctypes.c_int
    lib.lizard_qkvg_proj_bwd.argtypes = [_DP, ctypes.c_int64] + [_VP] * 9 + [ctypes.c_size_t, _VP]
    lib.lizard_qkvg_proj_bwd.restype = ctypes.c_int
    lib.lizard_attn_bwd.argtypes = [_DP] + [_VP] * 16 + [ctypes.c_size_t, _VP]
    lib.lizard_attn_bwd.restype = ctypes.c_int
    lib.lizard_decode_step.argtypes = [_DP, ctypes.c_int64] + [_VP] * 13 + [ctypes.c_size_t, _VP]
    lib.lizard_decode_step.restype = ctypes.c_int
    lib.lizard_decode_step_positions.argtypes = [_DP] + [_VP] * 14 + [ctypes.c_size_t, _VP]
    lib.lizard_decode_step_positions.restype = ctypes.c_int
    lib.lizard_gate_cache_fill.argtypes = [_DP, _VP, _VP, _VP]
    lib.lizard_gate_cache_fill.restype = ctypes.c_int
    lib.lizard_read_device_status.argtypes = [_VP, _VP]
    lib.lizard_read_device_status.restype = ctypes.c_int
    lib.lizard_status_string.argtypes = [ctypes.c_int]
    lib.lizard_status_string.restype = ctypes.c_char_p
    lib.lizard_profile_events.argtypes = [_VP, _VP]
    lib.lizard_profile_events.restype = ctypes.c_int
    lib.lizard_version.argtypes = []
    lib.lizard_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().lizard_status_string(status).decode()


def lizard_version() -> str:
    return load().lizard_version().decode()


def _check(status: int, where: str):
    if status != LIZARD_OK:
        raise LizardError(status, where)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return LIZARD_F32
    if t.dtype == torch.bfloat16:
        return LIZARD_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def make_dims(B, L, Hq, Hkv, d, D, w, M, dtype, scale: float = 0.0, chunk: int = 0,
              decay: int = LIZARD_DECAY_DELAYED) -> lizard_dims:
    code = dtype if isinstance(dtype, int) else _dtype_code(torch.empty(0, dtype=dtype))
    return lizard_dims(B, L, Hq, Hkv, d, D, w, M, chunk, float(scale), code, int(decay))


def dims_of(q, k, g, sinks, w: int, scale: float = 0.0,
            decay: int = LIZARD_DECAY_DELAYED) -> lizard_dims:
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    D = g.shape[-1]
    M = sinks.shape[1]
    return lizard_dims(B, L, Hq, Hkv, d, D, w, M, 0, float(scale), _dtype_code(q), int(decay))


def _need(t, name, shape, dtype):
    if t is None:
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype} != {dtype}")
    if not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def lizard_attn_fwd_workspace(dims: lizard_dims) -> int:
    return int(load().lizard_attn_fwd_workspace(ctypes.byref(dims)))


def lizard_attn_fwd_kernel(dims: lizard_dims) -> int:
    """1 if the tensor-core chunk walk serves these sizes, 0 for the SIMT walk, -1 invalid."""
    return int(load().lizard_attn_fwd_kernel(ctypes.byref(dims)))


def lizard_attn_bwd_workspace(dims: lizard_dims) -> int:
    return int(load().lizard_attn_bwd_workspace(ctypes.byref(dims)))


def lizard_decode_workspace(dims: lizard_dims) -> int:
    return int(load().lizard_decode_workspace(ctypes.byref(dims)))


def new_workspace(nbytes: int, device, stream=None) -> torch.Tensor:
    """Allocate a workspace (torch owns the memory) and zero its status word."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    _check(load().lizard_workspace_init(_p(ws), ws.numel(), _stream(stream)),
           "lizard_workspace_init")
    return ws


def lizard_profile_events(before=None, after=None):
    """Bracket the dominant kernel of later forward/backward calls with two
    torch.cuda.Event objects (None, None turns it off)."""
    handles = []
    for ev in (before, after):
        if ev is None:
            handles.append(None)
            continue
        if not ev.cuda_event:
            ev.record()  # torch creates the underlying cudaEvent_t on first record
        handles.append(ctypes.c_void_p(ev.cuda_event))
    _check(load().lizard_profile_events(*handles), "lizard_profile_events")


def lizard_selftest_wait_timeout(workspace, limit_cycles: int, stream=None):
    """Run the bounded-wait failure path once (see include/lizard.h).  workspace None targets
    the status word of lizard_attn_fwd_noalloc's fixed array."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().lizard_selftest_wait_timeout(_p(workspace), nbytes, int(limit_cycles),
                                               _stream(stream)), "lizard_selftest_wait_timeout")


def lizard_read_noalloc_status(stream=None) -> int:
    """Synchronise the stream, read and clear lizard_attn_fwd_noalloc's status word."""
    return int(load().lizard_read_noalloc_status(_stream(stream)))


def lizard_attn_fwd_noalloc_scratch(dims) -> int:
    return int(load().lizard_attn_fwd_noalloc_scratch(ctypes.byref(dims)))


def lizard_read_device_status(workspace: torch.Tensor, stream=None) -> int:
    return int(load().lizard_read_device_status(_p(workspace), _stream(stream)))


def lizard_attn_fwd(q, k, v, g, Wf, sinks, w: int, *, scale: float = 0.0, y=None, lse=None,
                    S_out=None, z_out=None, kcache_out=None, vcache_out=None, workspace=None,
                    stream=None, decay: int = LIZARD_DECAY_DELAYED):
    """Forward over L tokens.  Returns y [B, L, Hq, d] (allocated if not given).  `decay`
    selects the decay reading (LIZARD_DECAY_*)."""
    B, L, Hq, d = q.shape
    Hkv, D, M = k.shape[2], g.shape[-1], sinks.shape[1]
    dt = q.dtype
    _need(q, "q", (B, L, Hq, d), dt)
    _need(k, "k", (B, L, Hkv, d), dt)
    _need(v, "v", (B, L, Hkv, d), dt)
    _need(g, "g", (B, L, Hkv, D), dt)
    _need(Wf, "Wf", (Hkv, d, D // 2), dt)
    _need(sinks, "sinks", (Hq, M), torch.float32)
    if y is None:
        y = torch.empty_like(q)
    _need(y, "y", (B, L, Hq, d), dt)
    if lse is not None:
        _need(lse, "lse", (B, L, Hq), torch.float32)
    if S_out is not None:
        _need(S_out, "S_out", (B, Hkv, D, d), torch.float32)
        _need(z_out, "z_out", (B, Hkv, D), torch.float32)
    if kcache_out is not None:
        _need(kcache_out, "kcache_out", (B, Hkv, w + 1, d), dt)
        _need(vcache_out, "vcache_out", (B, Hkv, w + 1, d), dt)
    dims = dims_of(q, k, g, sinks, w, scale, decay)
    if workspace is None:
        workspace = new_workspace(lizard_attn_fwd_workspace(dims), q.device, stream)
    st = load().lizard_attn_fwd(ctypes.byref(dims), _p(q), _p(k), _p(v), _p(g), _p(Wf),
                                _p(sinks), _p(y), _p(lse), _p(S_out), _p(z_out), _p(kcache_out),
                                _p(vcache_out), _p(workspace), workspace.numel(),
                                _stream(stream))
    _check(st, "lizard_attn_fwd")
    return y


def lizard_attn_fwd_varlen_workspace(dims, cu_seqlens) -> int:
    """Workspace bytes for one launch of lizard_attn_fwd_varlen over all sequences."""
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    return int(load().lizard_attn_fwd_varlen_workspace(ctypes.byref(dims), cu.ctypes.data))


def lizard_attn_fwd_varlen(q, k, v, g, Wf, sinks, w: int, cu_seqlens, *, scale: float = 0.0,
                           y=None, lse=None, S_out=None, z_out=None, kcache_out=None,
                           vcache_out=None, workspace=None, stream=None,
                           decay: int = LIZARD_DECAY_DELAYED):
    """Forward over a packed batch: q [T, Hq, d], k, v [T, Hkv, d], g [T, Hkv, D], and
    cu_seqlens (host integers, B + 1 offsets) delimiting B sequences.  Returns y [T, Hq, d];
    S_out, z_out, kcache_out, vcache_out hold one entry per sequence."""
    T, Hq, d = q.shape
    Hkv, D, M = k.shape[1], g.shape[-1], sinks.shape[1]
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    nseq = cu.shape[0] - 1
    dt = q.dtype
    _need(q, "q", (T, Hq, d), dt)
    _need(k, "k", (T, Hkv, d), dt)
    _need(v, "v", (T, Hkv, d), dt)
    _need(g, "g", (T, Hkv, D), dt)
    _need(Wf, "Wf", (Hkv, d, D // 2), dt)
    _need(sinks, "sinks", (Hq, M), torch.float32)
    if y is None:
        y = torch.empty_like(q)
    _need(y, "y", (T, Hq, d), dt)
    if lse is not None:
        _need(lse, "lse", (T, Hq), torch.float32)
    if S_out is not None:
        _need(S_out, "S_out", (nseq, Hkv, D, d), torch.float32)
        _need(z_out, "z_out", (nseq, Hkv, D), torch.float32)
    if kcache_out is not None:
        _need(kcache_out, "kcache_out", (nseq, Hkv, w + 1, d), dt)
        _need(vcache_out, "vcache_out", (nseq, Hkv, w + 1, d), dt)
    dims = lizard_dims(nseq, T, Hq, Hkv, d, D, w, M, 0, float(scale), _dtype_code(q), int(decay))
    if workspace is None:  # the size of one launch over all sequences
        workspace = new_workspace(lizard_attn_fwd_varlen_workspace(dims, cu), q.device, stream)
    st = load().lizard_attn_fwd_varlen(ctypes.byref(dims), cu.ctypes.data, _p(q), _p(k), _p(v),
                                       _p(g), _p(Wf), _p(sinks), _p(y), _p(lse), _p(S_out),
                                       _p(z_out), _p(kcache_out), _p(vcache_out), _p(workspace),
                                       workspace.numel(), _stream(stream))
    _check(st, "lizard_attn_fwd_varlen")
    return y


def lizard_attn_fwd_noalloc(q, k, v, g, Wf, sinks, w: int, *, scale: float = 0.0, y=None,
                            lse=None, S_out=None, z_out=None, kcache_out=None, vcache_out=None,
                            stream=None, decay: int = LIZARD_DECAY_DELAYED):
    """The forward without a workspace, for callers that cannot allocate device memory.

    Same arguments and result as lizard_attn_fwd; the library keeps the scratch in a
    fixed 32 MiB device array (see include/lizard.h for the limit and the sharing rules).
    `y` is allocated here only for the Python caller's convenience when not given."""
    B, L, Hq, d = q.shape
    Hkv, D, M = k.shape[2], g.shape[-1], sinks.shape[1]
    dt = q.dtype
    _need(q, "q", (B, L, Hq, d), dt)
    _need(k, "k", (B, L, Hkv, d), dt)
    _need(v, "v", (B, L, Hkv, d), dt)
    _need(g, "g", (B, L, Hkv, D), dt)
    _need(Wf, "Wf", (Hkv, d, D // 2), dt)
    _need(sinks, "sinks", (Hq, M), torch.float32)
    if y is None:
        y = torch.empty_like(q)
    _need(y, "y", (B, L, Hq, d), dt)
    dims = dims_of(q, k, g, sinks, w, scale, decay)
    st = load().lizard_attn_fwd_noalloc(ctypes.byref(dims), _p(q), _p(k), _p(v), _p(g), _p(Wf),
                                        _p(sinks), _p(y), _p(lse), _p(S_out), _p(z_out),
                                        _p(kcache_out), _p(vcache_out), _stream(stream))
    _check(st, "lizard_attn_fwd_noalloc")
    return y


def lizard_attn_bwd(q, k, v, g, Wf, sinks, y, lse, dy, w: int, *, scale: float = 0.0,
                    dq=None, dk=None, dv=None, dg=None, dWf=None, dsinks=None, workspace=None,
                    stream=None, decay: int = LIZARD_DECAY_DELAYED):
    """Gradients (dq, dk, dv, dg, dWf, dsinks) of y against dy (same decay reading as the
    forward that made y)."""
    B, L, Hq, d = q.shape
    Hkv, D, M = k.shape[2], g.shape[-1], sinks.shape[1]
    dt = q.dtype
    for t, n, shp in ((q, "q", (B, L, Hq, d)), (k, "k", (B, L, Hkv, d)), (v, "v", (B, L, Hkv, d)),
                      (g, "g", (B, L, Hkv, D)), (Wf, "Wf", (Hkv, d, D // 2)),
                      (y, "y", (B, L, Hq, d)), (dy, "dy", (B, L, Hq, d))):
        _need(t, n, shp, dt)
    _need(sinks, "sinks", (Hq, M), torch.float32)
    _need(lse, "lse", (B, L, Hq), torch.float32)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    dg = torch.empty_like(g) if dg is None else dg
    dWf = torch.empty(Hkv, d, D // 2, dtype=torch.float32, device=q.device) if dWf is None else dWf
    dsinks = torch.empty(Hq, M, dtype=torch.float32, device=q.device) if dsinks is None else dsinks
    dims = dims_of(q, k, g, sinks, w, scale, decay)
    if workspace is None:
        workspace = new_workspace(lizard_attn_bwd_workspace(dims), q.device, stream)
    st = load().lizard_attn_bwd(ctypes.byref(dims), _p(q), _p(k), _p(v), _p(g), _p(Wf),
                                _p(sinks), _p(y), _p(lse), _p(dy), _p(dq), _p(dk), _p(dv),
                                _p(dg), _p(dWf), _p(dsinks), _p(workspace), workspace.numel(),
                                _stream(stream))
    _check(st, "lizard_attn_bwd")
    return dict(dq=dq, dk=dk, dv=dv, dg=dg, dWf=dWf, dsinks=dsinks)


def lizard_attn_bwd_varlen_workspace(dims, cu_seqlens) -> int:
    """Workspace bytes of lizard_attn_bwd_varlen for this packed batch (0: bad offsets)."""
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    return int(load().lizard_attn_bwd_varlen_workspace(ctypes.byref(dims), cu.ctypes.data))


def lizard_attn_bwd_varlen(q, k, v, g, Wf, sinks, y, lse, dy, w: int, cu_seqlens, *,
                           scale: float = 0.0, workspace=None, stream=None,
                           decay: int = LIZARD_DECAY_DELAYED):
    """Gradients of lizard_attn_fwd_varlen's y against dy for a packed batch: dq, dk, dv,
    dg packed like the inputs; dWf and dsinks summed over the sequences."""
    T, Hq, d = q.shape
    Hkv, D, M = k.shape[1], g.shape[-1], sinks.shape[1]
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    nseq = cu.shape[0] - 1
    dt = q.dtype
    for t, n, shp in ((q, "q", (T, Hq, d)), (k, "k", (T, Hkv, d)), (v, "v", (T, Hkv, d)),
                      (g, "g", (T, Hkv, D)), (Wf, "Wf", (Hkv, d, D // 2)),
                      (y, "y", (T, Hq, d)), (dy, "dy", (T, Hq, d))):
        _need(t, n, shp, dt)
    _need(sinks, "sinks", (Hq, M), torch.float32)
    _need(lse, "lse", (T, Hq), torch.float32)
    dq, dk, dv, dg = (torch.empty_like(x) for x in (q, k, v, g))
    dWf = torch.empty(Hkv, d, D // 2, dtype=torch.float32, device=q.device)
    dsinks = torch.empty(Hq, M, dtype=torch.float32, device=q.device)
    dims = lizard_dims(nseq, T, Hq, Hkv, d, D, w, M, 0, float(scale), _dtype_code(q), int(decay))
    if workspace is None:
        nbytes = int(load().lizard_attn_bwd_varlen_workspace(ctypes.byref(dims), cu.ctypes.data))
        if nbytes == 0:
            raise ValueError("cu_seqlens: inconsistent offsets")
        workspace = new_workspace(nbytes, q.device, stream)
    st = load().lizard_attn_bwd_varlen(ctypes.byref(dims), cu.ctypes.data, _p(q), _p(k), _p(v),
                                       _p(g), _p(Wf), _p(sinks), _p(y), _p(lse), _p(dy),
                                       _p(dq), _p(dk), _p(dv), _p(dg), _p(dWf), _p(dsinks),
                                       _p(workspace), workspace.numel(), _stream(stream))
    _check(st, "lizard_attn_bwd_varlen")
    return dict(dq=dq, dk=dk, dv=dv, dg=dg, dWf=dWf, dsinks=dsinks)


def _decode_common(q, k, v, g, Wf, sinks, S, z, kcache, vcache, gcache, w, decay):
    B, Hq, d = q.shape
    Hkv, D, M = k.shape[1], g.shape[-1], sinks.shape[1]
    dt = q.dtype
    _need(k, "k", (B, Hkv, d), dt)
    _need(v, "v", (B, Hkv, d), dt)
    _need(g, "g", (B, Hkv, D), dt)
    _need(Wf, "Wf", (Hkv, d, D // 2), dt)
    _need(sinks, "sinks", (Hq, M), torch.float32)
    _need(S, "S", (B, Hkv, D, d), torch.float32)
    _need(z, "z", (B, Hkv, D), torch.float32)
    _need(kcache, "kcache", (B, Hkv, w + 1, d), dt)
    _need(vcache, "vcache", (B, Hkv, w + 1, d), dt)
    if decay != LIZARD_DECAY_DELAYED or gcache is not None:
        _need(gcache, "gcache", (B, Hkv, w + 1, D), dt)
    return B, Hq, Hkv, d, D, M


def lizard_decode_step(pos: int, q, k, v, g, Wf, sinks, S, z, kcache, vcache, w: int, *,
                       scale: float = 0.0, y=None, workspace=None, stream=None, gcache=None,
                       decay: int = LIZARD_DECAY_DELAYED):
    """One decode step at position pos; S, z, kcache, vcache (and gcache, the gate ring the
    MASKED and LAGGED readings need) are updated in place."""
    B, Hq, Hkv, d, D, M = _decode_common(q, k, v, g, Wf, sinks, S, z, kcache, vcache, gcache,
                                         w, decay)
    y = torch.empty_like(q) if y is None else y
    dims = lizard_dims(B, 1, Hq, Hkv, d, D, w, M, 0, float(scale), _dtype_code(q), int(decay))
    if workspace is None:
        workspace = new_workspace(lizard_decode_workspace(dims), q.device, stream)
    st = load().lizard_decode_step(ctypes.byref(dims), int(pos), _p(q), _p(k), _p(v), _p(g),
                                   _p(Wf), _p(sinks), _p(y), _p(S), _p(z), _p(kcache),
                                   _p(vcache), _p(gcache), _p(workspace), workspace.numel(),
                                   _stream(stream))
    _check(st, "lizard_decode_step")
    return y


def lizard_decode_step_positions(pos, q, k, v, g, Wf, sinks, S, z, kcache, vcache, w: int, *,
                                 scale: float = 0.0, y=None, workspace=None, stream=None,
                                 gcache=None, decay: int = LIZARD_DECAY_DELAYED):
    """One decode step with a position per sequence: pos is an int64 device tensor [B],
    read when the kernel runs.  A negative entry is reported through the workspace status
    (lizard_read_device_status) and leaves that sequence untouched."""
    B = q.shape[0]
    _need(pos, "pos", (B,), torch.int64)
    B, Hq, Hkv, d, D, M = _decode_common(q, k, v, g, Wf, sinks, S, z, kcache, vcache, gcache,
                                         w, decay)
    y = torch.empty_like(q) if y is None else y
    dims = lizard_dims(B, 1, Hq, Hkv, d, D, w, M, 0, float(scale), _dtype_code(q), int(decay))
    if workspace is None:
        workspace = new_workspace(lizard_decode_workspace(dims), q.device, stream)
    st = load().lizard_decode_step_positions(ctypes.byref(dims), _p(pos), _p(q), _p(k), _p(v),
                                             _p(g), _p(Wf), _p(sinks), _p(y), _p(S), _p(z),
                                             _p(kcache), _p(vcache), _p(gcache), _p(workspace),
                                             workspace.numel(), _stream(stream))
    _check(st, "lizard_decode_step_positions")
    return y


def lizard_gate_cache_fill(g, gcache, w: int, *, stream=None):
    """Gate ring of a prefill: the gate rows of the last min(L, w) tokens of g [B, L, Hkv, D]
    go to slot t mod (w+1) of gcache [B, Hkv, w+1, D] (same dtype)."""
    B, L, Hkv, D = g.shape
    _need(g, "g", (B, L, Hkv, D), g.dtype)
    _need(gcache, "gcache", (B, Hkv, w + 1, D), g.dtype)
    dims = lizard_dims(B, L, Hkv, Hkv, D, D, w, 0, 0, 0.0, _dtype_code(g))
    _check(load().lizard_gate_cache_fill(ctypes.byref(dims), _p(g), _p(gcache), _stream(stream)),
           "lizard_gate_cache_fill")


def lizard_qkvg_proj(x, W, Hq: int, Hkv: int, d: int, D: int, *, q=None, k=None, v=None,
                     g=None, workspace=None, stream=None):
    """[q | k | v | g] = x W^T on the tensor cores.  x [B, L, dm], W [N, dm] (bf16).
    Returns (q, k, v, g) in the mixer's layouts (allocated if not given)."""
    B, L, dm = x.shape
    N = Hq * d + 2 * Hkv * d + Hkv * D
    _need(x, "x", (B, L, dm), torch.bfloat16)
    _need(W, "W", (N, dm), torch.bfloat16)
    outs = []
    for t, name, shape in ((q, "q", (B, L, Hq, d)), (k, "k", (B, L, Hkv, d)),
                           (v, "v", (B, L, Hkv, d)), (g, "g", (B, L, Hkv, D))):
        if t is None:
            t = torch.empty(shape, dtype=torch.bfloat16, device=x.device)
        _need(t, name, shape, torch.bfloat16)
        outs.append(t)
    dims = make_dims(B, L, Hq, Hkv, d, D, 1, 0, LIZARD_BF16)
    nb = 0 if workspace is None else workspace.numel()
    st = load().lizard_qkvg_proj(ctypes.byref(dims), dm, _p(x), _p(W), *[_p(t) for t in outs],
                                 _p(workspace), nb, _stream(stream))
    _check(st, "lizard_qkvg_proj")
    return tuple(outs)


def lizard_qkvg_proj_bwd(x, W, dq, dk, dv, dg, *, dx=None, dW=None, workspace=None,
                         stream=None):
    """dx = dY W (bf16) and dW = dY^T x (fp32) for dY = [dq | dk | dv | dg]."""
    B, L, dm = x.shape
    Hq, d = dq.shape[2], dq.shape[3]
    Hkv, D = dg.shape[2], dg.shape[3]
    N = Hq * d + 2 * Hkv * d + Hkv * D
    _need(x, "x", (B, L, dm), torch.bfloat16)
    _need(W, "W", (N, dm), torch.bfloat16)
    _need(dq, "dq", (B, L, Hq, d), torch.bfloat16)
    _need(dk, "dk", (B, L, Hkv, d), torch.bfloat16)
    _need(dv, "dv", (B, L, Hkv, d), torch.bfloat16)
    _need(dg, "dg", (B, L, Hkv, D), torch.bfloat16)
    if dx is None:
        dx = torch.empty_like(x)
    if dW is None:
        dW = torch.empty(N, dm, dtype=torch.float32, device=x.device)
    _need(dx, "dx", (B, L, dm), torch.bfloat16)
    _need(dW, "dW", (N, dm), torch.float32)
    dims = make_dims(B, L, Hq, Hkv, d, D, 1, 0, LIZARD_BF16)
    nb = 0 if workspace is None else workspace.numel()
    st = load().lizard_qkvg_proj_bwd(ctypes.byref(dims), dm, _p(x), _p(W), _p(dq), _p(dk),
                                     _p(dv), _p(dg), _p(dx), _p(dW), _p(workspace), nb,
                                     _stream(stream))
    _check(st, "lizard_qkvg_proj_bwd")
    return dx, dW
