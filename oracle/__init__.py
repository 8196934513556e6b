"""Float64 CPU oracle of the Lizard hybrid token mixer.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product library never imports it,
and this package imports nothing from the product package.

The main oracle is the token-by-token recurrence in `lizard_oracle.c` (plain C,
fp64, OpenMP over (batch, KV head) units), loaded here with ctypes.  The
projections in front of the mixer (q, k, v and the gate logits from the layer
input) are plain fp64 matrix products, `qkvg_proj` and `qkvg_proj_bwd`.  The
alternate forms in `forms.py` (brute force, quadratic-parallel, chunked with
explicit products, chunked in log space) exist to pin it.

Sources: Lizard summary (gist.science/ko/paper/2507.09025), sec. 2-A-1 (gated
linear attention with a sigmoid gate and a constant-size state), sec. 2-A-2
(sliding-window attention with meta-memory scalars in the denominator), sec.
2-C (non-negative Hedgehog feature map, log-space gates).
Parity status: pinned (see tests/test_oracle_*.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lizard_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/liboracle.so (gcc, OpenMP, -O2)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC,
                           "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_long) for n in ("B", "L", "Hq", "Hkv", "d", "D", "w", "M",
                                             "reading")] + [("scale", ctypes.c_double)]


# Readings of which gates decay a key that has left the window (the pages fix none):
# the weight of key j <= i - w at query i is the product of Gamma_s over
#   DELAYED  s = j+w+1 .. i   (the key enters the state undecayed as it leaves the window),
#   MASKED   s = j+1 .. i     (full gated linear attention with the window masked out),
#   LAGGED   s = j+1 .. i-w   (the query reads the state of token i-w).
DELAYED, MASKED, LAGGED = 0, 1, 2


_P = ctypes.POINTER(ctypes.c_double)


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.ora_fwd.argtypes = [ctypes.POINTER(_Dims)] + [_P] * 14
        lib.ora_fwd.restype = ctypes.c_int
        lib.ora_decode_step.argtypes = [ctypes.POINTER(_Dims), ctypes.c_long] + [_P] * 12
        lib.ora_decode_step.restype = ctypes.c_int
        lib.ora_bwd.argtypes = [ctypes.POINTER(_Dims)] + [_P] * 13
        lib.ora_bwd.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_P)


def _dims(q, k, g, sinks, w, scale, reading=DELAYED):
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    D = g.shape[3]
    M = sinks.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    return _Dims(B, L, Hq, Hkv, d, D, w, M, int(reading), float(scale))


def fwd(q, k, v, g, Wf, sinks, w: int, scale: float | None = None, parts: bool = False,
        state: bool = False, reading: int = DELAYED) -> dict:
    """Recurrent fp64 forward.  Returns {"y"} and optionally the state (S, z) after
    the last token and the parts num_gla, den_gla, num_win, den_win, den.  `reading`
    picks the decay reading (DELAYED, MASKED or LAGGED)."""
    lib = _load()
    q, k, v, g, Wf, sinks = map(_f64, (q, k, v, g, Wf, sinks))
    p = _dims(q, k, g, sinks, w, scale, reading)
    B, L, Hq, d = q.shape
    Hkv, D = k.shape[2], g.shape[3]
    out = {"y": np.zeros_like(q)}
    if state:
        out["S"] = np.zeros((B, Hkv, D, d))
        out["z"] = np.zeros((B, Hkv, D))
    if parts:
        out["num_gla"] = np.zeros_like(q)
        out["den_gla"] = np.zeros((B, L, Hq))
        out["num_win"] = np.zeros_like(q)
        out["den_win"] = np.zeros((B, L, Hq))
        out["den"] = np.zeros((B, L, Hq))
    rc = lib.ora_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(Wf), _ptr(sinks),
                     _ptr(out["y"]), _ptr(out.get("S")), _ptr(out.get("z")),
                     _ptr(out.get("num_gla")), _ptr(out.get("den_gla")),
                     _ptr(out.get("num_win")), _ptr(out.get("den_win")), _ptr(out.get("den")))
    if rc != 0:
        raise ValueError("ora_fwd rejected its arguments")
    return out


def decode_step(pos: int, q, k, v, g, Wf, sinks, S, z, kcache, vcache, w: int,
                scale: float | None = None, gcache=None, reading: int = DELAYED) -> np.ndarray:
    """One fp64 decode step.  q [B,Hq,d]; k, v [B,Hkv,d]; g [B,Hkv,D].  S, z,
    kcache, vcache (float64, contiguous) are updated in place, and so is gcache
    [B,Hkv,w+1,D], the ring of gate logits the MASKED and LAGGED readings need.
    Returns y [B,Hq,d]."""
    lib = _load()
    q, k, v, g, Wf, sinks = map(_f64, (q, k, v, g, Wf, sinks))
    for a in (S, z, kcache, vcache) + ((gcache,) if gcache is not None else ()):
        assert a.dtype == np.float64 and a.flags.c_contiguous
    B, Hq, d = q.shape
    p = _Dims(B, 1, Hq, k.shape[1], d, g.shape[2], w, sinks.shape[1], int(reading),
              float(1.0 / np.sqrt(d) if scale is None else scale))
    y = np.zeros_like(q)
    rc = lib.ora_decode_step(ctypes.byref(p), pos, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(Wf),
                             _ptr(sinks), _ptr(y), _ptr(S), _ptr(z), _ptr(kcache), _ptr(vcache),
                             _ptr(gcache))
    if rc != 0:
        raise ValueError("ora_decode_step rejected its arguments")
    return y


def bwd(q, k, v, g, Wf, sinks, dy, w: int, scale: float | None = None,
        reading: int = DELAYED) -> dict:
    """Exact fp64 gradient of fwd()["y"] (same reading) against the upstream gradient dy."""
    lib = _load()
    q, k, v, g, Wf, sinks, dy = map(_f64, (q, k, v, g, Wf, sinks, dy))
    p = _dims(q, k, g, sinks, w, scale, reading)
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dg=np.zeros_like(g), dWf=np.zeros_like(Wf), dsinks=np.zeros_like(sinks))
    rc = lib.ora_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(Wf), _ptr(sinks),
                     _ptr(dy), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                     _ptr(out["dg"]), _ptr(out["dWf"]), _ptr(out["dsinks"]))
    if rc != 0:
        raise ValueError("ora_bwd rejected its arguments")
    return out


def qkvg_proj(x, W, Hq: int, Hkv: int, d: int, D: int) -> dict:
    """The projections in front of the mixer, in fp64: [q | k | v | g] = x W^T.

    Lizard summary sec. 2-A-1: the gate logits are a learned projection of the layer input
    (Gamma_i = sigmoid(W_gamma x_i)), next to the attention projections of q, k and v.
    x [B, L, dm]; W [N, dm] with N = Hq d + 2 Hkv d + Hkv D, its rows in the order q, k, v, g.
    Returns q [B, L, Hq, d], k, v [B, L, Hkv, d], g [B, L, Hkv, D]."""
    x = np.asarray(x, np.float64)
    W = np.asarray(W, np.float64)
    B, L, dm = x.shape
    y = x.reshape(B * L, dm) @ W.T
    n = np.cumsum([0, Hq * d, Hkv * d, Hkv * d, Hkv * D])
    shapes = [(Hq, d), (Hkv, d), (Hkv, d), (Hkv, D)]
    return {name: y[:, n[i]:n[i + 1]].reshape(B, L, *shapes[i])
            for i, name in enumerate(("q", "k", "v", "g"))}


def qkvg_proj_bwd(x, W, dq, dk, dv, dg) -> dict:
    """Gradients of qkvg_proj: with dY = [dq | dk | dv | dg] (flattened per token),
    dx = dY W and dW = dY^T x, in fp64."""
    x = np.asarray(x, np.float64)
    W = np.asarray(W, np.float64)
    B, L, dm = x.shape
    dY = np.concatenate([np.asarray(t, np.float64).reshape(B * L, -1) for t in (dq, dk, dv, dg)],
                        axis=1)
    return {"dx": (dY @ W).reshape(B, L, dm), "dW": dY.T @ x.reshape(B * L, dm)}
