"""Out-of-bounds write guard for every output of the C ABI.

The sanitizer is closed on this machine, so bounds are checked the plain way: every output
buffer (and the tail of every workspace) sits inside a larger allocation whose slack before
and after is filled with a sentinel byte; after the call the slack must be byte-identical.
Lengths are ragged (1, 33, 517, 1000, 1100 tokens) so that partial tiles, partial 32-token
steps and partial TMA stores are written, on the tensor-core path (bf16, d = D = 128, four
query heads per KV head, window 64) and on the SIMT path (fp32).
"""
import ctypes

import numpy as np
import pytest

from gated_linear_sliding_gb300 import inputs as I
from helpers import assert_grad, assert_parity, to_dev, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SLACK = 4096  # bytes before and after each buffer (keeps the 16-byte alignment)
SENTINEL = 0xA5


@pytest.fixture(scope="module")
def lz():
    from gated_linear_sliding_gb300 import lizard

    lizard.load()
    return lizard


class Guarded:
    """Buffers with sentinel-filled slack on both sides."""

    def __init__(self):
        self.bufs = []

    def empty(self, shape, dtype, like=None):
        n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        buf = torch.full((SLACK + n + SLACK,), SENTINEL, dtype=torch.uint8, device="cuda")
        view = buf[SLACK:SLACK + n].view(dtype).view(*shape)
        if like is not None:
            view.copy_(like)
        self.bufs.append((buf, n, f"{tuple(shape)} {dtype}"))
        return view

    def check(self):
        torch.cuda.synchronize()
        for buf, n, what in self.bufs:
            front = buf[:SLACK]
            back = buf[SLACK + n:]
            assert bool((front == SENTINEL).all()), f"write before {what}"
            assert bool((back == SENTINEL).all()), f"write after {what}"


def _ws(lz, g, nbytes):
    """A workspace of exactly the queried size inside guarded slack, status word zeroed."""
    ws = g.empty((max(int(nbytes), 256),), torch.uint8)
    ws[:256].zero_()
    return ws


WORKLOADS = {
    "tc": I.LLAMA3_8B_L8K,
    "tc_closed": I.closed_gates(I.LLAMA3_8B_L8K, per_1k=8.0),
    "simt": I.TINY_F32.replace(Hq=4, Hkv=2, B=2),
}


@pytest.mark.parametrize("path", ["tc", "tc_closed", "simt"])
@pytest.mark.parametrize("L", [1, 33, 517, 1000, 1100])
def test_forward_writes_stay_in_bounds(lz, oracle_mod, path, L):
    wl = WORKLOADS[path]
    inp = I.make_inputs(wl, L=L)
    t = to_dev(inp, wl.dtype)
    B, Hq, Hkv, d, D = inp["q"].shape[0], wl.Hq, wl.Hkv, wl.d, wl.D
    dt = t["q"].dtype
    g = Guarded()
    y = g.empty((B, L, Hq, d), dt)
    lse = g.empty((B, L, Hq), torch.float32)
    S = g.empty((B, Hkv, D, d), torch.float32)
    z = g.empty((B, Hkv, D), torch.float32)
    kc = g.empty((B, Hkv, wl.w + 1, d), dt, like=torch.zeros(B, Hkv, wl.w + 1, d, dtype=dt))
    vc = g.empty((B, Hkv, wl.w + 1, d), dt, like=torch.zeros(B, Hkv, wl.w + 1, d, dtype=dt))
    dims = lz.dims_of(t["q"], t["k"], t["g"], t["sinks"], wl.w)
    ws = _ws(lz, g, lz.lizard_attn_fwd_workspace(dims))
    lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w, y=y, lse=lse,
                       S_out=S, z_out=z, kcache_out=kc, vcache_out=vc, workspace=ws)
    g.check()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK
    ref = oracle_mod.fwd(**inp, w=wl.w, state=True)
    assert_parity(to_np(y), ref["y"], wl.dtype, "y")
    assert_parity(to_np(S), ref["S"], wl.dtype, "S")


@pytest.mark.parametrize("path", ["tc", "tc_closed", "simt"])
@pytest.mark.parametrize("L", [33, 517, 1000])
def test_backward_writes_stay_in_bounds(lz, oracle_mod, path, L):
    wl = WORKLOADS[path] if path != "tc" else I.MISTRAL_7B_TRAIN
    inp = I.make_inputs(wl, L=L, B=1, with_dy=True)
    t = to_dev(inp, wl.dtype)
    B, Hq, Hkv, d, D, M = 1, wl.Hq, wl.Hkv, wl.d, wl.D, wl.M
    dt = t["q"].dtype
    lse = torch.empty(B, L, Hq, device="cuda")
    y = lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w, lse=lse)
    g = Guarded()
    out = dict(dq=g.empty((B, L, Hq, d), dt), dk=g.empty((B, L, Hkv, d), dt),
               dv=g.empty((B, L, Hkv, d), dt), dg=g.empty((B, L, Hkv, D), dt),
               dWf=g.empty((Hkv, d, D // 2), torch.float32),
               dsinks=g.empty((Hq, M), torch.float32))
    dims = lz.dims_of(t["q"], t["k"], t["g"], t["sinks"], wl.w)
    ws = _ws(lz, g, lz.lizard_attn_bwd_workspace(dims))
    lz.lizard_attn_bwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], y, lse, t["dy"],
                       wl.w, workspace=ws, **out)
    g.check()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w)
    for n in ("dq", "dk", "dv", "dg"):
        if not ref[n].any():  # L < w: no key leaves the window, the gates get no gradient
            scale = max(np.abs(ref["dq"]).max(), np.abs(ref["dv"]).max())
            assert np.abs(to_np(out[n])).max() <= 1e-6 * scale, n  # rounding noise at most
        else:
            assert_grad(to_np(out[n]), ref[n], wl.dtype, n)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_writes_stay_in_bounds(lz, oracle_mod, dtype):
    wl = I.DECODE_B64.replace(B=3, dtype=dtype)
    steps = 70
    inp = I.make_inputs(wl.replace(L=steps))
    t = to_dev(inp, dtype)
    dt = t["q"].dtype
    g = Guarded()
    S = g.empty((wl.B, wl.Hkv, wl.D, wl.d), torch.float32,
                like=torch.zeros(wl.B, wl.Hkv, wl.D, wl.d))
    z = g.empty((wl.B, wl.Hkv, wl.D), torch.float32, like=torch.zeros(wl.B, wl.Hkv, wl.D))
    kc = g.empty((wl.B, wl.Hkv, wl.w + 1, wl.d), dt,
                 like=torch.zeros(wl.B, wl.Hkv, wl.w + 1, wl.d, dtype=dt))
    vc = g.empty((wl.B, wl.Hkv, wl.w + 1, wl.d), dt,
                 like=torch.zeros(wl.B, wl.Hkv, wl.w + 1, wl.d, dtype=dt))
    dims = lz.make_dims(wl.B, 1, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w, wl.M, dt)
    ws = _ws(lz, g, lz.lizard_decode_workspace(dims))
    ys = []
    for pos in range(steps):
        y = g.empty((wl.B, wl.Hq, wl.d), dt)
        lz.lizard_decode_step(pos, t["q"][:, pos].contiguous(), t["k"][:, pos].contiguous(),
                              t["v"][:, pos].contiguous(), t["g"][:, pos].contiguous(), t["Wf"],
                              t["sinks"], S, z, kc, vc, wl.w, y=y, workspace=ws)
        ys.append(y)
    g.check()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK
    ref = oracle_mod.fwd(**inp, w=wl.w)["y"]
    assert_parity(to_np(torch.stack(ys, 1)), ref, dtype, "decode y")


@pytest.mark.parametrize("path", ["tc", "tc_one_launch", "simt"])
def test_varlen_writes_stay_in_bounds(lz, path):
    wl = WORKLOADS["tc" if path == "tc_one_launch" else path]
    lens = [1, 33, 0, 517, 1100]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    inp = I.make_inputs(wl.replace(B=1, L=T))
    t = to_dev(inp, wl.dtype)
    pk = {n: t[n][0] for n in ("q", "k", "v", "g")}
    dt = t["q"].dtype
    n = len(lens)
    g = Guarded()
    y = g.empty((T, wl.Hq, wl.d), dt)
    lse = g.empty((T, wl.Hq), torch.float32)
    S = g.empty((n, wl.Hkv, wl.D, wl.d), torch.float32)
    z = g.empty((n, wl.Hkv, wl.D), torch.float32)
    kc = g.empty((n, wl.Hkv, wl.w + 1, wl.d), dt)
    vc = g.empty((n, wl.Hkv, wl.w + 1, wl.d), dt)
    one = lz.make_dims(1, T, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w, wl.M, dt)
    if path == "tc_one_launch":  # every sequence in one launch (direct stores of ragged ends)
        dims = lz.make_dims(n, T, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w, wl.M, dt)
        ws = _ws(lz, g, lz.lizard_attn_fwd_varlen_workspace(dims, cu))
    else:  # one sequence after another
        ws = _ws(lz, g, lz.lizard_attn_fwd_workspace(one))
    lz.lizard_attn_fwd_varlen(pk["q"], pk["k"], pk["v"], pk["g"], t["Wf"], t["sinks"], wl.w, cu,
                              y=y, lse=lse, S_out=S, z_out=z, kcache_out=kc, vcache_out=vc,
                              workspace=ws)
    g.check()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK


def test_varlen_backward_writes_stay_in_bounds(lz):
    """The packed backward on four streams: dq, dk, dv, dg of every ragged sequence, dWf, dsinks
    and the workspace tail keep their slack untouched."""
    wl = I.MISTRAL_7B_TRAIN
    lens = [1, 33, 0, 517, 1100, 70]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, n = int(cu[-1]), len(lens)
    inp = I.make_inputs(wl.replace(B=1, L=T), with_dy=True)
    t = to_dev(inp, wl.dtype)
    pk = {k: t[k][0] for k in ("q", "k", "v", "g", "dy")}
    dt = pk["q"].dtype
    lse = torch.empty(T, wl.Hq, device="cuda")
    y = lz.lizard_attn_fwd_varlen(pk["q"], pk["k"], pk["v"], pk["g"], t["Wf"], t["sinks"], wl.w,
                                  cu, lse=lse)
    g = Guarded()
    out = dict(dq=g.empty((T, wl.Hq, wl.d), dt), dk=g.empty((T, wl.Hkv, wl.d), dt),
               dv=g.empty((T, wl.Hkv, wl.d), dt), dg=g.empty((T, wl.Hkv, wl.D), dt),
               dWf=g.empty((wl.Hkv, wl.d, wl.D // 2), torch.float32),
               dsinks=g.empty((wl.Hq, wl.M), torch.float32))
    dims = lz.make_dims(n, T, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w, wl.M, dt)
    ws = _ws(lz, g, lz.lizard_attn_bwd_varlen_workspace(dims, cu))
    lib = lz.load()
    st = lib.lizard_attn_bwd_varlen(
        ctypes.byref(dims), np.ascontiguousarray(cu).ctypes.data, *(lz._p(x) for x in (
            pk["q"], pk["k"], pk["v"], pk["g"], t["Wf"], t["sinks"], y, lse, pk["dy"],
            out["dq"], out["dk"], out["dv"], out["dg"], out["dWf"], out["dsinks"], ws)),
        ws.numel(), None)
    assert st == lz.LIZARD_OK
    g.check()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK
    for k in ("dq", "dk", "dv", "dg", "dWf", "dsinks"):
        assert bool(torch.isfinite(out[k].float()).all()), k
