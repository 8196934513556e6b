"""Parity of the two other decay readings, through the C ABI, against the float64 oracle.

The Lizard summary (gist.science 2507.09025, sec. 2-A-1) says the gate decays a state of the
tokens outside the window, not which gates such a key has seen.  Beside the delayed-key
reading the library runs the masked full-GLA reading (key j <= i - w weighed by
prod_{s=j+1..i} Gamma_s) and the lagged state (prod_{s=j+1..i-w} Gamma_s), selected by
lizard_dims.decay; the oracle's recurrence takes the same switch.  Forward (both paths),
packed batches, strongly closed gates, backward and decode through the gate ring.
"""
import numpy as np
import pytest

from gated_linear_sliding_gb300 import inputs as I
from helpers import assert_grad, assert_parity, rel_l2, to_dev, to_np
from oracle import LAGGED, MASKED

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

READINGS = [pytest.param(MASKED, id="masked"), pytest.param(LAGGED, id="lagged")]


@pytest.fixture(scope="module")
def lz():
    from gated_linear_sliding_gb300 import lizard

    lizard.load()
    return lizard


def gpu_fwd(lz, inp, wl, reading, lse=False, state=True):
    t = to_dev(inp, wl.dtype)
    B, L, Hq, d = inp["q"].shape
    kw = {}
    if state:
        kw = dict(S_out=torch.empty(B, wl.Hkv, wl.D, d, dtype=torch.float32, device="cuda"),
                  z_out=torch.empty(B, wl.Hkv, wl.D, dtype=torch.float32, device="cuda"))
    if lse:
        kw["lse"] = torch.empty(B, L, Hq, dtype=torch.float32, device="cuda")
    y = lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w,
                           decay=reading, **kw)
    torch.cuda.synchronize()
    out = {"y": to_np(y)}
    out.update({n: to_np(v) for n, v in kw.items()})
    return out


def check_fwd(lz, oracle_mod, wl, reading, L=None, B=None, scale=None):
    inp = I.make_inputs(wl, L=L, B=B)
    out = gpu_fwd(lz, inp, wl, reading)
    ref = oracle_mod.fwd(**inp, w=wl.w, scale=scale, state=True, reading=reading)
    sdt = "f32" if wl.dtype == "f32" else "bf16"
    assert_parity(out["y"], ref["y"], wl.dtype, "y")
    assert_parity(out["S_out"], ref["S"], sdt, "S")
    assert_parity(out["z_out"], ref["z"], sdt, "z")
    return inp, out, ref


@pytest.mark.parametrize("reading", READINGS)
@pytest.mark.parametrize("L,w", [(300, 8), (517, 64), (1100, 100), (40, 64)])
def test_fwd_f32(lz, oracle_mod, reading, L, w):
    check_fwd(lz, oracle_mod, I.TINY_F32.replace(L=L, w=w, Hq=4, Hkv=2, B=2), reading)


@pytest.mark.parametrize("reading", READINGS)
def test_fwd_f32_gla_sensitive_tells_readings_apart(lz, oracle_mod, reading):
    """Slow gates and peaked phi: the state carries real weight, and each reading's output
    differs from the delayed one's by more than ten times the fp32 tolerance (gates this
    close to 1 bring the readings together: the lagged one differs by ~3e-4), so the parity
    above is not vacuous."""
    wl = I.gla_sensitive(I.TINY_F32.replace(L=640, Hq=4, Hkv=2, w=16))
    inp, out, ref = check_fwd(lz, oracle_mod, wl, reading, scale=wl.scale)
    other = oracle_mod.fwd(**inp, w=wl.w, scale=wl.scale)["y"]
    assert rel_l2(ref["y"], other) > 10 * 1e-5
    assert rel_l2(out["y"], other) > 10 * 1e-5


@pytest.mark.parametrize("reading", READINGS)
def test_fwd_llama_shape(lz, oracle_mod, reading):
    """LLaMA-shaped heads at L = 1100 (several segments, a ragged last step), returning the
    final state: the lagged reading runs the tensor-core walk on the moved gates, the masked
    one (asked for the state) the SIMT walk."""
    wl = I.LLAMA3_8B_L8K
    dims = lz.make_dims(1, 1100, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w, wl.M, lz.LIZARD_BF16,
                        decay=reading)
    assert lz.lizard_attn_fwd_kernel(dims) == 1
    check_fwd(lz, oracle_mod, wl, reading, L=1100)


@pytest.mark.parametrize("reading", READINGS)
def test_fwd_llama_gla_sensitive(lz, oracle_mod, reading):
    wl = I.gla_sensitive(I.LLAMA3_8B_L8K)
    check_fwd(lz, oracle_mod, wl, reading, L=700, scale=wl.scale)


@pytest.mark.parametrize("reading", READINGS)
def test_fwd_closed_gates(lz, oracle_mod, reading):
    """Runs of strongly closed gates: the tensor-core walk hands such steps to the exact walk
    (at the moved positions for the lagged reading; with the keys' factors for the masked)."""
    check_fwd(lz, oracle_mod, I.closed_gates(I.LLAMA3_8B_L8K, per_1k=6.0), reading, L=1600)


@pytest.mark.parametrize("reading", READINGS)
def test_fwd_varlen_packed(lz, oracle_mod, reading):
    """A packed batch: the gates move (lagged, one launch over all sequences) or the keys'
    factors are taken (masked, sequence by sequence) within each sequence; each sequence
    equals its own forward."""
    wl = I.LLAMA3_8B_L8K
    lens = [1, 77, 0, 300, 1000, 130]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    inp = I.make_inputs(wl.replace(B=1, L=T))
    t = to_dev(inp, wl.dtype)
    nseq = len(lens)
    S = torch.empty(nseq, wl.Hkv, wl.D, wl.d, dtype=torch.float32, device="cuda")
    z = torch.empty(nseq, wl.Hkv, wl.D, dtype=torch.float32, device="cuda")
    y = lz.lizard_attn_fwd_varlen(t["q"][0], t["k"][0], t["v"][0], t["g"][0], t["Wf"],
                                  t["sinks"], wl.w, cu, S_out=S, z_out=z, decay=reading)
    torch.cuda.synchronize()
    y, S = to_np(y), to_np(S)
    for i in range(nseq):
        a, b = int(cu[i]), int(cu[i + 1])
        if a == b:
            assert not S[i].any()
            continue
        one = {n: (arr[:, a:b] if n in ("q", "k", "v", "g") else arr) for n, arr in inp.items()}
        ref = oracle_mod.fwd(**one, w=wl.w, state=True, reading=reading)
        assert_parity(y[a:b][None], ref["y"], "bf16", f"y of sequence {i}")
        assert_parity(S[i][None], ref["S"], "bf16", f"S of sequence {i}")


def test_noalloc_lagged_bit_identical(lz):
    """The no-allocation forward runs the same kernels on the same moved gates."""
    wl = I.LLAMA3_8B_L8K
    t = to_dev(I.make_inputs(wl, L=900), wl.dtype)
    args = (t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w)
    a = lz.lizard_attn_fwd(*args, decay=LAGGED)
    b = lz.lizard_attn_fwd_noalloc(*args, decay=LAGGED)
    torch.cuda.synchronize()
    assert lz.lizard_read_noalloc_status() == lz.LIZARD_OK
    assert torch.equal(a, b)


def gpu_fwd_bwd(lz, inp, wl, reading):
    t = to_dev(inp, wl.dtype)
    B, L, Hq, d = inp["q"].shape
    lse = torch.empty(B, L, Hq, dtype=torch.float32, device="cuda")
    y = lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w, lse=lse,
                           decay=reading)
    g = lz.lizard_attn_bwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], y, lse, t["dy"],
                           wl.w, decay=reading)
    torch.cuda.synchronize()
    return {n: to_np(v) for n, v in g.items()}


def check_bwd(lz, oracle_mod, wl, reading, L=None, B=None, scale=None):
    inp = I.make_inputs(wl, L=L, B=B, with_dy=True)
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w,
                         scale=scale, reading=reading)
    out = gpu_fwd_bwd(lz, inp, wl, reading)
    for n in ("dq", "dk", "dv", "dg", "dWf", "dsinks"):
        assert_grad(out[n], ref[n], wl.dtype, n)
    return out, ref


@pytest.mark.parametrize("reading", READINGS)
@pytest.mark.parametrize("L,w", [(300, 16), (257, 5), (100, 64)])
def test_bwd_f32(lz, oracle_mod, reading, L, w):
    check_bwd(lz, oracle_mod, I.TINY_F32.replace(L=L, w=w, B=2, Hq=4, Hkv=2), reading)


@pytest.mark.parametrize("reading", READINGS)
def test_bwd_f32_gla_sensitive(lz, oracle_mod, reading):
    wl = I.gla_sensitive(I.TINY_F32.replace(L=400, Hq=4, Hkv=2, w=16))
    out, ref = check_bwd(lz, oracle_mod, wl, reading, scale=wl.scale)
    assert np.abs(ref["dg"]).max() > 1e-3
    if reading == LAGGED:  # the last w gates decay nothing a query reads
        assert not out["dg"][:, wl.L - wl.w:].any()


@pytest.mark.parametrize("reading", READINGS)
def test_bwd_mistral_shape(lz, oracle_mod, reading):
    check_bwd(lz, oracle_mod, I.MISTRAL_7B_TRAIN, reading, L=520, B=2)


@pytest.mark.parametrize("reading", READINGS)
def test_bwd_mistral_gla_sensitive(lz, oracle_mod, reading):
    wl = I.gla_sensitive(I.MISTRAL_7B_TRAIN)
    check_bwd(lz, oracle_mod, wl, reading, L=640, B=1, scale=wl.scale)


def test_bwd_lagged_closed_gates(lz, oracle_mod):
    """Closed-gate runs under the lagged reading: the tensor-core walks leave the flagged
    segments (flagged on the moved gates) to the exact SIMT walks."""
    check_bwd(lz, oracle_mod, I.closed_gates(I.MISTRAL_7B_TRAIN, per_1k=6.0), LAGGED, L=900, B=1)


def test_bwd_masked_closed_gates(lz, oracle_mod):
    """Closed-gate runs under the masked reading: flagged segments go to the SIMT walks and the
    others stay on the tensor-core walks, both scaling the keys and writing their gate terms to
    the same key-term array."""
    check_bwd(lz, oracle_mod, I.closed_gates(I.MISTRAL_7B_TRAIN, per_1k=6.0), MASKED, L=900, B=2)


@pytest.mark.parametrize("reading", READINGS)
@pytest.mark.parametrize("dtype,d,D,G,w", [("f32", 64, 64, 2, 5), ("bf16", 128, 128, 4, 64)])
def test_decode_after_prefill(lz, oracle_mod, reading, dtype, d, D, G, w):
    """Prefill L0 tokens (state, k/v rings, gate ring), then decode the rest one token at a
    time through the gate ring: every step equals the oracle's prefill of the whole
    sequence under the same reading, and so does the final state."""
    L0, L = 150, 230
    base = I.LLAMA3_8B_L8K if dtype == "bf16" else I.TINY_F32
    wl = base.replace(B=3, L=L, d=d, D=D, Hkv=2, Hq=2 * G, w=w, dtype=dtype)
    inp = I.make_inputs(wl)
    ref = oracle_mod.fwd(**inp, w=w, state=True, reading=reading)
    t = to_dev(inp, dtype)
    tdt = t["q"].dtype
    pre = {n: (t[n][:, :L0].contiguous() if n in ("q", "k", "v", "g") else t[n]) for n in t}
    S = torch.empty(wl.B, wl.Hkv, D, d, dtype=torch.float32, device="cuda")
    z = torch.empty(wl.B, wl.Hkv, D, dtype=torch.float32, device="cuda")
    kc = torch.zeros(wl.B, wl.Hkv, w + 1, d, dtype=tdt, device="cuda")
    vc = torch.zeros_like(kc)
    gc = torch.zeros(wl.B, wl.Hkv, w + 1, D, dtype=tdt, device="cuda")
    y0 = lz.lizard_attn_fwd(pre["q"], pre["k"], pre["v"], pre["g"], t["Wf"], t["sinks"], w,
                            S_out=S, z_out=z, kcache_out=kc, vcache_out=vc, decay=reading)
    lz.lizard_gate_cache_fill(pre["g"], gc, w)
    dims = lz.make_dims(wl.B, 1, wl.Hq, wl.Hkv, d, D, w, wl.M, tdt, decay=reading)
    ws = lz.new_workspace(lz.lizard_decode_workspace(dims), "cuda")
    ys = []
    for pos in range(L0, L):
        ys.append(lz.lizard_decode_step(
            pos, t["q"][:, pos].contiguous(), t["k"][:, pos].contiguous(),
            t["v"][:, pos].contiguous(), t["g"][:, pos].contiguous(), t["Wf"], t["sinks"], S, z,
            kc, vc, w, workspace=ws, gcache=gc, decay=reading))
    torch.cuda.synchronize()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK
    assert_parity(to_np(y0), ref["y"][:, :L0], dtype, "prefill y")
    assert_parity(to_np(torch.stack(ys, 1)), ref["y"][:, L0:], dtype, "decode y")
    sdt = "f32" if dtype == "f32" else "bf16"
    assert_parity(to_np(S), ref["S"], sdt, "S")
    assert_parity(to_np(z), ref["z"], sdt, "z")


@pytest.mark.parametrize("reading", READINGS)
def test_decode_positions_from_scratch(lz, oracle_mod, reading):
    """Per-sequence positions (sequences started at different steps, one not yet started):
    each sequence's outputs follow the oracle from its own position 0."""
    wl = I.LLAMA3_8B_L8K.replace(B=3, L=90, Hq=8, Hkv=2)
    inp = I.make_inputs(wl)
    t = to_dev(inp, wl.dtype)
    tdt = t["q"].dtype
    B, w, d, D = wl.B, wl.w, wl.d, wl.D
    S = torch.zeros(B, wl.Hkv, D, d, dtype=torch.float32, device="cuda")
    z = torch.zeros(B, wl.Hkv, D, dtype=torch.float32, device="cuda")
    kc = torch.zeros(B, wl.Hkv, w + 1, d, dtype=tdt, device="cuda")
    vc = torch.zeros_like(kc)
    gc = torch.zeros(B, wl.Hkv, w + 1, D, dtype=tdt, device="cuda")
    start = [0, 7, 20]  # sequence b decodes its token p at loop step start[b] + p
    dims = lz.make_dims(B, 1, wl.Hq, wl.Hkv, d, D, w, wl.M, tdt, decay=reading)
    ws = lz.new_workspace(lz.lizard_decode_workspace(dims), "cuda")
    outs = {b: [] for b in range(B)}
    for stepi in range(wl.L + max(start)):
        p = [stepi - s for s in start]
        # a sequence not started or already finished takes position -1: left untouched, the
        # error noted in the status word
        pos = torch.tensor([pp if 0 <= pp < wl.L else -1 for pp in p], dtype=torch.int64,
                           device="cuda")
        idx = [min(max(pp, 0), wl.L - 1) for pp in p]
        tok = {n: torch.stack([t[n][b, idx[b]] for b in range(B)]).contiguous()
               for n in ("q", "k", "v", "g")}
        y = lz.lizard_decode_step_positions(pos, tok["q"], tok["k"], tok["v"], tok["g"], t["Wf"],
                                            t["sinks"], S, z, kc, vc, w, workspace=ws, gcache=gc,
                                            decay=reading)
        for b in range(B):
            if 0 <= p[b] < wl.L:
                outs[b].append(y[b])
    torch.cuda.synchronize()
    lz.lizard_read_device_status(ws)  # clears the noted negative positions
    ref = oracle_mod.fwd(**inp, w=w, reading=reading)["y"]
    for b in range(B):
        assert_parity(to_np(torch.stack(outs[b], 0))[None], ref[b:b + 1], "bf16", f"seq {b}")


# --- out-of-bounds write guard (the plain stand-in for the closed sanitizer) --------------

from test_gpu_canary import Guarded, _ws  # noqa: E402


@pytest.mark.parametrize("reading", READINGS)
@pytest.mark.parametrize("path,L", [("tc", 33), ("tc", 1100), ("simt", 517)])
def test_forward_writes_stay_in_bounds(lz, oracle_mod, reading, path, L):
    """Every output and the workspace (its reading scratch included, at exactly the queried
    size) sit in sentinel-filled slack that must stay untouched."""
    wl = I.LLAMA3_8B_L8K if path == "tc" else I.TINY_F32.replace(Hq=4, Hkv=2, B=2)
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
    dims = lz.dims_of(t["q"], t["k"], t["g"], t["sinks"], wl.w, decay=reading)
    ws = _ws(lz, g, lz.lizard_attn_fwd_workspace(dims))
    lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w, y=y, lse=lse,
                       S_out=S, z_out=z, kcache_out=kc, vcache_out=vc, workspace=ws,
                       decay=reading)
    g.check()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK
    ref = oracle_mod.fwd(**inp, w=wl.w, state=True, reading=reading)
    assert_parity(to_np(y), ref["y"], wl.dtype, "y")


@pytest.mark.parametrize("reading", READINGS)
@pytest.mark.parametrize("path,L", [("tc", 33), ("tc", 1000), ("simt", 517)])
def test_backward_writes_stay_in_bounds(lz, oracle_mod, reading, path, L):
    wl = I.MISTRAL_7B_TRAIN if path == "tc" else I.TINY_F32.replace(Hq=4, Hkv=2)
    inp = I.make_inputs(wl, L=L, B=1, with_dy=True)
    t = to_dev(inp, wl.dtype)
    B, Hq, Hkv, d, D, M = 1, wl.Hq, wl.Hkv, wl.d, wl.D, wl.M
    dt = t["q"].dtype
    lse = torch.empty(B, L, Hq, device="cuda")
    y = lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w, lse=lse,
                           decay=reading)
    g = Guarded()
    out = dict(dq=g.empty((B, L, Hq, d), dt), dk=g.empty((B, L, Hkv, d), dt),
               dv=g.empty((B, L, Hkv, d), dt), dg=g.empty((B, L, Hkv, D), dt),
               dWf=g.empty((Hkv, d, D // 2), torch.float32),
               dsinks=g.empty((Hq, M), torch.float32))
    dims = lz.dims_of(t["q"], t["k"], t["g"], t["sinks"], wl.w, decay=reading)
    ws = _ws(lz, g, lz.lizard_attn_bwd_workspace(dims))
    lz.lizard_attn_bwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], y, lse, t["dy"],
                       wl.w, workspace=ws, decay=reading, **out)
    g.check()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w,
                         reading=reading)
    for n in ("dq", "dk", "dv", "dg", "dWf"):
        assert_grad(to_np(out[n]), ref[n], wl.dtype, n)


@pytest.mark.parametrize("reading", READINGS)
def test_decode_writes_stay_in_bounds(lz, oracle_mod, reading):
    """Decode from position 0 through and past the window (the gate ring wraps): the ring,
    the state, y and the workspace at exactly the queried size stay in bounds."""
    wl = I.LLAMA3_8B_L8K.replace(B=2, L=80, Hq=8, Hkv=2)
    inp = I.make_inputs(wl)
    t = to_dev(inp, wl.dtype)
    B, Hq, Hkv, d, D, w = wl.B, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w
    dt = t["q"].dtype
    g = Guarded()
    S = g.empty((B, Hkv, D, d), torch.float32, like=torch.zeros(B, Hkv, D, d))
    z = g.empty((B, Hkv, D), torch.float32, like=torch.zeros(B, Hkv, D))
    kc = g.empty((B, Hkv, w + 1, d), dt, like=torch.zeros(B, Hkv, w + 1, d, dtype=dt))
    vc = g.empty((B, Hkv, w + 1, d), dt, like=torch.zeros(B, Hkv, w + 1, d, dtype=dt))
    gc = g.empty((B, Hkv, w + 1, D), dt, like=torch.zeros(B, Hkv, w + 1, D, dtype=dt))
    dims = lz.make_dims(B, 1, Hq, Hkv, d, D, w, wl.M, dt, decay=reading)
    ws = _ws(lz, g, lz.lizard_decode_workspace(dims))
    ys = []
    for pos in range(wl.L):
        y = g.empty((B, Hq, d), dt)
        lz.lizard_decode_step(pos, t["q"][:, pos].contiguous(), t["k"][:, pos].contiguous(),
                              t["v"][:, pos].contiguous(), t["g"][:, pos].contiguous(), t["Wf"],
                              t["sinks"], S, z, kc, vc, w, y=y, workspace=ws, gcache=gc,
                              decay=reading)
        ys.append(y)
    g.check()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK
    ref = oracle_mod.fwd(**inp, w=w, reading=reading)["y"]
    assert_parity(to_np(torch.stack(ys, 1)), ref, "bf16", "decode y")


@pytest.mark.parametrize("reading", READINGS)
def test_bwd_varlen_packed(lz, oracle_mod, reading):
    """The packed backward under each reading: every sequence's gradients equal the oracle's
    for that sequence alone; dWf sums over the sequences."""
    wl = I.MISTRAL_7B_TRAIN
    lens = [300, 0, 70, 513]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    inp = I.make_inputs(wl.replace(B=1, L=T), with_dy=True)
    t = to_dev(inp, wl.dtype)
    packed = {n: t[n][0] for n in ("q", "k", "v", "g", "dy")}
    lse = torch.empty(T, wl.Hq, dtype=torch.float32, device="cuda")
    y = lz.lizard_attn_fwd_varlen(packed["q"], packed["k"], packed["v"], packed["g"], t["Wf"],
                                  t["sinks"], wl.w, cu, lse=lse, decay=reading)
    gr = lz.lizard_attn_bwd_varlen(packed["q"], packed["k"], packed["v"], packed["g"], t["Wf"],
                                   t["sinks"], y, lse, packed["dy"], wl.w, cu, decay=reading)
    torch.cuda.synchronize()
    out = {n: to_np(v) for n, v in gr.items()}
    dWf = np.zeros_like(out["dWf"])
    for i in range(len(lens)):
        a, b = int(cu[i]), int(cu[i + 1])
        if a == b:
            continue
        one = {n: (arr[:, a:b] if n in ("q", "k", "v", "g", "dy") else arr)
               for n, arr in inp.items()}
        ref = oracle_mod.bwd(**{n: x for n, x in one.items() if n != "dy"}, dy=one["dy"],
                             w=wl.w, reading=reading)
        for n in ("dq", "dk", "dv", "dg"):
            assert_grad(out[n][a:b][None], ref[n], "bf16", f"{n} of sequence {i}")
        dWf += ref["dWf"]
    assert_grad(out["dWf"], dWf, "bf16", "dWf")


@pytest.mark.parametrize("reading", READINGS)
@pytest.mark.parametrize("d,D,G,w", [(64, 128, 2, 1), (128, 64, 1, 3)])
def test_fwd_bwd_small_windows_and_heads(lz, oracle_mod, reading, d, D, G, w):
    """w = 1 (the lagged gates move one token; the masked factor is the next token's gate)
    and the other compiled head sizes, forward and backward."""
    wl = I.TINY_F32.replace(L=150, d=d, D=D, Hkv=2, Hq=2 * G, w=w, B=2)
    check_fwd(lz, oracle_mod, wl, reading)
    check_bwd(lz, oracle_mod, wl, reading)


@pytest.mark.parametrize("reading", READINGS)
def test_fwd_llama_full_size(lz, oracle_mod, reading):
    """The bench's LLaMA-shaped forward at its full size (B = 1, L = 8192, all heads) in the
    bench's launch configuration, every output against the oracle."""
    wl = I.LLAMA3_8B_L8K
    check_fwd(lz, oracle_mod, wl, reading)


@pytest.mark.parametrize("reading", READINGS)
def test_stress_full_length_sampled_heads(lz, oracle_mod, reading):
    """L = 65536 with the stress gate mixture: the GPU runs all heads, the oracle one KV group
    (units are independent, so a head subset is an exact sub-problem)."""
    wl = I.STRESS_L64K
    inp = I.make_inputs(wl)
    out = gpu_fwd(lz, inp, wl, reading)
    G, kv = wl.G, 3
    sub = dict(q=inp["q"][:, :, kv * G:(kv + 1) * G], k=inp["k"][:, :, kv:kv + 1],
               v=inp["v"][:, :, kv:kv + 1], g=inp["g"][:, :, kv:kv + 1],
               Wf=inp["Wf"][kv:kv + 1], sinks=inp["sinks"][kv * G:(kv + 1) * G])
    ref = oracle_mod.fwd(**sub, w=wl.w, state=True, reading=reading)
    assert_parity(out["y"][:, :, kv * G:(kv + 1) * G], ref["y"], "bf16", f"y kv{kv}")
    assert_parity(out["S_out"][:, kv:kv + 1], ref["S"], "bf16", f"S kv{kv}")


@pytest.mark.parametrize("reading", READINGS)
def test_bwd_mistral_full_size_sampled(lz, oracle_mod, reading):
    """B = 8, L = 2048 (the bench's training step): the GPU runs the whole batch; the oracle
    checks one sequence's dq, dk, dv, dg (batch entries are independent)."""
    wl = I.MISTRAL_7B_TRAIN
    inp = I.make_inputs(wl, with_dy=True)
    out = gpu_fwd_bwd(lz, inp, wl, reading)
    b = 6
    sub = {n: (a[b:b + 1] if n in ("q", "k", "v", "g", "dy") else a) for n, a in inp.items()}
    ref = oracle_mod.bwd(**{n: a for n, a in sub.items() if n != "dy"}, dy=sub["dy"], w=wl.w,
                         reading=reading)
    for n in ("dq", "dk", "dv", "dg"):
        assert_grad(out[n][b:b + 1], ref[n], "bf16", f"{n} b{b}")


@pytest.mark.parametrize("L", [1100, 8192])
def test_fwd_masked_tensor_core_walk(lz, oracle_mod, L):
    """The masked reading on the tensor-core walk (a call that does not return the state):
    y and lse of the LLaMA-shaped layer against the oracle, up to the bench's full size."""
    wl = I.LLAMA3_8B_L8K
    inp = I.make_inputs(wl, L=L)
    out = gpu_fwd(lz, inp, wl, MASKED, lse=True, state=False)
    ref = oracle_mod.fwd(**inp, w=wl.w, parts=True, reading=MASKED)
    assert_parity(out["y"], ref["y"], "bf16", "y")
    assert rel_l2(out["lse"], np.log(ref["den"])) < 1e-3


def test_fwd_masked_tensor_core_walk_closed_gates(lz, oracle_mod):
    """Closed-gate runs on the masked tensor-core walk: the steps it hands to the exact walk
    take the keys' factors there too."""
    wl = I.closed_gates(I.LLAMA3_8B_L8K, per_1k=6.0)
    inp = I.make_inputs(wl, L=1600)
    out = gpu_fwd(lz, inp, wl, MASKED, state=False)
    ref = oracle_mod.fwd(**inp, w=wl.w, reading=MASKED)
    assert_parity(out["y"], ref["y"], "bf16", "y")


@pytest.mark.parametrize("reading", READINGS)
def test_decode_graph_replay_matches_eager(lz, reading):
    """The gate-ring step and the streaming decode step after it (launched as the ring
    step's programmatic dependent) captured in one CUDA graph: replays give the eager
    steps' outputs, states and rings bit for bit."""
    wl = I.DECODE_B64.replace(B=3)
    L0, steps, w = 100, 4, wl.w
    t = to_dev(I.make_inputs(wl.replace(L=L0 + steps)), wl.dtype)
    tdt = t["q"].dtype
    S = torch.empty(wl.B, wl.Hkv, wl.D, wl.d, dtype=torch.float32, device="cuda")
    z = torch.empty(wl.B, wl.Hkv, wl.D, dtype=torch.float32, device="cuda")
    kc = torch.zeros(wl.B, wl.Hkv, w + 1, wl.d, dtype=tdt, device="cuda")
    vc = torch.zeros_like(kc)
    gc = torch.zeros(wl.B, wl.Hkv, w + 1, wl.D, dtype=tdt, device="cuda")
    pre = {n: t[n][:, :L0].contiguous() for n in ("q", "k", "v", "g")}
    lz.lizard_attn_fwd(pre["q"], pre["k"], pre["v"], pre["g"], t["Wf"], t["sinks"], w,
                       S_out=S, z_out=z, kcache_out=kc, vcache_out=vc, decay=reading)
    lz.lizard_gate_cache_fill(pre["g"], gc, w)
    dims = lz.make_dims(wl.B, 1, wl.Hq, wl.Hkv, wl.d, wl.D, w, wl.M, tdt, decay=reading)
    ws = lz.new_workspace(lz.lizard_decode_workspace(dims), "cuda")
    torch.cuda.synchronize()
    states = (S, z, kc, vc, gc)
    start = [x.clone() for x in states]
    tok = {n: t[n][:, L0].contiguous() for n in ("q", "k", "v", "g")}
    y = torch.empty(wl.B, wl.Hq, wl.d, dtype=tdt, device="cuda")
    pos = torch.full((wl.B,), L0, dtype=torch.int64, device="cuda")

    def step():
        lz.lizard_decode_step_positions(pos, tok["q"], tok["k"], tok["v"], tok["g"], t["Wf"],
                                        t["sinks"], S, z, kc, vc, w, y=y, workspace=ws,
                                        gcache=gc, decay=reading)
        pos.add_(1)

    eager = []
    for i in range(steps):
        for n in tok:
            tok[n].copy_(t[n][:, L0 + i])
        step()
        eager.append(y.clone())
    torch.cuda.synchronize()
    end = [x.clone() for x in states]
    for x, x0 in zip(states, start):
        x.copy_(x0)
    pos.fill_(L0)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    replayed = []
    for i in range(steps):
        for n in tok:
            tok[n].copy_(t[n][:, L0 + i])
        graph.replay()
        replayed.append(y.clone())
    torch.cuda.synchronize()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK
    assert pos.tolist() == [L0 + steps] * wl.B
    for i, (a_, b_) in enumerate(zip(eager, replayed)):
        assert torch.equal(a_, b_), f"step {i}"
    for name, x, x1 in zip(("S", "z", "kcache", "vcache", "gcache"), states, end):
        assert torch.equal(x, x1), name
