"""Decode parity: lizard_decode_step (through the C ABI) against the float64 oracle.

Sec. 2-A-1 of the Lizard summary (gist.science 2507.09025): generation updates a
constant-size state token by token.  Each step must reproduce, token by token, the
output of a prefill over the whole sequence.
"""
import numpy as np
import pytest

from gated_linear_sliding_gb300 import inputs as I
from helpers import assert_parity, to_dev, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lz():
    from gated_linear_sliding_gb300 import lizard

    lizard.load()
    return lizard


def decode_all(lz, t, wl, pos0, npos, S, z, kc, vc):
    ys = []
    dims = lz.make_dims(wl.B, 1, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w, wl.M, t["q"].dtype)
    ws = lz.new_workspace(lz.lizard_decode_workspace(dims), "cuda")
    for pos in range(pos0, pos0 + npos):
        y = lz.lizard_decode_step(pos, t["q"][:, pos].contiguous(), t["k"][:, pos].contiguous(),
                                  t["v"][:, pos].contiguous(), t["g"][:, pos].contiguous(),
                                  t["Wf"], t["sinks"], S, z, kc, vc, wl.w, workspace=ws)
        ys.append(y)
    torch.cuda.synchronize()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK
    return to_np(torch.stack(ys, 1))


@pytest.mark.parametrize("dtype,d,D,G,w", [("f32", 64, 64, 2, 8), ("f32", 128, 128, 4, 5),
                                           ("bf16", 128, 128, 4, 64), ("bf16", 64, 128, 8, 3)])
def test_decode_from_scratch(lz, oracle_mod, dtype, d, D, G, w):
    wl = I.TINY_F32.replace(dtype=dtype, B=3, L=150, d=d, D=D, Hkv=2, Hq=2 * G, w=w)
    inp = I.make_inputs(wl)
    ref = oracle_mod.fwd(**inp, w=wl.w)["y"]
    t = to_dev(inp, dtype)
    tdt = t["q"].dtype
    S = torch.zeros(wl.B, wl.Hkv, D, d, dtype=torch.float32, device="cuda")
    z = torch.zeros(wl.B, wl.Hkv, D, dtype=torch.float32, device="cuda")
    kc = torch.zeros(wl.B, wl.Hkv, w + 1, d, dtype=tdt, device="cuda")
    vc = torch.zeros_like(kc)
    y = decode_all(lz, t, wl, 0, wl.L, S, z, kc, vc)
    assert_parity(y, ref, dtype, "decode y")
    fin = oracle_mod.fwd(**inp, w=wl.w, state=True)
    assert_parity(to_np(S), fin["S"], dtype, "S")
    assert_parity(to_np(z), fin["z"], dtype, "z")


@pytest.mark.parametrize("G,w,M", [(1, 1, 4), (2, 5, 0), (3, 17, 1), (4, 33, 64)])
def test_decode_streaming_kernel_shapes(lz, oracle_mod, G, w, M):
    """The streaming decode kernel's range (bf16, d = D = 128): one to four query heads per
    KV head, windows from 1 to 33 keys (the ring copies' box height is w + 1), no sinks up to
    64.  Decoded from position 0, so the window fills, wraps and the state starts admitting
    keys at token w."""
    wl = I.LLAMA3_8B_L8K.replace(B=3, L=110, Hkv=2, Hq=2 * G, w=w, M=M)
    inp = I.make_inputs(wl)
    ref = oracle_mod.fwd(**inp, w=w, state=True)
    t = to_dev(inp, "bf16")
    S = torch.zeros(wl.B, wl.Hkv, wl.D, wl.d, dtype=torch.float32, device="cuda")
    z = torch.zeros(wl.B, wl.Hkv, wl.D, dtype=torch.float32, device="cuda")
    kc = torch.zeros(wl.B, wl.Hkv, w + 1, wl.d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    y = decode_all(lz, t, wl, 0, wl.L, S, z, kc, vc)
    assert_parity(y, ref["y"], "bf16", "decode y")
    assert_parity(to_np(S), ref["S"], "bf16", "S")


def test_prefill_then_decode_matches_longer_prefill(lz, oracle_mod):
    """The forward hands off (S, z, ring caches); decode continues; the result equals the
    oracle prefill of the whole sequence, token by token."""
    wl = I.DECODE_B64.replace(B=4)
    L0, steps = 2048, 96
    inp = I.make_inputs(wl.replace(L=L0 + steps))
    ref = oracle_mod.fwd(**inp, w=wl.w)["y"]
    t = to_dev(inp, wl.dtype)
    tdt = t["q"].dtype
    S = torch.empty(wl.B, wl.Hkv, wl.D, wl.d, dtype=torch.float32, device="cuda")
    z = torch.empty(wl.B, wl.Hkv, wl.D, dtype=torch.float32, device="cuda")
    kc = torch.zeros(wl.B, wl.Hkv, wl.w + 1, wl.d, dtype=tdt, device="cuda")
    vc = torch.zeros_like(kc)
    pre = {n: (a[:, :L0].contiguous() if n in ("q", "k", "v", "g") else a) for n, a in t.items()}
    lz.lizard_attn_fwd(pre["q"], pre["k"], pre["v"], pre["g"], pre["Wf"], pre["sinks"], wl.w,
                       S_out=S, z_out=z, kcache_out=kc, vcache_out=vc)
    y = decode_all(lz, t, wl, L0, steps, S, z, kc, vc)
    assert_parity(y, ref[:, L0:], wl.dtype, "decode after prefill")


def test_decode_gla_sensitive(lz, oracle_mod):
    wl = I.gla_sensitive(I.DECODE_B64.replace(B=2))
    L0, steps = 1024, 64
    inp = I.make_inputs(wl.replace(L=L0 + steps))
    ref = oracle_mod.fwd(**inp, w=wl.w, scale=wl.scale)["y"]
    t = to_dev(inp, wl.dtype)
    S = torch.empty(wl.B, wl.Hkv, wl.D, wl.d, dtype=torch.float32, device="cuda")
    z = torch.empty(wl.B, wl.Hkv, wl.D, dtype=torch.float32, device="cuda")
    kc = torch.zeros(wl.B, wl.Hkv, wl.w + 1, wl.d, dtype=t["q"].dtype, device="cuda")
    vc = torch.zeros_like(kc)
    pre = {n: (a[:, :L0].contiguous() if n in ("q", "k", "v", "g") else a) for n, a in t.items()}
    lz.lizard_attn_fwd(pre["q"], pre["k"], pre["v"], pre["g"], pre["Wf"], pre["sinks"], wl.w,
                       S_out=S, z_out=z, kcache_out=kc, vcache_out=vc)
    y = decode_all(lz, t, wl, L0, steps, S, z, kc, vc)
    assert_parity(y, ref[:, L0:], wl.dtype, "decode gla-sensitive")


def test_decode_state_checkpoint_resume(lz):
    """The decode state (S, z, caches, pos) is the whole memory: copying it out and back
    in, then continuing, reproduces the uninterrupted run bit for bit."""
    wl = I.DECODE_B64.replace(B=2)
    inp = I.make_inputs(wl.replace(L=80))
    t = to_dev(inp, wl.dtype)
    tdt = t["q"].dtype

    def fresh():
        return (torch.zeros(wl.B, wl.Hkv, wl.D, wl.d, dtype=torch.float32, device="cuda"),
                torch.zeros(wl.B, wl.Hkv, wl.D, dtype=torch.float32, device="cuda"),
                torch.zeros(wl.B, wl.Hkv, wl.w + 1, wl.d, dtype=tdt, device="cuda"),
                torch.zeros(wl.B, wl.Hkv, wl.w + 1, wl.d, dtype=tdt, device="cuda"))

    st = fresh()
    y_all = decode_all(lz, t, wl, 0, 80, *st)
    st = fresh()
    decode_all(lz, t, wl, 0, 50, *st)
    saved = [x.cpu() for x in st]
    st2 = [x.to("cuda") for x in saved]
    y_tail = decode_all(lz, t, wl, 50, 30, *st2)
    np.testing.assert_array_equal(y_tail, y_all[:, 50:])


def test_decode_b64_full_size_sampled(lz, oracle_mod):
    """The decode workload at full size: B=64 sequences prefilled with 32768 tokens, then 1024
    single-token steps.  Inputs are drawn on the device (host generation of 15 G values would
    take minutes); two sampled sequences are copied back and checked against the oracle's
    prefill of all 33792 tokens, token by token."""
    wl = I.DECODE_B64
    T0, steps = wl.prefill, wl.steps
    B, Hq, Hkv, d, D, w = wl.B, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w
    pre = I.make_device_inputs(wl, "cuda", L=T0, B=B)
    S = torch.empty(B, Hkv, D, d, dtype=torch.float32, device="cuda")
    z = torch.empty(B, Hkv, D, dtype=torch.float32, device="cuda")
    kc = torch.zeros(B, Hkv, w + 1, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    lz.lizard_attn_fwd(pre["q"], pre["k"], pre["v"], pre["g"], pre["Wf"], pre["sinks"], w,
                       S_out=S, z_out=z, kcache_out=kc, vcache_out=vc)
    nxt = I.make_device_inputs(wl, "cuda", L=steps, B=B, seed_offset=1)
    qs, ks, vs, gs = (nxt[n].transpose(0, 1).contiguous() for n in ("q", "k", "v", "g"))
    dims = lz.make_dims(B, 1, Hq, Hkv, d, D, w, wl.M, torch.bfloat16)
    ws = lz.new_workspace(lz.lizard_decode_workspace(dims), "cuda")
    Y = torch.empty(steps, B, Hq, d, dtype=torch.bfloat16, device="cuda")
    for i in range(steps):
        lz.lizard_decode_step(T0 + i, qs[i], ks[i], vs[i], gs[i], pre["Wf"], pre["sinks"], S, z,
                              kc, vc, w, y=Y[i], workspace=ws)
    torch.cuda.synchronize()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK
    for b in (0, 37):
        seq = {n: torch.cat([pre[n][b:b + 1], nxt[n][b:b + 1]], dim=1).float().cpu().numpy()
               for n in ("q", "k", "v", "g")}
        seq["Wf"] = pre["Wf"].float().cpu().numpy()
        seq["sinks"] = pre["sinks"].cpu().numpy()
        ref = oracle_mod.fwd(**seq, w=w)["y"][0, T0:]          # [steps, Hq, d]
        got = Y[:, b].float().cpu().numpy().astype(np.float64)
        assert_parity(got, ref, "bf16", f"decode b{b}")


def _prefill_rows(lz, t, wl, lens, S, z, kc, vc):
    """State and ring caches of each sequence b after its first lens[b] tokens, one B=1
    forward per sequence writing into row b (rows of a sequence that has not started stay
    zero)."""
    S.zero_()
    z.zero_()
    kc.zero_()
    vc.zero_()
    for b, L0 in enumerate(lens):
        if L0 == 0:
            continue
        pre = {n: t[n][b:b + 1, :L0].contiguous() for n in ("q", "k", "v", "g")}
        lz.lizard_attn_fwd(pre["q"], pre["k"], pre["v"], pre["g"], t["Wf"], t["sinks"], wl.w,
                           S_out=S[b:b + 1], z_out=z[b:b + 1], kcache_out=kc[b:b + 1],
                           vcache_out=vc[b:b + 1])


def _token(t, lens, i):
    """The new token of every sequence at step i (sequence b is at position lens[b] + i)."""
    return {n: torch.stack([t[n][b, L0 + i] for b, L0 in enumerate(lens)]).contiguous()
            for n in ("q", "k", "v", "g")}


def _per_sequence_ref(oracle_mod, inp, wl, lens, steps):
    """Oracle outputs of each sequence at its own positions lens[b] .. lens[b] + steps - 1."""
    out = []
    for b, L0 in enumerate(lens):
        one = {n: (a[b:b + 1, :L0 + steps] if n in ("q", "k", "v", "g") else a)
               for n, a in inp.items()}
        out.append(oracle_mod.fwd(**one, w=wl.w)["y"][0, L0:L0 + steps])
    return np.stack(out)


def test_decode_positions_per_sequence(lz, oracle_mod):
    """Sequences of one batch at different positions (a fresh one, one inside the first
    window, one at the window edge, one long): each follows its own prefill, token by token."""
    wl = I.DECODE_B64.replace(B=4)
    lens, steps = [0, 5, 63, 700], 3
    inp = I.make_inputs(wl.replace(L=max(lens) + steps))
    ref = _per_sequence_ref(oracle_mod, inp, wl, lens, steps)
    t = to_dev(inp, wl.dtype)
    tdt = t["q"].dtype
    S = torch.empty(wl.B, wl.Hkv, wl.D, wl.d, dtype=torch.float32, device="cuda")
    z = torch.empty(wl.B, wl.Hkv, wl.D, dtype=torch.float32, device="cuda")
    kc = torch.empty(wl.B, wl.Hkv, wl.w + 1, wl.d, dtype=tdt, device="cuda")
    vc = torch.empty_like(kc)
    _prefill_rows(lz, t, wl, lens, S, z, kc, vc)
    dims = lz.make_dims(wl.B, 1, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w, wl.M, tdt)
    ws = lz.new_workspace(lz.lizard_decode_workspace(dims), "cuda")
    ys = []
    for i in range(steps):
        pos = torch.tensor([L0 + i for L0 in lens], dtype=torch.int64, device="cuda")
        tok = _token(t, lens, i)
        ys.append(lz.lizard_decode_step_positions(pos, tok["q"], tok["k"], tok["v"], tok["g"],
                                                  t["Wf"], t["sinks"], S, z, kc, vc, wl.w,
                                                  workspace=ws))
    torch.cuda.synchronize()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK
    assert_parity(to_np(torch.stack(ys, 1)), ref, wl.dtype, "per-sequence decode")


def test_decode_positions_negative_entry_is_reported(lz, oracle_mod):
    """A negative position is recorded in the workspace status and leaves that sequence's
    output, state and caches untouched; the other sequences are computed."""
    wl = I.DECODE_B64.replace(B=2)
    lens = [10, 70]
    inp = I.make_inputs(wl.replace(L=max(lens) + 1))
    ref = _per_sequence_ref(oracle_mod, inp, wl, lens, 1)
    t = to_dev(inp, wl.dtype)
    tdt = t["q"].dtype
    S = torch.empty(wl.B, wl.Hkv, wl.D, wl.d, dtype=torch.float32, device="cuda")
    z = torch.empty(wl.B, wl.Hkv, wl.D, dtype=torch.float32, device="cuda")
    kc = torch.empty(wl.B, wl.Hkv, wl.w + 1, wl.d, dtype=tdt, device="cuda")
    vc = torch.empty_like(kc)
    _prefill_rows(lz, t, wl, lens, S, z, kc, vc)
    before = [x[0].clone() for x in (S, z, kc, vc)]
    tok = _token(t, lens, 0)
    y = torch.full((wl.B, wl.Hq, wl.d), 7.0, dtype=tdt, device="cuda")
    dims = lz.make_dims(wl.B, 1, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w, wl.M, tdt)
    ws = lz.new_workspace(lz.lizard_decode_workspace(dims), "cuda")
    pos = torch.tensor([-1, lens[1]], dtype=torch.int64, device="cuda")
    lz.lizard_decode_step_positions(pos, tok["q"], tok["k"], tok["v"], tok["g"], t["Wf"],
                                    t["sinks"], S, z, kc, vc, wl.w, y=y, workspace=ws)
    torch.cuda.synchronize()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_ERR_INVALID_ARG
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK  # reading clears the word
    assert bool((y[0] == 7.0).all())
    for x, x0 in zip((S, z, kc, vc), before):
        assert torch.equal(x[0], x0)
    assert_parity(to_np(y[1:]), ref[1:, 0], wl.dtype, "the valid sequence")


def test_decode_positions_graph_replay(lz, oracle_mod):
    """The positions are read when the kernel runs: one captured step plus an on-device
    position increment, replayed, walks every sequence forward."""
    wl = I.DECODE_B64.replace(B=3)
    lens, steps = [3, 66, 129], 5
    inp = I.make_inputs(wl.replace(L=max(lens) + steps))
    ref = _per_sequence_ref(oracle_mod, inp, wl, lens, steps)
    t = to_dev(inp, wl.dtype)
    tdt = t["q"].dtype
    S = torch.empty(wl.B, wl.Hkv, wl.D, wl.d, dtype=torch.float32, device="cuda")
    z = torch.empty(wl.B, wl.Hkv, wl.D, dtype=torch.float32, device="cuda")
    kc = torch.empty(wl.B, wl.Hkv, wl.w + 1, wl.d, dtype=tdt, device="cuda")
    vc = torch.empty_like(kc)
    _prefill_rows(lz, t, wl, lens, S, z, kc, vc)
    dims = lz.make_dims(wl.B, 1, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w, wl.M, tdt)
    ws = lz.new_workspace(lz.lizard_decode_workspace(dims), "cuda")
    pos = torch.tensor(lens, dtype=torch.int64, device="cuda")
    tok = _token(t, lens, 0)
    y = torch.empty(wl.B, wl.Hq, wl.d, dtype=tdt, device="cuda")
    state0 = [x.clone() for x in (S, z, kc, vc)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # first call (attribute setup) outside the capture
        lz.lizard_decode_step_positions(pos, tok["q"], tok["k"], tok["v"], tok["g"], t["Wf"],
                                        t["sinks"], S, z, kc, vc, wl.w, y=y, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for x, x0 in zip((S, z, kc, vc), state0):
        x.copy_(x0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        lz.lizard_decode_step_positions(pos, tok["q"], tok["k"], tok["v"], tok["g"], t["Wf"],
                                        t["sinks"], S, z, kc, vc, wl.w, y=y, workspace=ws)
        pos.add_(1)
    ys = []
    for i in range(steps):
        for n, x in _token(t, lens, i).items():
            tok[n].copy_(x)
        graph.replay()
        ys.append(y.clone())
    torch.cuda.synchronize()
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK
    assert pos.tolist() == [L0 + steps for L0 in lens]
    assert_parity(to_np(torch.stack(ys, 1)), ref, wl.dtype, "graph-replayed decode")


def test_decode_closed_gate_runs(lz, oracle_mod):
    """Prefill and decode over gates with runs of strongly closed logits (N(-12, 1),
    N(-30, 1)): the state is decayed to nothing and rebuilt; decode follows the oracle."""
    wl = I.closed_gates(I.DECODE_B64.replace(B=4), per_1k=8.0)
    L0, steps = 1024, 128
    inp = I.make_inputs(wl.replace(L=L0 + steps))
    ref = oracle_mod.fwd(**inp, w=wl.w)["y"]
    t = to_dev(inp, wl.dtype)
    S = torch.empty(wl.B, wl.Hkv, wl.D, wl.d, dtype=torch.float32, device="cuda")
    z = torch.empty(wl.B, wl.Hkv, wl.D, dtype=torch.float32, device="cuda")
    kc = torch.zeros(wl.B, wl.Hkv, wl.w + 1, wl.d, dtype=t["q"].dtype, device="cuda")
    vc = torch.zeros_like(kc)
    pre = {n: (a[:, :L0].contiguous() if n in ("q", "k", "v", "g") else a) for n, a in t.items()}
    lz.lizard_attn_fwd(pre["q"], pre["k"], pre["v"], pre["g"], pre["Wf"], pre["sinks"], wl.w,
                       S_out=S, z_out=z, kcache_out=kc, vcache_out=vc)
    y = decode_all(lz, t, wl, L0, steps, S, z, kc, vc)
    assert_parity(y, ref[:, L0:], wl.dtype, "decode over closed gates")
