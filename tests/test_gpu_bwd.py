"""Backward parity: lizard_attn_bwd (through the C ABI) against the float64 oracle's exact
reverse pass (itself pinned by central finite differences).  The pages give no backward;
the reference is the adjoint of the forward definition (Lizard summary,
gist.science 2507.09025, sec. 2-A and 2-C)."""
import numpy as np
import pytest

from gated_linear_sliding_gb300 import inputs as I
from helpers import assert_grad, to_dev, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lz():
    from gated_linear_sliding_gb300 import lizard

    lizard.load()
    return lizard


def gpu_fwd_bwd(lz, inp, wl):
    t = to_dev(inp, wl.dtype)
    B, L, Hq, d = inp["q"].shape
    lse = torch.empty(B, L, Hq, dtype=torch.float32, device="cuda")
    y = lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w, lse=lse)
    g = lz.lizard_attn_bwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], y, lse, t["dy"],
                           wl.w)
    torch.cuda.synchronize()
    return {n: to_np(v) for n, v in g.items()}


def check(out, ref, dtype, names=("dq", "dk", "dv", "dg", "dWf", "dsinks")):
    for n in names:
        assert_grad(out[n], ref[n], dtype, n)


@pytest.mark.parametrize("L,w", [(100, 8), (300, 32), (40, 64), (257, 5)])
def test_bwd_f32_small(lz, oracle_mod, L, w):
    wl = I.TINY_F32.replace(L=L, w=w, B=2, Hq=4, Hkv=2)
    inp = I.make_inputs(wl, with_dy=True)
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=w)
    check(gpu_fwd_bwd(lz, inp, wl), ref, "f32")


def test_bwd_f32_tiny_workload(lz, oracle_mod):
    wl = I.TINY_F32
    inp = I.make_inputs(wl, with_dy=True)
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w)
    check(gpu_fwd_bwd(lz, inp, wl), ref, "f32")


def test_bwd_f32_gla_sensitive(lz, oracle_mod):
    wl = I.gla_sensitive(I.TINY_F32.replace(L=400, Hq=4, Hkv=2, w=16))
    inp = I.make_inputs(wl, with_dy=True)
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w,
                         scale=wl.scale)
    out = gpu_fwd_bwd(lz, inp, wl)
    check(out, ref, "f32")
    assert np.abs(ref["dg"]).max() > 1e-3  # the state carries gradient here


@pytest.mark.parametrize("d,D,G", [(128, 64, 2), (64, 128, 8)])
def test_bwd_f32_shapes(lz, oracle_mod, d, D, G):
    wl = I.TINY_F32.replace(L=200, d=d, D=D, Hkv=2, Hq=2 * G, w=16)
    inp = I.make_inputs(wl, with_dy=True)
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w)
    check(gpu_fwd_bwd(lz, inp, wl), ref, "f32")


def test_bwd_mistral_shape_reduced(lz, oracle_mod):
    wl = I.MISTRAL_7B_TRAIN
    inp = I.make_inputs(wl, L=512, B=2, with_dy=True)
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w)
    check(gpu_fwd_bwd(lz, inp, wl), ref, "bf16")


def test_bwd_mistral_gla_sensitive(lz, oracle_mod):
    wl = I.gla_sensitive(I.MISTRAL_7B_TRAIN)
    inp = I.make_inputs(wl, L=640, B=1, with_dy=True)
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w,
                         scale=wl.scale)
    check(gpu_fwd_bwd(lz, inp, wl), ref, "bf16")


def test_bwd_mistral_full_sampled_batch(lz, oracle_mod):
    """B=8, L=2048: the GPU runs the whole batch; the oracle checks two sequences (the
    batch entries are independent, except dWf and dsinks, which sum over the batch and are
    checked against the oracle over the same two sequences run alone)."""
    wl = I.MISTRAL_7B_TRAIN
    inp = I.make_inputs(wl, with_dy=True)
    out = gpu_fwd_bwd(lz, inp, wl)
    for b in (0, 5):
        sub = {n: (a[b:b + 1] if n in ("q", "k", "v", "g", "dy") else a) for n, a in inp.items()}
        ref = oracle_mod.bwd(**{n: a for n, a in sub.items() if n != "dy"}, dy=sub["dy"], w=wl.w)
        for n in ("dq", "dk", "dv", "dg"):
            assert_grad(out[n][b:b + 1], ref[n], "bf16", f"{n} b{b}")
    sub = {n: (a[[0, 5]] if n in ("q", "k", "v", "g", "dy") else a) for n, a in inp.items()}
    sub_out = gpu_fwd_bwd(lz, sub, wl)
    ref = oracle_mod.bwd(**{n: a for n, a in sub.items() if n != "dy"}, dy=sub["dy"], w=wl.w)
    assert_grad(sub_out["dWf"], ref["dWf"], "bf16", "dWf")
    assert_grad(sub_out["dsinks"], ref["dsinks"], "bf16", "dsinks")


def test_bwd_deterministic(lz):
    wl = I.MISTRAL_7B_TRAIN
    inp = I.make_inputs(wl, L=700, B=2, with_dy=True)
    a = gpu_fwd_bwd(lz, inp, wl)
    b = gpu_fwd_bwd(lz, inp, wl)
    for n in a:
        np.testing.assert_array_equal(a[n], b[n], err_msg=n)


def test_bwd_ragged_length_tensor_core_path(lz, oracle_mod):
    """L = 1000 is not a multiple of the 32-token steps: the last step of the tensor-core
    walks and window kernels is partial, and the sequence is cut into several segments."""
    wl = I.MISTRAL_7B_TRAIN
    inp = I.make_inputs(wl, L=1000, B=1, with_dy=True)
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w)
    check(gpu_fwd_bwd(lz, inp, wl), ref, "bf16")


def test_bwd_strong_decay_gates(lz, oracle_mod):
    """Gates drawn from the long-context stress mixture (30 % strongly decaying): the decay
    references and clamps of the tensor-core walks see cumulative log-gates far below zero."""
    wl = I.STRESS_L64K
    inp = I.make_inputs(wl, L=700, B=1, with_dy=True)
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w)
    check(gpu_fwd_bwd(lz, inp, wl), ref, "bf16")


def test_bwd_varlen_packed_batch(lz, oracle_mod):
    """Backward of a packed batch (sequences of 5, 0, 130 and 700 tokens, Mistral-shaped
    heads): each sequence's gradients equal its own backward; dWf and dsinks are the sums."""
    wl = I.MISTRAL_7B_TRAIN
    lens = [5, 0, 130, 700]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    inp = I.make_inputs(wl.replace(B=1, L=T), with_dy=True)
    t = to_dev(inp, wl.dtype)
    pk = {n: t[n][0] for n in ("q", "k", "v", "g", "dy")}
    lse = torch.empty(T, wl.Hq, dtype=torch.float32, device="cuda")
    y = lz.lizard_attn_fwd_varlen(pk["q"], pk["k"], pk["v"], pk["g"], t["Wf"], t["sinks"], wl.w,
                                  cu, lse=lse)
    gr = lz.lizard_attn_bwd_varlen(pk["q"], pk["k"], pk["v"], pk["g"], t["Wf"], t["sinks"], y,
                                   lse, pk["dy"], wl.w, cu)
    torch.cuda.synchronize()
    out = {n: to_np(v) for n, v in gr.items()}
    dW = np.zeros_like(out["dWf"], dtype=np.float64)
    dt = np.zeros_like(out["dsinks"], dtype=np.float64)
    for i in range(len(lens)):
        a, b = int(cu[i]), int(cu[i + 1])
        if b == a:
            continue
        one = {n: (arr[:, a:b] if n in ("q", "k", "v", "g", "dy") else arr)
               for n, arr in inp.items()}
        ref = oracle_mod.bwd(**{n: x for n, x in one.items() if n != "dy"}, dy=one["dy"], w=wl.w)
        for n in ("dq", "dk", "dv", "dg"):
            assert_grad(out[n][a:b][None], ref[n], "bf16", f"{n} of sequence {i}")
        dW += ref["dWf"]
        dt += ref["dsinks"]
    assert_grad(out["dWf"], dW, "bf16", "dWf (sum)")
    assert_grad(out["dsinks"], dt, "bf16", "dsinks (sum)")


@pytest.mark.parametrize("gla", [False, True])
def test_bwd_closed_gate_runs_mistral(lz, oracle_mod, gla):
    """Runs of strongly closed gates (logits N(-12, 1) and N(-30, 1)) inside the Mistral-shaped
    workload's gates: the segments they fall in take the exact SIMT walks, the others the
    tensor-core walks; all six gradients match the oracle."""
    wl = I.MISTRAL_7B_TRAIN
    if gla:
        wl = I.gla_sensitive(wl)
    wl = I.closed_gates(wl, per_1k=1.0)
    inp = I.make_inputs(wl, L=2048, B=2, with_dy=True)
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w,
                         scale=wl.scale)
    check(gpu_fwd_bwd(lz, inp, wl), ref, "bf16")


def test_bwd_closed_gate_runs_llama(lz, oracle_mod):
    wl = I.closed_gates(I.LLAMA3_8B_L8K, per_1k=0.5)
    inp = I.make_inputs(wl, L=4096, B=1, with_dy=True)
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w)
    check(gpu_fwd_bwd(lz, inp, wl), ref, "bf16")


def test_bwd_closed_gates_f32(lz, oracle_mod):
    """The fp32 path (SIMT walks only) under the same runs."""
    wl = I.closed_gates(I.TINY_F32.replace(L=400, B=2, Hq=4, Hkv=2, w=16), per_1k=5.0)
    inp = I.make_inputs(wl, with_dy=True)
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w)
    check(gpu_fwd_bwd(lz, inp, wl), ref, "f32")


def test_bwd_varlen_lanes_match_sequence_loop(lz):
    """The packed backward on four streams (full workspace) against one stream (a one-lane
    workspace), and against itself: per-sequence gradients are bit-identical (the same
    kernels on the same slices), dWf and dsinks equal up to the order of their sums, and a
    repeated call reproduces every output bit for bit."""
    wl = I.MISTRAL_7B_TRAIN
    lens = [700, 5, 0, 130, 1000, 64, 300]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    t = to_dev(I.make_inputs(wl.replace(B=1, L=T), with_dy=True), wl.dtype)
    pk = {n: t[n][0] for n in ("q", "k", "v", "g", "dy")}
    lse = torch.empty(T, wl.Hq, dtype=torch.float32, device="cuda")
    y = lz.lizard_attn_fwd_varlen(pk["q"], pk["k"], pk["v"], pk["g"], t["Wf"], t["sinks"], wl.w,
                                  cu, lse=lse)
    dims = lz.make_dims(len(lens), T, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w, wl.M, torch.bfloat16)
    full = lz.lizard_attn_bwd_varlen_workspace(dims, cu)
    assert full > 0 and full % 4 == 0
    ws_full = lz.new_workspace(full, torch.device("cuda"))
    ws_one = lz.new_workspace(full // 4, torch.device("cuda"))

    def run(ws):
        return lz.lizard_attn_bwd_varlen(pk["q"], pk["k"], pk["v"], pk["g"], t["Wf"], t["sinks"],
                                         y, lse, pk["dy"], wl.w, cu, workspace=ws)

    a, b, c = run(ws_full), run(ws_full), run(ws_one)
    torch.cuda.synchronize()
    assert lz.lizard_read_device_status(ws_full) == lz.LIZARD_OK
    assert lz.lizard_read_device_status(ws_one) == lz.LIZARD_OK
    for n in ("dq", "dk", "dv", "dg", "dWf", "dsinks"):
        assert torch.equal(a[n], b[n]), f"{n}: repeated call differs"
    for n in ("dq", "dk", "dv", "dg"):
        assert torch.equal(a[n], c[n]), f"{n}: lanes and one stream differ"
    for n in ("dWf", "dsinks"):
        x, r = to_np(a[n]), to_np(c[n])
        assert np.linalg.norm(x - r) <= 1e-5 * np.linalg.norm(r), n


@pytest.mark.parametrize("M", [0, 64])
def test_bwd_tensor_core_sink_counts(lz, oracle_mod, M):
    """The tensor-core backward with no sinks and with 64 per head (dsinks [Hq, M])."""
    wl = I.MISTRAL_7B_TRAIN.replace(M=M)
    inp = I.make_inputs(wl, L=300, B=1, with_dy=True)
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w)
    names = ("dq", "dk", "dv", "dg", "dWf") + (("dsinks",) if M > 0 else ())
    check(gpu_fwd_bwd(lz, inp, wl), ref, "bf16", names)


def test_bwd_tensor_core_batch_ragged(lz, oracle_mod):
    """Three batch entries with a ragged length on the tensor-core backward."""
    wl = I.MISTRAL_7B_TRAIN.replace(Hq=8, Hkv=2)
    inp = I.make_inputs(wl, L=1000, B=3, with_dy=True)
    ref = oracle_mod.bwd(**{n: a for n, a in inp.items() if n != "dy"}, dy=inp["dy"], w=wl.w)
    check(gpu_fwd_bwd(lz, inp, wl), ref, "bf16")
