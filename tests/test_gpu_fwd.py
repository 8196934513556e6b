"""Forward parity: lizard_attn_fwd (through the C ABI) against the float64 oracle.

The oracle is the token recurrence of the Lizard summary (gist.science 2507.09025,
sec. 2-A-1 and 2-A-2, shared normaliser); inputs come from the seeded generators.
"""
import numpy as np
import pytest

from gated_linear_sliding_gb300 import inputs as I
from helpers import assert_parity, rel_l2, to_dev, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lz():
    from gated_linear_sliding_gb300 import lizard

    lizard.load()
    return lizard


def gpu_fwd(lz, inp, wl, scale=0.0, state=False, cache=False, lse=False):
    t = to_dev(inp, wl.dtype)
    B, L, Hq, d = inp["q"].shape
    Hkv, D = wl.Hkv, wl.D
    kw = {}
    if lse:
        kw["lse"] = torch.empty(B, L, Hq, dtype=torch.float32, device="cuda")
    if state:
        kw["S_out"] = torch.empty(B, Hkv, D, d, dtype=torch.float32, device="cuda")
        kw["z_out"] = torch.empty(B, Hkv, D, dtype=torch.float32, device="cuda")
    if cache:
        kw["kcache_out"] = torch.zeros(B, Hkv, wl.w + 1, d, dtype=t["q"].dtype, device="cuda")
        kw["vcache_out"] = torch.zeros(B, Hkv, wl.w + 1, d, dtype=t["q"].dtype, device="cuda")
    y = lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w,
                           scale=scale, **kw)
    torch.cuda.synchronize()
    out = {"y": to_np(y)}
    for n, v in kw.items():
        out[n] = to_np(v)
    return out


def oracle_fwd(oracle_mod, inp, wl, **kw):
    return oracle_mod.fwd(**inp, w=wl.w, scale=wl.scale, **kw)


def test_tiny_f32(lz, oracle_mod):
    wl = I.TINY_F32
    inp = I.make_inputs(wl)
    out = gpu_fwd(lz, inp, wl, lse=True, state=True)
    ref = oracle_fwd(oracle_mod, inp, wl, parts=True, state=True)
    assert_parity(out["y"], ref["y"], "f32", "y")
    assert rel_l2(out["lse"], np.log(ref["den"])) < 1e-5
    assert_parity(out["S_out"], ref["S"], "f32", "S")
    assert_parity(out["z_out"], ref["z"], "f32", "z")


def test_tiny_f32_gla_sensitive(lz, oracle_mod):
    wl = I.gla_sensitive(I.TINY_F32.replace(L=640, Hq=4, Hkv=2))
    inp = I.make_inputs(wl)
    out = gpu_fwd(lz, inp, wl)
    assert_parity(out["y"], oracle_fwd(oracle_mod, inp, wl)["y"], "f32", "y")


@pytest.mark.parametrize("L,w", [(1, 32), (31, 32), (33, 32), (65, 1), (200, 5), (130, 300),
                                 (517, 64), (1100, 100)])
def test_f32_ragged_lengths_and_windows(lz, oracle_mod, L, w):
    wl = I.TINY_F32.replace(L=L, w=w, Hq=4, Hkv=2, B=2)
    inp = I.make_inputs(wl)
    out = gpu_fwd(lz, inp, wl, state=True)
    ref = oracle_fwd(oracle_mod, inp, wl, state=True)
    assert_parity(out["y"], ref["y"], "f32", "y")
    assert_parity(out["S_out"], ref["S"], "f32", "S")


@pytest.mark.parametrize("d,D,G", [(128, 64, 1), (64, 128, 8), (128, 128, 4), (64, 64, 3)])
def test_f32_shapes(lz, oracle_mod, d, D, G):
    wl = I.TINY_F32.replace(L=300, d=d, D=D, Hkv=2, Hq=2 * G, w=16)
    inp = I.make_inputs(wl)
    out = gpu_fwd(lz, inp, wl)
    assert_parity(out["y"], oracle_fwd(oracle_mod, inp, wl)["y"], "f32", "y")


def test_f32_no_sinks(lz, oracle_mod):
    wl = I.TINY_F32.replace(M=0, L=300)
    inp = I.make_inputs(wl)
    out = gpu_fwd(lz, inp, wl)
    assert_parity(out["y"], oracle_fwd(oracle_mod, inp, wl)["y"], "f32", "y")


def test_llama3_8b_shape_full(lz, oracle_mod):
    wl = I.LLAMA3_8B_L8K
    inp = I.make_inputs(wl)
    out = gpu_fwd(lz, inp, wl, lse=True, state=True, cache=True)
    ref = oracle_fwd(oracle_mod, inp, wl, parts=True, state=True)
    assert_parity(out["y"], ref["y"], "bf16", "y")
    assert rel_l2(out["lse"], np.log(ref["den"])) < 1e-3
    assert_parity(out["S_out"], ref["S"], "bf16", "S")
    assert_parity(out["z_out"], ref["z"], "bf16", "z")
    # ring caches hold the last w tokens at slot t mod (w+1)
    L, w = wl.L, wl.w
    for t in range(L - w, L):
        np.testing.assert_array_equal(out["kcache_out"][:, :, t % (w + 1)], inp["k"][:, t])
        np.testing.assert_array_equal(out["vcache_out"][:, :, t % (w + 1)], inp["v"][:, t])


@pytest.mark.parametrize("L", [64, 1000, 3000])
def test_llama3_8b_shape_ragged(lz, oracle_mod, L):
    wl = I.LLAMA3_8B_L8K
    inp = I.make_inputs(wl, L=L)
    out = gpu_fwd(lz, inp, wl)
    assert_parity(out["y"], oracle_fwd(oracle_mod, inp, wl)["y"], "bf16", "y")


def test_llama3_8b_gla_sensitive(lz, oracle_mod):
    wl = I.gla_sensitive(I.LLAMA3_8B_L8K)
    inp = I.make_inputs(wl, L=4096)
    out = gpu_fwd(lz, inp, wl, state=True)
    ref = oracle_fwd(oracle_mod, inp, wl, state=True, parts=True)
    assert np.median(ref["den_gla"][:, 2048:] / ref["den"][:, 2048:]) > 0.1
    assert_parity(out["y"], ref["y"], "bf16", "y")
    assert_parity(out["S_out"], ref["S"], "bf16", "S")


def test_stress_gates_underflow(lz, oracle_mod):
    """Gate mixture whose chunk products underflow: the log-space path stays finite."""
    wl = I.STRESS_L64K
    inp = I.make_inputs(wl, L=8192)
    out = gpu_fwd(lz, inp, wl)
    assert_parity(out["y"], oracle_fwd(oracle_mod, inp, wl)["y"], "bf16", "y")


def test_stress_full_length_sampled_heads(lz, oracle_mod):
    """L = 65536: the GPU runs all heads; the oracle checks two KV groups (the units are
    independent, so a head subset is an exact sub-problem)."""
    wl = I.STRESS_L64K
    inp = I.make_inputs(wl)
    out = gpu_fwd(lz, inp, wl)
    G = wl.G
    for kv in (0, 5):
        sub = dict(q=inp["q"][:, :, kv * G:(kv + 1) * G], k=inp["k"][:, :, kv:kv + 1],
                   v=inp["v"][:, :, kv:kv + 1], g=inp["g"][:, :, kv:kv + 1],
                   Wf=inp["Wf"][kv:kv + 1], sinks=inp["sinks"][kv * G:(kv + 1) * G])
        ref = oracle_mod.fwd(**sub, w=wl.w, scale=wl.scale)["y"]
        assert_parity(out["y"][:, :, kv * G:(kv + 1) * G], ref, "bf16", f"y kv{kv}")


def test_mistral_7b_train_shape(lz, oracle_mod):
    wl = I.MISTRAL_7B_TRAIN
    inp = I.make_inputs(wl)
    out = gpu_fwd(lz, inp, wl)
    assert_parity(out["y"], oracle_fwd(oracle_mod, inp, wl)["y"], "bf16", "y")


def test_workspace_reuse_and_determinism(lz):
    wl = I.LLAMA3_8B_L8K
    t = to_dev(I.make_inputs(wl, L=2048), wl.dtype)
    dims = lz.dims_of(t["q"], t["k"], t["g"], t["sinks"], wl.w)
    ws = lz.new_workspace(lz.lizard_attn_fwd_workspace(dims), "cuda")
    y1 = lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w,
                            workspace=ws)
    y2 = lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w,
                            workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK


def _varlen_run(lz, wl, t, cu, workspace=None):
    T, nseq = int(cu[-1]), len(cu) - 1
    packed = {n: t[n][0] for n in ("q", "k", "v", "g")}
    S = torch.empty(nseq, wl.Hkv, wl.D, wl.d, dtype=torch.float32, device="cuda")
    z = torch.empty(nseq, wl.Hkv, wl.D, dtype=torch.float32, device="cuda")
    lse = torch.empty(T, wl.Hq, dtype=torch.float32, device="cuda")
    y = lz.lizard_attn_fwd_varlen(packed["q"], packed["k"], packed["v"], packed["g"], t["Wf"],
                                  t["sinks"], wl.w, cu, lse=lse, S_out=S, z_out=z,
                                  workspace=workspace)
    return y, S, z, lse


def _varlen_case(lz, oracle_mod, wl, lens):
    """A packed batch of sequences against the oracle run on each sequence alone."""
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    inp = I.make_inputs(wl.replace(B=1, L=T))
    t = to_dev(inp, wl.dtype)
    nseq = len(lens)
    y, S, z, lse = _varlen_run(lz, wl, t, cu)
    torch.cuda.synchronize()
    y, S, z = to_np(y), to_np(S), to_np(z)
    for i in range(nseq):
        a, b = int(cu[i]), int(cu[i + 1])
        if b == a:
            assert not S[i].any() and not z[i].any()
            continue
        one = {n: (arr[:, a:b] if n in ("q", "k", "v", "g") else arr) for n, arr in inp.items()}
        ref = oracle_mod.fwd(**one, w=wl.w, state=True)
        assert_parity(y[a:b][None], ref["y"], wl.dtype, f"y of sequence {i}")
        assert_parity(S[i][None], ref["S"], "f32" if wl.dtype == "f32" else wl.dtype, f"S of {i}")


def test_varlen_packed_batch_bf16(lz, oracle_mod):
    """Sequences of 1, 77, 0, 300 and 1000 tokens in one packed batch (LLaMA-shaped heads):
    each equals its own forward; nothing crosses a boundary; the empty one has a zero state."""
    _varlen_case(lz, oracle_mod, I.LLAMA3_8B_L8K, [1, 77, 0, 300, 1000])


def test_varlen_packed_batch_f32(lz, oracle_mod):
    _varlen_case(lz, oracle_mod, I.TINY_F32.replace(Hq=4, Hkv=2), [40, 3, 129, 64])


def test_varlen_one_launch_several_segments(lz, oracle_mod):
    """One launch over sequences long enough to span several segments of the packed plan
    (the segment pass, whose first tile reaches 64 tokens before each sequence start, the
    scan and the main walk all cross packed boundaries), with ragged ends, a one-token and an
    empty sequence; each sequence equals its own forward."""
    _varlen_case(lz, oracle_mod, I.LLAMA3_8B_L8K, [2600, 33, 1, 0, 1500, 64, 2100])


def test_varlen_one_launch_closed_gates(lz, oracle_mod):
    """Strongly closed gates in a packed batch: steps handed to the exact tail walk, which
    walks each packed sequence from its own rows."""
    _varlen_case(lz, oracle_mod, I.closed_gates(I.LLAMA3_8B_L8K, per_1k=8.0), [1700, 300, 900])


def test_varlen_one_launch_matches_sequence_loop(lz):
    """The one-launch path and the sequence-by-sequence path (chosen by a workspace too small
    for the first) agree.  They cut segments differently, so the state reaches each boundary
    through different bf16-rounded update products: y within bf16 rounding, S, z and lse
    within 1e-3 relative (each path also meets the oracle bounds, tested above)."""
    wl = I.LLAMA3_8B_L8K
    lens = [700, 129, 2000, 5, 1000]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    t = to_dev(I.make_inputs(wl.replace(B=1, L=T)), wl.dtype)
    dims = lz.make_dims(len(lens), T, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w, wl.M, torch.bfloat16)
    one = lz.make_dims(1, T, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w, wl.M, torch.bfloat16)
    big, small = lz.lizard_attn_fwd_varlen_workspace(dims, cu), lz.lizard_attn_fwd_workspace(one)
    assert big > small > 0
    ws_big = lz.new_workspace(big, torch.device("cuda"))
    ws_small = lz.new_workspace(small, torch.device("cuda"))
    ya, Sa, za, la = _varlen_run(lz, wl, t, cu, ws_big)
    yb, Sb, zb, lb = _varlen_run(lz, wl, t, cu, ws_small)
    torch.cuda.synchronize()
    assert lz.lizard_read_device_status(ws_big) == lz.LIZARD_OK
    ya, yb = to_np(ya), to_np(yb)
    assert np.abs(ya - yb).max() <= 2e-2 * np.sqrt(np.mean(yb * yb)) + 1e-30
    for x, r in ((Sa, Sb), (za, zb), (la, lb)):
        x, r = to_np(x), to_np(r)
        assert np.linalg.norm(x - r) <= 1e-3 * np.linalg.norm(r)


def _closed_quarters(g) -> int:
    """Number of (batch, 8-token quarter, KV head, feature) cells whose gates decay by more
    than e^-36: the cells that take the tensor-core forward's exact tail walk."""
    B, L, H, D = g.shape
    ls = -np.logaddexp(0.0, -np.asarray(g, np.float64))
    n = L // 8 * 8
    return int((ls[:, :n].reshape(B, n // 8, 8, H, D).sum(2) < -36.0).sum())


@pytest.mark.parametrize("base,L,B,gla", [
    ("llama", 8192, 1, False),   # LLaMA-shaped heads, runs inside N(3, 1.5) gates
    ("llama", 1000, 1, True),    # ragged length, state term large (closing it matters)
    ("mistral", 2048, 2, False),
    ("mistral", 2048, 2, True),
])
def test_closed_gate_runs(lz, oracle_mod, base, L, B, gla):
    """Runs of 16-48 tokens whose gate logits are N(-12, 1) or N(-30, 1) (Lizard summary
    sec. 2-C: cumulative gate products that underflow).  The tensor-core walk hands each such
    step to the exact tail walk; y, lse, the final state and z match the oracle."""
    wl = {"llama": I.LLAMA3_8B_L8K, "mistral": I.MISTRAL_7B_TRAIN}[base]
    if gla:
        wl = I.gla_sensitive(wl)
    wl = I.closed_gates(wl)
    inp = I.make_inputs(wl, L=L, B=B)
    assert _closed_quarters(inp["g"]) > 0
    out = gpu_fwd(lz, inp, wl, lse=True, state=True)
    ref = oracle_fwd(oracle_mod, inp, wl, parts=True, state=True)
    assert_parity(out["y"], ref["y"], "bf16", "y")
    assert rel_l2(out["lse"], np.log(ref["den"])) < 1e-3
    assert_parity(out["S_out"], ref["S"], "bf16", "S")
    assert_parity(out["z_out"], ref["z"], "bf16", "z")


def test_closed_gates_every_step(lz, oracle_mod):
    """Every gate strongly closed (logits N(-20, 1)): the whole sequence runs on the exact
    walk from its first step; the state holds only the key that just left the window."""
    wl = I.LLAMA3_8B_L8K.replace(gate=("normal", -20.0, 1.0))
    inp = I.make_inputs(wl, L=700)
    out = gpu_fwd(lz, inp, wl, lse=True, state=True)
    ref = oracle_fwd(oracle_mod, inp, wl, parts=True, state=True)
    assert_parity(out["y"], ref["y"], "bf16", "y")
    assert_parity(out["S_out"], ref["S"], "bf16", "S")


def test_closed_gates_repeat_bitwise(lz):
    """The hand-off marks live in the workspace: a second call with open gates on the same
    workspace is unaffected by the first call's marks, and repeats are bit-identical."""
    wl = I.closed_gates(I.LLAMA3_8B_L8K)
    tc = to_dev(I.make_inputs(wl, L=4096), wl.dtype)
    to = to_dev(I.make_inputs(I.LLAMA3_8B_L8K, L=4096), wl.dtype)
    dims = lz.dims_of(tc["q"], tc["k"], tc["g"], tc["sinks"], wl.w)
    ws = lz.new_workspace(lz.lizard_attn_fwd_workspace(dims), "cuda")
    run = lambda t: lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"],
                                       wl.w, workspace=ws)
    yc1 = run(tc)
    yo1 = run(to)
    yc2 = run(tc)
    yo2 = run(to)
    torch.cuda.synchronize()
    assert torch.equal(yc1, yc2) and torch.equal(yo1, yo2)
    fresh = lz.lizard_attn_fwd(to["q"], to["k"], to["v"], to["g"], to["Wf"], to["sinks"], wl.w)
    torch.cuda.synchronize()
    assert torch.equal(yo1, fresh)
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK


@pytest.mark.parametrize("M", [0, 1, 64])
def test_tensor_core_forward_sink_counts(lz, oracle_mod, M):
    """The tensor-core walk with no sinks, one, and the most it takes (64 per head): the
    sinks only enter the shared denominator (and lse)."""
    wl = I.LLAMA3_8B_L8K.replace(M=M)
    inp = I.make_inputs(wl, L=700)
    out = gpu_fwd(lz, inp, wl, lse=True)
    ref = oracle_fwd(oracle_mod, inp, wl, parts=True)
    assert_parity(out["y"], ref["y"], "bf16", "y")
    assert rel_l2(out["lse"], np.log(ref["den"])) < 1e-3


@pytest.mark.parametrize("L", [1000, 1100])
def test_tensor_core_forward_batch_ragged(lz, oracle_mod, L):
    """Several batch entries with a ragged length on the tensor-core walk: the (batch, KV
    head) units and the segments of each entry, partial last steps, state and ring outputs."""
    wl = I.LLAMA3_8B_L8K.replace(B=3, L=L, Hq=8, Hkv=2)
    inp = I.make_inputs(wl)
    out = gpu_fwd(lz, inp, wl, lse=True, state=True, cache=True)
    ref = oracle_fwd(oracle_mod, inp, wl, parts=True, state=True)
    assert_parity(out["y"], ref["y"], "bf16", "y")
    assert rel_l2(out["lse"], np.log(ref["den"])) < 1e-3
    assert_parity(out["S_out"], ref["S"], "bf16", "S")
    for t in range(L - wl.w, L):
        np.testing.assert_array_equal(out["kcache_out"][:, :, t % (wl.w + 1)], inp["k"][:, t])
