"""Pins of the oracle's two other decay readings (no GPU).

The pages (Lizard summary, gist.science/ko/paper/2507.09025, sec. 2-A-1) say that the
gate decays a constant-size state of the tokens outside the window, not which gates a
key that has left the window has seen.  Beside the delayed-key reading the oracle keeps
two others; a key j <= i - w reaches query i with the gate product over
  masked (full GLA with the window masked out)   s = j+1 .. i,
  lagged (the query reads the state of i - w)    s = j+1 .. i-w.
Each is tied here to something the recurrence does not compute: hand-derived cases,
the brute-force weight definition, reductions to known cases, the shifted-gate identity
of the lagged reading, decode against prefill, and central finite differences.
"""
import json
import math
import os

import numpy as np
import pytest

from gated_linear_sliding_gb300 import inputs as I
from oracle import LAGGED, MASKED, forms

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small(**kw):
    base = I.TINY_F32.replace(L=16, d=6, D=8, Hq=4, Hkv=2, w=4, B=2)
    return base.replace(**kw)


def f64(inp):
    return {k: np.asarray(v, np.float64) for k, v in inp.items()}


def rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def test_golden_hand_derived(oracle_mod):
    spec = json.load(open(os.path.join(GOLDEN, "decay_readings_cases.json")))
    for case in spec["cases"]:
        L, w, D = len(case["v"]), case["w"], case["D"]
        q = np.zeros((1, L, 1, 1))
        k = np.linspace(-1.0, 1.0, L).reshape(1, L, 1, 1)  # phi(k) = [1, 1] whatever k is
        v = np.asarray(case["v"], np.float64).reshape(1, L, 1, 1)
        g = np.asarray(case["g"], np.float64).reshape(1, L, 1, D)
        Wf = np.full((1, 1, D // 2), 0.7)
        sinks = np.zeros((1, 1))
        y = oracle_mod.fwd(q, k, v, g, Wf, sinks, w=w, scale=1.0,
                           reading=case["reading"])["y"].reshape(-1)
        np.testing.assert_allclose(y, case["y"], rtol=1e-14, atol=0, err_msg=case["name"])


@pytest.mark.parametrize("reading", [MASKED, LAGGED])
@pytest.mark.parametrize("w", [1, 2, 4, 8])
def test_brute_force_matches_recurrence(oracle_mod, reading, w):
    inp = I.make_inputs(small(w=w))
    y = oracle_mod.fwd(**inp, w=w, reading=reading)["y"]
    assert rel(y, forms.brute_force(inp, w, reading=reading)) < 1e-13


@pytest.mark.parametrize("reading", [MASKED, LAGGED])
def test_quadratic_form_gla_sensitive(oracle_mod, reading):
    """Gates near 1 and unscaled q, k give the state term real weight; the L x L weight
    matrices of the definition agree with the recurrence."""
    wl = I.gla_sensitive(I.TINY_F32.replace(L=96, Hq=4, Hkv=2, d=8, D=8, w=8))
    inp = I.make_inputs(wl)
    y = oracle_mod.fwd(**inp, w=wl.w, scale=wl.scale, reading=reading)["y"]
    assert rel(y, forms.quadratic_parallel(inp, wl.w, scale=wl.scale, reading=reading)) < 1e-12
    # and the readings really differ from the delayed one on these gates
    y0 = oracle_mod.fwd(**inp, w=wl.w, scale=wl.scale)["y"]
    assert rel(y, y0) > 1e-4


def test_open_gates_make_the_readings_coincide(oracle_mod):
    """Gamma = 1 (g = 50 rounds sigmoid to 1 in fp64): every gate product is 1, so all
    three readings give the same y and the same final state."""
    wl = small(w=3, L=20)
    inp = f64(I.make_inputs(wl))
    inp["g"][:] = 50.0
    ref = oracle_mod.fwd(**inp, w=wl.w, state=True)
    for reading in (MASKED, LAGGED):
        out = oracle_mod.fwd(**inp, w=wl.w, state=True, reading=reading)
        for n in ("y", "S", "z"):
            assert rel(out[n], ref[n]) < 1e-15, (reading, n)


def test_masked_closed_gates_leave_window_softmax(oracle_mod):
    """Masked reading with every gate shut (g = -200): a key beyond the window carries at
    least w + 1 gate factors of ~1e-87, so y is the sliding-window softmax with the sinks
    in the denominator (the delayed reading would still hold key i - w)."""
    wl = small(w=3, L=20)
    inp = f64(I.make_inputs(wl))
    inp["g"][:] = -200.0
    y = oracle_mod.fwd(**inp, w=wl.w, reading=MASKED)["y"]
    q, k, v, t = inp["q"], inp["k"], inp["v"], inp["sinks"]
    B, L, Hq, d = q.shape
    G = Hq // wl.Hkv
    expect = np.zeros_like(y)
    for b in range(B):
        for h in range(Hq):
            kv = h // G
            for i in range(L):
                j0 = max(0, i - wl.w + 1)
                e = np.exp(k[b, j0:i + 1, kv] @ q[b, i, h] / math.sqrt(d))
                expect[b, i, h] = (e @ v[b, j0:i + 1, kv]) / (e.sum() + np.exp(t[h]).sum())
    assert rel(y, expect) < 1e-13


def test_lagged_is_delayed_on_gates_shifted_by_w(oracle_mod):
    """prod_{s=j+1..i-w} Gamma_s = prod_{s=j+w+1..i} Gamma'_s with Gamma'_s = Gamma_{s-w}:
    the lagged reading is the delayed one on the gate sequence moved w tokens later (the
    first w entries of the moved sequence only decay the empty state, so any value does)."""
    wl = small(w=4, L=40)
    inp = f64(I.make_inputs(wl))
    lag = oracle_mod.fwd(**inp, w=wl.w, state=True, reading=LAGGED)
    moved = dict(inp)
    moved["g"] = np.concatenate([np.full_like(inp["g"][:, :wl.w], -7.0),
                                 inp["g"][:, :wl.L - wl.w]], axis=1)
    ref = oracle_mod.fwd(**moved, w=wl.w, state=True)
    for n in ("y", "S", "z"):
        assert rel(lag[n], ref[n]) < 1e-14, n


@pytest.mark.parametrize("reading", [MASKED, LAGGED])
@pytest.mark.parametrize("L0", [0, 3, 37])
def test_decode_reproduces_prefill(oracle_mod, reading, L0):
    """Prefill of L0 tokens, then decode with the k, v and gate rings, equals the prefill
    of all tokens under the same reading."""
    wl = small(w=5, L=48)
    inp = f64(I.make_inputs(wl))
    full = oracle_mod.fwd(**inp, w=wl.w, reading=reading)["y"]
    R = wl.w + 1
    if L0 > 0:
        pre = oracle_mod.fwd(**{n: (a[:, :L0] if n in "qkvg" else a) for n, a in inp.items()},
                             w=wl.w, state=True, reading=reading)
        S, z = pre["S"].copy(), pre["z"].copy()
    else:
        S = np.zeros((wl.B, wl.Hkv, wl.D, wl.d))
        z = np.zeros((wl.B, wl.Hkv, wl.D))
    kc = np.zeros((wl.B, wl.Hkv, R, wl.d))
    vc = np.zeros((wl.B, wl.Hkv, R, wl.d))
    gc = np.zeros((wl.B, wl.Hkv, R, wl.D))
    for t in range(max(0, L0 - wl.w), L0):
        kc[:, :, t % R] = inp["k"][:, t]
        vc[:, :, t % R] = inp["v"][:, t]
        gc[:, :, t % R] = inp["g"][:, t]
    for pos in range(L0, wl.L):
        y = oracle_mod.decode_step(pos, inp["q"][:, pos], inp["k"][:, pos], inp["v"][:, pos],
                                   inp["g"][:, pos], inp["Wf"], inp["sinks"], S, z, kc, vc,
                                   w=wl.w, gcache=gc, reading=reading)
        assert rel(y, full[:, pos]) < 1e-13, pos


def test_decode_rejects_missing_gate_ring(oracle_mod):
    wl = small(w=2)
    inp = f64(I.make_inputs(wl))
    S = np.zeros((wl.B, wl.Hkv, wl.D, wl.d))
    z = np.zeros((wl.B, wl.Hkv, wl.D))
    kc = np.zeros((wl.B, wl.Hkv, 3, wl.d))
    vc = np.zeros_like(kc)
    with pytest.raises(ValueError):
        oracle_mod.decode_step(0, inp["q"][:, 0], inp["k"][:, 0], inp["v"][:, 0], inp["g"][:, 0],
                               inp["Wf"], inp["sinks"], S, z, kc, vc, w=2, reading=MASKED)


@pytest.mark.parametrize("reading", [MASKED, LAGGED])
def test_backward_finite_differences(oracle_mod, reading):
    """The adjoint of each reading's recurrence is the exact gradient: central differences
    (h = 1e-6) on B=1, Hq=2 (G=2), L=16, w=3, where dg and dWf are non-zero."""
    wl = I.TINY_F32.replace(B=1, L=16, Hq=2, Hkv=1, d=4, D=6, w=3)
    inp = f64(I.make_inputs(wl))
    dy = np.random.default_rng(17).standard_normal(inp["q"].shape)
    gr = oracle_mod.bwd(**inp, dy=dy, w=wl.w, reading=reading)

    def loss(x):
        return float((oracle_mod.fwd(**x, w=wl.w, reading=reading)["y"] * dy).sum())

    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("Wf", "dWf"),
                        ("sinks", "dsinks")):
        a = inp[name]
        fd = np.zeros_like(a)
        for idx in np.ndindex(a.shape):
            xp = dict(inp)
            xp[name] = a.copy()
            xp[name][idx] += 1e-6
            xm = dict(inp)
            xm[name] = a.copy()
            xm[name][idx] -= 1e-6
            fd[idx] = (loss(xp) - loss(xm)) / 2e-6
        err = np.abs(fd - gr[gname]).max() / max(np.abs(fd).max(), 1e-12)
        assert err < 1e-6, (name, err)
    assert np.abs(gr["dg"]).max() > 1e-4
    if reading == LAGGED:
        # the gates of the last w tokens never decay anything the queries read
        assert np.abs(gr["dg"][:, wl.L - wl.w:]).max() == 0.0


def test_lagged_gradient_is_delayed_gradient_on_moved_gates(oracle_mod):
    """The lagged reading is the delayed one on Gamma'_s = Gamma_{s-w}, so its gradients are
    the delayed reading's on the moved gates, with dg moved back: dg[j] = dg'[j + w], and 0 for
    the last w gates (they decay nothing a query reads).  Ties the lagged adjoint to the
    delayed one, which the finite differences pin."""
    wl = small(w=4, L=40, B=1)
    inp = f64(I.make_inputs(wl))
    dy = np.random.default_rng(23).standard_normal(inp["q"].shape)
    lag = oracle_mod.bwd(**inp, dy=dy, w=wl.w, reading=LAGGED)
    moved = dict(inp)
    moved["g"] = np.concatenate([np.full_like(inp["g"][:, :wl.w], 5.0),
                                 inp["g"][:, :wl.L - wl.w]], axis=1)
    ref = oracle_mod.bwd(**moved, dy=dy, w=wl.w)
    for n in ("dq", "dk", "dv", "dWf", "dsinks"):
        assert rel(lag[n], ref[n]) < 1e-12, n
    assert rel(lag["dg"][:, :wl.L - wl.w], ref["dg"][:, wl.w:]) < 1e-12
    assert not lag["dg"][:, wl.L - wl.w:].any()
