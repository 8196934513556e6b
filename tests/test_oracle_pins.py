"""Pins of the float64 oracle to facts outside itself (no GPU).

Each test ties the recurrent oracle to something it does not compute: a brute
force written from the weight definition, hand-derived closed forms, a library
attention routine, invariants of the formula, finite differences, and the
alternate chunked and log-space forms of the Lizard summary
(gist.science/ko/paper/2507.09025, sec. 2-A and 2-C).
"""
import json
import math
import os

import numpy as np
import pytest

from gated_linear_sliding_gb300 import inputs as I
from oracle import forms

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small(**kw):
    base = I.TINY_F32.replace(L=16, d=6, D=8, Hq=4, Hkv=2, w=4, B=2)
    return base.replace(**kw)


def f64(inp):
    return {k: np.asarray(v, np.float64) for k, v in inp.items()}


def rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("w", [1, 2, 4, 8, 16])
def test_brute_force_matches_recurrence(oracle_mod, w):
    wl = small(w=w)
    inp = I.make_inputs(wl)
    y = oracle_mod.fwd(**inp, w=w)["y"]
    yb = forms.brute_force(inp, w)
    assert rel(y, yb) < 1e-13


def test_brute_force_gla_sensitive(oracle_mod):
    wl = I.gla_sensitive(small(w=3, L=14))
    inp = I.make_inputs(wl)
    y = oracle_mod.fwd(**inp, w=3, scale=wl.scale)["y"]
    yb = forms.brute_force(inp, 3, scale=wl.scale)
    assert rel(y, yb) < 1e-13


def test_closed_form_golden(oracle_mod):
    spec = json.load(open(os.path.join(GOLDEN, "closed_form_cases.json")))
    for case in spec["cases"]:
        L, w, D = len(case["v"]), case["w"], case["D"]
        q = np.zeros((1, L, 1, 1))
        k = np.linspace(-1.0, 1.0, L).reshape(1, L, 1, 1)  # phi(k) = [1, 1] whatever k is
        v = np.asarray(case["v"], np.float64).reshape(1, L, 1, 1)
        g = np.asarray(case["g"], np.float64).reshape(1, L, 1, D)
        Wf = np.full((1, 1, D // 2), 0.7)
        sinks = np.zeros((1, 1))
        y = oracle_mod.fwd(q, k, v, g, Wf, sinks, w=w, scale=1.0)["y"].reshape(-1)
        np.testing.assert_allclose(y, case["y"], rtol=1e-14, atol=0, err_msg=case["name"])


def test_phi_sign_structure_closed_form(oracle_mod):
    """D/2 = 2: softmax([a, b]) = [sig(a-b), sig(b-a)], softmax([-a, -b]) = [sig(b-a), sig(a-b)].

    With gates at 1 (g = 50 rounds sigmoid to 1.0 in fp64), the state weight of
    key j for query i is phi(q_i).phi(k_j) = 2[sig(x)sig(y) + sig(-x)sig(-y)],
    x = q(w1 - w2), y = k(w1 - w2).  With w = 1 and L = 2, query 1 sees key 0
    through the state and key 1 through the window.
    """
    sig = lambda x: 1.0 / (1.0 + math.exp(-x))
    w1, w2 = 0.9, -0.4
    qv, kv0, kv1 = [0.3, 1.7], [-1.1, 0.5], [2.0, 3.0]
    q = np.array(qv).reshape(1, 2, 1, 1)
    k = np.array(kv0).reshape(1, 2, 1, 1)
    v = np.array(kv1).reshape(1, 2, 1, 1)
    g = np.full((1, 2, 1, 4), 50.0)
    Wf = np.array([[[w1, w2]]])
    sinks = np.array([[-1e4]])
    y = oracle_mod.fwd(q, k, v, g, Wf, sinks, w=1, scale=1.0)["y"].reshape(-1)
    a = qv[1] * (w1 - w2)
    b = kv0[0] * (w1 - w2)
    lin = 2 * (sig(a) * sig(b) + sig(-a) * sig(-b))
    e11 = math.exp(qv[1] * kv0[1])
    expect1 = (lin * kv1[0] + e11 * kv1[1]) / (lin + e11)
    assert abs(y[1] - expect1) < 1e-14
    assert abs(y[0] - kv1[0]) < 1e-14  # only key 0 in the window, no sinks


def test_forms_agree_tiny_workload(oracle_mod):
    wl = I.TINY_F32
    inp = I.make_inputs(wl)
    y = oracle_mod.fwd(**inp, w=wl.w)["y"]
    assert rel(forms.quadratic_parallel(inp, wl.w), y) < 1e-12
    assert rel(forms.chunked_cumprod(inp, wl.w, C=64), y) < 1e-12
    assert rel(forms.chunked_logspace(inp, wl.w, C=64), y) < 1e-12
    # ragged chunking (last chunk shorter than the others)
    assert rel(forms.chunked_logspace(inp, wl.w, C=48), y) < 1e-12


def test_forms_agree_gla_sensitive(oracle_mod):
    wl = I.gla_sensitive(I.TINY_F32.replace(L=192, Hq=4, Hkv=2))
    inp = I.make_inputs(wl)
    y = oracle_mod.fwd(**inp, w=wl.w, scale=wl.scale)["y"]
    parts = oracle_mod.fwd(**inp, w=wl.w, scale=wl.scale, parts=True)
    # the state term carries real weight in this variant
    assert np.median(parts["den_gla"][:, wl.L // 2:] / parts["den"][:, wl.L // 2:]) > 0.1
    assert rel(forms.chunked_cumprod(inp, wl.w, C=64, scale=wl.scale), y) < 1e-12
    assert rel(forms.chunked_logspace(inp, wl.w, C=64, scale=wl.scale), y) < 1e-12


def test_logspace_equals_cumprod_under_stress_gates():
    """Sec. 2-C: the log-space form equals the product form in fp64, also with the
    stress mixture (30 % of gate logits near -3) that drives chunk products far below 1."""
    wl = I.STRESS_L64K.replace(L=160, d=16, D=16, Hq=2, Hkv=1, dtype="f32")
    inp = I.make_inputs(wl)
    a = forms.chunked_cumprod(inp, wl.w, C=64)
    b = forms.chunked_logspace(inp, wl.w, C=64)
    assert rel(a, b) < 1e-12


def test_gates_one_no_sinks_is_window_softmax_plus_linear(oracle_mod):
    """Gates at 1 and t -> -inf: y is causal sliding-window softmax plus ungated linear
    attention over the keys that have left the window, with one normaliser."""
    wl = small(w=5, L=24)
    inp = f64(I.make_inputs(wl))
    inp["g"][:] = 50.0
    inp["sinks"][:] = -1e4
    y = oracle_mod.fwd(**inp, w=wl.w)["y"]
    q, k, v, Wf = inp["q"], inp["k"], inp["v"], inp["Wf"]
    B, L, Hq, d = q.shape
    G = Hq // wl.Hkv
    expect = np.zeros_like(y)
    for b in range(B):
        for h in range(Hq):
            kv = h // G
            pq, pk = forms.phi(q[b, :, h], Wf[kv]), forms.phi(k[b, :, kv], Wf[kv])
            lin = np.tril(pq @ pk.T, -wl.w)
            s = (q[b, :, h] @ k[b, :, kv].T) / math.sqrt(d)
            i, j = np.indices((L, L))
            win = np.where((j <= i) & (j > i - wl.w), np.exp(s), 0.0)
            A = lin + win
            expect[b, :, h] = (A @ v[b, :, kv]) / A.sum(1, keepdims=True)
    assert rel(y, expect) < 1e-13


def test_closed_gates_state_holds_only_the_leaving_key(oracle_mod):
    """Every gate shut (g = -200, Gamma ~ 1e-87): each step's decay wipes the state, so it
    holds only the key that has just left the window.  y_i is then a softmax-like average
    over the w window keys and key i - w, the latter weighted by phi(q_i).phi(k_{i-w}) instead
    of e^{s q.k}, with the sinks in the denominator (Lizard summary sec. 2-A-1, 2-A-2)."""
    wl = small(w=3, L=20)
    inp = f64(I.make_inputs(wl))
    inp["g"][:] = -200.0
    y = oracle_mod.fwd(**inp, w=wl.w)["y"]
    q, k, v, Wf, t = inp["q"], inp["k"], inp["v"], inp["Wf"], inp["sinks"]
    B, L, Hq, d = q.shape
    G = Hq // wl.Hkv
    expect = np.zeros_like(y)
    for b in range(B):
        for h in range(Hq):
            kv = h // G
            pq, pk = forms.phi(q[b, :, h], Wf[kv]), forms.phi(k[b, :, kv], Wf[kv])
            for i in range(L):
                num = np.zeros(d)
                den = np.exp(t[h]).sum()
                for j in range(max(0, i - wl.w + 1), i + 1):
                    e = math.exp(q[b, i, h] @ k[b, j, kv] / math.sqrt(d))
                    num += e * v[b, j, kv]
                    den += e
                if i >= wl.w:
                    a = pq[i] @ pk[i - wl.w]
                    num += a * v[b, i - wl.w, kv]
                    den += a
                expect[b, i, h] = num / den
    assert rel(y, expect) < 1e-13


def test_full_window_no_sinks_is_causal_softmax_attention(oracle_mod):
    """w >= L and no sinks: y is textbook causal softmax attention (torch SDPA, fp64)."""
    import torch

    wl = small(L=20, w=20)
    inp = f64(I.make_inputs(wl))
    inp["sinks"][:] = -1e4
    y = oracle_mod.fwd(**inp, w=wl.w)["y"]
    G = wl.Hq // wl.Hkv
    q = torch.from_numpy(inp["q"]).permute(0, 2, 1, 3)
    k = torch.from_numpy(inp["k"]).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    v = torch.from_numpy(inp["v"]).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                           scale=wl.scale)
    assert rel(y, ref.permute(0, 2, 1, 3).numpy()) < 1e-13


def test_uniform_phi_closed_form(oracle_mod):
    """Wf = 0 makes phi uniform (2/D per feature), so phi(q).phi(k) = 4/D; with gates at 1,
    the state denominator of query i is (i - w + 1) * 4/D."""
    wl = small(w=3, L=16)
    inp = f64(I.make_inputs(wl))
    inp["Wf"][:] = 0.0
    inp["g"][:] = 50.0
    out = oracle_mod.fwd(**inp, w=wl.w, parts=True)
    i = np.arange(wl.L)
    expect = np.maximum(i - wl.w + 1, 0) * 4.0 / wl.D
    np.testing.assert_allclose(out["den_gla"], np.broadcast_to(expect[None, :, None],
                                                               out["den_gla"].shape),
                               rtol=1e-14, atol=1e-15)


def test_value_ones_identity_and_convex_hull(oracle_mod):
    """Sinks only add to the denominator: v = 1 gives y = 1 - sum_m e^{t_m} / den.
    And y is a sub-convex combination of the values, so |y| <= max |v|."""
    wl = small(w=4, L=32)
    inp = f64(I.make_inputs(wl))
    out = oracle_mod.fwd(**inp, w=wl.w, parts=True)
    assert np.abs(out["y"]).max() <= np.abs(inp["v"]).max() + 1e-12
    ones = dict(inp, v=np.ones_like(inp["v"]))
    o1 = oracle_mod.fwd(**ones, w=wl.w, parts=True)
    sink = np.exp(inp["sinks"]).sum(1)  # [Hq]
    expect = 1.0 - sink[None, None, :, None] / o1["den"][..., None]
    np.testing.assert_allclose(o1["y"], np.broadcast_to(expect, o1["y"].shape), rtol=1e-13)
    np.testing.assert_allclose(o1["den"], o1["den_gla"] + o1["den_win"] + sink[None, None],
                               rtol=1e-14)


def test_gqa_head_mapping(oracle_mod):
    """Query head h reads KV head h // G: GQA equals the un-grouped run with every KV
    tensor repeated G times along the head axis."""
    wl = small(Hq=6, Hkv=2, w=3, L=16)
    inp = f64(I.make_inputs(wl))
    y = oracle_mod.fwd(**inp, w=wl.w)["y"]
    G = 3
    rep = dict(inp)
    for n in ("k", "v", "g"):
        rep[n] = np.repeat(inp[n], G, axis=2)
    rep["Wf"] = np.repeat(inp["Wf"], G, axis=0)
    y2 = oracle_mod.fwd(**rep, w=wl.w)["y"]
    assert rel(y, y2) < 1e-15


def test_state_is_constant_size(oracle_mod):
    """Sec. 2-A-1: inference keeps a constant-size state; the oracle's final state has the
    same shape at every L, and continuing from it equals the longer prefill."""
    wl = small(w=4)
    for L in (8, 64):
        out = oracle_mod.fwd(**I.make_inputs(wl, L=L), w=wl.w, state=True)
        assert out["S"].shape == (wl.B, wl.Hkv, wl.D, wl.d)
        assert out["z"].shape == (wl.B, wl.Hkv, wl.D)


@pytest.mark.parametrize("L0", [0, 3, 37])
def test_decode_reproduces_prefill(oracle_mod, L0):
    """Prefill of L0 tokens, then token-by-token decode, equals the prefill of all tokens."""
    wl = small(w=5, L=48)
    inp = f64(I.make_inputs(wl))
    full = oracle_mod.fwd(**inp, w=wl.w)["y"]
    R = wl.w + 1
    if L0 > 0:
        pre = oracle_mod.fwd(**{n: (a[:, :L0] if n in "qkvg" else a) for n, a in inp.items()},
                             w=wl.w, state=True)
        S, z = pre["S"].copy(), pre["z"].copy()
    else:
        S = np.zeros((wl.B, wl.Hkv, wl.D, wl.d))
        z = np.zeros((wl.B, wl.Hkv, wl.D))
    kc = np.zeros((wl.B, wl.Hkv, R, wl.d))
    vc = np.zeros((wl.B, wl.Hkv, R, wl.d))
    for t in range(max(0, L0 - wl.w), L0):
        kc[:, :, t % R] = inp["k"][:, t]
        vc[:, :, t % R] = inp["v"][:, t]
    for pos in range(L0, wl.L):
        y = oracle_mod.decode_step(pos, inp["q"][:, pos], inp["k"][:, pos], inp["v"][:, pos],
                                   inp["g"][:, pos], inp["Wf"], inp["sinks"], S, z, kc, vc,
                                   w=wl.w)
        assert rel(y, full[:, pos]) < 1e-13


def _fd_check(oracle_mod, wl, h=1e-6, tol=1e-6):
    inp = f64(I.make_inputs(wl))
    dy = np.random.default_rng(11).standard_normal(inp["q"].shape)
    gr = oracle_mod.bwd(**inp, dy=dy, w=wl.w)

    def loss(x):
        return float((oracle_mod.fwd(**x, w=wl.w)["y"] * dy).sum())

    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("Wf", "dWf"),
                        ("sinks", "dsinks")):
        a = inp[name]
        fd = np.zeros_like(a)
        for idx in np.ndindex(a.shape):
            xp = dict(inp)
            xp[name] = a.copy()
            xp[name][idx] += h
            xm = dict(inp)
            xm[name] = a.copy()
            xm[name][idx] -= h
            fd[idx] = (loss(xp) - loss(xm)) / (2 * h)
        scale = max(np.abs(fd).max(), 1e-12)
        err = np.abs(fd - gr[gname]).max() / scale
        assert err < tol, (name, err)
    return gr


def test_backward_finite_differences_w4(oracle_mod):
    """The reverse pass is the exact gradient: central differences (h = 1e-6) on B=1,
    Hq=2 (G=2), L=16, w=4, where dg and dWf are non-zero."""
    gr = _fd_check(oracle_mod, I.TINY_F32.replace(B=1, L=16, Hq=2, Hkv=1, d=6, D=8, w=4))
    assert np.abs(gr["dg"]).max() > 1e-4


def test_backward_finite_differences_w64(oracle_mod):
    """w = 64 > L: the state term is empty, so dg must vanish."""
    gr = _fd_check(oracle_mod, I.TINY_F32.replace(B=1, L=16, Hq=1, Hkv=1, d=6, D=8, w=64))
    assert np.abs(gr["dg"]).max() == 0.0


def test_backward_finite_differences_gla_sensitive(oracle_mod):
    wl = I.gla_sensitive(I.TINY_F32.replace(B=1, L=12, Hq=2, Hkv=1, d=4, D=6, w=2))
    inp = f64(I.make_inputs(wl))
    dy = np.random.default_rng(3).standard_normal(inp["q"].shape)
    gr = oracle_mod.bwd(**inp, dy=dy, w=wl.w, scale=wl.scale)

    def loss(x):
        return float((oracle_mod.fwd(**x, w=wl.w, scale=wl.scale)["y"] * dy).sum())

    for name, gname in (("g", "dg"), ("Wf", "dWf"), ("k", "dk")):
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
        # slow gates make dg small (Gamma (1 - Gamma) ~ 3e-4): the bound is the FD roundoff
        assert np.abs(fd - gr[gname]).max() / np.abs(fd).max() < 2e-5, name


def test_bf16_product_form_breaks_log_space_holds():
    """Sec. 2-C: with the stress mixture of gate logits, the product of gates over one
    64-token chunk leaves the fp32/bf16 range when it is folded into the keys as a
    reciprocal, while the log-space fold referenced to each 16-token sub-block keeps
    every factor finite and <= e^{88}."""
    wl = I.STRESS_L64K
    g = I.make_inputs(wl.replace(L=64 * 64, Hq=8, Hkv=1, d=16))["g"][0, :, 0, :]
    g = g.reshape(64, 64, wl.D).astype(np.float32)  # [chunk, token, feature]
    gam = (1.0 / (1.0 + np.exp(-g.astype(np.float64)))).astype(np.float32)
    with np.errstate(over="ignore", under="ignore", divide="ignore"):
        cp = np.cumprod(gam, axis=1)                  # fp32 product from the chunk start
        naive_fold = 1.0 / cp                         # key-side factor of the product form
    assert np.isinf(naive_fold).any() or (cp == 0).any()
    lam = -np.logaddexp(0.0, -g.astype(np.float64))
    b = np.cumsum(lam, axis=1)
    # sub-block reference: the last position before each 16-token sub-block
    ref = np.concatenate([np.zeros((64, 1, wl.D)), b[:, 15:-1:16]], axis=1)  # [chunk, 4, D]
    rb = np.repeat(ref, 16, axis=1)
    k_side = np.exp(rb - b)                           # >= 1 inside a sub-block only
    assert np.isfinite(k_side.astype(np.float32)).all()
    assert (rb - b).max() < 88.0
