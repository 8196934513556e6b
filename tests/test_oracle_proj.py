"""Pins of the fp64 projection oracle (no GPU).

[q | k | v | g] = x W^T is the step in front of the mixer: the gate logits are a learned
projection of the layer input (Lizard summary, gist.science/ko/paper/2507.09025, sec.
2-A-1: Gamma_i = sigmoid(W_gamma x_i)), beside the attention projections.  The oracle is a
library matrix product; these tests tie it to a brute-force sum written out loop by loop, to
the row order of W, and (for the backward) to central finite differences of the whole
layer, projection followed by the mixer.
"""
import math

import numpy as np

from gated_linear_sliding_gb300 import inputs as I


def tiny(**kw):
    base = I.TINY_F32.replace(B=1, L=3, Hq=2, Hkv=1, d=2, D=2, w=2, M=1)
    return base.replace(**kw)


def test_projection_brute_force_and_row_order(oracle_mod):
    wl = tiny()
    dm = 5
    inp = I.make_proj_inputs(wl, dm)
    x, W = inp["x"].astype(np.float64), inp["W"].astype(np.float64)
    out = oracle_mod.qkvg_proj(x, W, wl.Hq, wl.Hkv, wl.d, wl.D)
    # W's rows: q heads (Hq d), then k (Hkv d), v (Hkv d), gate (Hkv D), each head's
    # features contiguous
    order = ([("q", h, e) for h in range(wl.Hq) for e in range(wl.d)]
             + [("k", h, e) for h in range(wl.Hkv) for e in range(wl.d)]
             + [("v", h, e) for h in range(wl.Hkv) for e in range(wl.d)]
             + [("g", h, e) for h in range(wl.Hkv) for e in range(wl.D)])
    assert len(order) == W.shape[0]
    for t in range(wl.L):
        for n, (name, h, e) in enumerate(order):
            s = 0.0
            for c in range(dm):
                s += x[0, t, c] * W[n, c]
            assert math.isclose(out[name][0, t, h, e], s, rel_tol=1e-13, abs_tol=1e-15)


def test_projection_backward_brute_force(oracle_mod):
    wl = tiny()
    dm = 4
    inp = I.make_proj_inputs(wl, dm, with_grads=True)
    x, W = inp["x"].astype(np.float64), inp["W"].astype(np.float64)
    g = oracle_mod.qkvg_proj_bwd(x, W, inp["dq"], inp["dk"], inp["dv"], inp["dg"])
    dY = np.concatenate([inp[n].reshape(wl.L, -1) for n in ("dq", "dk", "dv", "dg")], axis=1)
    N = W.shape[0]
    for t in range(wl.L):
        for c in range(dm):
            s = sum(dY[t, n] * W[n, c] for n in range(N))
            assert math.isclose(g["dx"][0, t, c], s, rel_tol=1e-13, abs_tol=1e-15)
    for n in range(N):
        for c in range(dm):
            s = sum(dY[t, n] * x[0, t, c] for t in range(wl.L))
            assert math.isclose(g["dW"][n, c], s, rel_tol=1e-13, abs_tol=1e-15)


def test_layer_gradient_finite_differences(oracle_mod):
    """Projection then mixer: loss = sum(dy * y).  The chain of the oracle's mixer reverse
    pass and qkvg_proj_bwd gives dloss/dx and dloss/dW; central differences (h = 1e-6) of the
    fp64 forward agree with them on sampled entries."""
    wl = tiny(L=7, Hq=2, Hkv=1, d=3, D=4, w=2, M=2)
    dm = 5
    inp = I.make_proj_inputs(wl, dm)
    x, W = inp["x"].astype(np.float64), inp["W"].astype(np.float64)
    rng = np.random.default_rng(11)
    Wf = rng.standard_normal((wl.Hkv, wl.d, wl.D // 2))
    sinks = rng.standard_normal((wl.Hq, wl.M))
    dy = rng.standard_normal((1, wl.L, wl.Hq, wl.d))

    def loss(xx, WW):
        p = oracle_mod.qkvg_proj(xx, WW, wl.Hq, wl.Hkv, wl.d, wl.D)
        y = oracle_mod.fwd(p["q"], p["k"], p["v"], p["g"], Wf, sinks, w=wl.w)["y"]
        return float((dy * y).sum())

    p = oracle_mod.qkvg_proj(x, W, wl.Hq, wl.Hkv, wl.d, wl.D)
    gm = oracle_mod.bwd(p["q"], p["k"], p["v"], p["g"], Wf, sinks, dy, w=wl.w)
    gp = oracle_mod.qkvg_proj_bwd(x, W, gm["dq"], gm["dk"], gm["dv"], gm["dg"])
    h = 1e-6
    for _ in range(8):
        t, c = rng.integers(wl.L), rng.integers(dm)
        e = np.zeros_like(x)
        e[0, t, c] = h
        fd = (loss(x + e, W) - loss(x - e, W)) / (2 * h)
        assert math.isclose(gp["dx"][0, t, c], fd, rel_tol=1e-5, abs_tol=1e-8)
        n = rng.integers(W.shape[0])
        e = np.zeros_like(W)
        e[n, c] = h
        fd = (loss(x, W + e) - loss(x, W - e)) / (2 * h)
        assert math.isclose(gp["dW"][n, c], fd, rel_tol=1e-5, abs_tol=1e-8)
