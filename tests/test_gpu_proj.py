"""Parity of the projections in front of the mixer (lizard_qkvg_proj and its backward, through
the C ABI) against the fp64 oracle.  Lizard summary (gist.science 2507.09025) sec. 2-A-1: the
gate logits are a learned projection of the layer input, next to q, k and v.
"""
import numpy as np
import pytest

from gated_linear_sliding_gb300 import inputs as I
from helpers import assert_grad, assert_parity, rel_l2, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lz():
    from gated_linear_sliding_gb300 import lizard

    lizard.load()
    return lizard


def dev(a, dt=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda().to(dt)


def heads(wl):
    return wl.Hq, wl.Hkv, wl.d, wl.D


@pytest.mark.parametrize("wl,dm,L,B", [
    (I.LLAMA3_8B_L8K, 256, 300, 1),      # 256-wide output tiles, ragged token count
    (I.MISTRAL_7B_TRAIN, 512, 1000, 2),
    (I.LLAMA3_8B_L8K.replace(Hq=4, Hkv=1), 192, 77, 1),  # widths 512/128/128/128: 128-wide tiles
])
def test_projection_forward_and_backward(lz, oracle_mod, wl, dm, L, B):
    inp = I.make_proj_inputs(wl, dm, L=L, B=B, with_grads=True)
    x, W = dev(inp["x"]), dev(inp["W"])
    q, k, v, g = lz.lizard_qkvg_proj(x, W, *heads(wl))
    ref = oracle_mod.qkvg_proj(inp["x"], inp["W"], *heads(wl))
    torch.cuda.synchronize()
    for name, t in zip("qkvg", (q, k, v, g)):
        assert_parity(to_np(t), ref[name], "bf16", name)
    grads = {n: dev(inp[n]) for n in ("dq", "dk", "dv", "dg")}
    dx, dW = lz.lizard_qkvg_proj_bwd(x, W, grads["dq"], grads["dk"], grads["dv"], grads["dg"])
    refb = oracle_mod.qkvg_proj_bwd(inp["x"], inp["W"], inp["dq"], inp["dk"], inp["dv"],
                                    inp["dg"])
    torch.cuda.synchronize()
    assert_parity(to_np(dx), refb["dx"], "bf16", "dx")
    assert rel_l2(to_np(dW), refb["dW"]) <= 1e-5, rel_l2(to_np(dW), refb["dW"])


def test_projection_full_llama_size_sampled(lz, oracle_mod):
    """x [8192, 4096] and W [7168, 4096]: the GPU computes everything; the oracle checks 48
    sampled tokens of q, k, v, g and dx and 48 sampled rows of dW, each in full."""
    wl = I.LLAMA3_8B_L8K
    dm = 4096
    inp = I.make_proj_inputs(wl, dm, with_grads=True)
    x, W = dev(inp["x"]), dev(inp["W"])
    q, k, v, g = lz.lizard_qkvg_proj(x, W, *heads(wl))
    grads = {n: dev(inp[n]) for n in ("dq", "dk", "dv", "dg")}
    dx, dW = lz.lizard_qkvg_proj_bwd(x, W, grads["dq"], grads["dk"], grads["dv"], grads["dg"])
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    toks = np.sort(rng.choice(wl.L, 48, replace=False))
    sub = {"x": inp["x"][:, toks]}
    ref = oracle_mod.qkvg_proj(sub["x"], inp["W"], *heads(wl))
    for name, t in zip("qkvg", (q, k, v, g)):
        assert_parity(to_np(t[:, toks]), ref[name], "bf16", name)
    refb = oracle_mod.qkvg_proj_bwd(sub["x"], inp["W"], *(inp[n][:, toks] for n in
                                                         ("dq", "dk", "dv", "dg")))
    assert_parity(to_np(dx[:, toks]), refb["dx"], "bf16", "dx")
    rows = np.sort(rng.choice(W.shape[0], 48, replace=False))
    dY = np.concatenate([inp[n].reshape(wl.L, -1) for n in ("dq", "dk", "dv", "dg")], axis=1)
    refw = dY[:, rows].astype(np.float64).T @ inp["x"][0].astype(np.float64)
    assert rel_l2(to_np(dW[rows]), refw) <= 1e-5


def test_layer_gradient_through_projection_and_mixer(lz, oracle_mod):
    """x -> projections -> mixer -> y, then the mixer's backward and the projections' backward:
    dx and dW of the whole layer against the oracle chain (LLaMA-shaped heads, dm = 256)."""
    wl = I.LLAMA3_8B_L8K
    dm, L = 256, 640
    inp = I.make_proj_inputs(wl, dm, L=L)
    mix = I.make_inputs(wl, L=L, with_dy=True)
    x, W = dev(inp["x"]), dev(inp["W"])
    Wf, sinks, dy = dev(mix["Wf"]), torch.from_numpy(mix["sinks"]).cuda(), dev(mix["dy"])
    q, k, v, g = lz.lizard_qkvg_proj(x, W, *heads(wl))
    lse = torch.empty(1, L, wl.Hq, device="cuda")
    y = lz.lizard_attn_fwd(q, k, v, g, Wf, sinks, wl.w, lse=lse)
    gm = lz.lizard_attn_bwd(q, k, v, g, Wf, sinks, y, lse, dy, wl.w)
    dx, dW = lz.lizard_qkvg_proj_bwd(x, W, gm["dq"], gm["dk"], gm["dv"], gm["dg"])
    torch.cuda.synchronize()
    # the oracle chain runs on the GPU's own bf16 projections, so it checks the backward chain
    qn, kn, vn, gn = (to_np(t) for t in (q, k, v, g))
    ref = oracle_mod.bwd(qn, kn, vn, gn, mix["Wf"], mix["sinks"], mix["dy"], w=wl.w)
    refp = oracle_mod.qkvg_proj_bwd(inp["x"], inp["W"], ref["dq"], ref["dk"], ref["dv"], ref["dg"])
    assert_grad(to_np(dx), refp["dx"], "bf16", "dx")
    assert_grad(to_np(dW), refp["dW"], "bf16", "dW")
