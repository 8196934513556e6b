"""Seeded synthetic inputs for the Lizard hybrid token mixer.

This module only draws random numbers and rounds them to the storage type; it
holds none of the mixer's arithmetic, so that the CPU oracle and the CUDA
library can both be fed from it without sharing any computation.

Shapes (row-major, contiguous):
    q      [B, L, Hq,  d]
    k, v   [B, L, Hkv, d]
    g      [B, L, Hkv, D]   gate logits, Gamma = sigmoid(g) per phi-feature
    Wf     [Hkv, d, D/2]    Hedgehog projection, one per KV head
    sinks  [Hq, M]          meta-memory scalars t_m (always fp32)
    dy     [B, L, Hq, d]    upstream gradient (training workload only)

Workloads follow the Lizard pages (gist.science 2507.09025, section 2-ga
"hybrid attention" and section 4 "results": LLaMA-3-8B / Mistral-7B teachers,
contexts up to 64K, generation at 32K) with synthetic values:
q, k, v ~ N(0, 1) with q and k multiplied by 1/sqrt(d); Wf ~ N(0, 1/d);
t_m ~ N(0, 1); gate logits from a per-workload normal (or mixture).
Draw order from one numpy PCG64 stream: q, k, v, g, Wf, t, then dy.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    L: int
    Hq: int
    Hkv: int
    d: int
    D: int
    w: int
    M: int
    dtype: str  # "f32" or "bf16"
    gate: tuple  # ("normal", mu, sigma) or ("mix", p1, mu1, s1, mu2, s2)
    seed: int
    chunk: int = 64
    scale_qk: bool = True       # multiply q, k by 1/sqrt(d) at generation
    wf_std: float | None = None  # default 1/sqrt(d)
    prefill: int = 0            # decode workloads: context length before decoding
    steps: int = 0              # decode workloads: number of single-token steps

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads.  Seed = workload index - 1.
TINY_F32 = Workload("tiny_f32_B1_H2_L256_d64", B=1, L=256, Hq=2, Hkv=2, d=64, D=64, w=32, M=4,
                    dtype="f32", gate=("normal", 2.0, 1.0), seed=0)
LLAMA3_8B_L8K = Workload("llama3_8b_fwd_B1_L8192_Hq32_Hkv8_d128_w64", B=1, L=8192, Hq=32, Hkv=8,
                         d=128, D=128, w=64, M=4, dtype="bf16", gate=("normal", 3.0, 1.5), seed=1)
STRESS_L64K = Workload("stress_fwd_B1_L65536_Hq32_Hkv8_d128_w64", B=1, L=65536, Hq=32, Hkv=8,
                       d=128, D=128, w=64, M=4, dtype="bf16",
                       gate=("mix", 0.7, 4.0, 1.0, -3.0, 1.0), seed=2)
MISTRAL_7B_TRAIN = Workload("mistral7b_train_B8_L2048_Hq32_Hkv8_d128_w64", B=8, L=2048, Hq=32,
                            Hkv=8, d=128, D=128, w=64, M=4, dtype="bf16",
                            gate=("normal", 2.0, 1.0), seed=3)
DECODE_B64 = Workload("decode_B64_Hq32_Hkv8_d128_ctx32768_steps1024", B=64, L=1, Hq=32, Hkv=8,
                      d=128, D=128, w=64, M=4, dtype="bf16", gate=("normal", 3.0, 1.5), seed=4,
                      prefill=32768, steps=1024)

WORKLOADS = [TINY_F32, LLAMA3_8B_L8K, STRESS_L64K, MISTRAL_7B_TRAIN, DECODE_B64]


def gla_sensitive(wl: Workload) -> Workload:
    """Variant whose gated-linear term dominates the output.

    With the stated inputs the state term is about 1 % of the shared
    denominator, so a fault in it would hide under a bf16 tolerance.  Slow gates
    (logits ~ N(8, 1)) let the state hold thousands of tokens and Wf ~ N(0, 1)
    makes phi peaked; the state then carries 15-30 % of the denominator.
    """
    return wl.replace(name=wl.name + "_glasens", gate=("normal", 8.0, 1.0), wf_std=1.0)


def closed_gates(wl: Workload, per_1k: float = 2.0) -> Workload:
    """Variant whose gate logits hold runs of strongly closed gates.

    The Lizard summary (sec. 2-C) builds its chunk algorithm around cumulative gate
    products that underflow.  Here the workload's gate stream is broken, about per_1k
    times per 1000 tokens of each (batch, KV head), by a run of 16 to 48 consecutive tokens
    whose logits are N(-12, 1) (a quarter of the runs: N(-30, 1)), on every feature or on a
    random half of them.  Such a run closes the gates: 16 tokens at -12 decay the state by
    about e^-190.
    """
    return wl.replace(name=wl.name + "_closed", gate=("runs", wl.gate, per_1k, 16, 48, 0.25))


def round_to(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp32 values to the storage dtype and return them as fp32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    if dtype == "f32":
        return a
    if dtype == "bf16":
        # round to nearest even on the upper 16 bits (inputs are finite)
        u = a.view(np.uint32).astype(np.uint64)
        lsb = (u >> 16) & 1
        u = (u + 0x7FFF + lsb) >> 16
        return (u.astype(np.uint32) << 16).view(np.float32).reshape(a.shape)
    raise ValueError(dtype)


def _gates(rng: np.random.Generator, shape, spec) -> np.ndarray:
    if spec[0] == "normal":
        _, mu, sd = spec
        return (mu + sd * rng.standard_normal(shape, dtype=np.float32)).astype(np.float32)
    if spec[0] == "mix":
        _, p1, mu1, s1, mu2, s2 = spec
        a = rng.standard_normal(shape, dtype=np.float32)
        u = rng.random(shape, dtype=np.float32)
        first = u < p1
        return np.where(first, mu1 + s1 * a, mu2 + s2 * a).astype(np.float32)
    if spec[0] == "runs":
        _, base, per_1k, lo, hi, p_deep = spec
        out = _gates(rng, shape, base)
        B, L, H, D = shape
        nrun = max(1, int(round(L * per_1k / 1000.0)))
        for b in range(B):
            for h in range(H):
                starts = rng.integers(0, L, size=nrun)
                lens = rng.integers(lo, hi + 1, size=nrun)
                deep = rng.random(nrun) < p_deep
                every = rng.random(nrun) < 0.5
                for s0, n, dp, ev in zip(starts, lens, deep, every):
                    feats = np.arange(D) if ev else np.sort(rng.permutation(D)[: D // 2])
                    e = min(L, int(s0) + int(n))
                    vals = rng.standard_normal((e - int(s0), len(feats)), dtype=np.float32)
                    view = out[b, int(s0):e, h]
                    view[:, feats] = (-30.0 if dp else -12.0) + vals
        return out
    raise ValueError(spec)


def make_inputs(wl: Workload, L: int | None = None, B: int | None = None,
                with_dy: bool = False) -> dict:
    """Draw one workload's inputs on the host as fp32 arrays already rounded to wl.dtype.

    L and B override the workload's sizes (parity cases at reduced length).
    """
    L = wl.L if L is None else L
    B = wl.B if B is None else B
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    s = wl.scale if wl.scale_qk else 1.0
    wf_std = (1.0 / math.sqrt(wl.d)) if wl.wf_std is None else wl.wf_std
    q = rng.standard_normal((B, L, wl.Hq, wl.d), dtype=np.float32) * np.float32(s)
    k = rng.standard_normal((B, L, wl.Hkv, wl.d), dtype=np.float32) * np.float32(s)
    v = rng.standard_normal((B, L, wl.Hkv, wl.d), dtype=np.float32)
    g = _gates(rng, (B, L, wl.Hkv, wl.D), wl.gate)
    Wf = rng.standard_normal((wl.Hkv, wl.d, wl.D // 2), dtype=np.float32) * np.float32(wf_std)
    sinks = rng.standard_normal((wl.Hq, wl.M), dtype=np.float32)
    out = dict(q=q, k=k, v=v, g=g, Wf=Wf)
    out = {n: round_to(a, wl.dtype) for n, a in out.items()}
    out["sinks"] = np.ascontiguousarray(sinks, dtype=np.float32)
    if with_dy:
        dy = rng.standard_normal((B, L, wl.Hq, wl.d), dtype=np.float32)
        out["dy"] = round_to(dy, wl.dtype)
    return out


def make_proj_inputs(wl: Workload, dm: int, L: int | None = None, B: int | None = None,
                     with_grads: bool = False, seed_offset: int = 100) -> dict:
    """Inputs of the projections in front of the mixer: the layer input x [B, L, dm] ~ N(0, 1)
    and the stacked weight W [N, dm] ~ N(0, 1/dm), N = Hq d + 2 Hkv d + Hkv D (rows q, k, v,
    gate), rounded to the workload's dtype; optionally upstream gradients dq, dk, dv, dg ~
    N(0, 1).  Own stream: seed = 1000 * (workload seed + seed_offset)."""
    L = wl.L if L is None else L
    B = wl.B if B is None else B
    rng = np.random.Generator(np.random.PCG64(1000 * (wl.seed + seed_offset)))
    N = wl.Hq * wl.d + 2 * wl.Hkv * wl.d + wl.Hkv * wl.D
    x = rng.standard_normal((B, L, dm), dtype=np.float32)
    W = rng.standard_normal((N, dm), dtype=np.float32) * np.float32(1.0 / math.sqrt(dm))
    out = {"x": round_to(x, wl.dtype), "W": round_to(W, wl.dtype)}
    if with_grads:
        for n, h, e in (("dq", wl.Hq, wl.d), ("dk", wl.Hkv, wl.d), ("dv", wl.Hkv, wl.d),
                        ("dg", wl.Hkv, wl.D)):
            out[n] = round_to(rng.standard_normal((B, L, h, e), dtype=np.float32), wl.dtype)
    return out


def make_decode_inputs(wl: Workload, batch_index: int, T: int) -> dict:
    """Inputs of one sequence of a decode workload: T = prefill + steps tokens.

    Each sequence b has its own stream (seed = 1000 * wl.seed + b) so that a
    sampled subset of the batch can be regenerated on the host alone.
    Wf and sinks are shared by the batch and come from the workload seed.
    """
    rng = np.random.Generator(np.random.PCG64(1000 * wl.seed + batch_index))
    s = wl.scale if wl.scale_qk else 1.0
    q = rng.standard_normal((1, T, wl.Hq, wl.d), dtype=np.float32) * np.float32(s)
    k = rng.standard_normal((1, T, wl.Hkv, wl.d), dtype=np.float32) * np.float32(s)
    v = rng.standard_normal((1, T, wl.Hkv, wl.d), dtype=np.float32)
    g = _gates(rng, (1, T, wl.Hkv, wl.D), wl.gate)
    out = dict(q=q, k=k, v=v, g=g)
    return {n: round_to(a, wl.dtype) for n, a in out.items()}


def make_shared_params(wl: Workload) -> dict:
    """Wf and sinks of a decode workload (shared by all sequences of the batch)."""
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    wf_std = (1.0 / math.sqrt(wl.d)) if wl.wf_std is None else wl.wf_std
    Wf = rng.standard_normal((wl.Hkv, wl.d, wl.D // 2), dtype=np.float32) * np.float32(wf_std)
    sinks = rng.standard_normal((wl.Hq, wl.M), dtype=np.float32)
    return dict(Wf=round_to(Wf, wl.dtype), sinks=np.ascontiguousarray(sinks, np.float32))


def varlen_lengths(n: int = 64, lo: int = 128, hi: int = 4096, seed: int = 5) -> list:
    """Lengths of a packed serving batch: n sequences, lengths uniform on [lo, hi] (seeded)."""
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)]


def make_device_inputs(wl: Workload, device, L: int | None = None, B: int | None = None,
                       with_dy: bool = False, seed_offset: int = 0) -> dict:
    """Same laws as make_inputs, drawn on the device with torch's Philox generator.

    For throughput runs whose sizes make host generation slow.  The values are
    not the host stream's values; parity cases use make_inputs.
    """
    import torch

    L = wl.L if L is None else L
    B = wl.B if B is None else B
    gen = torch.Generator(device=device)
    gen.manual_seed(10007 * (wl.seed + 1) + seed_offset)
    tdt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    s = wl.scale if wl.scale_qk else 1.0
    wf_std = (1.0 / math.sqrt(wl.d)) if wl.wf_std is None else wl.wf_std

    def randn(*shape, mul=1.0, add=0.0):
        x = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
        if mul != 1.0:
            x.mul_(mul)
        if add != 0.0:
            x.add_(add)
        return x.to(tdt)

    out = {}
    out["q"] = randn(B, L, wl.Hq, wl.d, mul=s)
    out["k"] = randn(B, L, wl.Hkv, wl.d, mul=s)
    out["v"] = randn(B, L, wl.Hkv, wl.d)
    if wl.gate[0] == "normal":
        out["g"] = randn(B, L, wl.Hkv, wl.D, mul=wl.gate[2], add=wl.gate[1])
    else:
        _, p1, mu1, s1, mu2, s2 = wl.gate
        a = torch.randn(B, L, wl.Hkv, wl.D, generator=gen, device=device)
        u = torch.rand(B, L, wl.Hkv, wl.D, generator=gen, device=device)
        out["g"] = torch.where(u < p1, mu1 + s1 * a, mu2 + s2 * a).to(tdt)
        del a, u
    out["Wf"] = randn(wl.Hkv, wl.d, wl.D // 2, mul=wf_std)
    out["sinks"] = torch.randn(wl.Hq, wl.M, generator=gen, device=device, dtype=torch.float32)
    if with_dy:
        out["dy"] = randn(B, L, wl.Hq, wl.d)
    return out
