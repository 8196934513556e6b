"""Alternate float64 forms of the Lizard token mixer, used to pin the recurrent oracle.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

All forms compute the same y (Lizard summary, gist.science/ko/paper/2507.09025,
sec. 2-A-1 and 2-A-2, with one shared normaliser): a key j that has left the
window (j <= i - w) reaches query i through the state with the per-feature
weight

    phi(k_j)_f * prod_{s=j+w+1..i} Gamma_{s,f},      Gamma = sigmoid(g),

(the delayed-key reading; `brute_force` and `quadratic_parallel` also take the
masked reading, product over s = j+1..i, and the lagged reading, s = j+1..i-w)

and a key inside the window (i - w < j <= i) with e^{scale q_i.k_j}; the
meta-memory scalars add sum_m e^{t_m} to the denominator only.

  brute_force        pure Python loops, products written out term by term (tiny L)
  quadratic_parallel the L x L weight matrix at once (numpy), reverse cumprods
  chunked_cumprod    chunks of C tokens, inter-chunk state, explicit products
  chunked_logspace   the same chunks with gates in log space (sec. 2-C: the
                     gate terms move to log space; decays become exp of
                     differences of cumulative log-gates)
"""
from __future__ import annotations

import math

import numpy as np


def phi(x: np.ndarray, Wf_kv: np.ndarray) -> np.ndarray:
    """Hedgehog map [softmax(x Wf), softmax(-x Wf)] over the last axis (fp64)."""
    u = np.asarray(x, np.float64) @ np.asarray(Wf_kv, np.float64)

    def sm(a):
        a = a - a.max(axis=-1, keepdims=True)
        e = np.exp(a)
        return e / e.sum(axis=-1, keepdims=True)

    return np.concatenate([sm(u), sm(-u)], axis=-1)


def gate_range(reading: int, i: int, j: int, w: int) -> tuple[int, int]:
    """First and last s of the gate product that weighs key j <= i - w at query i:
    0 delayed key (j+w+1 .. i), 1 masked full GLA (j+1 .. i), 2 lagged state (j+1 .. i-w).
    An empty range (first > last) is the product 1."""
    if reading == 0:
        return j + w + 1, i
    if reading == 1:
        return j + 1, i
    if reading == 2:
        return j + 1, i - w
    raise ValueError(f"unknown reading {reading}")


def _unpack(inp):
    q, k, v, g, Wf, sinks = (np.asarray(inp[n], np.float64)
                             for n in ("q", "k", "v", "g", "Wf", "sinks"))
    return q, k, v, g, Wf, sinks


def brute_force(inp: dict, w: int, scale: float | None = None, reading: int = 0) -> np.ndarray:
    """Output y by the weight definition, one scalar product at a time (L <= 16)."""
    q, k, v, g, Wf, sinks = _unpack(inp)
    B, L, Hq, d = q.shape
    Hkv, D = k.shape[2], g.shape[3]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    y = np.zeros_like(q)
    for b in range(B):
        for h in range(Hq):
            kv = h // G
            for i in range(L):
                pq = phi(q[b, i, h], Wf[kv])
                num = [0.0] * d
                den = 0.0
                for j in range(0, i - w + 1):
                    pk = phi(k[b, j, kv], Wf[kv])
                    a = 0.0
                    lo, hi = gate_range(reading, i, j, w)
                    for f in range(D):
                        prod = 1.0
                        for s in range(lo, hi + 1):
                            prod *= 1.0 / (1.0 + math.exp(-g[b, s, kv, f]))
                        a += pq[f] * pk[f] * prod
                    for c in range(d):
                        num[c] += a * v[b, j, kv, c]
                    den += a
                for j in range(max(0, i - w + 1), i + 1):
                    s_ = 0.0
                    for c in range(d):
                        s_ += q[b, i, h, c] * k[b, j, kv, c]
                    e = math.exp(scale * s_)
                    for c in range(d):
                        num[c] += e * v[b, j, kv, c]
                    den += e
                for m in range(sinks.shape[1]):
                    den += math.exp(sinks[h, m])
                for c in range(d):
                    y[b, i, h, c] = num[c] / den
    return y


def quadratic_parallel(inp: dict, w: int, scale: float | None = None,
                       reading: int = 0) -> np.ndarray:
    """Output y from the full L x L weight matrices (gated-linear part and window part)."""
    q, k, v, g, Wf, sinks = _unpack(inp)
    B, L, Hq, d = q.shape
    Hkv, D = k.shape[2], g.shape[3]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    gam = 1.0 / (1.0 + np.exp(-g))
    y = np.zeros_like(q)
    ii = np.arange(L)[:, None]
    jj = np.arange(L)[None, :]
    win = (jj <= ii) & (jj > ii - w)
    for b in range(B):
        for kv in range(Hkv):
            pk = phi(k[b, :, kv], Wf[kv])                       # [L, D]
            # decay[i, j, f] = prod_{s=lo..hi} Gamma_s,f for j <= i-w (gate_range)
            decay = np.zeros((L, L, D))
            for i in range(w, L):
                for j in range(0, i - w + 1):
                    lo, hi = gate_range(reading, i, j, w)
                    decay[i, j] = np.prod(gam[b, lo:hi + 1, kv], axis=0)  # 1 when empty
            for hh in range(G):
                h = kv * G + hh
                pq = phi(q[b, :, h], Wf[kv])                   # [L, D]
                A = np.einsum("if,jf,ijf->ij", pq, pk, decay)
                s = scale * (q[b, :, h] @ k[b, :, kv].T)
                A = A + np.where(win, np.exp(np.where(win, s, 0.0)), 0.0)
                num = A @ v[b, :, kv]
                den = A.sum(axis=1) + np.exp(sinks[h]).sum()
                y[b, :, h] = num / den[:, None]
    return y


def _window_parts(qh, kk, vv, w, scale, i0, i1):
    """Window numerator/denominator for queries i0..i1-1 (keys (i-w, i])."""
    n = i1 - i0
    d = vv.shape[1]
    num = np.zeros((n, d))
    den = np.zeros(n)
    for r, i in enumerate(range(i0, i1)):
        j0 = max(0, i - w + 1)
        e = np.exp(scale * (kk[j0:i + 1] @ qh[i]))
        num[r] = e @ vv[j0:i + 1]
        den[r] = e.sum()
    return num, den


def _chunked(inp: dict, w: int, C: int, scale, logspace: bool) -> np.ndarray:
    q, k, v, g, Wf, sinks = _unpack(inp)
    B, L, Hq, d = q.shape
    Hkv, D = k.shape[2], g.shape[3]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    y = np.zeros_like(q)
    for b in range(B):
        for kv in range(Hkv):
            # delayed stream: token t of the state stream carries key t-w
            pk = phi(k[b, :, kv], Wf[kv])
            pkd = np.zeros((L, D))
            vd = np.zeros((L, d))
            if L > w:
                pkd[w:] = pk[:L - w]
                vd[w:] = v[b, :L - w, kv]
            gam = 1.0 / (1.0 + np.exp(-g[b, :, kv]))          # [L, D]
            lam = -np.logaddexp(0.0, -g[b, :, kv])            # log sigmoid, [L, D]
            H = np.zeros((D, d))
            z = np.zeros(D)
            pqs = [phi(q[b, :, kv * G + hh], Wf[kv]) for hh in range(G)]
            for t0 in range(0, L, C):
                t1 = min(L, t0 + C)
                n = t1 - t0
                if logspace:
                    bl = np.cumsum(lam[t0:t1], axis=0)          # chunk-local, inclusive
                    dq_ = np.exp(bl)                             # decay chunk start -> i
                    lower = (np.arange(n)[:, None] >= np.arange(n)[None, :])[:, :, None]
                    # i, t -> e^{b_i - b_t} for t <= i (the upper triangle is masked out)
                    dqk = np.exp(np.where(lower, bl[:, None, :] - bl[None, :, :], -np.inf))
                    dlast = np.exp(bl[-1][None, :] - bl)        # t -> e^{b_last - b_t}
                    dtot = np.exp(bl[-1])
                else:
                    dq_ = np.cumprod(gam[t0:t1], axis=0)
                    dqk = np.ones((n, n, D))
                    for i in range(n):
                        rc = np.cumprod(gam[t0 + i:t0:-1], axis=0) if i > 0 else None
                        # rc[m] = prod_{s=t0+i-m .. t0+i}; decay i<-t = prod_{s=t+1..i}
                        for t in range(i):
                            dqk[i, t] = rc[i - t - 1]
                    dlast = np.ones((n, D))
                    rcl = np.cumprod(gam[t1 - 1:t0:-1], axis=0)
                    for t in range(n - 1):
                        dlast[t] = rcl[n - 2 - t]
                    dtot = dq_[-1]
                causal = np.tril(np.ones((n, n)))
                for hh in range(G):
                    h = kv * G + hh
                    pq = pqs[hh][t0:t1]
                    qt = pq * dq_
                    num = qt @ H
                    den = qt @ z
                    A = np.einsum("if,tf,itf->it", pq, pkd[t0:t1], dqk) * causal
                    num = num + A @ vd[t0:t1]
                    den = den + A.sum(axis=1)
                    nw, dw = _window_parts(q[b, :, h], k[b, :, kv], v[b, :, kv], w, scale,
                                           t0, t1)
                    den = den + dw + np.exp(sinks[h]).sum()
                    y[b, t0:t1, h] = (num + nw) / den[:, None]
                kt = pkd[t0:t1] * dlast
                H = dtot[:, None] * H + kt.T @ vd[t0:t1]
                z = dtot * z + kt.sum(axis=0)
    return y


def chunked_cumprod(inp: dict, w: int, C: int = 64, scale: float | None = None) -> np.ndarray:
    """Chunked form with decays as explicit products of gates."""
    return _chunked(inp, w, C, scale, logspace=False)


def chunked_logspace(inp: dict, w: int, C: int = 64, scale: float | None = None) -> np.ndarray:
    """Chunked form with decays as exp of differences of chunk-local cumulative log-gates."""
    return _chunked(inp, w, C, scale, logspace=True)
