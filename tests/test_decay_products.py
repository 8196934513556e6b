"""The decay factors of the tensor-core segment passes are products of Gamma = sigmoid(g)
formed in fp32 rather than exponentials of summed log-sigmoids (Lizard summary, gist.science
2507.09025, sec. 2-C folds the gates in log space).  Emulated on the host in fp32 and compared
with fp64 log space, on the long-context stress gate mixture where products fall far below one:
the factors agree to fp32 accuracy wherever they are not negligible, and the log-decay taken
from quarter products renormalised every 4 tokens matches the sum of log-sigmoids."""
import numpy as np

from gated_linear_sliding_gb300 import inputs as I


def _gates(n_tok=128, n_f=128, seed=7):
    """One 128-token step of gate logits drawn by the workload generator's own law."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return I._gates(rng, (n_tok, n_f), I.STRESS_L64K.gate).astype(np.float32)


def _suffix_products_fp32(g):
    """e^{b_end - b_t} per token as the segment pass forms it: suffix products inside 32-token
    quarters times the later quarters' products, all in fp32."""
    gam = (1.0 / (1.0 + np.exp(-g.astype(np.float32)))).astype(np.float32)
    T = g.shape[0]
    out = np.empty_like(gam)
    quarters = [(q, min(T, q + 32)) for q in range(0, T, 32)]
    qprod = []
    for a, b in quarters:
        sp = np.ones(g.shape[1], np.float32)
        for t in range(b - 1, a - 1, -1):
            out[t] = sp
            sp = (sp * gam[t]).astype(np.float32)
        qprod.append(sp)
    for qi, (a, b) in enumerate(quarters):
        later = np.ones(g.shape[1], np.float32)
        for qj in range(qi + 1, len(quarters)):
            later = (later * qprod[qj]).astype(np.float32)
        out[a:b] = (out[a:b] * later).astype(np.float32)
    return out, gam


def _log_decay_renormalised(gam):
    """Sum over tokens of log Gamma from products renormalised every 4 tokens (frexp)."""
    m = np.ones(gam.shape[1], np.float32)
    e = np.zeros(gam.shape[1], np.int64)
    for t in range(gam.shape[0]):
        m = (m * gam[t]).astype(np.float32)
        if t % 4 == 3:
            mant, ex = np.frexp(m)
            m, e = mant.astype(np.float32), e + ex
    return np.log2(m.astype(np.float64)) * np.log(2.0) + e * np.log(2.0)


def test_suffix_products_match_log_space():
    g = _gates()
    got, _ = _suffix_products_fp32(g)
    lam = -np.logaddexp(0.0, -g.astype(np.float64))          # log sigmoid, fp64
    b = np.cumsum(lam, axis=0)
    ref = np.exp(b[-1][None, :] - b)                          # e^{b_end - b_t}
    big = ref > 1e-30                                         # factors that matter
    rel = np.abs(got[big] - ref[big]) / ref[big]
    assert rel.max() < 2e-5, rel.max()
    # where the exact factor is negligible the product is negligible too (or zero)
    assert np.all(got[~big] < 1e-29)


def test_renormalised_log_decay_matches_sum_of_log_sigmoids():
    g = _gates()
    _, gam = _suffix_products_fp32(g)
    ref = (-np.logaddexp(0.0, -g.astype(np.float64))).sum(axis=0)
    got = _log_decay_renormalised(gam)
    assert np.all(np.isfinite(got))
    assert np.abs(got - ref).max() < 1e-3 * np.abs(ref).max()
    # without renormalisation the fp32 product of 128 strong gates underflows
    plain = np.prod(gam.astype(np.float32), axis=0, dtype=np.float32)
    assert (plain == 0).any()
