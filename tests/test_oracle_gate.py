"""Pins of the oracle's gate preprocessing (no GPU).

The log decay comes from a raw gate logit x and a positive per-head scale
a_h as g = -a_h softplus(x) (the pages' "gate preprocessing", aivizor,
FLA-flow paragraph; the form is the GDN layer's decay gate).  The pins:
closed forms of softplus, and the gradients of the whole gated recurrence
(gate, then the sequential recurrence, then a scalar loss) against central
finite differences with respect to the logits and the scales.
"""
import numpy as np

import oracle


def test_softplus_closed_forms():
    a = np.array([0.25, 1.0, 3.0])
    assert np.allclose(oracle.gate(np.zeros((1, 3)), a), -a * np.log(2.0), rtol=1e-15)
    big = np.full((1, 3), 60.0)                   # softplus(x) = x + e^-x + ...
    assert np.allclose(oracle.gate(big, a), -a * 60.0, rtol=1e-15)
    small = np.full((1, 3), -60.0)                # softplus(x) = e^x + ...
    assert np.allclose(oracle.gate(small, a), -a * np.exp(-60.0), rtol=1e-12)


def test_gated_recurrence_gradients_match_central_differences():
    r = np.random.default_rng(5)
    B, T, H, K, V = 1, 6, 2, 3, 2
    q, k = r.standard_normal((B, T, H, K)), r.standard_normal((B, T, H, K))
    v, beta = r.standard_normal((B, T, H, V)), r.uniform(0.2, 0.8, (B, T, H))
    x, a = r.standard_normal((B, T, H)), r.uniform(0.2, 1.5, H)
    h0 = r.standard_normal((B, H, K, V))
    do, dht = r.standard_normal((B, T, H, V)), r.standard_normal((B, H, K, V))

    def loss(xx, aa):
        o, ht = oracle.fwd(q, k, v, oracle.gate(xx, aa), beta, h0=h0)
        return float((o * do).sum() + (ht * dht).sum())

    g = oracle.gate(x, a)
    dg = oracle.bwd(q, k, v, g, beta, do=do, h0=h0, dht=dht)["dg"]
    dx, da = oracle.gate_bwd(x, a, dg)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += 1e-6
        xm[idx] -= 1e-6
        fd = (loss(xp, a) - loss(xm, a)) / 2e-6
        assert abs(fd - dx[idx]) <= 1e-6 * max(1.0, abs(dx[idx]))
    for h in range(H):
        ap, am = a.copy(), a.copy()
        ap[h] += 1e-6
        am[h] -= 1e-6
        fd = (loss(x, ap) - loss(x, am)) / 2e-6
        assert abs(fd - da[h]) <= 1e-6 * max(1.0, abs(da[h]))
