"""Plants plausible mistakes in copies of the oracle's C source and checks that
the pins catch every one (no GPU).  Each mutant is one textual change: a
dropped term, a flipped sign, a wrong operand or a wrong order."""
import json
import os
import shutil
import tempfile

import numpy as np
import pytest

import gdn_synth
import oracle
from oracle import build as obuild
from oracle import chunked

MUTANTS = [
    ("r[j] -= row[j] * ki;", "r[j] += row[j] * ki;"),
    ("H[i] *= alpha;", "H[i] *= 1.0;"),
    ("ot[j] *= scale;", "ot[j] *= 1.0;"),
    ("const double bk = beta * kt[i];", "const double bk = kt[i];"),
    ("step_forward(H, K, V, exp(p->g[th]), p->beta[th], kt, p->v + th * V, r);\n"
     "        if (p->o) output_row(H, K, V, p->scale, qt, p->o + th * V);",
     "if (p->o) output_row(H, K, V, p->scale, qt, p->o + th * V);\n"
     "        step_forward(H, K, V, exp(p->g[th]), p->beta[th], kt, p->v + th * V, r);"),
    ("dg += dhb * Hbar[ij];", "dg += dH[ij] * Hbar[ij];"),
    ("dkh[i] -= s;", "dkh[i] += s;"),
    ("dH[ij] = alpha * dhb;", "dH[ij] = dhb;"),
    ("for (int j = 0; j < V; ++j) dr[j] *= beta;", ""),
    ("dq_out[i] = (dqh[i] - qt[i] * pq) * sq;", "dq_out[i] = dqh[i] * sq;"),
    ("dk_out[i] = (dkh[i] - kt[i] * pk) * sk;", "dk_out[i] = (dkh[i] - kt[i] * pk);"),
    ("s = 1.0 / sqrt(ss + eps);", "s = 1.0 / sqrt(ss);"),
    ("s += Ht[(long)i * V + j] * dot[j];", "s += Hbar[(long)i * V + j] * dot[j];"),
    ("dbeta += kt[i] * s;", "dbeta += s;"),
    ("dH[(long)i * V + j] += p->scale * qt[i] * dot[j];", "dH[(long)i * V + j] += qt[i] * dot[j];"),
    ("const long th = (bos + t) * Hh + h;\n            const double *Hprev",
     "const long th = (bos + t) * Hh + (Hh - 1 - h);\n            const double *Hprev"),
    # gate preprocessing
    ("return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));", "return x > 0.0 ? x : log1p(exp(x));"),
    ("dx[t * Hh + h] = -a[h] * d / (1.0 + exp(-xv));", "dx[t * Hh + h] = a[h] * d / (1.0 + exp(-xv));"),
    ("/ (1.0 + exp(-xv));", "/ (1.0 + exp(xv));"),
    ("acc -= d * softplus(xv);", "acc -= d * xv;"),
    ("g[t * Hh + h] = -a[h] * softplus(x[t * Hh + h]);", "g[t * Hh + h] = -softplus(x[t * Hh + h]);"),
]


def _hand(lib):
    ex = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "hand_worked_T3_K2_V2.json")))
    a = [np.array(ex[n])[None, :, None] for n in ("q", "k", "v")]
    o, ht = oracle.fwd(*a, np.log(np.array(ex["alpha"]))[None, :, None],
                       np.array(ex["beta"])[None, :, None], h0=np.array(ex["h0"])[None, None],
                       scale=ex["scale"], lib=lib)
    return np.allclose(o[0, :, 0], ex["o"], atol=1e-12) and np.allclose(ht[0, 0], ex["hT"],
                                                                        atol=1e-12)


def _chunked(lib, l2):
    pr = gdn_synth.make("tiny", T=40, K=6, V=5, H=2, h0_std=0.3, normalise=not l2)
    a = [x.double() for x in (pr.q, pr.k, pr.v, pr.g, pr.beta)]
    o, ht = oracle.fwd(*a, h0=pr.h0, use_l2norm=l2, lib=lib)
    oc, hc = chunked.forward(*a, h0=pr.h0.double(), C=16, use_l2norm=l2)
    return np.allclose(oc.numpy(), o, atol=1e-11) and np.allclose(hc.numpy(), ht, atol=1e-11)


def _eps(lib):
    q = np.zeros((1, 1, 1, 3))
    q[..., 1] = 1e-3
    h0 = np.arange(6.0).reshape(1, 1, 3, 2)
    o, _ = oracle.fwd(q, np.ones((1, 1, 1, 3)), np.zeros((1, 1, 1, 2)), np.zeros((1, 1, 1)),
                      np.zeros((1, 1, 1)), h0=h0, scale=1.0, use_l2norm=True, eps=1e-6, lib=lib)
    return np.allclose(o[0, 0, 0], h0[0, 0, 1] * 1e-3 / np.sqrt(2e-6), rtol=1e-12)


def _fd(lib, l2):
    r = np.random.default_rng(31)
    p = dict(q=r.standard_normal((1, 4, 2, 3)), k=r.standard_normal((1, 4, 2, 3)),
             v=r.standard_normal((1, 4, 2, 2)), g=-r.uniform(0.1, 0.5, (1, 4, 2)),
             beta=r.uniform(0.2, 0.8, (1, 4, 2)), h0=r.standard_normal((1, 2, 3, 2)))
    do, dht = r.standard_normal((1, 4, 2, 2)), r.standard_normal((1, 2, 3, 2))
    kw = dict(scale=0.7, use_l2norm=l2, lib=lib)
    d = oracle.bwd(**p, do=do, dht=dht, **kw)

    def loss():
        o, ht = oracle.fwd(**p, **kw)
        return float((o * do).sum() + (ht * dht).sum())

    for name, gname in dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", h0="dh0").items():
        x = p[name]
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + 1e-6
            lp = loss()
            x[idx] = old - 1e-6
            lm = loss()
            x[idx] = old
            if abs((lp - lm) / 2e-6 - d[gname][idx]) > 1e-6 * max(1.0, abs(d[gname][idx])):
                return False
    return True


def _gate(lib):
    # closed forms: softplus(0) = ln 2; a = 0 gives no decay; very negative logits none either
    g0 = oracle.gate(np.zeros((2, 3)), np.array([0.5, 1.0, 2.0]), lib=lib)
    if not np.allclose(g0, -np.array([0.5, 1.0, 2.0]) * np.log(2.0), rtol=1e-14):
        return False
    r = np.random.default_rng(7)
    x, a = 4.0 * r.standard_normal((5, 3)), r.uniform(0.1, 2.0, 3)
    if np.any(oracle.gate(x, np.zeros(3), lib=lib) != 0.0):
        return False
    if not np.allclose(oracle.gate(x + 40.0, a, lib=lib), -a * (x + 40.0), rtol=1e-12):
        return False
    # the backward against central differences of the forward
    dg = r.standard_normal(x.shape)
    dx, da = oracle.gate_bwd(x, a, dg, lib=lib)

    def loss(xx, aa):
        return float((oracle.gate(xx, aa, lib=lib) * dg).sum())

    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += 1e-6
        xm[idx] -= 1e-6
        if abs((loss(xp, a) - loss(xm, a)) / 2e-6 - dx[idx]) > 1e-7 * max(1.0, abs(dx[idx])):
            return False
    for h in range(3):
        ap, am = a.copy(), a.copy()
        ap[h] += 1e-6
        am[h] -= 1e-6
        if abs((loss(x, ap) - loss(x, am)) / 2e-6 - da[h]) > 1e-7 * max(1.0, abs(da[h])):
            return False
    return True


def pins_pass(lib):
    return (_hand(lib) and _chunked(lib, False) and _chunked(lib, True) and _eps(lib)
            and _fd(lib, False) and _fd(lib, True) and _gate(lib))


def test_unmutated_oracle_passes_the_quick_pins():
    assert pins_pass(oracle.open_library(obuild.build()))


@pytest.mark.parametrize("i", range(len(MUTANTS)))
def test_every_planted_mistake_is_caught(i):
    old, new = MUTANTS[i]
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    tmp = tempfile.mkdtemp()
    try:
        path = os.path.join(tmp, "mutant.c")
        open(path, "w").write(src.replace(old, new))
        lib = oracle.open_library(obuild.build(force=True, src=path,
                                               out=os.path.join(tmp, "libmutant.so")))
        assert not pins_pass(lib), f"mutant survived: {old!r} -> {new!r}"
    finally:
        shutil.rmtree(tmp)
