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


def pins_pass(lib):
    return (_hand(lib) and _chunked(lib, False) and _chunked(lib, True) and _eps(lib)
            and _fd(lib, False) and _fd(lib, True))


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
