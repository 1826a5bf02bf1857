"""Pins for the fp64 CPU oracle (no GPU).

The pages print no formula and no worked example, so the oracle is pinned to
things other than itself:
  * a three-step example worked by hand (tests/golden/);
  * closed forms: beta = 0 (pure decay of the initial state, forward and
    every gradient), g = 0 with beta = 0 (identity), g = 0 with beta = 1 and
    orthonormal keys (exact key -> value overwrite and retrieval);
  * an independent chunk-wise restatement (oracle/chunked.py) for chunk sizes
    1, 16, 64 and T, with a partial last chunk;
  * central finite differences of the oracle's own forward for every
    gradient, and torch autograd through the chunk-wise form;
  * invariants: varlen == separate runs, state continuation (forward and
    backward hand-over), joint linearity in (v, h0), unit subsets.
"""
import json
import os

import numpy as np
import pytest
import torch

import gdn_synth
import oracle
from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_problem(seed, B=1, T=9, H=2, K=4, V=3, h0=True, unit_keys=True):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, T, H, K))
    k = r.standard_normal((B, T, H, K))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((B, T, H, V))
    g = -r.uniform(0.05, 0.8, (B, T, H))
    beta = r.uniform(0.1, 0.9, (B, T, H))
    hh = r.standard_normal((B, H, K, V)) * 0.5 if h0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=hh)


# ---------------------------------------------------------------- hand example
def test_hand_worked_example():
    ex = json.load(open(os.path.join(GOLDEN, "hand_worked_T3_K2_V2.json")))
    q = np.array(ex["q"])[None, :, None, :]
    k = np.array(ex["k"])[None, :, None, :]
    v = np.array(ex["v"])[None, :, None, :]
    g = np.log(np.array(ex["alpha"]))[None, :, None]
    beta = np.array(ex["beta"])[None, :, None]
    h0 = np.array(ex["h0"])[None, None]
    o, ht = oracle.fwd(q, k, v, g, beta, h0=h0, scale=ex["scale"])
    np.testing.assert_allclose(o[0, :, 0], np.array(ex["o"]), atol=1e-14)
    np.testing.assert_allclose(ht[0, 0], np.array(ex["hT"]), atol=1e-14)


# ---------------------------------------------------------------- closed forms
def test_beta_zero_is_pure_decay_forward_and_backward():
    """beta = 0: H_t = e^{gamma_t} H0, o_t = s e^{gamma_t} H0^T q_t, and every
    gradient has a closed form."""
    p = rand_problem(1, T=11, K=5, V=4)
    p["beta"][:] = 0.0
    s = 0.37
    r = np.random.default_rng(2)
    do = r.standard_normal(p["v"].shape)
    dht = r.standard_normal(p["h0"].shape)
    o, ht = oracle.fwd(**p, scale=s)
    gam = np.cumsum(p["g"], axis=1)                             # [B,T,H]
    H0 = p["h0"][0]                                             # [H,K,V]
    o_ref = s * np.exp(gam)[..., None] * np.einsum("hkv,bthk->bthv", H0, p["q"])
    np.testing.assert_allclose(o, o_ref, atol=1e-13)
    np.testing.assert_allclose(ht[0], np.exp(gam[0, -1])[:, None, None] * H0, atol=1e-13)

    d = oracle.bwd(**p, do=do, dht=dht, scale=s)
    T = p["q"].shape[1]
    # dH_t (gradient with respect to the state after token t)
    dH = np.zeros((T,) + H0.shape)
    for t in range(T):
        acc = np.exp(gam[0, -1] - gam[0, t])[:, None, None] * dht[0]
        for u in range(t, T):
            acc = acc + s * np.exp(gam[0, u] - gam[0, t])[:, None, None] * np.einsum(
                "hk,hv->hkv", p["q"][0, u], do[0, u])
        dH[t] = acc
    Ht = np.exp(gam[0])[:, :, None, None] * H0[None]            # [T,H,K,V]
    np.testing.assert_allclose(d["dq"][0], s * np.einsum("thkv,thv->thk", Ht, do[0]), atol=1e-12)
    np.testing.assert_allclose(d["dv"], 0.0, atol=0)
    np.testing.assert_allclose(d["dk"], 0.0, atol=0)
    r_t = p["v"][0] - np.einsum("thkv,thk->thv", Ht, p["k"][0])
    np.testing.assert_allclose(d["dbeta"][0], np.einsum("thk,thkv,thv->th", p["k"][0], dH, r_t),
                               atol=1e-12)
    # L = sum_t s e^{gamma_t} q_t^T H0 do_t + e^{gamma_T} <H0, dht>
    per_tok = s * np.exp(gam[0]) * np.einsum("thk,hkv,thv->th", p["q"][0], H0, do[0])
    tail = np.exp(gam[0, -1]) * np.einsum("hkv,hkv->h", H0, dht[0])
    dg_ref = np.cumsum(per_tok[::-1], axis=0)[::-1] + tail[None]
    np.testing.assert_allclose(d["dg"][0], dg_ref, atol=1e-12)
    dh0_ref = np.exp(gam[0, -1])[:, None, None] * dht[0] + s * np.einsum(
        "th,thk,thv->hkv", np.exp(gam[0]), p["q"][0], do[0])
    np.testing.assert_allclose(d["dh0"][0], dh0_ref, atol=1e-12)


def test_no_decay_no_write_is_identity():
    p = rand_problem(3, T=6)
    p["g"][:] = 0.0
    p["beta"][:] = 0.0
    o, ht = oracle.fwd(**p, scale=0.5)
    np.testing.assert_allclose(ht, p["h0"], atol=0)
    np.testing.assert_allclose(o, 0.5 * np.einsum("bhkv,bthk->bthv", p["h0"], p["q"]), atol=1e-14)


def orthonormal_keys(K, n, seed):
    m = np.random.default_rng(seed).standard_normal((K, K))
    Q, _ = np.linalg.qr(m)
    return Q[:, :n].T                                            # n orthonormal rows


def test_orthonormal_keys_overwrite_and_retrieval():
    """g = 0, beta = 1, orthonormal keys: H_T = sum k_s v_s^T + (I - sum k_s k_s^T) H0,
    and querying with q_t = k_s (s <= t) returns scale * v_s."""
    K, V, T = 8, 5, 6
    keys = orthonormal_keys(K, T, 4)
    r = np.random.default_rng(5)
    v = r.standard_normal((T, V))
    h0 = r.standard_normal((K, V))
    lookup = [0, 1, 0, 3, 2, 5]                                  # q_t = k_{lookup[t]}, lookup[t] <= t
    q = keys[lookup]
    args = dict(q=q[None, :, None], k=keys[None, :, None], v=v[None, :, None],
                g=np.zeros((1, T, 1)), beta=np.ones((1, T, 1)), h0=h0[None, None])
    o, ht = oracle.fwd(**args, scale=0.25)
    ref = keys.T @ v + (np.eye(K) - keys.T @ keys) @ h0
    np.testing.assert_allclose(ht[0, 0], ref, atol=1e-13)
    np.testing.assert_allclose(o[0, :, 0], 0.25 * v[lookup], atol=1e-13)


def test_repeated_key_keeps_last_value():
    K, V = 6, 4
    key = orthonormal_keys(K, 1, 6)[0]
    r = np.random.default_rng(7)
    v = r.standard_normal((2, V))
    args = dict(q=np.stack([key, key])[None, :, None], k=np.stack([key, key])[None, :, None],
                v=v[None, :, None], g=np.zeros((1, 2, 1)), beta=np.ones((1, 2, 1)))
    o, ht = oracle.fwd(**args, scale=1.0)
    np.testing.assert_allclose(o[0, 1, 0], v[1], atol=1e-14)
    np.testing.assert_allclose(ht[0, 0], np.outer(key, v[1]), atol=1e-14)


def test_l2norm_closed_form_with_eps():
    """With g = 0, beta = 0: o = scale * H0^T q_hat, q_hat = q / sqrt(|q|^2 + eps);
    a short q makes the eps term visible."""
    K, V = 4, 3
    r = np.random.default_rng(8)
    h0 = r.standard_normal((1, 1, K, V))
    q = np.zeros((1, 1, 1, K))
    q[0, 0, 0, 2] = 1e-3
    eps = 1e-6
    args = dict(q=q, k=np.ones((1, 1, 1, K)), v=np.zeros((1, 1, 1, V)), g=np.zeros((1, 1, 1)),
                beta=np.zeros((1, 1, 1)), h0=h0)
    o, _ = oracle.fwd(**args, scale=1.0, use_l2norm=True, eps=eps)
    expect = h0[0, 0][2] * (1e-3 / np.sqrt(1e-6 + eps))
    np.testing.assert_allclose(o[0, 0, 0], expect, rtol=1e-13)


# ------------------------------------------------- independent chunked restatement
@pytest.mark.parametrize("C", [1, 16, 64, 200])
@pytest.mark.parametrize("l2", [False, True])
def test_chunked_form_matches_sequential(C, l2):
    pr = gdn_synth.make("tiny", T=200, K=16, V=12, H=2, h0_std=0.3, normalise=not l2)
    a = [x.double() for x in (pr.q, pr.k, pr.v, pr.g, pr.beta)]
    o, ht = oracle.fwd(*a, h0=pr.h0, use_l2norm=l2)
    oc, hc = chunked.forward(*a, h0=pr.h0.double(), C=C, use_l2norm=l2)
    np.testing.assert_allclose(oc.numpy(), o, atol=1e-12)
    np.testing.assert_allclose(hc.numpy(), ht, atol=1e-12)


# ---------------------------------------------------------------- gradients
def _loss(p, do, dht, **kw):
    o, ht = oracle.fwd(**p, **kw)
    return float((o * do).sum() + (ht * dht).sum())


@pytest.mark.parametrize("l2", [False, True])
def test_gradients_match_central_differences(l2):
    p = rand_problem(11, T=7, K=4, V=3, H=1, unit_keys=not l2)
    r = np.random.default_rng(12)
    do = r.standard_normal(p["v"].shape)
    dht = r.standard_normal(p["h0"].shape)
    kw = dict(scale=0.6, use_l2norm=l2)
    d = oracle.bwd(**p, do=do, dht=dht, **kw)
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", h0="dh0")
    h = 1e-6
    for name, gname in names.items():
        x = p[name]
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = _loss(p, do, dht, **kw)
            x[idx] = old - h
            lm = _loss(p, do, dht, **kw)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.abs(num - d[gname]).max() / max(1.0, np.abs(num).max())
        assert err < 1e-7, (name, err)


def test_gradients_match_autograd_of_chunked_form():
    pr = gdn_synth.make("tiny", T=150, K=16, V=16, H=2, h0_std=0.3, dht_std=0.2)
    leaves = [x.double().clone().requires_grad_(True)
              for x in (pr.q, pr.k, pr.v, pr.g, pr.beta, pr.h0)]
    q, k, v, g, beta, h0 = leaves
    o, ht = chunked.forward(q, k, v, g, beta, h0=h0, C=64, use_l2norm=True)
    loss = (o * pr.do.double()).sum() + (ht * pr.dht.double()).sum()
    loss.backward()
    d = oracle.bwd(*(x.detach() for x in leaves[:5]), do=pr.do, h0=pr.h0, dht=pr.dht,
                   use_l2norm=True)
    for leaf, name in zip(leaves, ["dq", "dk", "dv", "dg", "dbeta", "dh0"]):
        np.testing.assert_allclose(d[name], leaf.grad.numpy(), atol=1e-10, err_msg=name)


# ---------------------------------------------------------------- invariants
def test_varlen_equals_separate_runs():
    lens = [5, 0, 17, 1, 9]
    pr = gdn_synth.make("tiny", K=8, V=6, H=2, lengths=lens, h0_std=0.2, dht_std=0.1)
    o, ht = oracle.fwd(pr.q, pr.k, pr.v, pr.g, pr.beta, h0=pr.h0, cu_seqlens=pr.cu_seqlens)
    d = oracle.bwd(pr.q, pr.k, pr.v, pr.g, pr.beta, do=pr.do, h0=pr.h0, dht=pr.dht,
                   cu_seqlens=pr.cu_seqlens)
    cu = pr.cu_seqlens.tolist()
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        sub = [x[:, sl] for x in (pr.q, pr.k, pr.v, pr.g, pr.beta)]
        o1, h1 = oracle.fwd(*sub, h0=pr.h0[n:n + 1])
        d1 = oracle.bwd(*sub, do=pr.do[:, sl], h0=pr.h0[n:n + 1], dht=pr.dht[n:n + 1])
        np.testing.assert_allclose(o[:, sl], o1, atol=0)
        np.testing.assert_allclose(ht[n], h1[0], atol=0)
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            np.testing.assert_allclose(d[key][:, sl], d1[key], atol=0)
        np.testing.assert_allclose(d["dh0"][n], d1["dh0"][0], atol=0)
    # a zero-length sequence hands its state straight through
    np.testing.assert_allclose(ht[1], pr.h0[1].double().numpy(), atol=0)
    np.testing.assert_allclose(d["dh0"][1], pr.dht[1].double().numpy(), atol=0)


def test_state_continuation_forward_and_backward():
    pr = gdn_synth.make("tiny", T=130, K=8, V=8, H=2, h0_std=0.2, dht_std=0.1)
    full = [x for x in (pr.q, pr.k, pr.v, pr.g, pr.beta)]
    o, ht = oracle.fwd(*full, h0=pr.h0)
    d = oracle.bwd(*full, do=pr.do, h0=pr.h0, dht=pr.dht)
    cut = 77
    a = [x[:, :cut] for x in full]
    b = [x[:, cut:] for x in full]
    oa, ha = oracle.fwd(*a, h0=pr.h0)
    ob, hb = oracle.fwd(*b, h0=ha)
    np.testing.assert_allclose(np.concatenate([oa, ob], 1), o, atol=1e-13)
    np.testing.assert_allclose(hb, ht, atol=1e-13)
    db = oracle.bwd(*b, do=pr.do[:, cut:], h0=ha, dht=pr.dht)
    da = oracle.bwd(*a, do=pr.do[:, :cut], h0=pr.h0, dht=db["dh0"])
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        np.testing.assert_allclose(np.concatenate([da[key], db[key]], 1), d[key], atol=1e-12)
    np.testing.assert_allclose(da["dh0"], d["dh0"], atol=1e-12)


def test_joint_linearity_in_values_and_initial_state():
    p = rand_problem(21, T=10)
    p2 = dict(p, v=np.random.default_rng(22).standard_normal(p["v"].shape),
              h0=np.random.default_rng(23).standard_normal(p["h0"].shape))
    a, b = 0.7, -1.3
    pc = dict(p, v=a * p["v"] + b * p2["v"], h0=a * p["h0"] + b * p2["h0"])
    o1, h1 = oracle.fwd(**p)
    o2, h2 = oracle.fwd(**p2)
    oc, hc = oracle.fwd(**pc)
    np.testing.assert_allclose(oc, a * o1 + b * o2, atol=1e-12)
    np.testing.assert_allclose(hc, a * h1 + b * h2, atol=1e-12)


def test_unit_subset_matches_full_run():
    pr = gdn_synth.make("tiny", T=40, K=8, V=8, H=3, B=2, h0_std=0.2)
    o, ht = oracle.fwd(pr.q, pr.k, pr.v, pr.g, pr.beta, h0=pr.h0)
    units = [1, 5]                                                # (b=0,h=1), (b=1,h=2)
    os_, hs = oracle.fwd(pr.q, pr.k, pr.v, pr.g, pr.beta, h0=pr.h0, units=units)
    for u in units:
        b, h = divmod(u, 3)
        np.testing.assert_array_equal(os_[b, :, h], o[b, :, h])
        np.testing.assert_array_equal(hs[b, h], ht[b, h])
    assert np.isnan(os_[0, :, 0]).all()
