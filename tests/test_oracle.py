"""Pins for the fp64 oracle: each test checks it against something other than
itself -- values the pages print, closed forms, special cases that reduce to
a library routine, and brute force on tiny inputs.  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_mixture_experts_51_b300 import workloads as W


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- worked examples

def test_worked_gating_example(golden_dir):
    """Mixture-of-experts Models, Level 2: the printed top-two example."""
    g = _load(golden_dir, "gating_example.json")
    H = np.array([g["scores"]])
    # the scores reach the oracle through its logits step (x = 1, W_g = scores)
    H_from_logits = O.logits(np.ones((1, 1)), np.array([g["scores"]]))
    np.testing.assert_array_equal(H_from_logits, H)
    # printed softmax weights (3 decimals), independent of the oracle's gates()
    p = torch.softmax(torch.tensor(H, dtype=torch.float64), dim=1).numpy()[0]
    np.testing.assert_allclose(np.round(p, 3), g["printed_router_weights"], atol=0)
    idx = O.topk(H, g["top_k"])[0]
    assert sorted(idx.tolist()) == sorted(g["printed_experts_ascending"])
    # the page prints ascending-weight order; the oracle returns largest first
    assert idx.tolist() == list(reversed(g["printed_experts_ascending"]))
    w = O.gates(H, O.topk(H, g["top_k"]))[0]
    np.testing.assert_allclose(np.round(w[::-1], 3), g["printed_renormalised_ascending"], atol=0)
    assert abs(w[0] - 0.64566) < 1e-5 and abs(w[1] - 0.35434) < 1e-5


def test_worked_capacity_example(golden_dir):
    """Mixture-of-experts Models, Level 2: loads and overflow printed for C=2."""
    g = _load(golden_dir, "capacity_example.json")
    idx = np.array(g["assignments"])[:, None]
    d = O.dispatch(idx, g["n_experts"], g["capacity"])
    assert d["load"].tolist() == g["printed_loads"]
    assert np.maximum(d["load"] - g["capacity"], 0).tolist() == g["printed_overflow"]
    assert d["dropped"] == sum(g["printed_overflow"])
    # first come, first served (Lab 3): the third request for expert 0 is dropped
    assert d["pos"][:, 0].tolist() == [0, 1, -1, 0, 1, 0, 0, 1]
    assert d["counts"].tolist() == [2, 2, 1, 2]
    assert d["offsets"].tolist() == [0, 2, 4, 5, 7]


def test_capacities_of_the_five_layers(golden_dir):
    g = _load(golden_dir, "configs.json")
    for name, C in g["capacities"].items():
        w = W.WORKLOADS[name]
        assert O.capacity(w.T, w.k, w.E, w.capacity_factor) == C, name
    # no-drop layer: C equals T
    w = W.WORKLOADS["mixtral_t16384"]
    assert O.capacity(w.T, w.k, w.E, w.capacity_factor) == w.T


# ---------------------------------------------------------------- brute force

def _brute_topk(H, k):
    """rank(e) = #{e' : H[e'] > H[e] or (H[e'] == H[e] and e' < e)}; chosen iff rank < k."""
    T, E = H.shape
    out = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        for e in range(E):
            rank = sum(1 for e2 in range(E) if H[t, e2] > H[t, e] or (H[t, e2] == H[t, e] and e2 < e))
            if rank < k:
                out[t, rank] = e
    return out


def _brute_dispatch(idx, E, C):
    """pos(t,r) = #{(t',r') earlier in priority with the same expert}, O((Tk)^2)."""
    T, k = idx.shape
    order = [(r, t) for r in range(k) for t in range(T)]
    pos = np.full((T, k), -1, dtype=np.int64)
    load = [0] * E
    for j, (r, t) in enumerate(order):
        e = idx[t, r]
        earlier = sum(1 for (r2, t2) in order[:j] if idx[t2, r2] == e)
        load[e] += 1
        if earlier < C:
            pos[t, r] = earlier
    return pos, np.array(load)


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    T, E = 40, 7
    # small integers force many exact ties
    H = rng.integers(-3, 4, size=(T, E)).astype(np.float64)
    for k in (1, 2, 3, E):
        np.testing.assert_array_equal(O.topk(H, k), _brute_topk(H, k))


def test_tie_goes_to_lower_index_through_logits():
    # duplicated router columns give exactly equal logits (integer-valued, exact sums)
    x = np.array([[1.0, 2.0, -1.0], [0.0, 1.0, 3.0]])
    col = np.array([1.0, -2.0, 4.0])
    W_g = np.stack([col * 0, col, col, col * -1], axis=1)  # experts 1 and 2 identical
    H = O.logits(x, W_g)
    assert H[0, 1] == H[0, 2] and H[1, 1] == H[1, 2]
    idx = O.topk(H, 2)
    assert idx[1].tolist() == [1, 2]  # H[1] = [0, 10, 10, -10]: tie 1 vs 2 -> 1 first
    assert 1 in idx[0].tolist() or 0 in idx[0].tolist()


@pytest.mark.parametrize("seed,T,E,k,C", [(0, 9, 3, 2, 4), (1, 12, 4, 3, 5), (2, 7, 5, 1, 1),
                                          (3, 15, 4, 2, 3), (4, 6, 6, 6, 2), (5, 11, 2, 2, 100)])
def test_dispatch_brute_force(seed, T, E, k, C):
    rng = np.random.default_rng(seed)
    # distinct experts per token, like a real top-k table
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    d = O.dispatch(idx, E, C)
    pos, load = _brute_dispatch(idx, E, C)
    np.testing.assert_array_equal(d["pos"], pos)
    np.testing.assert_array_equal(d["load"], load)
    assert d["dropped"] == int(np.maximum(load - C, 0).sum())
    assert (d["counts"] <= C).all()
    assert int(d["counts"].sum()) + d["dropped"] == T * k
    # slots of each expert are exactly 0..counts-1
    for e in range(E):
        slots = sorted(d["pos"][(idx == e) & (d["pos"] >= 0)].tolist())
        assert slots == list(range(int(d["counts"][e])))


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("seed", range(4))
def test_gates_equal_renormalised_softmax(seed):
    """softmax over the selected logits (LLM part 09 s2) equals the renormalised
    top-k of the full softmax (Lab 1, Level 2, SimpleRouter)."""
    rng = np.random.default_rng(seed)
    H = rng.normal(size=(50, 9)) * 3
    for k in (1, 2, 4, 9):
        idx = O.topk(H, k)
        w = O.gates(H, idx)
        p = torch.softmax(torch.tensor(H), dim=1).numpy()
        sel = np.take_along_axis(p, idx, axis=1)
        np.testing.assert_allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-13)
        assert (np.diff(w, axis=1) <= 1e-15).all()  # largest first
    # top-1 gate is exactly 1
    assert (O.gates(H, O.topk(H, 1)) == 1.0).all()


def test_activation_functions_match_torch():
    a = np.linspace(-9, 9, 2001)
    ta = torch.tensor(a)
    np.testing.assert_allclose(O.gelu(a), torch.nn.functional.gelu(ta).numpy(), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(O.silu(a), torch.nn.functional.silu(ta).numpy(), rtol=1e-14, atol=1e-15)
    z = np.linspace(-40, 40, 2001)
    np.testing.assert_allclose(O.softplus(z), torch.nn.functional.softplus(torch.tensor(z), threshold=1e9).numpy(),
                               rtol=1e-14, atol=1e-300)


def test_noise_term_closed_forms():
    rng = np.random.default_rng(7)
    T, d, E = 5, 4, 3
    x = rng.normal(size=(T, d))
    W_g = rng.normal(size=(d, E))
    b_g = rng.normal(size=E)
    eps = rng.normal(size=(T, E))
    base = x @ W_g + b_g
    # W_noise = 0 -> softplus(0) = ln 2
    H = O.logits(x, W_g, b_g, np.zeros((d, E)), eps)
    np.testing.assert_allclose(H, base + eps * math.log(2.0), rtol=1e-14, atol=1e-14)
    # eps = 0 -> noiseless
    Wn = rng.normal(size=(d, E))
    np.testing.assert_allclose(O.logits(x, W_g, b_g, Wn, np.zeros((T, E))), base, rtol=0, atol=0)
    # one scalar entry by hand
    t, e = 2, 1
    z = sum(x[t, j] * Wn[j, e] for j in range(d))
    want = sum(x[t, j] * W_g[j, e] for j in range(d)) + b_g[e] + eps[t, e] * math.log1p(math.exp(z))
    assert abs(O.logits(x, W_g, b_g, Wn, eps)[t, e] - want) < 1e-12


def _loop_expert(xrow, e, act, W1, W3, W2, b1, b2):
    """Pure-Python per-element expert (nn.Linear layout: out_f = sum_j x_j W[f, j])."""
    F, d = W1.shape[1], W1.shape[2]
    h = []
    for f in range(F):
        a = sum(xrow[j] * W1[e, f, j] for j in range(d))
        if act == O.GELU:
            a += 0.0 if b1 is None else b1[e, f]
            h.append(a * 0.5 * (1 + math.erf(a / math.sqrt(2))))
        else:
            u = sum(xrow[j] * W3[e, f, j] for j in range(d))
            h.append(a / (1 + math.exp(-a)) * u)
    return np.array([sum(h[f] * W2[e, i, f] for f in range(F)) + (0.0 if b2 is None else b2[e, i])
                     for i in range(d)])


@pytest.mark.parametrize("act", [O.GELU, O.SWIGLU])
def test_expert_matches_elementwise_loops(act):
    rng = np.random.default_rng(11)
    E, d, F = 3, 5, 7  # non-square so a transposed operand cannot pass
    W1 = rng.normal(size=(E, F, d))
    W3 = rng.normal(size=(E, F, d))
    W2 = rng.normal(size=(E, d, F))
    b1 = rng.normal(size=(E, F)) if act == O.GELU else None
    b2 = rng.normal(size=(E, d))
    xr = rng.normal(size=(4, d))
    for e in range(E):
        y = O.expert(xr, e, act, W1, W3, W2, b1, b2)
        for i in range(4):
            np.testing.assert_allclose(y[i], _loop_expert(xr[i], e, act, W1, W3, W2, b1, b2), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- layer-level special cases

def _tiny_layer(seed, T=24, d=6, E=4, F=5, act=O.GELU, bias=True):
    rng = np.random.default_rng(seed)
    return dict(x=rng.normal(size=(T, d)), W_g=rng.normal(size=(d, E)),
                b_g=rng.normal(size=E) if bias else None,
                W1=rng.normal(size=(E, F, d)) / math.sqrt(d), W3=rng.normal(size=(E, F, d)) / math.sqrt(d),
                W2=rng.normal(size=(E, d, F)) / math.sqrt(F),
                b1=rng.normal(size=(E, F)) if (bias and act == O.GELU) else None,
                b2=rng.normal(size=(E, d)) if bias else None)


@pytest.mark.parametrize("act", [O.GELU, O.SWIGLU])
def test_k_equals_E_is_dense_softmax_mixture(act):
    """With k = E and C >= T every expert sees every token: the layer is the
    dense softmax-weighted mixture of the 'Mathematical Formulation' with k = N."""
    L = _tiny_layer(3, act=act)
    T, E = L["x"].shape[0], L["W_g"].shape[1]
    res = O.forward(L["x"], L["W_g"], E, act, L["W1"], L["W2"], L["W3"], L["b1"], L["b2"],
                    b_g=L["b_g"], C=T)
    assert res["dropped"] == 0
    # dense form in torch fp64: softmax over all experts, every expert on every token
    x = torch.tensor(L["x"])
    p = torch.softmax(x @ torch.tensor(L["W_g"]) + torch.tensor(L["b_g"]), dim=1)
    moe = torch.zeros_like(x)
    for e in range(E):
        a = x @ torch.tensor(L["W1"][e]).T
        if act == O.GELU:
            h = torch.nn.functional.gelu(a + torch.tensor(L["b1"][e]))
        else:
            h = torch.nn.functional.silu(a) * (x @ torch.tensor(L["W3"][e]).T)
        y = h @ torch.tensor(L["W2"][e]).T + torch.tensor(L["b2"][e])
        moe += p[:, e:e + 1] * y
    np.testing.assert_allclose(res["moe"], moe.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(res["out"], (x + moe).numpy(), rtol=1e-11, atol=1e-12)


def test_k1_is_argmax_expert_with_unit_gate():
    L = _tiny_layer(4, act=O.SWIGLU)
    T = L["x"].shape[0]
    res = O.forward(L["x"], L["W_g"], 1, O.SWIGLU, L["W1"], L["W2"], L["W3"], None, L["b2"], b_g=L["b_g"], C=T)
    H = L["x"] @ L["W_g"] + L["b_g"]
    for t in range(T):
        e = int(np.argmax(H[t]))
        assert res["idx"][t, 0] == e and res["w"][t, 0] == 1.0
        y = O.expert(L["x"][t:t + 1], e, O.SWIGLU, L["W1"], L["W3"], L["W2"], None, L["b2"])[0]
        np.testing.assert_allclose(res["moe"][t], y, rtol=1e-13, atol=1e-14)


def test_dropped_tokens_pass_through_and_gates_are_not_renormalised():
    L = _tiny_layer(5, T=30)
    k, C = 2, 3
    res = O.forward(L["x"], L["W_g"], k, O.GELU, L["W1"], L["W2"], None, L["b1"], L["b2"], b_g=L["b_g"], C=C)
    assert res["dropped"] > 0
    pos, w, idx = res["pos"], res["w"], res["idx"]
    for t in range(30):
        kept = [r for r in range(k) if pos[t, r] >= 0]
        if not kept:
            np.testing.assert_array_equal(res["out"][t], L["x"][t])
            assert not res["moe"][t].any()
        want = np.zeros(L["x"].shape[1])
        for r in kept:
            want += w[t, r] * O.expert(L["x"][t:t + 1], int(idx[t, r]), O.GELU, L["W1"], None, L["W2"], L["b1"], L["b2"])[0]
        np.testing.assert_allclose(res["moe"][t], want, rtol=1e-12, atol=1e-13)


def test_token_subset_matches_full_evaluation():
    L = _tiny_layer(6, T=40)
    full = O.forward(L["x"], L["W_g"], 2, O.GELU, L["W1"], L["W2"], None, L["b1"], L["b2"], b_g=L["b_g"], C=14)
    sub = [0, 7, 13, 39]
    part = O.forward(L["x"], L["W_g"], 2, O.GELU, L["W1"], L["W2"], None, L["b1"], L["b2"], b_g=L["b_g"], C=14, tokens=sub)
    np.testing.assert_allclose(part["out"], full["out"][sub], rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(part["pos"], full["pos"])


# ---------------------------------------------------------------- Lab invariants

def test_lab1_invariants_no_drop():
    """Lab 1: every token reaches exactly k experts; more than one expert is used."""
    L = _tiny_layer(8, T=20, d=6, E=8)
    res = O.forward(L["x"], L["W_g"], 2, O.GELU, L["W1"], L["W2"], None, L["b1"], L["b2"], C=20)
    assert int(res["counts"].sum()) == 20 * 2 and res["dropped"] == 0
    assert (res["counts"] > 0).sum() >= 2


@pytest.mark.parametrize("seed", range(5))
def test_lab3_capacity_behaviour(seed):
    """Lab 3: balanced routing with factor 1.5 drops < 5%; skewed routing with
    factor 1.0 drops more; no expert exceeds its capacity."""
    rng = np.random.default_rng(100 + seed)
    n, E = 100, 4
    balanced = rng.integers(0, E, size=n)
    skewed = np.concatenate([np.zeros(60, dtype=np.int64), rng.integers(1, E, size=40)])
    rng.shuffle(skewed)
    Ca = O.capacity(n, 1, E, 1.5)
    Cb = O.capacity(n, 1, E, 1.0)
    da = O.dispatch(balanced[:, None], E, Ca)
    db = O.dispatch(skewed[:, None], E, Cb)
    ra, rb = da["dropped"] / n, db["dropped"] / n
    assert ra < 0.05 and rb > ra
    assert da["counts"].max() <= Ca and db["counts"].max() <= Cb


def test_near_tie_report():
    H = np.array([[1.0, 1.00005, 0.0, -1.0],   # adjacent inside top-2
                  [2.0, 1.0, 0.99995, -1.0],   # boundary k-th vs (k+1)-th
                  [3.0, 2.0, 1.0, 0.0]])
    r = O.near_ties(H, 2)
    assert r["boundary"].tolist() == [1]
    assert r["any_adjacent"].tolist() == [0, 1]


def test_workload_generator_is_deterministic():
    w = W.WORKLOADS["tiny_fp32"]
    a, b = W.make_inputs(w), W.make_inputs(w)
    for key in a:
        if a[key] is None:
            assert b[key] is None
        else:
            assert torch.equal(a[key], b[key])
    s = W.make_inputs(W.WORKLOADS["switch_top1"].scaled(64))
    np.testing.assert_allclose(s["b_g"].numpy()[:3], [0.0, 2 * math.log(0.5), 2 * math.log(1 / 3)], rtol=1e-6)


# ----------------------------------------------------------------------------
# routing diagnostics and the auxiliary load-balancing loss
# ----------------------------------------------------------------------------

def _softmax_rows(H):
    z = np.exp(H - H.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def test_aux_loss_is_one_for_uniform_routing():
    """[P1] Mathematical Formulation: uniform f and P give L_aux = 1 exactly;
    uniform probabilities have entropy ln E; equal loads have zero CV."""
    T, E, k = 24, 6, 2
    H = np.zeros((T, E))
    idx = np.array([[t % E, (t + 1) % E] for t in range(T)])
    counts = np.full(E, T * k // E)
    st = O.routing_stats(H, idx, counts, 0)
    assert st["aux_loss"] == pytest.approx(1.0, abs=1e-15)
    assert st["entropy"] == pytest.approx(math.log(E), abs=1e-12)
    assert st["load_cv"] == 0.0 and st["kept_cv"] == 0.0
    assert st["utilisation"] == 1.0 and st["overflow"] == 0.0
    np.testing.assert_allclose(st["f"], 1.0 / E)
    np.testing.assert_allclose(st["P"], 1.0 / E)


def test_aux_loss_is_E_for_full_collapse():
    """Every token routed to one expert with probability ~1: f = P = e_0, so
    L_aux -> E and the per-token entropy -> 0."""
    T, E = 50, 8
    H = np.full((T, E), -80.0)
    H[:, 0] = 80.0
    idx = np.zeros((T, 1), dtype=np.int64)
    st = O.routing_stats(H, idx, np.array([T] + [0] * (E - 1)), 0)
    assert st["aux_loss"] == pytest.approx(E, rel=1e-12)
    assert st["entropy"] < 1e-60
    assert st["utilisation"] == 1.0 / E


@pytest.mark.parametrize("seed", [3, 4, 5])
def test_aux_loss_detects_collapse(seed):
    """[P1] Lab 2: logits N(0, 0.5^2) per expert, top-1 routing; adding 5 to
    expert 0's logit (collapse) lifts the loss above 1.5, the balanced router
    stays below 1.5 (our seeds, the lab's thresholds)."""
    rng = np.random.default_rng(seed)
    T, E = 200, 6
    base = rng.standard_normal((T, E)) * 0.5
    out = {}
    for name, bias in (("balanced", 0.0), ("collapsed", 5.0)):
        H = base.copy()
        H[:, 0] += bias
        idx = O.topk(H, 1)
        d = O.dispatch(idx, E, T)
        out[name] = O.routing_stats(H, idx, d["counts"], d["dropped"])
    assert out["balanced"]["aux_loss"] < 1.5 < out["collapsed"]["aux_loss"]
    assert out["collapsed"]["f"][0] > 0.9
    assert out["collapsed"]["load_cv"] > out["balanced"]["load_cv"]


def test_routing_stats_brute_force_and_token_order():
    """f, P, the loss and the entropy against element-by-element loops on a
    small batch with top-3 routing and capacity drops; the statistics do not
    depend on the order of the tokens."""
    rng = np.random.default_rng(11)
    T, E, k, C = 13, 5, 3, 6
    H = rng.standard_normal((T, E)) * 2.0
    idx = O.topk(H, k)
    d = O.dispatch(idx, E, C)
    st = O.routing_stats(H, idx, d["counts"], d["dropped"])
    f = [0.0] * E
    P = [0.0] * E
    ent = 0.0
    for t in range(T):
        m = max(H[t])
        ex = [math.exp(H[t, e] - m) for e in range(E)]
        s = sum(ex)
        for e in range(E):
            P[e] += ex[e] / s / T
            ent -= (ex[e] / s) * math.log(ex[e] / s) / T
        for r in range(k):
            f[idx[t, r]] += 1.0 / (T * k)
    np.testing.assert_allclose(st["f"], f, rtol=0, atol=1e-15)
    np.testing.assert_allclose(st["P"], P, rtol=0, atol=1e-15)
    assert st["aux_loss"] == pytest.approx(E * sum(a * b for a, b in zip(f, P)), abs=1e-14)
    assert st["entropy"] == pytest.approx(ent, abs=1e-14)
    # f is taken before the capacity cut: the drops change the kept CV, not f
    assert d["dropped"] > 0
    loads = np.array(f) * T * k
    assert st["load_cv"] == pytest.approx(float(np.std(loads) / np.mean(loads)), abs=1e-14)
    assert st["overflow"] == pytest.approx(d["dropped"] / (T * k))
    perm = rng.permutation(T)
    st2 = O.routing_stats(H[perm], idx[perm], d["counts"], d["dropped"])
    for key in ("f", "P"):
        np.testing.assert_allclose(st2[key], st[key], atol=1e-15)
    assert st2["aux_loss"] == pytest.approx(st["aux_loss"], abs=1e-14)


# ---------------------------------------------------------------- shared experts

def _shared(seed, S=2, d=6, Fs=5, act=O.GELU, bias=True):
    rng = np.random.default_rng(seed)
    return dict(W1s=rng.normal(size=(S, Fs, d)) / math.sqrt(d), W3s=rng.normal(size=(S, Fs, d)) / math.sqrt(d),
                W2s=rng.normal(size=(S, d, Fs)) / math.sqrt(Fs),
                b1s=rng.normal(size=(S, Fs)) if (bias and act == O.GELU) else None,
                b2s=rng.normal(size=(S, d)) if bias else None)


def _torch_ffn(x, act, W1, W3, W2, b1, b2):
    """One FFN in torch fp64 via F.linear (nn.Linear layout)."""
    lin = torch.nn.functional.linear
    t = lambda a: None if a is None else torch.tensor(a)
    if act == O.GELU:
        h = torch.nn.functional.gelu(lin(x, t(W1), t(b1)))
    else:
        h = torch.nn.functional.silu(lin(x, t(W1))) * lin(x, t(W3))
    return lin(h, t(W2), t(b2))


@pytest.mark.parametrize("act", [O.GELU, O.SWIGLU])
def test_shared_experts_alone_when_every_assignment_is_dropped(act):
    """C = 0 drops every routed assignment: the layer is x + the shared experts'
    sum, every token through every shared expert with weight 1 (torch fp64)."""
    L = _tiny_layer(31, act=act)
    S = _shared(32, act=act)
    res = O.forward(L["x"], L["W_g"], 2, act, L["W1"], L["W2"], L["W3"], L["b1"], L["b2"], b_g=L["b_g"], C=0,
                    shared=S)
    assert res["dropped"] == 2 * L["x"].shape[0]
    x = torch.tensor(L["x"])
    want = sum(_torch_ffn(x, act, S["W1s"][s], S["W3s"][s], S["W2s"][s],
                          None if S["b1s"] is None else S["b1s"][s], S["b2s"][s]) for s in range(2))
    np.testing.assert_allclose(res["moe"], want.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(res["out"], (x + want).numpy(), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("act", [O.GELU, O.SWIGLU])
def test_k_equals_E_with_shared_is_dense_mixture_plus_shared(act):
    L = _tiny_layer(33, act=act)
    S = _shared(34, S=1, act=act)
    T, E = L["x"].shape[0], L["W_g"].shape[1]
    res = O.forward(L["x"], L["W_g"], E, act, L["W1"], L["W2"], L["W3"], L["b1"], L["b2"], b_g=L["b_g"], C=T,
                    shared=S)
    x = torch.tensor(L["x"])
    p = torch.softmax(x @ torch.tensor(L["W_g"]) + torch.tensor(L["b_g"]), dim=1)
    moe = _torch_ffn(x, act, S["W1s"][0], S["W3s"][0], S["W2s"][0],
                     None if S["b1s"] is None else S["b1s"][0], S["b2s"][0])
    for e in range(E):
        moe = moe + p[:, e:e + 1] * _torch_ffn(x, act, L["W1"][e], L["W3"][e], L["W2"][e],
                                               None if L["b1"] is None else L["b1"][e], L["b2"][e])
    np.testing.assert_allclose(res["moe"], moe.numpy(), rtol=1e-11, atol=1e-12)


def test_shared_expert_matches_elementwise_loops():
    S = _shared(35, S=3, d=5, Fs=4, act=O.SWIGLU)
    xr = np.random.default_rng(36).normal(size=(3, 5))
    y = O.shared_experts(xr, O.SWIGLU, S["W1s"], S["W2s"], S["W3s"], None, S["b2s"])
    for i in range(3):
        want = sum(_loop_expert(xr[i], s, O.SWIGLU, S["W1s"], S["W3s"], S["W2s"], None, S["b2s"]) for s in range(3))
        np.testing.assert_allclose(y[i], want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", [O.GELU, O.SWIGLU])
def test_shared_experts_equal_one_wide_ffn(act):
    """S shared experts of width F_s are one FFN of width S*F_s: W1/W3 rows
    stacked, W2 columns stacked, b1 concatenated, b2 summed (the form the
    library takes them in)."""
    S = _shared(37, S=3, d=6, Fs=4, act=act)
    x = np.random.default_rng(38).normal(size=(9, 6))
    wide = dict(W1s=S["W1s"].reshape(1, 12, 6), W3s=S["W3s"].reshape(1, 12, 6),
                W2s=np.concatenate(list(S["W2s"]), axis=1)[None], b2s=S["b2s"].sum(axis=0)[None],
                b1s=None if S["b1s"] is None else S["b1s"].reshape(1, 12))
    a = O.shared_experts(x, act, S["W1s"], S["W2s"], S["W3s"], S["b1s"], S["b2s"])
    b = O.shared_experts(x, act, wide["W1s"], wide["W2s"], wide["W3s"], wide["b1s"], wide["b2s"])
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- expert-choice routing

def _check_top_sets(H, sel):
    """Definition of an expert's top-C set, checked pair by pair: every chosen
    token beats every unchosen one (larger score, or equal score and lower index)."""
    T, E = H.shape
    for e in range(E):
        ch = set(int(t) for t in sel[e])
        assert len(ch) == sel.shape[1] == min(sel.shape[1], T)
        for t in ch:
            for u in range(T):
                if u not in ch:
                    assert H[t, e] > H[u, e] or (H[t, e] == H[u, e] and t < u), (e, t, u)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_expert_choice_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    T, E = 23, 5
    H = rng.integers(-3, 4, size=(T, E)).astype(np.float64)  # many exact ties
    for C in [0, 1, 4, 9, 23, 40]:
        ec = O.expert_choice(H, C)
        assert ec["sel"].shape == (E, min(C, T))
        _check_top_sets(H, ec["sel"])
        assert (np.diff(ec["sel"], axis=1) > 0).all()   # ascending token order
        np.testing.assert_array_equal(ec["counts"], np.full(E, min(C, T)))  # every expert filled
        assert ec["dropped"] == int((~ec["chosen"].any(axis=1)).sum())


def test_expert_choice_gates_are_router_probabilities():
    rng = np.random.default_rng(5)
    H = rng.normal(size=(12, 4))
    ec = O.expert_choice(H, 5)
    p = torch.softmax(torch.tensor(H), dim=1).numpy()
    for e in range(4):
        for j, t in enumerate(ec["sel"][e]):
            assert abs(ec["gates"][e, j] - p[t, e]) < 1e-15


@pytest.mark.parametrize("act", [O.GELU, O.SWIGLU])
def test_expert_choice_with_full_capacity_is_dense_softmax_mixture(act):
    """C >= T: every expert takes every token, so the layer is the dense
    softmax-weighted mixture sum_e p_e E_e(x) (torch fp64), the same layer
    as token choice with k = E."""
    L = _tiny_layer(41, act=act)
    T, E = L["x"].shape[0], L["W_g"].shape[1]
    res = O.forward_expert_choice(L["x"], L["W_g"], act, L["W1"], L["W2"], L["W3"], L["b1"], L["b2"],
                                  b_g=L["b_g"], C=T + 3)
    x = torch.tensor(L["x"])
    p = torch.softmax(x @ torch.tensor(L["W_g"]) + torch.tensor(L["b_g"]), dim=1)
    moe = torch.zeros_like(x)
    for e in range(E):
        moe = moe + p[:, e:e + 1] * _torch_ffn(x, act, L["W1"][e], L["W3"][e], L["W2"][e],
                                               None if L["b1"] is None else L["b1"][e], L["b2"][e])
    np.testing.assert_allclose(res["moe"], moe.numpy(), rtol=1e-11, atol=1e-12)
    assert res["dropped"] == 0


def test_expert_choice_unchosen_tokens_pass_through_and_multi_expert_tokens_sum():
    L = _tiny_layer(42, T=30, E=4)
    res = O.forward_expert_choice(L["x"], L["W_g"], O.GELU, L["W1"], L["W2"], None, L["b1"], L["b2"],
                                  b_g=L["b_g"], C=5)
    ch = res["chosen"]
    assert res["dropped"] > 0 and (ch.sum(axis=1) > 1).any()
    for t in range(30):
        want = np.zeros(L["x"].shape[1])
        for e in range(4):
            if ch[t, e]:
                want += res["P"][t, e] * O.expert(L["x"][t:t + 1], e, O.GELU, L["W1"], None, L["W2"], L["b1"],
                                                  L["b2"])[0]
        np.testing.assert_allclose(res["moe"][t], want, rtol=1e-12, atol=1e-13)
        if not ch[t].any():
            np.testing.assert_array_equal(res["out"][t], L["x"][t])


def test_expert_choice_capacity_default_and_token_subset():
    L = _tiny_layer(43, T=40)
    full = O.forward_expert_choice(L["x"], L["W_g"], O.GELU, L["W1"], L["W2"], None, L["b1"], L["b2"],
                                   b_g=L["b_g"], capacity_factor=1.0, k=2)
    assert full["C"] == 20  # ceil(1.0 * 40 * 2 / 4)
    sub = [1, 8, 39]
    part = O.forward_expert_choice(L["x"], L["W_g"], O.GELU, L["W1"], L["W2"], None, L["b1"], L["b2"],
                                   b_g=L["b_g"], capacity_factor=1.0, k=2, tokens=sub)
    np.testing.assert_allclose(part["out"], full["out"][sub], rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- overflow variants

def test_reroute_worked_example():
    """The worked capacity example of "Mixture-of-experts Models" (top-1
    assignments [0,0,0,1,1,2,3,3], capacity 2: the third token overflows
    expert 0), with per-token backups: the overflow goes to its backup when
    that expert has room, and stays dropped when it is full.  Values worked
    by hand."""
    idx = np.array([[0], [0], [0], [1], [1], [2], [3], [3]])
    disp = O.dispatch(idx, 4, 2)
    assert disp["dropped"] == 1 and list(disp["counts"]) == [2, 2, 1, 2]
    rr = O.reroute(idx, disp, np.array([1, 2, 2, 0, 3, 3, 2, 0]), 2)
    assert rr["idx"][:, 0].tolist() == [0, 0, 2, 1, 1, 2, 3, 3]
    assert rr["pos"][:, 0].tolist() == [0, 1, 1, 0, 1, 0, 0, 1]
    assert rr["counts"].tolist() == [2, 2, 2, 2] and rr["offsets"].tolist() == [0, 2, 4, 6, 8]
    assert rr["dropped"] == 0 and rr["rerouted"] == 1
    full = O.reroute(idx, disp, np.array([1, 2, 1, 0, 3, 3, 2, 0]), 2)  # token 2's backup (1) is full
    assert full["idx"][2, 0] == 0 and full["pos"][2, 0] == -1 and full["dropped"] == 1 and full["rerouted"] == 0


def test_reroute_through_the_layer_uses_the_next_ranked_expert():
    """Logits built so every token's ranking is known: the backup is the
    (k+1)-th expert of the token's own ranking."""
    T, E = 8, 4
    top = [0, 0, 0, 1, 1, 2, 3, 3]
    nxt = [1, 2, 2, 0, 3, 3, 2, 0]
    H = np.zeros((T, E))
    for t in range(T):
        H[t, top[t]] = 10.0
        H[t, nxt[t]] = 5.0
    # identity-like x and W_g so that logits == H exactly
    x = np.eye(T)
    res = O.forward(x, H, 1, O.GELU, np.zeros((E, 2, T)), np.zeros((E, T, 2)), C=2, overflow="reroute")
    assert res["idx"][:, 0].tolist() == [0, 0, 2, 1, 1, 2, 3, 3]
    assert res["dropped"] == 0 and res["rerouted"] == 1
    np.testing.assert_array_equal(res["backup"], nxt)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_reroute_invariants(seed):
    rng = np.random.default_rng(seed)
    T, E, k, C = 40, 6, 2, 9
    H = rng.normal(size=(T, E)) + np.linspace(2, 0, E)  # skewed: drops happen
    idx0 = O.topk(H, k)
    disp = O.dispatch(idx0, E, C)
    backup = O.topk(H, k + 1)[:, k]
    rr = O.reroute(idx0, disp, backup, C)
    assert disp["dropped"] > 0
    assert (rr["counts"] <= C).all() and rr["counts"].sum() + rr["dropped"] == T * k
    assert rr["dropped"] == disp["dropped"] - rr["rerouted"]
    for t in range(T):
        assert len(set(rr["idx"][t][rr["pos"][t] >= 0])) == int((rr["pos"][t] >= 0).sum())  # no expert twice
        for r in range(k):
            if rr["idx"][t, r] != idx0[t, r]:           # moved: only the first dropped rank, to the backup
                assert rr["idx"][t, r] == backup[t] and disp["pos"][t, r] < 0
                assert all(disp["pos"][t, q] >= 0 for q in range(r))
            elif rr["pos"][t, r] < 0 and all(disp["pos"][t, q] >= 0 for q in range(r)):
                assert rr["counts"][backup[t]] == C   # a refused request found its backup full
    # the rows of each expert are numbered 0..counts-1 without gaps
    for e in range(E):
        slots = sorted(rr["pos"][(rr["idx"] == e) & (rr["pos"] >= 0)].tolist())
        assert slots == list(range(rr["counts"][e]))
    # with room for everything, re-routing changes nothing
    big = O.dispatch(idx0, E, T * k)
    same = O.reroute(idx0, big, backup, T * k)
    np.testing.assert_array_equal(same["idx"], idx0)
    assert same["rerouted"] == 0


def test_raw_gates_are_routing_probabilities():
    rng = np.random.default_rng(7)
    H = rng.normal(size=(10, 5))
    idx = O.topk(H, 2)
    p = torch.softmax(torch.tensor(H), dim=1).numpy()
    w = O.gates_raw(H, idx)
    np.testing.assert_allclose(w, np.take_along_axis(p, idx, axis=1), rtol=1e-15, atol=0)
    assert (w.sum(axis=1) < 1).all()
    # renormalising the raw gates gives the default gates
    np.testing.assert_allclose(w / w.sum(axis=1, keepdims=True), O.gates(H, idx), rtol=1e-13, atol=1e-15)
    # k = E: the raw gates are the whole distribution
    np.testing.assert_allclose(O.gates_raw(H, O.topk(H, 5)).sum(axis=1), 1.0, rtol=1e-14)
