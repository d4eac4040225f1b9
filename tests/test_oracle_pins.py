"""Pins for the CPU oracle: each check ties it to something other than itself.

These run on the CPU only.  A plausible slip in the oracle (a dropped term, a wrong sign
or index, a transposed operand, silu on the wrong branch, a wrong tie rule, a missing
inverse-permutation entry) fails at least one of them.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng


# ----------------------------------------------------------------------------- rounding


def _bits_bf16(v):
    return int(np.asarray(O.round_bf16(np.array([v]))[0], np.float32).view(np.uint32)) >> 16


def test_bf16_rounding_hand_derived_bit_patterns():
    assert _bits_bf16(1.0) == 0x3F80
    # 1 + 2^-8 sits exactly half-way between 1.0 and 1 + 2^-7: ties go to the even 0x3F80
    assert _bits_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 is half-way with an odd kept bit: rounds up to 0x3F82
    assert _bits_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # just above half-way rounds up
    assert _bits_bf16(1.0 + 2.0 ** -8 + 2.0 ** -20) == 0x3F81
    assert _bits_bf16(-2.5) == 0xC020
    # the largest fp32 rounds up past the largest bf16 to +inf
    assert _bits_bf16(float(np.finfo(np.float32).max)) == 0x7F80


def test_bf16_rounding_matches_torch_conversion():
    v = rng(7).standard_normal(100_000) * np.exp(rng(8).uniform(-30, 30, 100_000))
    ours = O.round_bf16(v)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, ref)


# ----------------------------------------------------------------------------- gating


def brute_topk(l, k):
    """k rounds of selection: take the largest remaining logit, lower index on ties."""
    T, E = l.shape
    out = np.zeros((T, k), np.int32)
    for t in range(T):
        left = list(range(E))
        for j in range(k):
            best = left[0]
            for e in left[1:]:
                if l[t, e] > l[t, best]:
                    best = e
            out[t, j] = best
            left.remove(best)
    return out


@pytest.mark.parametrize("E,k", [(2, 1), (4, 2), (8, 2), (16, 6), (7, 7), (33, 5)])
def test_topk_matches_bruteforce_selection(E, k):
    l = rng(E * 100 + k).standard_normal((40, E)).astype(np.float32)
    np.testing.assert_array_equal(O.topk(l, k), brute_topk(l, k))
    # small integer logits force many ties
    li = rng(E + k).integers(-2, 3, size=(40, E)).astype(np.float32)
    np.testing.assert_array_equal(O.topk(li, k), brute_topk(li, k))


def test_topk_ties_go_to_lower_index():
    l = np.array([[1.0, 3.0, 3.0, 2.0], [0.0, 0.0, 0.0, 0.0], [5.0, -1.0, 5.0, 5.0]])
    np.testing.assert_array_equal(O.topk(l, 2), [[1, 2], [0, 1], [0, 2]])
    np.testing.assert_array_equal(O.topk(l, 4), [[1, 2, 3, 0], [0, 1, 2, 3], [0, 2, 3, 1]])


def test_softmax_two_expert_closed_form():
    l = rng(1).standard_normal((50, 2)) * 4
    p = O.softmax(l)
    p0 = 1.0 / (1.0 + np.exp(l[:, 1] - l[:, 0]))
    np.testing.assert_allclose(p[:, 0], p0, rtol=1e-14, atol=0)
    np.testing.assert_allclose(p[:, 1], 1.0 - p0, rtol=1e-13, atol=1e-16)


def test_softmax_normalised_positive_and_shift_invariant():
    l = rng(2).standard_normal((30, 17)) * 10
    p = O.softmax(l)
    assert (p > 0).all()
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(O.softmax(l + 123.0), p, rtol=1e-12)


def test_route_weights_are_selected_probabilities_not_renormalised():
    l = rng(3).standard_normal((20, 8)).astype(np.float32)
    r = O.route_from_logits(l, 3, "f32")
    p = O.softmax(l)
    for t in range(20):
        for j in range(3):
            assert abs(r["topk_w"][t, j] - p[t, r["topk_idx"][t, j]]) < 1e-7
        assert r["topk_w"][t].sum() < 1.0
        # descending weights follow descending logits
        assert all(r["topk_w"][t, j] >= r["topk_w"][t, j + 1] for j in range(2))


def test_router_logits_bias_added_after_product():
    x = np.array([[1.0, 2.0]])
    Wg = np.array([[1.0, 0.0, -1.0], [0.5, 1.0, 0.0]])
    b = np.array([0.0, -1.0, 3.0])
    np.testing.assert_array_equal(O.router_logits(x, Wg, b, "f64"), [[2.0, 1.0, 2.0]])


# ----------------------------------------------------------------------------- PFT


def _routing(T, E, k, seed, skew=False):
    l = rng(seed).standard_normal((T, E)).astype(np.float32)
    if skew:
        l = l + (-1.6 * np.log(np.arange(E) + 1.0)).astype(np.float32)
    return O.topk(l, k)


@pytest.mark.parametrize("T,E,k,skew", [(1, 4, 2, False), (37, 8, 2, False), (64, 16, 6, True),
                                        (50, 5, 5, False), (33, 1, 1, False), (100, 64, 6, True)])
def test_pft_invariants_and_bruteforce_recount(T, E, k, skew):
    idx = _routing(T, E, k, T * 7 + E, skew)
    p = O.pft_build(idx, E)
    Tk = T * k
    # brute-force recount over every (t, j, e)
    counts = np.zeros(E, np.int64)
    for t in range(T):
        for j in range(k):
            for e in range(E):
                if idx[t, j] == e:
                    counts[e] += 1
    np.testing.assert_array_equal(p["num_ids"], counts)
    assert p["num_ids"].sum() == Tk and p["offsets"][0] == 0 and p["offsets"][E] == Tk
    assert len(p["token_ids"]) == Tk  # exactly T*k rows: no padded rows
    assert (np.diff(p["expert_ids"]) >= 0).all()
    for e in range(E):
        seg = p["token_ids"][p["offsets"][e]:p["offsets"][e + 1]]
        assert (np.diff(seg) > 0).all()
        assert (p["expert_ids"][p["offsets"][e]:p["offsets"][e + 1]] == e).all()
    # slot_of is a permutation and the inverse of (token_ids, expert_ids)
    assert sorted(p["slot_of"].tolist()) == list(range(Tk))
    for t in range(T):
        for j in range(k):
            s = p["slot_of"][t * k + j]
            assert p["token_ids"][s] == t and p["expert_ids"][s] == idx[t, j]


def test_pft_positions_by_counting_earlier_tokens():
    """Position of (t, e) = (tokens routed to experts < e) + (tokens t' < t routed to e)."""
    T, E, k = 29, 6, 3
    idx = _routing(T, E, k, 5)
    p = O.pft_build(idx, E)
    chose = [[e in idx[t] for e in range(E)] for t in range(T)]
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            before = sum(chose[tt][ee] for tt in range(T) for ee in range(e))
            earlier = sum(chose[tt][e] for tt in range(t))
            assert p["slot_of"][t * k + j] == before + earlier


# ----------------------------------------------------------------------------- dispatch / combine


def test_dispatch_adjoint_identity():
    T, E, k, h = 23, 6, 2, 5
    idx = _routing(T, E, k, 11)
    p = O.pft_build(idx, E)
    x = rng(12).standard_normal((T, h))
    u = rng(13).standard_normal((T * k, h))
    lhs = np.sum(O.dispatch(x, p["token_ids"]) * u)
    rhs = np.sum(x * O.dispatch_bwd(u, p["slot_of"], k, None, "f64"))
    assert abs(lhs - rhs) < 1e-11 * (1 + abs(lhs))


def test_dispatch_then_dispatch_bwd_gives_k_times_x():
    T, E, k, h = 19, 7, 4, 3
    idx = _routing(T, E, k, 21)
    p = O.pft_build(idx, E)
    x = rng(22).standard_normal((T, h))
    np.testing.assert_allclose(O.dispatch_bwd(O.dispatch(x, p["token_ids"]), p["slot_of"], k, None, "f64"),
                               k * x, rtol=1e-14)


def test_combine_of_identity_experts_scales_by_weight_sum():
    T, E, k, h = 31, 8, 3, 6
    r = O.route_from_logits(rng(31).standard_normal((T, E)).astype(np.float32), k, "f64")
    p = O.pft_build(r["topk_idx"], E)
    x = rng(32).standard_normal((T, h))
    y = O.combine(O.dispatch(x, p["token_ids"]), p["slot_of"], r["topk_w"], "f64")
    np.testing.assert_allclose(y, r["topk_w"].sum(axis=1, keepdims=True) * x, rtol=1e-13)


def test_combine_bwd_adjoint_and_weight_gradient():
    T, E, k, h = 17, 5, 2, 4
    r = O.route_from_logits(rng(41).standard_normal((T, E)).astype(np.float32), k, "f64")
    p = O.pft_build(r["topk_idx"], E)
    u = rng(42).standard_normal((T * k, h))
    v = rng(43).standard_normal((T, h))
    dybuf, dw = O.combine_bwd(v, u, p["slot_of"], r["topk_w"], "f64")
    lhs = np.sum(O.combine(u, p["slot_of"], r["topk_w"], "f64") * v)
    assert abs(lhs - np.sum(u * dybuf)) < 1e-11 * (1 + abs(lhs))
    # d<combine(u; w), v>/dw by central differences
    eps = 1e-6
    for t, j in [(0, 0), (3, 1), (16, 0)]:
        wp = r["topk_w"].copy(); wp[t, j] += eps
        wm = r["topk_w"].copy(); wm[t, j] -= eps
        fd = (np.sum(O.combine(u, p["slot_of"], wp, "f64") * v)
              - np.sum(O.combine(u, p["slot_of"], wm, "f64") * v)) / (2 * eps)
        assert abs(fd - dw[t, j]) < 1e-7


# ----------------------------------------------------------------------------- experts


def test_swiglu_closed_form_case():
    g = json.load(open(os.path.join(GOLDEN, "swiglu_closed_form.json")))
    x = np.array(g["x"]); W1 = np.array(g["W1"]); W3 = np.array(g["W3"]); W2 = np.array(g["W2"])
    out = O.expert_ffn(x, np.array([0, 1]), W1, W3, W2, "f64")
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))  # noqa: E731
    a = np.array([2.0 * sig(2.0) * 3.0, 1.0 * sig(1.0) * -1.5])
    np.testing.assert_allclose(out["h1"][0], g["closed_form_terms"]["h1"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out["h3"][0], g["closed_form_terms"]["h3"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out["a"][0], a, rtol=1e-15)
    np.testing.assert_allclose(out["ybuf"][0], a[0] * W2[0, 0] + a[1] * W2[0, 1], rtol=1e-14)


@pytest.mark.parametrize("T,h,E,k,f,skew", [(24, 6, 4, 2, 5, False), (40, 8, 8, 3, 4, True)])
def test_pft_layer_equals_gshard_capacity_layer(T, h, E, k, f, skew):
    """X-MoE's claim: the padding-free layer is a lossless change of data structure, so the
    capacity-buffer layer with C = the largest load gives the same outputs."""
    g = rng(T + E)
    x = g.standard_normal((T, h)); Wg = g.standard_normal((h, E)) / math.sqrt(h)
    W1 = g.standard_normal((E, h, f)); W3 = g.standard_normal((E, h, f)); W2 = g.standard_normal((E, f, h))
    bias = -1.6 * np.log(np.arange(E) + 1.0) if skew else None
    fw = O.layer_forward(x, Wg, W1, W3, W2, k, bias, "f64")
    gs = O.gshard_layer_forward(x, Wg, W1, W3, W2, k, None, bias, "f64")
    np.testing.assert_allclose(gs["y"], fw["y"], rtol=1e-12, atol=1e-12)
    # the padded buffer holds the PFT buffer's rows at the same positions within each expert
    for e in range(E):
        n = fw["num_ids"][e]
        np.testing.assert_array_equal(gs["xe"][e, :n], fw["xbuf"][fw["offsets"][e]:fw["offsets"][e + 1]])
        assert (gs["xe"][e, n:] == 0).all()
    assert gs["C"] == fw["num_ids"].max()


def test_gshard_gate_by_brute_force_and_its_invariants():
    """Masks against a plain recount (slot = earlier tokens of the same expert), the drop rule
    at a capacity below the largest load, and the sums the masks must keep."""
    T, E, k = 30, 5, 2
    g = rng(11)
    idx = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    w = g.uniform(0.1, 1.0, (T, k))
    loads = np.bincount(idx.ravel(), minlength=E)
    for C in (int(loads.max()), int(loads.max()) - 3):
        m = O.gshard_capacity_gate(idx, w, E, C)
        np.testing.assert_array_equal(m["loads"], loads)
        kept = 0
        for t in range(T):
            for j in range(k):
                e = idx[t, j]
                c = sum(1 for u in range(t) if e in idx[u])
                if c < C:
                    assert m["dispatch_mask"][t, e, c] == 1.0 and m["combine_weights"][t, e, c] == w[t, j]
                    kept += 1
        assert m["dispatch_mask"].sum() == kept
        assert (m["dispatch_mask"].sum(axis=0) <= 1).all()  # one token per padded row
        if C == loads.max():
            assert kept == T * k
            np.testing.assert_allclose(m["combine_weights"].sum(axis=(1, 2)), w.sum(axis=1), rtol=1e-15)
        else:
            assert kept < T * k


def test_gshard_dispatch_and_combine_are_the_contractions():
    """One-hot masks make the contractions a gather and a weighted sum of picked rows."""
    T, E, C, h = 7, 3, 4, 5
    g = rng(12)
    x = g.standard_normal((T, h)); ye = g.standard_normal((E, C, h))
    mask = np.zeros((T, E, C)); cw = np.zeros((T, E, C))
    mask[2, 1, 0] = 1.0; mask[5, 1, 1] = 1.0; mask[0, 2, 3] = 1.0
    cw[2, 1, 0] = 0.25; cw[2, 0, 2] = 0.5; cw[6, 2, 1] = -2.0
    xe = O.gshard_dispatch(mask, x)
    np.testing.assert_array_equal(xe[1, 0], x[2]); np.testing.assert_array_equal(xe[1, 1], x[5])
    np.testing.assert_array_equal(xe[2, 3], x[0])
    assert np.count_nonzero(np.abs(xe).sum(axis=2)) == 3
    y = O.gshard_combine(cw, ye, "f64")
    np.testing.assert_allclose(y[2], 0.25 * ye[1, 0] + 0.5 * ye[0, 2], rtol=1e-15)
    np.testing.assert_allclose(y[6], -2.0 * ye[2, 1], rtol=1e-15)
    assert (y[[0, 1, 3, 4, 5]] == 0).all()


def test_identical_experts_scale_one_dense_ffn():
    T, h, E, k, f = 16, 5, 6, 3, 4
    g = rng(77)
    x = g.standard_normal((T, h)); Wg = g.standard_normal((h, E))
    w1 = g.standard_normal((h, f)); w3 = g.standard_normal((h, f)); w2 = g.standard_normal((f, h))
    W1 = np.stack([w1] * E); W3 = np.stack([w3] * E); W2 = np.stack([w2] * E)
    fw = O.layer_forward(x, Wg, W1, W3, W2, k, None, "f64")
    dense = O.expert_ffn(x, np.array([0, T]), W1[:1], W3[:1], W2[:1], "f64")["ybuf"]
    np.testing.assert_allclose(fw["y"], fw["topk_w"].sum(axis=1, keepdims=True) * dense, rtol=1e-12)


def test_empty_expert_gets_exact_zero_weight_gradient():
    T, h, E, k, f = 20, 4, 6, 2, 3
    g = rng(5)
    x = g.standard_normal((T, h)); Wg = g.standard_normal((h, E))
    W1 = g.standard_normal((E, h, f)); W3 = g.standard_normal((E, h, f)); W2 = g.standard_normal((E, f, h))
    bias = np.zeros(E); bias[E - 1] = -1e4  # nothing can choose the last expert
    fw = O.layer_forward(x, Wg, W1, W3, W2, k, bias, "bf16")
    assert fw["num_ids"][E - 1] == 0
    bw = O.layer_backward(fw, x, Wg, W1, W3, W2, g.standard_normal((T, h)), "bf16")
    for n in ("dW1", "dW3", "dW2"):
        assert (bw[n][E - 1] == 0).all() and np.abs(bw[n][:E - 1]).sum() > 0


# ----------------------------------------------------------------------------- gradients


@pytest.mark.parametrize("gate,renorm", [("softmax", False), ("softmax", True), ("sigmoid", False),
                                         ("sigmoid", True)])
def test_every_gradient_matches_central_finite_differences(gate, renorm):
    T, h, E, k, f = 5, 4, 4, 2, 3
    g = rng(2024)
    x = g.standard_normal((T, h)); Wg = g.standard_normal((h, E))
    W1 = g.standard_normal((E, h, f)) * 0.7; W3 = g.standard_normal((E, h, f)) * 0.7
    W2 = g.standard_normal((E, f, h)) * 0.7; dy = g.standard_normal((T, h))
    bias = np.array([0.3, -0.2, 0.0, 0.1])

    def loss(x_, Wg_, W1_, W3_, W2_):
        return np.sum(O.layer_forward(x_, Wg_, W1_, W3_, W2_, k, bias, "f64", gate, renorm)["y"] * dy)

    fw = O.layer_forward(x, Wg, W1, W3, W2, k, bias, "f64", gate, renorm)
    bw = O.layer_backward(fw, x, Wg, W1, W3, W2, dy, "f64")
    params = {"x": x, "Wg": Wg, "W1": W1, "W3": W3, "W2": W2}
    grads = {"x": bw["dx"], "Wg": bw["dWg"], "W1": bw["dW1"], "W3": bw["dW3"], "W2": bw["dW2"]}
    eps = 1e-6
    for name, P in params.items():
        fd = np.zeros_like(P)
        for i in itertools.product(*[range(s) for s in P.shape]):
            keep = P[i]
            P[i] = keep + eps
            lp = loss(x, Wg, W1, W3, W2)
            P[i] = keep - eps
            lm = loss(x, Wg, W1, W3, W2)
            P[i] = keep
            fd[i] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grads[name], fd, rtol=1e-6, atol=1e-8, err_msg=name)


def test_sigmoid_gate_closed_form_and_selection():
    l = rng(9).standard_normal((25, 6)) * 3
    r = O.route_from_logits(l, 3, "f64", gate="sigmoid")
    for t in range(25):
        for e in range(6):
            assert abs(r["probs"][t, e] - 1.0 / (1.0 + math.exp(-l[t, e]))) < 1e-15
    # the selection is the k largest scores (brute force on the scores themselves)
    np.testing.assert_array_equal(r["topk_idx"], brute_topk(r["probs"], 3))


@pytest.mark.parametrize("gate", ["softmax", "sigmoid"])
def test_renormalised_weights_sum_to_one_in_proportion(gate):
    l = rng(10).standard_normal((30, 8)).astype(np.float32)
    r = O.route_from_logits(l, 3, "f64", gate=gate, renorm=True)
    plain = O.route_from_logits(l, 3, "f64", gate=gate)
    np.testing.assert_array_equal(r["topk_idx"], plain["topk_idx"])
    np.testing.assert_allclose(r["topk_w"].sum(axis=1), 1.0, rtol=1e-14)
    ratio = r["topk_w"] / plain["topk_w"]
    np.testing.assert_allclose(ratio, ratio[:, :1] * np.ones_like(ratio), rtol=1e-13)


# ----------------------------------------------------------------------------- workloads


def test_workload_shapes_match_the_pages_model_table():
    from mixture_experts_layer_pft_gb300.workloads import WORKLOADS

    g = json.load(open(os.path.join(GOLDEN, "xmoe_model_table.json")))
    for w, name in zip(WORKLOADS[1:4] + WORKLOADS[5:6], ["Small", "Medium", "Large", "Super"]):
        s, hm, hf, E, k, _ = g["models"][name]
        assert (w.T, w.h, w.f, w.E, w.k) == (s, hm, hf, E, k)
    fl = g["flashdmoe"]
    w4 = WORKLOADS[4]
    assert w4.T == fl["max_seq_len"] and w4.k == fl["top_k"] and w4.E <= fl["max_experts"]
