"""CPU oracle for the padding-free (PFT) MoE layer: the plain definition of every stage.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or run this
module: only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It
shares no code with the CUDA library (no kernels, headers, helpers or tables) and is
written to be checked against the pages by eye, not to be fast.

What it computes, stage by stage, and where each stage comes from:

* Gating -- X-MoE review, §3 "Training pipeline" step 2 (padding-free gating) and the
  FlashDMoE blog, §1.1 "DMoE operator definition" (gating picks a few experts per
  token).  The pages fix no gate formula.  Reading adopted: router logits l = x·W_g
  (+ an optional fixed per-expert bias), softmax over all E experts, the k largest
  logits, descending, ties to the lower expert index; each selected expert's weight is
  its softmax probability, not renormalised.  Variants (FSMoE report, part 6: the system
  supports several routers, sigmoid among them): sigmoid scores instead of the softmax, and
  renormalising the k selected weights to sum to one.
* PFT build -- X-MoE review, §3 "Training pipeline" step 1 (flatten and sort the
  top_experts array into token_ids / expert_ids) and §3 "Model components" (the PFT
  holds token_ids, expert_ids, num_ids and only valid tokens).  Reading adopted: the
  sort key is (expert, token); num_ids[e] is the number of tokens routed to expert e;
  offsets is its exclusive prefix sum with E+1 entries; slot_of[t*k+j] is the buffer
  row that holds (token t, its j-th expert) -- the inverse permutation ("I-Order" in
  the FSMoE report, part 3, item 1).
* Dispatch -- X-MoE review, §3 "Training pipeline" step 3 and FlashDMoE blog §5
  "payload-efficient data handling": only routed tokens are moved, into one buffer with
  exactly T*k rows (X-MoE review, §3 "Core formulas": O(B x H) instead of O(E x C x H)).
* Expert compute -- X-MoE review, §3 "Training pipeline" step 5 (GEMMs over the uneven
  token buffer).  The pages give no FFN formula.  Reading adopted: SwiGLU,
  A = silu(X·W1[e]) * (X·W3[e]), Y = A·W2[e], silu(z) = z·sigmoid(z).
* Combine -- X-MoE review, §3 "Training pipeline" step 6 and FlashDMoE blog §1.1 (the
  expert outputs return to their token and are merged with the gate weights):
  y[t] = sum_j w[t,j] · ybuf[slot_of[t*k+j]], j ascending.
* Backward -- the pages describe none; each stage's backward is the textbook adjoint of
  its forward (chain rule, softmax Jacobian, SwiGLU derivative).
* Capacity-buffer baseline -- X-MoE review, §3 "Core formulas" (GShard-style dispatching
  holds an E x C x H buffer, C a fixed capacity) and §3 "Training pipeline" step 2 (the PFT
  gate avoids building a dispatch_mask).  Reading adopted: the gate turns the same top-k
  selection into dispatch_mask [T,E,C] and combine_weights [T,E,C]; a token's slot c in
  expert e's C rows is the number of earlier tokens that chose e; slots at or beyond C are
  dropped; dispatch is the contraction xe[e,c] = sum_t mask[t,e,c] x[t] and combine is
  y[t] = sum_{e,c} combine_weights[t,e,c] ye[e,c]; the experts run on all E*C padded rows.

Precision policy (``dtype``):

* ``"f64"``: nothing is rounded; used by the finite-difference pins.
* ``"f32"`` / ``"bf16"``: every product is accumulated in fp64, and each tensor is
  rounded to the storage type at the point where the layer stores it: gating tensors
  (logits, probabilities, gate weights, their gradients, dW_g and the router part of
  dx) to fp32; activations, expert intermediates (H1, H3, A), expert outputs and all
  other gradients to ``dtype``.  bf16 rounding is round-to-nearest-even applied to the
  fp32-rounded value, as a value held in an fp32 accumulator is stored.

Parity pins (tests marked "not gpu" check each of them): top-k against a brute-force
selection and constructed ties; softmax against the two-expert closed form; the PFT
arrays against a brute-force recount and the inverse-permutation identity; dispatch and
combine against identity experts and adjoint identities; the expert FFN against a
hand-derived SwiGLU case and the capacity-buffer formulation below (equal to the PFT layer);
every gradient against central finite differences in fp64; bf16 rounding against
hand-derived bit patterns and torch's own conversion.  No function here is unpinned.
"""

from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------- rounding


def round_f32(a):
    """Round to IEEE fp32 (round-to-nearest-even) and return float64 values."""
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_bf16(a):
    """Round to bfloat16 (8-bit mantissa, round-to-nearest-even) via fp32.

    bfloat16 is the upper 16 bits of an fp32 word.  Rounding adds 0x7FFF plus the lowest
    kept bit to the fp32 bit pattern and truncates, which rounds to nearest with ties to
    even.  NaN stays NaN (its payload is forced quiet).
    """
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + keep_lsb) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32).astype(np.float64)
    nan = np.isnan(f)
    if nan.any():
        out[nan] = np.nan
    return out


def store(a, dtype):
    """Round ``a`` to the storage type ``dtype`` ("f64", "f32" or "bf16")."""
    if dtype == "f64":
        return np.asarray(a, dtype=np.float64)
    if dtype == "f32":
        return round_f32(a)
    if dtype == "bf16":
        return round_bf16(a)
    raise ValueError(f"unknown dtype {dtype!r}")


def gate_store(a, dtype):
    """Gating tensors are fp32 whatever the activation type (fp64 only in "f64" mode)."""
    return np.asarray(a, dtype=np.float64) if dtype == "f64" else round_f32(a)


# ----------------------------------------------------------------------------- gating


def router_logits(x, Wg, bias=None, dtype="f32"):
    """l[t,e] = sum_c x[t,c]·W_g[c,e] (+ bias[e]), accumulated in fp64.

    The product is rounded to fp32 before the bias is added and the sum is rounded
    again, the two points where an fp32 layer holds the value.
    """
    l = gate_store(np.asarray(x, np.float64) @ np.asarray(Wg, np.float64), dtype)
    if bias is not None:
        l = gate_store(l + np.asarray(bias, np.float64)[None, :], dtype)
    return l


def softmax(logits):
    """p[t,e] = exp(l[t,e] - max_e l) / sum_e exp(l[t,e] - max_e l), in fp64."""
    l = np.asarray(logits, np.float64)
    z = np.exp(l - l.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def topk(logits, k):
    """Indices of the k largest logits per token, descending, ties to the lower index.

    A full stable sort of every token's (logit descending, index ascending) pairs; the
    first k entries are taken.  Softmax is monotone, so ranking the logits ranks the
    probabilities in exact arithmetic.
    """
    l = np.asarray(logits, np.float64)
    T, E = l.shape
    idx = np.empty((T, k), dtype=np.int32)
    e_ids = np.arange(E)
    for t in range(T):
        order = np.lexsort((e_ids, -l[t]))  # last key is primary: -logit, then index
        idx[t] = order[:k]
    return idx


def route(x, Wg, k, bias=None, dtype="f32", gate="softmax", renorm=False):
    """Gating stage: logits, probabilities, top-k expert ids and gate weights."""
    logits = router_logits(x, Wg, bias, dtype)
    return route_from_logits(logits, k, dtype, gate, renorm)


def route_from_logits(logits, k, dtype="f32", gate="softmax", renorm=False):
    """Scores, top-k selection and gate weights from the router logits.

    gate="softmax" (the layer's default): p = softmax over the E experts.  gate="sigmoid": each
    expert's score is p_e = sigmoid(l_e) on its own -- the FSMoE report (part 6, "highlights")
    lists a sigmoid router beside the GShard and X-MoE ones.  Both maps are monotone, so the
    selection is the k largest logits either way.  renorm=True divides the k selected scores
    by their sum (taken from the stored scores), so a token's gate weights add up to one.
    """
    l = np.asarray(logits, np.float64)
    p = softmax(l) if gate == "softmax" else sigmoid(l)
    probs = gate_store(p, dtype)
    idx = topk(logits, k)
    w = np.take_along_axis(probs, idx.astype(np.int64), axis=1)
    if renorm:
        w = gate_store(w / w.sum(axis=1, keepdims=True), dtype)
    return {"logits": l, "probs": probs, "topk_idx": idx, "topk_w": w}


# ----------------------------------------------------------------------------- PFT build


def pft_build(topk_idx, E):
    """Build the padding-free token buffer index arrays from top_experts [T,k].

    For e = 0..E-1 and, inside each e, t = 0..T-1 ascending: if token t chose expert e,
    append (t, e).  This is the sort of the flattened (token, expert) pairs by the key
    (expert, token), written as its plain definition.
    """
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, k = idx.shape
    token_ids, expert_ids = [], []
    num_ids = np.zeros(E, dtype=np.int32)
    for e in range(E):
        ts = np.nonzero((idx == e).any(axis=1))[0]  # ascending token order
        token_ids.extend(ts.tolist())
        expert_ids.extend([e] * len(ts))
        num_ids[e] = len(ts)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(num_ids)
    token_ids = np.asarray(token_ids, dtype=np.int32)
    expert_ids = np.asarray(expert_ids, dtype=np.int32)
    slot_of = np.full(T * k, -1, dtype=np.int32)
    for p in range(len(token_ids)):
        t, e = int(token_ids[p]), int(expert_ids[p])
        j = int(np.nonzero(idx[t] == e)[0][0])
        slot_of[t * k + j] = p
    return {"num_ids": num_ids, "offsets": offsets, "token_ids": token_ids,
            "expert_ids": expert_ids, "slot_of": slot_of}


# ----------------------------------------------------------------------------- dispatch


def dispatch(x, token_ids):
    """xbuf[p] = x[token_ids[p]]: one contiguous buffer of exactly T*k rows."""
    return np.asarray(x, np.float64)[np.asarray(token_ids, np.int64)]


def dispatch_bwd(dxbuf, slot_of, k, dx_add=None, dtype="f32"):
    """dx[t] = dx_add[t] + sum_j dxbuf[slot_of[t*k+j]] (adjoint of dispatch)."""
    slot = np.asarray(slot_of, np.int64)
    T = slot.shape[0] // k
    dxb = np.asarray(dxbuf, np.float64)
    acc = np.zeros((T, dxb.shape[1])) if dx_add is None else np.array(dx_add, np.float64)
    for j in range(k):
        acc = acc + dxb[slot[j::k]]
    return store(acc, dtype)


# ----------------------------------------------------------------------------- experts


def silu(z):
    return z / (1.0 + np.exp(-z))


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def expert_ffn(xbuf, offsets, W1, W3, W2, dtype="f32"):
    """Per-expert SwiGLU over the uneven segments rows [offsets[e], offsets[e+1]).

    H1 = X·W1[e], H3 = X·W3[e], A = silu(H1)*H3, Y = A·W2[e].  W1, W3 are [E,h,f] and
    W2 is [E,f,h].  H1, H3 and A are returned as stored (for the backward).
    """
    X = np.asarray(xbuf, np.float64)
    off = np.asarray(offsets, np.int64)
    E = off.shape[0] - 1
    f = W1.shape[2]
    Tk, h = X.shape
    H1 = np.zeros((Tk, f)); H3 = np.zeros((Tk, f)); A = np.zeros((Tk, f)); Y = np.zeros((Tk, h))
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        Xe = X[r0:r1]
        h1 = Xe @ np.asarray(W1[e], np.float64)
        h3 = Xe @ np.asarray(W3[e], np.float64)
        a = store(silu(h1) * h3, dtype)
        H1[r0:r1] = store(h1, dtype)
        H3[r0:r1] = store(h3, dtype)
        A[r0:r1] = a
        Y[r0:r1] = store(a @ np.asarray(W2[e], np.float64), dtype)
    return {"ybuf": Y, "h1": H1, "h3": H3, "a": A}


def expert_ffn_bwd(dybuf, xbuf, h1, h3, a, offsets, W1, W3, W2, dtype="f32"):
    """Backward of the per-expert SwiGLU, from the stored H1, H3 and A.

    dA = dY·W2[e]^T; dH1 = dA*H3*silu'(H1) with silu'(z) = s(z)(1 + z(1 - s(z)));
    dH3 = dA*silu(H1); dX = dH1·W1[e]^T + dH3·W3[e]^T; dW2[e] = A^T·dY;
    dW1[e] = X^T·dH1; dW3[e] = X^T·dH3.  An expert with no rows gets dW = 0.
    """
    dY = np.asarray(dybuf, np.float64)
    X = np.asarray(xbuf, np.float64)
    off = np.asarray(offsets, np.int64)
    E = off.shape[0] - 1
    Tk, h = X.shape
    f = W1.shape[2]
    dX = np.zeros((Tk, h))
    dW1 = np.zeros((E, h, f)); dW3 = np.zeros((E, h, f)); dW2 = np.zeros((E, f, h))
    dH1 = np.zeros((Tk, f)); dH3 = np.zeros((Tk, f))
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        z1 = np.asarray(h1[r0:r1], np.float64)
        z3 = np.asarray(h3[r0:r1], np.float64)
        dA = dY[r0:r1] @ np.asarray(W2[e], np.float64).T
        s = sigmoid(z1)
        d1 = store(dA * z3 * s * (1.0 + z1 * (1.0 - s)), dtype)
        d3 = store(dA * silu(z1), dtype)
        dH1[r0:r1] = d1
        dH3[r0:r1] = d3
        dX[r0:r1] = store(d1 @ np.asarray(W1[e], np.float64).T + d3 @ np.asarray(W3[e], np.float64).T, dtype)
        Xe = X[r0:r1]
        dW1[e] = store(Xe.T @ d1, dtype)
        dW3[e] = store(Xe.T @ d3, dtype)
        dW2[e] = store(np.asarray(a[r0:r1], np.float64).T @ dY[r0:r1], dtype)
    return {"dxbuf": dX, "dW1": dW1, "dW3": dW3, "dW2": dW2, "dh1": dH1, "dh3": dH3}


# ----------------------------------------------------------------------------- combine


def combine(ybuf, slot_of, topk_w, dtype="f32"):
    """y[t] = sum_{j ascending} w[t,j] · ybuf[slot_of[t*k+j]]."""
    w = np.asarray(topk_w, np.float64)
    T, k = w.shape
    slot = np.asarray(slot_of, np.int64)
    Yb = np.asarray(ybuf, np.float64)
    y = np.zeros((T, Yb.shape[1]))
    for j in range(k):
        y = y + w[:, j:j + 1] * Yb[slot[j::k]]
    return store(y, dtype)


def combine_bwd(dy, ybuf, slot_of, topk_w, dtype="f32"):
    """Adjoint of combine: dybuf[slot_of[t*k+j]] = w[t,j]·dy[t] and
    d_w[t,j] = <dy[t], ybuf[slot_of[t*k+j]]>."""
    w = np.asarray(topk_w, np.float64)
    T, k = w.shape
    slot = np.asarray(slot_of, np.int64)
    Yb = np.asarray(ybuf, np.float64)
    d = np.asarray(dy, np.float64)
    dybuf = np.zeros_like(Yb)
    dw = np.zeros((T, k))
    for j in range(k):
        rows = slot[j::k]
        dybuf[rows] = w[:, j:j + 1] * d
        dw[:, j] = np.einsum("th,th->t", d, Yb[rows])
    return store(dybuf, dtype), gate_store(dw, dtype)


# ----------------------------------------------------------------------------- gating bwd


def route_bwd(x, Wg, probs, topk_idx, d_topk_w, dtype="f32", gate="softmax", renorm=False):
    """Backward of the gate scores + top-k gate weights.

    Without renormalisation w[t,j] = p[t, idx[t,j]], so the gradient g with respect to the
    scores is d_w[t,j] at e = idx[t,j] and zero elsewhere.  With renormalisation
    w_j = p_j / S, S = sum of the selected scores, so g at the selected entries is
    (d_w_j - sum_i d_w_i w_i) / S.  Through the softmax Jacobian d_l = p*(g - sum_e p*g);
    through the sigmoid d_l = p*(1-p)*g.  Then dW_g = x^T·d_l and the router's share of dx is
    d_l·W_g^T.  The selection is piecewise constant and contributes no gradient.
    """
    p = np.asarray(probs, np.float64)
    T, E = p.shape
    idx = np.asarray(topk_idx, np.int64)
    dw = np.asarray(d_topk_w, np.float64)
    if renorm:
        sel = np.take_along_axis(p, idx, axis=1)
        S = sel.sum(axis=1, keepdims=True)
        dw = (dw - (dw * (sel / S)).sum(axis=1, keepdims=True)) / S
    g = np.zeros((T, E))
    np.put_along_axis(g, idx, dw, axis=1)
    if gate == "softmax":
        d_logits = p * (g - (p * g).sum(axis=1, keepdims=True))
    else:
        d_logits = p * (1.0 - p) * g
    d_logits = gate_store(d_logits, dtype)
    dWg = gate_store(np.asarray(x, np.float64).T @ d_logits, dtype)
    dx_router = gate_store(d_logits @ np.asarray(Wg, np.float64).T, dtype)
    return {"d_logits": d_logits, "dWg": dWg, "dx_router": dx_router}


# ----------------------------------------------------------------------------- layer


def layer_forward(x, Wg, W1, W3, W2, k, bias=None, dtype="f32", gate="softmax", renorm=False):
    """The whole forward pass: gate -> PFT build -> dispatch -> experts -> combine."""
    E = W1.shape[0]
    r = route(x, Wg, k, bias, dtype, gate, renorm)
    pft = pft_build(r["topk_idx"], E)
    xbuf = dispatch(x, pft["token_ids"])
    ffn = expert_ffn(xbuf, pft["offsets"], W1, W3, W2, dtype)
    y = combine(ffn["ybuf"], pft["slot_of"], r["topk_w"], dtype)
    out = dict(r)
    out.update(pft)
    out.update(ffn)
    out["xbuf"] = xbuf
    out["y"] = y
    out["gate"], out["renorm"] = gate, renorm
    return out


def layer_backward(fwd, x, Wg, W1, W3, W2, dy, dtype="f32"):
    """The whole backward pass, in reverse stage order, from a ``layer_forward`` result."""
    k = fwd["topk_idx"].shape[1]
    dybuf, d_w = combine_bwd(dy, fwd["ybuf"], fwd["slot_of"], fwd["topk_w"], dtype)
    eb = expert_ffn_bwd(dybuf, fwd["xbuf"], fwd["h1"], fwd["h3"], fwd["a"], fwd["offsets"],
                        W1, W3, W2, dtype)
    rb = route_bwd(x, Wg, fwd["probs"], fwd["topk_idx"], d_w, dtype, fwd.get("gate", "softmax"),
                   fwd.get("renorm", False))
    dx = dispatch_bwd(eb["dxbuf"], fwd["slot_of"], k, rb["dx_router"], dtype)
    out = {"dybuf": dybuf, "d_topk_w": d_w, "dx": dx}
    out.update(eb)
    out.update(rb)
    return out



# ----------------------------------------------------------------------------- capacity-buffer baseline


def gshard_capacity_gate(topk_idx, topk_w, E, C):
    """dispatch_mask, combine_weights [T,E,C] and per-expert loads from a top-k selection.

    The token-by-expert choice matrix is scanned down the tokens: token t's slot in expert e is
    the number of tokens before t that chose e.  Each (t, j) with slot c < C sets
    dispatch_mask[t,e,c] = 1 and combine_weights[t,e,c] = topk_w[t,j]; a slot at or beyond the
    capacity is dropped.  loads[e] counts every token that chose e, dropped or not."""
    idx = np.asarray(topk_idx, np.int64)
    w = np.asarray(topk_w, np.float64)
    T, k = idx.shape
    chose = np.zeros((T, E))
    for j in range(k):
        chose[np.arange(T), idx[:, j]] = 1.0
    slot = np.cumsum(chose, axis=0) - chose  # tokens before t that chose e
    mask = np.zeros((T, E, C))
    cw = np.zeros((T, E, C))
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            c = int(slot[t, e])
            if c < C:
                mask[t, e, c] = 1.0
                cw[t, e, c] = w[t, j]
    return {"dispatch_mask": mask, "combine_weights": cw, "loads": chose.sum(axis=0).astype(np.int64)}


def gshard_dispatch(dispatch_mask, x):
    """xe[e,c,:] = sum_t dispatch_mask[t,e,c] * x[t,:]: the padded [E,C,h] expert buffer."""
    return np.einsum("tec,th->ech", np.asarray(dispatch_mask, np.float64), np.asarray(x, np.float64))


def gshard_combine(combine_weights, ye, dtype="f32"):
    """y[t,:] = sum_{e,c} combine_weights[t,e,c] * ye[e,c,:], rounded once."""
    y = np.einsum("tec,ech->th", np.asarray(combine_weights, np.float64), np.asarray(ye, np.float64))
    return store(y, dtype)


def gshard_layer_forward(x, Wg, W1, W3, W2, k, C=None, bias=None, dtype="f32"):
    """The capacity-buffer forward: gate -> masks -> padded dispatch -> experts on all E*C rows
    -> combine.  C defaults to the largest expert load, so no token is dropped."""
    E = W1.shape[0]
    r = route(x, Wg, k, bias, dtype)
    if C is None:
        C = int(np.bincount(r["topk_idx"].ravel(), minlength=E).max())
    g = gshard_capacity_gate(r["topk_idx"], r["topk_w"], E, C)
    xe = gshard_dispatch(g["dispatch_mask"], x)
    h = xe.shape[2]
    ffn = expert_ffn(xe.reshape(E * C, h), np.arange(E + 1) * C, W1, W3, W2, dtype)
    ye = ffn["ybuf"].reshape(E, C, h)
    out = dict(r)
    out.update(g)
    out.update({"C": C, "xe": xe, "ye": ye, "y": gshard_combine(g["combine_weights"], ye, dtype)})
    return out
