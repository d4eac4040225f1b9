"""Whole-layer parity: the GPU step (forward + backward, as the benchmark runs it) against the
oracle on the same seeded workload.

Small workloads are compared in full.  At the full sizes the oracle recomputes a seeded
sample of tokens (every token's outputs depend only on its own input and the weights) and
the weight gradients of a few sampled experts.

The router logits are fp32 sums on the GPU and exact sums in the oracle; a token whose
top-(k+1) logits lie closer than the rounding error admits several correct selections.
Those tokens are checked for validity and left out of the element-wise comparison, as are
experts whose token set depends on them.
"""

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from helpers import TOL, check_valid_topk, dtype_name, np64, npi, rel_l2, unambiguous_tokens
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from mixture_experts_layer_pft_gb300 import build, layer, workloads

    build.build()
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    return layer, workloads


class LazyExperts:
    """Stacked expert weights on the GPU, handed to the oracle one expert at a time."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, e):
        return np64(self.t[e])


def gpu_step(M, w, T=None):
    layer, workloads = M
    inp = workloads.make_inputs(w, "cuda", T=T)
    T_ = inp["x"].shape[0]
    b = layer.LayerBuffers(T_, w.h, w.E, w.k, w.f, w.torch_dtype(), backward=w.backward)
    layer.step(inp, b)
    torch.cuda.synchronize()
    return inp, b


def routing_checks(b, exact, k):
    """GPU logits within rounding of the exact ones; selection unique where it must be."""
    err = np.abs(np64(b.logits) - exact).max()
    assert err < 1e-3, err
    delta = 2.0 * err + 1e-7
    una = unambiguous_tokens(exact, k, delta)
    check_valid_topk(npi(b.topk_idx), exact, k, delta)
    exact_idx = O.topk(exact, k)
    np.testing.assert_array_equal(npi(b.topk_idx)[una], exact_idx[una])
    return una


@pytest.mark.parametrize("cfg", [0, 1])
def test_full_layer_small_workloads(M, cfg):
    _, workloads = M
    w = workloads.WORKLOADS[cfg]
    dn = w.dtype
    inp, b = gpu_step(M, w)
    x, Wg = np64(inp["x"]), np64(inp["Wg"])
    bias = None if inp["bias"] is None else np64(inp["bias"])
    W1, W3, W2, dy = np64(inp["W1"]), np64(inp["W3"]), np64(inp["W2"]), np64(inp["dy"])
    fw = O.layer_forward(x, Wg, W1, W3, W2, w.k, bias, dn)
    bw = O.layer_backward(fw, x, Wg, W1, W3, W2, dy, dn)
    exact = O.router_logits(x, Wg, bias, "f64")
    una = routing_checks(b, exact, w.k)
    assert rel_l2(np64(b.logits), fw["logits"]) <= TOL["f32"]
    check_layer_against_oracle(b, fw, bw, una, npi(b.topk_idx), O.topk(exact, w.k), w.E, dn)
    if not una.all():
        pytest.skip(f"{(~una).sum()} tokens with near-tied logits: compared token by token above")
    for n in ("num_ids", "offsets", "token_ids", "expert_ids", "slot_of"):
        np.testing.assert_array_equal(npi(getattr(b, n)), fw[n], err_msg=n)
    if b.xbuf is not None:  # the fused layer never writes the dispatched buffer
        np.testing.assert_array_equal(np64(b.xbuf), fw["xbuf"])
    for n in ("probs", "topk_w"):
        assert rel_l2(np64(getattr(b, n)), fw[n]) <= TOL["f32"], n
    # stored in fp32, but d_topk_w = <dy, ybuf> carries ybuf's rounding in the layer's dtype,
    # and the gate gradients below it inherit that
    for n in ("d_topk_w", "d_logits", "dWg", "dx_router"):
        assert rel_l2(np64(getattr(b, n)), bw[n]) <= TOL[dn], n
    for n in ("h1", "h3", "a", "ybuf", "y"):
        assert rel_l2(np64(getattr(b, n)), fw[n]) <= TOL[dn], n
    for n in ("dybuf", "dxbuf", "dW1", "dW3", "dW2", "dx"):
        assert rel_l2(np64(getattr(b, n)), bw[n]) <= TOL[dn], n


def _sample_unambiguous(n, una, seed):
    """n unambiguous tokens in a seeded order, plus the first and last token when unambiguous."""
    T = una.shape[0]
    g = np.random.default_rng(seed)
    cand = [t for t in g.permutation(T) if una[t]][:n]
    cand += [t for t in (0, T - 1) if una[t]]
    return np.array(sorted(set(int(t) for t in cand)))


def oracle_token_rows(x_s, Wg, bias, W1, W3, W2, k, dn, dy_s=None):
    """The oracle's layer on a token sample, stage by stage as layer_forward / layer_backward
    compose it, with the expert backward run one expert at a time (so no E x h x f array of
    weight gradients is allocated).  Every per-token output (y, dx, the token's buffer rows) depends
    only on that token and the weights, so these rows equal the full layer's rows."""
    E = W1.shape[0]
    r = O.route(x_s, Wg, k, bias, dn)
    pft = O.pft_build(r["topk_idx"], E)
    xbuf = O.dispatch(x_s, pft["token_ids"])
    off = pft["offsets"]
    experts = np.nonzero(np.diff(off))[0]

    def one(t, e):
        return LazyExperts(t.t[e:e + 1]) if isinstance(t, LazyExperts) else t[e:e + 1]

    # the oracle's expert stages one expert segment at a time (each expert's rows depend on that
    # expert alone), several experts at once on the host's cores
    def fwd(e):
        return e, O.expert_ffn(xbuf[off[e]:off[e + 1]], np.array([0, off[e + 1] - off[e]]), one(W1, e), one(W3, e),
                               one(W2, e), dn)

    Tk_s, h = xbuf.shape
    f = W1.shape[2]
    ffn = {"h1": np.zeros((Tk_s, f)), "h3": np.zeros((Tk_s, f)), "a": np.zeros((Tk_s, f)),
           "ybuf": np.zeros((Tk_s, h))}
    with ThreadPoolExecutor(max_workers=8) as ex:
        for e, res in ex.map(fwd, experts):
            for n in ffn:
                ffn[n][off[e]:off[e + 1]] = res[n]
    out = dict(r)
    out.update(pft)
    out.update(ffn)
    out["xbuf"] = xbuf
    out["y"] = O.combine(ffn["ybuf"], pft["slot_of"], r["topk_w"], dn)
    if dy_s is None:
        return out
    dybuf, d_w = O.combine_bwd(dy_s, ffn["ybuf"], pft["slot_of"], r["topk_w"], dn)
    dxbuf, dh1, dh3 = np.zeros((Tk_s, h)), np.zeros((Tk_s, f)), np.zeros((Tk_s, f))

    def bwd(e):
        sl = slice(off[e], off[e + 1])
        return e, O.expert_ffn_bwd(dybuf[sl], xbuf[sl], ffn["h1"][sl], ffn["h3"][sl], ffn["a"][sl],
                                   np.array([0, off[e + 1] - off[e]]), one(W1, e), one(W3, e), one(W2, e), dn)

    with ThreadPoolExecutor(max_workers=8) as ex:
        for e, eb in ex.map(bwd, experts):
            sl = slice(off[e], off[e + 1])
            dxbuf[sl], dh1[sl], dh3[sl] = eb["dxbuf"], eb["dh1"], eb["dh3"]
    rb = O.route_bwd(x_s, Wg, r["probs"], r["topk_idx"], d_w, dn)
    out.update({"dybuf": dybuf, "d_topk_w": d_w, "dxbuf": dxbuf, "dh1": dh1, "dh3": dh3,
                "d_logits": rb["d_logits"], "dx_router": rb["dx_router"],
                "dx": O.dispatch_bwd(dxbuf, pft["slot_of"], k, rb["dx_router"], dn)})
    return out


def take(t: torch.Tensor, idx) -> torch.Tensor:
    """Rows idx (a numpy integer array) of a device tensor."""
    return t[torch.as_tensor(np.asarray(idx, np.int64), device=t.device)]


def assert_rows_close(got, want, tol, what):
    """rel-L2 <= tol on every row on its own, so one wrong row cannot hide in a norm."""
    got, want = np.atleast_2d(got), np.atleast_2d(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    for i in range(got.shape[0]):
        r = rel_l2(got[i], want[i])
        assert r <= tol, (what, i, r)


def check_sampled_tokens(b, inp, w, S, dn):
    """GPU outputs on the token sample S (unambiguous tokens) against the oracle's rows."""
    x, Wg = np64(inp["x"]), np64(inp["Wg"])
    bias = None if inp["bias"] is None else np64(inp["bias"])
    W1, W3, W2 = LazyExperts(inp["W1"]), LazyExperts(inp["W3"]), LazyExperts(inp["W2"])
    dy_s = np64(take(inp["dy"], S)) if b.backward else None
    o = oracle_token_rows(x[S], Wg, bias, W1, W3, W2, w.k, dn, dy_s)
    np.testing.assert_array_equal(npi(take(b.topk_idx, S)), o["topk_idx"])
    assert_rows_close(np64(take(b.y, S)), o["y"], TOL[dn], "y")
    assert_rows_close(np64(take(b.topk_w, S)), o["topk_w"], TOL["f32"], "topk_w")
    assert_rows_close(np64(take(b.probs, S)), o["probs"], TOL["f32"], "probs")
    # the token's k buffer rows: GPU row slot_of[t*k+j] against the sample's row for (s, j)
    g_rows = npi(b.slot_of).reshape(-1, w.k)[S].ravel()
    o_rows = o["slot_of"]
    np.testing.assert_array_equal(npi(b.token_ids)[g_rows], np.repeat(S, w.k))
    np.testing.assert_array_equal(npi(b.expert_ids)[g_rows], o["expert_ids"][o_rows])
    for n in ("h1", "h3", "a", "ybuf"):
        assert_rows_close(np64(take(getattr(b, n), g_rows)), o[n][o_rows], TOL[dn], n)
    if b.xbuf is not None:
        np.testing.assert_array_equal(np64(take(b.xbuf, g_rows)), o["xbuf"][o_rows])
    if not b.backward:
        return
    assert_rows_close(np64(take(b.dx, S)), o["dx"], TOL[dn], "dx")
    assert_rows_close(np64(take(b.dybuf, g_rows)), o["dybuf"][o_rows], TOL[dn], "dybuf")
    assert_rows_close(np64(take(b.dxbuf, g_rows)), o["dxbuf"][o_rows], TOL[dn], "dxbuf")
    # fp32 gate gradients carry ybuf's rounding in the layer's dtype (d_w = <dy, ybuf>)
    assert rel_l2(np64(take(b.d_topk_w, S)), o["d_topk_w"]) <= TOL[dn]
    assert rel_l2(np64(take(b.d_logits, S)), o["d_logits"]) <= TOL[dn]
    assert rel_l2(np64(take(b.dx_router, S)), o["dx_router"]) <= TOL[dn]


def check_router_gemms_at_full_size(b, inp):
    """The router GEMMs are fp32 sums of exact products: dW_g = x^T d_logits and the router's
    part of dx = d_logits W_g^T, checked against the definition in fp64 on the GPU's own d_logits
    (a property that holds at any size)."""
    x, Wg, dl = np64(inp["x"]), np64(inp["Wg"]), np64(b.d_logits)
    assert rel_l2(np64(b.dWg), x.T @ dl) <= TOL["f32"]
    assert rel_l2(np64(b.dx_router), dl @ Wg.T) <= TOL["f32"]


def unambiguous_experts(exact_idx, gpu_idx, una, E):
    """Experts every one of whose tokens -- in the exact routing and in the GPU's -- is
    unambiguous: their token sets are unique, so their weight gradients have one correct value."""
    amb = ~una
    touched_by_ambiguous = np.zeros(E, bool)
    touched_by_ambiguous[exact_idx[amb].ravel()] = True
    touched_by_ambiguous[gpu_idx[amb].ravel()] = True
    used = np.bincount(exact_idx.ravel(), minlength=E) > 0
    return np.nonzero(used & ~touched_by_ambiguous)[0]


def check_sampled_experts(b, inp, w, exact, una, nexp, seed, dn):
    """Weight gradients of nexp seeded experts whose token sets are unambiguous, each against the
    oracle's single-expert forward and backward over exactly that expert's tokens."""
    x, Wg = np64(inp["x"]), np64(inp["Wg"])
    bias = None if inp["bias"] is None else np64(inp["bias"])
    dy = np64(inp["dy"])
    tok, off = npi(b.token_ids), npi(b.offsets)
    ex_idx = O.topk(exact, w.k)
    eligible = unambiguous_experts(ex_idx, npi(b.topk_idx), una, w.E)
    assert len(eligible) >= nexp // 2, f"only {len(eligible)} experts with unambiguous token sets"
    nexp = min(nexp, len(eligible))
    g = np.random.default_rng(seed)
    checked = 0
    for e in g.permutation(eligible):
        toks = np.nonzero((ex_idx == e).any(axis=1))[0]
        np.testing.assert_array_equal(tok[off[e]:off[e + 1]], toks)
        r = O.route(x[toks], Wg, w.k, bias, dn)
        wts = r["probs"][:, e]
        xe = x[toks]
        dyb = O.store(wts[:, None] * dy[toks], dn)
        one = np.array([0, len(toks)])
        We = [LazyExperts(inp[n][e:e + 1]) for n in ("W1", "W3", "W2")]
        f1 = O.expert_ffn(xe, one, *We, dn)
        gb = O.expert_ffn_bwd(dyb, xe, f1["h1"], f1["h3"], f1["a"], one, *We, dn)
        for n in ("dW1", "dW3", "dW2"):
            assert rel_l2(np64(getattr(b, n)[e]), gb[n][0]) <= TOL[dn], (n, e)
        checked += 1
        if checked == nexp:
            break
    assert checked == nexp
    empty = np.nonzero(npi(b.num_ids) == 0)[0]
    for e in empty[:4]:
        assert (np64(b.dW1[e]) == 0).all() and (np64(b.dW2[e]) == 0).all()


@pytest.mark.parametrize("cfg,ntok,nexp", [(2, 64, 16), (3, 64, 16), (4, 64, 0), (5, 64, 16)])
def test_full_size_layer_sampled(M, cfg, ntok, nexp):
    """The benchmark's full-size layers: 64 unambiguous tokens row by row (outputs, the tokens'
    buffer rows, gate gradients), the router GEMMs against their definition, and the weight
    gradients of 16 sampled experts."""
    _, workloads = M
    w = workloads.WORKLOADS[cfg]
    dn = w.dtype
    inp, b = gpu_step(M, w)
    x, Wg = np64(inp["x"]), np64(inp["Wg"])
    bias = None if inp["bias"] is None else np64(inp["bias"])
    exact = O.router_logits(x, Wg, bias, "f64")
    una = routing_checks(b, exact, w.k)
    assert rel_l2(np64(b.logits), O.router_logits(x, Wg, bias, "f32")) <= TOL["f32"]
    # invariants of the PFT arrays at full size
    Tk = w.T * w.k
    off = npi(b.offsets)
    assert off[0] == 0 and off[-1] == Tk and (np.diff(off) == npi(b.num_ids)).all()
    tok, slot, idx = npi(b.token_ids), npi(b.slot_of), npi(b.topk_idx)
    assert (tok[slot] == np.repeat(np.arange(w.T), w.k)).all()
    assert (npi(b.expert_ids)[slot] == idx.ravel()).all()

    S = _sample_unambiguous(ntok, una, cfg)
    assert len(S) >= ntok, f"only {len(S)} unambiguous sampled tokens"
    check_sampled_tokens(b, inp, w, S, dn)
    if not w.backward:
        return
    check_router_gemms_at_full_size(b, inp)
    check_sampled_experts(b, inp, w, exact, una, nexp, 100 + cfg, dn)


def test_full_size_fused_fp32_forward_sampled(M):
    """The long-sequence fp32 forward at full size (T = 16384) with the dispatch folded into the
    row split: 64 unambiguous tokens row by row against the oracle, and every output bit for bit
    against the layer with the dispatch call."""
    layer, workloads = M
    w = workloads.WORKLOADS[4]
    inp = workloads.make_inputs(w, "cuda")
    outs = []
    for fused in (False, True):
        b = layer.LayerBuffers(w.T, w.h, w.E, w.k, w.f, torch.float32, backward=False, fused=fused)
        layer.step(inp, b)
        torch.cuda.synchronize()
        assert binding_status(b) == 0
        outs.append(b)
    ref, b = outs
    for n in ("ybuf", "h1", "h3", "a", "y"):
        assert torch.equal(getattr(b, n), getattr(ref, n)), n
    x, Wg = np64(inp["x"]), np64(inp["Wg"])
    bias = None if inp["bias"] is None else np64(inp["bias"])
    una = routing_checks(b, O.router_logits(x, Wg, bias, "f64"), w.k)
    S = _sample_unambiguous(64, una, 44)
    assert len(S) >= 64, f"only {len(S)} unambiguous sampled tokens"
    check_sampled_tokens(b, inp, w, S, "f32")


@pytest.mark.parametrize("T,h,E,k,f,dt", [(1, 128, 8, 2, 64, torch.float32), (5, 64, 4, 4, 16, torch.bfloat16),
                                          (33, 72, 12, 12, 24, torch.float32), (17, 256, 4, 1, 128, torch.bfloat16),
                                          (300, 256, 4, 4, 256, torch.bfloat16)])  # k = E on the tensor cores
def test_edge_case_layers(M, T, h, E, k, f, dt):
    layer, workloads = M
    w = workloads.Workload("edge", T, h, E, k, f, dtype_name(dt), False, True, 7)
    inp, b = gpu_step(M, w)
    dn = dtype_name(dt)
    x, Wg = np64(inp["x"]), np64(inp["Wg"])
    W1, W3, W2, dy = np64(inp["W1"]), np64(inp["W3"]), np64(inp["W2"]), np64(inp["dy"])
    exact = O.router_logits(x, Wg, None, "f64")
    una = routing_checks(b, exact, k)
    if not una.all():
        pytest.skip("near-tied logits")
    fw = O.layer_forward(x, Wg, W1, W3, W2, k, None, dn)
    bw = O.layer_backward(fw, x, Wg, W1, W3, W2, dy, dn)
    assert rel_l2(np64(b.y), fw["y"]) <= TOL[dn]
    for n in ("dx", "dW1", "dW3", "dW2"):
        assert rel_l2(np64(getattr(b, n)), bw[n]) <= TOL[dn], n
    assert rel_l2(np64(b.dWg), bw["dWg"]) <= TOL[dn]


@pytest.mark.parametrize("gate,renorm,dt", [("sigmoid", True, torch.float32), ("softmax", True, torch.bfloat16),
                                           ("sigmoid", False, torch.bfloat16)])
def test_layer_with_router_variants(M, gate, renorm, dt):
    layer, workloads = M
    w = workloads.Workload("variant", 192, 256, 16, 4, 128, dtype_name(dt), True, True, 11)
    inp = workloads.make_inputs(w, "cuda")
    b = layer.LayerBuffers(w.T, w.h, w.E, w.k, w.f, dt, gate=gate, renorm=renorm)
    layer.step(inp, b)
    torch.cuda.synchronize()
    dn = dtype_name(dt)
    x, Wg, bias = np64(inp["x"]), np64(inp["Wg"]), np64(inp["bias"])
    W1, W3, W2, dy = np64(inp["W1"]), np64(inp["W3"]), np64(inp["W2"]), np64(inp["dy"])
    exact = O.router_logits(x, Wg, bias, "f64")
    una = routing_checks(b, exact, w.k)
    if not una.all():
        pytest.skip("near-tied logits")
    fw = O.layer_forward(x, Wg, W1, W3, W2, w.k, bias, dn, gate, renorm)
    bw = O.layer_backward(fw, x, Wg, W1, W3, W2, dy, dn)
    assert rel_l2(np64(b.topk_w), fw["topk_w"]) <= TOL["f32"]
    assert rel_l2(np64(b.y), fw["y"]) <= TOL[dn]
    for n in ("dx", "dW1", "dW2", "dWg", "d_logits"):
        assert rel_l2(np64(getattr(b, n)), bw[n]) <= TOL[dn], n


def test_layer_step_is_bitwise_deterministic(M):
    layer, workloads = M
    w = workloads.WORKLOADS[1]
    inp = workloads.make_inputs(w, "cuda")
    b = layer.LayerBuffers(w.T, w.h, w.E, w.k, w.f, w.torch_dtype())
    outs = []
    for _ in range(2):
        layer.step(inp, b)
        torch.cuda.synchronize()
        outs.append([getattr(b, n).clone() for n in ("y", "dx", "dW1", "dW2", "dWg", "slot_of")])
    for a, c in zip(*outs):
        assert torch.equal(a, c)


@pytest.mark.parametrize("cfg", [1, 4])
def test_host_buffer_step_equals_device_step(M, cfg):
    """step_host (pinned host tokens in, outputs back, copies overlapped on a second stream)
    gives the same bits as the device-resident step, over two back-to-back steps."""
    layer, workloads = M
    w = workloads.WORKLOADS[cfg]
    T = min(w.T, 2048)
    inp = workloads.make_inputs(w, "cuda", T=T)
    b = layer.LayerBuffers(T, w.h, w.E, w.k, w.f, w.torch_dtype(), backward=w.backward)
    layer.step(inp, b)
    torch.cuda.synchronize()
    want_y = b.y.cpu()
    want_dx = b.dx.cpu() if w.backward else None
    hx = inp["x"].cpu().pin_memory()
    hdy = inp["dy"].cpu().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    hdx = torch.empty_like(hx).pin_memory() if w.backward else None
    for _ in range(2):
        inp["x"].zero_()
        inp["dy"].zero_()
        b.y.zero_()
        hy.zero_()
        layer.step_host(inp, b, hx, hy, hdy, hdx)
        torch.cuda.current_stream().synchronize()
        assert torch.equal(hy, want_y)
        if w.backward:
            assert torch.equal(hdx, want_dx)


@pytest.mark.parametrize("graphs", [True, False])
@pytest.mark.parametrize("cfg", [0, 1, 4])
def test_host_pipeline_equals_device_steps(M, cfg, graphs):
    """HostPipeline over four different batches (two device slots, uploads and downloads on
    copy streams beside the compute): each batch's y and dx are the bits of a device-resident
    step on that batch."""
    layer, workloads = M
    w = workloads.WORKLOADS[cfg]
    T = min(w.T, 2048)
    batches = []
    for i in range(4):  # the same weights, different tokens; one copy of the weights kept
        inp = workloads.make_inputs(w, "cuda", T=T, token_seed=500 + i)
        batches.append(inp if i == 0 else dict(batches[0], x=inp["x"], dy=inp["dy"]))
        del inp
    b = layer.LayerBuffers(T, w.h, w.E, w.k, w.f, w.torch_dtype(), backward=w.backward)
    want = []
    for inp in batches:
        layer.step(inp, b)
        torch.cuda.synchronize()
        want.append((b.y.cpu(), b.dx.cpu() if w.backward else None))
    host = [(inp["x"].cpu().pin_memory(), inp["dy"].cpu().pin_memory()) for inp in batches]
    outs = [(torch.zeros_like(hx).pin_memory(), torch.zeros_like(hx).pin_memory() if w.backward else None)
            for hx, _ in host]
    weights = dict(batches[0], x=torch.zeros_like(batches[0]["x"]), dy=torch.zeros_like(batches[0]["dy"]))
    pipe = layer.HostPipeline(weights, b, graphs=graphs)
    for (hx, hdy), (hy, hdx) in zip(host, outs):
        pipe.submit(hx, hy, hdy, hdx)
    pipe.finish()
    torch.cuda.current_stream().synchronize()
    for i, ((hy, hdx), (wy, wdx)) in enumerate(zip(outs, want)):
        assert torch.equal(hy, wy), i
        if w.backward:
            assert torch.equal(hdx, wdx), i


def test_captured_step_replays_the_same_bits(M):
    """CapturedStep (the step as one CUDA graph) reproduces the stream-launched step exactly."""
    layer, workloads = M
    w = workloads.WORKLOADS[1]
    inp = workloads.make_inputs(w, "cuda")
    b = layer.LayerBuffers(w.T, w.h, w.E, w.k, w.f, w.torch_dtype())
    names = ("y", "dx", "dW1", "dW3", "dW2", "dWg", "slot_of")
    layer.step(inp, b)
    torch.cuda.synchronize()
    want = [getattr(b, n).clone() for n in names]
    g = layer.CapturedStep(lambda: layer.step(inp, b))
    assert g.launches >= 15
    for _ in range(2):
        for n in names:
            getattr(b, n).zero_()
        g.replay()
        torch.cuda.synchronize()
        for n, t in zip(names, want):
            assert torch.equal(getattr(b, n), t), n


@pytest.mark.parametrize("cfg", [1, 2])
def test_fused_layer_equals_dispatched_layer(M, cfg):
    """Dispatch folded into the expert GEMMs, the combine folded into the down projection, or
    both, give the same bits as the separate calls."""
    layer, workloads = M
    w = workloads.WORKLOADS[cfg]
    T = min(w.T, 2048)
    inp = workloads.make_inputs(w, "cuda", T=T)
    outs = []
    for fused, fold in ((False, False), (True, False), (False, True), (True, True)):
        b = layer.LayerBuffers(T, w.h, w.E, w.k, w.f, w.torch_dtype(), fused=fused, fold_combine=fold)
        assert b.fused == fused and (b.xbuf is None) == fused
        layer.step(inp, b)
        torch.cuda.synchronize()
        outs.append({n: getattr(b, n).clone() for n in ("ybuf", "h1", "h3", "a", "y", "dxbuf", "dW1", "dW3",
                                                        "dW2", "dWg", "dx")})
        del b
    for o in outs[1:]:
        for n, t in outs[0].items():
            assert torch.equal(o[n], t), n


@pytest.mark.parametrize("shape", [("longseq", 2048, 2048, 128, 2, 2048, True, False),
                                   ("fp32-fwd-bwd", 600, 256, 12, 3, 384, False, True)])
def test_fused_fp32_layer_equals_dispatched_layer(M, shape):
    """fp32 on the tensor cores: the layer whose expert FFN gathers its rows from x (the forward
    splits them into planes, the backward gathers them into dxbuf) gives the same bits as the
    layer with a dispatch call, forward only at the long-sequence shape and fwd+bwd."""
    layer, workloads = M
    name, T, h, E, k, f, skew, bwd = shape
    w = workloads.Workload(name, T, h, E, k, f, "f32", skew, bwd, 40 + T)
    inp = workloads.make_inputs(w, "cuda")
    outs = []
    for fused in (False, True):
        b = layer.LayerBuffers(T, h, E, k, f, torch.float32, backward=bwd, fused=fused)
        assert (b.xbuf is None) == fused
        layer.step(inp, b)
        torch.cuda.synchronize()
        assert binding_status(b) == 0
        names = ("ybuf", "h1", "h3", "a", "y") + (("dxbuf", "dW1", "dW3", "dW2", "dWg", "dx") if bwd else ())
        outs.append({n: getattr(b, n).clone() for n in names})
        del b
    for n, t in outs[0].items():
        assert torch.equal(outs[1][n], t), n


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_empty_batch_layer(M, dt):
    """A step over zero tokens runs every stage, leaves nothing to route or combine and gives
    exactly zero weight gradients."""
    layer, workloads = M
    w = workloads.Workload("empty", 0, 256, 8, 2, 256, dtype_name(dt), False, True, 9)
    inp = workloads.make_inputs(w, "cuda")
    b = layer.LayerBuffers(0, w.h, w.E, w.k, w.f, dt)
    for n in ("dW1", "dW3", "dW2", "dWg"):
        getattr(b, n).fill_(1.0)
    layer.step(inp, b)
    torch.cuda.synchronize()
    assert b.y.shape == (0, w.h) and b.dx.shape == (0, w.h)
    assert int(b.offsets.abs().sum()) == 0 and int(b.num_ids.abs().sum()) == 0
    for n in ("dW1", "dW3", "dW2", "dWg"):
        assert int(torch.count_nonzero(getattr(b, n))) == 0, n


def _random_layer_shapes(n, seed):
    g = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        E = 4 * int(g.integers(1, 41))
        out.append((int(g.choice([1, 7, 64, 129, 300, 513, 1000, 2047])), 128 * int(g.integers(1, 7)), E,
                    int(g.integers(1, min(8, E) + 1)), 128 * int(g.integers(1, 7)), bool(g.random() < 0.4)))
    return out


def check_layer_against_oracle(v, fw, bw, una, gpu_idx, exact_idx, E, dn):
    """A whole layer step against the oracle's full layer: every unambiguous token row by row
    (y, dx and, with the token's own buffer rows, h1, h3, a, ybuf, dybuf, dxbuf), and every
    expert whose token set is unambiguous (dW1, dW3, dW2); all of it when no token is ambiguous."""
    S = np.nonzero(una)[0]
    if len(S):
        assert_rows_close(np64(take(v.y, S)), fw["y"][S], TOL[dn], "y")
        assert_rows_close(np64(take(v.dx, S)), bw["dx"][S], TOL[dn], "dx")
        k = gpu_idx.shape[1]
        g_rows = npi(v.slot_of).reshape(-1, k)[S].ravel()
        o_rows = fw["slot_of"].reshape(-1, k)[S].ravel()
        for n in ("h1", "h3", "a", "ybuf"):
            assert_rows_close(np64(take(getattr(v, n), g_rows)), fw[n][o_rows], TOL[dn], n)
        for n in ("dybuf", "dxbuf"):
            assert_rows_close(np64(take(getattr(v, n), g_rows)), bw[n][o_rows], TOL[dn], n)
    for e in unambiguous_experts(exact_idx, gpu_idx, una, E):
        for n in ("dW1", "dW3", "dW2"):
            assert rel_l2(np64(getattr(v, n)[e]), bw[n][e]) <= TOL[dn], (n, e)
    if una.all():
        assert rel_l2(np64(v.dWg), bw["dWg"]) <= TOL[dn]


@pytest.mark.parametrize("T,h,E,k,f,skew", _random_layer_shapes(24, 2024))
def test_random_bf16_layers(M, T, h, E, k, f, skew):
    """Seeded random shapes on the tensor-core path: the layer, the gathered layer and the
    combine-folded layers each against the oracle (unambiguous tokens and experts), and the
    folded layers bit for bit against the layer with separate calls."""
    layer, workloads = M
    w = workloads.Workload("random", T, h, E, k, f, "bf16", skew, True, T + h + E)
    inp = workloads.make_inputs(w, "cuda")
    b = layer.LayerBuffers(T, h, E, k, f, torch.bfloat16)
    layer.step(inp, b)
    torch.cuda.synchronize()
    x, Wg = np64(inp["x"]), np64(inp["Wg"])
    bias = None if inp["bias"] is None else np64(inp["bias"])
    exact = O.router_logits(x, Wg, bias, "f64")
    una = routing_checks(b, exact, k)
    W1, W3, W2, dy = np64(inp["W1"]), np64(inp["W3"]), np64(inp["W2"]), np64(inp["dy"])
    fw = O.layer_forward(x, Wg, W1, W3, W2, k, bias, "bf16")
    bw = O.layer_backward(fw, x, Wg, W1, W3, W2, dy, "bf16")
    gpu_idx, exact_idx = npi(b.topk_idx), O.topk(exact, k)
    check_layer_against_oracle(b, fw, bw, una, gpu_idx, exact_idx, E, "bf16")
    ref = {n: getattr(b, n).clone() for n in ("y", "dx", "dW1", "dW3", "dW2", "dWg")}
    for fused, fold in [(True, False)] + ([(False, True), (True, True)] if h % 256 == 0 else []):
        bf = layer.LayerBuffers(T, h, E, k, f, torch.bfloat16, fused=fused, fold_combine=fold)
        layer.step(inp, bf)
        torch.cuda.synchronize()
        assert binding_status(bf) == 0
        check_layer_against_oracle(bf, fw, bw, una, npi(bf.topk_idx), exact_idx, E, "bf16")
        for n, t in ref.items():
            assert torch.equal(getattr(bf, n), t), (fused, fold, n)
    assert binding_status(b) == 0


@pytest.mark.parametrize("T,h,E,k,f,skew", _random_layer_shapes(8, 4242))
def test_random_fp32_layers(M, T, h, E, k, f, skew):
    """Seeded random fp32 shapes (h and f multiples of 128: the forward on the tensor cores over
    exact bf16 planes, the backward on the FMA engine): the layer against the oracle at the fp32
    tolerance, and the layer with the rows gathered from x bit for bit against it."""
    layer, workloads = M
    w = workloads.Workload("random-fp32", T, h, E, k, f, "f32", skew, True, T + h + E + 1)
    inp = workloads.make_inputs(w, "cuda")
    b = layer.LayerBuffers(T, h, E, k, f, torch.float32)
    layer.step(inp, b)
    torch.cuda.synchronize()
    assert binding_status(b) == 0
    x, Wg = np64(inp["x"]), np64(inp["Wg"])
    bias = None if inp["bias"] is None else np64(inp["bias"])
    exact = O.router_logits(x, Wg, bias, "f64")
    una = routing_checks(b, exact, k)
    W1, W3, W2, dy = np64(inp["W1"]), np64(inp["W3"]), np64(inp["W2"]), np64(inp["dy"])
    fw = O.layer_forward(x, Wg, W1, W3, W2, k, bias, "f32")
    bw = O.layer_backward(fw, x, Wg, W1, W3, W2, dy, "f32")
    check_layer_against_oracle(b, fw, bw, una, npi(b.topk_idx), O.topk(exact, k), E, "f32")
    ref = {n: getattr(b, n).clone() for n in ("y", "h1", "h3", "a", "dx", "dW1", "dW3", "dW2", "dWg")}
    bf = layer.LayerBuffers(T, h, E, k, f, torch.float32, fused=True)
    layer.step(inp, bf)
    torch.cuda.synchronize()
    assert binding_status(bf) == 0
    for n, t in ref.items():
        assert torch.equal(getattr(bf, n), t), n


def binding_status(b):
    from mixture_experts_layer_pft_gb300 import binding

    return binding.moe_check_status(b.ws)
