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
    if not una.all():
        pytest.skip(f"{(~una).sum()} tokens with near-tied logits; covered by the sampled test")
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


def _sample(n, hi, seed):
    g = np.random.default_rng(seed)
    s = set(g.choice(hi, size=min(n, hi), replace=False).tolist()) | {0, hi - 1}
    return np.array(sorted(s))


@pytest.mark.parametrize("cfg,ntok,nexp", [(2, 6, 2), (3, 4, 2), (4, 16, 0), (5, 3, 1)])
def test_full_size_layer_sampled(M, cfg, ntok, nexp):
    _, workloads = M
    w = workloads.WORKLOADS[cfg]
    dn = w.dtype
    inp, b = gpu_step(M, w)
    x, Wg = np64(inp["x"]), np64(inp["Wg"])
    bias = None if inp["bias"] is None else np64(inp["bias"])
    W1, W3, W2 = LazyExperts(inp["W1"]), LazyExperts(inp["W3"]), LazyExperts(inp["W2"])
    exact = O.router_logits(x, Wg, bias, "f64")
    una = routing_checks(b, exact, w.k)
    # invariants of the PFT arrays at full size
    Tk = w.T * w.k
    off = npi(b.offsets)
    assert off[0] == 0 and off[-1] == Tk and (np.diff(off) == npi(b.num_ids)).all()
    tok, slot, idx = npi(b.token_ids), npi(b.slot_of), npi(b.topk_idx)
    assert (tok[slot] == np.repeat(np.arange(w.T), w.k)).all()
    assert (npi(b.expert_ids)[slot] == idx.ravel()).all()

    S = [t for t in _sample(ntok, w.T, cfg) if una[t]]
    assert S, "no unambiguous sampled token"
    fw = O.layer_forward(x[S], Wg, W1, W3, W2, w.k, bias, dn)
    assert rel_l2(np64(b.y[S]), fw["y"]) <= TOL[dn]
    assert rel_l2(np64(b.topk_w[S]), fw["topk_w"]) <= TOL["f32"]
    if not w.backward:
        return
    dy = np64(inp["dy"])
    bw = O.layer_backward(fw, x[S], Wg, W1, W3, W2, dy[S], dn)
    assert rel_l2(np64(b.dx[S]), bw["dx"]) <= TOL[dn]
    assert rel_l2(np64(b.d_topk_w[S]), bw["d_topk_w"]) <= TOL[dn]

    # weight gradients of sampled experts whose token set is unambiguous
    ex_idx = O.topk(exact, w.k)
    counts = np.bincount(ex_idx.ravel(), minlength=w.E)
    g = np.random.default_rng(100 + cfg)
    checked = 0
    for e in g.permutation(np.nonzero(counts)[0]):
        toks = np.nonzero((ex_idx == e).any(axis=1))[0]
        if not una[toks].all():
            continue
        np.testing.assert_array_equal(tok[off[e]:off[e + 1]], toks)
        wts = O.route(x[toks], Wg, w.k, bias, dn)["probs"][:, e]
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


@pytest.mark.parametrize("T,h,E,k,f,skew", _random_layer_shapes(24, 2024))
def test_random_bf16_layers(M, T, h, E, k, f, skew):
    """Seeded random shapes on the tensor-core path: the layer against the oracle (where the
    routing is unique), and the gathered and combine-folded layers bit for bit against it."""
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
    if una.all():
        W1, W3, W2, dy = np64(inp["W1"]), np64(inp["W3"]), np64(inp["W2"]), np64(inp["dy"])
        fw = O.layer_forward(x, Wg, W1, W3, W2, k, bias, "bf16")
        bw = O.layer_backward(fw, x, Wg, W1, W3, W2, dy, "bf16")
        assert rel_l2(np64(b.y), fw["y"]) <= TOL["bf16"]
        for n in ("dx", "dW1", "dW3", "dW2", "dWg"):
            assert rel_l2(np64(getattr(b, n)), bw[n]) <= TOL["bf16"], n
    ref = {n: getattr(b, n).clone() for n in ("y", "dx", "dW1", "dW3", "dW2", "dWg")}
    for fused, fold in [(True, False)] + ([(False, True), (True, True)] if h % 256 == 0 else []):
        bf = layer.LayerBuffers(T, h, E, k, f, torch.bfloat16, fused=fused, fold_combine=fold)
        layer.step(inp, bf)
        torch.cuda.synchronize()
        assert binding_status(bf) == 0
        for n, t in ref.items():
            assert torch.equal(getattr(bf, n), t), (fused, fold, n)
    assert binding_status(b) == 0


def binding_status(b):
    from mixture_experts_layer_pft_gb300 import binding

    return binding.moe_check_status(b.ws)
