"""Per-stage parity: each C-ABI call against the oracle on identical seeded inputs.

Each stage gets generated inputs (never another stage's GPU output), so a failure points at
one kernel.  Integer outputs (top-k ids, PFT arrays) and copies are compared bit-exactly;
floating outputs by rel-L2 against the oracle's fp64 result (1e-5 fp32, 1e-2 bf16).
"""

import numpy as np
import pytest
import torch

from helpers import TOL, dtype_name, np64, npi, rel_l2
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from mixture_experts_layer_pft_gb300 import binding, build

    build.build()
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    return binding


def gen_logits(T, E, seed, skew=False, ties=False):
    from mixture_experts_layer_pft_gb300.workloads import random_logits, skew_bias

    l = random_logits(T, E, seed, "cuda")
    if ties:
        l = torch.round(l * 2.0) / 2.0  # many exact ties
    if skew:
        l = l + skew_bias(E, "cuda")[None, :]
    return l.contiguous()


def oracle_routing(T, E, k, seed, skew=False):
    """top-k ids from the oracle on generated logits (an oracle-derived input)."""
    l = gen_logits(T, E, seed, skew).cpu().numpy()
    return O.topk(l, k)


def route_from_logits(B, logits, k):
    T, E = logits.shape
    probs = torch.empty(T, E, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, device="cuda")
    ws = B.new_workspace(B.MOE_OP_ROUTE, T, 8, E, k, 8, torch.float32)
    B.moe_route(None, None, None, k, logits, probs, idx, w, ws, from_logits=True)
    return probs, idx, w, ws


# ----------------------------------------------------------------------------- gate


@pytest.mark.parametrize("T,E,k,ties", [(1, 8, 2, False), (37, 8, 2, False), (300, 64, 6, False),
                                        (513, 128, 6, True), (257, 256, 8, False), (64, 256, 8, True),
                                        (33, 1000, 7, False), (20, 16, 16, True), (100, 4, 1, False)])
def test_topk_bitexact_given_the_same_logits(B, T, E, k, ties):
    logits = gen_logits(T, E, T + E + k, ties=ties)
    probs, idx, w, _ = route_from_logits(B, logits, k)
    r = O.route_from_logits(logits.cpu().numpy(), k, "f32")
    np.testing.assert_array_equal(npi(idx), r["topk_idx"])
    assert rel_l2(np64(probs), r["probs"]) <= TOL["f32"]
    assert rel_l2(np64(w), r["topk_w"]) <= TOL["f32"]
    # the gate weight is exactly the stored probability of the chosen expert
    np.testing.assert_array_equal(np64(w), np.take_along_axis(np64(probs), npi(idx), axis=1))


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,h,E,skew", [(130, 128, 8, False), (300, 2048, 64, False), (77, 512, 128, True)])
def test_router_logits_and_topk_of_them(B, dt, T, h, E, skew):
    from mixture_experts_layer_pft_gb300.workloads import random_tensor, skew_bias

    x = random_tensor((T, h), 5, dt, "cuda")
    Wg = random_tensor((h, E), 6, torch.float32, "cuda", std=h ** -0.5)
    bias = skew_bias(E, "cuda") if skew else None
    k = 2
    logits = torch.empty(T, E, device="cuda")
    probs = torch.empty(T, E, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, device="cuda")
    ws = B.new_workspace(B.MOE_OP_ROUTE, T, h, E, k, 8, dt)
    B.moe_route(x, Wg, bias, k, logits, probs, idx, w, ws)
    want = O.router_logits(np64(x), np64(Wg), None if bias is None else np64(bias), "f32")
    assert rel_l2(np64(logits), want) <= TOL["f32"]
    # the selection on the GPU's own logits is the oracle's selection on those logits
    np.testing.assert_array_equal(npi(idx), O.topk(logits.cpu().numpy(), k))


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,h,E,k", [(200, 128, 8, 2), (129, 256, 64, 6), (64, 512, 256, 8)])
def test_route_bwd(B, dt, T, h, E, k):
    from mixture_experts_layer_pft_gb300.workloads import random_tensor

    x = random_tensor((T, h), 11, dt, "cuda")
    Wg = random_tensor((h, E), 12, torch.float32, "cuda", std=h ** -0.5)
    logits = gen_logits(T, E, 13)
    probs, idx, w, ws = route_from_logits(B, logits, k)
    d_w = random_tensor((T, k), 14, torch.float32, "cuda")
    d_logits = torch.empty(T, E, device="cuda")
    dWg = torch.empty(h, E, device="cuda")
    dxr = torch.empty(T, h, device="cuda")
    ws = B.new_workspace(B.MOE_OP_ROUTE_BWD, T, h, E, k, 8, dt)
    B.moe_route_bwd(x, Wg, probs, idx, d_w, d_logits, dWg, dxr, ws)
    r = O.route_bwd(np64(x), np64(Wg), np64(probs), npi(idx), np64(d_w), "f32")
    assert rel_l2(np64(d_logits), r["d_logits"]) <= TOL["f32"]
    assert rel_l2(np64(dWg), r["dWg"]) <= TOL["f32"]
    assert rel_l2(np64(dxr), r["dx_router"]) <= TOL["f32"]
    assert B.moe_check_status(ws) == 0


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,h,E", [(300, 7168, 256), (4096, 2048, 64), (1000, 5120, 128), (257, 2048, 80),
                                   (100, 256, 1024), (16384, 2048, 128)])
def test_router_gemms_at_full_widths(B, dt, T, h, E):
    """bf16 or fp32 activations with an fp32 router at the pages' widths (long sums over h = 7168
    and T up to 16384): logits, dWg and dx stay within the fp32 tolerance of the exact sums."""
    from mixture_experts_layer_pft_gb300.workloads import random_tensor

    k = 2
    x = random_tensor((T, h), 21, dt, "cuda")
    Wg = random_tensor((h, E), 22, torch.float32, "cuda", std=h ** -0.5)
    logits = torch.empty(T, E, device="cuda")
    probs = torch.empty(T, E, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, device="cuda")
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, 8, dt)
    B.moe_route(x, Wg, None, k, logits, probs, idx, w, ws)
    want = O.router_logits(np64(x), np64(Wg), None, "f32")
    assert rel_l2(np64(logits), want) <= TOL["f32"]
    d_w = random_tensor((T, k), 23, torch.float32, "cuda")
    d_logits = torch.empty(T, E, device="cuda")
    dWg = torch.empty(h, E, device="cuda")
    dxr = torch.empty(T, h, device="cuda")
    B.moe_route_bwd(x, Wg, probs, idx, d_w, d_logits, dWg, dxr, ws)
    r = O.route_bwd(np64(x), np64(Wg), np64(probs), npi(idx), np64(d_w), "f32")
    assert rel_l2(np64(d_logits), r["d_logits"]) <= TOL["f32"]
    assert rel_l2(np64(dWg), r["dWg"]) <= TOL["f32"]
    assert rel_l2(np64(dxr), r["dx_router"]) <= TOL["f32"]
    assert B.moe_check_status(ws) == 0


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,h,E", [(300, 2048, 64), (77, 512, 256)])
def test_tensor_core_router_matches_fp32_fma_router(B, monkeypatch, dt, T, h, E):
    """The tensor-core router (exact bf16 planes, short truncated chains) and the fp32 FMA router
    agree to fp32 accuracy on the same inputs."""
    from mixture_experts_layer_pft_gb300.workloads import random_tensor

    k = 4
    x = random_tensor((T, h), 31, dt, "cuda")
    Wg = random_tensor((h, E), 32, torch.float32, "cuda", std=h ** -0.5)
    d_w = random_tensor((T, k), 33, torch.float32, "cuda")
    probs0, idx0, _, _ = route_from_logits(B, gen_logits(T, E, 34), k)
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, 8, dt)
    outs = {}
    for engine in ("tc", "simt"):
        if engine == "simt":
            monkeypatch.setenv("MOE_PFT_GEMM", "simt")
        else:
            monkeypatch.delenv("MOE_PFT_GEMM", raising=False)
        o = {"logits": torch.empty(T, E, device="cuda"), "d_logits": torch.empty(T, E, device="cuda"),
             "dWg": torch.empty(h, E, device="cuda"), "dx": torch.empty(T, h, device="cuda")}
        probs = torch.empty(T, E, device="cuda")
        idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
        w = torch.empty(T, k, device="cuda")
        B.moe_route(x, Wg, None, k, o["logits"], probs, idx, w, ws)
        B.moe_route_bwd(x, Wg, probs0, idx0, d_w, o["d_logits"], o["dWg"], o["dx"], ws)
        torch.cuda.synchronize()
        outs[engine] = o
    assert B.moe_check_status(ws) == 0
    for n in outs["tc"]:
        assert rel_l2(np64(outs["tc"][n]), np64(outs["simt"][n])) <= TOL["f32"], n


@pytest.mark.parametrize("gate,renorm", [("softmax", True), ("sigmoid", False), ("sigmoid", True)])
@pytest.mark.parametrize("T,E,k", [(37, 8, 2), (300, 64, 6), (129, 256, 8), (40, 1000, 5)])
def test_gate_variants_given_the_same_logits(B, gate, renorm, T, E, k):
    logits = gen_logits(T, E, 7 * T + E)
    probs = torch.empty(T, E, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, device="cuda")
    ws = B.new_workspace(B.MOE_OP_ROUTE, T, 8, E, k, 8, torch.float32)
    B.moe_route(None, None, None, k, logits, probs, idx, w, ws, from_logits=True, gate=gate, renorm=renorm)
    r = O.route_from_logits(logits.cpu().numpy(), k, "f32", gate, renorm)
    np.testing.assert_array_equal(npi(idx), r["topk_idx"])
    assert rel_l2(np64(probs), r["probs"]) <= TOL["f32"]
    assert rel_l2(np64(w), r["topk_w"]) <= TOL["f32"]


@pytest.mark.parametrize("gate,renorm", [("softmax", True), ("sigmoid", False), ("sigmoid", True)])
@pytest.mark.parametrize("T,h,E,k", [(200, 128, 8, 2), (129, 256, 64, 6), (64, 512, 256, 8)])
def test_route_bwd_gate_variants(B, gate, renorm, T, h, E, k):
    from mixture_experts_layer_pft_gb300.workloads import random_tensor

    x = random_tensor((T, h), 21, torch.float32, "cuda")
    Wg = random_tensor((h, E), 22, torch.float32, "cuda", std=h ** -0.5)
    logits = gen_logits(T, E, 23)
    probs = torch.empty(T, E, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, device="cuda")
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, 8, torch.float32)
    B.moe_route(None, None, None, k, logits, probs, idx, w, ws, from_logits=True, gate=gate, renorm=renorm)
    # both sides of the backward take the oracle gate's scores and selection
    r = O.route_from_logits(logits.cpu().numpy(), k, "f32", gate, renorm)
    probs = torch.from_numpy(r["probs"].astype(np.float32)).cuda()
    idx = torch.from_numpy(r["topk_idx"].astype(np.int32)).cuda()
    d_w = random_tensor((T, k), 24, torch.float32, "cuda")
    d_logits = torch.empty(T, E, device="cuda")
    dWg = torch.empty(h, E, device="cuda")
    dxr = torch.empty(T, h, device="cuda")
    B.moe_route_bwd(x, Wg, probs, idx, d_w, d_logits, dWg, dxr, ws, gate=gate, renorm=renorm)
    want = O.route_bwd(np64(x), np64(Wg), r["probs"], r["topk_idx"], np64(d_w), "f32", gate, renorm)
    for n, got in (("d_logits", d_logits), ("dWg", dWg), ("dx_router", dxr)):
        assert rel_l2(np64(got), want[n]) <= TOL["f32"], n
    assert B.moe_check_status(ws) == 0


# ----------------------------------------------------------------------------- PFT


def run_pft(B, idx_np, E):
    T, k = idx_np.shape
    idx = torch.from_numpy(idx_np.astype(np.int32)).cuda()
    Tk = T * k
    out = {n: torch.full((Tk,), -7, dtype=torch.int32, device="cuda") for n in ("token_ids", "expert_ids", "slot_of")}
    out["num_ids"] = torch.empty(E, dtype=torch.int32, device="cuda")
    out["offsets"] = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    ws = B.new_workspace(B.MOE_OP_PFT_BUILD, T, 8, E, k, 8, torch.float32)
    B.moe_pft_build(idx, E, out["num_ids"], out["offsets"], out["token_ids"], out["expert_ids"],
                    out["slot_of"], ws)
    return out, ws


@pytest.mark.parametrize("T,E,k,skew", [(1, 8, 2, False), (37, 8, 2, False), (2048, 64, 6, False),
                                        (4096, 128, 6, True), (4096, 256, 8, False), (5000, 7, 7, False),
                                        (333, 1, 1, False), (16384, 128, 2, True), (131072, 256, 8, False),
                                        (999, 1000, 3, False), (200000, 16, 1, False), (40000, 1024, 2, False),
                                        (257, 600, 300, False)])
def test_pft_build_bitexact(B, T, E, k, skew):
    idx = oracle_routing(T, E, k, 100 + T, skew)
    out, ws = run_pft(B, idx, E)
    want = O.pft_build(idx, E)
    for n in ("num_ids", "offsets", "token_ids", "expert_ids", "slot_of"):
        np.testing.assert_array_equal(npi(out[n]), want[n], err_msg=n)
    assert B.moe_check_status(ws) == 0
    # the workspace is left clean: a second build on it gives the same arrays
    out2, _ = run_pft(B, idx, E)
    for n in ("token_ids", "slot_of"):
        np.testing.assert_array_equal(npi(out2[n]), want[n])


def _random_pft_shapes(n, seed):
    """Seeded (T, E, k, skew): T log-uniform up to 60000, E up to 1024, k up to min(E, 16), with
    T * E kept small enough for the oracle's top-k."""
    g = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        E = int(g.integers(1, 1025))
        k = int(g.integers(1, min(E, 16) + 1))
        T = int(np.exp(g.uniform(0, np.log(60000))))
        if T * E <= 20_000_000:
            out.append((max(T, 1), E, k, bool(g.random() < 0.3)))
    return out


@pytest.mark.parametrize("T,E,k,skew", _random_pft_shapes(16, 31337))
def test_pft_build_random_shapes(B, T, E, k, skew):
    """Seeded random shapes (bitmap tiles of every width, ranges of one to several tiles):
    bit for bit against the oracle."""
    idx = oracle_routing(T, E, k, 7 * T + E, skew)
    out, ws = run_pft(B, idx, E)
    want = O.pft_build(idx, E)
    for n in ("num_ids", "offsets", "token_ids", "expert_ids", "slot_of"):
        np.testing.assert_array_equal(npi(out[n]), want[n], err_msg=n)
    assert B.moe_check_status(ws) == 0


def test_pft_build_at_the_scaled_benchmark_size(B):
    """T = 2^20 tokens, k = 8, E = 256 (8.4 M rows), where the oracle's plain loops would take
    minutes: properties that fix the arrays uniquely.  The pairs (token_ids[p], expert_ids[p]) are
    exactly the flattened (t, topk_idx[t, j]) (slot_of is a permutation and their inverse), sorted by
    the unique key (expert, token), with num_ids and offsets the counts and their scan."""
    from mixture_experts_layer_pft_gb300.workloads import random_logits

    T, E, k = 1 << 20, 256, 8
    idx = torch.topk(random_logits(T, E, 77, "cuda"), k, dim=1).indices.to(torch.int32).contiguous()
    Tk = T * k
    out = {n: torch.full((Tk,), -7, dtype=torch.int32, device="cuda") for n in ("token_ids", "expert_ids", "slot_of")}
    num_ids = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    ws = B.new_workspace(B.MOE_OP_PFT_BUILD, T, 8, E, k, 8, torch.float32)
    B.moe_pft_build(idx, E, num_ids, offsets, out["token_ids"], out["expert_ids"], out["slot_of"], ws)
    assert B.moe_check_status(ws) == 0
    ids = npi(idx).ravel()
    tok, exp, slot = npi(out["token_ids"]), npi(out["expert_ids"]), npi(out["slot_of"])
    cnt = np.bincount(ids, minlength=E)
    np.testing.assert_array_equal(npi(num_ids), cnt)
    np.testing.assert_array_equal(npi(offsets), np.concatenate([[0], np.cumsum(cnt)]))
    np.testing.assert_array_equal(exp, np.repeat(np.arange(E), cnt))
    assert (np.bincount(slot, minlength=Tk) == 1).all()  # a permutation of the rows
    np.testing.assert_array_equal(tok[slot], np.repeat(np.arange(T), k))
    np.testing.assert_array_equal(exp[slot], ids)
    same = exp[1:] == exp[:-1]
    assert (tok[1:][same] > tok[:-1][same]).all()  # tokens ascending inside every segment


def test_pft_build_all_tokens_to_one_expert(B):
    T, E = 3000, 16
    idx = np.zeros((T, 1), np.int32)
    out, _ = run_pft(B, idx, E)
    want = O.pft_build(idx, E)
    for n in want:
        np.testing.assert_array_equal(npi(out[n]), want[n], err_msg=n)


def test_pft_build_flags_an_expert_id_repeated_within_a_row(B):
    """Rows must hold k distinct ids; a repeat is reported, and every write stays in range."""
    T, E, k = 300, 8, 3
    idx = oracle_routing(T, E, k, 5)
    idx[10, 2] = idx[10, 0]
    out, ws = run_pft(B, idx, E)
    assert B.moe_check_status(ws) & B.MOE_STATUS_BAD_INDEX
    cnt = np.bincount(idx.ravel(), minlength=E)
    np.testing.assert_array_equal(npi(out["num_ids"]), cnt)
    slot = npi(out["slot_of"])
    assert ((slot >= 0) & (slot < T * k)).all()
    assert slot[10 * k + 2] == slot[10 * k]
    # every other row is the oracle's build of the same ids with the repeat taken out
    keep = np.ones(T * k, bool)
    keep[10 * k + 2] = False
    tok = npi(out["token_ids"])
    assert (tok[slot[keep]] == np.repeat(np.arange(T), k)[keep]).all()


def test_pft_build_flags_an_out_of_range_expert_id(B):
    idx = oracle_routing(64, 8, 2, 3)
    idx[10, 1] = 8  # an expert id equal to E: reported, not dereferenced
    out, ws = run_pft(B, idx, 8)
    assert B.moe_check_status(ws) & B.MOE_STATUS_BAD_INDEX
    assert npi(out["slot_of"])[21] == -1
    assert npi(out["offsets"])[8] == 64 * 2 - 1


# ----------------------------------------------------------------------------- dispatch / combine


def pft_inputs(T, E, k, seed, skew=False):
    idx = oracle_routing(T, E, k, seed, skew)
    return idx, O.pft_build(idx, E)


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,h,E,k", [(1, 8, 4, 2), (77, 136, 8, 2), (2048, 2048, 64, 6), (512, 7168, 256, 8)])
def test_dispatch_bitexact_and_bwd(B, dt, T, h, E, k):
    from mixture_experts_layer_pft_gb300.workloads import random_tensor

    idx, p = pft_inputs(T, E, k, T + h)
    x = random_tensor((T, h), 21, dt, "cuda")
    tok = torch.from_numpy(p["token_ids"]).cuda()
    slot = torch.from_numpy(p["slot_of"]).cuda()
    xbuf = torch.empty(T * k, h, dtype=dt, device="cuda")
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, 8, dt)
    B.moe_dispatch(x, tok, k, xbuf, ws)
    np.testing.assert_array_equal(np64(xbuf), O.dispatch(np64(x), p["token_ids"]))
    dxbuf = random_tensor((T * k, h), 22, dt, "cuda")
    dx_add = random_tensor((T, h), 23, torch.float32, "cuda")
    dx = torch.empty(T, h, dtype=dt, device="cuda")
    for add in (None, dx_add):
        B.moe_dispatch_bwd(dxbuf, slot, add, k, dx, ws)
        want = O.dispatch_bwd(np64(dxbuf), p["slot_of"], k, None if add is None else np64(add), dtype_name(dt))
        assert rel_l2(np64(dx), want) <= TOL[dtype_name(dt)] / 10
    assert B.moe_check_status(ws) == 0


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,h,E,k", [(1, 8, 4, 2), (77, 136, 8, 2), (2048, 2048, 64, 6), (300, 7168, 256, 8),
                                     (65, 64, 40, 32)])
def test_combine_and_combine_bwd(B, dt, T, h, E, k):
    from mixture_experts_layer_pft_gb300.workloads import random_tensor

    logits = gen_logits(T, E, 31 + T)
    r = O.route_from_logits(logits.cpu().numpy(), k, "f32")
    p = O.pft_build(r["topk_idx"], E)
    slot = torch.from_numpy(p["slot_of"]).cuda()
    w = torch.from_numpy(r["topk_w"].astype(np.float32)).cuda()
    ybuf = random_tensor((T * k, h), 32, dt, "cuda")
    y = torch.empty(T, h, dtype=dt, device="cuda")
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, 8, dt)
    B.moe_combine(ybuf, slot, w, y, ws)
    tol = TOL[dtype_name(dt)] / 10
    assert rel_l2(np64(y), O.combine(np64(ybuf), p["slot_of"], r["topk_w"], dtype_name(dt))) <= tol
    dy = random_tensor((T, h), 33, dt, "cuda")
    dybuf = torch.empty(T * k, h, dtype=dt, device="cuda")
    d_w = torch.empty(T, k, device="cuda")
    B.moe_combine_bwd(dy, ybuf, slot, w, dybuf, d_w, ws)
    want_dyb, want_dw = O.combine_bwd(np64(dy), np64(ybuf), p["slot_of"], r["topk_w"], dtype_name(dt))
    assert rel_l2(np64(dybuf), want_dyb) <= tol
    assert rel_l2(np64(d_w), want_dw) <= TOL["f32"]
    assert B.moe_check_status(ws) == 0


# ----------------------------------------------------------------------------- experts


def expert_inputs(T, h, E, k, f, dt, seed, skew=False):
    from mixture_experts_layer_pft_gb300.workloads import random_tensor

    idx, p = pft_inputs(T, E, k, seed, skew)
    Tk = T * k
    d = {
        "offsets": torch.from_numpy(p["offsets"]).cuda(),
        "xbuf": random_tensor((Tk, h), seed + 1, dt, "cuda"),
        "W1": random_tensor((E, h, f), seed + 2, dt, "cuda", std=h ** -0.5),
        "W3": random_tensor((E, h, f), seed + 3, dt, "cuda", std=h ** -0.5),
        "W2": random_tensor((E, f, h), seed + 4, dt, "cuda", std=f ** -0.5),
        "dybuf": random_tensor((Tk, h), seed + 5, dt, "cuda"),
    }
    return p, d


EXPERT_SHAPES = [
    # T, h, E, k, f, dtype, skew
    (256, 128, 8, 2, 64, torch.float32, False),     # the tiny fp32 layer
    (300, 256, 8, 2, 192, torch.bfloat16, False),   # several tiles, ragged segment tails
    (200, 512, 16, 4, 256, torch.bfloat16, True),   # Zipf load: empty experts
    (97, 384, 40, 6, 128, torch.float32, True),     # many small segments at every residue
    (64, 256, 4, 1, 136, torch.bfloat16, False),    # f not a multiple of the tile
    # tensor-core engine (bf16, h and f multiples of 128)
    (333, 384, 12, 3, 256, torch.bfloat16, False),  # ragged segments below one chunk
    (1000, 256, 4, 2, 128, torch.bfloat16, True),   # segments of several 256-row chunks, Zipf
    (96, 640, 64, 6, 384, torch.bfloat16, True),    # many empty and tiny segments
    (600, 256, 4, 2, 256, torch.bfloat16, False),   # > 160 rows per expert: 256-row gate/up chunks
    (520, 384, 4, 2, 128, torch.bfloat16, True),    # 256-row chunks over Zipf-sized segments
    (400, 512, 80, 2, 512, torch.bfloat16, False),  # 160 paired units: the last 8 split into M tiles
    # fp32 on the tensor cores over exact bf16 planes (h and f multiples of 128)
    (700, 256, 12, 3, 256, torch.float32, True),    # Zipf segments, several 128-token chunks
    (300, 512, 8, 2, 384, torch.float32, False),    # K = 512 and 384: two and 1.5 drains of 256
    (64, 1024, 4, 1, 128, torch.float32, False),    # K = 1024 (four drains), one chunk per expert
]


@pytest.mark.parametrize("T,h,E,k,f,skew", [(512, 256, 8, 2, 256, False), (700, 384, 16, 4, 128, True)])
def test_tensor_core_engine_matches_simt_engine(B, monkeypatch, T, h, E, k, f, skew):
    dt = torch.bfloat16
    p, d = expert_inputs(T, h, E, k, f, dt, 90 + T, skew)
    Tk = T * k
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, f, dt)
    outs = {}
    for engine in ("tc", "simt"):
        if engine == "simt":
            monkeypatch.setenv("MOE_PFT_GEMM", "simt")
        else:
            monkeypatch.delenv("MOE_PFT_GEMM", raising=False)
        z = lambda *s: torch.empty(*s, dtype=dt, device="cuda")  # noqa: E731
        o = {"ybuf": z(Tk, h), "h1": z(Tk, f), "h3": z(Tk, f), "a": z(Tk, f), "dxbuf": z(Tk, h),
             "dW1": z(E, h, f), "dW3": z(E, h, f), "dW2": z(E, f, h)}
        B.moe_expert_ffn(d["xbuf"], d["offsets"], d["W1"], d["W3"], d["W2"], o["ybuf"], o["h1"], o["h3"], o["a"], ws)
        B.moe_expert_ffn_bwd(d["dybuf"], d["xbuf"], o["h1"], o["h3"], o["a"], d["offsets"], d["W1"], d["W3"],
                             d["W2"], o["dxbuf"], o["dW1"], o["dW3"], o["dW2"], ws)
        torch.cuda.synchronize()
        outs[engine] = o
    assert B.moe_check_status(ws) == 0
    for n in outs["tc"]:
        assert rel_l2(np64(outs["tc"][n]), np64(outs["simt"][n])) <= TOL["bf16"], n


@pytest.mark.parametrize("T,h,E,k,f,skew", [(640, 256, 8, 2, 256, False), (900, 384, 16, 4, 128, True),
                                             (2048, 2048, 32, 2, 2048, True)])
def test_fp32_tensor_core_forward_matches_the_fma_engine(B, monkeypatch, T, h, E, k, f, skew):
    """The fp32 forward over exact bf16 planes on the tensor cores against the FP32 FMA engine and
    the oracle: both within the fp32 tolerance, expert segment by expert segment."""
    p, d = expert_inputs(T, h, E, k, f, torch.float32, 90 + T, skew)
    Tk = T * k
    outs = {}
    for engine in ("tc", "simt"):
        if engine == "simt":
            monkeypatch.setenv("MOE_PFT_GEMM", "simt")
        z = lambda *s: torch.empty(*s, dtype=torch.float32, device="cuda")  # noqa: E731
        ybuf, h1, h3, a = z(Tk, h), z(Tk, f), z(Tk, f), z(Tk, f)
        ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, f, torch.float32)
        B.moe_expert_ffn(d["xbuf"], d["offsets"], d["W1"], d["W3"], d["W2"], ybuf, h1, h3, a, ws)
        assert B.moe_check_status(ws) == 0
        outs[engine] = {"ybuf": np64(ybuf), "h1": np64(h1), "h3": np64(h3), "a": np64(a)}
        monkeypatch.delenv("MOE_PFT_GEMM", raising=False)
    want = O.expert_ffn(np64(d["xbuf"]), p["offsets"], np64(d["W1"]), np64(d["W3"]), np64(d["W2"]), "f32")
    off = p["offsets"]
    for n in ("ybuf", "h1", "h3", "a"):
        for e in range(E):
            if off[e + 1] > off[e]:
                sl = slice(off[e], off[e + 1])
                assert rel_l2(outs["tc"][n][sl], want[n][sl]) <= TOL["f32"], (n, e)
                assert rel_l2(outs["tc"][n][sl], outs["simt"][n][sl]) <= TOL["f32"], (n, e)


@pytest.mark.parametrize("h,f", [(256, 384), (384, 256)])
def test_expert_forward_at_segment_length_edges(B, h, f):
    """Gate/up (256-token chunks, more than 96 rows per expert on average) and DOWN (two M tiles
    per unit when h % 256 == 0) over expert segments of 0..513 rows, built directly as PFT
    offsets; every expert's rows of h1, h3, a and y against the oracle on their own."""
    from mixture_experts_layer_pft_gb300.workloads import random_tensor

    dt = torch.bfloat16
    lens = np.array([0, 1, 15, 16, 17, 63, 64, 65, 255, 256, 257, 513], dtype=np.int64)
    E = len(lens)
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    Tk = int(offsets[-1])
    x = random_tensor((Tk, h), 61, dt, "cuda")
    W1 = random_tensor((E, h, f), 62, dt, "cuda", std=h ** -0.5)
    W3 = random_tensor((E, h, f), 63, dt, "cuda", std=h ** -0.5)
    W2 = random_tensor((E, f, h), 64, dt, "cuda", std=f ** -0.5)
    z = lambda *s: torch.full(s, float("nan"), dtype=dt, device="cuda")  # noqa: E731
    ybuf, h1, h3, a = z(Tk, h), z(Tk, f), z(Tk, f), z(Tk, f)
    ws = B.new_workspace(B.MOE_OP_ALL, Tk, h, E, 1, f, dt)
    B.moe_expert_ffn(x, torch.from_numpy(offsets).cuda(), W1, W3, W2, ybuf, h1, h3, a, ws)
    torch.cuda.synchronize()
    want = O.expert_ffn(np64(x), offsets, np64(W1), np64(W3), np64(W2), "bf16")
    for n, got in (("ybuf", ybuf), ("h1", h1), ("h3", h3), ("a", a)):
        g = np64(got)
        assert np.isfinite(g).all(), n
        for e in range(E):
            sl = slice(offsets[e], offsets[e + 1])
            if lens[e]:
                assert rel_l2(g[sl], want[n][sl]) <= TOL["bf16"], (n, e, lens[e])
    assert B.moe_check_status(ws) == 0


def test_weight_gradients_at_segment_length_edges(B):
    """Expert segments whose lengths straddle the 16-row MMA slice, the 64-row K step and the
    256-row resident chunk of the weight-gradient GEMMs (0, 1, 15, 16, 17, 63, 64, 65, 255, 256,
    257 and 513 rows), built directly as PFT offsets; dW1, dW3, dW2 and dX against the oracle."""
    from mixture_experts_layer_pft_gb300.workloads import random_tensor

    dt = torch.bfloat16
    lens = np.array([0, 1, 15, 16, 17, 63, 64, 65, 255, 256, 257, 513], dtype=np.int64)
    E, h, f = len(lens), 256, 384
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    Tk = int(offsets[-1])
    d = {
        "xbuf": random_tensor((Tk, h), 51, dt, "cuda"),
        "dybuf": random_tensor((Tk, h), 52, dt, "cuda"),
        "W1": random_tensor((E, h, f), 53, dt, "cuda", std=h ** -0.5),
        "W3": random_tensor((E, h, f), 54, dt, "cuda", std=h ** -0.5),
        "W2": random_tensor((E, f, h), 55, dt, "cuda", std=f ** -0.5),
    }
    off = torch.from_numpy(offsets).cuda()
    want = O.expert_ffn(np64(d["xbuf"]), offsets, np64(d["W1"]), np64(d["W3"]), np64(d["W2"]), "bf16")
    sv = {n: torch.from_numpy(want[n]).to(dt).cuda() for n in ("h1", "h3", "a")}
    z = lambda *s: torch.full(s, float("nan"), dtype=dt, device="cuda")  # noqa: E731
    dxbuf, dW1, dW3, dW2 = z(Tk, h), z(E, h, f), z(E, h, f), z(E, f, h)
    ws = B.new_workspace(B.MOE_OP_ALL, Tk, h, E, 1, f, dt)
    B.moe_expert_ffn_bwd(d["dybuf"], d["xbuf"], sv["h1"], sv["h3"], sv["a"], off, d["W1"], d["W3"], d["W2"],
                         dxbuf, dW1, dW3, dW2, ws)
    torch.cuda.synchronize()
    wb = O.expert_ffn_bwd(np64(d["dybuf"]), np64(d["xbuf"]), want["h1"], want["h3"], want["a"], offsets,
                          np64(d["W1"]), np64(d["W3"]), np64(d["W2"]), "bf16")
    for n, got in (("dxbuf", dxbuf), ("dW1", dW1), ("dW3", dW3), ("dW2", dW2)):
        g = np64(got)
        assert np.isfinite(g).all(), n
        for e in range(E):  # every expert on its own, so a wrong segment cannot hide in the norm
            if n == "dxbuf":
                sl = slice(offsets[e], offsets[e + 1])
                if lens[e]:
                    assert rel_l2(g[sl], wb[n][sl]) <= TOL["bf16"], (n, e)
            elif lens[e] == 0:
                assert (g[e] == 0).all(), (n, e)
            else:
                assert rel_l2(g[e], wb[n][e]) <= TOL["bf16"], (n, e, lens[e])
    assert B.moe_check_status(ws) == 0


@pytest.mark.parametrize("T,h,E,k,f,dt,skew", EXPERT_SHAPES)
def test_expert_ffn_forward_and_backward(B, T, h, E, k, f, dt, skew):
    p, d = expert_inputs(T, h, E, k, f, dt, 40 + T, skew)
    Tk = T * k
    z = lambda *s: torch.empty(*s, dtype=dt, device="cuda")  # noqa: E731
    ybuf, h1, h3, a = z(Tk, h), z(Tk, f), z(Tk, f), z(Tk, f)
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, f, dt)
    B.moe_expert_ffn(d["xbuf"], d["offsets"], d["W1"], d["W3"], d["W2"], ybuf, h1, h3, a, ws)
    dn = dtype_name(dt)
    want = O.expert_ffn(np64(d["xbuf"]), p["offsets"], np64(d["W1"]), np64(d["W3"]), np64(d["W2"]), dn)
    off = p["offsets"]
    for n, got in (("ybuf", ybuf), ("h1", h1), ("h3", h3), ("a", a)):
        g = np64(got)
        assert rel_l2(g, want[n]) <= TOL[dn], n
        for e in range(E):  # every expert segment on its own, so a wrong one cannot hide in the norm
            if off[e + 1] > off[e]:
                sl = slice(off[e], off[e + 1])
                assert rel_l2(g[sl], want[n][sl]) <= TOL[dn], (n, e)
    dxbuf, dW1, dW3, dW2 = z(Tk, h), z(E, h, f), z(E, h, f), z(E, f, h)
    # both sides of the backward get the oracle forward's saved tensors (exact in dtype)
    sv = {n: torch.from_numpy(want[n]).to(dt).cuda() for n in ("h1", "h3", "a")}
    B.moe_expert_ffn_bwd(d["dybuf"], d["xbuf"], sv["h1"], sv["h3"], sv["a"], d["offsets"], d["W1"],
                         d["W3"], d["W2"], dxbuf, dW1, dW3, dW2, ws)
    wb = O.expert_ffn_bwd(np64(d["dybuf"]), np64(d["xbuf"]), want["h1"], want["h3"], want["a"],
                          p["offsets"], np64(d["W1"]), np64(d["W3"]), np64(d["W2"]), dn)
    for n, got in (("dxbuf", dxbuf), ("dW1", dW1), ("dW3", dW3), ("dW2", dW2)):
        g = np64(got)
        assert rel_l2(g, wb[n]) <= TOL[dn], n
        for e in range(E):
            if off[e + 1] == off[e]:
                continue
            if n == "dxbuf":
                sl = slice(off[e], off[e + 1])
                assert rel_l2(g[sl], wb[n][sl]) <= TOL[dn], (n, e)
            else:
                assert rel_l2(g[e], wb[n][e]) <= TOL[dn], (n, e)
    empty = np.nonzero(p["num_ids"] == 0)[0]
    for e in empty:
        assert (np64(dW1[e]) == 0).all() and (np64(dW2[e]) == 0).all()
    assert B.moe_check_status(ws) == 0


GATHER_SHAPES = [s for s in EXPERT_SHAPES if s[1] % 128 == 0 and s[4] % 128 == 0]  # bf16 and fp32


@pytest.mark.parametrize("bad_id", [False, True])
@pytest.mark.parametrize("T,h,E,k,f,dt,skew", GATHER_SHAPES)
def test_gathered_expert_ffn_equals_dispatch_then_ffn(B, T, h, E, k, f, dt, skew, bad_id):
    """The expert GEMMs that gather their token rows from x give the same bits as dispatching
    xbuf first, forward and backward; an out-of-range token id reads as a zero row and sets the
    status bit on both paths.  In fp32 the forward splits the gathered rows straight into planes
    and the backward gathers them into dxbuf ahead of dW1/dW3."""
    from mixture_experts_layer_pft_gb300.workloads import random_tensor

    assert B.moe_expert_ffn_gather_supported(h, f, dt)
    p, d = expert_inputs(T, h, E, k, f, dt, 70 + T, skew)
    Tk = T * k
    x = random_tensor((T, h), 90 + T, dt, "cuda")
    tok = torch.from_numpy(p["token_ids"]).cuda()
    if bad_id:
        tok[Tk // 2] = T + 3
    z = lambda *s: torch.empty(*s, dtype=dt, device="cuda")  # noqa: E731
    outs = []
    for gathered in (False, True):
        ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, f, dt)
        ybuf, h1, h3, a = z(Tk, h), z(Tk, f), z(Tk, f), z(Tk, f)
        dxbuf, dW1, dW3, dW2 = z(Tk, h), z(E, h, f), z(E, h, f), z(E, f, h)
        if gathered:
            B.moe_expert_ffn_gather(x, tok, d["offsets"], d["W1"], d["W3"], d["W2"], ybuf, h1, h3, a, ws)
            B.moe_expert_ffn_bwd_gather(d["dybuf"], x, tok, h1, h3, a, d["offsets"], d["W1"], d["W3"], d["W2"],
                                        dxbuf, dW1, dW3, dW2, ws)
        else:
            xbuf = z(Tk, h)
            B.moe_dispatch(x, tok, k, xbuf, ws)
            B.moe_expert_ffn(xbuf, d["offsets"], d["W1"], d["W3"], d["W2"], ybuf, h1, h3, a, ws)
            B.moe_expert_ffn_bwd(d["dybuf"], xbuf, h1, h3, a, d["offsets"], d["W1"], d["W3"], d["W2"],
                                 dxbuf, dW1, dW3, dW2, ws)
        torch.cuda.synchronize()
        status = B.moe_check_status(ws)
        assert status == (B.MOE_STATUS_BAD_INDEX if bad_id else 0)
        outs.append({"ybuf": ybuf, "h1": h1, "h3": h3, "a": a, "dxbuf": dxbuf, "dW1": dW1, "dW3": dW3,
                     "dW2": dW2})
    for n, t in outs[0].items():
        assert torch.equal(outs[1][n], t), n


def test_gathered_expert_ffn_rejects_the_simt_engine(B):
    """Shapes only the FMA engine takes (f not a multiple of 128) have no gathered form: the
    call reports MOE_ERR_UNSUPPORTED."""
    assert B.moe_expert_ffn_gather_supported(256, 256, torch.float32)
    assert not B.moe_expert_ffn_gather_supported(256, 192, torch.float32)
    assert not B.moe_expert_ffn_gather_supported(256, 192, torch.bfloat16)
    T, h, E, k, f = 16, 256, 4, 2, 192
    x = torch.zeros(T, h, device="cuda")
    tok = torch.zeros(T * k, dtype=torch.int32, device="cuda")
    off = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    W = torch.zeros(E, h, f, device="cuda")
    o = torch.zeros(T * k, h, device="cuda")
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, f, torch.float32)
    with pytest.raises(B.MoEError):
        B.moe_expert_ffn_gather(x, tok, off, W, W, W.transpose(1, 2).contiguous(), o, o, o, o, ws)


FOLD_SHAPES = [s for s in GATHER_SHAPES if s[5] == torch.bfloat16 and s[1] % 256 == 0]


@pytest.mark.parametrize("gathered", [False, True])
@pytest.mark.parametrize("T,h,E,k,f,dt,skew", FOLD_SHAPES)
def test_combine_folded_into_down_projection(B, T, h, E, k, f, dt, skew, gathered):
    """moe_expert_ffn_fused with y: the down projection's epilogue writes the same y, bit for
    bit, as moe_combine over its ybuf (and the same ybuf, h1, h3, a as moe_expert_ffn), with the
    dispatch separate or folded in too."""
    from mixture_experts_layer_pft_gb300.workloads import random_tensor

    p, d = expert_inputs(T, h, E, k, f, dt, 110 + T, skew)
    Tk = T * k
    x = random_tensor((T, h), 120 + T, dt, "cuda")
    tok = torch.from_numpy(p["token_ids"]).cuda()
    slot = torch.from_numpy(p["slot_of"]).cuda()
    w = torch.rand(T, k, generator=torch.Generator().manual_seed(T), dtype=torch.float32).cuda()
    z = lambda *s: torch.empty(*s, dtype=dt, device="cuda")  # noqa: E731
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, f, dt)
    xbuf = z(Tk, h)
    B.moe_dispatch(x, tok, k, xbuf, ws)
    want = {n: z(*sh) for n, sh in (("ybuf", (Tk, h)), ("h1", (Tk, f)), ("h3", (Tk, f)), ("a", (Tk, f)), ("y", (T, h)))}
    B.moe_expert_ffn(xbuf, d["offsets"], d["W1"], d["W3"], d["W2"], want["ybuf"], want["h1"], want["h3"], want["a"], ws)
    B.moe_combine(want["ybuf"], slot, w, want["y"], ws)
    got = {n: torch.full_like(t, float("nan")) for n, t in want.items()}
    for _ in range(2):  # the counters are zeroed by each call
        B.moe_expert_ffn_fused(None if gathered else xbuf, x, tok, slot, w, d["offsets"], d["W1"], d["W3"],
                               d["W2"], got["ybuf"], got["h1"], got["h3"], got["a"], got["y"], ws)
        torch.cuda.synchronize()
        for n in want:
            assert torch.equal(got[n], want[n]), n
    assert B.moe_check_status(ws) == 0


def test_combine_fold_rejects_unsupported_shapes(B):
    """The combine fold lives in the paired down projection: h % 256 != 0 is MOE_ERR_UNSUPPORTED."""
    T, h, E, k, f = 16, 384, 4, 2, 128
    dt = torch.bfloat16
    z = lambda *s, d=dt: torch.zeros(*s, dtype=d, device="cuda")  # noqa: E731
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, f, dt)
    with pytest.raises(B.MoEError):
        B.moe_expert_ffn_fused(z(T * k, h), z(T, h), z(T * k, d=torch.int32), z(T * k, d=torch.int32),
                               z(T, k, d=torch.float32), z(E + 1, d=torch.int32), z(E, h, f), z(E, h, f), z(E, f, h),
                               z(T * k, h), z(T * k, f), z(T * k, f), z(T * k, f), z(T, h), ws)
