"""The capacity-buffer (GShard-style) comparison path against the oracle's capacity-buffer
formulation, and its layer against the padding-free layer (X-MoE review, §3 "Core formulas" and
§5 "Ablation": the padded dispatch the PFT replaces).

Masks, loads and the padded dispatch are compared bit for bit; the combine and the layer output
(sums in another order than the padding-free combine) by rel-L2 row by row."""

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


def routing(T, E, k, seed, skew=False):
    """top-k ids from the oracle on generated logits, and seeded gate weights."""
    from mixture_experts_layer_pft_gb300.workloads import random_logits, skew_bias

    l = random_logits(T, E, seed, "cpu")
    if skew:
        l = l + skew_bias(E)[None, :]
    idx = O.topk(l.numpy(), k)
    w = np.random.default_rng(seed).uniform(0.05, 1.0, (T, k)).astype(np.float32)
    return idx, w


def gate_on_gpu(B, idx, w, E, C, dt):
    T, k = idx.shape
    mask = torch.full((T, E, C), 7.0, dtype=dt, device="cuda")
    cw = torch.full((T, E, C), 7.0, dtype=torch.float32, device="cuda")
    loads = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    ws = B.new_workspace(B.MOE_OP_GSHARD, T, 8, E, k, 8, dt)
    B.moe_gshard_gate(torch.from_numpy(idx.astype(np.int32)).cuda(), torch.from_numpy(w).cuda(), E, C, mask, cw,
                      loads, ws)
    return mask, cw, loads, ws


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,E,k,skew,drop", [(1, 4, 2, False, 0), (300, 8, 2, False, 0), (1000, 64, 6, False, 0),
                                             (257, 256, 8, False, 0), (500, 32, 4, True, 0), (300, 8, 2, False, 5),
                                             (400, 16, 3, True, 40)])
def test_gshard_gate_bitexact(B, dt, T, E, k, skew, drop):
    idx, w = routing(T, E, k, T + E, skew)
    C = max(1, int(np.bincount(idx.ravel(), minlength=E).max()) - drop)
    want = O.gshard_capacity_gate(idx, w, E, C)
    mask, cw, loads, ws = gate_on_gpu(B, idx, w, E, C, dt)
    assert B.moe_check_status(ws) == 0
    np.testing.assert_array_equal(npi(loads), want["loads"])
    np.testing.assert_array_equal(np64(mask), want["dispatch_mask"])
    np.testing.assert_array_equal(np64(cw), want["combine_weights"].astype(np.float32).astype(np.float64))


def test_gshard_gate_flags_an_out_of_range_expert_id(B):
    idx, w = routing(64, 8, 2, 3)
    idx[10, 1] = 8
    C = int(np.bincount(idx[idx < 8], minlength=8).max())
    mask, cw, loads, ws = gate_on_gpu(B, idx, w, 8, C, torch.float32)
    assert B.moe_check_status(ws) & B.MOE_STATUS_BAD_INDEX
    assert int(mask.sum()) == 64 * 2 - 1


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,h,E,k,drop", [(1, 8, 4, 2, 0), (77, 136, 8, 2, 0), (600, 256, 16, 4, 0),
                                          (300, 2048, 64, 6, 0), (200, 128, 8, 3, 12)])
def test_gshard_dispatch_bitexact(B, dt, T, h, E, k, drop):
    from mixture_experts_layer_pft_gb300.workloads import random_tensor

    idx, w = routing(T, E, k, 5 + T)
    C = max(1, int(np.bincount(idx.ravel(), minlength=E).max()) - drop)
    g = O.gshard_capacity_gate(idx, w, E, C)
    x = random_tensor((T, h), 9 + T, dt, "cuda")
    mask = torch.from_numpy(g["dispatch_mask"]).to(dt).cuda()
    xe = torch.full((E, C, h), float("nan"), dtype=dt, device="cuda")
    ws = B.new_workspace(B.MOE_OP_GSHARD, T, h, E, k, 8, dt)
    B.moe_gshard_dispatch(x, mask, xe, ws)
    want = O.gshard_dispatch(g["dispatch_mask"], np64(x))
    np.testing.assert_array_equal(np64(xe), want)
    assert B.moe_check_status(ws) == 0


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,h,E,k,drop", [(1, 8, 4, 2, 0), (77, 136, 8, 2, 0), (600, 256, 16, 4, 0),
                                          (300, 2048, 64, 6, 0), (200, 128, 8, 3, 12)])
def test_gshard_combine(B, dt, T, h, E, k, drop):
    from mixture_experts_layer_pft_gb300.workloads import random_tensor

    idx, w = routing(T, E, k, 15 + T)
    C = max(1, int(np.bincount(idx.ravel(), minlength=E).max()) - drop)
    g = O.gshard_capacity_gate(idx, w, E, C)
    ye = random_tensor((E, C, h), 19 + T, dt, "cuda")
    cw = torch.from_numpy(g["combine_weights"].astype(np.float32)).cuda()
    y = torch.full((T, h), float("nan"), dtype=dt, device="cuda")
    ws = B.new_workspace(B.MOE_OP_GSHARD, T, h, E, k, 8, dt)
    B.moe_gshard_combine(cw, ye, y, ws)
    dn = dtype_name(dt)
    want = O.gshard_combine(g["combine_weights"].astype(np.float32), np64(ye), dn)
    got = np64(y)
    for t in range(T):
        if np.abs(want[t]).sum() == 0:
            assert (got[t] == 0).all()  # every slot of the token was dropped
        else:
            assert rel_l2(got[t], want[t]) <= TOL[dn], t
    assert B.moe_check_status(ws) == 0


@pytest.mark.parametrize("T,h,E,k,f,dt,skew", [(512, 256, 16, 4, 256, torch.bfloat16, False),
                                               (300, 256, 8, 2, 128, torch.float32, True),
                                               (2048, 2048, 64, 6, 1408, torch.bfloat16, False)])
def test_gshard_layer_equals_the_padding_free_layer(B, T, h, E, k, f, dt, skew):
    """With C the largest load no token is dropped: the capacity-buffer forward equals the oracle's
    capacity-buffer layer and the padding-free layer's output on the same inputs."""
    from mixture_experts_layer_pft_gb300 import layer, workloads

    w = workloads.Workload("gshard", T, h, E, k, f, dtype_name(dt), skew, False, 31 + T)
    inp = workloads.make_inputs(w, "cuda")
    x, Wg = np64(inp["x"]), np64(inp["Wg"])
    bias = None if inp["bias"] is None else np64(inp["bias"])
    r = O.route(x, Wg, k, bias, "f32")
    C = int(np.bincount(r["topk_idx"].ravel(), minlength=E).max())
    gb = layer.GShardBuffers(T, h, E, k, f, C, dt)
    layer.gshard_forward(inp, gb)
    pb = layer.LayerBuffers(T, h, E, k, f, dt, backward=False)
    layer.forward(inp, pb)
    torch.cuda.synchronize()
    assert B.moe_check_status(gb.ws_gshard) == 0 and B.moe_check_status(gb.ws) == 0
    dn = dtype_name(dt)
    if not np.array_equal(npi(gb.topk_idx), r["topk_idx"]):
        pytest.skip("near-tied logits: the selection is not unique")
    np.testing.assert_array_equal(npi(gb.loads), np.bincount(r["topk_idx"].ravel(), minlength=E))
    got, pft = np64(gb.y), np64(pb.y)
    for t in range(T):
        assert rel_l2(got[t], pft[t]) <= TOL[dn], t
    # the padded buffer holds the padding-free buffer's rows, then zeros
    off = npi(pb.offsets)
    xe = np64(gb.xe)
    for e in range(E):
        n = off[e + 1] - off[e]
        np.testing.assert_array_equal(xe[e, :n], np64(pb.xbuf[off[e]:off[e + 1]]))
        assert (xe[e, n:] == 0).all()
    if T <= 512:
        W1, W3, W2 = np64(inp["W1"]), np64(inp["W3"]), np64(inp["W2"])
        want = O.gshard_layer_forward(x, Wg, W1, W3, W2, k, C, bias, dn)
        for t in range(T):
            assert rel_l2(got[t], want["y"][t]) <= TOL[dn], t
