"""moe_pft_build_noalloc: the PFT build for callers that cannot allocate device memory.

Plugins whose host framework owns all device memory, or services with a fixed memory plan,
cannot call cudaMalloc or pass a workspace.  This entry point keeps its scratch in a static
device array instead.  Its arrays must equal those of moe_pft_build, which takes a workspace,
bit for bit (index arrays are compared exactly throughout these tests), on consecutive calls
that share the static array, on an empty batch and with corrupted expert ids; sizes beyond its
limits are refused on the host.  This file is collected last.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _routing(T, E, k, seed):
    from mixture_experts_layer_pft_gb300.workloads import random_logits

    logits = random_logits(T, E, seed, "cuda")
    return torch.topk(logits, k, dim=1).indices.to(torch.int32).contiguous()


def _outputs(T, E, k):
    Tk = T * k
    return {
        "num_ids": torch.full((E,), -9, dtype=torch.int32, device="cuda"),
        "offsets": torch.full((E + 1,), -9, dtype=torch.int32, device="cuda"),
        "token_ids": torch.full((Tk,), -9, dtype=torch.int32, device="cuda"),
        "expert_ids": torch.full((Tk,), -9, dtype=torch.int32, device="cuda"),
        "slot_of": torch.full((Tk,), -9, dtype=torch.int32, device="cuda"),
    }


def test_noalloc_pft_build_equals_the_workspace_version_on_consecutive_calls():
    from mixture_experts_layer_pft_gb300 import binding as B
    from mixture_experts_layer_pft_gb300 import build

    build.build()
    assert torch.cuda.is_available()
    # two calls in a row, different shapes: the second must not see the first one's state
    for T, E, k, seed in [(4096, 256, 8, 11), (2048, 64, 6, 12)]:
        idx = _routing(T, E, k, seed)
        ref = _outputs(T, E, k)
        ws = B.new_workspace(B.MOE_OP_PFT_BUILD, T, 8, E, k, 8, torch.float32)
        B.moe_pft_build(idx, E, ref["num_ids"], ref["offsets"], ref["token_ids"], ref["expert_ids"],
                        ref["slot_of"], ws)
        got = _outputs(T, E, k)
        B.moe_pft_build_noalloc(idx, E, got["num_ids"], got["offsets"], got["token_ids"],
                                got["expert_ids"], got["slot_of"])
        torch.cuda.synchronize()
        assert B.moe_check_status(ws) == 0
        for n in ref:
            np.testing.assert_array_equal(got[n].cpu().numpy(), ref[n].cpu().numpy(), err_msg=n)


def test_noalloc_pft_build_rejects_sizes_beyond_its_static_scratch():
    from mixture_experts_layer_pft_gb300 import binding as B
    from mixture_experts_layer_pft_gb300 import build

    build.build()
    # E = 1024 experts with T*k = 1024 * 1024 entries needs more than the 1 MiB scratch;
    # the call is refused on the host before any pointer is touched
    T, E, k = 1 << 17, 1024, 8
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoEError) as ei:
        B._call("moe_pft_build_noalloc", B._p(dummy), T, E, k, B._p(dummy), B._p(dummy), B._p(dummy),
                B._p(dummy), B._p(dummy), B._stream())
    assert ei.value.code == B.MOE_ERR_UNSUPPORTED
    assert "static maximum" in str(ei.value)


def test_noalloc_pft_build_rejects_more_than_2_to_the_30_entries():
    from mixture_experts_layer_pft_gb300 import binding as B
    from mixture_experts_layer_pft_gb300 import build

    build.build()
    # E = 8 needs only a few KB of histograms at any T, so the static scratch alone would let
    # this through; the int32 positions of the PFT arrays do not, and the call is refused on the
    # host as moe_pft_build refuses it
    T, E, k = (1 << 28) + 1, 8, 4
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoEError) as ei:
        B._call("moe_pft_build_noalloc", B._p(dummy), T, E, k, B._p(dummy), B._p(dummy), B._p(dummy),
                B._p(dummy), B._p(dummy), B._stream())
    assert ei.value.code == B.MOE_ERR_UNSUPPORTED
    assert "2^30" in str(ei.value)


def test_noalloc_pft_build_of_an_empty_batch():
    from mixture_experts_layer_pft_gb300 import binding as B
    from mixture_experts_layer_pft_gb300 import build

    build.build()
    E, k = 16, 2
    idx = torch.empty(0, k, dtype=torch.int32, device="cuda")
    got = _outputs(0, E, k)
    B.moe_pft_build_noalloc(idx, E, got["num_ids"], got["offsets"], got["token_ids"], got["expert_ids"],
                            got["slot_of"])
    torch.cuda.synchronize()
    assert int(got["num_ids"].abs().sum()) == 0 and int(got["offsets"].abs().sum()) == 0


def test_noalloc_pft_build_drops_an_out_of_range_expert_id():
    from mixture_experts_layer_pft_gb300 import binding as B
    from mixture_experts_layer_pft_gb300 import build

    build.build()
    T, E, k = 300, 64, 6
    idx = _routing(T, E, k, 13)
    bad = [(5, 0, E), (17, 3, -1), (299, 5, E + 40)]  # (token, slot j, corrupted id), set on the host
    h = idx.cpu()
    for t, j, v in bad:
        h[t, j] = v
    idx = h.cuda()
    ref = _outputs(T, E, k)
    ws = B.new_workspace(B.MOE_OP_PFT_BUILD, T, 8, E, k, 8, torch.float32)
    B.moe_pft_build(idx, E, ref["num_ids"], ref["offsets"], ref["token_ids"], ref["expert_ids"],
                    ref["slot_of"], ws)
    got = _outputs(T, E, k)
    B.moe_pft_build_noalloc(idx, E, got["num_ids"], got["offsets"], got["token_ids"], got["expert_ids"],
                            got["slot_of"])
    torch.cuda.synchronize()
    assert B.moe_check_status(ws) & B.MOE_STATUS_BAD_INDEX  # the workspace version reports it
    slot = got["slot_of"].cpu().numpy()
    for t, j, _ in bad:
        assert slot[t * k + j] == -1
    # the dropped entries leave T*k - 3 rows; every array matches the workspace version's
    assert int(got["offsets"][E]) == T * k - len(bad)
    for n in ("num_ids", "offsets", "slot_of"):
        np.testing.assert_array_equal(got[n].cpu().numpy(), ref[n].cpu().numpy(), err_msg=n)
    n_rows = T * k - len(bad)
    for n in ("token_ids", "expert_ids"):
        np.testing.assert_array_equal(got[n][:n_rows].cpu().numpy(), ref[n][:n_rows].cpu().numpy(), err_msg=n)
