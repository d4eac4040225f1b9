"""The bounded waits of the tensor-core kernels, made to run out on purpose.

The failure is injected on the host (moe_debug_withhold_stage): the TMA producer of the next
tcgen05 launch never fills its first pipeline stage, so the MMA warp waits on a barrier that
nothing completes.  The wait gives up after a short limit, the kernel sets MOE_STATUS_TIMEOUT,
every warp role unwinds and the tensor memory is freed.  Each test then clears the status word,
runs the same call again on the same workspace and requires the bits of a clean call: no warp
was left waiting, no tensor memory was left allocated.  Nothing here traps or faults the GPU:
every wait in those kernels is bounded by the device clock.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000  # 20 ms per wait for the withheld launches


@pytest.fixture(scope="module")
def B():
    from mixture_experts_layer_pft_gb300 import binding, build

    build.build()
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    yield binding
    binding.moe_debug_withhold_stage(0)


def _expert_inputs(T, h, E, k, f, seed):
    from mixture_experts_layer_pft_gb300.workloads import random_logits, random_tensor

    idx = torch.topk(random_logits(T, E, seed, "cuda"), k, dim=1).indices
    counts = torch.bincount(idx.flatten(), minlength=E)
    offsets = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    offsets[1:] = torch.cumsum(counts, 0).to(torch.int32)
    Tk, dt = T * k, torch.bfloat16
    return {
        "offsets": offsets,
        "x": random_tensor((T, h), seed + 6, dt, "cuda"),
        # buffer rows sorted by (expert, token): a stable sort of the flattened ids by expert
        "token_ids": (idx.flatten().argsort(stable=True) // k).to(torch.int32),
        "xbuf": random_tensor((Tk, h), seed + 1, dt, "cuda"),
        "W1": random_tensor((E, h, f), seed + 2, dt, "cuda", std=h ** -0.5),
        "W3": random_tensor((E, h, f), seed + 3, dt, "cuda", std=h ** -0.5),
        "W2": random_tensor((E, f, h), seed + 4, dt, "cuda", std=f ** -0.5),
        "dybuf": random_tensor((Tk, h), seed + 5, dt, "cuda"),
    }


def _timed_out(B, ws):
    code = B.moe_check_status(ws)
    return (code & B.MOE_STATUS_TIMEOUT) != 0


def _run_twice_with_a_timeout_between(B, ws, call, outputs, launches):
    """call() on clean state -> reference bits; the same call with `launches` withheld stages ->
    MOE_STATUS_TIMEOUT; cleared status and the call again -> the reference bits."""
    call()
    assert B.moe_check_status(ws) == 0
    want = [t.clone() for t in outputs]
    B.moe_debug_withhold_stage(launches, LIMIT_NS)
    call()
    assert _timed_out(B, ws)
    B.moe_debug_withhold_stage(0)
    B.moe_status_reset(ws)
    for t in outputs:
        t.fill_(float("nan")) if t.is_floating_point() else t.fill_(-1)
    call()
    assert B.moe_check_status(ws) == 0
    for got, ref in zip(outputs, want):
        assert torch.equal(got, ref)


def test_expert_forward_gemm_times_out_and_recovers(B):
    T, h, E, k, f = 512, 256, 8, 2, 256
    d = _expert_inputs(T, h, E, k, f, 61)
    Tk = T * k
    z = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    ybuf, h1, h3, a = z(Tk, h), z(Tk, f), z(Tk, f), z(Tk, f)
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, f, torch.bfloat16)

    def call():
        B.moe_expert_ffn(d["xbuf"], d["offsets"], d["W1"], d["W3"], d["W2"], ybuf, h1, h3, a, ws)

    # gate/up withheld; the down projection after it runs normally on what gate/up left
    _run_twice_with_a_timeout_between(B, ws, call, [ybuf, h1, h3, a], 1)
    # both GEMMs withheld
    _run_twice_with_a_timeout_between(B, ws, call, [ybuf, h1, h3, a], 2)


def test_expert_backward_gemms_time_out_and_recover(B):
    T, h, E, k, f = 512, 256, 8, 2, 256
    d = _expert_inputs(T, h, E, k, f, 62)
    Tk = T * k
    z = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    ybuf, h1, h3, a = z(Tk, h), z(Tk, f), z(Tk, f), z(Tk, f)
    dxbuf, dW1, dW3, dW2 = z(Tk, h), z(E, h, f), z(E, h, f), z(E, f, h)
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, f, torch.bfloat16)
    B.moe_expert_ffn(d["xbuf"], d["offsets"], d["W1"], d["W3"], d["W2"], ybuf, h1, h3, a, ws)
    torch.cuda.synchronize()

    def call():
        B.moe_expert_ffn_bwd(d["dybuf"], d["xbuf"], h1, h3, a, d["offsets"], d["W1"], d["W3"], d["W2"], dxbuf,
                             dW1, dW3, dW2, ws)

    # all four backward GEMMs (dA, dX, dW1/dW3 with tensor stores, dW2) withheld
    _run_twice_with_a_timeout_between(B, ws, call, [dxbuf, dW1, dW3, dW2], 4)


def test_gathered_gemm_times_out_and_recovers(B):
    """The gate/up GEMM whose producer warp gathers token rows itself (cp.async copies)."""
    T, h, E, k, f = 384, 256, 8, 2, 256
    d = _expert_inputs(T, h, E, k, f, 63)
    if not B.moe_expert_ffn_gather_supported(h, f, torch.bfloat16):
        pytest.skip("no tensor-core engine")
    Tk = T * k
    z = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    ybuf, h1, h3, a = z(Tk, h), z(Tk, f), z(Tk, f), z(Tk, f)
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, f, torch.bfloat16)

    def call():
        B.moe_expert_ffn_gather(d["x"], d["token_ids"], d["offsets"], d["W1"], d["W3"], d["W2"], ybuf, h1, h3,
                                a, ws)

    _run_twice_with_a_timeout_between(B, ws, call, [ybuf, h1, h3, a], 1)


def test_router_gemms_time_out_and_recover(B):
    from mixture_experts_layer_pft_gb300.workloads import random_tensor

    T, h, E, k = 300, 512, 64, 4
    x = random_tensor((T, h), 71, torch.bfloat16, "cuda")
    Wg = random_tensor((h, E), 72, torch.float32, "cuda", std=h ** -0.5)
    logits = torch.empty(T, E, device="cuda")
    probs = torch.empty(T, E, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, device="cuda")
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, 128, torch.bfloat16)

    def fwd():
        B.moe_route(x, Wg, None, k, logits, probs, idx, w, ws)

    _run_twice_with_a_timeout_between(B, ws, fwd, [logits, probs, idx, w], 1)

    d_w = random_tensor((T, k), 73, torch.float32, "cuda")
    d_logits = torch.empty(T, E, device="cuda")
    dWg = torch.empty(h, E, device="cuda")
    dxr = torch.empty(T, h, device="cuda")

    def bwd():
        B.moe_route_bwd(x, Wg, probs, idx, d_w, d_logits, dWg, dxr, ws)

    _run_twice_with_a_timeout_between(B, ws, bwd, [d_logits, dWg, dxr], 2)


def test_fp32_tensor_core_gemm_times_out_and_recovers(B):
    """The fp32 forward over bf16 planes: its first GEMM withheld, then all three."""
    from mixture_experts_layer_pft_gb300.workloads import random_logits, random_tensor

    T, h, E, k, f = 256, 256, 4, 2, 256
    idx = torch.topk(random_logits(T, E, 65, "cuda"), k, dim=1).indices
    counts = torch.bincount(idx.flatten(), minlength=E)
    offsets = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    offsets[1:] = torch.cumsum(counts, 0).to(torch.int32)
    Tk = T * k
    xbuf = random_tensor((Tk, h), 66, torch.float32, "cuda")
    W1 = random_tensor((E, h, f), 67, torch.float32, "cuda", std=h ** -0.5)
    W3 = random_tensor((E, h, f), 68, torch.float32, "cuda", std=h ** -0.5)
    W2 = random_tensor((E, f, h), 69, torch.float32, "cuda", std=f ** -0.5)
    z = lambda *s: torch.empty(*s, dtype=torch.float32, device="cuda")  # noqa: E731
    ybuf, h1, h3, a = z(Tk, h), z(Tk, f), z(Tk, f), z(Tk, f)
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, f, torch.float32)

    def call():
        B.moe_expert_ffn(xbuf, offsets, W1, W3, W2, ybuf, h1, h3, a, ws)

    _run_twice_with_a_timeout_between(B, ws, call, [ybuf, h1, h3, a], 1)
    _run_twice_with_a_timeout_between(B, ws, call, [ybuf, h1, h3, a], 3)


def test_hook_is_off_by_default_and_cancels(B):
    """A cancelled request leaves the next launch alone."""
    T, h, E, k, f = 256, 256, 4, 2, 128
    d = _expert_inputs(T, h, E, k, f, 64)
    Tk = T * k
    z = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    ybuf, h1, h3, a = z(Tk, h), z(Tk, f), z(Tk, f), z(Tk, f)
    ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, f, torch.bfloat16)
    B.moe_debug_withhold_stage(3, LIMIT_NS)
    B.moe_debug_withhold_stage(0)
    B.moe_expert_ffn(d["xbuf"], d["offsets"], d["W1"], d["W3"], d["W2"], ybuf, h1, h3, a, ws)
    assert B.moe_check_status(ws) == 0
    assert np.isfinite(ybuf.float().cpu().numpy()).all()
