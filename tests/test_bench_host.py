"""Host-side logic of bench.py (CPU only): the bounded oracle sample and its stage-by-stage
composition, which must give the oracle's own layer results."""

import numpy as np
import torch

import bench
from mixture_experts_layer_pft_gb300 import workloads
from oracle import moe_oracle as O


def test_oracle_sample_is_bounded_in_work_and_host_memory():
    W = workloads.WORKLOADS
    assert bench.oracle_sample_tokens(W[1]) == W[1].T  # the whole X-MoE Small layer
    # X-MoE Large: the experts 2 tokens can reach (16) hold about 5.6 GB of fp64 weights
    assert bench.oracle_sample_tokens(W[3]) == 2
    for w in W:
        Ts = bench.oracle_sample_tokens(w)
        per_expert = 3 * w.h * w.f * 8
        assert 1 <= Ts <= w.T
        if w.E * per_expert > 6e9:  # only the experts Ts tokens can reach are held on the host
            assert Ts * w.k * per_expert <= 6e9
        assert bench.model_flops(w, Ts) <= 1.2e12


def test_oracle_step_equals_the_oracle_layer():
    """The per-expert backward of the timed composition gives the oracle layer's y and dx."""
    w = workloads.Workload("host", 40, 64, 6, 2, 32, "bf16", True, True, 5)
    inp = workloads.make_inputs(w, "cpu")
    c = {k: (None if v is None else v.double().numpy()) for k, v in inp.items()}
    experts = {e: (c["W1"][e], c["W3"][e], c["W2"][e]) for e in range(w.E)}
    W1 = bench.HostExperts({e: v[0] for e, v in experts.items()}, (w.E, w.h, w.f))
    W3 = bench.HostExperts({e: v[1] for e, v in experts.items()}, (w.E, w.h, w.f))
    W2 = bench.HostExperts({e: v[2] for e, v in experts.items()}, (w.E, w.f, w.h))
    y, dx = bench.oracle_step(w, c["x"], c["Wg"], c["bias"], W1, W3, W2, c["dy"])
    fw = O.layer_forward(c["x"], c["Wg"], c["W1"], c["W3"], c["W2"], w.k, c["bias"], "bf16")
    bw = O.layer_backward(fw, c["x"], c["Wg"], c["W1"], c["W3"], c["W2"], c["dy"], "bf16")
    np.testing.assert_array_equal(y, fw["y"])
    np.testing.assert_array_equal(dx, bw["dx"])


def test_host_sample_inputs_reach_only_their_experts():
    w = workloads.WORKLOADS[2]  # Medium: 5120 x 1536 experts, Zipf router bias
    Ts = 3
    args, n_exp = bench.oracle_inputs(w.with_tokens(w.T), Ts)
    x_s, Wg, bias, W1, W3, W2, dy_s = args
    assert x_s.shape == (Ts, w.h) and dy_s.shape == (Ts, w.h) and bias is not None
    assert 1 <= n_exp <= Ts * w.k and len(W1.w) == n_exp
    e = next(iter(W1.w))
    assert W1[e].shape == (w.h, w.f) and W2[e].shape == (w.f, w.h) and W1[e].dtype == np.float64
    # the values are bf16 numbers held in fp64
    assert torch.equal(torch.from_numpy(W1[e]).to(torch.bfloat16).double(), torch.from_numpy(W1[e]))
