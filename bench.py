"""Benchmark of one padding-free MoE layer step (forward + backward) on GB300.

A step is one pass of the whole path over one batch of synthetic tokens: gate, PFT build,
dispatch, expert SwiGLU, combine, then combine backward, expert backward, gate backward and
dispatch backward.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]

Under torchrun each rank runs the step on its own GPU over its own tokens (weights drawn
identically), with no collective on the data path; ``value`` is the whole-job throughput,
the max over ranks of the timed region.

The timed region replays the layer step captured as a CUDA graph (``--no-graph``: one host call
per stage), one event pair per step.  Per-stage and per-kernel times, and the roofline's kernel
duration, come from a second pass of the same steps with an event after every launch.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd+bwd TFLOPS & tokens/s on 1×GB300; dispatch/combine HBM GB/s"
DEFAULT_CONFIG = 3  # the X-MoE Large layer, bf16, forward + backward
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP32_ALU_TFLOPS_NOMINAL = 152 * 128 * 2 * 2.07e9 / 1e12  # SMs x FP32 lanes x FMA x max clock

STAGES = ["route", "pft_build", "dispatch", "expert_ffn", "combine",
          "combine_bwd", "expert_ffn_bwd", "route_bwd", "dispatch_bwd"]


# ----------------------------------------------------------------------------- algorithmic counts


def stage_counts(w, T):
    """Algorithmic FLOPs and HBM bytes of each stage for workload ``w`` at T tokens."""
    s = 2 if w.dtype == "bf16" else 4
    h, E, k, f = w.h, w.E, w.k, w.f
    Tk = T * k
    c = {
        "route": {"flops": 2 * T * h * E, "bytes": T * h * s + h * E * 4 + 3 * T * E * 4 + 8 * Tk},
        "pft_build": {"flops": 0, "bytes": 4 * Tk + 12 * Tk + 8 * E},
        "dispatch": {"flops": 0, "bytes": T * h * s + Tk * h * s + 4 * Tk},
        "expert_ffn": {"flops": 6 * Tk * h * f, "bytes": 3 * E * h * f * s + 2 * Tk * h * s + 3 * Tk * f * s},
        "combine": {"flops": 2 * Tk * h, "bytes": Tk * h * s + T * h * s + 8 * Tk},
        "combine_bwd": {"flops": 3 * Tk * h, "bytes": T * h * s + 2 * Tk * h * s + 12 * Tk},
        "expert_ffn_bwd": {"flops": 12 * Tk * h * f,
                           "bytes": 6 * E * h * f * s + 3 * Tk * h * s + 7 * Tk * f * s},
        "route_bwd": {"flops": 4 * T * h * E, "bytes": T * h * s + h * E * 8 + 2 * T * E * 4 + T * h * 4},
        "dispatch_bwd": {"flops": Tk * h, "bytes": Tk * h * s + T * h * s + T * h * 4 + 4 * Tk},
    }
    if not w.backward:
        for n in ("combine_bwd", "expert_ffn_bwd", "route_bwd", "dispatch_bwd"):
            c.pop(n)
    return c


def model_flops(w, T):
    """Layer FLOPs as the headline counts them: expert GEMMs + router GEMMs."""
    Tk = T * w.k
    fwd = 6 * Tk * w.h * w.f + 2 * T * w.h * w.E
    bwd = 12 * Tk * w.h * w.f + 4 * T * w.h * w.E
    return fwd + (bwd if w.backward else 0)


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


CSRC = "mixture_experts_layer_pft_gb300/csrc/"
# headers every kernel source includes: a change there also invalidates recorded counters
KERNEL_HEADERS = [CSRC + "common.cuh", CSRC + "tc_ptx.cuh"]


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key, src_hash):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
    except (OSError, ValueError):
        return None
    e = d.get(kernel_key)
    if not e or e.get("source_hash") != src_hash:
        return None
    return e.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples every 100 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = open(os.devnull, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed helpers


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle baseline


def oracle_sample_tokens(w, budget_flops=1.2e12, host_bytes=6e9):
    """Token count of a bounded oracle sample: about ``budget_flops`` of layer work (10-30 s of
    fp64 numpy on a CPU host), and no more tokens than keep the fp64 weights of the experts they
    can reach (at most k per token) within ``host_bytes``."""
    per_tok = model_flops(w, 1)
    Ts = int(budget_flops // per_tok)
    per_expert = 3 * w.h * w.f * 8
    max_experts = int(host_bytes // per_expert)
    if w.E > max_experts:
        Ts = min(Ts, max(1, max_experts // w.k))
    return int(max(1, min(w.T, Ts)))


class HostExperts:
    """Expert weights of one kind (W1, W3 or W2) as fp64 host arrays for the experts a sample
    reaches, indexed like the stacked [E, ...] array the oracle takes."""

    def __init__(self, per_expert, shape):
        self.w = per_expert
        self.shape = tuple(shape)

    def __getitem__(self, e):
        if isinstance(e, slice):  # a one-expert view for the per-expert backward
            return HostExperts({0: self.w[int(e.start)]}, (1,) + self.shape[1:])
        return self.w[int(e)]


def oracle_step(w, x_s, Wg, bias, W1, W3, W2, dy_s):
    """One layer step of the oracle on a token sample, stage by stage in the order the oracle's
    layer_forward and layer_backward take them; the expert backward runs one expert at a time so
    that only one expert's fp64 weight gradients exist at once.  Returns (y, dx) of the sample."""
    import numpy as np

    from oracle import moe_oracle as O

    dn = w.dtype
    r = O.route(x_s, Wg, w.k, bias, dn)
    pft = O.pft_build(r["topk_idx"], w.E)
    xbuf = O.dispatch(x_s, pft["token_ids"])
    ffn = O.expert_ffn(xbuf, pft["offsets"], W1, W3, W2, dn)
    y = O.combine(ffn["ybuf"], pft["slot_of"], r["topk_w"], dn)
    if dy_s is None:
        return y, None
    dybuf, d_w = O.combine_bwd(dy_s, ffn["ybuf"], pft["slot_of"], r["topk_w"], dn)
    off = pft["offsets"]
    dxbuf = np.zeros_like(xbuf)
    for e in np.nonzero(np.diff(off))[0]:
        sl = slice(off[e], off[e + 1])
        one = np.array([0, off[e + 1] - off[e]])
        eb = O.expert_ffn_bwd(dybuf[sl], xbuf[sl], ffn["h1"][sl], ffn["h3"][sl], ffn["a"][sl], one,
                              W1[e:e + 1], W3[e:e + 1], W2[e:e + 1], dn)
        dxbuf[sl] = eb["dxbuf"]
    rb = O.route_bwd(x_s, Wg, r["probs"], r["topk_idx"], d_w, dn)
    return y, O.dispatch_bwd(dxbuf, pft["slot_of"], w.k, rb["dx_router"], dn)


def oracle_inputs(w, Ts, inp=None):
    """Host inputs of an oracle sample of Ts tokens: from the benchmark's device inputs ``inp``
    (a seeded choice of tokens, and only the experts they reach), or, without them, drawn on the
    host (workloads.make_token_sample / make_expert_sample)."""
    import numpy as np
    import torch

    from mixture_experts_layer_pft_gb300 import workloads
    from oracle import moe_oracle as O

    if inp is not None:
        sel = np.sort(np.random.default_rng(w.seed).choice(w.T, size=Ts, replace=False))
        ix = torch.as_tensor(sel, device=inp["x"].device)
        x_s = inp["x"][ix].double().cpu().numpy()
        dy_s = inp["dy"][ix].double().cpu().numpy() if w.backward else None
        Wg = inp["Wg"].double().cpu().numpy()
        bias = None if inp["bias"] is None else inp["bias"].double().cpu().numpy()
    else:
        smp = workloads.make_token_sample(w, Ts, "cpu")
        x_s, Wg = smp["x"].double().numpy(), smp["Wg"].double().numpy()
        dy_s = smp["dy"].double().numpy() if w.backward else None
        bias = None if smp["bias"] is None else smp["bias"].double().numpy()
    # the experts the sample reaches (the oracle's own gate decides)
    experts = np.unique(O.route(x_s, Wg, w.k, bias, w.dtype)["topk_idx"])
    if inp is not None:
        ws = {int(e): tuple(inp[n][int(e)].double().cpu().numpy() for n in ("W1", "W3", "W2")) for e in experts}
    else:
        ws = {e: tuple(t.double().numpy() for t in v) for e, v in workloads.make_expert_sample(w, experts).items()}
    W1 = HostExperts({e: v[0] for e, v in ws.items()}, (w.E, w.h, w.f))
    W3 = HostExperts({e: v[1] for e, v in ws.items()}, (w.E, w.h, w.f))
    W2 = HostExperts({e: v[2] for e, v in ws.items()}, (w.E, w.f, w.h))
    return (x_s, Wg, bias, W1, W3, W2, dy_s), len(experts)


def time_oracle(w, Ts, steps=1, inp=None):
    """Time the oracle on Ts tokens of workload ``w``; returns (seconds per step, experts reached)."""
    args, n_exp = oracle_inputs(w, Ts, inp)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle_step(w, *args)
        times.append(time.perf_counter() - t0)
    return times, n_exp


def cpu_cores():
    n = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    try:
        return int(n) if n else (os.cpu_count() or 1)
    except ValueError:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- main arms


def run_reference(args, w):
    """The oracle, as it stands, timed on the host cores as the reference arm."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    # about 10 s of oracle work per step at most: the warm-up and timed steps end within minutes
    Ts = oracle_sample_tokens(w, budget_flops=float(args.ref_budget_tflop) * 1e12, host_bytes=3e9)
    args_o, n_exp = oracle_inputs(w, Ts)
    for _ in range(args.warmup):
        oracle_step(w, *args_o)
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(w, *args_o)
        ts.append(time.perf_counter() - t0)
    tot = sum(ts)
    flops = model_flops(w, Ts) * len(ts)
    value = flops / tot / 1e12
    sample = (f"{Ts} of {w.T} tokens per step and the {n_exp} experts they reach (weights drawn on the host "
              f"per expert, held in fp64), fp64 numpy, forward{'+backward' if w.backward else ''}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot / len(ts), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; random-init weights)",
        "tokens_per_s": Ts * len(ts) / tot,
        "config": {"workload": workload_desc(w), "sample_tokens": Ts},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def oracle_single_thread(args):
    """The reference arm's sample (one step) in a child process whose BLAS may use one thread:
    the oracle on one core beside the all-core figure."""
    cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--config", str(args.config),
           "--steps", "1", "--warmup", "0"]
    if args.tokens:
        cmd += ["--tokens", str(args.tokens)]
    if args.experts:
        cmd += ["--experts", str(args.experts)]
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        env.pop(k, None)
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300)
        line = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")][-1]
        return {"value": line["value"], "unit": line["unit"], "cores": 1, "kind": "oracle",
                "sample": line["cpu_baseline"]["sample"] + ", one BLAS thread"}
    except Exception as e:  # noqa: BLE001 -- a baseline, not the product: report and go on
        return {"unavailable": f"{type(e).__name__}: {e}"[:200]}


def workload_desc(w):
    return (f"{w.name}: T={w.T} tokens, h={w.h}, E={w.E}, top-k={w.k}, SwiGLU f={w.f}, "
            f"{w.dtype}{' (fp32 gating)' if w.dtype == 'bf16' else ''}, "
            f"{'fwd+bwd' if w.backward else 'fwd only'}{', Zipf router bias' if w.skew else ''}")




def kernel_names(stage, n, w):
    """Names (and source file) of the n launches one stage call makes, in launch order."""
    simt_only = os.environ.get("MOE_PFT_GEMM") == "simt"
    tc = w.dtype == "bf16" and w.h % 128 == 0 and w.f % 128 == 0 and not simt_only
    tc_router = w.h % 64 == 0 and w.E % 16 == 0 and w.E >= 64 and not simt_only
    f32tc = w.dtype == "f32" and w.h % 128 == 0 and w.f % 128 == 0 and not simt_only
    if tc_router:
        # fp32 activations: x is split into bf16 planes too, before each of its two GEMMs
        xs = ["router_split_x"] if w.dtype == "f32" else []
        route = (["router_split_w"] + xs + ["tc_router_fwd", "softmax_topk"], CSRC + "router_tc.cu")
        # route_dlogits also writes d_logits' bf16 planes; the top-k kernel finishes a K-split logits GEMM
        route_bwd = ((["route_dlogits"] + xs + ["tc_router_dwg", "router_split_w", "tc_router_dx"] if n == 4 + len(xs)
                      else ["route_dlogits"] + xs + ["tc_router_dwg", "router_dwg_splitk_reduce", "router_split_w",
                                                     "tc_router_dx"]), CSRC + "router_tc.cu")
    else:
        route = (["router_gemm", "softmax_topk"] if n == 2 else ["router_gemm", "router_splitk_reduce", "softmax_topk"],
                 CSRC + "gemm_simt.cu")
        route_bwd = ((["route_dlogits", "router_dwg", "router_dx"] if n == 3
                      else ["route_dlogits", "router_dwg", "router_dwg_splitk_reduce", "router_dx"]),
                     CSRC + "gemm_simt.cu")
    table = {
        "route": route,
        "pft_build": (["pft_count", "pft_scan", "pft_scatter"], CSRC + "pft.cu"),
        "dispatch": (["dispatch"], CSRC + "gather.cu"),
        "expert_ffn": ((["tc_GATEUP", "tc_DOWN"], CSRC + "gemm_tc.cu") if tc
                       else (["f32_split_x", "f32_split_w1", "f32tc_H1", "f32tc_H3A", "f32tc_Y"],
                             CSRC + "gemm_f32tc.cu") if f32tc
                       else ((["simt_gateup", "simt_down"] if n == 2 else ["simt_h1", "simt_h3_swiglu", "simt_down"]),
                             CSRC + "gemm_simt.cu")),
        "combine": (["combine"], CSRC + "gather.cu"),
        "combine_bwd": (["combine_bwd"], CSRC + "gather.cu"),
        "expert_ffn_bwd": ((["tc_DA", "tc_DX", "tc_WGRAD13", "tc_WGRAD2"], CSRC + "gemm_tc.cu") if tc
                           # fp32 with the rows gathered from x: they land in dxbuf first
                           else ((["simt_dA", "simt_dW13", "simt_dX", "simt_dW2"] if n == 4 else
                                  ["gather_rows", "simt_dA", "simt_dW13", "simt_dX", "simt_dW2"]),
                                 CSRC + "gemm_simt.cu")),
        "route_bwd": route_bwd,
        "dispatch_bwd": (["dispatch_bwd"], CSRC + "gather.cu"),
    }
    names, src = table[stage]
    if stage in ("dispatch", "combine") and n == 0:  # folded into the expert GEMMs
        return [], src
    if len(names) != n:  # a launch sequence this table does not know: numbered, not named
        return [f"{stage}#{j}" for j in range(n)], src
    return names, src


def kernel_counts(w, T, e_active):
    """Algorithmic FLOPs and HBM bytes of one launch of each kernel."""
    s = 2 if w.dtype == "bf16" else 4
    h, E, k, f = w.h, w.E, w.k, w.f
    Tk = T * k
    Wb = h * f * s  # bytes of one expert's weight matrix
    d = {
        "router_gemm": {"flops": 2 * T * h * E, "bytes": T * h * s + h * E * 4 + T * E * 4},
        "router_splitk_reduce": {"flops": 0, "bytes": 2 * T * E * 4},
        "softmax_topk": {"flops": 0, "bytes": 2 * T * E * 4 + 8 * Tk},
        "pft_count": {"flops": 0, "bytes": 4 * Tk},
        "pft_scan": {"flops": 0, "bytes": 8 * E},
        "pft_scatter": {"flops": 0, "bytes": 16 * Tk},
        "dispatch": {"flops": 0, "bytes": T * h * s + Tk * h * s + 4 * Tk},
        "gather_rows": {"flops": 0, "bytes": T * h * s + Tk * h * s + 4 * Tk},
        "tc_GATEUP": {"flops": 4 * Tk * h * f, "bytes": 2 * e_active * Wb + Tk * h * s + 3 * Tk * f * s},
        "tc_DOWN": {"flops": 2 * Tk * h * f, "bytes": e_active * Wb + Tk * f * s + Tk * h * s},
        "combine": {"flops": 2 * Tk * h, "bytes": Tk * h * s + T * h * s + 8 * Tk},
        "combine_bwd": {"flops": 3 * Tk * h, "bytes": T * h * s + 2 * Tk * h * s + 12 * Tk},
        "tc_DA": {"flops": 2 * Tk * h * f, "bytes": e_active * Wb + Tk * h * s + 4 * Tk * f * s},
        "tc_DX": {"flops": 4 * Tk * h * f, "bytes": 2 * e_active * Wb + 2 * Tk * f * s + Tk * h * s},
        "tc_WGRAD13": {"flops": 4 * Tk * h * f, "bytes": Tk * h * s + 2 * Tk * f * s + 2 * E * Wb},
        "tc_WGRAD2": {"flops": 2 * Tk * h * f, "bytes": Tk * h * s + Tk * f * s + E * Wb},
        "route_dlogits": {"flops": 0, "bytes": 2 * T * E * 4 + 12 * Tk},  # (+ 6 * T * E with the planes)
        # tensor-core router: exact three-plane bf16 splits of the fp32 operands, then the GEMMs
        "router_split_w": {"flops": 0, "bytes": h * E * 4 + 3 * h * E * 2},
        "router_split_dl": {"flops": 0, "bytes": T * E * 4 + 3 * T * E * 2},
        "router_split_x": {"flops": 0, "bytes": T * h * 4 + 3 * T * h * 2},
        "tc_router_fwd": {"flops": 2 * T * h * E, "bytes": T * h * s + 3 * h * E * 2 + T * E * 4},
        "tc_router_dwg": {"flops": 2 * T * h * E, "bytes": T * h * s + 3 * T * E * 2 + h * E * 4},
        "tc_router_dx": {"flops": 2 * T * h * E, "bytes": 3 * T * E * 2 + 3 * h * E * 2 + T * h * 4},
        "router_dwg": {"flops": 2 * T * h * E, "bytes": T * h * s + T * E * 4 + h * E * 4},
        "router_dwg_splitk_reduce": {"flops": 0, "bytes": 2 * h * E * 4},
        "router_dx": {"flops": 2 * T * h * E, "bytes": T * E * 4 + h * E * 4 + T * h * 4},
        "dispatch_bwd": {"flops": 0, "bytes": Tk * h * s + T * h * s + T * h * 4 + 4 * Tk},
    }
    # fp32 expert forward on the tensor cores: exact three-plane bf16 splits, then one GEMM per
    # product (the FLOPs are the fp32 GEMM's; the tensor cores do six plane products for each)
    d["f32_split_x"] = {"flops": 0, "bytes": Tk * h * 4 + 3 * Tk * h * 2}
    # W1's planes have their own launch; H1 and H3A split W3 and W2 (the next GEMM's weights)
    # in a side warp while they run
    wsplit = e_active * h * f * (4 + 6)
    d["f32_split_w1"] = {"flops": 0, "bytes": wsplit}
    d["f32tc_H1"] = {"flops": 2 * Tk * h * f,
                     "bytes": 3 * e_active * h * f * 2 + 3 * Tk * h * 2 + Tk * f * 4 + wsplit}
    d["f32tc_H3A"] = {"flops": 2 * Tk * h * f,
                      "bytes": 3 * e_active * h * f * 2 + 3 * Tk * h * 2 + Tk * f * 4 * 3 + 3 * Tk * f * 2 + wsplit}
    d["f32tc_Y"] = {"flops": 2 * Tk * h * f, "bytes": 3 * e_active * h * f * 2 + 3 * Tk * f * 2 + Tk * h * 4}
    d["simt_h1"] = {"flops": 2 * Tk * h * f, "bytes": e_active * Wb + Tk * h * s + Tk * f * s}
    d["simt_h3_swiglu"] = {"flops": 2 * Tk * h * f, "bytes": e_active * Wb + Tk * h * s + 3 * Tk * f * s}
    for a, bname in (("simt_gateup", "tc_GATEUP"), ("simt_down", "tc_DOWN"), ("simt_dA", "tc_DA"),
                     ("simt_dX", "tc_DX"), ("simt_dW13", "tc_WGRAD13"), ("simt_dW2", "tc_WGRAD2")):
        d[a] = d[bname]
    return d


def stage_calls(binding, w, inp, b):
    """The layer step's C-ABI calls, one per stage (a no-op where a stage is folded away)."""
    calls = [
        lambda: binding.moe_route(inp["x"], inp["Wg"], inp["bias"], w.k, b.logits, b.probs,
                                  b.topk_idx, b.topk_w, b.ws),
        lambda: binding.moe_pft_build(b.topk_idx, w.E, b.num_ids, b.offsets, b.token_ids,
                                      b.expert_ids, b.slot_of, b.ws),
        # fused: no dispatch call; the gate/up GEMM gathers its token rows from x
        (lambda: None) if b.fused else
        (lambda: binding.moe_dispatch(inp["x"], b.token_ids, w.k, b.xbuf, b.ws)),
        (lambda: binding.moe_expert_ffn_fused(b.xbuf, inp["x"], b.token_ids, b.slot_of, b.topk_w, b.offsets,
                                              inp["W1"], inp["W3"], inp["W2"], b.ybuf, b.h1, b.h3, b.a,
                                              b.y, b.ws)) if b.fold_combine else
        (lambda: binding.moe_expert_ffn_gather(inp["x"], b.token_ids, b.offsets, inp["W1"], inp["W3"],
                                               inp["W2"], b.ybuf, b.h1, b.h3, b.a, b.ws)) if b.fused else
        (lambda: binding.moe_expert_ffn(b.xbuf, b.offsets, inp["W1"], inp["W3"], inp["W2"],
                                        b.ybuf, b.h1, b.h3, b.a, b.ws)),
        # fold_combine: the down projection already wrote y
        (lambda: None) if b.fold_combine else
        (lambda: binding.moe_combine(b.ybuf, b.slot_of, b.topk_w, b.y, b.ws)),
    ]
    if w.backward:
        calls += [
            lambda: binding.moe_combine_bwd(inp["dy"], b.ybuf, b.slot_of, b.topk_w, b.dybuf,
                                            b.d_topk_w, b.ws),
            (lambda: binding.moe_expert_ffn_bwd_gather(b.dybuf, inp["x"], b.token_ids, b.h1, b.h3, b.a,
                                                       b.offsets, inp["W1"], inp["W3"], inp["W2"],
                                                       b.dxbuf, b.dW1, b.dW3, b.dW2, b.ws)) if b.fused else
            (lambda: binding.moe_expert_ffn_bwd(b.dybuf, b.xbuf, b.h1, b.h3, b.a, b.offsets,
                                                inp["W1"], inp["W3"], inp["W2"], b.dxbuf,
                                                b.dW1, b.dW3, b.dW2, b.ws)),
            lambda: binding.moe_route_bwd(inp["x"], inp["Wg"], b.probs, b.topk_idx, b.d_topk_w,
                                          b.d_logits, b.dWg, b.dx_router, b.ws),
            lambda: binding.moe_dispatch_bwd(b.dxbuf, b.slot_of, b.dx_router, w.k, b.dx, b.ws),
        ]
    return calls


def run_calls(calls, stream, ev=None, timer=None, spans=None):
    """One step with an event before each stage call and one after the last.  With a kernel
    timer, spans[i] = (first, last) ring index of the launches call i made."""
    for i, c in enumerate(calls):
        if ev is not None:
            ev[i].record(stream)
        n0 = timer.count() if timer else 0
        c()
        if timer is not None:
            spans.append((n0, timer.count()))
    if ev is not None:
        ev[len(calls)].record(stream)


def measure_layer(w, T, inp, b, steps, warmup, flush, world, device, no_graph=False, clocks=None):
    """Warm-up, the timed region (whole steps; the captured step replayed as a CUDA graph unless
    no_graph, L2 flushed between steps outside the events) and the breakdown pass (an event
    before each stage call and after each kernel launch).  Returns a dict of the measurements."""
    import torch

    from mixture_experts_layer_pft_gb300 import binding, layer

    lib = binding.lib()
    stream = torch.cuda.current_stream()
    calls = stage_calls(binding, w, inp, b)
    nst = len(calls)
    for _ in range(warmup):
        run_calls(calls, stream)
    torch.cuda.synchronize()
    assert binding.moe_check_status(b.ws) == 0, "device status set during warm-up"

    graph = None if no_graph else layer.CapturedStep(lambda: run_calls(calls, stream))
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
    if clocks is not None:
        clocks.start()
    n_launch0 = lib.moe_kernel_launches()
    barrier(world)
    torch.cuda.synchronize()
    for s in range(steps):
        flush.zero_()
        step_ev[s][0].record(stream)
        if graph is not None:
            graph.replay()
        else:
            run_calls(calls, stream)
        step_ev[s][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = graph.launches * steps if graph is not None else lib.moe_kernel_launches() - n_launch0
    clk = clocks.stop() if clocks is not None else None
    assert binding.moe_check_status(b.ws) == 0, "device status set during the timed region"
    step_ms = [a.elapsed_time(e) for a, e in step_ev]
    total_ms = max_over_ranks(sum(step_ms), world, device)

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(steps)]
    timer = binding.KernelTimer(64 * steps)
    spans = [[] for _ in range(steps)]
    with timer:
        torch.cuda.synchronize()
        for s in range(steps):
            flush.zero_()
            run_calls(calls, stream, events[s], timer, spans[s])
        torch.cuda.synchronize()
    assert binding.moe_check_status(b.ws) == 0, "device status set during the breakdown pass"
    stage_ms = {STAGES[i]: [events[s][i].elapsed_time(events[s][i + 1]) for s in range(steps)]
                for i in range(nst)}
    kern_ms, kern_src = {}, {}
    for s in range(steps):
        for i, (a0, a1) in enumerate(spans[s]):
            names, src = kernel_names(STAGES[i], a1 - a0, w)
            prev = events[s][i]
            for j, q in enumerate(range(a0, a1)):
                ev = timer.event(q)
                kern_ms.setdefault(names[j], []).append(prev.elapsed_time(ev))
                kern_src[names[j]] = src
                prev = ev
    del graph
    return {"ms_per_step": total_ms / steps, "launches": int(launches),
            "per_step_launches": int(launches // steps), "graph": not no_graph, "clocks": clk,
            "stage_ms": stage_ms, "kern_ms": kern_ms, "kern_src": kern_src,
            "e_active": int((b.num_ids > 0).sum().item())}


def kernel_table(w, T, m):
    """Per-kernel average time, GB/s and TFLOP/s from a measure_layer result."""
    kc = kernel_counts(w, T, m["e_active"])
    kernels = {}
    for n, ms in m["kern_ms"].items():
        avg = sum(ms) / len(ms)
        c = kc.get(n, {"flops": 0, "bytes": 0})
        kernels[n] = {"us": round(1e3 * avg, 2), "GB/s": round(c["bytes"] / (avg * 1e-3) / 1e9, 1)}
        if c["flops"]:
            kernels[n]["TFLOP/s"] = round(c["flops"] / (avg * 1e-3) / 1e12, 2)
    return kernels, kc


def measure_pft_scaled(binding, flush, peaks, steps=20, T=1 << 20, k=8, E=256, seed=20):
    """moe_pft_build at a size where its HBM fraction means something (T = 2^20 tokens, k = 8,
    E = 256: 8.4 M routed rows): the mean of `steps` launches, L2 flushed before each, with the
    two kernels timed apart through the library's event ring."""
    import torch

    from mixture_experts_layer_pft_gb300 import workloads

    dev = flush.device
    logits = workloads.random_logits(T, E, seed, dev)
    idx = torch.topk(logits, k, dim=1).indices.to(torch.int32).contiguous()
    del logits
    Tk = T * k
    out = {n: torch.empty(Tk, dtype=torch.int32, device=dev) for n in ("token_ids", "expert_ids", "slot_of")}
    num_ids = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    ws = binding.new_workspace(binding.MOE_OP_PFT_BUILD, T, 8, E, k, 8, torch.float32, dev)
    stream = torch.cuda.current_stream()

    def call():
        binding.moe_pft_build(idx, E, num_ids, offsets, out["token_ids"], out["expert_ids"], out["slot_of"], ws)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    timer = binding.KernelTimer(8 * steps)
    per_kernel = []
    with timer:
        for s in range(steps):
            flush.zero_()
            ev[s][0].record(stream)
            n0 = timer.count()
            call()
            n1 = timer.count()
            ev[s][1].record(stream)
            per_kernel.append((n0, n1))
        torch.cuda.synchronize()
    assert binding.moe_check_status(ws) == 0, "device status set by the scaled PFT build"
    us = 1e3 * sum(a.elapsed_time(e) for a, e in ev) / steps
    kus = {}
    names = ["pft_count", "pft_scan", "pft_scatter"]
    for s, (n0, n1) in enumerate(per_kernel):
        prev = ev[s][0]
        for j, q in enumerate(range(n0, n1)):
            e = timer.event(q)
            name = names[j] if n1 - n0 == len(names) else f"launch{j}"
            kus.setdefault(name, []).append(1e3 * prev.elapsed_time(e))
            prev = e
    byts = 16 * Tk + 8 * E + 4
    gbs = byts / (us * 1e-6) / 1e9
    return {"T": T, "k": k, "E": E, "rows": Tk, "us": round(us, 2), "GB/s": round(gbs, 1),
            "frac_of_hbm": round(gbs / float(peaks["hbm_gbs"]), 4),
            "algorithmic_bytes": byts, "bytes_note": "topk_idx read once (4 Tk) + token_ids, expert_ids, "
            "slot_of written (12 Tk) + num_ids, offsets",
            "kernels_us": {n: round(sum(v) / len(v), 2) for n, v in kus.items()},
            "l2": "flushed before each launch (256 MB write)"}


def measure_supplementary(w, inp, peaks, flush, world, device, steps, warmup, T=16384):
    """The Large layer shape at T tokens per GPU (512 rows per expert at T = 16384), where the
    expert GEMMs' arithmetic intensity is above the bf16 ridge: step time, layer TFLOP/s and the
    fraction of the measured bf16 peak, for the step and for the tensor-core expert GEMMs alone."""
    import torch

    from mixture_experts_layer_pft_gb300 import layer, workloads

    ws_ = w.with_tokens(T)
    tok = workloads.make_token_sample(ws_, T, device)
    sup = {"x": tok["x"], "dy": tok["dy"], "Wg": inp["Wg"], "bias": inp["bias"],
           "W1": inp["W1"], "W3": inp["W3"], "W2": inp["W2"]}
    b = layer.LayerBuffers(T, w.h, w.E, w.k, w.f, w.torch_dtype(), device, backward=w.backward)
    m = measure_layer(ws_, T, sup, b, steps, warmup, flush, world, device)
    kernels, kc = kernel_table(ws_, T, m)
    fkey = "bf16_tflops"
    peak = float(peaks[fkey])
    flops = model_flops(ws_, T)
    gemm = [n for n in kernels if n.startswith("tc_") and not n.startswith("tc_router")]
    gemm_ms = sum(sum(m["kern_ms"][n]) / len(m["kern_ms"][n]) for n in gemm)
    gemm_flops = sum(kc[n]["flops"] for n in gemm)
    out = {"workload": f"{w.name} at T={T} tokens (Tk={T * w.k}, {T * w.k // w.E} rows per expert on average)",
           "ms_per_step": round(m["ms_per_step"], 4),
           "TFLOP/s": round(flops / (m["ms_per_step"] * 1e-3) / 1e12, 2),
           "tensor_frac_step": round(flops / (m["ms_per_step"] * 1e-3) / (peak * 1e12), 4),
           "expert_gemms": {"ms": round(gemm_ms, 4), "TFLOP/s": round(gemm_flops / (gemm_ms * 1e-3) / 1e12, 2),
                            "tensor_frac": round(gemm_flops / (gemm_ms * 1e-3) / (peak * 1e12), 4)},
           "kernels": {n: kernels[n] for n in gemm},
           "peak": f"MEASURED_PEAKS.json {fkey} = {peak}", "steps": steps}
    del b
    return out


def measure_gshard(flush, device, cfg=1, reps=20):
    """The capacity-buffer (GShard-style) forward beside the padding-free one on workload ``cfg``
    (X-MoE Small: the pages' ablation compares gating, dispatch and combine there), C = the largest
    expert load so that both compute the same layer.  Each stage is timed on its own, L2 flushed
    before it, averaged over ``reps``."""
    import torch

    from mixture_experts_layer_pft_gb300 import binding, layer, workloads

    w = workloads.WORKLOADS[cfg]
    inp = workloads.make_inputs(w, device)
    pb = layer.LayerBuffers(w.T, w.h, w.E, w.k, w.f, w.torch_dtype(), device, backward=False)
    layer.forward(inp, pb)
    torch.cuda.synchronize()
    C = int(pb.num_ids.max().item())
    gb = layer.GShardBuffers(w.T, w.h, w.E, w.k, w.f, C, w.torch_dtype(), device)
    layer.gshard_forward(inp, gb)
    torch.cuda.synchronize()
    g_calls = layer.gshard_forward(inp, gb, stages=True)
    route = lambda: binding.moe_route(inp["x"], inp["Wg"], inp["bias"], w.k, pb.logits, pb.probs,  # noqa: E731
                                      pb.topk_idx, pb.topk_w, pb.ws)
    pft = {
        "gating": lambda: (route(), binding.moe_pft_build(pb.topk_idx, w.E, pb.num_ids, pb.offsets, pb.token_ids,
                                                          pb.expert_ids, pb.slot_of, pb.ws)),
        "dispatch": lambda: binding.moe_dispatch(inp["x"], pb.token_ids, w.k, pb.xbuf, pb.ws),
        "experts": lambda: binding.moe_expert_ffn(pb.xbuf, pb.offsets, inp["W1"], inp["W3"], inp["W2"], pb.ybuf,
                                                  pb.h1, pb.h3, pb.a, pb.ws),
        "combine": lambda: binding.moe_combine(pb.ybuf, pb.slot_of, pb.topk_w, pb.y, pb.ws),
    }
    gsh = dict(zip(("gating", "dispatch", "experts", "combine"), g_calls))
    stream = torch.cuda.current_stream()

    def timed(fn):
        fn()
        ms = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return 1e3 * sum(ms) / len(ms)

    out = {"workload": workload_desc(w) + " (forward)", "capacity_C": C, "stages_us": {}}
    for n in ("gating", "dispatch", "experts", "combine"):
        tp, tg = timed(pft[n]), timed(gsh[n])
        out["stages_us"][n] = {"pft": round(tp, 2), "capacity_buffer": round(tg, 2),
                               "speedup": round(tg / tp, 2)}
    tp = sum(v["pft"] for v in out["stages_us"].values())
    tg = sum(v["capacity_buffer"] for v in out["stages_us"].values())
    out["forward_us"] = {"pft": round(tp, 2), "capacity_buffer": round(tg, 2), "speedup": round(tg / tp, 2)}
    s = 2 if w.dtype == "bf16" else 4
    out["buffer_bytes"] = {"pft_token_buffers": 2 * w.Tk * w.h * s,
                           "capacity_buffers": 2 * w.E * C * w.h * s + w.T * w.E * C * (s + 4)}
    diff = (gb.y.float() - pb.y.float()).norm() / pb.y.float().norm()
    out["rel_l2_y_vs_pft"] = float(diff)
    assert binding.moe_check_status(gb.ws_gshard) == 0 and binding.moe_check_status(pb.ws) == 0
    out["note"] = ("the pages' X-MoE ablation (Small, AMD MI250X) reports 5.7x / 35.7x / 8.1x for gating / "
                   "dispatch / combine; these are the same stages on one GB300")
    del gb, pb
    return out


def run_ours(args, w):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())

    from mixture_experts_layer_pft_gb300 import binding, build, layer, workloads

    build.build()
    binding.lib()
    T = w.T
    inp = workloads.make_inputs(w, device, token_seed=None if world == 1 else w.seed + 7919 * rank)
    b = layer.LayerBuffers(T, w.h, w.E, w.k, w.f, w.torch_dtype(), device, backward=w.backward,
                           fused=args.fused, fold_combine=args.fold_combine)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)  # 2x the 129 MB L2
    stream = torch.cuda.current_stream()

    # ---------------------------------------------------------------- timed region + breakdown pass
    m = measure_layer(w, T, inp, b, args.steps, args.warmup, flush, world, device, args.no_graph,
                      ClockSampler(device.index))
    ms_per_step = m["ms_per_step"]
    flops = model_flops(w, T)
    value = world * flops / (ms_per_step * 1e-3) / 1e12

    counts = stage_counts(w, T)
    stages = {}
    for n, ms in m["stage_ms"].items():
        avg = sum(ms) / len(ms)
        c = counts[n]
        if (b.fused and n == "dispatch") or (b.fold_combine and n == "combine"):
            stages[n] = {"ms": round(avg, 4), "GB/s": None, "note": "no launch: folded into the expert GEMMs"}
            continue
        stages[n] = {"ms": round(avg, 4), "GB/s": round(c["bytes"] / (avg * 1e-3) / 1e9, 1)}
        if c["flops"] and n.startswith(("expert", "route")):
            stages[n]["TFLOP/s"] = round(c["flops"] / (avg * 1e-3) / 1e12, 2)
    kernels, kc = kernel_table(w, T, m)
    kern_ms, kern_src = m["kern_ms"], m["kern_src"]

    # ---------------------------------------------------------------- roofline of the dominant kernel
    peaks, peak_src = read_peaks()
    known = [n for n in kern_ms if n in kc]
    dom = max(known, key=lambda n: sum(kern_ms[n]) / len(kern_ms[n]))
    dom_ms = sum(kern_ms[dom]) / len(kern_ms[dom])
    c = kc[dom]
    region_ms = ms_per_step * args.steps
    fkey = "bf16_tflops_sustained" if region_ms > 2000 else "bf16_tflops"
    if dom.startswith("f32tc_"):
        # six exact bf16 plane products per fp32 product: the tensor work is 6x the GEMM's FLOPs
        roof = {"bound": "tensor", "achieved": 6 * c["flops"] / (dom_ms * 1e-3) / 1e12,
                "peak": float(peaks[fkey]), "unit": "TFLOP/s"}
        which = (f"MEASURED_PEAKS.json {fkey} ({'of measured' if peak_src == 'measured' else 'of fallback'}); "
                 "achieved counts the six bf16 plane products of each fp32 product")
    elif dom.startswith("simt") or dom in ("router_gemm", "router_dwg", "router_dx"):
        roof = {"bound": "alu", "achieved": c["flops"] / (dom_ms * 1e-3) / 1e12,
                "peak": FP32_ALU_TFLOPS_NOMINAL, "unit": "TFLOP/s"}
        which = "derived FP32 FMA peak: 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz (nominal)"
    else:
        t_tensor = c["flops"] / (float(peaks[fkey]) * 1e12) if c["flops"] else 0.0
        t_hbm = c["bytes"] / (float(peaks["hbm_gbs"]) * 1e9)
        if t_tensor > t_hbm:
            roof = {"bound": "tensor", "achieved": c["flops"] / (dom_ms * 1e-3) / 1e12,
                    "peak": float(peaks[fkey]), "unit": "TFLOP/s"}
            which = f"MEASURED_PEAKS.json {fkey} ({'of measured' if peak_src == 'measured' else 'of fallback'})"
        else:
            roof = {"bound": "hbm", "achieved": c["bytes"] / (dom_ms * 1e-3) / 1e9,
                    "peak": float(peaks["hbm_gbs"]), "unit": "GB/s"}
            which = f"MEASURED_PEAKS.json hbm_gbs ({'of measured' if peak_src == 'measured' else 'of fallback'})"
        if c["flops"]:
            roof["tensor_frac"] = c["flops"] / (dom_ms * 1e-3) / (float(peaks[fkey]) * 1e12)
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = recorded_traffic(f"{dom}:{w.name}", source_hash([kern_src[dom]] + KERNEL_HEADERS))
    roof["kernel"] = dom
    roof["launch_us"] = round(1e3 * dom_ms, 2)
    roof["peak_source"] = which
    roof["algorithmic_per_launch"] = {"flops": c["flops"], "bytes": c["bytes"]}

    # ---------------------------------------------------------------- the grouped expert GEMMs together
    # the fraction of the tensor peak, and of the true roofline: per kernel the longer of its
    # FLOPs at the bf16 peak and its algorithmic bytes at the copy peak, summed, over the time
    gemm_names = [n for n in known if n.startswith("tc_") and not n.startswith("tc_router")]
    expert_gemms = None
    if gemm_names:
        gms = sum(sum(kern_ms[n]) / len(kern_ms[n]) for n in gemm_names)
        gfl = sum(kc[n]["flops"] for n in gemm_names)
        bound_ms = sum(max(kc[n]["flops"] / (float(peaks[fkey]) * 1e12),
                           kc[n]["bytes"] / (float(peaks["hbm_gbs"]) * 1e9)) * 1e3 for n in gemm_names)
        expert_gemms = {"kernels": gemm_names, "ms": round(gms, 4),
                        "TFLOP/s": round(gfl / (gms * 1e-3) / 1e12, 2),
                        "tensor_frac": round(gfl / (gms * 1e-3) / (float(peaks[fkey]) * 1e12), 4),
                        "roofline_ms": round(bound_ms, 4), "roofline_frac": round(bound_ms / gms, 4),
                        "peaks": f"MEASURED_PEAKS.json {fkey} and hbm_gbs"}

    # ---------------------------------------------------------------- end to end through host buffers
    e2e = None
    if not args.no_e2e:
        hx = torch.empty_like(inp["x"], device="cpu").pin_memory()
        hx.copy_(inp["x"])
        hdy = torch.empty_like(inp["dy"], device="cpu").pin_memory()
        hdy.copy_(inp["dy"])
        hy = torch.empty_like(b.y, device="cpu").pin_memory()
        hdx = torch.empty_like(b.dx, device="cpu").pin_memory() if w.backward else None
        # The layer's two-slot host pipeline: step i + 1's upload and step i's downloads run on
        # copy streams beside the compute.  Every step's copies are inside the timed region; the
        # first upload and the last download are exposed.  No L2 flush between these steps: the
        # weights every step reads (and the per-step traffic) are far larger than L2.
        pipe = layer.HostPipeline(inp, b, graphs=not args.no_graph)
        for _ in range(args.warmup):
            pipe.submit(hx, hy, hdy, hdx)
        pipe.finish()
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            pipe.submit(hx, hy, hdy, hdx)
        pipe.finish()
        e1.record(stream)
        e1.synchronize()
        e_ms = [e0.elapsed_time(e1)]
        e_steps = args.steps
        e2e_ms = max_over_ranks(sum(e_ms), world, device) / e_steps
        bi = hx.numel() * hx.element_size() + (hdy.numel() * hdy.element_size() if w.backward else 0)
        bo = hy.numel() * hy.element_size() + (hdx.numel() * hdx.element_size() if w.backward else 0)
        e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms,
               "copies": "pinned host buffers; layer.HostPipeline overlaps step i+1's upload and step i's "
                         "downloads with the compute (two device slots for x, dy, y and dx, each slot's step "
                         "one captured CUDA graph), all inside the timed region; no L2 flush between steps "
                         "(weights larger than L2)"}
        del pipe

    # ---------------------------------------------------------------- CPU oracle baseline (rank 0, N = 1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        Ts = oracle_sample_tokens(w)
        ts, n_exp = time_oracle(w, Ts, 1, inp)
        cpu = {"value": model_flops(w, Ts) / ts[0] / 1e12, "unit": "TFLOPS", "cores": cpu_cores(),
               "kind": "oracle",
               "sample": f"one {'forward+backward' if w.backward else 'forward'} of a seeded {Ts} of {w.T} "
                         f"tokens and the {n_exp} experts they reach (the benchmark's own inputs), fp64 "
                         f"numpy/OpenBLAS, {ts[0]:.1f} s; value = sample FLOPs / time"}
        if not args.no_single_thread:
            cpu["single_thread"] = oracle_single_thread(args)

    # ---------------------------------------------------------------- scaled PFT build and the T = 16384 run
    pft_scaled = None if args.no_pft_scaled else measure_pft_scaled(binding, flush, peaks)
    gshard = None
    if not args.no_gshard:
        gshard = measure_gshard(flush, device)
    supplementary = None
    is_large = (w.h, w.E, w.k, w.f, w.dtype) == (7168, 256, 8, 2048, "bf16")
    if is_large and not args.no_supplementary:
        del b
        torch.cuda.empty_cache()
        supplementary = measure_supplementary(w, inp, peaks, flush, world, device, steps=min(args.steps, 10),
                                              warmup=3)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic (seeded N(0,1) tokens, random-init weights)",
            "tokens_per_s": world * T / (ms_per_step * 1e-3),
            "dispatch_GBps": None if args.fused else stages["dispatch"]["GB/s"],
            "combine_GBps": None if args.fold_combine else stages["combine"]["GB/s"],
            "config": {"workload": workload_desc(w), "tokens_per_gpu": T,
                       "l2": "flushed between timed steps (256 MB write, outside the step events)",
                       "step": ("one host call per stage" if args.no_graph else
                                f"CUDA graph replay of the captured layer step ({m['per_step_launches']} "
                                f"library kernels)"),
                       "breakdown": "stages and kernels timed in a second pass with an event after each launch",
                       "dispatch": ("folded into the gate/up and dW1/dW3 GEMMs (rows gathered from x)"
                                    if args.fused else "its own kernel writing the padding-free buffer"),
                       "combine": ("folded into the down projection's epilogue" if args.fold_combine
                                   else "its own kernel over ybuf"),
                       "parallelism": f"replicas x{world} (independent tokens, no data-path collective)"},
            "stages": stages,
            "kernels": kernels,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "expert_gemms": expert_gemms,
            "pft_scaled": pft_scaled,
            "supplementary": supplementary,
            "gshard": gshard,
            "gpu_launches": m["launches"],
            "clocks": m["clocks"],
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fused", action="store_true",
                    help="fold dispatch into the expert GEMMs (tensor-core paths, bf16 or fp32; rows gathered from x)")
    ap.add_argument("--fold-combine", action="store_true",
                    help="fold the combine into the down projection (bf16 tensor-core path, h % 256 == 0)")
    ap.add_argument("--no-graph", action="store_true",
                    help="time steps as one host call per stage instead of a CUDA graph replay")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-single-thread", action="store_true",
                    help="skip the one-thread oracle timing beside the all-core cpu_baseline")
    ap.add_argument("--no-pft-scaled", action="store_true",
                    help="skip the PFT build at T = 2^20, k = 8, E = 256")
    ap.add_argument("--tokens", type=int, default=0, help="override the workload's token count T")
    ap.add_argument("--experts", type=int, default=0, help="override the workload's expert count E")
    ap.add_argument("--no-gshard", action="store_true",
                    help="skip the capacity-buffer (GShard-style) stages timed beside the PFT ones")
    ap.add_argument("--no-supplementary", action="store_true",
                    help="skip the Large layer shape at T = 16384 (run with the Large workload only)")
    ap.add_argument("--ref-budget-tflop", type=float, default=0.1,
                    help="reference arm: algorithmic TFLOP per step of the oracle sample")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    from mixture_experts_layer_pft_gb300 import workloads

    w = workloads.WORKLOADS[args.config]
    if args.tokens or args.experts:
        # a slice of the workload with the same expert shape (profiling captures stay small)
        import dataclasses

        T = args.tokens or w.T
        E = args.experts or w.E
        w = dataclasses.replace(w, T=T, E=E, name=f"{w.name}-slice-T{T}-E{E}")
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
