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
DEFAULT_CONFIG = 1  # the X-MoE Small layer, bf16, forward + backward
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
    """nvidia-smi samples every 200 ms while the timed region runs."""

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
                 "-lms", "200", "-i", str(self.gpu)],
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


def oracle_sample_tokens(w, budget_flops=1.2e12):
    """Token count of a bounded oracle sample (about 10-30 s of fp64 numpy on a CPU host)."""
    per_tok = model_flops(w, 1)
    return int(max(16, min(w.T, budget_flops // per_tok)))


def time_oracle(w, Ts, steps=1):
    """Time the oracle on Ts tokens of workload ``w`` (inputs drawn on the CPU)."""
    from mixture_experts_layer_pft_gb300 import workloads
    from oracle import moe_oracle as O

    inp = workloads.make_inputs(w, "cpu", T=Ts)
    c = {k: (None if v is None else v.double().numpy()) for k, v in inp.items()}
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        fw = O.layer_forward(c["x"], c["Wg"], c["W1"], c["W3"], c["W2"], w.k, c["bias"], w.dtype)
        if w.backward:
            O.layer_backward(fw, c["x"], c["Wg"], c["W1"], c["W3"], c["W2"], c["dy"], w.dtype)
        times.append(time.perf_counter() - t0)
    return times


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
    Ts = oracle_sample_tokens(w, budget_flops=float(args.ref_budget_tflop) * 1e12)
    for _ in range(args.warmup):
        time_oracle(w, Ts, 1)
    ts = time_oracle(w, Ts, args.steps)
    tot = sum(ts)
    flops = model_flops(w, Ts) * len(ts)
    value = flops / tot / 1e12
    sample = f"{Ts} of {w.T} tokens per step (full expert set), fp64 numpy, forward{'+backward' if w.backward else ''}"
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


def workload_desc(w):
    return (f"{w.name}: T={w.T} tokens, h={w.h}, E={w.E}, top-k={w.k}, SwiGLU f={w.f}, "
            f"{w.dtype}{' (fp32 gating)' if w.dtype == 'bf16' else ''}, "
            f"{'fwd+bwd' if w.backward else 'fwd only'}{', Zipf router bias' if w.skew else ''}")




def kernel_names(stage, n, w):
    """Names (and source file) of the n launches one stage call makes, in launch order."""
    simt_only = os.environ.get("MOE_PFT_GEMM") == "simt"
    tc = w.dtype == "bf16" and w.h % 128 == 0 and w.f % 128 == 0 and not simt_only
    tc_router = w.dtype == "bf16" and w.h % 64 == 0 and w.E % 16 == 0 and w.E >= 64 and not simt_only
    if tc_router:
        route = (["router_split_w", "tc_router_fwd", "softmax_topk"], CSRC + "router_tc.cu")
        # route_dlogits also writes d_logits' bf16 planes; the top-k kernel finishes a K-split logits GEMM
        route_bwd = ((["route_dlogits", "tc_router_dwg", "router_split_w", "tc_router_dx"] if n == 4
                      else ["route_dlogits", "tc_router_dwg", "router_dwg_splitk_reduce", "router_split_w",
                            "tc_router_dx"]), CSRC + "router_tc.cu")
    else:
        route = (["router_gemm", "softmax_topk"] if n == 2 else ["router_gemm", "router_splitk_reduce", "softmax_topk"],
                 CSRC + "gemm_simt.cu")
        route_bwd = ((["route_dlogits", "router_dwg", "router_dx"] if n == 3
                      else ["route_dlogits", "router_dwg", "router_dwg_splitk_reduce", "router_dx"]),
                     CSRC + "gemm_simt.cu")
    table = {
        "route": route,
        "pft_build": (["pft_hist", "pft_scatter"], CSRC + "pft.cu"),
        "dispatch": (["dispatch"], CSRC + "gather.cu"),
        "expert_ffn": ((["tc_GATEUP", "tc_DOWN"], CSRC + "gemm_tc.cu") if tc
                       else ((["simt_gateup", "simt_down"] if n == 2 else ["simt_h1", "simt_h3_swiglu", "simt_down"]),
                             CSRC + "gemm_simt.cu")),
        "combine": (["combine"], CSRC + "gather.cu"),
        "combine_bwd": (["combine_bwd"], CSRC + "gather.cu"),
        "expert_ffn_bwd": ((["tc_DA", "tc_DX", "tc_WGRAD13", "tc_WGRAD2"], CSRC + "gemm_tc.cu") if tc
                           else (["simt_dA", "simt_dX", "simt_dW13", "simt_dW2"], CSRC + "gemm_simt.cu")),
        "route_bwd": route_bwd,
        "dispatch_bwd": (["dispatch_bwd"], CSRC + "gather.cu"),
    }
    names, src = table[stage]
    if stage in ("dispatch", "combine") and n == 0:  # folded into the expert GEMMs
        return [], src
    assert len(names) == n, (stage, n, names)
    return names, src


def kernel_counts(w, T, e_active, binding=None):
    """Algorithmic FLOPs and HBM bytes of one launch of each kernel."""
    s = 2 if w.dtype == "bf16" else 4
    h, E, k, f = w.h, w.E, w.k, w.f
    Tk = T * k
    Wb = h * f * s  # bytes of one expert's weight matrix
    d = {
        "router_gemm": {"flops": 2 * T * h * E, "bytes": T * h * s + h * E * 4 + T * E * 4},
        "router_splitk_reduce": {"flops": 0, "bytes": 2 * T * E * 4},
        "softmax_topk": {"flops": 0, "bytes": 2 * T * E * 4 + 8 * Tk},
        "pft_hist": {"flops": 0, "bytes": 4 * Tk},
        "pft_scatter": {"flops": 0, "bytes": 16 * Tk},
        "dispatch": {"flops": 0, "bytes": T * h * s + Tk * h * s + 4 * Tk},
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
        "tc_router_fwd": {"flops": 2 * T * h * E, "bytes": T * h * s + 3 * h * E * 2 + T * E * 4},
        "tc_router_dwg": {"flops": 2 * T * h * E, "bytes": T * h * s + 3 * T * E * 2 + h * E * 4},
        "tc_router_dx": {"flops": 2 * T * h * E, "bytes": 3 * T * E * 2 + 3 * h * E * 2 + T * h * 4},
        "router_dwg": {"flops": 2 * T * h * E, "bytes": T * h * s + T * E * 4 + h * E * 4},
        "router_dwg_splitk_reduce": {"flops": 0, "bytes": 2 * h * E * 4},
        "router_dx": {"flops": 2 * T * h * E, "bytes": T * E * 4 + h * E * 4 + T * h * 4},
        "dispatch_bwd": {"flops": 0, "bytes": Tk * h * s + T * h * s + T * h * 4 + 4 * Tk},
    }
    d["simt_h1"] = {"flops": 2 * Tk * h * f, "bytes": e_active * Wb + Tk * h * s + Tk * f * s}
    d["simt_h3_swiglu"] = {"flops": 2 * Tk * h * f, "bytes": e_active * Wb + Tk * h * s + 3 * Tk * f * s}
    for a, bname in (("simt_gateup", "tc_GATEUP"), ("simt_down", "tc_DOWN"), ("simt_dA", "tc_DA"),
                     ("simt_dX", "tc_DX"), ("simt_dW13", "tc_WGRAD13"), ("simt_dW2", "tc_WGRAD2")):
        d[a] = d[bname]
    return d


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
    lib = binding.lib()
    T = w.T
    inp = workloads.make_inputs(w, device, token_seed=None if world == 1 else w.seed + 7919 * rank)
    b = layer.LayerBuffers(T, w.h, w.E, w.k, w.f, w.torch_dtype(), device, backward=w.backward,
                           fused=args.fused, fold_combine=args.fold_combine)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)  # 2x the 129 MB L2
    stream = torch.cuda.current_stream()

    def run_stages(ev, timer=None, spans=None):
        """One step with an event before each stage call and one after the last.  With a
        kernel timer, spans[i] = (first, last) ring index of the launches call i made."""
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
        for i, c in enumerate(calls):
            if ev is not None:
                ev[i].record(stream)
            n0 = timer.count() if timer else 0
            c()
            if timer is not None:
                spans.append((n0, timer.count()))
        if ev is not None:
            ev[len(calls)].record(stream)

    nst = len(STAGES) if w.backward else 5
    for _ in range(args.warmup):
        run_stages(None)
    torch.cuda.synchronize()
    assert binding.moe_check_status(b.ws) == 0, "device status set during warm-up"

    # ---------------------------------------------------------------- timed region: whole steps
    # Each step is the captured layer step (CUDA graph replay; --no-graph: one host call per
    # stage), bracketed by one event pair; L2 is flushed between steps, outside the events.
    if args.no_graph:
        graph = None
        per_step = None
    else:
        graph = layer.CapturedStep(lambda: run_stages(None))
        per_step = graph.launches
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    clocks = ClockSampler(device.index)
    clocks.start()
    n_launch0 = lib.moe_kernel_launches()
    barrier(world)
    torch.cuda.synchronize()
    for s in range(args.steps):
        flush.zero_()
        step_ev[s][0].record(stream)
        if graph is not None:
            graph.replay()
        else:
            run_stages(None)
        step_ev[s][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = (per_step * args.steps if graph is not None
                else lib.moe_kernel_launches() - n_launch0)
    clk = clocks.stop()
    assert binding.moe_check_status(b.ws) == 0, "device status set during the timed region"
    step_ms = [a.elapsed_time(e) for a, e in step_ev]
    total_ms = max_over_ranks(sum(step_ms), world, device)

    # ---------------------------------------------------------------- breakdown pass
    # The same steps again, with an event before each stage call and after each kernel launch:
    # per-stage and per-kernel times (the roofline's kernel duration) come from here.
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(args.steps)]
    timer = binding.KernelTimer(64 * args.steps)
    spans = [[] for _ in range(args.steps)]
    with timer:
        torch.cuda.synchronize()
        for s in range(args.steps):
            flush.zero_()
            run_stages(events[s], timer, spans[s])
        torch.cuda.synchronize()
    assert binding.moe_check_status(b.ws) == 0, "device status set during the breakdown pass"
    stage_ms = {STAGES[i]: [events[s][i].elapsed_time(events[s][i + 1]) for s in range(args.steps)]
                for i in range(nst)}
    ms_per_step = total_ms / args.steps
    flops = model_flops(w, T)
    value = world * flops / (ms_per_step * 1e-3) / 1e12

    counts = stage_counts(w, T)
    stages = {}
    for n, ms in stage_ms.items():
        avg = sum(ms) / len(ms)
        c = counts[n]
        if (b.fused and n == "dispatch") or (b.fold_combine and n == "combine"):
            stages[n] = {"ms": round(avg, 4), "GB/s": None, "note": "no launch: folded into the expert GEMMs"}
            continue
        stages[n] = {"ms": round(avg, 4), "GB/s": round(c["bytes"] / (avg * 1e-3) / 1e9, 1)}
        if c["flops"] and n.startswith(("expert", "route")):
            stages[n]["TFLOP/s"] = round(c["flops"] / (avg * 1e-3) / 1e12, 2)

    # ---------------------------------------------------------------- per-kernel times (event ring)
    e_active = int((b.num_ids > 0).sum().item())
    kern_ms = {}  # kernel name -> list of durations (ms)
    kern_src = {}
    for s in range(args.steps):
        for i, (a0, a1) in enumerate(spans[s]):
            names, src = kernel_names(STAGES[i], a1 - a0, w)
            prev = events[s][i]
            for j, q in enumerate(range(a0, a1)):
                ev = timer.event(q)
                kern_ms.setdefault(names[j], []).append(prev.elapsed_time(ev))
                kern_src[names[j]] = src
                prev = ev
    kernels = {}
    kc = kernel_counts(w, T, e_active, binding)
    for n, ms in kern_ms.items():
        avg = sum(ms) / len(ms)
        c = kc.get(n, {"flops": 0, "bytes": 0})
        kernels[n] = {"us": round(1e3 * avg, 2), "GB/s": round(c["bytes"] / (avg * 1e-3) / 1e9, 1)}
        if c["flops"]:
            kernels[n]["TFLOP/s"] = round(c["flops"] / (avg * 1e-3) / 1e12, 2)

    # ---------------------------------------------------------------- roofline of the dominant kernel
    peaks, peak_src = read_peaks()
    dom = max(kern_ms, key=lambda n: sum(kern_ms[n]) / len(kern_ms[n]))
    dom_ms = sum(kern_ms[dom]) / len(kern_ms[dom])
    c = kc[dom]
    region_ms = ms_per_step * args.steps
    fkey = "bf16_tflops_sustained" if region_ms > 2000 else "bf16_tflops"
    if dom.startswith("simt") or dom in ("router_gemm", "router_dwg", "router_dx"):
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

    # ---------------------------------------------------------------- end to end through host buffers
    e2e = None
    if not args.no_e2e:
        hx = torch.empty_like(inp["x"], device="cpu").pin_memory()
        hx.copy_(inp["x"])
        hdy = torch.empty_like(inp["dy"], device="cpu").pin_memory()
        hdy.copy_(inp["dy"])
        hy = torch.empty_like(b.y, device="cpu").pin_memory()
        hdx = torch.empty_like(b.dx, device="cpu").pin_memory() if w.backward else None
        host_step = lambda: layer.step_host(inp, b, hx, hy, hdy, hdx)  # noqa: E731
        hgraph = None if args.no_graph else layer.CapturedStep(host_step)
        e_ms = []
        for s in range(args.steps + args.warmup):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if hgraph is not None:
                hgraph.replay()
            else:
                host_step()
            e1.record(stream)
            e1.synchronize()
            if s >= args.warmup:
                e_ms.append(e0.elapsed_time(e1))
        e2e_ms = max_over_ranks(sum(e_ms), world, device) / len(e_ms)
        bi = hx.numel() * hx.element_size() + (hdy.numel() * hdy.element_size() if w.backward else 0)
        bo = hy.numel() * hy.element_size() + (hdx.numel() * hdx.element_size() if w.backward else 0)
        e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms}

    # ---------------------------------------------------------------- CPU oracle baseline (rank 0, N = 1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        Ts = oracle_sample_tokens(w)
        ts = time_oracle(w, Ts, 1)
        cpu = {"value": model_flops(w, Ts) / ts[0] / 1e12, "unit": "TFLOPS", "cores": cpu_cores(),
               "kind": "oracle",
               "sample": f"one {'forward+backward' if w.backward else 'forward'} of {Ts} of {w.T} tokens "
                         f"(all {w.E} experts' weights), fp64 numpy/OpenBLAS, {ts[0]:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic (seeded N(0,1) tokens, random-init weights)",
            "tokens_per_s": world * T / (ms_per_step * 1e-3),
            "dispatch_GBps": None if b.fused else stages["dispatch"]["GB/s"],
            "combine_GBps": None if b.fold_combine else stages["combine"]["GB/s"],
            "config": {"workload": workload_desc(w), "tokens_per_gpu": T,
                       "l2": "flushed between timed steps (256 MB write, outside the step events)",
                       "step": ("one host call per stage" if args.no_graph else
                                f"CUDA graph replay of the captured layer step ({per_step} library kernels)"),
                       "breakdown": "stages and kernels timed in a second pass with an event after each launch",
                       "dispatch": ("folded into the gate/up and dW1/dW3 GEMMs (rows gathered from x)"
                                    if b.fused else "its own kernel writing the padding-free buffer"),
                       "combine": ("folded into the down projection's epilogue" if b.fold_combine
                                   else "its own kernel over ybuf"),
                       "parallelism": f"replicas x{world} (independent tokens, no data-path collective)"},
            "stages": stages,
            "kernels": kernels,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": int(launches),
            "clocks": clk,
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
                    help="fold dispatch into the expert GEMMs (bf16 tensor-core path; rows gathered from x)")
    ap.add_argument("--fold-combine", action="store_true",
                    help="fold the combine into the down projection (bf16 tensor-core path, h % 256 == 0)")
    ap.add_argument("--no-graph", action="store_true",
                    help="time steps as one host call per stage instead of a CUDA graph replay")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget-tflop", type=float, default=0.1,
                    help="reference arm: algorithmic TFLOP per step of the oracle sample")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    from mixture_experts_layer_pft_gb300 import workloads

    w = workloads.WORKLOADS[args.config]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
