"""One padding-free MoE layer step (forward + backward) over the C ABI.

``LayerBuffers`` allocates every device buffer of the layer once (PyTorch owns the memory);
``forward`` and ``backward`` issue the stage calls in order on the current stream.  Each stage
runs in the library's kernels; this module only sequences them.  ``step_host`` runs a step whose
tokens live in pinned host memory, ``HostPipeline`` runs a stream of such steps with the copies
beside the compute of neighbouring steps, and ``CapturedStep`` replays a captured step as one CUDA
graph.
"""

from __future__ import annotations

import torch

from . import binding as B


class LayerBuffers:
    """Device buffers of one layer.

    With ``fused`` the expert GEMMs gather their token rows from x (the library's
    moe_expert_ffn_gather / moe_expert_ffn_bwd_gather: bf16 or fp32, h and f multiples of 128),
    so the dispatched buffer xbuf is never written and ``xbuf`` is None.  With ``fold_combine``
    the down projection also writes y (moe_expert_ffn_fused; bf16, h a multiple of 256), so no
    combine call runs.  Either way the results are the same bits as the separate calls.  The
    defaults are the separate calls: in bf16 the gathered loads, 16-byte copies from one producer
    warp, keep too few bytes in flight to match the tensor loads of a dispatched buffer.  In fp32
    the gathered forward is the faster one (its row split replaces both the dispatch copy and the
    split of xbuf).
    """

    def __init__(self, T: int, h: int, E: int, k: int, f: int, dtype: torch.dtype, device="cuda",
                 backward: bool = True, gate: str = "softmax", renorm: bool = False,
                 fused: bool = False, fold_combine: bool = False):
        self.T, self.h, self.E, self.k, self.f, self.dtype = T, h, E, k, f, dtype
        if (fused or fold_combine) and not B.moe_expert_ffn_gather_supported(h, f, dtype):
            raise ValueError("fused layer needs bf16 or fp32 with h and f multiples of 128")
        if fold_combine and (h % 256 != 0 or dtype != torch.bfloat16):
            raise ValueError("the combine fold needs bf16 and h a multiple of 256")
        self.fused = bool(fused)
        self.fold_combine = bool(fold_combine)
        self.gate, self.renorm = gate, renorm
        Tk = T * k
        f32, i32 = torch.float32, torch.int32
        d = dict(device=device)
        self.logits = torch.empty(T, E, dtype=f32, **d)
        self.probs = torch.empty(T, E, dtype=f32, **d)
        self.topk_idx = torch.empty(T, k, dtype=i32, **d)
        self.topk_w = torch.empty(T, k, dtype=f32, **d)
        self.num_ids = torch.empty(E, dtype=i32, **d)
        self.offsets = torch.empty(E + 1, dtype=i32, **d)
        self.token_ids = torch.empty(Tk, dtype=i32, **d)
        self.expert_ids = torch.empty(Tk, dtype=i32, **d)
        self.slot_of = torch.empty(Tk, dtype=i32, **d)
        self.xbuf = None if self.fused else torch.empty(Tk, h, dtype=dtype, **d)
        self.h1 = torch.empty(Tk, f, dtype=dtype, **d)
        self.h3 = torch.empty(Tk, f, dtype=dtype, **d)
        self.a = torch.empty(Tk, f, dtype=dtype, **d)
        self.ybuf = torch.empty(Tk, h, dtype=dtype, **d)
        self.y = torch.empty(T, h, dtype=dtype, **d)
        self.backward = backward
        if backward:
            self.dybuf = torch.empty(Tk, h, dtype=dtype, **d)
            self.d_topk_w = torch.empty(T, k, dtype=f32, **d)
            self.dxbuf = torch.empty(Tk, h, dtype=dtype, **d)
            self.dW1 = torch.empty(E, h, f, dtype=dtype, **d)
            self.dW3 = torch.empty(E, h, f, dtype=dtype, **d)
            self.dW2 = torch.empty(E, f, h, dtype=dtype, **d)
            self.d_logits = torch.empty(T, E, dtype=f32, **d)
            self.dWg = torch.empty(h, E, dtype=f32, **d)
            self.dx_router = torch.empty(T, h, dtype=f32, **d)
            self.dx = torch.empty(T, h, dtype=dtype, **d)
        self.ws = B.new_workspace(B.MOE_OP_ALL, T, h, E, k, f, dtype, device)


def forward(inp: dict, b: LayerBuffers):
    """Gate -> PFT build -> dispatch -> experts -> combine (dispatch folded into the expert
    GEMMs when b.fused, combine folded into the down projection when b.fold_combine).
    Returns b.y."""
    B.moe_route(inp["x"], inp["Wg"], inp.get("bias"), b.k, b.logits, b.probs, b.topk_idx, b.topk_w, b.ws,
                gate=b.gate, renorm=b.renorm)
    B.moe_pft_build(b.topk_idx, b.E, b.num_ids, b.offsets, b.token_ids, b.expert_ids, b.slot_of, b.ws)
    if not b.fused:
        B.moe_dispatch(inp["x"], b.token_ids, b.k, b.xbuf, b.ws)
    if b.fold_combine:
        B.moe_expert_ffn_fused(b.xbuf, inp["x"], b.token_ids, b.slot_of, b.topk_w, b.offsets, inp["W1"],
                               inp["W3"], inp["W2"], b.ybuf, b.h1, b.h3, b.a, b.y, b.ws)
        return b.y
    if b.fused:
        B.moe_expert_ffn_gather(inp["x"], b.token_ids, b.offsets, inp["W1"], inp["W3"], inp["W2"], b.ybuf,
                                b.h1, b.h3, b.a, b.ws)
    else:
        B.moe_expert_ffn(b.xbuf, b.offsets, inp["W1"], inp["W3"], inp["W2"], b.ybuf, b.h1, b.h3, b.a, b.ws)
    B.moe_combine(b.ybuf, b.slot_of, b.topk_w, b.y, b.ws)
    return b.y


def backward(inp: dict, dy: torch.Tensor, b: LayerBuffers):
    """Combine bwd -> experts bwd -> gate bwd -> dispatch bwd.  Returns b.dx."""
    B.moe_combine_bwd(dy, b.ybuf, b.slot_of, b.topk_w, b.dybuf, b.d_topk_w, b.ws)
    if b.fused:
        B.moe_expert_ffn_bwd_gather(b.dybuf, inp["x"], b.token_ids, b.h1, b.h3, b.a, b.offsets, inp["W1"],
                                    inp["W3"], inp["W2"], b.dxbuf, b.dW1, b.dW3, b.dW2, b.ws)
    else:
        B.moe_expert_ffn_bwd(b.dybuf, b.xbuf, b.h1, b.h3, b.a, b.offsets, inp["W1"], inp["W3"], inp["W2"],
                             b.dxbuf, b.dW1, b.dW3, b.dW2, b.ws)
    B.moe_route_bwd(inp["x"], inp["Wg"], b.probs, b.topk_idx, b.d_topk_w, b.d_logits, b.dWg,
                    b.dx_router, b.ws, gate=b.gate, renorm=b.renorm)
    B.moe_dispatch_bwd(b.dxbuf, b.slot_of, b.dx_router, b.k, b.dx, b.ws)
    return b.dx


def step(inp: dict, b: LayerBuffers):
    """One full layer step: forward, then (if the buffers have it) backward of inp['dy']."""
    forward(inp, b)
    if b.backward:
        backward(inp, inp["dy"], b)


def step_host(inp: dict, b: LayerBuffers, hx: torch.Tensor, hy: torch.Tensor,
              hdy: torch.Tensor | None = None, hdx: torch.Tensor | None = None):
    """One layer step with the step's tokens in pinned host memory.

    hx (and hdy) are copied into inp['x'] (and inp['dy']); y (and dx) come back into hy (and
    hdx).  The upload of dy overlaps the forward and the download of y overlaps the backward, on
    a second stream; the current stream waits for both, so the step is complete (host buffers
    included) once the current stream is.
    """
    cur = torch.cuda.current_stream()
    inp["x"].copy_(hx, non_blocking=True)
    if not b.backward:
        forward(inp, b)
        hy.copy_(b.y, non_blocking=True)
        return
    side = getattr(b, "copy_stream", None)
    if side is None:
        side = b.copy_stream = torch.cuda.Stream(device=inp["x"].device)
    side.wait_stream(cur)  # earlier readers of inp['dy'] and writers of hy are done
    with torch.cuda.stream(side):
        inp["dy"].copy_(hdy, non_blocking=True)
        dy_ready = torch.cuda.Event()
        dy_ready.record(side)
    forward(inp, b)
    side.wait_stream(cur)  # y is complete
    with torch.cuda.stream(side):
        hy.copy_(b.y, non_blocking=True)
    cur.wait_event(dy_ready)
    backward(inp, inp["dy"], b)
    hdx.copy_(b.dx, non_blocking=True)
    cur.wait_stream(side)


class CapturedStep:
    """A layer step captured once as a CUDA graph and then replayed.

    ``fn`` issues the step on the current stream (``lambda: step(inp, b)``, or ``step_host`` with
    its host buffers); it must use the same tensors on every call, as the graph keeps their
    addresses.  A replay runs the same kernels and copies in the same order on the caller's
    current stream, with one graph launch in place of one host call per kernel.  ``launches`` is
    the number of library kernels in the graph.
    """

    def __init__(self, fn, warmup: int = 1):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        n0 = B.lib().moe_kernel_launches()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            fn()
        self.launches = B.lib().moe_kernel_launches() - n0

    def replay(self):
        self.graph.replay()


class HostPipeline:
    """Layer steps over batches in pinned host memory, with the copies off the critical path.

    Two device slots hold the tokens (x, and dy for the backward) of consecutive steps: step
    i + 1's upload runs on a copy stream into the other slot while step i computes, and y and dx
    download on a second copy stream while later work runs.  ``submit`` returns at once.
    ``finish`` makes the current stream wait for every download, so the host buffers of every
    submitted step are complete once the current stream is.

    With ``graphs`` (the default) each slot's step is captured once as a CUDA graph that writes
    the slot's own y (and dx): a step waits for its upload and for the download of the outputs
    its slot held two steps back, and then replays as one launch.  Without it the calls are
    issued one by one on the current stream, y downloads while the backward runs, and a step
    waits for the previous step's y (and dx) to leave b.y (and b.dx) before overwriting them.

    ``inp`` holds the weights (and the router bias); its x and dy are slot 0.  The host buffers
    passed to ``submit`` must stay untouched until the current stream passes ``finish``.
    """

    def __init__(self, inp: dict, b: LayerBuffers, graphs: bool = True):
        self.b = b
        self.inp = inp
        dev = inp["x"].device
        bwd = b.backward
        self.x = [inp["x"], torch.zeros_like(inp["x"])]
        self.dy = [inp["dy"], torch.zeros_like(inp["dy"])] if bwd else [None, None]
        self.up = torch.cuda.Stream(device=dev)
        self.down = torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        self.slot_free = [ev(), ev()]   # the compute that last read a slot is done
        self.ready = [ev(), ev()]       # a slot's upload is done
        self.out_done, self.out_free = [ev(), ev()], [ev(), ev()]  # graphs: a slot's outputs
        self.y_done, self.y_free = ev(), ev()
        self.dx_done, self.dx_free = ev(), ev()
        self.graphs = None
        if graphs:
            self.y = [b.y, torch.zeros_like(b.y)]
            self.dx = [b.dx, torch.zeros_like(b.dx)] if bwd else [None, None]
            self.graphs = []
            for sl in range(2):
                b.y = self.y[sl]
                if bwd:
                    b.dx = self.dx[sl]
                inp_s = dict(inp, x=self.x[sl], dy=self.dy[sl])
                self.graphs.append(CapturedStep(lambda inp_s=inp_s: step(inp_s, b)))
            b.y = self.y[0]
            if bwd:
                b.dx = self.dx[0]
        cur = torch.cuda.current_stream()
        for e in self.slot_free + self.out_free + [self.y_free, self.dx_free]:
            e.record(cur)
        self.i = 0

    def submit(self, hx: torch.Tensor, hy: torch.Tensor, hdy: torch.Tensor | None = None,
               hdx: torch.Tensor | None = None):
        b, s = self.b, self.i % 2
        cur = torch.cuda.current_stream()
        self.up.wait_event(self.slot_free[s])
        with torch.cuda.stream(self.up):
            self.x[s].copy_(hx, non_blocking=True)
            if b.backward:
                self.dy[s].copy_(hdy, non_blocking=True)
            self.ready[s].record(self.up)
        cur.wait_event(self.ready[s])
        if self.graphs is not None:
            cur.wait_event(self.out_free[s])  # this slot's outputs of two steps back have left
            self.graphs[s].replay()
            self.out_done[s].record(cur)
            self.slot_free[s].record(cur)
            self.down.wait_event(self.out_done[s])
            with torch.cuda.stream(self.down):
                hy.copy_(self.y[s], non_blocking=True)
                if b.backward:
                    hdx.copy_(self.dx[s], non_blocking=True)
                self.out_free[s].record(self.down)
            self.i += 1
            return
        inp = dict(self.inp, x=self.x[s], dy=self.dy[s])
        cur.wait_event(self.y_free)  # the previous step's y has left b.y
        forward(inp, b)
        self.y_done.record(cur)
        self.down.wait_event(self.y_done)
        with torch.cuda.stream(self.down):
            hy.copy_(b.y, non_blocking=True)
            self.y_free.record(self.down)
        if b.backward:
            cur.wait_event(self.dx_free)  # the previous step's dx has left b.dx
            backward(inp, inp["dy"], b)
            self.dx_done.record(cur)
            self.down.wait_event(self.dx_done)
            with torch.cuda.stream(self.down):
                hdx.copy_(b.dx, non_blocking=True)
                self.dx_free.record(self.down)
        self.slot_free[s].record(cur)
        self.i += 1

    def finish(self):
        torch.cuda.current_stream().wait_stream(self.down)


class GShardBuffers:
    """Device buffers of the capacity-buffer (GShard-style) forward at capacity C: the masks
    [T,E,C], the padded expert buffers [E*C, ...] and the padded segment offsets e*C.  The gate's
    probabilities and top-k come from the same moe_route as the padding-free layer."""

    def __init__(self, T: int, h: int, E: int, k: int, f: int, C: int, dtype: torch.dtype, device="cuda"):
        self.T, self.h, self.E, self.k, self.f, self.C, self.dtype = T, h, E, k, f, C, dtype
        f32, i32 = torch.float32, torch.int32
        d = dict(device=device)
        self.logits = torch.empty(T, E, dtype=f32, **d)
        self.probs = torch.empty(T, E, dtype=f32, **d)
        self.topk_idx = torch.empty(T, k, dtype=i32, **d)
        self.topk_w = torch.empty(T, k, dtype=f32, **d)
        self.dispatch_mask = torch.empty(T, E, C, dtype=dtype, **d)
        self.combine_w = torch.empty(T, E, C, dtype=f32, **d)
        self.loads = torch.empty(E, dtype=i32, **d)
        self.offsets = (torch.arange(E + 1, dtype=i32, **d) * C).contiguous()
        self.xe = torch.empty(E, C, h, dtype=dtype, **d)
        self.h1 = torch.empty(E * C, f, dtype=dtype, **d)
        self.h3 = torch.empty(E * C, f, dtype=dtype, **d)
        self.a = torch.empty(E * C, f, dtype=dtype, **d)
        self.ye = torch.empty(E, C, h, dtype=dtype, **d)
        self.y = torch.empty(T, h, dtype=dtype, **d)
        # the experts run on E*C padded rows, more than the T*k of the padding-free layer
        nbytes = max(B.workspace_size(B.MOE_OP_ALL, T, h, E, k, f, dtype),
                     B.workspace_size(B.MOE_OP_EXPERT_FFN, E * C, h, E, 1, f, dtype))
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        self.ws_gshard = B.new_workspace(B.MOE_OP_GSHARD, T, h, E, k, f, dtype, device)


def gshard_forward(inp: dict, g: GShardBuffers, stages=None):
    """Gate -> masks -> padded dispatch -> experts on every padded row -> combine.  With
    ``stages`` (a list of callables) the four stage calls are returned instead of run."""
    calls = [
        lambda: (B.moe_route(inp["x"], inp["Wg"], inp.get("bias"), g.k, g.logits, g.probs, g.topk_idx, g.topk_w,
                             g.ws),
                 B.moe_gshard_gate(g.topk_idx, g.topk_w, g.E, g.C, g.dispatch_mask, g.combine_w, g.loads,
                                   g.ws_gshard)),
        lambda: B.moe_gshard_dispatch(inp["x"], g.dispatch_mask, g.xe, g.ws_gshard),
        lambda: B.moe_expert_ffn(g.xe.view(g.E * g.C, g.h), g.offsets, inp["W1"], inp["W3"], inp["W2"],
                                 g.ye.view(g.E * g.C, g.h), g.h1, g.h3, g.a, g.ws),
        lambda: B.moe_gshard_combine(g.combine_w, g.ye, g.y, g.ws_gshard),
    ]
    if stages is not None:
        return calls
    for c in calls:
        c()
    return g.y
