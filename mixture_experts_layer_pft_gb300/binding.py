"""Python binding of the C ABI in include/moe_pft.h (ctypes; argument marshalling only).

Every function takes torch CUDA tensors that the caller allocated, passes their device
pointers and the current CUDA stream to the function of the same name in libmoe_pft.so, and
raises ``MoEError`` on a non-zero status.  There is no CPU path: without the built library or
a CUDA device the first call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_pft.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_DEVICE = (
    0, -1, -2, -3, -4, -5)
MOE_F32, MOE_BF16 = 0, 1
MOE_STATUS_BAD_INDEX, MOE_STATUS_TIMEOUT = 1, 2
MOE_ROUTE_FROM_LOGITS, MOE_ROUTE_SIGMOID, MOE_ROUTE_RENORM = 1, 2, 4
(MOE_OP_ROUTE, MOE_OP_ROUTE_BWD, MOE_OP_PFT_BUILD, MOE_OP_DISPATCH, MOE_OP_DISPATCH_BWD,
 MOE_OP_EXPERT_FFN, MOE_OP_EXPERT_FFN_BWD, MOE_OP_COMBINE, MOE_OP_COMBINE_BWD, MOE_OP_ALL, MOE_OP_GSHARD) = range(11)

# C signatures: (name, restype, argtypes).  P = pointer, I = int, Z = size_t.
_P, _I, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "moe_abi_version": (_I, []),
    "moe_kernel_launches": (ctypes.c_uint64, []),
    "moe_profile_events": (_I, [ctypes.POINTER(ctypes.c_void_p), _I]),
    "moe_profile_count": (ctypes.c_uint64, []),
    "moe_debug_withhold_stage": (_I, [_I, ctypes.c_ulonglong]),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I, _I]),
    "moe_status_reset": (_I, [_P, _P]),
    "moe_check_status": (_I, [_P, _P, ctypes.POINTER(ctypes.c_int)]),
    "moe_route": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_route_bwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "moe_pft_build": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_pft_build_noalloc": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "moe_dispatch": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_dispatch_bwd": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_expert_ffn": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_expert_ffn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                _P, _P, _P, _P, _P, _Z, _P]),
    "moe_expert_ffn_gather": (_I, [_P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                   _P, _Z, _P]),
    "moe_expert_ffn_bwd_gather": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                       _P, _P, _P, _P, _P, _Z, _P]),
    "moe_expert_ffn_gather_supported": (_I, [_I, _I, _I]),
    "moe_expert_ffn_fused": (_I, [_P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                  _P, _P, _Z, _P]),
    "moe_combine": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_gshard_gate": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "moe_gshard_dispatch": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_gshard_combine": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_combine_bwd": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _Z, _P]),
}


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed with status {code}: {msg}")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoe_pft.so once; raise if it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build() first")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MOE_F32
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _p(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _call(name, *args):
    rc = getattr(lib(), name)(*args)
    if rc != MOE_OK:
        raise MoEError(name, rc, (lib().moe_last_error() or b"").decode())


def workspace_size(op: int, T: int, h: int, E: int, k: int, f: int, dtype: torch.dtype) -> int:
    code = MOE_BF16 if dtype == torch.bfloat16 else MOE_F32
    return int(lib().moe_workspace_size(op, T, h, E, k, f, code))


def new_workspace(op: int, T: int, h: int, E: int, k: int, f: int, dtype: torch.dtype, device="cuda"):
    """A zeroed uint8 workspace of moe_workspace_size bytes (status word cleared)."""
    return torch.zeros(workspace_size(op, T, h, E, k, f, dtype), dtype=torch.uint8, device=device)


class KernelTimer:
    """Per-kernel CUDA-event timing through moe_profile_events: the library records one event
    after each of its launches, on the launching stream."""

    def __init__(self, capacity: int):
        stream = torch.cuda.current_stream()
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        for e in self.events:  # materialise the underlying cudaEvent_t
            e.record(stream)
        self._handles = (ctypes.c_void_p * capacity)(*[e.cuda_event for e in self.events])
        self.capacity = capacity

    def __enter__(self):
        rc = lib().moe_profile_events(self._handles, self.capacity)
        if rc != MOE_OK:
            raise MoEError("moe_profile_events", rc, (lib().moe_last_error() or b"").decode())
        return self

    def count(self) -> int:
        return int(lib().moe_profile_count())

    def event(self, n: int):
        return self.events[n % self.capacity]

    def __exit__(self, *exc):
        lib().moe_profile_events(None, 0)
        return False


def moe_status_reset(ws):
    _call("moe_status_reset", _p(ws), _stream())


def moe_check_status(ws) -> int:
    """Synchronise the current stream and return the device status word (0 = clean)."""
    code = ctypes.c_int(0)
    rc = lib().moe_check_status(_p(ws), _stream(), ctypes.byref(code))
    if rc not in (MOE_OK, MOE_ERR_DEVICE):
        raise MoEError("moe_check_status", rc, (lib().moe_last_error() or b"").decode())
    return code.value


def moe_debug_withhold_stage(launches: int, wait_limit_ns: int = 0):
    """Test hook: the next ``launches`` tensor-core kernel launches withhold their first pipeline
    stage, so their bounded waits run out (after ``wait_limit_ns``; 0 = the default limit) and
    they report MOE_STATUS_TIMEOUT.  ``launches=0`` cancels."""
    rc = lib().moe_debug_withhold_stage(int(launches), int(wait_limit_ns))
    if rc != MOE_OK:
        raise MoEError("moe_debug_withhold_stage", rc, (lib().moe_last_error() or b"").decode())


def gate_flags(gate: str = "softmax", renorm: bool = False) -> int:
    if gate not in ("softmax", "sigmoid"):
        raise ValueError(f"unknown gate {gate!r}")
    return (MOE_ROUTE_SIGMOID if gate == "sigmoid" else 0) | (MOE_ROUTE_RENORM if renorm else 0)


def moe_route(x, Wg, bias, k, logits, probs, topk_idx, topk_w, ws, from_logits=False, dtype=None,
              gate="softmax", renorm=False):
    T, E = logits.shape
    h = x.shape[1] if x is not None else 0
    dt = _dtype_code(x) if x is not None else (MOE_BF16 if dtype == torch.bfloat16 else MOE_F32)
    flags = gate_flags(gate, renorm) | (MOE_ROUTE_FROM_LOGITS if from_logits else 0)
    _call("moe_route", _p(x), _p(Wg), _p(bias), T, h, E, k, dt, flags, _p(logits), _p(probs),
          _p(topk_idx), _p(topk_w), _p(ws), ws.numel(), _stream())


def moe_route_bwd(x, Wg, probs, topk_idx, d_topk_w, d_logits, dWg, dx_router, ws, gate="softmax",
                  renorm=False):
    T, h = x.shape
    E = Wg.shape[1]
    k = topk_idx.shape[1]
    _call("moe_route_bwd", _p(x), _p(Wg), _p(probs), _p(topk_idx), _p(d_topk_w), T, h, E, k,
          _dtype_code(x), gate_flags(gate, renorm), _p(d_logits), _p(dWg), _p(dx_router), _p(ws),
          ws.numel(), _stream())


def moe_pft_build(topk_idx, E, num_ids, offsets, token_ids, expert_ids, slot_of, ws):
    T, k = topk_idx.shape
    _call("moe_pft_build", _p(topk_idx), T, E, k, _p(num_ids), _p(offsets), _p(token_ids),
          _p(expert_ids), _p(slot_of), _p(ws), ws.numel(), _stream())


def moe_pft_build_noalloc(topk_idx, E, num_ids, offsets, token_ids, expert_ids, slot_of):
    """moe_pft_build without a workspace: its scratch is the library's static device array,
    for callers that cannot allocate.  Calls that overlap on the GPU race."""
    T, k = topk_idx.shape
    _call("moe_pft_build_noalloc", _p(topk_idx), T, E, k, _p(num_ids), _p(offsets), _p(token_ids),
          _p(expert_ids), _p(slot_of), _stream())


def moe_dispatch(x, token_ids, k, xbuf, ws):
    T, h = x.shape
    _call("moe_dispatch", _p(x), _p(token_ids), T, k, h, _dtype_code(x), _p(xbuf), _p(ws),
          ws.numel(), _stream())


def moe_dispatch_bwd(dxbuf, slot_of, dx_add, k, dx, ws):
    T, h = dx.shape
    _call("moe_dispatch_bwd", _p(dxbuf), _p(slot_of), _p(dx_add), T, k, h, _dtype_code(dx), _p(dx),
          _p(ws), ws.numel(), _stream())


def moe_expert_ffn(xbuf, offsets, W1, W3, W2, ybuf, h1, h3, a, ws):
    Tk, h = xbuf.shape
    E, _, f = W1.shape
    _call("moe_expert_ffn", _p(xbuf), _p(offsets), _p(W1), _p(W3), _p(W2), Tk, E, h, f,
          _dtype_code(xbuf), _p(ybuf), _p(h1), _p(h3), _p(a), _p(ws), ws.numel(), _stream())


def moe_expert_ffn_bwd(dybuf, xbuf, h1, h3, a, offsets, W1, W3, W2, dxbuf, dW1, dW3, dW2, ws):
    Tk, h = xbuf.shape
    E, _, f = W1.shape
    _call("moe_expert_ffn_bwd", _p(dybuf), _p(xbuf), _p(h1), _p(h3), _p(a), _p(offsets), _p(W1),
          _p(W3), _p(W2), Tk, E, h, f, _dtype_code(xbuf), _p(dxbuf), _p(dW1), _p(dW3), _p(dW2),
          _p(ws), ws.numel(), _stream())


def moe_expert_ffn_gather(x, token_ids, offsets, W1, W3, W2, ybuf, h1, h3, a, ws):
    T, h = x.shape
    Tk = token_ids.shape[0]
    E, _, f = W1.shape
    _call("moe_expert_ffn_gather", _p(x), _p(token_ids), T, _p(offsets), _p(W1), _p(W3), _p(W2), Tk, E,
          h, f, _dtype_code(x), _p(ybuf), _p(h1), _p(h3), _p(a), _p(ws), ws.numel(), _stream())


def moe_expert_ffn_bwd_gather(dybuf, x, token_ids, h1, h3, a, offsets, W1, W3, W2, dxbuf, dW1, dW3, dW2,
                              ws):
    T, h = x.shape
    Tk = token_ids.shape[0]
    E, _, f = W1.shape
    _call("moe_expert_ffn_bwd_gather", _p(dybuf), _p(x), _p(token_ids), T, _p(h1), _p(h3), _p(a),
          _p(offsets), _p(W1), _p(W3), _p(W2), Tk, E, h, f, _dtype_code(x), _p(dxbuf), _p(dW1), _p(dW3),
          _p(dW2), _p(ws), ws.numel(), _stream())


def moe_expert_ffn_gather_supported(h: int, f: int, dtype: torch.dtype) -> bool:
    code = MOE_BF16 if dtype == torch.bfloat16 else MOE_F32
    return bool(lib().moe_expert_ffn_gather_supported(h, f, code))


def moe_expert_ffn_fused(xbuf, x, token_ids, slot_of, topk_w, offsets, W1, W3, W2, ybuf, h1, h3, a, y, ws):
    """Expert FFN with the dispatch (xbuf None: rows gathered from x) and/or the combine (y not
    None) folded into its GEMMs."""
    T, k = topk_w.shape
    Tk = token_ids.shape[0]
    E, h, f = W1.shape
    dt = (xbuf if xbuf is not None else x).dtype
    code = MOE_BF16 if dt == torch.bfloat16 else MOE_F32
    _call("moe_expert_ffn_fused", _p(xbuf), _p(x), _p(token_ids), T, k, _p(slot_of), _p(topk_w), _p(offsets),
          _p(W1), _p(W3), _p(W2), Tk, E, h, f, code, _p(ybuf), _p(h1), _p(h3), _p(a), _p(y), _p(ws), ws.numel(),
          _stream())


def moe_combine(ybuf, slot_of, topk_w, y, ws):
    T, h = y.shape
    k = topk_w.shape[1]
    _call("moe_combine", _p(ybuf), _p(slot_of), _p(topk_w), T, k, h, _dtype_code(y), _p(y), _p(ws),
          ws.numel(), _stream())


def moe_combine_bwd(dy, ybuf, slot_of, topk_w, dybuf, d_topk_w, ws):
    T, h = dy.shape
    k = topk_w.shape[1]
    _call("moe_combine_bwd", _p(dy), _p(ybuf), _p(slot_of), _p(topk_w), T, k, h, _dtype_code(dy),
          _p(dybuf), _p(d_topk_w), _p(ws), ws.numel(), _stream())


def moe_gshard_gate(topk_idx, topk_w, E, C, dispatch_mask, combine_w, loads, ws):
    """Capacity-buffer gate: dispatch_mask [T,E,C] (activation dtype) and combine_w [T,E,C] fp32."""
    T, k = topk_idx.shape
    _call("moe_gshard_gate", _p(topk_idx), _p(topk_w), T, E, k, C, _dtype_code(dispatch_mask),
          _p(dispatch_mask), _p(combine_w), _p(loads), _p(ws), ws.numel(), _stream())


def moe_gshard_dispatch(x, dispatch_mask, xe, ws):
    """xe [E,C,h] = the contraction of dispatch_mask [T,E,C] with x [T,h] over the tokens."""
    T, E, C = dispatch_mask.shape
    h = x.shape[1]
    _call("moe_gshard_dispatch", _p(x), _p(dispatch_mask), T, E, C, h, _dtype_code(x), _p(xe), _p(ws),
          ws.numel(), _stream())


def moe_gshard_combine(combine_w, ye, y, ws):
    """y [T,h] = the contraction of combine_w [T,E,C] with ye [E,C,h] over (e, c)."""
    T, E, C = combine_w.shape
    h = ye.shape[2]
    _call("moe_gshard_combine", _p(combine_w), _p(ye), T, E, C, h, _dtype_code(ye), _p(y), _p(ws), ws.numel(),
          _stream())
