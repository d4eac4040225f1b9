"""Helpers shared by the GPU parity tests (comparison metrics, routing ambiguity)."""

from __future__ import annotations

import numpy as np
import torch

# Acceptance: bit-exact for indices and copies; rel-L2 on floating outputs and gradients.
TOL = {"f32": 1e-5, "bf16": 1e-2}


def rel_l2(got, want) -> float:
    g = np.asarray(got, np.float64)
    w = np.asarray(want, np.float64)
    den = np.linalg.norm(w.ravel())
    num = np.linalg.norm((g - w).ravel())
    if den == 0.0:
        return float(num)
    return float(num / den)


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def npi(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.int64)


def dtype_name(dt: torch.dtype) -> str:
    return "bf16" if dt == torch.bfloat16 else "f32"


def unambiguous_tokens(exact_logits: np.ndarray, k: int, delta: float) -> np.ndarray:
    """Tokens whose top-(k+1) sorted logits are separated by more than ``delta``.

    For such a token every fp32 evaluation of the logits within ``delta``/2 of the exact
    values selects the same experts in the same order, so the selection is unique; for the
    others several selections are correct within rounding.
    """
    s = -np.sort(-exact_logits, axis=1)
    kk = min(k + 1, exact_logits.shape[1])
    gaps = s[:, : kk - 1] - s[:, 1:kk]
    return (gaps > delta).all(axis=1)


def check_valid_topk(gpu_idx: np.ndarray, exact_logits: np.ndarray, k: int, delta: float):
    """Any selection is valid if it picks k distinct experts whose logits are each within
    ``delta`` of the exact k largest, in order within ``delta``."""
    T, E = exact_logits.shape
    s = -np.sort(-exact_logits, axis=1)
    for t in range(T):
        row = gpu_idx[t]
        assert len(set(row.tolist())) == k and row.min() >= 0 and row.max() < E
        vals = exact_logits[t, row]
        assert (np.abs(vals - s[t, :k]) <= delta).all(), (t, row, vals, s[t, : k + 1])
