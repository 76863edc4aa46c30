"""Shared test helpers: tensor conversion and comparison metrics.  No layer arithmetic."""
from __future__ import annotations

import numpy as np
import torch


def to_np(t):
    """torch tensor (any device) -> numpy; bf16 becomes uint16 bit patterns."""
    if isinstance(t, np.ndarray):
        return t
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float16:
        return t.numpy()
    return t.numpy()


def np_inputs(weights: dict, step: dict):
    w = {k: to_np(v) for k, v in weights.items()}
    s = {k: (to_np(v) if isinstance(v, torch.Tensor) else v) for k, v in step.items()}
    return w, s


def bf16_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rel_l2(a, b) -> float:
    a, b = np.asarray(a, np.float64).ravel(), np.asarray(b, np.float64).ravel()
    d = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (d if d > 0 else 1.0))


def cosine(a, b) -> float:
    a, b = np.asarray(a, np.float64).ravel(), np.asarray(b, np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))
