"""Helpers shared by the GPU parity tests: layout mapping between the library's padded
workspace arrays and the oracle's natural [T, H, 128] arrays, error metrics, and oracle runs.
Nothing here computes attention."""
from __future__ import annotations

import math

import numpy as np
import torch

SCALE = 1.0 / math.sqrt(128)


def bits(t: torch.Tensor) -> np.ndarray:
    """BF16 CPU tensor (any strides, unit channel stride) -> uint16 numpy view, same strides."""
    t = t.cpu() if t.is_cuda else t
    return t.view(torch.int16).numpy().view(np.uint16)


def padded_rows(cu, row_offsets):
    """Padded-axis row of every token (length T) and the set of padding rows."""
    rows = []
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        rows.extend(range(row_offsets[s], row_offsets[s] + (b - a)))
    rows = np.asarray(rows, np.int64)
    tpad = row_offsets[-1]
    pad = np.setdiff1d(np.arange(tpad), rows)
    return rows, pad


def rel_rms(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def out_rows(out: torch.Tensor, rows) -> np.ndarray:
    """Gather (token, head) rows of a BF16 [T, H, 128] tensor -> float64 [n, 128]."""
    o = out.float().cpu().numpy()
    r = np.asarray(rows, np.int64).reshape(-1, 2)
    return o[r[:, 0], r[:, 1]].astype(np.float64)


def all_rows(cu, heads):
    return [(t, h) for t in range(cu[-1]) for h in range(heads)]


def bf16_of(out64: np.ndarray) -> np.ndarray:
    return torch.from_numpy(out64.astype(np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)
