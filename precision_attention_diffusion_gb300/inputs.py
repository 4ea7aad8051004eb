"""Seeded synthetic inputs shaped like the MiniMax-H3 attention workloads.

This module holds no arithmetic of the attention method: it only draws random BF16 tensors and
names the segment layouts, so that the CUDA path, the oracle checks and the benchmark all see the
same bytes. Recipe: ``torch.Generator().manual_seed(seed)`` on the CPU, ``randn`` in FP32, then a
cast to BF16 (i.i.d. N(0, 1)), as in the pages' Gaussian synthetic Q/K/V (SGLang PR #40175,
Accuracy Tests and Speed Tests).
"""
from __future__ import annotations

import torch

HEAD_DIM = 128

# Named workloads: (segment lengths as cu_seqlens, heads).
WORKLOADS = {
    # one segment S=256, H=2 (the oracle finishes it in seconds)
    "fp8_s256_h2": dict(cu=[0, 256], heads=2),
    # one segment S=4096, H=56
    "fp8_s4096_h56": dict(cu=[0, 4096], heads=56),
    # MiniMax-H3 shapes, single segments, H=56
    "fp8_s20440_h56": dict(cu=[0, 20440], heads=56),
    "fp8_s30272_h56": dict(cu=[0, 30272], heads=56),
    # packed varlen with empty, sub-tile and trailing-padding segments
    "fp8_varlen_32768_h56": dict(cu=[0, 0, 17, 4113, 4113, 31800, 32768], heads=56),
    # NVFP4 at the H3 shape, and a small case of the same kernel (profiling)
    "nvfp4_s30272_h56": dict(cu=[0, 30272], heads=56),
    "nvfp4_s4096_h56": dict(cu=[0, 4096], heads=56),
}


def gaussian_bf16(shape, seed: int, std: float = 1.0) -> torch.Tensor:
    g = torch.Generator().manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16)


def qkv_separate(tokens: int, heads: int, seed: int = 0):
    """Three contiguous BF16 [T, H, 128] tensors, N(0,1), drawn from seeds seed, seed+1, seed+2."""
    shape = (tokens, heads, HEAD_DIM)
    return tuple(gaussian_bf16(shape, seed + i) for i in range(3))


def qkv_fused(tokens: int, heads: int, seed: int = 0):
    """One BF16 [T, 3, H, 128] buffer (N(0,1)) and its three strided [T, H, 128] views (token
    stride 3*H*128, head stride 128), the layout of a fused QKV projection."""
    buf = gaussian_bf16((tokens, 3, heads, HEAD_DIM), seed)
    return buf, buf[:, 0], buf[:, 1], buf[:, 2]


def k_channel_offset(heads: int, seed: int, std: float = 2.0) -> torch.Tensor:
    """Per-(head, channel) offset, N(0, std^2), constant over tokens (exercises K centring)."""
    g = torch.Generator().manual_seed(int(seed) + 1000)
    return (torch.randn(heads, HEAD_DIM, generator=g) * std).to(torch.float32)


def sample_rows(cu, heads: int, n_heads: int, n_rows: int, seed: int):
    """A seeded sample of (token, head) query rows: n_heads heads x n_rows tokens drawn from the
    non-empty segments (uniformly over tokens)."""
    g = torch.Generator().manual_seed(int(seed))
    tokens = int(cu[-1])
    hs = torch.randperm(heads, generator=g)[:n_heads].tolist()
    if tokens == 0:
        return []
    ts = torch.randint(0, tokens, (n_rows,), generator=g).tolist()
    return [(t, h) for h in hs for t in sorted(ts)]
