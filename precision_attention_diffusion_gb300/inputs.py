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
    # block-sparse FP8 at the H3 shape: 64-row query blocks x 64-key blocks, about a quarter of
    # the key blocks listed per query block (the pages' sparsity 0.75), and a small case
    "sparse_fp8_s30272_h56": dict(cu=[0, 30272], heads=56, density=0.25),
    "sparse_fp8_s4096_h56": dict(cu=[0, 4096], heads=56, density=0.25),
}

SPARSE_BLOCK = 64  # rows of a query block and keys of a key block of the block-sparse lists


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


def block_sparse_lists(cu, heads: int, density: float, seed: int, dense_every: int = 0,
                       empty_every: int = 0):
    """A seeded block-sparse pattern in the form the block-sparse forward takes.

    Query blocks are the 64-row blocks of every segment (counted from the segment's first token,
    the last one partial), numbered g = 0 .. G-1 over the segments in order; key blocks are the
    64-key blocks of the same segment. For every (head h, query block g) the list holds distinct
    key-block indices in ascending order: its length is density x (key blocks of the segment) x
    u, u uniform in [0.5, 1.5), rounded, at least 1; its blocks are drawn uniformly without
    replacement. Every `dense_every`-th list (counted over h G + g) names every key block and
    every `empty_every`-th none (mixed sparse/dense rows and empty rows). Returns (offsets int32
    [H G + 1], indices int32 [nnz]); the list of (h, g) is indices[offsets[h G + g] :
    offsets[h G + g + 1]]."""
    import numpy as np

    rng = np.random.default_rng(int(seed))
    lens = [int(b) - int(a) for a, b in zip(cu[:-1], cu[1:])]
    nblk = [(L + SPARSE_BLOCK - 1) // SPARSE_BLOCK for L in lens]
    G = sum(nblk)
    lists = [[None] * G for _ in range(heads)]
    g0 = 0
    for n in nblk:  # a segment of n blocks: n query blocks, each choosing among n key blocks
        if n == 0:
            continue
        k = np.clip(np.rint(density * n * (0.5 + rng.random((heads, n)))), 1, n).astype(np.int64)
        ranks = np.argsort(np.argsort(rng.random((heads, n, n)), axis=2), axis=2)
        for h in range(heads):
            for i in range(n):
                j = h * G + g0 + i
                if empty_every and j % empty_every == empty_every - 1:
                    lists[h][g0 + i] = np.zeros(0, np.int64)
                elif dense_every and j % dense_every == dense_every - 1:
                    lists[h][g0 + i] = np.arange(n)
                else:
                    lists[h][g0 + i] = np.nonzero(ranks[h, i] < k[h, i])[0]
        g0 += n
    flat = [lists[h][g] for h in range(heads) for g in range(G)]
    offsets = np.zeros(heads * G + 1, np.int64)
    offsets[1:] = np.cumsum([len(x) for x in flat])
    idx = np.concatenate(flat) if flat else np.zeros(0, np.int64)
    return offsets.astype(np.int32), idx.astype(np.int32)
