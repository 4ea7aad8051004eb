"""Pins for the oracle's block-sparse attention (reading r16; SGLang PR #40116 "Add SM120 Sage
compute for SubBlock sparse attention", Modifications: 64-row query blocks x 64-key blocks,
partial blocks, variable per-row block counts, mixed sparse and dense rows; Accuracy Tests:
ragged lengths, variable block counts, empty rows against an FP32 reference). CPU only.

What pins what (nothing here retypes the oracle's own loops):
  * full lists reduce to the dense oracle, bit for bit (C1 and C2 with 64-key tiles), which is
    pinned by its own tests;
  * C1 under lists against a brute force that builds the dense key mask of every row from the
    lists and applies scipy's softmax over the allowed keys;
  * rows with an empty list give 0 (and LSE -inf); keys of blocks that are not listed do not
    change the output, keys of a listed block do (negative control);
  * C2 under lists: constant V returns deq(V) exactly; empty rows give 0 there as well;
  * lists that break the contract (outside the segment, unsorted, repeated) are rejected.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from precision_attention_diffusion_gb300 import inputs

SCALE = 1.0 / math.sqrt(128)
B = 64


def bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).numpy().view(np.uint16)


def qkv(cu, H, seed):
    return inputs.qkv_separate(cu[-1], H, seed)


def full_lists(cu, H):
    lens = [b - a for a, b in zip(cu[:-1], cu[1:])]
    per_g = [n for L in lens for n in [(L + B - 1) // B] * ((L + B - 1) // B)]
    flat = [np.arange(n) for _ in range(H) for n in per_g]
    off = np.zeros(len(flat) + 1, np.int32)
    off[1:] = np.cumsum([len(x) for x in flat])
    return off, (np.concatenate(flat) if flat else np.zeros(0)).astype(np.int32)


def list_of(cu, off, idx, H, t, h):
    """(segment start, segment end, the list) of query row (t, h)."""
    lens = [b - a for a, b in zip(cu[:-1], cu[1:])]
    G = sum((L + B - 1) // B for L in lens)
    g0 = 0
    for s, L in enumerate(lens):
        a = cu[s]
        if a <= t < a + L:
            g = g0 + (t - a) // B
            return a, a + L, idx[off[h * G + g]:off[h * G + g + 1]]
        g0 += (L + B - 1) // B
    raise AssertionError("token outside every segment")


CU = [0, 100, 100, 300, 301]  # partial blocks, an empty segment, a one-token segment
H = 2


def test_full_lists_equal_dense_exact_and_fp8():
    q, k, v = qkv(CU, H, 7)
    rows = [(t, h) for t in range(CU[-1]) for h in range(H)]
    off, idx = full_lists(CU, H)
    dense = oracle.attn_exact(bits(q), bits(k), bits(v), CU, rows, SCALE)
    sparse = oracle.attn_exact_sparse(bits(q), bits(k), bits(v), CU, off, idx, rows, SCALE)
    assert np.array_equal(dense, sparse)
    cq, dq = oracle.fp8_quantize(bits(q))
    ck, dk = oracle.fp8_quantize(bits(k))
    cv, dv = oracle.fp8_quantize(bits(v))
    for tau in (0.0, 8.0):
        d64, d16, dl = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, CU, rows, SCALE, n_kv=64, tau=tau,
                                       lse=True)
        s64, s16, sl = oracle.attn_fp8_sparse(cq, ck, cv, dq, dk, dv, CU, off, idx, rows, SCALE,
                                              tau=tau, lse=True)
        assert np.array_equal(d64, s64) and np.array_equal(d16, s16) and np.array_equal(dl, sl)


def test_exact_against_masked_softmax_brute_force():
    q, k, v = qkv(CU, H, 11)
    off, idx = inputs.block_sparse_lists(CU, H, density=0.5, seed=3, dense_every=4,
                                         empty_every=5)
    rows = [(t, h) for t in range(CU[-1]) for h in range(H)]
    got, lse = oracle.attn_exact_sparse(bits(q), bits(k), bits(v), CU, off, idx, rows, SCALE,
                                        lse=True)
    qf, kf, vf = (x.float().numpy().astype(np.float64) for x in (q, k, v))
    nonempty = 0
    for r, (t, h) in enumerate(rows):
        a, b, lst = list_of(CU, off, idx, H, t, h)
        allowed = np.zeros(CU[-1], bool)
        for kb in lst:
            allowed[a + B * kb:min(b, a + B * (kb + 1))] = True
        if not allowed.any():
            assert np.all(got[r] == 0.0) and lse[r] == -np.inf
            continue
        nonempty += 1
        s = kf[allowed, h] @ qf[t, h] * SCALE
        p = scipy.special.softmax(s)
        want = p @ vf[allowed, h]
        np.testing.assert_allclose(got[r], want, rtol=1e-11, atol=1e-13)
        assert abs(lse[r] - scipy.special.logsumexp(s)) < 1e-11
    assert 0 < nonempty < len(rows)  # the pattern has both empty and non-empty rows


def test_unlisted_keys_do_not_matter_listed_keys_do():
    cu = [0, 256]
    q, k, v = qkv(cu, 1, 5)
    # query block 1 lists key blocks 0 and 2 only; the others list everything
    lists = [np.arange(4), np.array([0, 2]), np.arange(4), np.arange(4)]
    off = np.zeros(5, np.int32)
    off[1:] = np.cumsum([len(x) for x in lists])
    idx = np.concatenate(lists).astype(np.int32)
    rows = [(t, 0) for t in range(64, 128)]
    base = oracle.attn_exact_sparse(bits(q), bits(k), bits(v), cu, off, idx, rows, SCALE)
    k2, v2 = k.clone(), v.clone()
    k2[64:128] = -k2[64:128]
    v2[192:256] = 3 * v2[192:256]
    same = oracle.attn_exact_sparse(bits(q), bits(k2), bits(v2), cu, off, idx, rows, SCALE)
    assert np.array_equal(base, same)
    v3 = v.clone()
    v3[128:192] = 3 * v3[128:192]  # key block 2 is listed
    diff = oracle.attn_exact_sparse(bits(q), bits(k), bits(v3), cu, off, idx, rows, SCALE)
    assert np.max(np.abs(diff - base)) > 0.05


def test_fp8_constant_v_and_empty_rows():
    q, k, _ = qkv(CU, H, 13)
    v = torch.full((CU[-1], H, 128), 0.8125).to(torch.bfloat16)
    cq, dq = oracle.fp8_quantize(bits(q))
    ck, dk = oracle.fp8_quantize(bits(k))
    cv, dv = oracle.fp8_quantize(bits(v))
    off, idx = inputs.block_sparse_lists(CU, H, density=0.3, seed=4, empty_every=3)
    rows = [(t, h) for t in range(CU[-1]) for h in range(H)]
    o64, o16, lse = oracle.attn_fp8_sparse(cq, ck, cv, dq, dk, dv, CU, off, idx, rows, SCALE,
                                           tau=8.0, lse=True)
    want = oracle.e4m3_decode_table()[cv[0, 0, 0]] * np.float64(dv[0])
    for r, (t, h) in enumerate(rows):
        if len(list_of(CU, off, idx, H, t, h)[2]) == 0:
            assert np.all(o64[r] == 0.0) and np.all(o16[r] == 0) and lse[r] == -np.inf
        else:
            np.testing.assert_array_equal(o64[r], np.full(128, want))


def test_a_proper_subset_of_blocks_differs_from_dense():
    """Negative control: listing only some key blocks must not reproduce dense attention."""
    cu = [0, 320]
    q, k, v = qkv(cu, 1, 17)
    lst = np.array([0, 2, 4], np.int32)
    off = np.array([0] + [3 * (i + 1) for i in range(5)], np.int32)
    idx = np.tile(lst, 5)
    rows = [(t, 0) for t in range(0, 320, 7)]
    a = oracle.attn_exact_sparse(bits(q), bits(k), bits(v), cu, off, idx, rows, SCALE)
    full = oracle.attn_exact(bits(q), bits(k), bits(v), cu, rows, SCALE)
    assert np.max(np.abs(a - full)) > 1e-3  # dropping blocks changes the result


@pytest.mark.parametrize("bad", [[1, 0], [0, 0], [5], [-1]])
def test_lists_breaking_the_contract_are_rejected(bad):
    cu = [0, 256]
    q, k, v = qkv(cu, 1, 1)
    lists = [np.array(bad), np.arange(4), np.arange(4), np.arange(4)]
    off = np.zeros(5, np.int32)
    off[1:] = np.cumsum([len(x) for x in lists])
    idx = np.concatenate(lists).astype(np.int32)
    with pytest.raises(ValueError):
        oracle.attn_exact_sparse(bits(q), bits(k), bits(v), cu, off, idx, [(0, 0)], SCALE)


def test_generator_shapes_and_order():
    cu = [0, 0, 17, 4113, 4113, 4500]
    off, idx = inputs.block_sparse_lists(cu, 3, density=0.25, seed=0, dense_every=7,
                                         empty_every=11)
    lens = [b - a for a, b in zip(cu[:-1], cu[1:])]
    G = sum((L + 63) // 64 for L in lens)
    assert off.shape == (3 * G + 1,) and off[0] == 0 and off[-1] == len(idx)
    assert np.all(np.diff(off) >= 0)
    for j in range(3 * G):
        lst = idx[off[j]:off[j + 1]]
        assert np.all(np.diff(lst) > 0)
