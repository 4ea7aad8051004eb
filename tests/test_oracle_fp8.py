"""Pins for the oracle's FP8 path: quantization (a1), exact attention (C1) and the
FP8-emulating attention (C2). CPU only.

What pins what (nothing here retypes the oracle's own formula):
  * quantization: a hand-derived head (golden), the amax element mapping to 448, a
    dequantization error bound, and strided-view invariance;
  * C1: a textbook closed form (logistic pair), scipy's softmax on tiny inputs, constant V,
    one-hot keys, single-key segments, and segment isolation;
  * C2: constant V returns V exactly, a one-hot key returns that V row exactly (SGLang PR #36904's
    one-hot exactness test), a single-tile brute force with library E4M3 rounding, relative RMS
    against C1 inside the pages' FP8 band (SGLang PR #40175, Accuracy Tests: 0.0535-0.0539), and a
    scrambled-key negative control that must fail (SGLang PR #36904's control).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from precision_attention_diffusion_gb300 import inputs

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))
SCALE = 1.0 / math.sqrt(128)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_tensor(values, shape):
    return torch.tensor(values, dtype=torch.float32).reshape(shape).to(torch.bfloat16)


def rel_rms(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


# ---------------------------------------------------------------------------------------------
# a1 quantization
# ---------------------------------------------------------------------------------------------
def test_quantize_golden_head():
    g = GOLD["fp8_quantize_head"]
    x = torch.zeros(1, 1, 128)
    x[0, 0, :4] = torch.tensor(g["x"])
    codes, d = oracle.fp8_quantize(bits(x.to(torch.bfloat16)))
    assert list(codes[0, 0, :4]) == g["codes"]
    assert np.all(codes[0, 0, 4:] == 0)
    assert d[0] == np.float32(g["descale"])


def test_quantize_amax_maps_to_448_and_error_bound():
    x = inputs.gaussian_bf16((300, 3, 128), seed=3)
    codes, d = oracle.fp8_quantize(bits(x))
    dec = oracle.e4m3_decode_table()[codes]
    xf = x.float().numpy()
    for h in range(3):
        assert np.max(np.abs(dec[:, h])) == 448.0
        amax = np.abs(xf[:, h]).max()
        assert d[h] == np.float32(amax / np.float32(448.0))
        # E4M3 keeps 4 significant bits: relative error <= 2^-4 for normals, absolute <= 2^-10
        # (half the subnormal step) below 2^-6, before the descale
        err = np.abs(dec[:, h] * d[h] - xf[:, h])
        bound = np.maximum(np.abs(xf[:, h]) * 2.0 ** -4, d[h] * 2.0 ** -10) * 1.0001 + 1e-12
        assert np.all(err <= bound)


def test_quantize_strided_view_matches_contiguous():
    buf, q, k, v = inputs.qkv_fused(64, 4, seed=5)
    for view in (q, k, v):
        c1, d1 = oracle.fp8_quantize(bits(view))
        c2, d2 = oracle.fp8_quantize(bits(view.contiguous()))
        assert np.array_equal(c1, c2) and np.array_equal(d1, d2)


def test_quantize_zero_head():
    x = torch.zeros(10, 2, 128, dtype=torch.bfloat16)
    x[:, 1] = 1.0
    codes, d = oracle.fp8_quantize(bits(x))
    assert d[0] == 1.0 and np.all(codes[:, 0] == 0)
    assert np.all(codes[:, 1] == 126) and d[1] == np.float32(1.0 / 448.0)


# ---------------------------------------------------------------------------------------------
# C1 exact attention
# ---------------------------------------------------------------------------------------------
def test_exact_logistic_closed_form():
    q = torch.zeros(2, 1, 128); k = torch.zeros(2, 1, 128); v = torch.zeros(2, 1, 128)
    q[0, 0, 0] = 1.0
    k[1, 0, 0] = 2.0
    v[0, 0, 0] = 1.0
    v[1, 0, 1] = 1.0
    out = oracle.attn_exact(*(bits(t.to(torch.bfloat16)) for t in (q, k, v)), [0, 2], [(0, 0)], 1.0)
    w = GOLD["attention_logistic"]["out_first_two"]
    assert abs(out[0, 0] - w[0]) < 1e-15 and abs(out[0, 1] - w[1]) < 1e-15
    assert np.all(out[0, 2:] == 0)


def test_exact_tiny_bruteforce_against_scipy():
    special = pytest.importorskip("scipy.special")
    cu = [0, 3, 3, 8]
    q, k, v = inputs.qkv_separate(8, 2, seed=11)
    rows = [(t, h) for t in range(8) for h in range(2)]
    out = oracle.attn_exact(bits(q), bits(k), bits(v), cu, rows, SCALE)
    qf, kf, vf = (t.double().numpy() for t in (q, k, v))
    for r, (t, h) in enumerate(rows):
        a, b = (0, 3) if t < 3 else (3, 8)
        p = special.softmax(qf[t, h] @ kf[a:b, h].T * SCALE)
        assert np.allclose(out[r], p @ vf[a:b, h], rtol=1e-13, atol=1e-14)


def test_exact_invariants():
    T, H = 200, 2
    q, k, _ = inputs.qkv_separate(T, H, seed=2)
    cu = [0, 1, 57, 200]
    rows = [(t, h) for t in (0, 1, 30, 56, 57, 199) for h in range(H)]
    # constant V -> V; rows sum to one (V = ones)
    vconst = torch.full((T, H, 128), 0.75).to(torch.bfloat16)
    out = oracle.attn_exact(bits(q), bits(k), bits(vconst), cu, rows, SCALE)
    assert np.allclose(out, 0.75, rtol=0, atol=1e-15)
    # single-key segment returns its v row
    _, _, v = inputs.qkv_separate(T, H, seed=4)
    out = oracle.attn_exact(bits(q), bits(k), bits(v), cu, [(0, 0), (0, 1)], SCALE)
    assert np.array_equal(out, v[0].double().numpy())
    # one dominant key returns that v row
    q2 = torch.zeros(T, H, 128); k2 = torch.zeros(T, H, 128)
    q2[:, :, 0] = 8.0
    k2[100, :, 0] = 8.0
    out = oracle.attn_exact(bits(q2.to(torch.bfloat16)), bits(k2.to(torch.bfloat16)), bits(v), cu,
                            [(60, 0), (150, 1)], 1.0)
    assert np.allclose(out[0], v[100, 0].double().numpy(), atol=1e-20, rtol=1e-12)
    assert np.allclose(out[1], v[100, 1].double().numpy(), atol=1e-20, rtol=1e-12)


def test_exact_segment_isolation():
    T, H = 64, 1
    q, k, v = inputs.qkv_separate(T, H, seed=8)
    cu = [0, 20, 64]
    rows = [(t, 0) for t in range(20)]
    base = oracle.attn_exact(bits(q), bits(k), bits(v), cu, rows, SCALE)
    k2, v2 = k.clone(), v.clone()
    k2[20:] = 5.0
    v2[20:] = -3.0
    moved = oracle.attn_exact(bits(q), bits(k2), bits(v2), cu, rows, SCALE)
    assert np.array_equal(base, moved)


# ---------------------------------------------------------------------------------------------
# C2 FP8-emulating attention
# ---------------------------------------------------------------------------------------------
def quant3(q, k, v):
    (cq, dq), (ck, dk), (cv, dv) = (oracle.fp8_quantize(bits(t)) for t in (q, k, v))
    return cq, ck, cv, dq, dk, dv


def test_fp8_constant_v_returns_v():
    T, H = 700, 2
    q, k, _ = inputs.qkv_separate(T, H, seed=1)
    v = torch.full((T, H, 128), -1.5).to(torch.bfloat16)
    cu = [0, 300, 700]
    rows = [(t, h) for t in (0, 299, 300, 699) for h in range(H)]
    o64, o16 = oracle.attn_fp8(*quant3(q, k, v), cu, rows, SCALE)
    assert np.all(o16 == 0xBFC0)  # BF16 bits of -1.5
    assert np.allclose(o64, -1.5, rtol=1e-6)


def test_fp8_one_hot_key_is_exact():
    """A dominant key: every other probability underflows E4M3, so out = deq(v row) exactly."""
    T, H = 400, 1
    q = torch.zeros(T, H, 128); k = torch.zeros(T, H, 128)
    q[:, :, 0] = 1.0
    k[:, :, 0] = 0.01
    k[50, :, 0] = 1.0    # dominant key inside the first 128-key tile: exact
    _, _, v = inputs.qkv_separate(T, H, seed=9)
    cq, ck, cv, dq, dk, dv = quant3(q.to(torch.bfloat16), k.to(torch.bfloat16), v)
    o64, _ = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, [0, T], [(5, 0), (390, 0)], 40.0)
    want = oracle.e4m3_decode_table()[cv[50, 0]].astype(np.float64) * np.float64(dv[0])
    assert np.array_equal(o64[0], want) and np.array_equal(o64[1], want)
    # dominant key in a later tile: earlier tiles leave only alpha-scaled residues
    # (alpha = exp(0.4 - 40) ~ 6e-18 per earlier key), far below BF16 resolution
    k[50, :, 0] = 0.01
    k[333, :, 0] = 1.0
    cq, ck, cv, dq, dk, dv = quant3(q.to(torch.bfloat16), k.to(torch.bfloat16), v)
    o64, o16 = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, [0, T], [(5, 0)], 40.0)
    want = oracle.e4m3_decode_table()[cv[333, 0]].astype(np.float64) * np.float64(dv[0])
    assert np.max(np.abs(o64[0] - want)) <= 1e-14 * np.abs(want).max()
    assert np.array_equal(o16[0], oracle.f64_to_bf16(want))


def test_fp8_single_tile_bruteforce_with_library_rounding():
    """L <= n_kv: the online softmax is one tile, so C2 equals the global-max formula computed
    with numpy and torch's E4M3 rounding."""
    T, H = 96, 2
    q, k, v = inputs.qkv_separate(T, H, seed=21)
    cq, ck, cv, dq, dk, dv = quant3(q, k, v)
    rows = [(t, h) for t in range(0, T, 7) for h in range(H)]
    o64, _ = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, [0, T], rows, SCALE, n_kv=128)
    dec = lambda c: torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).double().numpy()
    for r, (t, h) in enumerate(rows):
        s = (dec(cq[t, h]) @ dec(ck[:, h]).T) * (float(dq[h]) * float(dk[h]) * SCALE)
        p = np.exp(s - s.max()).astype(np.float32)
        pq = torch.from_numpy(p).to(torch.float8_e4m3fn).double().numpy()
        want = (pq @ dec(cv[:, h])) * float(dv[h]) / pq.sum()
        assert np.allclose(o64[r], want, rtol=1e-12, atol=1e-14)


@pytest.fixture(scope="module")
def gaussian_2048():
    T, H = 2048, 4
    q, k, v = inputs.qkv_separate(T, H, seed=0)
    rows = inputs.sample_rows([0, T], H, n_heads=2, n_rows=96, seed=1)
    exact = oracle.attn_exact(bits(q), bits(k), bits(v), [0, T], rows, SCALE)
    return q, k, v, rows, exact


def test_fp8_relative_rms_in_page_band(gaussian_2048):
    q, k, v, rows, exact = gaussian_2048
    o64, _ = oracle.attn_fp8(*quant3(q, k, v), [0, 2048], rows, SCALE)
    e = rel_rms(o64, exact)
    # FP8 Q/K/V/P error on Gaussian inputs: the pages report 0.0535-0.0539 at S=20440/30272
    assert 0.02 < e < 0.06, e


def test_fp8_kv_tile_width_changes_little(gaussian_2048):
    q, k, v, rows, exact = gaussian_2048
    qz = quant3(q, k, v)
    a, _ = oracle.attn_fp8(*qz, [0, 2048], rows, SCALE, n_kv=128)
    b, _ = oracle.attn_fp8(*qz, [0, 2048], rows, SCALE, n_kv=64)
    c, _ = oracle.attn_fp8(*qz, [0, 2048], rows, SCALE, n_kv=4096)
    # neighbouring tile widths move the emulated output a little ...
    assert 0 < rel_rms(a, b) < 0.02
    # ... but quantizing P against the global row max (one tile) moves it by more than the 1e-2
    # kernel gate: the emulation must replay the kernel's own tile width and max rule
    assert 0.01 < rel_rms(a, c) < 0.05
    assert rel_rms(c, exact) < 0.06
    p8, _ = oracle.attn_fp8(*qz, [0, 2048], rows, SCALE, n_kv=128, p_shift=8)
    assert rel_rms(p8, exact) < 0.06


def test_fp8_scrambled_keys_negative_control(gaussian_2048):
    q, k, v, rows, exact = gaussian_2048
    perm = torch.randperm(2048, generator=torch.Generator().manual_seed(3))
    o64, _ = oracle.attn_fp8(*quant3(q, k[perm].contiguous(), v), [0, 2048], rows, SCALE)
    assert rel_rms(o64, exact) > 0.5


def test_fp8_varlen_rows_match_single_segment_runs():
    """Each segment of a packed batch gives the same rows as that segment run alone (the
    quantization scales are shared, so quantize once over the packed tensor)."""
    cu = [0, 0, 17, 150, 150, 333]
    T, H = 333, 2
    q, k, v = inputs.qkv_separate(T, H, seed=6)
    qz = quant3(q, k, v)
    rows = [(t, h) for t in (0, 16, 17, 149, 150, 332) for h in range(H)]
    packed, _ = oracle.attn_fp8(*qz, cu, rows, SCALE)
    for r, (t, h) in enumerate(rows):
        a, b = (0, 17) if t < 17 else ((17, 150) if t < 150 else (150, 333))
        cq, ck, cv, dq, dk, dv = qz
        alone, _ = oracle.attn_fp8(cq[a:b], ck[a:b], cv[a:b], dq, dk, dv, [0, b - a], [(t - a, h)], SCALE)
        assert np.array_equal(packed[r], alone[0])


def test_fp8_lazy_reference_max_rule():
    """tau > 0: while no later tile's maximum exceeds the first tile's by more than tau (log2
    units), every probability is taken against the first tile's maximum -- checked with the
    global formula on a 3-tile row, using torch's E4M3 rounding; tau = 0 is the exact rule."""
    T, H = 300, 1
    q, k, v = inputs.qkv_separate(T, H, seed=31)
    cq, ck, cv, dq, dk, dv = quant3(q, k, v)
    rows = [(t, 0) for t in range(0, T, 29)]
    dec = lambda c: torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).double().numpy()
    lazy, _ = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, [0, T], rows, SCALE, n_kv=128, tau=8.0)
    for r, (t, h) in enumerate(rows):
        s = (dec(cq[t, h]) @ dec(ck[:, h]).T) * (float(dq[h]) * float(dk[h]) * SCALE)
        m0 = s[:128].max()
        assert s.max() - m0 <= 8 * np.log(2)  # the rule never moves the reference here
        p = np.exp(s - m0).astype(np.float32)
        pq = torch.from_numpy(p).to(torch.float8_e4m3fn).double().numpy()
        want = (pq @ dec(cv[:, h])) * float(dv[h]) / pq.sum()
        assert np.allclose(lazy[r], want, rtol=1e-12, atol=1e-14)
    exact0, _ = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, [0, T], rows, SCALE, n_kv=128, tau=0.0)
    exact1, _ = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, [0, T], rows, SCALE, n_kv=128)
    assert np.array_equal(exact0, exact1)
    # a tile whose maximum jumps by more than tau moves the reference: tile 2 holds a key 12 log2
    # units above the rest, so the result equals the exact rule's on that row
    k2 = k.clone()
    k2[260] = q[0] * 4.0
    cq, ck, cv, dq, dk, dv = quant3(q, k2, v)
    a, _ = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, [0, T], [(0, 0)], SCALE, tau=8.0)
    b, _ = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, [0, T], [(0, 0)], SCALE, tau=0.0)
    s = (dec(cq[0, 0]) @ dec(ck[:, 0]).T) * (float(dq[0]) * float(dk[0]) * SCALE)
    assert s[256:].max() - s[:256].max() > 8 * np.log(2)
    assert np.allclose(a, b, rtol=1e-3)


# ---------------------------------------------------------------------------------------------
# The per-segment FP8 mode (the alternative of reading r1 that SGLang PR #40175's per-head amax
# leaves open for packed batches): one scale per (segment, tensor, head). Pinned by reduction to
# the per-tensor path, which is pinned above: a packed batch quantized per segment gives, for
# every segment, exactly the codes, descales and attention rows of that segment quantized and run
# alone.
# ---------------------------------------------------------------------------------------------
def test_fp8_segment_scales_equal_each_segment_alone():
    cu = [0, 0, 17, 150, 150, 333]
    T, H = 333, 2
    q, k, v = inputs.qkv_separate(T, H, seed=61)
    # segment amax 100x apart: the short middle segment is small, the last one large
    scale_rows = torch.ones(T, 1, 1)
    scale_rows[17:150] = 0.01
    scale_rows[150:] = 3.0
    q, k, v = ((x.float() * scale_rows).to(torch.bfloat16) for x in (q, k, v))
    quant = [oracle.fp8_quantize_seg(bits(x), cu) for x in (q, k, v)]
    cq, ck, cv = (z[0] for z in quant)
    dq, dk, dv = (z[1] for z in quant)
    assert dq.shape == (5, H)
    assert np.all(dq[[0, 3]] == 1.0)          # empty segments: descale 1
    rows = [(t, h) for t in (0, 16, 17, 80, 149, 150, 332) for h in range(H)]
    packed, _ = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, cu, rows, SCALE, n_kv=64, tau=8.0)
    for s, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        if a == b:
            continue
        alone = [oracle.fp8_quantize(bits(x[a:b].contiguous())) for x in (q, k, v)]
        for (c_seg, d_seg), (c_alone, d_alone) in zip(quant, alone):
            assert np.array_equal(c_seg[a:b], c_alone)
            assert np.array_equal(d_seg[s], d_alone)
        for r, (t, h) in enumerate(rows):
            if a <= t < b:
                want, _ = oracle.attn_fp8(*(z[0] for z in alone), *(z[1] for z in alone),
                                          [0, b - a], [(t - a, h)], SCALE, n_kv=64, tau=8.0)
                assert np.array_equal(packed[r], want[0])
    # one segment: the per-segment mode is the per-tensor mode
    c1, d1 = oracle.fp8_quantize_seg(bits(v), [0, T])
    c0, d0 = oracle.fp8_quantize(bits(v))
    assert np.array_equal(c1, c0) and np.array_equal(d1[0], d0)


def test_fp8_segment_scales_help_a_small_segment_beside_a_large_one():
    """Why the mode exists: a segment whose V is 3e-5 times its neighbour's falls into the E4M3
    subnormal range under the shared per-head scale (error 0.18 against exact attention) and keeps
    the FP8 error band (below 0.06, the pages' 0.0535-0.0539) with its own scale."""
    cu = [0, 200, 400]
    T, H = 400, 1
    q, k, v = inputs.qkv_separate(T, H, seed=62)
    sr = torch.ones(T, 1, 1)
    sr[:200] = 3e-5
    v = (v.float() * sr).to(torch.bfloat16)
    rows = [(t, 0) for t in range(0, 200, 9)]
    exact = oracle.attn_exact(bits(q), bits(k), bits(v), cu, rows, SCALE)
    shq = [oracle.fp8_quantize(bits(x)) for x in (q, k, v)]
    shared, _ = oracle.attn_fp8(*(z[0] for z in shq), *(z[1] for z in shq), cu, rows, SCALE,
                                n_kv=64, tau=8.0)
    segq = [oracle.fp8_quantize_seg(bits(x), cu) for x in (q, k, v)]
    own, _ = oracle.attn_fp8(*(z[0] for z in segq), *(z[1] for z in segq), cu, rows, SCALE,
                             n_kv=64, tau=8.0)
    assert rel_rms(own, exact) < 0.06
    assert rel_rms(shared, exact) > 0.15
