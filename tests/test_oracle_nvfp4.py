"""Pins for the oracle's NVFP4 path (FlashInfer docs,
``minimax_h3_sm120_varlen_attention_nvfp4``, description): K means (a6), Q block means and
E2M1/UE4M3 packing (a7) and the NVFP4-emulating attention (C3). CPU only.

Pinned by: numpy means (an independent reduction), a hand-derived scale group (golden), a
reconstruction error bound, the segment-aligned group layout on ragged segments, softmax shift
invariance (the reason K can be centred), constant-V and one-hot exactness, the pages' FP4
tolerance (atol 1.0 / rtol 0.1 against FP32/FP64 attention, error about 4x FP8's), and a
scrambled-key negative control.
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
E2M1 = None


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def rel_rms(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def deq_rows(codes, sf):
    """[T,H,128] codes and [T,H,8] scales -> float64 values."""
    e2 = oracle.e2m1_decode_table()
    e4 = oracle.e4m3_decode_table()
    return e2[codes] * np.repeat(e4[sf], 16, axis=-1)


def test_kmean_and_qmean_match_numpy():
    cu = [0, 0, 17, 300, 300, 333]
    T, H = 333, 3
    q, k, v = inputs.qkv_separate(T, H, seed=4)
    off = inputs.k_channel_offset(H, seed=4)
    k = (k.float() + off[None]).to(torch.bfloat16)
    z = oracle.nvfp4_quantize(bits(q), bits(k), bits(v), cu)
    kf, qf = k.double().numpy(), q.double().numpy()
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        if a == b:
            assert np.all(z["km"][s] == 0)
            continue
        assert np.array_equal(z["km"][s], kf[a:b].mean(axis=0).astype(np.float32))
        for blk in range((b - a + 127) // 128):
            r0, r1 = a + 128 * blk, min(b, a + 128 * blk + 128)
            qb = z["qoff"][s] + blk
            assert np.array_equal(z["qm"][qb], qf[r0:r1].mean(axis=0).astype(np.float32))
    assert list(z["qoff"]) == [0, 0, 1, 4, 4, 5]
    assert list(z["goff"]) == [0, 0, 2, 20, 20, 23]


def test_golden_scale_group_on_v_and_k():
    g = GOLD["nvfp4_group"]
    x = torch.tensor(g["x"])
    T, H = 16, 1
    v = torch.zeros(T, H, 128)
    v[:, 0, 0] = x                       # 16 consecutive keys of channel 0 -> one V group
    k = torch.zeros(2, H, 128)
    k[0, 0, :16] = x                     # two K rows with zero mean -> centring is the identity
    k[1, 0, :16] = -x
    q = torch.zeros(T, H, 128)
    z = oracle.nvfp4_quantize(bits(q.to(torch.bfloat16)), bits(k.repeat(8, 1, 1).to(torch.bfloat16)),
                              bits(v.to(torch.bfloat16)), [0, T])
    assert z["sv"][0, 0, 0] == g["scale_code"]
    assert list(z["cv"][:, 0, 0]) == g["codes"]
    assert z["sk"][0, 0, 0] == g["scale_code"]
    assert list(z["ck"][0, 0, :16]) == g["codes"]
    flipped = [c ^ 8 for c in g["codes"]]  # -x: zeros become -0.0, whose code keeps the sign
    assert list(z["ck"][1, 0, :16]) == flipped
    # an all-zero group gets scale code 0 and codes 0
    assert z["sk"][0, 0, 1] == 0 and np.all(z["ck"][0, 0, 16:] == 0)


def test_reconstruction_error_bound():
    T, H = 256, 2
    q, k, v = inputs.qkv_separate(T, H, seed=12)
    z = oracle.nvfp4_quantize(bits(q), bits(k), bits(v), [0, T])
    e4 = oracle.e4m3_decode_table()
    kc = k.double().numpy() - z["km"][0][None].astype(np.float64)
    dk = deq_rows(z["ck"], z["sk"])
    sfk = np.repeat(e4[z["sk"]], 16, axis=-1)
    # E2M1 rounding error is at most half the widest gap (4 -> 6) times the scale, and the
    # E4M3 rounding of amax/6 keeps amax / scale <= 6.4, which saturates to 6 (error 0.4 scale)
    assert np.all(np.abs(kc - dk) <= sfk * 1.0 + 1e-7)
    e = rel_rms(dk, kc)
    assert 0.05 < e < 0.2, e


def test_v_groups_are_segment_aligned():
    cu = [0, 17, 17, 40]
    T, H = 40, 1
    q, k, v = inputs.qkv_separate(T, H, seed=13)
    z = oracle.nvfp4_quantize(bits(q), bits(k), bits(v), cu)
    assert list(z["goff"]) == [0, 2, 2, 4]
    v2 = v.clone()
    v2[17:] *= 64.0                     # other segment: scales of segment 0 must not move
    z2 = oracle.nvfp4_quantize(bits(q), bits(k), bits(v2), cu)
    assert np.array_equal(z["sv"][..., :2], z2["sv"][..., :2])
    assert np.array_equal(z["cv"][:17], z2["cv"][:17])
    assert not np.array_equal(z["sv"][..., 2:], z2["sv"][..., 2:])
    # a group holding only key 16 (15 zero pads): its scale is |v| / 6 rounded
    e4 = oracle.e4m3_decode_table()
    for c in range(0, 128, 17):
        a = abs(float(v[16, 0, c]))
        want = oracle.e4m3_encode(np.array([np.float32(a) / np.float32(6.0)]))[0]
        assert z["sv"][0, c, 1] == want


@pytest.fixture(scope="module")
def gauss():
    T, H = 2048, 4
    q, k, v = inputs.qkv_separate(T, H, seed=0)
    off = inputs.k_channel_offset(H, seed=0)
    k_off = (k.float() + off[None]).to(torch.bfloat16)
    rows = inputs.sample_rows([0, T], H, n_heads=2, n_rows=64, seed=1)
    return T, q, k, k_off, v, rows


def test_nvfp4_tolerance_against_exact(gauss):
    T, q, k, k_off, v, rows = gauss
    for kk in (k, k_off):
        exact = oracle.attn_exact(bits(q), bits(kk), bits(v), [0, T], rows, SCALE)
        z = oracle.nvfp4_quantize(bits(q), bits(kk), bits(v), [0, T])
        o64, _ = oracle.attn_nvfp4(z, [0, T], rows, SCALE)
        e = rel_rms(o64, exact)
        assert 0.1 < e < 0.25, e
        assert np.allclose(o64, exact, atol=1.0, rtol=0.1)
        # about 4x the FP8 error on Gaussian inputs
        (cq, dq), (ck, dk), (cv, dv) = (oracle.fp8_quantize(bits(t)) for t in (q, kk, v))
        f8, _ = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, [0, T], rows, SCALE)
        ratio = e / rel_rms(f8, exact)
        assert 2.5 < ratio < 6.0, ratio


def test_softmax_shift_invariance_and_centring():
    """q.(k + o) adds the same q.o to every score of a row: exact attention is unchanged, and the
    centred NVFP4 emulation stays within its error band."""
    T, H = 512, 2
    g = torch.Generator().manual_seed(7)
    q = (torch.randint(-16, 16, (T, H, 128), generator=g) / 8.0).to(torch.bfloat16)
    k = (torch.randint(-16, 16, (T, H, 128), generator=g) / 8.0).to(torch.bfloat16)
    v = inputs.gaussian_bf16((T, H, 128), seed=7)
    o = torch.randint(-8, 9, (H, 128), generator=g).float()
    k2 = (k.float() + o[None]).to(torch.bfloat16)
    assert torch.equal(k2.float() - o[None], k.float())  # exact in BF16
    rows = [(t, h) for t in range(0, T, 37) for h in range(H)]
    sc = 0.05
    e1 = oracle.attn_exact(bits(q), bits(k), bits(v), [0, T], rows, sc)
    e2 = oracle.attn_exact(bits(q), bits(k2), bits(v), [0, T], rows, sc)
    assert np.allclose(e1, e2, rtol=1e-10, atol=1e-12)
    z1 = oracle.nvfp4_quantize(bits(q), bits(k), bits(v), [0, T])
    z2 = oracle.nvfp4_quantize(bits(q), bits(k2), bits(v), [0, T])
    a, _ = oracle.attn_nvfp4(z1, [0, T], rows, sc)
    b, _ = oracle.attn_nvfp4(z2, [0, T], rows, sc)
    assert rel_rms(a, e1) < 0.25 and rel_rms(b, e1) < 0.25
    assert rel_rms(a, b) < 0.1


def test_nvfp4_constant_v_and_one_hot():
    T, H = 300, 1
    q, k, _ = inputs.qkv_separate(T, H, seed=3)
    v = torch.full((T, H, 128), 0.75).to(torch.bfloat16)   # 0.75 = 6 * 2^-3: scale exact
    z = oracle.nvfp4_quantize(bits(q), bits(k), bits(v), [0, T])
    _, o16 = oracle.attn_nvfp4(z, [0, T], [(0, 0), (299, 0)], SCALE)
    assert np.all(o16 == 0x3F40)  # BF16 0.75
    # one dominant key inside the first tile
    q1 = torch.zeros(T, H, 128); k1 = torch.zeros(T, H, 128)
    q1[:, :, 0] = 1.0
    k1[77, :, 0] = 1.0
    _, _, v1 = inputs.qkv_separate(T, H, seed=5)
    z = oracle.nvfp4_quantize(bits(q1.to(torch.bfloat16)), bits(k1.to(torch.bfloat16)), bits(v1), [0, T])
    o64, _ = oracle.attn_nvfp4(z, [0, T], [(3, 0), (250, 0)], 60.0)
    e2 = oracle.e2m1_decode_table(); e4 = oracle.e4m3_decode_table()
    g = z["goff"][0] + 77 // 16
    want = e2[z["cv"][77, 0]] * e4[z["sv"][0, :, g]]
    assert np.array_equal(o64[0], want) and np.array_equal(o64[1], want)


def test_nvfp4_scrambled_negative_control(gauss):
    T, q, k, k_off, v, rows = gauss
    exact = oracle.attn_exact(bits(q), bits(k), bits(v), [0, T], rows, SCALE)
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(9))
    z = oracle.nvfp4_quantize(bits(q), bits(k[perm].contiguous()), bits(v), [0, T])
    o64, _ = oracle.attn_nvfp4(z, [0, T], rows, SCALE)
    assert rel_rms(o64, exact) > 0.5


def _dominant_key_case(pos, T=2048, H=2, seed=11):
    """Every query row has its largest score at key `pos`: channel 0 of every q is raised by 8 and
    channel 0 of key `pos` is 30, so q.k_pos exceeds every other score by about 100 (raw units);
    with softmax scale 0.02 the other keys still carry weight."""
    q, k, v = inputs.qkv_separate(T, H, seed=seed)
    q = q.float(); k = k.float()
    q[:, :, 0] += 8.0
    k[pos, :, 0] = 30.0
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v


def _argmax_keys(q, k, rows):
    qf, kf = q.double(), k.double()
    return np.array([int((kf[:, h] @ qf[r, h]).argmax()) for r, h in rows])


def test_nvfp4_tile_width_invariance_when_max_is_first():
    """With the exact running maximum, the tile width only matters through the moments the
    maximum moves: when each row's maximum lies in the first 16 keys, every tile width (a multiple
    of 16) quantizes every P' against the same m, so the outputs agree bit for bit."""
    T = 2048
    q, k, v = _dominant_key_case(5, T)
    z = oracle.nvfp4_quantize(bits(q), bits(k), bits(v), [0, T])
    rows = inputs.sample_rows([0, T], 2, n_heads=2, n_rows=48, seed=3)
    assert np.all(_argmax_keys(q, k, rows) == 5)
    outs = [oracle.attn_nvfp4(z, [0, T], rows, 0.02, n_kv=n)[0] for n in (16, 64, 128, 4096)]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    # not degenerate: other keys still carry weight, so the output is not V of the dominant key
    e2 = oracle.e2m1_decode_table(); e4 = oracle.e4m3_decode_table()
    dom = e2[z["cv"][5, 0]] * e4[z["sv"][0, :, 0]]
    assert np.abs(outs[0][np.asarray(rows)[:, 1] == 0] - dom).max() > 1e-2


def test_nvfp4_tile_width_matters_when_max_moves():
    """The same rows with the dominant key at 1000: tiles before it are quantized against smaller
    maxima, so a 16-key and a 4096-key tiling give different (both valid) outputs."""
    T = 2048
    q, k, v = _dominant_key_case(1000, T)
    z = oracle.nvfp4_quantize(bits(q), bits(k), bits(v), [0, T])
    rows = inputs.sample_rows([0, T], 2, n_heads=2, n_rows=48, seed=3)
    assert np.all(_argmax_keys(q, k, rows) == 1000)
    a, _ = oracle.attn_nvfp4(z, [0, T], rows, 0.02, n_kv=16)
    b, _ = oracle.attn_nvfp4(z, [0, T], rows, 0.02, n_kv=4096)
    exact = oracle.attn_exact(bits(q), bits(k), bits(v), [0, T], rows, 0.02)
    assert not np.array_equal(a, b)
    assert rel_rms(a, exact) < 0.25 and rel_rms(b, exact) < 0.25


# ---------------------------------------------------------------------------------------------
# Brute force of C3 on rows whose segment fits one key tile: the online softmax then sees the
# whole row at once (its running maximum is the row maximum), so C3 must equal the global formula
# of the FlashInfer NVFP4 op's description, written here with numpy and ml_dtypes' own E2M1 /
# E4M3 conversions (a library independent of the oracle's converters):
#   S'  = scale (deq(Qc) + qm) deq(Kc)^T                      (qm K^T added back, reading r12)
#   P'  = fl32(2688 exp(S' - max S'))                          (row maximum to 448 * 6, r11)
#   per 16 keys from the segment start: sf = E4M3(fl32(amax16 / 6)),
#                                       code = E2M1(fl32(P' / deq(sf)))   (r9; sf 0 -> codes 0)
#   out = sum deq(P') deq(V) / sum deq(P')                      (l sums the dequantized P)
# The negative controls plant each plausible slip in this brute force (32-key groups, groups
# aligned to absolute token multiples of 16, 448 where 2688 belongs, the amax instead of amax / 6,
# the qm K^T term dropped) and check that the oracle disagrees with every one of them.
# ---------------------------------------------------------------------------------------------
def _bruteforce_nvfp4_row(z, cu, t, h, scale, group=16, aligned_abs=False, first_level=2688.0,
                          sf_div=6.0, with_qm=True):
    md = pytest.importorskip("ml_dtypes")
    e2 = lambda c: np.asarray(c, np.uint8).view(md.float4_e2m1fn).astype(np.float64)
    e4 = lambda c: np.asarray(c, np.uint8).view(md.float8_e4m3fn).astype(np.float64)
    s = max(i for i in range(len(cu) - 1) if cu[i] <= t < cu[i + 1])
    a, b = cu[s], cu[s + 1]
    qb = z["qoff"][s] + (t - a) // 128
    H = z["cq"].shape[1]
    dq = e2(z["cq"][t, h]) * np.repeat(e4(z["sq"][t, h]), 16)
    qm = z["qm"][qb, h].astype(np.float64) if with_qm else 0.0
    dk = e2(z["ck"][a:b, h]) * np.repeat(e4(z["sk"][a:b, h]), 16, axis=-1)
    sc = ((dq + qm) @ dk.T) * scale
    p = (first_level * np.exp(sc - sc.max())).astype(np.float32)
    pd = np.zeros(b - a)
    starts = range(a - (a % group if aligned_abs else 0), b, group)
    for g0 in starts:
        lo, hi = max(g0, a) - a, min(g0 + group, b) - a
        amax = p[lo:hi].max()
        # E4M3 satfinite (the correct path never exceeds 448: amax <= 2688)
        sf = np.minimum(np.float32(amax) / np.float32(sf_div), np.float32(448)).astype(md.float8_e4m3fn)
        dsf = np.float32(np.asarray(sf).astype(np.float64))
        if dsf == 0:
            continue
        y = np.clip(p[lo:hi] / dsf, -6.0, 6.0)  # E2M1 satfinite: nothing rounds past 6
        pd[lo:hi] = y.astype(md.float4_e2m1fn).astype(np.float64) * np.float64(dsf)
    G = z["sv"].shape[2]
    gi = z["goff"][s] + (np.arange(a, b) - a) // 16
    dv = e2(z["cv"][a:b, h]) * e4(z["sv"][h][:, gi]).T
    return (pd @ dv) / pd.sum()


@pytest.mark.parametrize("case", ["gaussian_ragged", "offsets_qm_matters"])
def test_nvfp4_single_tile_bruteforce_with_library_rounding(case):
    pytest.importorskip("ml_dtypes")
    if case == "gaussian_ragged":
        # segments of 37 (not a multiple of 16, starting at token 0) and 90 (starting at 37)
        cu, H, seed = [0, 37, 127], 2, 41
        q, k, v = inputs.qkv_separate(cu[-1], H, seed=seed)
    else:
        # per-channel K and Q offsets: K is centred away, and Q's block mean qm is large, so the
        # qm K^T term carries a visible share of every score
        cu, H, seed = [0, 0, 128, 203], 2, 43
        q, k, v = inputs.qkv_separate(cu[-1], H, seed=seed)
        k = (k.float() + inputs.k_channel_offset(H, seed=seed)[None]).to(torch.bfloat16)
        q = (q.float() + inputs.k_channel_offset(H, seed=seed + 1, std=1.5)[None]).to(torch.bfloat16)
    T = cu[-1]
    z = oracle.nvfp4_quantize(bits(q), bits(k), bits(v), cu)
    rows = [(t, h) for t in range(0, T, 5) for h in range(H)]
    o64, _ = oracle.attn_nvfp4(z, cu, rows, SCALE, n_kv=128)
    for r, (t, h) in enumerate(rows):
        want = _bruteforce_nvfp4_row(z, cu, t, h, SCALE)
        assert np.allclose(o64[r], want, rtol=1e-12, atol=1e-12), (t, h)
    # every planted slip moves some row by far more than the agreement above
    slips = [dict(group=32), dict(first_level=448.0), dict(sf_div=1.0)]
    # the ragged layout has a segment starting at token 37; the offset case has a large qm
    slips += [dict(aligned_abs=True)] if case == "gaussian_ragged" else [dict(with_qm=False)]
    for slip in slips:
        worst = max(np.abs(o64[r] - _bruteforce_nvfp4_row(z, cu, t, h, SCALE, **slip)).max()
                    for r, (t, h) in enumerate(rows))
        assert worst > 1e-4, slip
