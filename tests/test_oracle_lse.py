"""Pins for the oracle's row log-sum-exp (reading r15: LSE = m + log(l) in the natural units of
S = q.k scale; the SGLang PR #40175 kernel returns output and LSE, review thread). CPU only.

What pins what (nothing here retypes the oracle's own formula):
  * C1: scipy.special.logsumexp of scores computed here with numpy; the normalization identity
    sum_j exp(s_j - lse) = 1; a zero query gives log(L) exactly;
  * C2 (FP8) and C3 (NVFP4): a zero query makes every score 0, every quantized P exact (E4M3 1.0;
    UE4M3 448 x E2M1 6 = 2688), so the LSE is log(L) to rounding; against C1 the LSE differs by the
    P quantization only (|d| well below 0.1 on Gaussian inputs), and by much more when the softmax
    scale is wrong (negative control; the LSE does not depend on the order of the keys); C3's
    LSE follows the exact LSE of keys with a per-channel offset (the K centring is undone).
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from precision_attention_diffusion_gb300 import inputs

SCALE = 1.0 / math.sqrt(128)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).numpy().view(np.uint16)


def test_exact_lse_matches_scipy_logsumexp():
    T, H = 300, 2
    cu = [0, 120, 300]
    q, k, v = inputs.qkv_separate(T, H, seed=21)
    rows = [(t, h) for t in (0, 57, 119, 120, 233, 299) for h in range(H)]
    _, lse = oracle.attn_exact(bits(q), bits(k), bits(v), cu, rows, SCALE, lse=True)
    qf, kf = q.double().numpy(), k.double().numpy()
    for i, (t, h) in enumerate(rows):
        a, b = (0, 120) if t < 120 else (120, 300)
        s = kf[a:b, h] @ qf[t, h] * SCALE
        assert abs(lse[i] - logsumexp(s)) < 1e-12
        assert abs(np.exp(s - lse[i]).sum() - 1.0) < 1e-12


def test_zero_query_gives_log_length():
    T, H = 200, 1
    cu = [0, 37, 200]
    q = torch.zeros(T, H, 128, dtype=torch.bfloat16)
    _, k, v = inputs.qkv_separate(T, H, seed=22)
    rows = [(5, 0), (36, 0), (37, 0), (199, 0)]
    want = np.array([math.log(37)] * 2 + [math.log(163)] * 2)
    _, l1 = oracle.attn_exact(bits(q), bits(k), bits(v), cu, rows, SCALE, lse=True)
    assert np.allclose(l1, want, rtol=0, atol=1e-12)
    (cq, dq), (ck, dk), (cv, dv) = (oracle.fp8_quantize(bits(x)) for x in (q, k, v))
    for n_kv, tau in ((128, 0.0), (64, 8.0)):
        _, _, l2 = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, cu, rows, SCALE, n_kv=n_kv, tau=tau,
                                   lse=True)
        assert np.allclose(l2, want, rtol=0, atol=1e-12)
    z = oracle.nvfp4_quantize(bits(q), bits(k), bits(v), cu)
    _, _, l3 = oracle.attn_nvfp4(z, cu, rows, SCALE, n_kv=64, lse=True)
    assert np.allclose(l3, want, rtol=0, atol=1e-12)


@pytest.fixture(scope="module")
def gauss():
    T, H = 2048, 2
    q, k, v = inputs.qkv_separate(T, H, seed=23)
    rows = inputs.sample_rows([0, T], H, n_heads=2, n_rows=48, seed=4)
    _, exact = oracle.attn_exact(bits(q), bits(k), bits(v), [0, T], rows, SCALE, lse=True)
    return T, q, k, v, rows, exact


def test_fp8_lse_close_to_exact(gauss):
    T, q, k, v, rows, exact = gauss
    (cq, dq), (ck, dk), (cv, dv) = (oracle.fp8_quantize(bits(x)) for x in (q, k, v))
    _, _, l2 = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, [0, T], rows, SCALE, n_kv=64, tau=8.0,
                               lse=True)
    d = np.abs(l2 - exact)
    # |LSE| ~ 8 here: a log2 / ln mix-up (x 1.44 on log l) or a dropped m would be off by > 1
    assert d.max() < 0.05 and d.mean() < 0.02
    # doubling the softmax scale changes the LSE by far more than the quantization does
    _, _, l2x = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, [0, T], rows, 2 * SCALE, n_kv=64,
                                tau=8.0, lse=True)
    assert np.abs(l2x - exact).mean() > 10 * d.mean()


def test_nvfp4_lse_close_to_exact(gauss):
    T, q, k, v, rows, exact = gauss
    off = inputs.k_channel_offset(2, seed=23)
    k_off = (k.float() + off[None]).to(torch.bfloat16)
    # the K offset adds q.o to every score of a row: the exact LSE moves by exactly that
    _, exact_off = oracle.attn_exact(bits(q), bits(k_off), bits(v), [0, T], rows, SCALE,
                                     lse=True)
    z = oracle.nvfp4_quantize(bits(q), bits(k_off), bits(v), [0, T])
    _, _, l3 = oracle.attn_nvfp4(z, [0, T], rows, SCALE, n_kv=64, lse=True)
    # C3 restores the uncentred scores for its LSE: it tracks the exact LSE of the offset keys
    d = np.abs(l3 - exact_off)
    assert d.max() < 0.1 and d.mean() < 0.04
    # ... and differs from it by q.km scale (about 2 here) without that term: the offset matters
    qf = q.double().numpy()
    km = z["km"][0].astype(np.float64)
    shift = np.array([qf[t, h] @ km[h] * SCALE for t, h in rows])
    assert np.abs(shift).mean() > 20 * d.mean()
    assert np.allclose([z["qkm"][t, h] * SCALE for t, h in rows], shift, rtol=1e-12, atol=1e-12)
