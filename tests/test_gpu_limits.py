"""Limits of the plan on the GPU, through the C ABI, against the oracle: the largest head count a
plan accepts (1024) and a single segment much longer than the benchmark's (131072 tokens, past
every 16-bit index of the token axis), for the FP8 and the NVFP4 path.

Bars as in test_gpu_fp8.py / test_gpu_nvfp4.py: codes bit-exact where checked; FP8 outputs within
relative RMS 1e-2 of the FP8-emulating oracle and 0.06 of exact attention; NVFP4 outputs within
atol 1.0 / rtol 0.1 of exact attention and relative RMS 1e-2 of the NVFP4-emulating oracle."""
import numpy as np
import pytest
import torch

import oracle
from precision_attention_diffusion_gb300 import inputs
from parity import SCALE, bits, out_rows, padded_rows, rel_rms

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from precision_attention_diffusion_gb300 import build, fa_lp
    build.build()
    fa_lp.load()
    return fa_lp


def run(fa, mode, q, k, v, cu, H):
    plan = fa.Plan(cu, H, mode=mode)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    plan.attention(q.cuda(), k.cuda(), v.cuda(), torch.tensor(cu, dtype=torch.int32,
                                                              device="cuda"), out=out)
    torch.cuda.synchronize()
    assert plan.last_error() == 0
    return plan, out


def fp8_natural(fa, plan, cu):
    rows, _ = padded_rows(cu, plan.row_offsets())
    qc = plan.quantized(fa.Q_CODES).cpu().numpy()
    kc = plan.quantized(fa.K_CODES).cpu().numpy()
    vt = plan.quantized(fa.V_CODES).cpu().numpy()
    ds = plan.quantized(fa.DESCALE).cpu().numpy()[0]
    return (qc[:, rows].transpose(1, 0, 2), kc[:, rows].transpose(1, 0, 2),
            vt[:, :, rows].transpose(2, 0, 1), ds)


def check_fp8(fa, plan, out, q, k, v, cu, rows, codes_exact=True):
    cq, ck, cv, ds = fp8_natural(fa, plan, cu)
    if codes_exact:
        for got, x, i in ((cq, q, 0), (ck, k, 1), (cv, v, 2)):
            want, d = oracle.fp8_quantize(bits(x))
            assert np.array_equal(got, want) and np.array_equal(ds[i], d)
    emu, _ = oracle.attn_fp8(cq, ck, cv, ds[0], ds[1], ds[2], cu, rows, SCALE, n_kv=64, tau=8.0)
    exact = oracle.attn_exact(bits(q), bits(k), bits(v), cu, rows, SCALE)
    got = out_rows(out, rows)
    per_row = np.linalg.norm(got - emu, axis=1) / np.maximum(np.linalg.norm(emu, axis=1), 1e-30)
    assert rel_rms(got, emu) <= 1e-2 and per_row.max() <= 5e-2, (rel_rms(got, emu), per_row.max())
    assert rel_rms(got, exact) <= 0.06


def check_nvfp4(out, q, k, v, cu, rows):
    z = oracle.nvfp4_quantize(bits(q), bits(k), bits(v), cu)
    emu, _ = oracle.attn_nvfp4(z, cu, rows, SCALE, n_kv=64)
    exact = oracle.attn_exact(bits(q), bits(k), bits(v), cu, rows, SCALE)
    got = out_rows(out, rows)
    per_row = np.linalg.norm(got - emu, axis=1) / np.maximum(np.linalg.norm(emu, axis=1), 1e-30)
    assert rel_rms(got, emu) <= 1e-2 and per_row.max() <= 5e-2, (rel_rms(got, emu), per_row.max())
    assert np.allclose(got, exact, atol=1.0, rtol=0.1)


def test_fp8_and_nvfp4_at_the_largest_head_count(fa):
    """H = 1024 (the plan's limit) over a ragged two-segment batch: every head's scales and codes
    (FP8), rows of the first, middle and last heads against the oracles."""
    cu, H = [0, 77, 300], 1024
    q, k, v = inputs.qkv_separate(cu[-1], H, seed=91)
    plan, out = run(fa, fa.MODE_FP8, q, k, v, cu, H)
    rows = [(t, h) for t in (0, 76, 77, 150, 299) for h in (0, 1, 511, 512, 1022, 1023)]
    check_fp8(fa, plan, out, q, k, v, cu, rows)
    k4 = (k.float() + inputs.k_channel_offset(H, seed=91)[None]).to(torch.bfloat16)
    _, out4 = run(fa, fa.MODE_NVFP4, q, k4, v, cu, H)
    check_nvfp4(out4, q, k4, v, cu, rows)


def test_fp8_and_nvfp4_on_a_131072_token_segment(fa):
    """One segment of 131072 tokens (four times the benchmark's), two heads: FP8 codes bit-exact
    over the whole segment, sampled rows against the oracles, for both paths."""
    S, H = 131072, 2
    cu = [0, S]
    q, k, v = inputs.qkv_separate(S, H, seed=92)
    rows = inputs.sample_rows(cu, H, n_heads=2, n_rows=24, seed=3)
    plan, out = run(fa, fa.MODE_FP8, q, k, v, cu, H)
    check_fp8(fa, plan, out, q, k, v, cu, rows)
    del plan
    k4 = (k.float() + inputs.k_channel_offset(H, seed=92)[None]).to(torch.bfloat16)
    _, out4 = run(fa, fa.MODE_NVFP4, q, k4, v, cu, H)
    check_nvfp4(out4, q, k4, v, cu, rows)
