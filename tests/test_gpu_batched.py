"""Batch > 1 through varlen packing (fa_lp.attention_batched) on the GPU.

The batched front end only builds cu_seqlens = [0, S, 2S, ...] and packs the [B, S, H, 128]
views without copying; so its output must equal the packed varlen call bit for bit, and the
packed call's parity against the oracle (every row of every sequence) covers the rest. Also: a
fused [B, S, 3, H, 128] QKV buffer, and NVFP4.
"""
import numpy as np
import pytest
import torch

import oracle
from precision_attention_diffusion_gb300 import inputs
from parity import SCALE, all_rows, bits, out_rows, rel_rms

pytestmark = pytest.mark.gpu

KV_TILE, TAU = 64, 8.0


@pytest.fixture(scope="module")
def fa():
    from precision_attention_diffusion_gb300 import build, fa_lp
    build.build()
    fa_lp.load()
    return fa_lp


def fused_batch(B, S, H, seed):
    buf = inputs.gaussian_bf16((B, S, 3, H, 128), seed).cuda()
    return buf, buf[:, :, 0], buf[:, :, 1], buf[:, :, 2]


@pytest.mark.parametrize("mode", [0, 1])
def test_batched_equals_packed_varlen_call(fa, mode):
    B, S, H = 3, 300, 4
    _, q, k, v = fused_batch(B, S, H, seed=60)
    out_b = fa.attention_batched(q, k, v, mode=mode)
    cu = [i * S for i in range(B + 1)]
    qp, kp, vp = (fa.merge_batch(x, n) for x, n in ((q, "q"), (k, "k"), (v, "v")))
    plan = fa.Plan(cu, H, mode=mode)
    out_v = plan.attention(qp, kp, vp, torch.tensor(cu, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(out_b.reshape(B * S, H, 128).view(torch.int16), out_v.view(torch.int16))


def test_batched_fp8_parity_every_row(fa):
    """Each sequence attends to itself only: every row against the FP8-emulating oracle and the
    exact attention of its own sequence."""
    B, S, H = 2, 200, 2
    _, q, k, v = fused_batch(B, S, H, seed=61)
    out = fa.attention_batched(q, k, v)
    torch.cuda.synchronize()
    cu = [i * S for i in range(B + 1)]
    qp, kp, vp = (fa.merge_batch(x, n).cpu().contiguous() for x, n in ((q, "q"), (k, "k"), (v, "v")))
    (cq, dq), (ck, dk), (cv, dv) = (oracle.fp8_quantize(bits(x)) for x in (qp, kp, vp))
    rows = all_rows(cu, H)
    emu, _ = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, cu, rows, SCALE, n_kv=KV_TILE, tau=TAU)
    exact = oracle.attn_exact(bits(qp), bits(kp), bits(vp), cu, rows, SCALE)
    got = out_rows(out.reshape(B * S, H, 128), rows)
    assert rel_rms(got, emu) <= 1e-2
    assert rel_rms(got, exact) <= 0.06
    # no attention across sequences: sequence 1 alone gives the same exact reference
    one = oracle.attn_exact(bits(qp[S:]), bits(kp[S:]), bits(vp[S:]), [0, S],
                            [(t - S, h) for t, h in rows if t >= S], SCALE)
    assert np.allclose(exact[[i for i, (t, h) in enumerate(rows) if t >= S]], one, rtol=0, atol=0)
