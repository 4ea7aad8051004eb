"""NVFP4 quantization (FlashInfer docs, minimax_h3_sm120_varlen_attention_nvfp4, description) on
the GPU through the C ABI, bit-exact against the oracle: K segment means, Q block means, E2M1
codes and UE4M3 scales of Q, K and V^T, padding bytes zero."""
import numpy as np
import pytest
import torch

import oracle
from precision_attention_diffusion_gb300 import inputs
from parity import bits, padded_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from precision_attention_diffusion_gb300 import build, fa_lp
    build.build()
    fa_lp.load()
    return fa_lp


def unpack_nibbles(a):
    lo = a & 0xF
    hi = a >> 4
    return np.stack([lo, hi], axis=-1).reshape(*a.shape[:-1], a.shape[-1] * 2)


def quantize_gpu(fa, q, k, v, cu, H):
    plan = fa.Plan(cu, H, mode=fa.MODE_NVFP4)
    plan.quantize(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    return plan


def gpu_natural(fa, plan, cu):
    offs = plan.row_offsets()
    rows, pad = padded_rows(cu, offs)
    g = {name: plan.quantized(getattr(fa, name)).cpu().numpy()
         for name in ("Q_CODES", "K_CODES", "V_CODES", "Q_SCALES", "K_SCALES", "V_SCALES",
                      "Q_MEANS", "K_MEANS")}
    qc, kc = unpack_nibbles(g["Q_CODES"]), unpack_nibbles(g["K_CODES"])   # [H][Tp][128]
    vc = unpack_nibbles(g["V_CODES"])                                      # [H][128][Tp]
    nat = dict(cq=qc[:, rows].transpose(1, 0, 2), ck=kc[:, rows].transpose(1, 0, 2),
               cv=vc[:, :, rows].transpose(2, 0, 1),
               sq=g["Q_SCALES"][:, rows].transpose(1, 0, 2),
               sk=g["K_SCALES"][:, rows].transpose(1, 0, 2), km=g["K_MEANS"])
    pads = dict(q=qc[:, pad], k=kc[:, pad], v=vc[:, :, pad], sq=g["Q_SCALES"][:, pad],
                sk=g["K_SCALES"][:, pad])
    return nat, pads, g, offs


def check_nvfp4_quant(fa, q, k, v, cu, H):
    plan = quantize_gpu(fa, q, k, v, cu, H)
    nat, pads, g, offs = gpu_natural(fa, plan, cu)
    z = oracle.nvfp4_quantize(bits(q), bits(k), bits(v), cu)
    for key in ("cq", "ck", "cv", "sq", "sk"):
        assert np.array_equal(nat[key], z[key]), key
    assert np.array_equal(nat["km"].view(np.uint32), z["km"].view(np.uint32)), "k means"
    for name, a in pads.items():
        assert np.all(a == 0), f"{name} padding not zero"
    # Q block means and V group scales: per segment, map the padded layout to the oracle's
    for s in range(len(cu) - 1):
        L = cu[s + 1] - cu[s]
        nb, ng = (L + 127) // 128, (L + 15) // 16
        b0, g0 = offs[s] // 128, offs[s] // 16
        got = g["Q_MEANS"][:, b0:b0 + nb].transpose(1, 0, 2)          # [nb][H][128]
        want = z["qm"][z["qoff"][s]:z["qoff"][s] + nb]
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), f"q means seg {s}"
        assert np.array_equal(g["V_SCALES"][:, :, g0:g0 + ng],
                              z["sv"][:, :, z["goff"][s]:z["goff"][s] + ng]), f"v scales seg {s}"
    return plan, z


def with_k_offset(k, H, seed):
    off = inputs.k_channel_offset(H, seed=seed)
    return (k.float() + off[None]).to(torch.bfloat16)


def test_nvfp4_quantize_small(fa):
    cu, H = [0, 256], 2
    q, k, v = inputs.qkv_separate(256, H, seed=0)
    check_nvfp4_quant(fa, q, with_k_offset(k, H, 0), v, cu, H)


def test_nvfp4_quantize_ragged_varlen(fa):
    cu, H = [0, 0, 17, 300, 300, 1400, 1500], 3
    q, k, v = inputs.qkv_separate(1500, H, seed=2)
    check_nvfp4_quant(fa, q, with_k_offset(k, H, 2), v, cu, H)


def test_nvfp4_quantize_strided_views(fa):
    buf, q, k, v = inputs.qkv_fused(333, 4, seed=4)
    check_nvfp4_quant(fa, q, k, v, [0, 100, 333], 4)


def test_nvfp4_quantize_h3_shape(fa):
    """S=30272, H=56 with the per-(head, channel) K offset N(0, 4): every code, scale and mean."""
    S, H = 30272, 56
    q, k, v = inputs.qkv_separate(S, H, seed=0)
    check_nvfp4_quant(fa, q, with_k_offset(k, H, 0), v, [0, S], H)
