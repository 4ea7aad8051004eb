"""Device memory returns to its baseline across distinct shapes (SGLang PR #40175, review: the
regression test that memory returns to baseline across sequence lengths).

Plans of several lengths run the FP8, NVFP4 and block-sparse forwards and the host-buffer entry;
after every plan is destroyed and the shared workspace released, the device's free memory is
back where it started (the stream-ordered pool trims at the synchronization), up to a few MB of
slack for the driver's own bookkeeping."""
import numpy as np
import pytest
import torch

from precision_attention_diffusion_gb300 import inputs

pytestmark = pytest.mark.gpu

SLACK = 16 << 20


@pytest.fixture(scope="module")
def fa():
    from precision_attention_diffusion_gb300 import build, fa_lp
    build.build()
    fa_lp.load()
    return fa_lp


def free_bytes(fa):
    torch.cuda.synchronize()
    fa.release_workspace()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return torch.cuda.mem_get_info()[0]


def test_distinct_shapes_release_memory(fa):
    H = 4
    base = free_bytes(fa)
    for S in (1052, 4096, 5980):
        cu = [0, 17, S]
        q, k, v = (x.cuda() for x in inputs.qkv_separate(S, H, seed=S))
        out = torch.empty((S, H, 128), dtype=torch.bfloat16, device="cuda")
        for mode in (fa.MODE_FP8, fa.MODE_NVFP4):
            plan = fa.Plan(cu, H, mode=mode)
            plan.attention(q, k, v, out=out)
            if mode == fa.MODE_FP8:
                off, idx = inputs.block_sparse_lists(cu, H, density=0.5, seed=S)
                plan.forward_sparse(torch.from_numpy(off).cuda(), torch.from_numpy(idx).cuda(),
                                    out)
                hq = torch.stack([q, k, v], dim=1).cpu().pin_memory()
                hout = torch.empty((S, H, 128), dtype=torch.bfloat16).pin_memory()
                plan.attention_host(hq[:, 0], hq[:, 1], hq[:, 2], hout, heads_per_chunk=2)
            torch.cuda.synchronize()
            assert plan.last_error() == 0
            plan.close()
        del q, k, v, out
    after = free_bytes(fa)
    assert after >= base - SLACK, (base - after) / 2**20


def test_forward_refuses_a_workspace_another_plan_overwrote(fa):
    """The quantized operands live in one workspace per device shared by every plan: after plan
    B quantizes, plan A's codes are gone, and A's forward returns FA_LP_ERR_STATE instead of
    attending over B's codes. Quantizing A again makes its forward valid again."""
    H = 2
    qa, ka, va = (x.cuda() for x in inputs.qkv_separate(300, H, seed=1))
    qb, kb, vb = (x.cuda() for x in inputs.qkv_separate(500, H, seed=2))
    a = fa.Plan([0, 300], H)
    b = fa.Plan([0, 200, 500], H)
    out = torch.empty((300, H, 128), dtype=torch.bfloat16, device="cuda")
    a.quantize(qa, ka, va)
    b.quantize(qb, kb, vb)
    with pytest.raises(fa.FaLpError) as e:
        a.forward(out)
    assert e.value.status == fa.FA_LP_ERR_STATE
    a.quantize(qa, ka, va)
    a.forward(out)
    want = torch.empty_like(out)
    a.attention(qa, ka, va, out=want)
    torch.cuda.synchronize()
    assert torch.equal(out, want)
    a.close()
    b.close()
