"""The no-allocation FP8 descale entry point, checked against the regular path.

fa_lp_fp8_descale_noalloc is for callers that cannot let the library allocate device memory (their
memory belongs to their own pool, or their footprint is fixed after start-up, or cudaMalloc's
implicit synchronization is not acceptable where they call). Its scratch is a fixed device array
inside the library that every call shares. This file is collected last so that a run stopping at
the first failure has already run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from precision_attention_diffusion_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from precision_attention_diffusion_gb300 import build, fa_lp
    build.build()
    fa_lp.load()
    return fa_lp


def descale_regular(fa, q, k, v, T, H):
    plan = fa.Plan([0, T], H)
    plan.quantize(q, k, v)
    return plan.quantized(fa.DESCALE)[0].clone()


def test_noalloc_descale_matches_regular_path_on_two_calls(fa):
    T, H = 1000, 6
    _, q1, k1, v1 = inputs.qkv_fused(T, H, seed=21)
    q2, k2, v2 = (x * 3.0 for x in inputs.qkv_separate(T, H, seed=22))  # larger amax
    q1, k1, v1, q2, k2, v2 = (x.cuda() for x in (q1, k1, v1, q2, k2, v2))
    want1 = descale_regular(fa, q1, k1, v1, T, H)
    want2 = descale_regular(fa, q2, k2, v2, T, H)
    out = torch.full((3, H), -1.0, device="cuda")
    # two calls in a row on different inputs: the second must not see the first's scratch
    got1 = fa.fp8_descale_noalloc(q1, k1, v1).clone()
    fa.fp8_descale_noalloc(q2, k2, v2, out=out)
    torch.cuda.synchronize()
    # the descales are exact (amax / 448 with IEEE division), so the tolerance is zero
    assert torch.equal(got1, want1)
    assert torch.equal(out, want2)
    # and the second call after a larger one: clearing, not max with stale contents
    got3 = fa.fp8_descale_noalloc(q1, k1, v1)
    torch.cuda.synchronize()
    assert torch.equal(got3, want1)


def test_noalloc_allocates_no_device_memory(fa):
    """The property the entry point exists for: after a first call (which loads its kernels and
    looks up the scratch address), further calls at other sizes leave the device's free memory
    unchanged. Every tensor the calls touch is created before the first reading."""
    cases = [(1000, 6), (3000, 40), (1, 1), (4097, 1024)]
    ins = [tuple(x.cuda() for x in inputs.qkv_separate(T, H, seed=30 + i))
           for i, (T, H) in enumerate(cases)]
    outs = [torch.empty((3, H), dtype=torch.float32, device="cuda") for _, H in cases]
    fa.fp8_descale_noalloc(*ins[0], out=outs[0])
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for (q, k, v), o in zip(ins[1:], outs[1:]):
        fa.fp8_descale_noalloc(q, k, v, out=o)
        fa.fp8_descale_noalloc(q, k, v, out=o)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    for (q, k, v), o in zip(ins, outs):
        assert torch.equal(o, descale_regular(fa, q, k, v, q.shape[0], q.shape[1]))


def test_noalloc_rejects_sizes_beyond_its_scratch(fa):
    T, H = 4, 1025
    x = torch.zeros((T, H, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FaLpError) as e:
        fa.fp8_descale_noalloc(x, x, x)
    assert e.value.status == fa.FA_LP_ERR_INVALID_ARG
