"""The host-buffer entry point (fa_lp_attention_host) on the GPU.

Every step of the path is independent per head (FP8 scales per (tensor, head); NVFP4 means and
scales per head), so the head-chunked, copy-overlapped schedule must return exactly what the
device-buffer call returns on the same data: compared bit for bit, for several chunk sizes, a
fused-QKV host layout, pageable and page-locked memory, a strided host output, and both modes.
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


def fused_host(T, H, seed, pin=True):
    q, k, v = inputs.qkv_separate(T, H, seed=seed)
    buf = torch.stack([q, k, v], dim=1).contiguous()  # [T, 3, H, 128]
    return buf.pin_memory() if pin else buf


def device_reference(fa, plan, buf):
    d = buf.cuda()
    out = torch.empty((buf.shape[0], buf.shape[2], 128), dtype=torch.bfloat16, device="cuda")
    plan.attention(d[:, 0], d[:, 1], d[:, 2], out=out)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("mode", [0, 1])
def test_host_entry_equals_device_call(fa, mode):
    T, H = 1500, 6
    cu = [0, 17, 700, 1500]
    buf = fused_host(T, H, seed=31)
    plan = fa.Plan(cu, H, mode=mode)
    ref = device_reference(fa, plan, buf)
    for nh in (0, 1, 4, 6):
        out = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16).pin_memory()
        plan.attention_host(buf[:, 0], buf[:, 1], buf[:, 2], out, heads_per_chunk=nh)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"heads_per_chunk={nh}"
    assert plan.last_error() == 0


def test_host_entry_nvfp4_under_a_table_limit(fa):
    """NVFP4 through the host entry with the plan's qm K^T table limited to one head per slot: the
    chunk plans take the limit (their tables become rings of one-head slots) and the result still
    equals the whole-table device call bit for bit."""
    T, H = 1500, 6
    cu = [0, 17, 700, 1500]
    buf = fused_host(T, H, seed=33)
    plan = fa.Plan(cu, H, mode=1)
    ref = device_reference(fa, plan, buf)
    head_bytes = sum(((b - a + 127) // 128) ** 2 for a, b in zip(cu[:-1], cu[1:])) * 128 * 4
    try:
        plan.set_table_limit(2 * head_bytes)
        for nh in (0, 3):
            out = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16).pin_memory()
            plan.attention_host(buf[:, 0], buf[:, 1], buf[:, 2], out, heads_per_chunk=nh)
            torch.cuda.synchronize()
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"heads_per_chunk={nh}"
            sub = fa.Plan(cu, 3, mode=1)  # the 3-head chunk plan (from the plan cache)
            if nh == 3:
                assert sub.table_layout() == dict(heads_per_slot=1, slots=2, slot_bytes=head_bytes)
        assert plan.last_error() == 0
    finally:
        plan.set_table_limit(0)
        fa.Plan(cu, 3, mode=1).set_table_limit(0)


def test_host_entry_pageable_memory_and_strided_output(fa):
    T, H = 900, 5
    cu = [0, 300, 301, 900]
    buf = fused_host(T, H, seed=32, pin=False)
    plan = fa.Plan(cu, H, mode=0)
    ref = device_reference(fa, plan, buf)
    # output heads 256 channels apart inside a larger host buffer: the gaps stay untouched
    big = torch.full((T, H, 256), 7.0, dtype=torch.bfloat16)
    out = big[:, :, :128]
    plan.attention_host(buf[:, 0], buf[:, 1], buf[:, 2], out, heads_per_chunk=2)
    torch.cuda.synchronize()
    assert torch.equal(out.contiguous().view(torch.int16), ref.view(torch.int16))
    assert bool((big[:, :, 128:] == 7.0).all())


def test_host_entry_repeated_calls_and_chunk_changes(fa):
    T, H = 640, 8
    cu = [0, 640]
    plan = fa.Plan(cu, H, mode=0)
    for i, nh in enumerate((3, 3, 8, 0, 1)):
        buf = fused_host(T, H, seed=40 + i)
        ref = device_reference(fa, plan, buf)
        out = torch.empty((T, H, 128), dtype=torch.bfloat16).pin_memory()
        plan.attention_host(buf[:, 0], buf[:, 1], buf[:, 2], out, heads_per_chunk=nh)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), (i, nh)


def test_host_entry_reports_device_wait_expiry(fa):
    """An expired device-side wait inside a chunk is reported on the plan the caller holds."""
    T, H = 512, 4
    plan = fa.Plan([0, T], H, mode=0)
    buf = fused_host(T, H, seed=50)
    out = torch.empty((T, H, 128), dtype=torch.bfloat16).pin_memory()
    plan.set_wait_limit(1)
    try:
        plan.attention_host(buf[:, 0], buf[:, 1], buf[:, 2], out, heads_per_chunk=2)
        torch.cuda.synchronize()
        assert plan.last_error() != 0
    finally:
        plan.set_wait_limit(20000)
    plan.attention_host(buf[:, 0], buf[:, 1], buf[:, 2], out, heads_per_chunk=2)
    torch.cuda.synchronize()
    assert plan.last_error() == 0
    assert torch.equal(out.view(torch.int16), device_reference(fa, plan, buf).view(torch.int16))


def test_host_entry_default_schedule_many_heads(fa):
    """The library's default chunking with enough heads for several chunks and a two-segment
    segmentation."""
    T, H = 2048, 24
    buf = fused_host(T, H, seed=55)
    plan = fa.Plan([0, 1000, T], H, mode=0)
    ref = device_reference(fa, plan, buf)
    out = torch.empty((T, H, 128), dtype=torch.bfloat16).pin_memory()
    plan.attention_host(buf[:, 0], buf[:, 1], buf[:, 2], out)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("hpc", [0, 3, 7])
def test_sparse_host_entry_equals_device_call(fa, hpc):
    """fa_lp_attention_sparse_host (block lists from host memory, head chunks with their lists'
    offsets from h0 G on) returns the device-buffer block-sparse forward's output bit for bit."""
    cu, H = [0, 0, 17, 300, 300, 1400, 1500], 7
    T = cu[-1]
    buf = fused_host(T, H, seed=21)
    off, idx = inputs.block_sparse_lists(cu, H, density=0.4, seed=2, dense_every=5, empty_every=6)
    plan = fa.Plan(cu, H, mode=fa.MODE_FP8)
    d = buf.cuda()
    ref = torch.empty((T, H, 128), dtype=torch.bfloat16, device="cuda")
    plan.quantize(d[:, 0], d[:, 1], d[:, 2])
    plan.forward_sparse(torch.from_numpy(off).cuda(), torch.from_numpy(idx).cuda(), ref)
    torch.cuda.synchronize()
    ref = ref.cpu()
    out = torch.full((T, H, 128), 5.0, dtype=torch.bfloat16).pin_memory()
    plan.attention_sparse_host(buf[:, 0], buf[:, 1], buf[:, 2], torch.from_numpy(off),
                               torch.from_numpy(idx), out, heads_per_chunk=hpc)
    torch.cuda.synchronize()
    assert plan.last_error() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
