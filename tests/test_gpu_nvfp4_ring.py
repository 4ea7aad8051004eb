"""NVFP4 forward with the qm K^T table held as a ring of two head-group slots (FlashInfer docs,
minimax_h3_sm120_varlen_attention_nvfp4, description: the qm K^T term added back to the
scores). The ring changes where and when the table is built, not a single value: outputs and LSE
must equal those of the whole-table plan bit for bit, and match the NVFP4-emulating oracle."""
import numpy as np
import pytest
import torch

import oracle
from precision_attention_diffusion_gb300 import inputs
from parity import SCALE, all_rows, bits, rel_rms

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from precision_attention_diffusion_gb300 import build, fa_lp
    build.build()
    fa_lp.load()
    return fa_lp


def with_k_offset(k, H, seed):
    off = inputs.k_channel_offset(H, seed=seed)
    return (k.float() + off[None]).to(torch.bfloat16)


def head_table_bytes(cu):
    return sum(((b - a + 127) // 128) ** 2 for a, b in zip(cu[:-1], cu[1:])) * 128 * 4


def run(fa, plan, q, k, v, T, H, stream=None):
    out = torch.full((T, H, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H, T), 7.0, dtype=torch.float32, device="cuda")
    plan.quantize(q, k, v, stream=stream)
    plan.forward(out, lse=lse, stream=stream)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("per_slot", [1, 2])
def test_ring_equals_whole_table_ragged(fa, per_slot):
    """Five heads over empty, 17-token and ragged segments; slots of one head (5 groups) and of two
    (groups of 2, 2, 1)."""
    cu, H = [0, 0, 17, 300, 300, 1400, 1500], 5
    T = cu[-1]
    q, k, v = inputs.qkv_separate(T, H, seed=21)
    k = with_k_offset(k, H, 21)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    plan = fa.Plan(cu, H, mode=fa.MODE_NVFP4)
    try:
        plan.set_table_limit(0)
        assert plan.table_layout()["slots"] == 1
        ref_out, ref_lse = run(fa, plan, q, k, v, T, H)
        plan.set_table_limit(2 * per_slot * head_table_bytes(cu))
        lay = plan.table_layout()
        assert lay["slots"] == 2 and lay["heads_per_slot"] == per_slot
        for _ in range(2):  # the table is rebuilt by every forward
            out, lse = run(fa, plan, q, k, v, T, H)
            assert torch.equal(out, ref_out)
            assert torch.equal(lse, ref_lse)
        assert plan.last_error() == 0
        with pytest.raises(fa.FaLpError):
            plan.quantized(fa.QMK_TABLE)
    finally:
        plan.set_table_limit(0)
    z = oracle.nvfp4_quantize(bits(q.cpu()), bits(k.cpu()), bits(v.cpu()), cu)
    rows = all_rows(cu, H)
    emu = oracle.attn_nvfp4(z, cu, rows, SCALE, n_kv=64)[0]
    got = np.stack([out[t, h].float().cpu().numpy() for t, h in rows])
    assert rel_rms(got, emu) < 1e-2


def test_ring_on_a_side_stream(fa):
    """The ring's internal streams start after the caller's stream and the caller's stream waits
    for them: a forward issued on a side stream, followed there by a copy of the output, sees the
    finished output."""
    cu, H = [0, 900, 2000], 3
    T = cu[-1]
    q, k, v = inputs.qkv_separate(T, H, seed=22)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    plan = fa.Plan(cu, H, mode=fa.MODE_NVFP4)
    try:
        ref_out, _ = run(fa, plan, q, k, v, T, H)
        plan.set_table_limit(2 * head_table_bytes(cu))
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            out = torch.empty((T, H, 128), dtype=torch.bfloat16, device="cuda")
            plan.quantize(q, k, v, stream=s)
            plan.forward(out, stream=s)
            copy = out.clone()
        torch.cuda.synchronize()
        assert torch.equal(copy, ref_out)
    finally:
        plan.set_table_limit(0)


def test_ring_equals_whole_table_h3_shape(fa):
    """S=30272, H=56 (K offset N(0, 4)): a 64 MB limit (one 29 MB head per slot, 56 groups) and a
    workspace under 0.5 GB; every output and LSE value equals the whole-table run's."""
    S, H = 30272, 56
    cu = [0, S]
    q, k, v = inputs.qkv_separate(S, H, seed=0)
    k = with_k_offset(k, H, 0)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    plan = fa.Plan(cu, H, mode=fa.MODE_NVFP4)
    try:
        ref_out, ref_lse = run(fa, plan, q, k, v, S, H)
        plan.set_table_limit(64 << 20)
        assert plan.table_layout()["heads_per_slot"] == 1
        assert plan.info()["workspace_bytes"] < 500_000_000
        out, lse = run(fa, plan, q, k, v, S, H)
        assert torch.equal(out, ref_out)
        assert torch.equal(lse, ref_lse)
        assert plan.last_error() == 0
    finally:
        plan.set_table_limit(0)


def test_ring_device_wait_limit_returns_error_not_hang(fa):
    """A wait limit of one probe in ring mode: the launches of the head groups on the two internal
    streams report the expiry through the plan's error word (0x100 | role), nothing hangs, and a
    correct ring run follows on the same plan."""
    cu, H = [0, 640], 3
    q, k, v = inputs.qkv_separate(640, H, seed=23)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    plan = fa.Plan(cu, H, mode=fa.MODE_NVFP4)
    try:
        ref_out, ref_lse = run(fa, plan, q, k, v, 640, H)
        plan.set_table_limit(2 * head_table_bytes(cu))
        assert plan.table_layout()["slots"] == 2
        plan.last_error()  # clear
        plan.set_wait_limit(1)
        run(fa, plan, q, k, v, 640, H)
        status = plan.last_error()
        assert status != 0 and (status & 0xFF00) == 0x100
        plan.set_wait_limit(20000)
        out, lse = run(fa, plan, q, k, v, 640, H)
        assert plan.last_error() == 0
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    finally:
        plan.set_wait_limit(20000)
        plan.set_table_limit(0)
