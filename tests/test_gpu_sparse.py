"""Block-sparse FP8 forward on the GPU through the C ABI, against the oracle.

Semantics (reading r16; SGLang PR #40116, Modifications and Accuracy Tests): 64-row query blocks
x 64-key blocks counted from each segment start, the last ones partial; a row attends to the keys
of its block's list; a row with an empty list is 0. The kernel takes the listed blocks in list
order as its online-softmax tiles with the dense path's rule (reference maximum moving by more
than 8 in log2 units), which the emulating oracle replays.

Bar: as the dense FP8 path -- relative RMS <= 1e-2 against the FP8-emulating oracle, <= 0.06
against FP64 exact sparse attention, worst row <= 5e-2; rows with empty lists exactly 0 with LSE
-inf; with every block listed, the output equals the dense forward's bit for bit (same tiles,
same arithmetic).
"""
import numpy as np
import pytest
import torch

import oracle
from precision_attention_diffusion_gb300 import inputs
from parity import SCALE, all_rows, bits, out_rows, rel_rms
from test_gpu_fp8 import TAU, TOL_LSE, check_codes, gpu_codes_natural

pytestmark = pytest.mark.gpu

TOL_EMU, TOL_EXACT, TOL_ROW = 1e-2, 0.06, 5e-2
B = 64


@pytest.fixture(scope="module")
def fa():
    from precision_attention_diffusion_gb300 import build, fa_lp
    build.build()
    fa_lp.load()
    return fa_lp


def full_lists(cu, H):
    lens = [b - a for a, b in zip(cu[:-1], cu[1:])]
    flat = [np.arange((L + B - 1) // B) for _ in range(H) for L in lens
            for _ in range((L + B - 1) // B)]
    off = np.zeros(len(flat) + 1, np.int32)
    off[1:] = np.cumsum([len(x) for x in flat])
    return off, np.concatenate(flat).astype(np.int32)


def lists_from(per_block, H):
    """per_block: list over h * G + g of index lists -> (offsets, indices)."""
    off = np.zeros(len(per_block) + 1, np.int32)
    off[1:] = np.cumsum([len(x) for x in per_block])
    idx = np.concatenate([np.asarray(x, np.int64) for x in per_block]) if per_block else []
    return off, np.asarray(idx, np.int32)


def run_sparse(fa, q, k, v, cu, H, off, idx, lse=False):
    plan = fa.Plan(cu, H, mode=fa.MODE_FP8)
    plan.quantize(q.cuda(), k.cuda(), v.cuda())
    out = torch.full(q.shape, 7.0, dtype=torch.bfloat16, device="cuda")
    lse_t = torch.full((H, cu[-1]), 3.0, dtype=torch.float32, device="cuda") if lse else None
    d_off = torch.from_numpy(np.asarray(off, np.int32)).cuda()
    d_idx = torch.from_numpy(np.asarray(idx, np.int32).reshape(-1)).cuda()
    if d_idx.numel() == 0:
        d_idx = torch.zeros(1, dtype=torch.int32, device="cuda")[:0]
    plan.forward_sparse(d_off, d_idx, out, lse=lse_t)
    torch.cuda.synchronize()
    assert plan.last_error() == 0
    return plan, out, lse_t


def check_sparse(fa, plan, out, q, k, v, cu, H, off, idx, rows, lse_t=None):
    nat, ds = check_codes(fa, plan, cu, q, k, v)
    got = out_rows(out, rows)
    emu, _, emu_lse = oracle.attn_fp8_sparse(nat["q"], nat["k"], nat["v"], ds[0], ds[1], ds[2],
                                             cu, off, idx, rows, SCALE, tau=TAU, lse=True)
    exact = oracle.attn_exact_sparse(bits(q), bits(k), bits(v), cu, off, idx, rows, SCALE)
    empty = np.all(emu == 0.0, axis=1)
    assert np.all(got[empty] == 0.0), "rows with an empty list must be 0"
    live = ~empty
    assert live.any()
    g, e, x = got[live], emu[live], exact[live]
    assert rel_rms(g, e) <= TOL_EMU, rel_rms(g, e)
    assert rel_rms(g, x) <= TOL_EXACT, rel_rms(g, x)
    per_row = np.linalg.norm(g - e, axis=1) / np.maximum(np.linalg.norm(e, axis=1), 1e-30)
    assert per_row.max() <= TOL_ROW, per_row.max()
    if lse_t is not None:
        r = np.asarray(rows, np.int64).reshape(-1, 2)
        lg = lse_t.cpu().numpy()[r[:, 1], r[:, 0]].astype(np.float64)
        assert np.all(np.isneginf(lg[empty]))
        assert np.max(np.abs(lg[live] - emu_lse[live])) <= TOL_LSE
    return empty


def test_sparse_full_lists_equal_dense_forward(fa):
    cu, H = [0, 0, 17, 300, 300, 1400, 1500], 3
    q, k, v = inputs.qkv_separate(cu[-1], H, seed=2)
    off, idx = full_lists(cu, H)
    plan, out, lse = run_sparse(fa, q, k, v, cu, H, off, idx, lse=True)
    dense = torch.empty_like(out)
    dlse = torch.empty_like(lse)
    plan.forward(dense, lse=dlse)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), dense.view(torch.int16))
    assert torch.equal(lse, dlse)


def test_sparse_ragged_varlen_all_rows(fa):
    """Partial query and key blocks, empty and one-token segments, variable list lengths, dense
    and empty lists mixed in; every row against the oracle."""
    cu, H = [0, 0, 17, 300, 300, 1400, 1401, 1500], 3
    q, k, v = inputs.qkv_separate(cu[-1], H, seed=5)
    off, idx = inputs.block_sparse_lists(cu, H, density=0.4, seed=6, dense_every=5,
                                         empty_every=7)
    plan, out, lse = run_sparse(fa, q, k, v, cu, H, off, idx, lse=True)
    empty = check_sparse(fa, plan, out, q, k, v, cu, H, off, idx, all_rows(cu, H), lse)
    assert empty.any()


def test_sparse_halves_of_a_tile_differ(fa):
    """The two 64-row halves of each 128-row tile list different blocks (one lists none)."""
    cu, H = [0, 320], 1
    q, k, v = inputs.qkv_separate(320, H, seed=8)
    per_block = [[0], [3], [], [1, 2, 4], [4]]
    off, idx = lists_from(per_block, H)
    plan, out, lse = run_sparse(fa, q, k, v, cu, H, off, idx, lse=True)
    empty = check_sparse(fa, plan, out, q, k, v, cu, H, off, idx, all_rows(cu, H), lse)
    assert empty.sum() == 64


@pytest.mark.parametrize("cu,H,density,dense_every,empty_every", [
    ([0, 192], 1, 0.5, 0, 2),            # a tile holding one full 64-row block only
    ([0, 64, 128, 129, 257], 2, 1.0, 0, 0),  # long lists (half to all blocks), short segments
    ([0, 0, 17, 4113, 4113, 5200], 4, 0.2, 3, 4),  # the varlen layout's empty / short segments
])
def test_sparse_shapes(fa, cu, H, density, dense_every, empty_every):
    q, k, v = inputs.qkv_separate(cu[-1], H, seed=10 + H)
    off, idx = inputs.block_sparse_lists(cu, H, density=density, seed=H, dense_every=dense_every,
                                         empty_every=empty_every)
    plan, out, lse = run_sparse(fa, q, k, v, cu, H, off, idx, lse=True)
    rows = all_rows(cu, H) if cu[-1] * H <= 3000 else inputs.sample_rows(cu, H, H, 512, seed=3)
    check_sparse(fa, plan, out, q, k, v, cu, H, off, idx, rows, lse)


def test_sparse_list_breaking_the_contract_is_reported(fa):
    """A descending list is caught by the device-side check: status 0x200, INVALID_ARG, no
    access outside the arrays; the next valid call is clean."""
    cu, H = [0, 256], 1
    q, k, v = inputs.qkv_separate(256, H, seed=9)
    off, idx = lists_from([[2, 1], [0], [0, 1, 2, 3], [3]], H)
    plan = fa.Plan(cu, H, mode=fa.MODE_FP8)
    plan.quantize(q.cuda(), k.cuda(), v.cuda())
    out = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    plan.forward_sparse(torch.from_numpy(off).cuda(), torch.from_numpy(idx).cuda(), out)
    torch.cuda.synchronize()
    assert plan.last_error() == 0x200
    off, idx = lists_from([[1, 2], [0], [0, 1, 2, 3], [3]], H)
    plan.forward_sparse(torch.from_numpy(off).cuda(), torch.from_numpy(idx).cuda(), out)
    torch.cuda.synchronize()
    assert plan.last_error() == 0


def test_sparse_deterministic_and_wait_limit(fa):
    """Repeated calls give the same bits (the tiles are ordered on the device, ties in any order,
    but every tile is computed on its own); a wait limit of one probe makes the block-sparse
    kernel record an expired wait and return, and the next call with the normal limit is clean
    and correct."""
    cu, H = [0, 17, 700], 2
    q, k, v = inputs.qkv_separate(cu[-1], H, seed=12)
    off, idx = inputs.block_sparse_lists(cu, H, density=0.5, seed=3, empty_every=4)
    plan, out, _ = run_sparse(fa, q, k, v, cu, H, off, idx)
    d_off, d_idx = torch.from_numpy(off).cuda(), torch.from_numpy(idx).cuda()
    again = torch.empty_like(out)
    plan.forward_sparse(d_off, d_idx, again)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    plan.set_wait_limit(1)
    plan.forward_sparse(d_off, d_idx, again)
    torch.cuda.synchronize()
    status = plan.last_error()
    assert status != 0 and (status & 0xFF00) == 0x100
    plan.set_wait_limit(20000)
    plan.forward_sparse(d_off, d_idx, again)
    torch.cuda.synchronize()
    assert plan.last_error() == 0
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


@pytest.mark.parametrize("cu", [[0, 30272], [0, 0, 17, 4113, 4113, 31800, 32768]])
def test_sparse_h3_sampled(fa, cu):
    """H=56, a quarter of the key blocks listed per query block (the pages' sparsity 0.75), every
    16th list dense: the bench's launch at S=30272, and the packed varlen layout with empty, short
    and trailing segments; sampled rows against the oracle."""
    H = 56
    q, k, v = inputs.qkv_separate(cu[-1], H, seed=0)
    off, idx = inputs.block_sparse_lists(cu, H, density=0.25, seed=0, dense_every=16)
    plan, out, _ = run_sparse(fa, q, k, v, cu, H, off, idx)
    rows = inputs.sample_rows(cu, H, n_heads=4, n_rows=64, seed=1)
    check_sparse(fa, plan, out, q, k, v, cu, H, off, idx, rows)


def test_sparse_many_small_segments(fa):
    """300 segments of 0 to 200 tokens (seeded), H=2, variable lists with dense and empty ones:
    every row against the oracle."""
    g = np.random.default_rng(33)
    lens = g.integers(0, 201, 300)
    lens[g.integers(0, 300, 40)] = 0
    cu = [0] + np.cumsum(lens).tolist()
    H = 2
    q, k, v = inputs.qkv_separate(cu[-1], H, seed=33)
    off, idx = inputs.block_sparse_lists(cu, H, density=0.5, seed=33, dense_every=5,
                                         empty_every=7)
    plan, out, lse = run_sparse(fa, q, k, v, cu, H, off, idx, lse=True)
    check_sparse(fa, plan, out, q, k, v, cu, H, off, idx, all_rows(cu, H), lse)
