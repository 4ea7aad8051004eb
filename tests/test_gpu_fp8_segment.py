"""The per-segment FP8 mode (FA_LP_MODE_FP8_SEGMENT: one scale per (segment, tensor, head), the
alternative of reading r1 for packed batches; SGLang PR #40175, Modifications, fused_prep.py takes
one amax per head) on the GPU through the C ABI, against the oracle's per-segment quantization.

Bar as for the FP8 mode: codes and descales bit-exact, output within relative RMS 1e-2 of the
FP8-emulating oracle (per-segment descales) and 0.06 of exact attention, worst row 5e-2."""
import numpy as np
import pytest
import torch

import oracle
from precision_attention_diffusion_gb300 import inputs
from parity import SCALE, all_rows, bits, out_rows, padded_rows, rel_rms

pytestmark = pytest.mark.gpu

TOL_EMU, TOL_EXACT, TOL_ROW = 1e-2, 0.06, 5e-2
KV_TILE, TAU = 64, 8.0


@pytest.fixture(scope="module")
def fa():
    from precision_attention_diffusion_gb300 import build, fa_lp
    build.build()
    fa_lp.load()
    return fa_lp


def scaled_segments(cu, H, seed, factors):
    """Gaussian Q/K/V whose segment s has Q and V multiplied and K divided by factors[s]: the
    segments' amax lie far apart while every segment's scores (and so its attention pattern) stay
    those of unit Gaussians."""
    q, k, v = inputs.qkv_separate(cu[-1], H, seed=seed)
    f = torch.ones(cu[-1], 1, 1)
    for s, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        f[a:b] = factors[s]
    return tuple((x.float() * g).to(torch.bfloat16) for x, g in ((q, f), (k, 1.0 / f), (v, f)))


def run(fa, q, k, v, cu, H, out=None):
    plan = fa.Plan(cu, H, mode=fa.MODE_FP8_SEGMENT)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    plan.attention(q.cuda(), k.cuda(), v.cuda(), torch.tensor(cu, dtype=torch.int32,
                                                              device="cuda"), out=out)
    torch.cuda.synchronize()
    return plan, out


def check_codes(fa, plan, cu, q, k, v):
    rows, pad = padded_rows(cu, plan.row_offsets())
    qc = plan.quantized(fa.Q_CODES).cpu().numpy()
    kc = plan.quantized(fa.K_CODES).cpu().numpy()
    vt = plan.quantized(fa.V_CODES).cpu().numpy()
    ds = plan.quantized(fa.DESCALE).cpu().numpy()          # [3][nseg][H]
    assert ds.shape == (3, len(cu) - 1, q.shape[1])
    nat = dict(q=qc[:, rows].transpose(1, 0, 2), k=kc[:, rows].transpose(1, 0, 2),
               v=vt[:, :, rows].transpose(2, 0, 1))
    for i, (name, x) in enumerate((("q", q), ("k", k), ("v", v))):
        codes, d = oracle.fp8_quantize_seg(bits(x), cu)
        assert np.array_equal(nat[name], codes), f"{name} codes differ"
        assert np.array_equal(ds[i], d), f"{name} descales differ"
    assert np.all(qc[:, pad] == 0) and np.all(kc[:, pad] == 0) and np.all(vt[:, :, pad] == 0)
    return nat, ds


def check_outputs(out, q, k, v, nat, ds, cu, rows):
    got = out_rows(out, rows)
    emu, _ = oracle.attn_fp8(nat["q"], nat["k"], nat["v"], ds[0], ds[1], ds[2], cu, rows, SCALE,
                             n_kv=KV_TILE, tau=TAU)
    exact = oracle.attn_exact(bits(q), bits(k), bits(v), cu, rows, SCALE)
    per_row = np.linalg.norm(got - emu, axis=1) / np.maximum(np.linalg.norm(emu, axis=1), 1e-30)
    assert rel_rms(got, emu) <= TOL_EMU, rel_rms(got, emu)
    assert rel_rms(got, exact) <= TOL_EXACT, rel_rms(got, exact)
    assert per_row.max() <= TOL_ROW, per_row.max()


def test_fp8_segment_ragged_full_parity(fa):
    """Empty segments, a 17-row segment and ragged tiles; segment amax 1e4 apart; every row."""
    cu, H = [0, 0, 17, 300, 300, 1400, 1500], 3
    q, k, v = scaled_segments(cu, H, 71, [1.0, 0.01, 1.0, 1.0, 100.0, 0.5])
    plan, out = run(fa, q, k, v, cu, H)
    nat, ds = check_codes(fa, plan, cu, q, k, v)
    check_outputs(out, q, k, v, nat, ds, cu, all_rows(cu, H))
    # block-sparse forward on the same per-segment operands: full lists give the dense bits
    off, idx = inputs.block_sparse_lists(cu, H, density=1.0, seed=0, dense_every=1)
    outs = torch.empty_like(out)
    plan.forward_sparse(torch.from_numpy(off).cuda(), torch.from_numpy(idx).cuda(), outs)
    torch.cuda.synchronize()
    assert plan.last_error() == 0
    assert torch.equal(outs, out)


def test_fp8_segment_packed_varlen_32768(fa):
    """The packed varlen configuration (cu = [0, 0, 17, 4113, 4113, 31800, 32768], H = 56) with
    segment scales 1000x apart: codes and descales bit-exact; the 17- and 968-row segments in
    full, sampled rows of the rest."""
    cu, H = [0, 0, 17, 4113, 4113, 31800, 32768], 56
    q, k, v = scaled_segments(cu, H, 0, [1.0, 0.01, 3.0, 1.0, 1.0, 0.003])
    sentinel = torch.full((32768, H, 256), 3.0, dtype=torch.bfloat16, device="cuda")
    out = sentinel[:, :, :128]
    plan, _ = run(fa, q, k, v, cu, H, out=out)
    assert torch.all(sentinel[:, :, 128:] == 3.0)
    nat, ds = check_codes(fa, plan, cu, q, k, v)
    full = [(t, h) for t in list(range(0, 17)) + list(range(31800, 32768)) for h in range(H)]
    check_outputs(out, q, k, v, nat, ds, cu, full)
    check_outputs(out, q, k, v, nat, ds, cu, inputs.sample_rows(cu, H, n_heads=4, n_rows=256,
                                                                seed=1))


def test_fp8_segment_host_entry_equals_device_call(fa):
    """fa_lp_attention_host on a per-segment plan returns the device call's bits (every step is
    per head, and the per-segment scales too)."""
    cu, H = [0, 100, 700, 777], 6
    q, k, v = scaled_segments(cu, H, 5, [0.02, 1.0, 10.0])
    plan, out = run(fa, q, k, v, cu, H)
    hbuf = torch.stack([q, k, v], dim=1).pin_memory()
    hout = torch.empty((cu[-1], H, 128), dtype=torch.bfloat16).pin_memory()
    plan.attention_host(hbuf[:, 0], hbuf[:, 1], hbuf[:, 2], hout, heads_per_chunk=4)
    torch.cuda.synchronize()
    assert torch.equal(hout, out.cpu())


def test_fp8_segment_lse(fa):
    """Row log-sum-exp on a per-segment plan: within the f16 row-sum bound (2.5e-3, as for the
    FP8 mode) of the emulating oracle run with the per-segment descales."""
    cu, H = [0, 0, 17, 300, 300, 1400, 1500], 3
    T = cu[-1]
    q, k, v = scaled_segments(cu, H, 73, [1.0, 0.02, 4.0, 1.0, 0.25, 30.0])
    plan = fa.Plan(cu, H, mode=fa.MODE_FP8_SEGMENT)
    plan.quantize(q.cuda(), k.cuda(), v.cuda())
    out = torch.empty(T, H, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H, T), 7.0, dtype=torch.float32, device="cuda")
    plan.forward(out, lse=lse)
    torch.cuda.synchronize()
    nat, ds = check_codes(fa, plan, cu, q, k, v)
    rows = all_rows(cu, H)
    _, _, emu = oracle.attn_fp8(nat["q"], nat["k"], nat["v"], ds[0], ds[1], ds[2], cu, rows,
                                SCALE, n_kv=KV_TILE, tau=TAU, lse=True)
    g = lse.cpu().numpy()
    got = np.array([g[h, t] for t, h in rows], np.float64)
    assert np.abs(got - emu).max() < 2.5e-3, np.abs(got - emu).max()
