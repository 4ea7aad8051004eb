"""FP8 E4M3 path on the GPU through the C ABI, against the oracle.

Bar: quantized codes and descales bit-exact; output within relative RMS 1e-2 of the
FP8-emulating oracle (C2, replaying the kernel's 64-key tiles and reference-max rule) and within
0.06 of FP64 exact attention (C1) on Gaussian inputs. Per row, the error is also bounded
(relative RMS of any one row <= 5e-2 of C2) so that a single wrong row cannot hide in the mean.
"""
import numpy as np
import pytest
import torch

import oracle
from precision_attention_diffusion_gb300 import inputs
from parity import SCALE, all_rows, bits, out_rows, padded_rows, rel_rms

pytestmark = pytest.mark.gpu

TOL_EMU = 1e-2      # relative RMS against the FP8-emulating oracle
TOL_EXACT = 0.06    # relative RMS against FP64 exact attention (pages: 0.0535-0.0539)
TOL_ROW = 5e-2      # worst single row against the emulating oracle
# Row LSE against the emulating oracle's m + log(l): the kernel sums a thread's 32 quantized P in
# f16 pairs (one add per key pair, then a three-level tree, so a value passes through four f16
# additions, each rounding by at most 2^-11 of its result); P spans 2^-9 .. 2^8 under the lazy
# maximum, so those sums are not exact, and l carries a relative error of at most 4 x 2^-11 =
# 1.95e-3 (the log of l the same in absolute terms); 2.5e-3 leaves room for ex2.approx.
TOL_LSE = 2.5e-3


@pytest.fixture(scope="module")
def fa():
    from precision_attention_diffusion_gb300 import build, fa_lp
    build.build()
    fa_lp.load()
    return fa_lp


def run_fp8(fa, q, k, v, cu, heads, out=None):
    plan = fa.Plan(cu, heads, mode=fa.MODE_FP8)
    dq, dk, dv = q.cuda() if not q.is_cuda else q, k.cuda() if not k.is_cuda else k, v.cuda() if not v.is_cuda else v
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    cu_dev = torch.tensor(cu, dtype=torch.int32, device="cuda")
    plan.attention(dq, dk, dv, cu_dev, out=out)
    torch.cuda.synchronize()
    return plan, out


def gpu_codes_natural(fa, plan, cu):
    """Map the plan's workspace arrays back to natural [T, H, 128] order; also the padding."""
    rows, pad = padded_rows(cu, plan.row_offsets())
    qc = plan.quantized(fa.Q_CODES).cpu().numpy()      # [H][Tp][128]
    kc = plan.quantized(fa.K_CODES).cpu().numpy()
    vt = plan.quantized(fa.V_CODES).cpu().numpy()      # [H][128][Tp]
    ds = plan.quantized(fa.DESCALE).cpu().numpy()[0]   # [3][H]
    nat = dict(q=qc[:, rows].transpose(1, 0, 2), k=kc[:, rows].transpose(1, 0, 2),
               v=vt[:, :, rows].transpose(2, 0, 1))
    pads = dict(q=qc[:, pad], k=kc[:, pad], v=vt[:, :, pad])
    return nat, pads, ds


def check_codes(fa, plan, cu, q, k, v):
    nat, pads, ds = gpu_codes_natural(fa, plan, cu)
    for i, (name, x) in enumerate((("q", q), ("k", k), ("v", v))):
        codes, d = oracle.fp8_quantize(bits(x))
        assert np.array_equal(nat[name], codes), f"{name} codes differ"
        assert np.array_equal(ds[i], d), f"{name} descales differ"
        assert np.all(pads[name] == 0), f"{name} padding not zero"
    return nat, ds


# The kernel's online-softmax rule, as documented for fa_lp_forward_varlen in include/fa_lp.h:
# 64-key tiles from each segment start; the reference maximum moves only by more than 8 (log2).
KV_TILE, TAU = 64, 8.0


def oracle_fp8(nat, ds, cu, rows):
    return oracle.attn_fp8(nat["q"], nat["k"], nat["v"], ds[0], ds[1], ds[2], cu, rows, SCALE,
                           n_kv=KV_TILE, tau=TAU)


def check_outputs(out, q, k, v, nat, ds, cu, rows):
    got = out_rows(out, rows)
    emu, _ = oracle_fp8(nat, ds, cu, rows)
    exact = oracle.attn_exact(bits(q), bits(k), bits(v), cu, rows, SCALE)
    e_emu, e_exact = rel_rms(got, emu), rel_rms(got, exact)
    per_row = np.linalg.norm(got - emu, axis=1) / np.maximum(np.linalg.norm(emu, axis=1), 1e-30)
    assert e_emu <= TOL_EMU, e_emu
    assert e_exact <= TOL_EXACT, e_exact
    assert per_row.max() <= TOL_ROW, per_row.max()
    return e_emu, e_exact


# ------------------------------------------------------------------------------------------------
def test_hw_e4m3_conversion_matches_definition(fa):
    x = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    x = x[np.isfinite(x)]
    got = fa.encode(0, torch.from_numpy(x).cuda()).cpu().numpy()
    assert np.array_equal(got, oracle.e4m3_encode(x))


def test_hw_e2m1_conversion_matches_definition(fa):
    x = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    x = x[np.isfinite(x)]
    got = fa.encode(1, torch.from_numpy(x).cuda()).cpu().numpy()
    assert np.array_equal(got, oracle.e2m1_encode(x))


def test_fp8_small_full_parity(fa):
    """One segment S=256, H=2, seed 0: every row against the oracle."""
    cu, H = [0, 256], 2
    q, k, v = inputs.qkv_separate(256, H, seed=0)
    plan, out = run_fp8(fa, q, k, v, cu, H)
    nat, ds = check_codes(fa, plan, cu, q, k, v)
    check_outputs(out, q, k, v, nat, ds, cu, all_rows(cu, H))


def test_fp8_ragged_varlen_full_parity(fa):
    """Empty segments, a 17-row segment, ragged tails of key and query tiles; all rows."""
    cu, H = [0, 0, 17, 300, 300, 1400, 1500], 3
    q, k, v = inputs.qkv_separate(1500, H, seed=2)
    plan, out = run_fp8(fa, q, k, v, cu, H)
    nat, ds = check_codes(fa, plan, cu, q, k, v)
    check_outputs(out, q, k, v, nat, ds, cu, all_rows(cu, H))


def test_fp8_single_row_segments(fa):
    cu, H = [0, 1, 2, 130, 131], 2
    q, k, v = inputs.qkv_separate(131, H, seed=3)
    plan, out = run_fp8(fa, q, k, v, cu, H)
    nat, ds = check_codes(fa, plan, cu, q, k, v)
    check_outputs(out, q, k, v, nat, ds, cu, all_rows(cu, H))
    # a one-token segment returns its own dequantized v row
    o = out.float().cpu().numpy()
    dec = oracle.e4m3_decode_table()
    for t in (0, 1, 130):
        for h in range(H):
            want = torch.tensor(dec[nat["v"][t, h]] * np.float64(ds[2][h])).to(torch.bfloat16).float().numpy()
            assert np.array_equal(o[t, h], want)


def test_fp8_strided_out_leaves_other_bytes_untouched(fa):
    cu, H = [0, 77, 333], 2
    q, k, v = inputs.qkv_separate(333, H, seed=4)
    big = torch.full((333, H, 256), -7.0, dtype=torch.bfloat16, device="cuda")
    out = big[:, :, :128]
    plan, _ = run_fp8(fa, q, k, v, cu, H, out=out)
    assert torch.all(big[:, :, 128:] == -7.0)
    nat, ds = check_codes(fa, plan, cu, q, k, v)
    check_outputs(out, q, k, v, nat, ds, cu, all_rows(cu, H))


def test_fp8_constant_v_returns_v(fa):
    cu, H = [0, 1000], 2
    q, k, _ = inputs.qkv_separate(1000, H, seed=5)
    v = torch.full((1000, H, 128), 0.8125, dtype=torch.bfloat16)
    _, out = run_fp8(fa, q, k, v, cu, H)
    assert torch.all(out.cpu() == v)


def test_fp8_deterministic(fa):
    cu, H = [0, 700], 4
    q, k, v = inputs.qkv_separate(700, H, seed=6)
    _, o1 = run_fp8(fa, q, k, v, cu, H)
    o1 = o1.clone()
    _, o2 = run_fp8(fa, q, k, v, cu, H)
    assert torch.equal(o1, o2)


def test_fp8_scrambled_keys_negative_control(fa):
    """The comparator must fail when the keys are permuted (guards against a vacuous check)."""
    cu, H = [0, 512], 2
    q, k, v = inputs.qkv_separate(512, H, seed=7)
    _, out = run_fp8(fa, q, k, v, cu, H)
    rows = all_rows(cu, H)
    perm = torch.randperm(512, generator=torch.Generator().manual_seed(1))
    kp = k[perm].contiguous()
    (cq, dq), (ck, dk), (cv, dv) = (oracle.fp8_quantize(bits(x)) for x in (q, kp, v))
    wrong, _ = oracle.attn_fp8(cq, ck, cv, dq, dk, dv, cu, rows, SCALE, n_kv=KV_TILE, tau=TAU)
    assert rel_rms(out_rows(out, rows), wrong) > 0.3


def test_device_wait_limit_returns_error_not_hang(fa):
    """A wait limit of one probe expires on the first wait that is not already complete: the
    kernel must record an error and return; the context stays usable."""
    cu, H = [0, 640], 2
    q, k, v = inputs.qkv_separate(640, H, seed=8)
    plan = fa.Plan(cu, H)
    plan.last_error()  # clear
    plan.set_wait_limit(1)
    out = torch.zeros(640, H, 128, dtype=torch.bfloat16, device="cuda")
    plan.attention(q.cuda(), k.cuda(), v.cuda(), out=out)
    torch.cuda.synchronize()
    status = plan.last_error()
    assert status != 0 and (status & 0xFF00) == 0x100
    plan.set_wait_limit(20000)
    plan.attention(q.cuda(), k.cuda(), v.cuda(), out=out)
    torch.cuda.synchronize()
    assert plan.last_error() == 0
    nat, ds = check_codes(fa, plan, cu, q, k, v)
    check_outputs(out, q, k, v, nat, ds, cu, all_rows(cu, H))


def test_padding_bytes_are_rewritten(fa):
    """Fill the workspace with non-zero codes through a plan whose single segment covers the whole
    padded axis, then quantize a ragged plan over the same bytes: every padding byte must be 0
    (SGLang PR #40175 review: the pack pass writes every padding position)."""
    cu, H = [0, 5, 200, 333], 2
    plan = fa.Plan(cu, H)
    tp = plan.info()["padded_tokens"]
    fill = torch.full((tp, H, 128), -300.0, dtype=torch.bfloat16)
    run_fp8(fa, fill, fill, fill, [0, tp], H)
    q, k, v = inputs.qkv_separate(333, H, seed=9)
    plan, out = run_fp8(fa, q, k, v, cu, H)
    check_codes(fa, plan, cu, q, k, v)


# ------------------------------------------------------------------------------------------------
# Full-size configurations, in the launch configuration the benchmark times: codes bit-exact for
# every head, outputs on a seeded sample of rows the oracle computes one by one.
# ------------------------------------------------------------------------------------------------
def test_fp8_s4096_h56_sampled(fa):
    cu, H = [0, 4096], 56
    q, k, v = inputs.qkv_separate(4096, H, seed=0)
    plan, out = run_fp8(fa, q, k, v, cu, H)
    nat, ds = check_codes(fa, plan, cu, q, k, v)
    rows = inputs.sample_rows(cu, H, n_heads=4, n_rows=256, seed=1)
    check_outputs(out, q, k, v, nat, ds, cu, rows)


@pytest.mark.parametrize("S", [20440, 30272])
def test_fp8_h3_shape_strided_views_sampled(fa, S):
    H = 56
    buf, q, k, v = inputs.qkv_fused(S, H, seed=0)
    dbuf = buf.cuda()
    dq, dk, dv = dbuf[:, 0], dbuf[:, 1], dbuf[:, 2]
    cu = [0, S]
    plan, out = run_fp8(fa, dq, dk, dv, cu, H)
    nat, ds = check_codes(fa, plan, cu, q, k, v)
    rows = inputs.sample_rows(cu, H, n_heads=4, n_rows=256, seed=1)
    check_outputs(out, q, k, v, nat, ds, cu, rows)


def test_fp8_packed_varlen_32768(fa):
    cu, H = [0, 0, 17, 4113, 4113, 31800, 32768], 56
    q, k, v = inputs.qkv_separate(32768, H, seed=0)
    sentinel = torch.full((32768, H, 256), 3.0, dtype=torch.bfloat16, device="cuda")
    out = sentinel[:, :, :128]
    plan, _ = run_fp8(fa, q, k, v, cu, H, out=out)
    assert torch.all(sentinel[:, :, 128:] == 3.0)
    nat, ds = check_codes(fa, plan, cu, q, k, v)
    full = [(t, h) for t in list(range(0, 17)) + list(range(31800, 32768)) for h in range(H)]
    check_outputs(out, q, k, v, nat, ds, cu, full)
    rows = inputs.sample_rows(cu, H, n_heads=4, n_rows=256, seed=1)
    check_outputs(out, q, k, v, nat, ds, cu, rows)


def test_fp8_lse_ragged_varlen(fa):
    """Row log-sum-exp (fa_lp_forward_varlen_lse, reading r15) on empty, short and long segments:
    within TOL_LSE of the FP8-emulating oracle's m + log(l), within the E4M3 bound of exact
    attention's LSE; columns past the last token untouched."""
    cu, H = [0, 0, 17, 300, 300, 1400, 1500], 3
    T = cu[-1]
    q, k, v = inputs.qkv_separate(T, H, seed=12)
    plan = fa.Plan(cu, H)
    plan.quantize(q.cuda(), k.cuda(), v.cuda())
    out = torch.empty(T, H, 128, dtype=torch.bfloat16, device="cuda")
    lse_buf = torch.full((H, T + 5), 7.0, dtype=torch.float32, device="cuda")
    plan.forward(out, torch.tensor(cu, dtype=torch.int32, device="cuda"), lse=lse_buf)
    torch.cuda.synchronize()
    got = lse_buf.cpu().numpy()
    assert np.all(got[:, T:] == 7.0)
    rows = all_rows(cu, H)
    nat, ds = check_codes(fa, plan, cu, q, k, v)
    _, _, emu = oracle.attn_fp8(nat["q"], nat["k"], nat["v"], ds[0], ds[1], ds[2], cu, rows,
                                SCALE, n_kv=KV_TILE, tau=TAU, lse=True)
    _, exact = oracle.attn_exact(bits(q), bits(k), bits(v), cu, rows, SCALE, lse=True)
    g = np.array([got[h, t] for t, h in rows], np.float64)
    assert np.abs(g - emu).max() < TOL_LSE, np.abs(g - emu).max()
    # against exact attention: E4M3 rounding moves each P by at most 2^-4 (so log l by at most
    # ln(1 + 2^-4) = 0.061) plus the score quantization; short segments do not average it out
    d = np.abs(g - exact)
    assert d.max() < 0.1 and d.mean() < 0.02, (d.max(), d.mean())


def test_fp8_many_small_segments(fa):
    """300 segments of 0 to 200 tokens (seeded), H=2: hundreds of work items of one or two
    partial tiles, empty segments between them; every row against the oracle."""
    g = np.random.default_rng(31)
    lens = g.integers(0, 201, 300)
    lens[g.integers(0, 300, 40)] = 0
    cu = [0] + np.cumsum(lens).tolist()
    H = 2
    q, k, v = inputs.qkv_separate(cu[-1], H, seed=31)
    plan, out = run_fp8(fa, q, k, v, cu, H)
    nat, ds = check_codes(fa, plan, cu, q, k, v)
    check_outputs(out, q, k, v, nat, ds, cu, all_rows(cu, H))
