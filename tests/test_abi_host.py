"""C-ABI checks that need no GPU: the library builds for sm_103a and loads, it exports every
function include/fa_lp.h declares, and the host-only plan logic (cu_seqlens validation, padded
token axis, work list, workspace size) behaves as documented. No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_lp.h")


@pytest.fixture(scope="module")
def lib():
    from precision_attention_diffusion_gb300 import build, fa_lp
    build.build()
    return fa_lp.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^FA_LP_API\s+(?:int|const char\*)\s+(fa_lp_\w+)\s*\(", text, re.M)))


def test_header_declares_the_documented_calls():
    names = declared_functions()
    for must in ("fa_lp_plan_create", "fa_lp_quantize", "fa_lp_forward_varlen",
                 "fa_lp_attention", "fa_lp_plan_destroy", "fa_lp_workspace_bytes",
                 "fa_lp_get_last_error", "fa_lp_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    from precision_attention_diffusion_gb300 import fa_lp
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(fa_lp.EXPORTS)


def test_status_strings(lib):
    for s in range(7):
        assert lib.fa_lp_status_string(s)
    assert b"unknown" in lib.fa_lp_status_string(99)


def _create(lib, cu, heads=4, mode=0, scale=0.0, tokens=None):
    arr = (ctypes.c_int32 * len(cu))(*cu)
    h = ctypes.c_void_p()
    t = cu[-1] if tokens is None else tokens
    st = lib.fa_lp_plan_create(t, heads, arr, len(cu) - 1, scale, mode, 0, ctypes.byref(h))
    return st, h


@pytest.mark.parametrize("cu,tokens", [([1, 5], None), ([0, 5, 3], None), ([0, 5], 6),
                                       ([0, -1, 5], None)])
def test_plan_rejects_malformed_cu_seqlens(lib, cu, tokens):
    st, h = _create(lib, cu, tokens=tokens)
    assert st == 1 and not h.value


def test_plan_rejects_bad_heads_and_mode(lib):
    assert _create(lib, [0, 5], heads=0)[0] == 1
    assert _create(lib, [0, 5], mode=7)[0] == 1


def test_plan_padded_axis_and_work_list(lib):
    from precision_attention_diffusion_gb300 import fa_lp
    cu = [0, 0, 17, 4113, 4113, 31800, 32768]
    st, h = _create(lib, cu, heads=56)
    assert st == 0
    try:
        tp, wi, ws = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_size_t()
        assert lib.fa_lp_plan_info(h, ctypes.byref(tp), ctypes.byref(wi), ctypes.byref(ws)) == 0
        lens = [b - a for a, b in zip(cu[:-1], cu[1:])]
        blocks = [(L + 127) // 128 for L in lens]
        assert tp.value == 128 * sum(blocks)
        assert wi.value == 56 * sum((b + 1) // 2 for b in blocks)
        # FP8 workspace: Q, K codes [H][Tp][128], V^T [H][128][Tp], plus two [3][H] arrays
        assert ws.value >= 3 * 56 * 128 * tp.value
        offs = (ctypes.c_int64 * len(cu))()
        assert lib.fa_lp_plan_row_offsets(h, offs) == 0
        want, acc = [], 0
        for b in blocks:
            want.append(acc)
            acc += 128 * b
        want.append(acc)
        assert list(offs) == want
        assert all(o % 128 == 0 for o in offs)
    finally:
        assert lib.fa_lp_plan_destroy(h) == 0


def test_plan_cache_shares_identical_keys(lib):
    st1, h1 = _create(lib, [0, 100, 300], heads=2)
    st2, h2 = _create(lib, [0, 100, 300], heads=2)
    st3, h3 = _create(lib, [0, 100, 300], heads=3)
    try:
        assert st1 == st2 == st3 == 0
        assert h1.value == h2.value and h1.value != h3.value
    finally:
        for h in (h1, h2, h3):
            assert lib.fa_lp_plan_destroy(h) == 0


def test_calls_validate_before_touching_the_device(lib):
    st, h = _create(lib, [0, 64], heads=1)
    try:
        # NULL views are rejected before any CUDA call
        assert lib.fa_lp_quantize(h, None, 128, 128, None, 128, 128, None, 128, 128, None) == 1
        # forward before quantize is out of order
        assert lib.fa_lp_forward_varlen(h, None, ctypes.c_void_p(16), 128, 128, None) == 6
        assert lib.fa_lp_plan_set_wait_limit(h, 0) == 1
        assert lib.fa_lp_plan_set_wait_limit(h, 5) == 0
        assert lib.fa_lp_encode(3, None, 0, None, None) == 1
        # host-buffer entry: NULL views and chunk sizes outside 0..heads are rejected first
        hb = ctypes.create_string_buffer(64 * 128 * 2 + 16)
        hp = ctypes.c_void_p((ctypes.addressof(hb) + 15) // 16 * 16)
        assert lib.fa_lp_attention_host(h, None, 128, 128, hp, 128, 128, hp, 128, 128, hp, 128,
                                        128, 0, None) == 1
        assert lib.fa_lp_attention_host(h, hp, 128, 128, hp, 128, 128, hp, 128, 128, hp, 128,
                                        128, 2, None) == 1
        assert lib.fa_lp_attention_host(h, hp, 128, 128, hp, 128, 128, hp, 128, 128, hp, 128,
                                        128, -1, None) == 1
        assert lib.fa_lp_attention_host(h, hp, 127, 128, hp, 128, 128, hp, 128, 128, hp, 128,
                                        128, 1, None) == 1
    finally:
        lib.fa_lp_plan_destroy(h)


def test_nvfp4_workspace_holds_the_qmk_table(lib):
    """NVFP4 plans size their workspace for the qm K^T table: H nb_s^2 128 floats per segment
    (quadratic in the segment length), on top of the codes, scales and means."""
    def ws_of(cu, heads):
        st, h = _create(lib, cu, heads=heads, mode=1)
        assert st == 0
        try:
            ws = ctypes.c_size_t()
            assert lib.fa_lp_workspace_bytes(h, ctypes.byref(ws)) == 0
            return ws.value
        finally:
            assert lib.fa_lp_plan_destroy(h) == 0
    one = ws_of([0, 30272], 56)
    table = 56 * 237 * 237 * 128 * 4
    assert table <= one <= table + 2 * 30336 * 56 * 128
    # the same tokens in two segments: half the blocks each, a quarter of the table each
    two = ws_of([0, 15136, 30272], 56)
    assert two <= one - 0.49 * table
    # an empty segment adds no table (only its K-means row: H x 128 floats, aligned)
    assert ws_of([0, 0, 30272], 56) <= one + 56 * 128 * 4 + 2048


def test_nvfp4_table_ring_bounds_the_workspace(lib):
    """A table limit below the whole qm K^T table makes the plan hold two slots of whole head
    groups (equal groups, one head's table at the least); the work list keeps every item; the
    limit 0 restores the whole table. At S = 30272, H = 56 a 64 MB limit puts the workspace under
    0.5 GB (one head's table is 237^2 x 128 floats = 29 MB)."""
    def layout(h):
        hg, ns, sb = ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
        assert lib.fa_lp_plan_table_layout(h, ctypes.byref(hg), ctypes.byref(ns),
                                           ctypes.byref(sb)) == 0
        tp, wi, ws = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_size_t()
        assert lib.fa_lp_plan_info(h, ctypes.byref(tp), ctypes.byref(wi), ctypes.byref(ws)) == 0
        return hg.value, ns.value, sb.value, wi.value, ws.value

    head = 237 * 237 * 128 * 4
    st, h = _create(lib, [0, 30272], heads=56, mode=1)
    assert st == 0
    try:
        hg, ns, sb, wi, ws_full = layout(h)
        assert (hg, ns, sb) == (56, 1, 56 * head)
        assert lib.fa_lp_plan_set_table_limit(h, 64 << 20) == 0
        hg, ns, sb, wi2, ws = layout(h)
        assert (hg, ns, sb) == (1, 2, head) and wi2 == wi
        assert ws < 500_000_000 and ws_full - ws == 56 * head - 2 * head
        # 200 MB: three heads per 100 MB slot, 19 groups -> equal groups of 3 (the last of 2)
        assert lib.fa_lp_plan_set_table_limit(h, 200 << 20) == 0
        assert layout(h)[:3] == (3, 2, 3 * head)
        assert lib.fa_lp_plan_set_table_limit(h, 0) == 0
        assert layout(h) == (56, 1, 56 * head, wi, ws_full)
    finally:
        assert lib.fa_lp_plan_destroy(h) == 0
    # the default limit (4 GB) holds a 49456-token segment's table whole and rings a 50000-token
    # one: 391^2 x 512 B = 78 MB per head, 27 heads per 2 GB slot -> 3 equal groups of 19
    for L, want in ((49456, (56, 1)), (50000, (19, 2))):
        st, h = _create(lib, [0, L], heads=56, mode=1)
        assert st == 0
        try:
            assert layout(h)[:2] == want
        finally:
            assert lib.fa_lp_plan_destroy(h) == 0
    # FP8 plans hold no table: the limit has no effect
    st, h = _create(lib, [0, 4096], heads=4, mode=0)
    try:
        assert lib.fa_lp_plan_set_table_limit(h, 1) == 0
        assert layout(h)[:3] == (0, 0, 0)
    finally:
        assert lib.fa_lp_plan_destroy(h) == 0


def test_batched_front_end_packs_without_copies():
    """[batch, seq, heads, 128] views become the packed token axis only when no copy is needed."""
    import torch
    from precision_attention_diffusion_gb300 import fa_lp
    x = torch.zeros(3, 5, 2, 128, dtype=torch.bfloat16)
    p = fa_lp.merge_batch(x, "x")
    assert tuple(p.shape) == (15, 2, 128) and p.data_ptr() == x.data_ptr()
    assert p.stride() == (256, 128, 1)
    fused = torch.zeros(3, 5, 3, 2, 128, dtype=torch.bfloat16)
    q = fa_lp.merge_batch(fused[:, :, 0], "q")
    assert q.stride() == (768, 128, 1) and tuple(q.shape) == (15, 2, 128)
    # token 7 of the packed view is sequence 1, token 2 of the batch
    fused[1, 2, 0, 1, 5] = 3.0
    assert float(q[7, 1, 5]) == 3.0
    with pytest.raises(ValueError):
        fa_lp.merge_batch(x.transpose(0, 1), "x")  # seq-major storage: batch cannot be packed
    with pytest.raises(ValueError):
        fa_lp.merge_batch(x[0], "x")


def test_sparse_query_blocks_and_argument_checks(lib):
    """G = sum over segments of ceil(L_s / 64) (64-row query blocks, SGLang PR #40116,
    Modifications); fa_lp_forward_sparse refuses NVFP4 plans and calls before quantize."""
    cu = [0, 0, 17, 4113, 4113, 31800, 32768]
    st, h = _create(lib, cu, heads=3)
    assert st == 0
    try:
        g = ctypes.c_int64()
        assert lib.fa_lp_sparse_query_blocks(h, ctypes.byref(g)) == 0
        assert g.value == sum((b - a + 63) // 64 for a, b in zip(cu[:-1], cu[1:]))
        assert lib.fa_lp_sparse_query_blocks(h, None) == 1
        # before quantize: out of order
        assert lib.fa_lp_forward_sparse(h, None, ctypes.c_void_p(16), ctypes.c_void_p(16), 4,
                                        ctypes.c_void_p(16), 128, 128, None, 0, None) == 6
    finally:
        lib.fa_lp_plan_destroy(h)
    st, h = _create(lib, [0, 256], heads=1, mode=1)
    assert st == 0
    try:
        assert lib.fa_lp_forward_sparse(h, None, ctypes.c_void_p(16), ctypes.c_void_p(16), 4,
                                        ctypes.c_void_p(16), 128, 128, None, 0, None) == 2
    finally:
        lib.fa_lp_plan_destroy(h)


def test_noalloc_rejects_misaligned_or_oversized_arguments_before_any_cuda_call(lib):
    """fa_lp_fp8_descale_noalloc validates its host-visible arguments first: a descale pointer
    that is not 4-byte aligned, or more heads than its fixed scratch holds, returns
    FA_LP_ERR_INVALID_ARG without touching a GPU (the pointers below are never dereferenced)."""
    fake = ctypes.c_void_p(0x10000)
    misaligned = ctypes.c_void_p(0x10002)
    st = lib.fa_lp_fp8_descale_noalloc(fake, 512, 128, fake, 512, 128, fake, 512, 128, 0, 4,
                                       misaligned, None)
    assert st == 1
    st = lib.fa_lp_fp8_descale_noalloc(fake, 512, 128, fake, 512, 128, fake, 512, 128, 0, 1025,
                                       fake, None)
    assert st == 1
