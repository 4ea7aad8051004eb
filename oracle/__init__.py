"""CPU oracle for the low-precision varlen attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package. The product (the CUDA library and its Python binding) never does, and the two share
no code. The arithmetic lives in ``fa_lp_oracle.cpp`` (plain C++17, FP64, no fast-math); this
module only builds it with g++ and marshals numpy arrays through ctypes.

Sources followed (page title and section):
  * SGLang PR #40175 "add fp8_fa_sm120 FP8 backend for SM120 GPUs", Modifications.
  * SGLang PR #40116 "Add SM120 Sage compute for SubBlock sparse attention", Modifications and
    Accuracy Tests (block-sparse lists).
  * FlashInfer docs, ``flashinfer.diffusion_ops.minimax_h3_sm120_varlen_attention_nvfp4``,
    description and Parameters.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_lp_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libfa_lp_oracle.so")
_lock = threading.Lock()
_lib = None

D = 128


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (IEEE single operations: no contraction, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            P = ctypes.c_void_p
            i64, i32, f32, f64, u8 = (ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                      ctypes.c_double, ctypes.c_uint8)
            L.orc_e4m3_encode.argtypes = [f32]; L.orc_e4m3_encode.restype = u8
            L.orc_e4m3_decode.argtypes = [u8]; L.orc_e4m3_decode.restype = f64
            L.orc_e2m1_encode.argtypes = [f32]; L.orc_e2m1_encode.restype = u8
            L.orc_e2m1_decode.argtypes = [u8]; L.orc_e2m1_decode.restype = f64
            L.orc_f64_to_bf16.argtypes = [f64]; L.orc_f64_to_bf16.restype = ctypes.c_uint16
            L.orc_e4m3_encode_array.argtypes = [P, i64, P]
            L.orc_e2m1_encode_array.argtypes = [P, i64, P]
            L.orc_fp8_quantize.argtypes = [P, i64, i32, i64, i64, P, P, i32]
            L.orc_attn_exact.argtypes = [P, i64, i64, P, i64, i64, P, i64, i64, i64, i32, P, i32,
                                         f64, P, i64, P, P, i32]
            L.orc_fp8_quantize_seg.argtypes = [P, i64, i32, i64, i64, P, i32, P, P, i32]
            L.orc_attn_fp8.argtypes = [P, P, P, P, P, P, i64, i32, P, i32, f64, i32, i32, f64, P,
                                       i64, P, P, P, i32, i32]
            L.orc_attn_exact_sparse.argtypes = [P, i64, i64, P, i64, i64, P, i64, i64, i64, i32,
                                                P, i32, f64, P, P, P, i64, P, P, i32]
            L.orc_attn_exact_sparse.restype = i32
            L.orc_attn_fp8_sparse.argtypes = [P, P, P, P, P, P, i64, i32, P, i32, f64, P, P, i32,
                                              f64, P, i64, P, P, P, i32, i32]
            L.orc_attn_fp8_sparse.restype = i32
            L.orc_nvfp4_kmean.argtypes = [P, i64, i64, i64, i32, P, i32, P, i32]
            L.orc_nvfp4_qblock_offsets.argtypes = [P, i32, P]; L.orc_nvfp4_qblock_offsets.restype = i64
            L.orc_nvfp4_vgroup_offsets.argtypes = [P, i32, P]; L.orc_nvfp4_vgroup_offsets.restype = i64
            L.orc_nvfp4_quantize_q.argtypes = [P, i64, i64, i64, i32, P, i32, P, P, P, i32]
            L.orc_nvfp4_quantize_k.argtypes = [P, i64, i64, i64, i32, P, i32, P, P, P, i32]
            L.orc_nvfp4_quantize_v.argtypes = [P, i64, i64, i64, i32, P, i32, P, P, i32]
            L.orc_attn_nvfp4.argtypes = [P, P, P, P, P, P, P, P, i64, i32, P, i32, f64, i32, P,
                                         i64, P, P, P, i32]
            L.orc_nvfp4_qkm.argtypes = [P, i64, i64, i64, i32, P, i32, P, P, i32]
            _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_view(x):
    """Accept a uint16 ndarray of BF16 bits or a torch bfloat16 CPU tensor, shaped [T, H, 128]
    with unit channel stride and any positive token/head strides (a strided view is fine).
    Returns (array, token stride, head stride), strides in elements."""
    if hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch
        assert x.device.type == "cpu"
        x = x.view(torch.int16).numpy().view(np.uint16)
    assert x.dtype == np.uint16 and x.ndim == 3 and x.strides[2] == 2
    assert x.strides[0] > 0 and x.strides[1] > 0
    return x, x.strides[0] // 2, x.strides[1] // 2


def _threads(n):
    return int(n) if n else 0


# ------------------------------------------------------------------------------------------------
# converters
# ------------------------------------------------------------------------------------------------
def e4m3_encode(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().orc_e4m3_encode_array(_p(x), x.size, _p(out))
    return out


def e2m1_encode(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().orc_e2m1_encode_array(_p(x), x.size, _p(out))
    return out


def e4m3_decode_table() -> np.ndarray:
    return np.array([lib().orc_e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e2m1_decode_table() -> np.ndarray:
    return np.array([lib().orc_e2m1_decode(c) for c in range(16)], dtype=np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    flat = np.asarray(x, dtype=np.float64).ravel()
    return np.array([lib().orc_f64_to_bf16(float(v)) for v in flat], np.uint16).reshape(np.shape(x))


# ------------------------------------------------------------------------------------------------
# FP8 path
# ------------------------------------------------------------------------------------------------
def fp8_quantize(x, nthreads=0):
    """x: [T,H,128] BF16 bits (uint16 ndarray, any token/head strides) -> (codes [T,H,128] uint8,
    descale [H] float32)."""
    arr, st, sh = _bf16_view(x)
    T, H = x.shape[0], x.shape[1]
    codes = np.empty((T, H, D), np.uint8)
    d = np.empty(H, np.float32)
    lib().orc_fp8_quantize(_p(arr), T, H, st, sh, _p(codes), _p(d), _threads(nthreads))
    return codes, d


def fp8_quantize_seg(x, cu, nthreads=0):
    """Per-segment FP8 mode: x [T,H,128] BF16 bits, cu_seqlens -> (codes [T,H,128] uint8,
    descale [nseg,H] float32): one amax per (segment, head) over the segment's own tokens."""
    arr, st, sh = _bf16_view(x)
    T, H = x.shape[0], x.shape[1]
    cu = np.ascontiguousarray(cu, np.int32)
    codes = np.zeros((T, H, D), np.uint8)
    d = np.empty((len(cu) - 1, H), np.float32)
    lib().orc_fp8_quantize_seg(_p(arr), T, H, st, sh, _p(cu), len(cu) - 1, _p(codes), _p(d),
                               _threads(nthreads))
    return codes, d


def attn_exact(q, k, v, cu, rows, scale, nthreads=0, lse=False):
    """C1: exact FP64 attention for rows [(token, head)] -> [n,128] float64; with lse=True also
    the row's log-sum-exp log sum_j exp(q.k_j scale) -> (out, lse [n])."""
    (qa, qst, qsh), (ka, kst, ksh), (va, vst, vsh) = _bf16_view(q), _bf16_view(k), _bf16_view(v)
    cu = np.ascontiguousarray(cu, np.int32)
    rows = np.ascontiguousarray(rows, np.int64).reshape(-1, 2)
    out = np.empty((rows.shape[0], D), np.float64)
    ls = np.empty(rows.shape[0], np.float64)
    lib().orc_attn_exact(_p(qa), qst, qsh, _p(ka), kst, ksh, _p(va), vst, vsh, q.shape[0],
                         q.shape[1], _p(cu), len(cu) - 1, float(scale), _p(rows), rows.shape[0],
                         _p(out), _p(ls), _threads(nthreads))
    return (out, ls) if lse else out


def _seg_scales(dq, dk, dv, cu, H):
    """1 when the descales are per (segment, head) ([nseg, H]), 0 when per head ([H])."""
    nseg = len(cu) - 1
    shapes = {tuple(np.shape(a)) for a in (dq, dk, dv)}
    if shapes == {(H,)}:
        return 0
    if shapes == {(nseg, H)}:
        return 1
    raise ValueError("descales must all be [H] or all [nseg, H]")


def attn_fp8(cq, ck, cv, dq, dk, dv, cu, rows, scale, n_kv=128, p_shift=0, tau=0.0,
             nthreads=0, lse=False):
    """C2: FP8-emulating attention from codes/descales -> (out fp64 [n,128], out bf16 bits).
    Descales [H] (one per head, reading r1) or [nseg, H] (the per-segment mode).
    n_kv: key-tile width; tau: threshold (log2 units) for moving the reference maximum, 0 = the
    exact running maximum; p_shift: power-of-two shift applied to P before E4M3 rounding.
    lse=True appends the row's m + log(l) (reading r15) -> (o64, o16, lse [n])."""
    cq, ck, cv = (np.ascontiguousarray(a, np.uint8) for a in (cq, ck, cv))
    dq, dk, dv = (np.ascontiguousarray(a, np.float32) for a in (dq, dk, dv))
    cu = np.ascontiguousarray(cu, np.int32)
    rows = np.ascontiguousarray(rows, np.int64).reshape(-1, 2)
    o64 = np.empty((rows.shape[0], D), np.float64)
    o16 = np.empty((rows.shape[0], D), np.uint16)
    ls = np.empty(rows.shape[0], np.float64)
    seg = _seg_scales(dq, dk, dv, cu, cq.shape[1])
    lib().orc_attn_fp8(_p(cq), _p(ck), _p(cv), _p(dq), _p(dk), _p(dv), cq.shape[0], cq.shape[1],
                       _p(cu), len(cu) - 1, float(scale), int(n_kv), int(p_shift), float(tau),
                       _p(rows),
                       rows.shape[0], _p(o64), _p(o16), _p(ls), _threads(nthreads), seg)
    return (o64, o16, ls) if lse else (o64, o16)


# ------------------------------------------------------------------------------------------------
# block-sparse (64-row query blocks x 64-key key blocks, reading r16)
# ------------------------------------------------------------------------------------------------
def _lists(blk_off, blk_idx):
    off = np.ascontiguousarray(blk_off, np.int32)
    idx = np.ascontiguousarray(blk_idx, np.int32)
    if idx.size == 0:
        idx = np.zeros(1, np.int32)
    return off, idx


def attn_exact_sparse(q, k, v, cu, blk_off, blk_idx, rows, scale, nthreads=0, lse=False):
    """C1 under block lists -> out [n,128] float64 (and lse [n] with lse=True). Raises
    ValueError when a list breaks the contract (index outside the segment, not ascending)."""
    (qa, qst, qsh), (ka, kst, ksh), (va, vst, vsh) = _bf16_view(q), _bf16_view(k), _bf16_view(v)
    cu = np.ascontiguousarray(cu, np.int32)
    off, idx = _lists(blk_off, blk_idx)
    rows = np.ascontiguousarray(rows, np.int64).reshape(-1, 2)
    out = np.empty((rows.shape[0], D), np.float64)
    ls = np.empty(rows.shape[0], np.float64)
    st = lib().orc_attn_exact_sparse(_p(qa), qst, qsh, _p(ka), kst, ksh, _p(va), vst, vsh,
                                     q.shape[0], q.shape[1], _p(cu), len(cu) - 1, float(scale),
                                     _p(off), _p(idx), _p(rows), rows.shape[0], _p(out), _p(ls),
                                     _threads(nthreads))
    if st != 0:
        raise ValueError("block list outside its segment or not strictly ascending")
    return (out, ls) if lse else out


def attn_fp8_sparse(cq, ck, cv, dq, dk, dv, cu, blk_off, blk_idx, rows, scale, p_shift=0,
                    tau=0.0, nthreads=0, lse=False):
    """C2 under block lists: the listed 64-key blocks, in list order, are the online softmax's
    key tiles -> (out fp64 [n,128], out bf16 bits[, lse])."""
    cq, ck, cv = (np.ascontiguousarray(a, np.uint8) for a in (cq, ck, cv))
    dq, dk, dv = (np.ascontiguousarray(a, np.float32) for a in (dq, dk, dv))
    cu = np.ascontiguousarray(cu, np.int32)
    off, idx = _lists(blk_off, blk_idx)
    rows = np.ascontiguousarray(rows, np.int64).reshape(-1, 2)
    o64 = np.empty((rows.shape[0], D), np.float64)
    o16 = np.empty((rows.shape[0], D), np.uint16)
    ls = np.empty(rows.shape[0], np.float64)
    seg = _seg_scales(dq, dk, dv, cu, cq.shape[1])
    st = lib().orc_attn_fp8_sparse(_p(cq), _p(ck), _p(cv), _p(dq), _p(dk), _p(dv), cq.shape[0],
                                   cq.shape[1], _p(cu), len(cu) - 1, float(scale), _p(off),
                                   _p(idx), int(p_shift), float(tau), _p(rows), rows.shape[0],
                                   _p(o64), _p(o16), _p(ls), _threads(nthreads), seg)
    if st != 0:
        raise ValueError("block list outside its segment or not strictly ascending")
    return (o64, o16, ls) if lse else (o64, o16)


# ------------------------------------------------------------------------------------------------
# NVFP4 path
# ------------------------------------------------------------------------------------------------
def nvfp4_offsets(cu):
    cu = np.ascontiguousarray(cu, np.int32)
    ns = len(cu) - 1
    qo = np.empty(ns + 1, np.int64)
    go = np.empty(ns + 1, np.int64)
    lib().orc_nvfp4_qblock_offsets(_p(cu), ns, _p(qo))
    lib().orc_nvfp4_vgroup_offsets(_p(cu), ns, _p(go))
    return qo, go


def nvfp4_quantize(q, k, v, cu, nthreads=0):
    """a6+a7 -> dict with km [nseg,H,128] f32, qm [QB,H,128] f32, q/k/v codes [T,H,128] (one
    4-bit code per byte), q/k scales [T,H,8] (UE4M3 bytes), v scales [H,128,G] (UE4M3 bytes),
    qkm [T,H] f64 = q . km (for the LSE, reading r15)."""
    (qa, qst, qsh), (ka, kst, ksh), (va, vst, vsh) = _bf16_view(q), _bf16_view(k), _bf16_view(v)
    T, H = q.shape[0], q.shape[1]
    cu = np.ascontiguousarray(cu, np.int32)
    ns = len(cu) - 1
    qo, go = nvfp4_offsets(cu)
    L = lib()
    nt = _threads(nthreads)
    km = np.empty((ns, H, D), np.float32)
    L.orc_nvfp4_kmean(_p(ka), kst, ksh, T, H, _p(cu), ns, _p(km), nt)
    qm = np.empty((int(qo[-1]), H, D), np.float32)
    cq = np.zeros((T, H, D), np.uint8)
    sq = np.zeros((T, H, 8), np.uint8)
    L.orc_nvfp4_quantize_q(_p(qa), qst, qsh, T, H, _p(cu), ns, _p(qm), _p(cq), _p(sq), nt)
    ck = np.zeros((T, H, D), np.uint8)
    sk = np.zeros((T, H, 8), np.uint8)
    L.orc_nvfp4_quantize_k(_p(ka), kst, ksh, T, H, _p(cu), ns, _p(km), _p(ck), _p(sk), nt)
    cv = np.zeros((T, H, D), np.uint8)
    sv = np.zeros((H, D, int(go[-1])), np.uint8)
    L.orc_nvfp4_quantize_v(_p(va), vst, vsh, T, H, _p(cu), ns, _p(cv), _p(sv), nt)
    qkm = np.empty((T, H), np.float64)
    L.orc_nvfp4_qkm(_p(qa), qst, qsh, T, H, _p(cu), ns, _p(km), _p(qkm), nt)
    return dict(km=km, qm=qm, cq=cq, sq=sq, ck=ck, sk=sk, cv=cv, sv=sv, qoff=qo, goff=go, qkm=qkm)


def attn_nvfp4(qz, cu, rows, scale, n_kv=128, nthreads=0, lse=False):
    """C3: NVFP4-emulating attention from nvfp4_quantize()'s dict -> (out fp64, out bf16).

    n_kv: width of the online-softmax key tiles (a multiple of 16), counted from each segment
    start; the running maximum is exact. lse=True appends m + log(l / 2688) + q . km scale with
    the BF16 q (reading r15: the LSE of the uncentred scores)."""
    if n_kv <= 0 or n_kv % 16:
        raise ValueError("n_kv must be a positive multiple of 16")
    cu = np.ascontiguousarray(cu, np.int32)
    rows = np.ascontiguousarray(rows, np.int64).reshape(-1, 2)
    T, H = qz["cq"].shape[0], qz["cq"].shape[1]
    o64 = np.empty((rows.shape[0], D), np.float64)
    o16 = np.empty((rows.shape[0], D), np.uint16)
    ls = np.empty(rows.shape[0], np.float64)
    lib().orc_attn_nvfp4(_p(qz["cq"]), _p(qz["sq"]), _p(qz["qm"]), _p(qz["qkm"]), _p(qz["ck"]),
                         _p(qz["sk"]),
                         _p(qz["cv"]), _p(qz["sv"]), T, H, _p(cu), len(cu) - 1, float(scale),
                         int(n_kv), _p(rows), rows.shape[0], _p(o64), _p(o16), _p(ls),
                         _threads(nthreads))
    return (o64, o16, ls) if lse else (o64, o16)
