"""Thin Python binding over the C ABI of libfa_lp.so (``include/fa_lp.h``).

Argument marshalling only: torch tensors become device pointers and element strides, torch streams
become ``cudaStream_t`` handles. Every step of the computation runs in the library's CUDA kernels;
there is no Python or CPU fallback. If the library is missing this module raises on first use.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

FA_LP_OK = 0
FA_LP_ERR_INVALID_ARG = 1
FA_LP_ERR_UNSUPPORTED = 2
FA_LP_ERR_CUDA = 3
FA_LP_ERR_OOM = 4
FA_LP_ERR_DEVICE_TIMEOUT = 5
FA_LP_ERR_STATE = 6

MODE_FP8 = 0
MODE_NVFP4 = 1
MODE_FP8_SEGMENT = 2  # FP8 with one scale per (segment, tensor, head)

(Q_CODES, K_CODES, V_CODES, DESCALE, Q_SCALES, K_SCALES, V_SCALES, Q_MEANS, K_MEANS, Q_KM,
 QMK_TABLE) = range(11)

# Every symbol include/fa_lp.h declares.
EXPORTS = (
    "fa_lp_status_string", "fa_lp_plan_create", "fa_lp_plan_destroy", "fa_lp_plan_info",
    "fa_lp_workspace_bytes", "fa_lp_quantize", "fa_lp_forward_varlen", "fa_lp_attention",
    "fa_lp_plan_row_offsets", "fa_lp_get_quantized", "fa_lp_copy_quantized",
    "fa_lp_get_last_error", "fa_lp_plan_set_wait_limit", "fa_lp_release_workspace",
    "fa_lp_encode", "fa_lp_fp8_descale_noalloc", "fa_lp_forward_varlen_lse",
    "fa_lp_attention_host", "fa_lp_forward_sparse", "fa_lp_sparse_query_blocks",
    "fa_lp_attention_sparse_host", "fa_lp_plan_set_table_limit", "fa_lp_plan_table_layout",
)

_lib = None
_lock = threading.Lock()


class FaLpError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class _ArrayDesc(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dims", ctypes.c_int64 * 3),
                ("strides", ctypes.c_int64 * 3), ("elem_bytes", ctypes.c_int)]


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libfa_lp.so. Raises if it has not been built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"libfa_lp.so is not built ({path}); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            _build.build()
        L = ctypes.CDLL(path)
        P, i64, i32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                ctypes.c_size_t)
        L.fa_lp_status_string.argtypes = [i32]
        L.fa_lp_status_string.restype = ctypes.c_char_p
        L.fa_lp_plan_create.argtypes = [i64, i32, P, i32, f32, i32, i32, ctypes.POINTER(P)]
        L.fa_lp_plan_destroy.argtypes = [P]
        L.fa_lp_plan_info.argtypes = [P, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                      ctypes.POINTER(sz)]
        L.fa_lp_workspace_bytes.argtypes = [P, ctypes.POINTER(sz)]
        L.fa_lp_quantize.argtypes = [P, P, i64, i64, P, i64, i64, P, i64, i64, P]
        L.fa_lp_forward_varlen.argtypes = [P, P, P, i64, i64, P]
        L.fa_lp_forward_varlen_lse.argtypes = [P, P, P, i64, i64, P, i64, P]
        L.fa_lp_forward_sparse.argtypes = [P, P, P, P, i64, P, i64, i64, P, i64, P]
        L.fa_lp_sparse_query_blocks.argtypes = [P, ctypes.POINTER(i64)]
        L.fa_lp_attention_sparse_host.argtypes = [P, P, i64, i64, P, i64, i64, P, i64, i64, P, P,
                                                  i64, P, i64, i64, i32, P]
        L.fa_lp_attention.argtypes = [P, P, i64, i64, P, i64, i64, P, i64, i64, P, P, i64, i64, P]
        L.fa_lp_attention_host.argtypes = [P, P, i64, i64, P, i64, i64, P, i64, i64, P, i64, i64,
                                           i32, P]
        L.fa_lp_plan_row_offsets.argtypes = [P, ctypes.POINTER(i64)]
        L.fa_lp_get_quantized.argtypes = [P, i32, ctypes.POINTER(_ArrayDesc)]
        L.fa_lp_copy_quantized.argtypes = [P, i32, P, sz, P]
        L.fa_lp_get_last_error.argtypes = [P, ctypes.POINTER(i32)]
        L.fa_lp_plan_set_wait_limit.argtypes = [P, i64]
        L.fa_lp_plan_set_table_limit.argtypes = [P, sz]
        L.fa_lp_plan_table_layout.argtypes = [P, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                              ctypes.POINTER(sz)]
        L.fa_lp_release_workspace.argtypes = [i32, P]
        L.fa_lp_encode.argtypes = [i32, P, i64, P, P]
        L.fa_lp_fp8_descale_noalloc.argtypes = [P, i64, i64, P, i64, i64, P, i64, i64, i64, i32, P,
                                                P]
        for name in EXPORTS:
            if name != "fa_lp_status_string":
                getattr(L, name).restype = i32
        _lib = L
        return L


def status_string(status: int) -> str:
    try:
        return load().fa_lp_status_string(int(status)).decode()
    except Exception:  # pragma: no cover - library missing
        return f"status {status}"


def _check(status: int, what: str):
    if status != FA_LP_OK:
        raise FaLpError(status, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _view(x: torch.Tensor, name: str, host: bool = False):
    if x.dtype != torch.bfloat16 or x.dim() != 3 or x.shape[2] != 128 or x.stride(2) != 1:
        raise ValueError(f"{name} must be a bfloat16 [tokens, heads, 128] view with unit channel "
                         f"stride (got {tuple(x.shape)} {x.dtype} strides {x.stride()})")
    if x.is_cuda == host:
        raise ValueError(f"{name} must be a {'host (CPU)' if host else 'CUDA'} tensor")
    return ctypes.c_void_p(x.data_ptr()), int(x.stride(0)), int(x.stride(1))


class Plan:
    """A cached segment plan (FlashInfer docs: cached per (cu_seqlens, heads, device))."""

    def __init__(self, cu_seqlens_host, heads: int, softmax_scale: float | None = None,
                 mode: int = MODE_FP8, device: int | None = None):
        L = load()
        cu = [int(c) for c in cu_seqlens_host]
        self.cu = cu
        self.heads = int(heads)
        self.mode = int(mode)
        self.device = torch.cuda.current_device() if device is None else int(device)
        self.tokens = cu[-1]
        self.scale = (1.0 / math.sqrt(128)) if softmax_scale is None else float(softmax_scale)
        arr = (ctypes.c_int32 * len(cu))(*cu)
        h = ctypes.c_void_p()
        _check(L.fa_lp_plan_create(self.tokens, self.heads, arr, len(cu) - 1, self.scale,
                                   self.mode, self.device, ctypes.byref(h)), "fa_lp_plan_create")
        self._h = h

    # -- lifetime ---------------------------------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _check(load().fa_lp_plan_destroy(self._h), "fa_lp_plan_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    # -- facts ------------------------------------------------------------------------------------
    def info(self):
        tp, wi, ws = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_size_t()
        _check(load().fa_lp_plan_info(self._h, ctypes.byref(tp), ctypes.byref(wi),
                                      ctypes.byref(ws)), "fa_lp_plan_info")
        return dict(padded_tokens=tp.value, work_items=wi.value, workspace_bytes=ws.value)

    def row_offsets(self):
        n = len(self.cu)
        arr = (ctypes.c_int64 * n)()
        _check(load().fa_lp_plan_row_offsets(self._h, arr), "fa_lp_plan_row_offsets")
        return list(arr)

    def set_wait_limit(self, spins: int):
        _check(load().fa_lp_plan_set_wait_limit(self._h, int(spins)), "fa_lp_plan_set_wait_limit")

    def set_table_limit(self, nbytes: int):
        """NVFP4: the largest qm K^T table held at once (0: the library default)."""
        _check(load().fa_lp_plan_set_table_limit(self._h, int(nbytes)),
               "fa_lp_plan_set_table_limit")

    def table_layout(self):
        hg, ns, sb = ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
        _check(load().fa_lp_plan_table_layout(self._h, ctypes.byref(hg), ctypes.byref(ns),
                                              ctypes.byref(sb)), "fa_lp_plan_table_layout")
        return dict(heads_per_slot=hg.value, slots=ns.value, slot_bytes=sb.value)

    def last_error(self) -> int:
        v = ctypes.c_int()
        st = load().fa_lp_get_last_error(self._h, ctypes.byref(v))
        if v.value == 0:  # a non-zero device status comes with DEVICE_TIMEOUT or INVALID_ARG
            _check(st, "fa_lp_get_last_error")
        return v.value

    # -- compute ----------------------------------------------------------------------------------
    def quantize(self, q, k, v, stream=None):
        qa, qs, qh = _view(q, "q")
        ka, ks, kh = _view(k, "k")
        va, vs, vh = _view(v, "v")
        _check(load().fa_lp_quantize(self._h, qa, qs, qh, ka, ks, kh, va, vs, vh, _stream(stream)),
               "fa_lp_quantize")

    def forward(self, out, cu_seqlens_dev=None, stream=None, lse=None):
        """Attention over the last quantize; `lse` (optional, float32 [heads, >= tokens] on the
        device) receives each row's log-sum-exp."""
        oa, os_, oh = _view(out, "out")
        cu = ctypes.c_void_p(cu_seqlens_dev.data_ptr()) if cu_seqlens_dev is not None else None
        if lse is None:
            _check(load().fa_lp_forward_varlen(self._h, cu, oa, os_, oh, _stream(stream)),
                   "fa_lp_forward_varlen")
            return out
        if (lse.dtype != torch.float32 or lse.dim() != 2 or lse.stride(1) != 1 or not lse.is_cuda
                or lse.shape[0] != self.heads or lse.shape[1] < self.tokens):
            raise ValueError("lse must be a CUDA float32 [heads, >= tokens] tensor with unit "
                             "token stride")
        _check(load().fa_lp_forward_varlen_lse(self._h, cu, oa, os_, oh,
                                               ctypes.c_void_p(lse.data_ptr()),
                                               int(lse.stride(0)), _stream(stream)),
               "fa_lp_forward_varlen_lse")
        return out

    def sparse_query_blocks(self) -> int:
        """G: the 64-row query blocks of the plan (block lists are indexed h * G + g)."""
        g = ctypes.c_int64()
        _check(load().fa_lp_sparse_query_blocks(self._h, ctypes.byref(g)),
               "fa_lp_sparse_query_blocks")
        return g.value

    def forward_sparse(self, block_offsets, block_indices, out, stream=None, lse=None):
        """Block-sparse attention over the last quantize: `block_offsets` (int32 [heads G + 1])
        and `block_indices` (int32) on the device, the list of (head h, query block g) being
        block_indices[block_offsets[h G + g] : block_offsets[h G + g + 1]]."""
        oa, os_, oh = _view(out, "out")
        for name, x in (("block_offsets", block_offsets), ("block_indices", block_indices)):
            if x.dtype != torch.int32 or not x.is_cuda or not x.is_contiguous():
                raise ValueError(f"{name} must be a contiguous CUDA int32 tensor")
        if block_offsets.numel() != self.heads * self.sparse_query_blocks() + 1:
            raise ValueError("block_offsets must hold heads * G + 1 entries")
        lp, ls = None, 0
        if lse is not None:
            if (lse.dtype != torch.float32 or lse.dim() != 2 or lse.stride(1) != 1
                    or not lse.is_cuda or lse.shape[0] != self.heads
                    or lse.shape[1] < self.tokens):
                raise ValueError("lse must be a CUDA float32 [heads, >= tokens] tensor with unit "
                                 "token stride")
            lp, ls = ctypes.c_void_p(lse.data_ptr()), int(lse.stride(0))
        _check(load().fa_lp_forward_sparse(self._h, None, ctypes.c_void_p(block_offsets.data_ptr()),
                                           ctypes.c_void_p(block_indices.data_ptr()),
                                           int(block_indices.numel()), oa, os_, oh, lp, ls,
                                           _stream(stream)), "fa_lp_forward_sparse")
        return out

    def attention(self, q, k, v, cu_seqlens_dev=None, out=None, stream=None):
        if out is None:
            out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
        qa, qs, qh = _view(q, "q")
        ka, ks, kh = _view(k, "k")
        va, vs, vh = _view(v, "v")
        oa, os_, oh = _view(out, "out")
        cu = ctypes.c_void_p(cu_seqlens_dev.data_ptr()) if cu_seqlens_dev is not None else None
        _check(load().fa_lp_attention(self._h, qa, qs, qh, ka, ks, kh, va, vs, vh, cu, oa, os_, oh,
                                      _stream(stream)), "fa_lp_attention")
        return out

    def attention_host(self, q, k, v, out, heads_per_chunk: int = 0, stream=None):
        """out = attention(q, k, v) with q, k, v and out in host memory (CPU tensors; page-locked
        ones let the copies overlap the compute). Heads go through the device in chunks whose
        copy-in, compute and copy-out overlap; `out` is complete once `stream` is."""
        qa, qs, qh = _view(q, "q", host=True)
        ka, ks, kh = _view(k, "k", host=True)
        va, vs, vh = _view(v, "v", host=True)
        oa, os_, oh = _view(out, "out", host=True)
        _check(load().fa_lp_attention_host(self._h, qa, qs, qh, ka, ks, kh, va, vs, vh, oa, os_,
                                           oh, int(heads_per_chunk), _stream(stream)),
               "fa_lp_attention_host")
        return out

    def attention_sparse_host(self, q, k, v, block_offsets, block_indices, out,
                              heads_per_chunk: int = 0, stream=None):
        """fa_lp_attention_sparse_host: q, k, v, out BF16 [tokens, heads, 128] CPU tensors
        (page-locked for overlap); block_offsets (int32 [heads G + 1]) and block_indices
        (int32) contiguous CPU tensors."""
        qa, qs, qh = _view(q, "q", host=True)
        ka, ks, kh = _view(k, "k", host=True)
        va, vs, vh = _view(v, "v", host=True)
        oa, os_, oh = _view(out, "out", host=True)
        for name, x in (("block_offsets", block_offsets), ("block_indices", block_indices)):
            if x.dtype != torch.int32 or x.is_cuda or not x.is_contiguous():
                raise ValueError(f"{name} must be a contiguous CPU int32 tensor")
        if block_offsets.numel() != self.heads * self.sparse_query_blocks() + 1:
            raise ValueError("block_offsets must hold heads * G + 1 entries")
        _check(load().fa_lp_attention_sparse_host(
            self._h, qa, qs, qh, ka, ks, kh, va, vs, vh, ctypes.c_void_p(block_offsets.data_ptr()),
            ctypes.c_void_p(block_indices.data_ptr()), int(block_indices.numel()), oa, os_, oh,
            int(heads_per_chunk), _stream(stream)), "fa_lp_attention_sparse_host")
        return out

    # -- inspection -------------------------------------------------------------------------------
    def quantized(self, which: int, stream=None) -> torch.Tensor:
        """Copy one quantized array out of the workspace into a new device tensor."""
        d = _ArrayDesc()
        _check(load().fa_lp_get_quantized(self._h, int(which), ctypes.byref(d)),
               "fa_lp_get_quantized")
        dims = [int(x) for x in d.dims]
        dtype = torch.uint8 if d.elem_bytes == 1 else torch.float32
        out = torch.empty(dims, dtype=dtype, device=f"cuda:{self.device}")
        _check(load().fa_lp_copy_quantized(self._h, int(which), ctypes.c_void_p(out.data_ptr()),
                                           out.numel() * out.element_size(), _stream(stream)),
               "fa_lp_copy_quantized")
        return out


def encode(fmt: int, x: torch.Tensor, stream=None) -> torch.Tensor:
    """Hardware E4M3 (fmt 0) / E2M1 (fmt 1) round-to-nearest-even saturating conversion."""
    assert x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()
    out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(load().fa_lp_encode(int(fmt), ctypes.c_void_p(x.data_ptr()), x.numel(),
                               ctypes.c_void_p(out.data_ptr()), _stream(stream)), "fa_lp_encode")
    return out


def fp8_descale_noalloc(q, k, v, out=None, stream=None) -> torch.Tensor:
    """FP8 descales [3, heads] (q, k, v) through the entry point that allocates nothing inside
    the library; `out` (float32 [3, heads] on the device) may be passed in."""
    qa, qs, qh = _view(q, "q")
    ka, ks, kh = _view(k, "k")
    va, vs, vh = _view(v, "v")
    heads = q.shape[1]
    if out is None:
        out = torch.empty((3, heads), dtype=torch.float32, device=q.device)
    assert out.dtype == torch.float32 and out.is_contiguous() and out.numel() >= 3 * heads
    _check(load().fa_lp_fp8_descale_noalloc(qa, qs, qh, ka, ks, kh, va, vs, vh, q.shape[0], heads,
                                            ctypes.c_void_p(out.data_ptr()), _stream(stream)),
           "fa_lp_fp8_descale_noalloc")
    return out


def release_workspace(device: int | None = None, stream=None):
    dev = torch.cuda.current_device() if device is None else int(device)
    _check(load().fa_lp_release_workspace(dev, _stream(stream)), "fa_lp_release_workspace")


def attention(q, k, v, cu_seqlens, out=None, *, cu_seqlens_host=None, softmax_scale=None,
              mode: int = MODE_FP8, stream=None):
    """out[a:b, h] = softmax(q[a:b, h] k[a:b, h]^T * scale) v[a:b, h] for every cu_seqlens
    segment, on FP8 (mode 0) or NVFP4 (mode 1) operands. The plan is cached by the library."""
    host = list(cu_seqlens_host) if cu_seqlens_host is not None else cu_seqlens.tolist()
    plan = _plan_cache_get(tuple(host), q.shape[1], softmax_scale, mode, q.device.index)
    return plan.attention(q, k, v, cu_seqlens, out=out, stream=stream)


def merge_batch(x: torch.Tensor, name: str) -> torch.Tensor:
    """View a [batch, seq, heads, 128] tensor as the packed [batch * seq, heads, 128] token axis,
    without copying: the batch stride must equal seq times the token stride (true for contiguous
    tensors and for slices of a fused [batch, seq, 3, heads, 128] QKV buffer)."""
    if x.dim() != 4:
        raise ValueError(f"{name} must be [batch, seq, heads, 128] (got {tuple(x.shape)})")
    B, S = x.shape[0], x.shape[1]
    if B > 1 and S > 0 and x.stride(0) != S * x.stride(1):
        raise ValueError(f"{name}: batch stride {x.stride(0)} is not seq x token stride "
                         f"({S} x {x.stride(1)}); the batch cannot be packed without a copy")
    return x.as_strided((B * S, x.shape[2], x.shape[3]), (x.stride(1), x.stride(2), x.stride(3)))


def attention_batched(q, k, v, out=None, *, softmax_scale=None, mode: int = MODE_FP8,
                      stream=None):
    """Batch > 1 through varlen packing: q, k, v [batch, seq, heads, 128] become one packed call
    with cu_seqlens = [0, seq, 2 seq, ..., batch seq] (each sequence attends to itself only).
    Scales follow the packed call (per (tensor, head) over every token of the batch). Returns
    out [batch, seq, heads, 128]."""
    B, S, H = q.shape[0], q.shape[1], q.shape[2]
    for name, x in (("k", k), ("v", v)):
        if tuple(x.shape) != tuple(q.shape):
            raise ValueError(f"{name} shape {tuple(x.shape)} differs from q {tuple(q.shape)}")
    qp, kp, vp = merge_batch(q, "q"), merge_batch(k, "k"), merge_batch(v, "v")
    if out is None:
        out = torch.empty((B, S, H, q.shape[3]), dtype=torch.bfloat16, device=q.device)
    op = merge_batch(out, "out")
    cu_host = [i * S for i in range(B + 1)]
    cu_dev = torch.tensor(cu_host, dtype=torch.int32, device=q.device)
    attention(qp, kp, vp, cu_dev, out=op, cu_seqlens_host=cu_host, softmax_scale=softmax_scale,
              mode=mode, stream=stream)
    return out


_plans = {}


def _plan_cache_get(cu, heads, scale, mode, device):
    key = (cu, int(heads), scale, int(mode), device)
    p = _plans.get(key)
    if p is None:
        p = Plan(list(cu), heads, softmax_scale=scale, mode=mode, device=device)
        _plans[key] = p
    return p
