"""Python binding of libdsv4attn.so (ctypes).

Argument marshalling only: every step of the attention computation runs in
the library's CUDA kernels.  PyTorch supplies device memory (outputs and the
workspace are allocated here when the caller passes none) and the current
stream.  Loading fails loudly when the library has not been built; there is
no fallback path.

The entry points mirror include/dsv4attn.h:
  dsv4_attn_swa, dsv4_attn_c4_sparse, dsv4_attn_c128_dense, dsv4_attn_verify,
  dsv4_attn_plan, dsv4_attn_workspace_size, dsv4_attn_get_device_error,
  dsv4_attn_strerror;
include/dsv4kvstore.h (the cache write before the step):
  dsv4_kv_store;
and include/dsv4topk.h (the top-k selection that makes the C4 index lists):
  dsv4_topk, dsv4_topk_max_length.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsv4attn.so")

DSV4_KV_BF16 = 0
DSV4_KV_FP8_PACKED = 1
DEV_ERR = {
    "SWA_PAGE": 0x01, "EXTRA_PAGE": 0x02, "INDEX_RANGE": 0x04, "POSITION": 0x08,
    "PLAN": 0x10, "TIMEOUT": 0x20, "REQ_ROW": 0x40, "STORE_ROW": 0x80, "TOPK_LENGTH": 0x100,
}
EXPORTED = [
    "dsv4_attn_swa", "dsv4_attn_c4_sparse", "dsv4_attn_c128_dense", "dsv4_attn_verify",
    "dsv4_attn_plan", "dsv4_attn_workspace_size", "dsv4_attn_get_device_error",
    "dsv4_attn_strerror", "dsv4_attn_c4_sparse_noalloc", "dsv4_kv_store",
    "dsv4_topk", "dsv4_topk_max_length",
]
NOALLOC_SCRATCH_BYTES = 16 << 20


class KvPool(ctypes.Structure):
    _fields_ = [
        ("rows", ctypes.c_void_p),
        ("num_pages", ctypes.c_int64),
        ("row_bytes", ctypes.c_int32),
        ("format", ctypes.c_int32),
        ("page_table", ctypes.c_void_p),
        ("page_table_rows", ctypes.c_int32),
        ("page_table_stride", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
    ]


class Dsv4Error(RuntimeError):
    pass


def load_library(path=LIB_PATH):
    if not os.path.exists(path):
        raise Dsv4Error(f"{path} is missing: build it with hybrid_sparse_mqa_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I32, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    PP = ctypes.POINTER(KvPool)
    lib.dsv4_attn_swa.argtypes = [P, I32, I32, P, P, PP, I32, P, F32, P, P, I32, P, SZ, P, P]
    lib.dsv4_attn_c4_sparse.argtypes = [P, I32, I32, P, P, PP, I32, PP, P, I32, P, F32, P, P, I32, P, SZ, P, P]
    lib.dsv4_attn_c128_dense.argtypes = [P, I32, I32, P, P, PP, I32, PP, I32, P, F32, P, P, I32, P, SZ, P, P]
    lib.dsv4_attn_verify.argtypes = [P, I32, I32, I32, P, P, P, PP, I32, I32, PP, P, I32, I32, P, F32,
                                     P, P, I32, P, SZ, P, P]
    lib.dsv4_attn_c4_sparse_noalloc.argtypes = [P, I32, I32, P, P, PP, I32, PP, P, I32, P, F32, P, P, I32, P, P]
    for name in ("dsv4_attn_swa", "dsv4_attn_c4_sparse", "dsv4_attn_c128_dense", "dsv4_attn_verify",
                 "dsv4_attn_c4_sparse_noalloc"):
        getattr(lib, name).restype = ctypes.c_int
    lib.dsv4_attn_plan.argtypes = [I32, I32, I32, I32, I32, I32, I32,
                                   ctypes.POINTER(I32), ctypes.POINTER(I32)]
    lib.dsv4_attn_plan.restype = ctypes.c_int
    lib.dsv4_attn_workspace_size.argtypes = [I32, I32, I32, I32, I32, I32, I32]
    lib.dsv4_attn_workspace_size.restype = SZ
    lib.dsv4_attn_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), P]
    lib.dsv4_attn_get_device_error.restype = ctypes.c_int
    lib.dsv4_attn_strerror.argtypes = [ctypes.c_int]
    lib.dsv4_attn_strerror.restype = ctypes.c_char_p
    lib.dsv4_kv_store.argtypes = [P, I32, P, P, PP, P]
    lib.dsv4_kv_store.restype = ctypes.c_int
    lib.dsv4_topk.argtypes = [P, I32, ctypes.c_int64, P, I32, I32, P, P]
    lib.dsv4_topk.restype = ctypes.c_int
    lib.dsv4_topk_max_length.argtypes = [I32]
    lib.dsv4_topk_max_length.restype = I32
    return lib


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = load_library()
    return _lib


# ---------------------------------------------------------------- helpers
def _ptr(x):
    return None if x is None else ctypes.c_void_p(x.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_pool(rows, page_table, kv_format=None):
    """dsv4_kv_pool for a device pool tensor ([rows, 512] bf16 or [rows, 608]
    uint8) and its int32 page table [request rows, logical pages]."""
    if kv_format is None:
        kv_format = DSV4_KV_BF16 if rows.dtype == torch.bfloat16 else DSV4_KV_FP8_PACKED
    row_bytes = rows.shape[1] * rows.element_size()
    pool = KvPool()
    pool.rows = rows.data_ptr()
    pool.num_pages = rows.shape[0] // 256
    pool.row_bytes = row_bytes
    pool.format = kv_format
    pool.page_table = page_table.data_ptr()
    pool.page_table_rows = page_table.shape[0]
    pool.page_table_stride = page_table.stride(0)
    pool.page_size = 256
    pool._keep = (rows, page_table)
    return pool


def _check(rc):
    if rc != 0:
        raise Dsv4Error(f"dsv4attn: {lib().dsv4_attn_strerror(rc).decode()} ({rc})")


def _outputs(q, out, lse):
    T, H = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(T, H, dtype=torch.float32, device=q.device)
    return out, lse


def _workspace(workspace, T, H, ratio, window, topk, max_seq_len, num_splits, device):
    need = lib().dsv4_attn_workspace_size(T, H, ratio, window, topk, max_seq_len, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    return workspace, (0 if workspace is None else workspace.numel() * workspace.element_size())


def debug_stride(ratio, window, topk=0, max_seq_len=0):
    return window + (topk if ratio == 4 else (max_seq_len // 128 if ratio == 128 else 0))


# ---------------------------------------------------------------- entry points
def dsv4_attn_swa(q, seq_lens, swa_pool, sink, *, scale=1.0 / math.sqrt(512), window=128,
                  req_pool_indices=None, out=None, lse=None, num_splits=0, workspace=None,
                  debug_rows=None, stream=None):
    T, H = q.shape[0], q.shape[1]
    out, lse = _outputs(q, out, lse)
    workspace, wsb = _workspace(workspace, T, H, 0, window, 0, 0, num_splits, q.device)
    _check(lib().dsv4_attn_swa(_ptr(q), T, H, _ptr(seq_lens), _ptr(req_pool_indices),
                               ctypes.byref(swa_pool), window, _ptr(sink), scale, _ptr(out), _ptr(lse),
                               num_splits, _ptr(workspace), wsb, _ptr(debug_rows), _stream(stream)))
    return out, lse


def dsv4_attn_c4_sparse(q, seq_lens, swa_pool, extra_pool, topk_idx, sink, *,
                        scale=1.0 / math.sqrt(512), window=128, req_pool_indices=None, out=None,
                        lse=None, num_splits=0, workspace=None, debug_rows=None, stream=None):
    T, H = q.shape[0], q.shape[1]
    topk = topk_idx.shape[1]
    out, lse = _outputs(q, out, lse)
    workspace, wsb = _workspace(workspace, T, H, 4, window, topk, 0, num_splits, q.device)
    _check(lib().dsv4_attn_c4_sparse(_ptr(q), T, H, _ptr(seq_lens), _ptr(req_pool_indices),
                                     ctypes.byref(swa_pool), window, ctypes.byref(extra_pool),
                                     _ptr(topk_idx), topk, _ptr(sink), scale, _ptr(out), _ptr(lse),
                                     num_splits, _ptr(workspace), wsb, _ptr(debug_rows), _stream(stream)))
    return out, lse


def dsv4_attn_c4_sparse_noalloc(q, seq_lens, swa_pool, extra_pool, topk_idx, sink, *,
                                scale=1.0 / math.sqrt(512), window=128, req_pool_indices=None,
                                out=None, lse=None, num_splits=0, debug_rows=None, stream=None):
    """dsv4_attn_c4_sparse without a workspace argument: for callers that
    cannot allocate device memory, the split merge uses the library's own
    static scratch buffer (see include/dsv4attn.h for its limits)."""
    T, H = q.shape[0], q.shape[1]
    topk = topk_idx.shape[1]
    if out is None or lse is None:
        out, lse = _outputs(q, out, lse)
    _check(lib().dsv4_attn_c4_sparse_noalloc(_ptr(q), T, H, _ptr(seq_lens), _ptr(req_pool_indices),
                                             ctypes.byref(swa_pool), window, ctypes.byref(extra_pool),
                                             _ptr(topk_idx), topk, _ptr(sink), scale, _ptr(out), _ptr(lse),
                                             num_splits, _ptr(debug_rows), _stream(stream)))
    return out, lse


def dsv4_attn_c128_dense(q, seq_lens, swa_pool, extra_pool, sink, *, max_seq_len,
                         scale=1.0 / math.sqrt(512), window=128, req_pool_indices=None, out=None,
                         lse=None, num_splits=0, workspace=None, debug_rows=None, stream=None):
    T, H = q.shape[0], q.shape[1]
    out, lse = _outputs(q, out, lse)
    workspace, wsb = _workspace(workspace, T, H, 128, window, 0, max_seq_len, num_splits, q.device)
    _check(lib().dsv4_attn_c128_dense(_ptr(q), T, H, _ptr(seq_lens), _ptr(req_pool_indices),
                                      ctypes.byref(swa_pool), window, ctypes.byref(extra_pool),
                                      max_seq_len, _ptr(sink), scale, _ptr(out), _ptr(lse), num_splits,
                                      _ptr(workspace), wsb, _ptr(debug_rows), _stream(stream)))
    return out, lse


def dsv4_attn_verify(q, seq_lens, cu_seqlens_q, swa_pool, sink, *, compress_ratio, batch,
                     extra_pool=None, topk_idx=None, max_seq_len=0, scale=1.0 / math.sqrt(512),
                     window=128, req_pool_indices=None, out=None, lse=None, num_splits=0,
                     workspace=None, debug_rows=None, stream=None):
    T, H = q.shape[0], q.shape[1]
    topk = 0 if topk_idx is None else topk_idx.shape[1]
    out, lse = _outputs(q, out, lse)
    workspace, wsb = _workspace(workspace, T, H, compress_ratio, window, topk, max_seq_len,
                                num_splits, q.device)
    _check(lib().dsv4_attn_verify(_ptr(q), T, batch, H, _ptr(seq_lens), _ptr(cu_seqlens_q),
                                  _ptr(req_pool_indices), ctypes.byref(swa_pool), window,
                                  compress_ratio,
                                  None if extra_pool is None else ctypes.byref(extra_pool),
                                  _ptr(topk_idx), topk, max_seq_len, _ptr(sink), scale, _ptr(out),
                                  _ptr(lse), num_splits, _ptr(workspace), wsb, _ptr(debug_rows),
                                  _stream(stream)))
    return out, lse


def dsv4_attn_plan(num_tokens, num_heads, compress_ratio, window=128, topk=0, max_seq_len=0,
                   num_splits=0):
    sc, sg = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().dsv4_attn_plan(num_tokens, num_heads, compress_ratio, window, topk, max_seq_len,
                                num_splits, ctypes.byref(sc), ctypes.byref(sg)))
    return sc.value, sg.value


def dsv4_attn_workspace_size(num_tokens, num_heads, compress_ratio, window=128, topk=0,
                             max_seq_len=0, num_splits=0):
    return lib().dsv4_attn_workspace_size(num_tokens, num_heads, compress_ratio, window, topk,
                                          max_seq_len, num_splits)


def dsv4_attn_get_device_error(stream=None):
    v = ctypes.c_uint32()
    _check(lib().dsv4_attn_get_device_error(ctypes.byref(v), _stream(stream)))
    return v.value


def dsv4_attn_strerror(status):
    return lib().dsv4_attn_strerror(status).decode()


# ---------------------------------------------------------------- one call per workload
def dsv4_kv_store(k, req_rows, positions, pool, *, stream=None):
    """Store new key rows k (bf16 [n, 512]) into `pool` (a make_pool()
    descriptor) at logical row positions[i] of page-table row req_rows[i]
    (int32 [n] each), packing them to FP8 for a packed pool."""
    if k.dtype != torch.bfloat16 or k.dim() != 2 or k.shape[1] != 512 or not k.is_contiguous():
        raise Dsv4Error("k must be a contiguous bf16 [n, 512] tensor")
    n = k.shape[0]
    for name, x in (("req_rows", req_rows), ("positions", positions)):
        if x.dtype != torch.int32 or x.numel() != n or not x.is_contiguous():
            raise Dsv4Error(f"{name} must be a contiguous int32 tensor of {n} entries")
    _check(lib().dsv4_kv_store(_ptr(k), n, _ptr(req_rows), _ptr(positions), ctypes.byref(pool),
                               _stream(stream)))


def dsv4_topk_max_length(k):
    return lib().dsv4_topk_max_length(k)


def dsv4_topk(scores, lengths, k, *, max_length=None, out=None, stream=None):
    """Indices of the k best scores of every row (ascending, -1 padded):
    scores fp32 [rows, stride] (stride a multiple of 4), lengths int32 [rows]."""
    if scores.dtype != torch.float32 or scores.dim() != 2 or scores.stride(1) != 1:
        raise Dsv4Error("scores must be a row-major fp32 [rows, stride] tensor")
    rows = scores.shape[0]
    if lengths.dtype != torch.int32 or lengths.numel() != rows or not lengths.is_contiguous():
        raise Dsv4Error(f"lengths must be a contiguous int32 tensor of {rows} entries")
    if max_length is None:
        max_length = scores.shape[1]
    if out is None:
        out = torch.empty(rows, k, dtype=torch.int32, device=scores.device)
    _check(lib().dsv4_topk(_ptr(scores), rows, scores.stride(0), _ptr(lengths), max_length, k, _ptr(out),
                           _stream(stream)))
    return out


def run_inputs(inp, *, num_splits=0, debug_rows=None, out=None, lse=None, workspace=None, stream=None):
    """Dispatch a synth.Inputs batch (already on the GPU) to the matching entry point."""
    w = inp.work
    swa = make_pool(inp.swa_pool, inp.swa_page_table)
    kw = dict(scale=inp.scale, window=w.window, req_pool_indices=inp.req_pool_indices, out=out,
              lse=lse, num_splits=num_splits, workspace=workspace, debug_rows=debug_rows, stream=stream)
    extra = None if inp.extra_pool is None else make_pool(inp.extra_pool, inp.extra_page_table)
    if inp.cu_seqlens_q is not None:
        return dsv4_attn_verify(inp.q, inp.seq_lens, inp.cu_seqlens_q, swa, inp.sink,
                                compress_ratio=w.ratio, batch=w.batch, extra_pool=extra,
                                topk_idx=inp.topk_idx, max_seq_len=inp.max_seq_len, **kw)
    if w.ratio == 0:
        return dsv4_attn_swa(inp.q, inp.seq_lens, swa, inp.sink, **kw)
    if w.ratio == 4:
        return dsv4_attn_c4_sparse(inp.q, inp.seq_lens, swa, extra, inp.topk_idx, inp.sink, **kw)
    return dsv4_attn_c128_dense(inp.q, inp.seq_lens, swa, extra, inp.sink,
                                max_seq_len=inp.max_seq_len, **kw)


def debug_stride_for(inp):
    w = inp.work
    return debug_stride(w.ratio, w.window, w.topk if w.ratio == 4 else 0, inp.max_seq_len)
