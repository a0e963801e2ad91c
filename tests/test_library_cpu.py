"""The C ABI library without a GPU: it builds, loads, exports every entry point
the header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def A():
    from hybrid_sparse_mqa_gb300 import build
    build.build()
    from hybrid_sparse_mqa_gb300 import attn
    attn.lib()
    return attn


def header_functions():
    names = set()
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(dsv4_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = header_functions()
    for want in ("dsv4_attn_swa", "dsv4_attn_c4_sparse", "dsv4_attn_c128_dense", "dsv4_attn_verify",
                 "dsv4_kv_store"):
        assert want in names


def test_every_declared_symbol_is_exported(A):
    lib = ctypes.CDLL(A.LIB_PATH)
    for name in header_functions():
        assert hasattr(lib, name), name
    assert sorted(A.EXPORTED) == header_functions()


def test_strerror(A):
    assert A.dsv4_attn_strerror(0) == "ok"
    assert "invalid" in A.dsv4_attn_strerror(-1)
    assert "unsupported" in A.dsv4_attn_strerror(-2)
    assert "workspace" in A.dsv4_attn_strerror(-3)


def _pool(A, page_size=256, row_bytes=1024, fmt=0, pages=4):
    p = A.KvPool()
    p.rows = 4096
    p.num_pages = pages
    p.row_bytes = row_bytes
    p.format = fmt
    p.page_table = 8192
    p.page_table_rows = 2
    p.page_table_stride = 4
    p.page_size = page_size
    return p


def _swa(A, pool, H=64, window=128, q=4096, out=4096, sink=4096, seq=4096, batch=2):
    return A.lib().dsv4_attn_swa(q, batch, H, seq, None, ctypes.byref(pool), window, sink, 0.044,
                                 out, None, 0, None, 0, None, None)


def test_host_validation(A):
    ok = _pool(A)
    assert _swa(A, ok, q=None) == -1
    assert _swa(A, ok, out=None) == -1
    assert _swa(A, ok, H=0) == -1
    assert _swa(A, ok, H=129) == -1
    assert _swa(A, ok, window=0) == -1
    assert _swa(A, ok, batch=0) == -1
    assert _swa(A, _pool(A, page_size=255)) == -2          # page_size must be 256
    assert _swa(A, _pool(A, row_bytes=1000)) == -2         # bf16 rows are 1024 bytes
    assert _swa(A, _pool(A, pages=0)) == -1
    lib = A.lib()
    # compress ratio outside {0, 4, 128}
    rc = lib.dsv4_attn_verify(4096, 2, 2, 64, 4096, 4096, None, ctypes.byref(ok), 128, 5,
                              ctypes.byref(ok), None, 0, 0, 4096, 0.044, 4096, None, 0, None, 0,
                              None, None)
    assert rc == -2
    # C4 without an index list
    rc = lib.dsv4_attn_c4_sparse(4096, 2, 64, 4096, None, ctypes.byref(ok), 128, ctypes.byref(ok),
                                 None, 512, 4096, 0.044, 4096, None, 0, None, 0, None, None)
    assert rc == -1
    # verify without cu_seqlens_q
    rc = lib.dsv4_attn_verify(4096, 2, 2, 64, 4096, None, None, ctypes.byref(ok), 128, 0, None, None,
                              0, 0, 4096, 0.044, 4096, None, 0, None, 0, None, None)
    assert rc == -1


def test_kv_store_host_validation(A):
    lib = A.lib()
    ok = _pool(A)
    fp8 = _pool(A, row_bytes=608, fmt=1)
    assert lib.dsv4_kv_store(4096, -1, 4096, 4096, ctypes.byref(ok), None) == -1
    assert lib.dsv4_kv_store(4096, 4, 4096, 4096, None, None) == -1
    assert lib.dsv4_kv_store(4096, 4, 4096, 4096, ctypes.byref(_pool(A, page_size=128)), None) == -2
    assert lib.dsv4_kv_store(4096, 4, 4096, 4096, ctypes.byref(_pool(A, row_bytes=1024, fmt=1)), None) == -2
    assert lib.dsv4_kv_store(4096, 4, 4096, 4096, ctypes.byref(_pool(A, pages=0)), None) == -1
    assert lib.dsv4_kv_store(None, 4, 4096, 4096, ctypes.byref(ok), None) == -1
    assert lib.dsv4_kv_store(4096, 4, None, 4096, ctypes.byref(fp8), None) == -1
    assert lib.dsv4_kv_store(4096, 4, 4096, None, ctypes.byref(fp8), None) == -1
    assert lib.dsv4_kv_store(4104, 4, 4096, 4096, ctypes.byref(fp8), None) == -1     # k not 16-byte aligned
    assert lib.dsv4_kv_store(None, 0, None, None, ctypes.byref(fp8), None) == 0       # nothing to store


def test_topk_host_validation(A):
    lib = A.lib()
    assert lib.dsv4_topk_max_length(512) == 524288 and lib.dsv4_topk_max_length(1024) == 524288
    assert lib.dsv4_topk_max_length(0) == 0 and lib.dsv4_topk_max_length(1025) == 0
    assert lib.dsv4_topk(4096, 0, 16, 4096, 16, 4, 4096, None) == -1          # no rows
    assert lib.dsv4_topk(4096, 65536, 16, 4096, 16, 4, 4096, None) == -1      # too many rows
    assert lib.dsv4_topk(4096, 2, 16, 4096, 16, 0, 4096, None) == -1          # k = 0
    assert lib.dsv4_topk(4096, 2, 16, 4096, 16, 1025, 4096, None) == -1       # k too large
    assert lib.dsv4_topk(4096, 2, 16, 4096, -1, 4, 4096, None) == -1          # negative max_length
    assert lib.dsv4_topk(4096, 2, 14, 4096, 16, 4, 4096, None) == -1          # stride < max_length
    assert lib.dsv4_topk(4096, 2, 18, 4096, 16, 4, 4096, None) == -1          # stride not a multiple of 4
    assert lib.dsv4_topk(4100, 2, 16, 4096, 16, 4, 4096, None) == -1          # scores misaligned
    assert lib.dsv4_topk(None, 2, 16, 4096, 16, 4, 4096, None) == -1
    assert lib.dsv4_topk(4096, 2, 16, None, 16, 4, 4096, None) == -1
    assert lib.dsv4_topk(4096, 2, 16, 4096, 16, 4, None, None) == -1
    assert lib.dsv4_topk(4096, 2, 524292, 4096, 524292, 512, 4096, None) == -2   # too long


def test_kv_store_without_device_reports_cuda_error(A):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert A.lib().dsv4_kv_store(4096, 4, 4096, 4096, ctypes.byref(_pool(A, row_bytes=608, fmt=1)), None) == -4


def test_topk_without_device_reports_cuda_error(A):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert A.lib().dsv4_topk(4096, 2, 16, 4096, 16, 4, 4096, None) == -4


def test_plan_without_device_reports_cuda_error(A):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    sc, sg = ctypes.c_int32(), ctypes.c_int32()
    assert A.lib().dsv4_attn_plan(32, 64, 4, 128, 512, 0, 0, ctypes.byref(sc), ctypes.byref(sg)) == -4
