"""The allocation-free C4 entry point against the regular one.

dsv4_attn_c4_sparse_noalloc exists for callers that cannot allocate device
memory (code running where no allocator may be called, or a process whose
memory is reserved up front): it takes no workspace and keeps the scratch a
split plan needs (the partial rows the slices of a cluster exchange and the
fp32 partial results that the combine kernel merges) in a static buffer
inside the library.  These tests call it through
the C ABI on problems whose plan does need that scratch, one after another
with different inputs so that a read of the previous call's scratch would
show, and check each result against dsv4_attn_c4_sparse, which takes a
caller workspace.  The file is named so that pytest collects it after every
other test.
"""
import numpy as np
import pytest
import torch

from hybrid_sparse_mqa_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN, TOL_LSE = 1e-2, 1e-3, 1e-3
SPLITS = 16          # 8 slices per cluster x 2 cluster groups merged through the scratch


@pytest.fixture(scope="module")
def A():
    from hybrid_sparse_mqa_gb300 import build
    build.build()
    from hybrid_sparse_mqa_gb300 import attn
    attn.lib()
    attn.dsv4_attn_get_device_error()
    return attn


def _inputs(seq_lens, seed):
    return synth.make_inputs(
        synth.Workload("noalloc_c4", batch=len(seq_lens), heads=64, ratio=4, seq_lens=tuple(seq_lens),
                       seed=seed), device="cuda")


def _check(A, inp):
    """One no-allocation call (into outputs prefilled with junk) against the
    allocating entry point on the same inputs."""
    w = inp.work
    swa = A.make_pool(inp.swa_pool, inp.swa_page_table)
    extra = A.make_pool(inp.extra_pool, inp.extra_page_table)
    ref_out, ref_lse = A.dsv4_attn_c4_sparse(inp.q, inp.seq_lens, swa, extra, inp.topk_idx, inp.sink,
                                             scale=inp.scale, window=w.window, num_splits=SPLITS)
    out = torch.full_like(inp.q, 7.0)
    lse = torch.full((inp.T, inp.H), 7.0, dtype=torch.float32, device="cuda")
    A.dsv4_attn_c4_sparse_noalloc(inp.q, inp.seq_lens, swa, extra, inp.topk_idx, inp.sink,
                                  scale=inp.scale, window=w.window, out=out, lse=lse, num_splits=SPLITS)
    torch.cuda.synchronize()
    assert A.dsv4_attn_get_device_error() == 0
    err = np.abs(out.float().cpu().numpy() - ref_out.float().cpu().numpy())
    assert err.max() <= TOL_MAX, err.max()
    assert err.mean() <= TOL_MEAN, err.mean()
    assert np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy()).max() <= TOL_LSE


def test_noalloc_matches_allocating_entry_point_on_consecutive_calls(A):
    first = _inputs((3000, 9000, 700, 20000, 5000, 65536, 1200, 40000), seed=21)
    second = _inputs((65536, 2500, 33000, 900, 12000, 7000, 50000, 4100), seed=22)
    sc, sg = A.dsv4_attn_plan(first.T, first.H, 4, first.work.window, first.work.topk, 0, SPLITS)
    assert sg > 1, (sc, sg)                                  # the plan merges through the scratch
    need = A.dsv4_attn_workspace_size(first.T, first.H, 4, first.work.window, first.work.topk, 0, SPLITS)
    assert 0 < need <= A.NOALLOC_SCRATCH_BYTES, need
    # each call follows one on different inputs: stale scratch would give wrong rows
    for inp in (first, second, first):
        _check(A, inp)


def test_noalloc_rejects_plans_beyond_its_scratch(A):
    inp = _inputs((3000, 9000, 700, 20000, 5000, 65536, 1200, 40000), seed=21)
    w = inp.work
    # 128 tokens x 16 slices of 64 heads x 512 partial values > 16 MiB
    q = inp.q.repeat(16, 1, 1)
    seq = inp.seq_lens.repeat(16)
    idx = inp.topk_idx.repeat(16, 1)
    need = A.dsv4_attn_workspace_size(q.shape[0], inp.H, 4, w.window, w.topk, 0, SPLITS)
    assert need > A.NOALLOC_SCRATCH_BYTES
    swa = A.make_pool(inp.swa_pool, inp.swa_page_table)
    extra = A.make_pool(inp.extra_pool, inp.extra_page_table)
    rpi = torch.arange(8, dtype=torch.int32, device="cuda").repeat(16)
    with pytest.raises(A.Dsv4Error, match="scratch"):
        A.dsv4_attn_c4_sparse_noalloc(q, seq, swa, extra, idx, inp.sink, scale=inp.scale,
                                      window=w.window, req_pool_indices=rpi, num_splits=SPLITS)
