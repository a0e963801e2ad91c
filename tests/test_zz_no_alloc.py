"""The allocation-free C4 entry point against the regular one.

dsv4_attn_c4_sparse_noalloc exists for callers that cannot allocate device
memory (code running where no allocator may be called, or a process whose
memory is reserved up front): it takes no workspace and keeps the scratch its
split merge needs in a static buffer inside the library.  These tests call it
through the C ABI twice in a row on a problem whose plan does need scratch and
check each result against dsv4_attn_c4_sparse, which takes a caller workspace.
The file is named so that pytest collects it after every other test.
"""
import numpy as np
import pytest
import torch

from hybrid_sparse_mqa_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN, TOL_LSE = 1e-2, 1e-3, 1e-3


@pytest.fixture(scope="module")
def A():
    from hybrid_sparse_mqa_gb300 import build
    build.build()
    from hybrid_sparse_mqa_gb300 import attn
    attn.lib()
    attn.dsv4_attn_get_device_error()
    return attn


def _inputs():
    # 8 decode tokens of 640 keys each: the plan splits every token across a
    # cluster, so the merge needs scratch memory
    return synth.make_inputs(
        synth.Workload("noalloc_c4", batch=8, heads=64, ratio=4,
                       seq_lens=(3000, 9000, 700, 20000, 5000, 65536, 1200, 40000), seed=21),
        device="cuda")


def test_noalloc_matches_allocating_entry_point_twice(A):
    inp = _inputs()
    w = inp.work
    need = A.dsv4_attn_workspace_size(inp.T, inp.H, 4, w.window, w.topk, 0, 0)
    assert 0 < need <= A.NOALLOC_SCRATCH_BYTES, need      # the path under test uses scratch
    swa = A.make_pool(inp.swa_pool, inp.swa_page_table)
    extra = A.make_pool(inp.extra_pool, inp.extra_page_table)
    ref_out, ref_lse = A.dsv4_attn_c4_sparse(inp.q, inp.seq_lens, swa, extra, inp.topk_idx, inp.sink,
                                             scale=inp.scale, window=w.window)
    torch.cuda.synchronize()
    ref_out = ref_out.float().cpu().numpy()
    ref_lse = ref_lse.cpu().numpy()
    out = torch.empty_like(inp.q)
    lse = torch.empty(inp.T, inp.H, dtype=torch.float32, device="cuda")
    for call in range(2):
        out.fill_(7.0)
        lse.fill_(7.0)
        A.dsv4_attn_c4_sparse_noalloc(inp.q, inp.seq_lens, swa, extra, inp.topk_idx, inp.sink,
                                      scale=inp.scale, window=w.window, out=out, lse=lse)
        torch.cuda.synchronize()
        assert A.dsv4_attn_get_device_error() == 0
        err = np.abs(out.float().cpu().numpy() - ref_out)
        assert err.max() <= TOL_MAX, (call, err.max())
        assert err.mean() <= TOL_MEAN, (call, err.mean())
        assert np.abs(lse.cpu().numpy() - ref_lse).max() <= TOL_LSE, call


def test_noalloc_rejects_plans_beyond_its_scratch(A):
    inp = _inputs()
    w = inp.work
    # force 8 slices per token on 64 tokens: 64 x 8 x 64 KB of merge scratch > 16 MiB
    q = inp.q.repeat(8, 1, 1)
    seq = inp.seq_lens.repeat(8)
    idx = inp.topk_idx.repeat(8, 1)
    need = A.dsv4_attn_workspace_size(q.shape[0], inp.H, 4, w.window, w.topk, 0, 8)
    assert need > A.NOALLOC_SCRATCH_BYTES
    swa = A.make_pool(inp.swa_pool, inp.swa_page_table)
    extra = A.make_pool(inp.extra_pool, inp.extra_page_table)
    rpi = torch.arange(8, dtype=torch.int32, device="cuda").repeat(8)
    with pytest.raises(A.Dsv4Error, match="scratch"):
        A.dsv4_attn_c4_sparse_noalloc(q, seq, swa, extra, idx, inp.sink, scale=inp.scale,
                                      window=w.window, req_pool_indices=rpi, num_splits=8)
