"""Top-k index selection (dsv4_topk, through the C ABI) against the oracle.

The selected set is unique (ties go to the lower index, -0 ranks below +0)
and the output order is ascending, so the bar is exact equality of the index
lists.  At the 1M-context size the oracle checks sampled rows and every row
is checked for the properties that define the result.
"""
import numpy as np
import pytest
import torch

from hybrid_sparse_mqa_gb300 import synth
from oracle import dsv4_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from hybrid_sparse_mqa_gb300 import build
    build.build()
    from hybrid_sparse_mqa_gb300 import attn
    attn.lib()
    attn.dsv4_attn_get_device_error()
    return attn


def run(A, scores, lengths, k, max_length=None):
    s = scores.cuda() if scores.device.type != "cuda" else scores
    l = lengths.cuda() if lengths.device.type != "cuda" else lengths
    out = A.dsv4_topk(s, l, k, max_length=max_length)
    torch.cuda.synchronize()
    return out.cpu().numpy(), A.dsv4_attn_get_device_error()


@pytest.mark.parametrize("name", ["topk_tiny", "topk_c4_decode"])
def test_topk_matches_oracle(A, name):
    inp = synth.make_topk_inputs(name)
    got, flags = run(A, inp.scores, inp.lengths, inp.work.k)
    assert flags == 0
    assert np.array_equal(got, O.topk_indices(**inp.oracle_kwargs()))


def test_topk_1m_context(A):
    # 32 rows of 262144 candidates (the pages' 1M-context shape): rows 0, 13
    # and 31 against the oracle; every row: 512 distinct ascending indices
    # below the row length whose scores are exactly the 512 best values
    inp = synth.make_topk_inputs("topk_1m", device="cuda")
    k = inp.work.k
    got, flags = run(A, inp.scores, inp.lengths, k)
    assert flags == 0
    kw = inp.oracle_kwargs()
    for r in (0, 13, 31):
        want = O.topk_indices(kw["scores"][r:r + 1], kw["lengths"][r:r + 1], k)[0]
        assert np.array_equal(got[r], want), r
    g = torch.from_numpy(got).cuda().long()
    assert bool((g[:, 1:] > g[:, :-1]).all()) and bool((g >= 0).all())
    assert bool((g < inp.lengths[:, None].long()).all())
    best = torch.topk(inp.scores[:, :inp.lengths.max()], k, dim=1).values.sort(dim=1).values
    assert torch.equal(torch.gather(inp.scores, 1, g).sort(dim=1).values, best)


def test_topk_long_ragged_rows(A):
    # 16 rows of up to 262144 candidates: the launch holds 64 scores per
    # thread (half of them in shared memory) and rows end inside a group of
    # four, inside the shared-memory half, at a CTA boundary and past it
    rows, n = 16, 262144
    g = torch.Generator().manual_seed(21)
    scores = torch.randn(rows, n, generator=g)
    scores[3, 70000:70600] = 5.0                                     # a tied block above the rest
    scores[9] = torch.randint(-4, 4, (n,), generator=g).float()      # heavy ties
    lengths = torch.tensor([n, n - 3, 200001, 131075, 65536, 65539, 40000, 513, 1025, 150002, 32768 + 34,
                            32768 * 3 + 129, 262141, 99999, 7, 0], dtype=torch.int32)
    for k in (512, 1024):
        got, flags = run(A, scores, lengths, k)
        assert flags == 0
        assert np.array_equal(got, O.topk_indices(scores.numpy(), lengths.numpy(), k)), k


@pytest.mark.parametrize("rows,n", [(32, 16384), (8, 40000), (32, 65536), (8, 262144), (16, 262144)])
def test_topk_ties_every_launch_shape(A, rows, n):
    # integer-valued scores (long runs of equal values across warps, CTAs and
    # the cluster) at lengths that select each launch shape: 4, 8, 16, 32 and
    # 64 scores per thread; row lengths end inside a group of four
    g = torch.Generator().manual_seed(rows * 7 + n)
    scores = torch.randint(-6, 6, (rows, n), generator=g).float()
    scores[0] = 1.0                                                  # one value everywhere
    scores[1, n // 3:] = 7.0                                         # the top value in one late run
    lengths = torch.full((rows,), n, dtype=torch.int32)
    lengths[2::3] = torch.randint(n // 2, n, (len(range(2, rows, 3)),), generator=g, dtype=torch.int32)
    for k in (512, 1000):
        got, flags = run(A, scores, lengths, k)
        assert flags == 0
        assert np.array_equal(got, O.topk_indices(scores.numpy(), lengths.numpy(), k)), k


def test_topk_longest_rows(A):
    # rows up to the longest length the call takes (524288: eight CTAs of
    # 65536 scores per row), ragged, with a tied block near the end
    n = A.dsv4_topk_max_length(512)
    assert n == 524288
    g = torch.Generator().manual_seed(23)
    scores = torch.randn(4, n, generator=g)
    scores[1, n - 700:n - 100] = 6.0
    lengths = torch.tensor([n, n - 1, 300001, 65537], dtype=torch.int32)
    for k in (512, 1024):
        got, flags = run(A, scores, lengths, k)
        assert flags == 0
        assert np.array_equal(got, O.topk_indices(scores.numpy(), lengths.numpy(), k)), k


def test_topk_edges(A):
    n = 40000
    g = torch.Generator().manual_seed(9)
    rows = []
    rows.append(torch.zeros(n))                                       # all equal -> lowest indices
    rows.append(torch.randn(n, generator=g))
    z = torch.zeros(n)
    z[torch.randperm(n, generator=g)[: n // 2]] = -0.0                # signed zeros
    z[5], z[77] = -1.0, -2.0
    rows.append(z)
    rows.append(torch.randint(-3, 3, (n,), generator=g).float())      # heavy ties across chunks
    rows.append(torch.arange(n).float())                              # rising: the last k
    rows.append(-torch.arange(n).float())                             # falling: the first k
    rows.append(torch.randn(n, generator=g))
    rows.append(torch.randn(n, generator=g))
    scores = torch.stack(rows)
    lengths = torch.tensor([n, 16384, 16385, 32769, n, n, 0, 1], dtype=torch.int32)
    for k in (1, 7, 512, 1024):
        got, flags = run(A, scores, lengths, k)
        assert flags == 0
        assert np.array_equal(got, O.topk_indices(scores.numpy(), lengths.numpy(), k)), k


def test_topk_length_out_of_range_is_clamped_and_reported(A):
    scores = torch.randn(3, 2048)
    lengths = torch.tensor([2048, 3000, -4], dtype=torch.int32)
    got, flags = run(A, scores, lengths, 100, max_length=2048)
    assert flags == 0x100
    want = O.topk_indices(scores.numpy(), [2048, 2048, 0], 100)
    assert np.array_equal(got, want)


def test_topk_repeated_and_back_to_back_calls(A):
    # calls queued back to back on one stream (each may start while the one
    # before drains) give the same answers as calls made one at a time
    inp = synth.make_topk_inputs("topk_1m", device="cuda")
    rows = 4
    scores, lengths = inp.scores[:rows].contiguous(), inp.lengths[:rows].contiguous()
    flipped = scores.flip(1).contiguous()
    a, _ = run(A, scores, lengths, 512)
    outs = [A.dsv4_topk(x, lengths, 512) for x in (scores, flipped, scores, flipped)]
    torch.cuda.synchronize()
    assert A.dsv4_attn_get_device_error() == 0
    kw = dict(scores=flipped.cpu().numpy()[:1], lengths=lengths.cpu().numpy()[:1], k=512)
    want_flipped = O.topk_indices(**kw)[0]
    for j, o in enumerate(outs):
        o = o.cpu().numpy()
        if j % 2 == 0:
            assert np.array_equal(o, a)
        else:
            assert np.array_equal(o[0], want_flipped)


def test_topk_feeds_c4_attention(A):
    # indexer scores -> top-512 -> C4 decode, on the GPU, against the oracle
    # doing both steps
    work = synth.Workload("topk_c4", batch=4, heads=64, ratio=4, seq_lens=(9000, 70000, 2500, 33000), seed=12)
    inp = synth.make_inputs(work, device="cuda")
    n_c = [(s) // 4 for s in work.seq_lens]                  # rows visible to the token at position s - 1
    stride = (max(n_c) + 3) // 4 * 4
    g = torch.Generator(device="cuda").manual_seed(3)
    scores = torch.randn(work.batch, stride, generator=g, device="cuda")
    lengths = torch.tensor(n_c, dtype=torch.int32, device="cuda")
    idx = A.dsv4_topk(scores, lengths, 512)
    inp.topk_idx = idx
    out, lse = A.run_inputs(inp)
    torch.cuda.synchronize()
    assert A.dsv4_attn_get_device_error() == 0
    want_idx = O.topk_indices(scores.cpu().numpy(), n_c, 512)
    assert np.array_equal(idx.cpu().numpy(), want_idx)
    kw = inp.oracle_kwargs()
    kw["topk_idx"] = want_idx
    res = O.dsv4_attention(**kw)
    assert res.errors == 0
    e = np.abs(out.float().cpu().numpy() - res.out)
    assert e.max() <= 1e-2 and e.mean() <= 1e-3
    assert np.abs(lse.cpu().numpy() - res.lse).max() <= 1e-3
