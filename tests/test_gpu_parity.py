"""CUDA path (through the C ABI) against the float64 oracle.

Tolerances: bf16 inputs ~ N(0,1)*0.5 -> max |out - oracle| <= 1e-2 and mean
|out - oracle| <= 1e-3; packed FP8 KV -> max <= 3e-2 against the oracle on the
same dequantised values; lse within 1e-3.  The gathered row sets must match
the oracle's bit for bit (debug dump).
"""
import numpy as np
import pytest
import torch

from hybrid_sparse_mqa_gb300 import synth
from oracle import dsv4_oracle as O

pytestmark = pytest.mark.gpu

TOL_MAX_BF16, TOL_MEAN_BF16, TOL_MAX_FP8, TOL_LSE = 1e-2, 1e-3, 3e-2, 1e-3


@pytest.fixture(scope="module")
def attn():
    from hybrid_sparse_mqa_gb300 import build
    build.build()
    from hybrid_sparse_mqa_gb300 import attn as A
    A.lib()
    A.dsv4_attn_get_device_error()     # start from a clean error word
    return A


def run_and_compare(A, inp, *, tokens=None, num_splits=0, check_rows=True):
    dev = torch.device("cuda")
    g = inp.to(dev) if inp.q.device.type != "cuda" else inp
    stride = A.debug_stride_for(g)
    dbg = torch.full((g.T, stride), -7, dtype=torch.int32, device=dev) if check_rows else None
    out, lse = A.run_inputs(g, num_splits=num_splits, debug_rows=dbg)
    torch.cuda.synchronize()
    flags = A.dsv4_attn_get_device_error()
    res = O.dsv4_attention(**g.oracle_kwargs(), tokens=tokens)
    assert res.errors == 0, f"oracle flagged input errors {res.errors}"
    assert flags == 0, f"device error flags {flags:#x}"
    toks = list(range(g.T)) if tokens is None else list(tokens)
    o = out.float().cpu().numpy()[toks]
    ref = res.out[toks]
    assert np.all(np.isfinite(o))
    err = np.abs(o - ref)
    fp8 = g.work.kv_format == "fp8"
    assert err.max() <= (TOL_MAX_FP8 if fp8 else TOL_MAX_BF16), f"max abs err {err.max():.3e}"
    if not fp8:
        assert err.mean() <= TOL_MEAN_BF16, f"mean abs err {err.mean():.3e}"
    lerr = np.abs(lse.cpu().numpy()[toks] - res.lse[toks])
    assert lerr.max() <= TOL_LSE, f"lse err {lerr.max():.3e}"
    if check_rows:
        rows = dbg.cpu().numpy()
        for t in toks:
            want = np.full(stride, -1, dtype=np.int64)
            want[:len(res.rows[t])] = res.rows[t]
            assert np.array_equal(rows[t], want), f"token {t}: gathered rows differ"
    return out, lse, float(err.max())


def small(kind, heads, seq_lens, *, qlen=1, topk=512, kv_format="bf16", seed=0, rpi=None, sink=None, window=128):
    ratio = dict(swa=0, c4=4, c128=128)[kind]
    inp = synth.make_inputs(
        synth.Workload(f"t_{kind}", batch=len(seq_lens), heads=heads, ratio=ratio,
                       seq_lens=tuple(seq_lens), qlen=qlen, topk=topk, kv_format=kv_format,
                       req_pool_indices=rpi, window=window, seed=seed), device="cuda")
    if sink is not None:
        inp.sink.fill_(sink)
    return inp


def test_swa_tiny_all_tokens(attn):
    inp = synth.make_inputs("swa_tiny", device="cuda")
    run_and_compare(attn, inp)


@pytest.mark.parametrize("heads", [8, 16, 32, 64, 128])
def test_swa_decode_boundaries(attn, heads):
    # window edge (128), page edge (255/256/257), single token, multi-page windows
    run_and_compare(attn, small("swa", heads, (1, 7, 127, 128, 129, 255, 256, 257, 300, 1000), seed=heads))


@pytest.mark.parametrize("heads", [1, 16, 64, 96, 128])
def test_c4_decode_small(attn, heads):
    # no compressed row visible yet (lengths 1 and 3: every index slot is
    # absent), n_c(p) below and above topk (short lists are padded with -1)
    run_and_compare(attn, small("c4", heads, (1, 3, 4, 100, 515, 2048, 2049, 9000), seed=10 + heads))


@pytest.mark.parametrize("kind,window", [("swa", 1), ("swa", 64), ("swa", 200), ("swa", 512),
                                         ("c4", 64), ("c4", 200), ("c4", 512), ("c128", 300)])
def test_window_sizes(attn, kind, window):
    # windows shorter than a tile, spanning several index chunks (192 slots),
    # and longer than the C4 list
    run_and_compare(attn, small(kind, 64, (2, 150, 700, 3000), qlen=2, window=window, seed=window),
                    num_splits=0)


@pytest.mark.parametrize("topk", [16, 100, 512])
def test_c4_topk_sizes(attn, topk):
    run_and_compare(attn, small("c4", 64, (3000, 700, 5000), topk=topk, seed=topk))


@pytest.mark.parametrize("heads", [64, 128])
def test_c128_decode_small(attn, heads):
    run_and_compare(attn, small("c128", heads, (127, 128, 129, 640, 20000, 70000), seed=20 + heads))


@pytest.mark.parametrize("kind", ["swa", "c4", "c128"])
def test_verify_small(attn, kind):
    run_and_compare(attn, small(kind, 64, (300, 1029, 5000), qlen=3, seed=30))


@pytest.mark.parametrize("kind,chunks", [("swa", (257, 1, 130)), ("c4", (257, 1, 130)), ("c128", (257, 1, 130)),
                                         ("c4", (5, 0, 130)), ("swa", (0, 64, 0))])
def test_extend_chunks(attn, kind, chunks):
    # sparse prefill / extend: requests appending chunks of 1..257 tokens,
    # ragged, across page and window boundaries (every token checked); a
    # request may bring no query token at all
    work = synth.Workload(f"extend_{kind}", batch=3, heads=64, ratio={"swa": 0, "c4": 4, "c128": 128}[kind],
                          seq_lens=(300, 2000, 9000), qlen=1, swa_resident="all", seed=33)
    inp = synth.make_inputs(work)
    # replace the one-token boundaries by the ragged extend chunks
    cu = torch.tensor([0] + list(np.cumsum(chunks)), dtype=torch.int32)
    T = int(cu[-1])
    g = torch.Generator().manual_seed(34)
    inp.cu_seqlens_q = cu
    inp.q = (torch.randn(T, 64, 512, generator=g) * 0.5).to(torch.bfloat16)
    if work.ratio == 4:
        seq = inp.seq_lens.tolist()
        rows = []
        for b, (lo, hi) in enumerate(zip(cu[:-1].tolist(), cu[1:].tolist())):
            for i in range(hi - lo):
                p = seq[b] - (hi - lo) + i
                n_c = (p + 1) // 4
                row = torch.full((512,), -1, dtype=torch.int32)
                k = min(512, n_c)
                row[:k] = torch.randperm(n_c, generator=g)[:k].to(torch.int32)
                rows.append(row)
        inp.topk_idx = torch.stack(rows)
    run_and_compare(attn, inp)


def test_req_pool_indices(attn):
    inp = small("c4", 32, (900, 3000), rpi=(5, 9), seed=40)
    run_and_compare(attn, inp)


@pytest.mark.parametrize("sink", [float("-inf"), 0.0, 30.0])
def test_sink_values(attn, sink):
    run_and_compare(attn, small("c4", 64, (600, 4000), sink=sink, seed=50))


@pytest.mark.parametrize("splits", [1, 2, 3, 4, 7, 8, 12])
def test_split_invariance(attn, splits):
    inp = small("c128", 64, (33000, 60000, 129), seed=60)
    out, _, _ = run_and_compare(attn, inp, num_splits=splits)
    ref, _, _ = run_and_compare(attn, inp, num_splits=1, check_rows=False)
    assert (out.float() - ref.float()).abs().max().item() <= 1e-2


def test_device_errors_are_flagged_not_trapped(attn):
    inp = small("c4", 64, (900, 3000, 5000), seed=70)
    bad_pt = inp.swa_page_table.clone()
    bad_pt[0, 899 // 256] = inp.swa_pool.shape[0] // 256        # page id past the pool
    idx = inp.topk_idx.clone()
    idx[1, 0] = 3000 // 4                                       # >= n_c(2999) = 750
    from dataclasses import replace
    bad = replace(inp, swa_page_table=bad_pt, topk_idx=idx)
    out, lse = attn.run_inputs(bad)
    torch.cuda.synchronize()
    flags = attn.dsv4_attn_get_device_error()
    assert flags & attn.DEV_ERR["SWA_PAGE"] and flags & attn.DEV_ERR["INDEX_RANGE"]
    assert attn.dsv4_attn_get_device_error() == 0               # read clears
    res = O.dsv4_attention(**bad.oracle_kwargs())
    assert res.errors == (O.ERR_SWA_PAGE | O.ERR_INDEX_RANGE)
    # skipped slots are skipped identically on both sides
    err = np.abs(out.float().cpu().numpy() - res.out).max()
    assert err <= TOL_MAX_BF16


def test_position_and_extra_page_errors(attn):
    # a request with no tokens yet (seq_len 0: its decode position is -1) and
    # a C4 index on an extra page id past the pool: both flagged, and the
    # outputs still match the oracle's (the position-less token attends to the
    # sink alone: zero output, lse = sink)
    inp = small("c4", 64, (900, 3000, 5000), seed=71)
    from dataclasses import replace
    seq = inp.seq_lens.clone()
    seq[0] = 0
    ept = inp.extra_page_table.clone()
    i2 = int(inp.topk_idx[2, 0])
    ept[2, i2 // 256] = inp.extra_pool.shape[0] // 256
    bad = replace(inp, seq_lens=seq, extra_page_table=ept)
    out, lse = attn.run_inputs(bad)
    torch.cuda.synchronize()
    flags = attn.dsv4_attn_get_device_error()
    assert flags == attn.DEV_ERR["EXTRA_PAGE"] | attn.DEV_ERR["POSITION"], hex(flags)
    res = O.dsv4_attention(**bad.oracle_kwargs())
    assert res.errors == (O.ERR_EXTRA_PAGE | O.ERR_TOKEN_POSITION)
    assert np.abs(out.float().cpu().numpy() - res.out).max() <= TOL_MAX_BF16
    assert np.abs(lse.cpu().numpy() - res.lse).max() <= TOL_LSE


def test_req_row_error(attn):
    # a req_pool_indices entry past the page tables is flagged, not trapped
    inp = small("c4", 32, (900, 3000), rpi=(5, 9), seed=72)
    from dataclasses import replace
    rpi = inp.req_pool_indices.clone()
    rpi[1] = inp.swa_page_table.shape[0] + 3
    attn.run_inputs(replace(inp, req_pool_indices=rpi))
    torch.cuda.synchronize()
    assert attn.dsv4_attn_get_device_error() & attn.DEV_ERR["REQ_ROW"]


def test_plan_too_short_is_flagged(attn):
    # C128 with max_seq_len below a request's length: the plan covers fewer
    # key slots than that token has; the call is flagged, nothing traps, and
    # the library stays usable for a correct call afterwards
    inp = small("c128", 64, (20000, 3000), seed=73)
    swa = attn.make_pool(inp.swa_pool, inp.swa_page_table)
    extra = attn.make_pool(inp.extra_pool, inp.extra_page_table)
    attn.dsv4_attn_c128_dense(inp.q, inp.seq_lens, swa, extra, inp.sink, max_seq_len=4000, scale=inp.scale)
    torch.cuda.synchronize()
    assert attn.dsv4_attn_get_device_error() & attn.DEV_ERR["PLAN"]
    run_and_compare(attn, inp)


# ---------------------------------------------------------------- full-size workloads
@pytest.mark.parametrize("name,tokens", [
    ("swa_decode", None),                        # every token
    ("c4_decode", None),
    ("c128_decode", None),
    ("c128_decode_b2", None),                    # grid-split plan: the combine kernel
    ("c4_prefill", list(range(0, 4096, 8)) + [1023, 1024, 4095]),
])
def test_full_size(attn, name, tokens):
    inp = synth.make_inputs(name, device="cuda")
    run_and_compare(attn, inp, tokens=tokens)


@pytest.mark.parametrize("splits", [4, 16])
def test_c128_long_slices(attn, splits):
    # one token at 1M context: 8192 compressed rows + the window, cut into
    # slices of about 2080 keys (44 tiles) or 520 keys over 2 cluster groups
    inp = small("c128", 128, (1048576,), seed=61)
    run_and_compare(attn, inp, num_splits=splits)


def test_more_tokens_than_a_grid_row(attn):
    # one call with 70000 query tokens (two extend chunks of 35000): tokens
    # beyond 65535 are addressed like the others
    work = synth.Workload("t_many", batch=2, heads=8, ratio=0, seq_lens=(40000, 38000), qlen=35000,
                          swa_resident="all", seed=62)
    inp = synth.make_inputs(work, device="cuda")
    assert inp.T == 70000
    run_and_compare(attn, inp, tokens=[0, 34999, 35000, 65534, 65535, 65536, 69999])


# ---------------------------------------------------------------- packed FP8 KV
@pytest.mark.parametrize("kind,qlen", [("swa", 1), ("c4", 1), ("c128", 1), ("c4", 4), ("c128", 3)])
def test_fp8_small(attn, kind, qlen):
    run_and_compare(attn, small(kind, 64, (300, 1029, 5000), qlen=qlen, kv_format="fp8", seed=80))


def test_fp8_h128(attn):
    run_and_compare(attn, small("c128", 128, (700, 3000), kv_format="fp8", seed=81))


def test_fp8_h96_verify(attn):
    # a partial second head group, several query tokens per request
    run_and_compare(attn, small("c4", 96, (800, 6000), qlen=3, kv_format="fp8", seed=83))


@pytest.mark.parametrize("kind,splits", [("c4", 8), ("c4", 16), ("c128", 6), ("c128", 14)])
def test_fp8_split_merge(attn, kind, splits):
    # packed-FP8 rows (values up to a few units) through the cluster merge's
    # bf16 exchange and, past 8 slices, the combine kernel's fp32 partials
    run_and_compare(attn, small(kind, 64, (2000, 9000), qlen=2, kv_format="fp8", seed=82), num_splits=splits)


def test_full_size_c4_verify_fp8(attn):
    inp = synth.make_inputs("c4_verify_fp8", device="cuda")
    # every request's first and last query token, and all four of every 8th request
    toks = sorted(set([4 * b for b in range(64)] + [4 * b + 3 for b in range(64)] +
                      [4 * b + i for b in range(0, 64, 8) for i in range(4)]))
    run_and_compare(attn, inp, tokens=toks)


def test_back_to_back_calls_read_inputs_after_the_previous_kernel(attn):
    """Attention launches carry programmatic stream serialisation: a launch may
    start while the previous kernel of the stream drains, but must read none
    of its inputs before that kernel has finished.  Chain calls on one stream
    without synchronising, each taking the previous call's output as its
    query (including a grid-split plan, whose combine kernel precedes the next
    launch), and compare every link with the oracle on the query it got."""
    import dataclasses
    inp = small("c4", 64, (3000, 9000, 20000, 65000, 700, 40000), seed=91)
    links = []
    q = inp.q
    for k, splits in enumerate((0, 16, 0, 4, 0)):
        g = dataclasses.replace(inp, q=q)
        out, lse = attn.run_inputs(g, num_splits=splits)
        links.append((g, out, lse))
        q = out
    torch.cuda.synchronize()
    assert attn.dsv4_attn_get_device_error() == 0
    for k, (g, out, lse) in enumerate(links):
        res = O.dsv4_attention(**g.oracle_kwargs())
        err = np.abs(out.float().cpu().numpy() - res.out)
        assert err.max() <= TOL_MAX_BF16, (k, float(err.max()))
        assert err.mean() <= TOL_MEAN_BF16, (k, float(err.mean()))
        assert np.abs(lse.cpu().numpy() - res.lse).max() <= TOL_LSE, k
