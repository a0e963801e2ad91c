"""The KV cache write (dsv4_kv_store, through the C ABI) against the oracle.

Storing is byte work and the quantisation decision is taken in float32 on
both sides (reading R13), so the bar is bit-exact: after a call, every byte
of the pool equals the oracle's pool (rows not addressed keep their random
content).  The last test stores rows with the CUDA writer and attends over
them with the CUDA attention step, against the oracle doing both.
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


def _bits(x):
    x = x.detach().cpu()
    return x.view(torch.int16).numpy().view(np.uint16) if x.dtype == torch.bfloat16 else x.numpy()


def gpu_store(A, s):
    pool = s.pool.clone()
    A.dsv4_kv_store(s.k, s.req_rows, s.positions, A.make_pool(pool, s.page_table))
    torch.cuda.synchronize()
    return pool, A.dsv4_attn_get_device_error()


def check_store(A, s, want_flags=0):
    pool, flags = gpu_store(A, s)
    want, err = O.kv_store(**s.oracle_kwargs())
    assert flags == want_flags and err == want_flags, (flags, err)
    got = _bits(pool)
    bad = np.nonzero(np.any(got != want, axis=1))[0]
    assert bad.size == 0, f"{bad.size} pool rows differ, first {bad[:5].tolist()}"
    return pool


@pytest.mark.parametrize("name", ["kv_store_tiny", "kv_store_tiny_bf16", "kv_store_decode"])
def test_store_matches_oracle(A, name):
    check_store(A, synth.make_store_inputs(name, device="cuda"))


def test_store_full_size(A):
    # the benchmark's prefill chunk: 64 requests x 1024 rows into a packed pool
    check_store(A, synth.make_store_inputs("kv_store_prefill", device="cuda"))


def _edge_rows():
    """bf16 rows that stress the packer: exact e4m3 ties, zero and negative
    zero blocks, a block amax that is negative, amax at the bottom and top of
    the bf16 range, and blocks spanning 2^-30 .. 2^30."""
    dec = O.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    mids = ((dec[:-1] + dec[1:]) / 2).astype(np.float32)          # 125 exact midpoints
    rng = np.random.default_rng(17)
    rows = np.zeros((12, 512), dtype=np.float32)
    for b in range(7):
        k = float(2.0 ** (b - 3))
        blk = np.concatenate([[448.0], rng.choice(mids, 63) * rng.choice([-1.0, 1.0], 63)]).astype(np.float32)
        rows[0, 64 * b:64 * b + 64] = blk * np.float32(k)
    rows[1, :] = 0.0
    rows[1, 64:128] = -0.0
    rows[1, 448:] = rng.standard_normal(64).astype(np.float32)
    rows[2, :448] = rng.standard_normal(448).astype(np.float32) * 0.1
    rows[2, 5] = -3.0                                              # negative amax in block 0
    rows[3, :448] = np.float32(1.2e-38) * rng.standard_normal(448).astype(np.float32)
    rows[4, :448] = np.float32(1.0e38) * rng.uniform(-3.0, 3.0, 448).astype(np.float32)
    for r in range(5, 12):
        mag = np.exp2(rng.integers(-30, 31, 8)).astype(np.float32)
        rows[r] = rng.standard_normal(512).astype(np.float32) * np.repeat(mag, 64)
    bits = (rows.view(np.uint32) >> 16).astype(np.uint16)            # truncate to bf16 (finite here)
    return bits


def test_store_edge_values(A):
    s = synth.make_store_inputs("kv_store_tiny")
    bits = _edge_rows()
    n = bits.shape[0]
    s = synth.StoreInputs(work=s.work, k=torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16),
                          req_rows=s.req_rows[:n].clone(), positions=s.positions[:n].clone(),
                          pool=s.pool, page_table=s.page_table).to("cuda")
    check_store(A, s)


def test_store_reports_rows_it_cannot_place(A):
    s = synth.make_store_inputs("kv_store_tiny")
    n = s.k.shape[0]
    req, pos = s.req_rows.clone(), s.positions.clone()
    req[3] = -1                                  # no such request row
    req[10] = s.page_table.shape[0]              # past the table
    req[20] = 1                                  # a table row with no pages (stride 2)
    pos[30] = -5                                 # negative position
    pos[40] = s.page_table.shape[1] * 256        # past the table's width
    s = synth.StoreInputs(work=s.work, k=s.k, req_rows=req, positions=pos, pool=s.pool,
                          page_table=s.page_table).to("cuda")
    check_store(A, s, want_flags=O.ERR_STORE_ROW)
    assert n > 40


def test_store_nothing(A):
    s = synth.make_store_inputs("kv_store_tiny", device="cuda")
    pool = s.pool.clone()
    A.dsv4_kv_store(s.k[:0], s.req_rows[:0], s.positions[:0], A.make_pool(pool, s.page_table))
    torch.cuda.synchronize()
    assert A.dsv4_attn_get_device_error() == 0
    assert torch.equal(pool, s.pool)


def test_store_then_attend(A):
    # verify step over a packed-FP8 cache: the 4 newest positions of every
    # request are first written by the cache writer, then attended
    work = synth.Workload("store_attend", batch=6, heads=64, ratio=4, seq_lens=(1000, 5000, 300, 12000, 700, 9000),
                          qlen=4, kv_format="fp8", seed=31)
    inp_cpu = synth.make_inputs(work)
    pool0 = _bits(inp_cpu.swa_pool).copy()                      # the cache before the write
    inp = inp_cpu.to("cuda")
    g = torch.Generator(device="cuda").manual_seed(7)
    T = inp.T
    k_new = (torch.randn(T, 512, generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    seq = inp.seq_lens.tolist()
    req = torch.tensor([b for b in range(work.batch) for _ in range(4)], dtype=torch.int32, device="cuda")
    pos = torch.tensor([seq[b] - 4 + i for b in range(work.batch) for i in range(4)], dtype=torch.int32,
                       device="cuda")
    A.dsv4_kv_store(k_new, req, pos, A.make_pool(inp.swa_pool, inp.swa_page_table))
    out, lse = A.run_inputs(inp)
    torch.cuda.synchronize()
    assert A.dsv4_attn_get_device_error() == 0
    kw = inp.oracle_kwargs()
    kw["swa_pool"], err = O.kv_store(pool0, _bits(k_new), req.cpu().numpy(), pos.cpu().numpy(),
                                     inp.swa_page_table.cpu().numpy(), "fp8")
    assert err == 0
    assert np.array_equal(kw["swa_pool"], _bits(inp.swa_pool))
    res = O.dsv4_attention(**kw)
    assert res.errors == 0
    e = np.abs(out.float().cpu().numpy() - res.out)
    assert e.max() <= 3e-2, e.max()
    assert np.abs(lse.cpu().numpy() - res.lse).max() <= 1e-3
