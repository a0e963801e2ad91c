"""Seeded synthetic inputs for the hybrid sparse MQA attention step.

This module only draws random numbers and lays them out the way the step reads
them: query rows, per-head sinks, paged KV pools with their page tables,
sequence lengths, query boundaries and top-k index lists.  It holds none of
the step's arithmetic, so both the CUDA path and the float64 oracle can take
their inputs from it.

Packed FP8 pools are drawn directly in their stored layout (448 e4m3 nope
codes, 64 bf16 rope values, 7 fp32 block scales, 608-byte stride): random
finite e4m3 codes, random positive scales and random bf16 rope values.  No
quantisation happens here; the cache writer that quantises bf16 rows is part
of the library (dsv4_kv_store), and its tests feed it bf16 rows drawn below.

Shapes follow the five workloads of the step:
  swa_tiny       batch 2, seq_lens (7,7), H=8, SWA only
  swa_decode     batch 64, H=64, seq_len uniform 2K..32K, SWA only, all pages
                 resident and randomly permuted
  c4_decode      batch 32, H=64, context 65536 (16384 compressed rows), 512
                 distinct uniform indices per token
  c128_decode    batch 16, H=128, context 1,048,576 (8192 compressed rows, all
                 attended)
  c4_verify_fp8  batch 64 x 4 query tokens, H=64, context 262144, top-512,
                 packed FP8 KV
  c4_prefill     batch 4 x 1024 query tokens (extend chunk), H=64, context
                 65536, top-512
Values: q and KV ~ N(0,1)*0.5 in bf16, sink ~ N(0,1) in fp32,
scale = 1/sqrt(512).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

PAGE = 256
DIM = 512
NOPE = 448
ROPE = 64
BLOCK = 64
FP8_STRIDE = 608


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    ratio: int = 0                 # 0 = SWA only, 4 = C4 top-k, 128 = C128 dense
    window: int = 128
    topk: int = 512
    seq_lens: tuple | None = None  # fixed lengths, else drawn from seq_range
    seq_range: tuple = (0, 0)
    qlen: int = 1                  # query tokens per request (verify when > 1)
    kv_format: str = "bf16"        # "bf16" or "fp8"
    swa_resident: str = "window"   # "window": only pages the window touches; "all"
    req_pool_indices: tuple | None = None
    decoy_pages: int = 4           # unused pool pages with random content
    seed: int = 0

    @property
    def tokens(self):
        return self.batch * self.qlen


PRESETS = {
    "swa_tiny": Workload("swa_tiny", batch=2, heads=8, seq_lens=(7, 7),
                         req_pool_indices=(5, 9), decoy_pages=3, seed=0),
    "swa_decode": Workload("swa_decode", batch=64, heads=64, seq_range=(2048, 32768),
                           swa_resident="all", seed=1),
    "c4_decode": Workload("c4_decode", batch=32, heads=64, ratio=4,
                          seq_lens=(65536,) * 32, seed=2),
    "c128_decode": Workload("c128_decode", batch=16, heads=128, ratio=128,
                            seq_lens=(1048576,) * 16, seed=3),
    "c4_verify_fp8": Workload("c4_verify_fp8", batch=64, heads=64, ratio=4,
                              seq_lens=(262144,) * 64, qlen=4, kv_format="fp8", seed=4),
    # sparse prefill / extend: 4 requests each appending a 1024-token chunk at
    # the end of a 65536-token context, C4 top-512 per query token
    "c4_prefill": Workload("c4_prefill", batch=4, heads=64, ratio=4, seq_lens=(65536,) * 4, qlen=1024, seed=5),
    # small batch x long compressed list: C128 decode of 2 requests at 1M
    # context, whose split plan merges cluster groups with the combine kernel
    "c128_decode_b2": Workload("c128_decode_b2", batch=2, heads=128, ratio=128, seq_lens=(1048576,) * 2, seed=6),
}


@dataclass
class Inputs:
    """One batch of step inputs (torch tensors on one device)."""
    work: Workload
    q: torch.Tensor                     # [T, H, 512] bf16
    sink: torch.Tensor                  # [H] fp32
    seq_lens: torch.Tensor              # [B] int32
    cu_seqlens_q: torch.Tensor | None   # [B+1] int32, None for decode
    req_pool_indices: torch.Tensor | None
    swa_pool: torch.Tensor              # [rows, 512] bf16 or [rows, 608] uint8
    swa_page_table: torch.Tensor        # [R, P] int32
    extra_pool: torch.Tensor | None
    extra_page_table: torch.Tensor | None
    topk_idx: torch.Tensor | None       # [T, topk] int32
    scale: float = 1.0 / math.sqrt(DIM)
    max_seq_len: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def T(self):
        return self.q.shape[0]

    @property
    def H(self):
        return self.q.shape[1]

    def to(self, device):
        def mv(x):
            return None if x is None else x.to(device)
        return replace(self, q=mv(self.q), sink=mv(self.sink), seq_lens=mv(self.seq_lens),
                       cu_seqlens_q=mv(self.cu_seqlens_q),
                       req_pool_indices=mv(self.req_pool_indices),
                       swa_pool=mv(self.swa_pool), swa_page_table=mv(self.swa_page_table),
                       extra_pool=mv(self.extra_pool),
                       extra_page_table=mv(self.extra_page_table),
                       topk_idx=mv(self.topk_idx))

    def oracle_kwargs(self):
        """numpy views of every input, in the oracle's argument names."""
        def np_(x):
            return None if x is None else x.detach().cpu().numpy()
        def bits(x):
            if x is None:
                return None
            x = x.detach().cpu()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16)
            return x.numpy()
        return dict(
            q_bits=bits(self.q), sink=np_(self.sink), scale=self.scale,
            seq_lens=np_(self.seq_lens), window=self.work.window,
            swa_pool=bits(self.swa_pool), swa_page_table=np_(self.swa_page_table),
            kv_format=self.work.kv_format, compress_ratio=self.work.ratio,
            extra_pool=bits(self.extra_pool), extra_page_table=np_(self.extra_page_table),
            topk_idx=np_(self.topk_idx), cu_seqlens_q=np_(self.cu_seqlens_q),
            req_pool_indices=np_(self.req_pool_indices))


# --------------------------------------------------------------------------
def _randn_bf16(shape, gen, device, chunk_rows=1 << 20):
    """N(0,1)*0.5 in bf16, drawn in chunks to bound temporary fp32 memory."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        flat[r0:r1] = (torch.randn((r1 - r0, flat.shape[1]), generator=gen, device=device) * 0.5).to(torch.bfloat16)
    return out


def _pool(num_rows, kv_format, gen, device):
    if kv_format == "bf16":
        return _randn_bf16((num_rows, DIM), gen, device)
    out = torch.empty(num_rows, FP8_STRIDE, dtype=torch.uint8, device=device)
    step = 1 << 18
    for r0 in range(0, num_rows, step):
        r1 = min(num_rows, r0 + step)
        out[r0:r1] = _fp8_rows(r1 - r0, gen, device)
    return out


def _fp8_rows(n, gen, device):
    """n packed FP8 rows: finite e4m3 codes uniform over the 254 non-NaN codes
    (0x7F and 0xFF are skipped), block scales uniform in [0.005, 0.012),
    bf16 rope ~ N(0,1)*0.5, zero padding."""
    out = torch.zeros(n, FP8_STRIDE, dtype=torch.uint8, device=device)
    r = torch.randint(0, 254, (n, NOPE), generator=gen, device=device, dtype=torch.int32)
    out[:, :NOPE] = (r + (r >= 0x7F).to(torch.int32)).to(torch.uint8)
    out[:, NOPE:NOPE + 2 * ROPE] = _randn_bf16((n, ROPE), gen, device).view(torch.uint8).reshape(n, 2 * ROPE)
    scales = 0.005 + 0.007 * torch.rand((n, NOPE // BLOCK), generator=gen, device=device)
    out[:, NOPE + 2 * ROPE:NOPE + 2 * ROPE + 4 * (NOPE // BLOCK)] = \
        scales.float().contiguous().view(torch.uint8).reshape(n, 4 * (NOPE // BLOCK))
    return out


def _page_tables(needed, num_req_rows, width, decoys, gen_cpu):
    """Assign a random distinct physical page to every (request row, logical
    page) in `needed`; pages not needed stay -1.  Returns (table, num_pages)."""
    total = len(needed) + decoys
    perm = torch.randperm(total, generator=gen_cpu).tolist()
    table = torch.full((num_req_rows, max(width, 1)), -1, dtype=torch.int32)
    for k, (r, lp) in enumerate(needed):
        table[r, lp] = perm[k]
    return table, total


def make_inputs(work: Workload | str, device="cpu", seed=None, **overrides) -> Inputs:
    """Draw one batch of inputs for a workload (a preset name or a Workload)."""
    if isinstance(work, str):
        work = PRESETS[work]
    if overrides:
        work = replace(work, **overrides)
    if seed is not None:
        work = replace(work, seed=seed)
    gen_cpu = torch.Generator().manual_seed(work.seed)
    dev = torch.device(device)
    gen_dev = gen_cpu if dev.type == "cpu" else torch.Generator(device=dev).manual_seed(work.seed)

    B, H = work.batch, work.heads
    if work.seq_lens is not None:
        seq = [int(s) for s in work.seq_lens]
        assert len(seq) == B
    else:
        lo, hi = work.seq_range
        seq = torch.randint(lo, hi + 1, (B,), generator=gen_cpu).tolist()
    qlen = work.qlen
    T = B * qlen
    cu = None if qlen == 1 else torch.arange(0, T + 1, qlen, dtype=torch.int32)
    rpi = work.req_pool_indices
    table_rows = [b if rpi is None else rpi[b] for b in range(B)]
    num_req_rows = (max(table_rows) + 1) if table_rows else 1

    # ---- SWA pool: pages covering each request's windows (or every page).
    needed = []
    width = 0
    for b in range(B):
        p_max = seq[b] - 1
        p_min = seq[b] - qlen
        first = 0 if work.swa_resident == "all" else max(0, p_min - work.window + 1) // PAGE
        last = p_max // PAGE
        width = max(width, last + 1)
        needed += [(table_rows[b], lp) for lp in range(first, last + 1)]
    swa_table, swa_pages = _page_tables(needed, num_req_rows, width, work.decoy_pages, gen_cpu)
    swa_pool = _pool(swa_pages * PAGE, work.kv_format, gen_dev, dev)

    # ---- extra (compressed) pool: every compressed row of every request.
    extra_pool = extra_table = topk = None
    if work.ratio:
        needed = []
        width = 0
        for b in range(B):
            n_c = seq[b] // work.ratio
            pages = (n_c + PAGE - 1) // PAGE
            width = max(width, pages)
            needed += [(table_rows[b], lp) for lp in range(pages)]
        extra_table, extra_pages = _page_tables(needed, num_req_rows, width, work.decoy_pages, gen_cpu)
        extra_pool = _pool(extra_pages * PAGE, work.kv_format, gen_dev, dev)
    if work.ratio == 4:
        # the workloads hold valid index lists: a query token at position p
        # draws from the compressed rows of its complete groups of 4 positions
        visible = [(s_ - qlen + i + 1) // 4 for s_ in seq for i in range(qlen)]
        topk = _topk_lists(visible, work.topk, gen_cpu)

    q = _randn_bf16((T, H, DIM), gen_dev, dev)
    sink = torch.randn(H, generator=gen_cpu).float()
    inp = Inputs(work=work, q=q, sink=sink,
                 seq_lens=torch.tensor(seq, dtype=torch.int32),
                 cu_seqlens_q=cu,
                 req_pool_indices=None if rpi is None else torch.tensor(rpi, dtype=torch.int32),
                 swa_pool=swa_pool, swa_page_table=swa_table,
                 extra_pool=extra_pool, extra_page_table=extra_table, topk_idx=topk,
                 max_seq_len=max(seq) if seq else 0)
    return inp.to(dev)


# --------------------------------------------------------------------------
# Cache-write inputs: new key rows for a paged pool
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class StoreWorkload:
    """`requests` requests each receive `rows_per_request` consecutive
    logical rows starting at a random row below `max_len` (a prefill chunk;
    one row per request is a decode step).  Request r uses page-table row
    r * req_row_stride."""
    name: str
    requests: int
    rows_per_request: int
    kv_format: str = "fp8"
    max_len: int = 65536
    req_row_stride: int = 1
    decoy_pages: int = 8
    seed: int = 0

    @property
    def rows(self):
        return self.requests * self.rows_per_request


STORE_PRESETS = {
    "kv_store_tiny": StoreWorkload("kv_store_tiny", requests=3, rows_per_request=341, max_len=4096,
                                   req_row_stride=2, seed=21),
    "kv_store_tiny_bf16": StoreWorkload("kv_store_tiny_bf16", requests=3, rows_per_request=341,
                                        kv_format="bf16", max_len=4096, req_row_stride=2, seed=22),
    "kv_store_prefill": StoreWorkload("kv_store_prefill", requests=64, rows_per_request=1024, seed=23),
    "kv_store_decode": StoreWorkload("kv_store_decode", requests=64, rows_per_request=1, seed=24),
}


@dataclass
class StoreInputs:
    """One batch of new rows and the pool they go to (torch tensors)."""
    work: StoreWorkload
    k: torch.Tensor             # [n, 512] bf16
    req_rows: torch.Tensor      # [n] int32
    positions: torch.Tensor     # [n] int32
    pool: torch.Tensor          # [rows, 608] uint8 or [rows, 512] bf16, random content
    page_table: torch.Tensor    # [R, W] int32

    def to(self, device):
        return replace(self, k=self.k.to(device), req_rows=self.req_rows.to(device),
                       positions=self.positions.to(device), pool=self.pool.to(device),
                       page_table=self.page_table.to(device))

    def oracle_kwargs(self):
        def bits(x):
            x = x.detach().cpu()
            return x.view(torch.int16).numpy().view(np.uint16) if x.dtype == torch.bfloat16 else x.numpy()
        return dict(pool=bits(self.pool), bits=bits(self.k), req_rows=self.req_rows.cpu().numpy(),
                    positions=self.positions.cpu().numpy(), page_table=self.page_table.cpu().numpy(),
                    kv_format=self.work.kv_format)


def make_store_inputs(work: StoreWorkload | str, device="cpu", seed=None) -> StoreInputs:
    """Draw new rows ~ N(0,1)*0.5 in bf16, their request rows and positions,
    and a pool of randomly permuted pages (random content, so that a write
    to the wrong row shows) covering every page the rows land on."""
    if isinstance(work, str):
        work = STORE_PRESETS[work]
    if seed is not None:
        work = replace(work, seed=seed)
    gen_cpu = torch.Generator().manual_seed(work.seed)
    dev = torch.device(device)
    gen_dev = gen_cpu if dev.type == "cpu" else torch.Generator(device=dev).manual_seed(work.seed)
    n_req, per = work.requests, work.rows_per_request
    starts = torch.randint(0, work.max_len - per + 1, (n_req,), generator=gen_cpu).tolist()
    table_rows = [r * work.req_row_stride for r in range(n_req)]
    needed = []
    for r in range(n_req):
        needed += [(table_rows[r], lp) for lp in range(starts[r] // PAGE, (starts[r] + per - 1) // PAGE + 1)]
    table, pages = _page_tables(needed, max(table_rows) + 1, work.max_len // PAGE, work.decoy_pages, gen_cpu)
    pool = _pool(pages * PAGE, work.kv_format, gen_dev, dev)
    req_rows = torch.tensor([table_rows[r] for r in range(n_req) for _ in range(per)], dtype=torch.int32)
    positions = torch.tensor([starts[r] + i for r in range(n_req) for i in range(per)], dtype=torch.int32)
    k = _randn_bf16((work.rows, DIM), gen_dev, dev)
    return StoreInputs(work=work, k=k, req_rows=req_rows, positions=positions, pool=pool,
                       page_table=table).to(dev)


# --------------------------------------------------------------------------
# Top-k selection inputs: indexer scores per query token
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class TopkWorkload:
    """`rows` query tokens, each with `length` candidate scores (or the
    given per-row lengths), fp32 ~ N(0,1); rows listed in `repeat_rows`
    draw their scores from 64 values only, so many scores repeat."""
    name: str
    rows: int
    length: int = 0
    lengths: tuple | None = None
    k: int = 512
    repeat_rows: tuple = ()
    seed: int = 0


TOPK_PRESETS = {
    "topk_tiny": TopkWorkload("topk_tiny", rows=6, lengths=(3000, 700, 512, 100, 2999, 513), k=512,
                              repeat_rows=(4,), seed=41),
    "topk_c4_decode": TopkWorkload("topk_c4_decode", rows=32, length=16384, seed=42),
    "topk_1m": TopkWorkload("topk_1m", rows=32, length=262144, seed=43),
}


@dataclass
class TopkInputs:
    work: TopkWorkload
    scores: torch.Tensor        # [rows, stride] fp32 (stride a multiple of 4)
    lengths: torch.Tensor       # [rows] int32

    def to(self, device):
        return replace(self, scores=self.scores.to(device), lengths=self.lengths.to(device))

    def oracle_kwargs(self):
        return dict(scores=self.scores.cpu().numpy(), lengths=self.lengths.cpu().numpy(), k=self.work.k)


def make_topk_inputs(work: TopkWorkload | str, device="cpu", seed=None) -> TopkInputs:
    if isinstance(work, str):
        work = TOPK_PRESETS[work]
    if seed is not None:
        work = replace(work, seed=seed)
    lengths = list(work.lengths) if work.lengths is not None else [work.length] * work.rows
    stride = max(4, (max(lengths) + 3) // 4 * 4)
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(work.seed) if dev.type != "cpu" else \
        torch.Generator().manual_seed(work.seed)
    scores = torch.randn((work.rows, stride), generator=gen, device=dev, dtype=torch.float32)
    for r in work.repeat_rows:
        scores[r] = torch.randint(-32, 32, (stride,), generator=gen, device=dev).float() / 8.0
    return TopkInputs(work=work, scores=scores, lengths=torch.tensor(lengths, dtype=torch.int32, device=dev))


def _topk_lists(visible, topk, gen_cpu):
    """Per query token: min(topk, n) distinct uniform indices in [0, n),
    unsorted, padded with -1, where n is that token's entry of `visible`
    (the number of compressed rows it may index, given by the caller)."""
    rows = []
    for n_c in visible:
        k = min(topk, n_c)
        if n_c <= 4 * topk:
            pick = torch.randperm(n_c, generator=gen_cpu)[:k]
        else:
            # rejection-free distinct draw: random keys, keep the k largest
            pick = torch.rand(n_c, generator=gen_cpu).topk(k).indices
            pick = pick[torch.randperm(k, generator=gen_cpu)]
        row = torch.full((topk,), -1, dtype=torch.int32)
        row[:k] = pick.to(torch.int32)
        rows.append(row)
    return torch.stack(rows) if rows else torch.zeros((0, topk), dtype=torch.int32)
