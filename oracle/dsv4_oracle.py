"""Float64 CPU oracle for the DeepSeek-V4 hybrid sparse MQA attention step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes this module: it exists so that tests, the smoke check and the CPU
baseline leg of the benchmark can state what the step must compute.  It shares
no code, constants or helpers with the CUDA library; it reads the same seeded
inputs (as numpy arrays) and nothing else.

What the step computes (one query token t, its H query heads, one shared KV
head of 512 values per key row, K and V being the same row):

    keys(t) = SWA window of t  ++  extra compressed rows of t
    s_j     = scale * <q[t, h, :], k_j>
    L       = exp(sink_h) + sum_j exp(s_j)
    out     = sum_j exp(s_j) * k_j / L
    lse     = ln L

Sources (page title, section):
  * "SGLang DeepSeek-V4 Attention Test Capability Matrix" (trdm.cn),
    "Input And Config Coverage": head_dim 512 = 448 nope + 64 rope, page_size
    256, SWA window 128, packed FP8 nope + BF16 rope KV;
    "Reference Implementation Notes": the reference is a vanilla softmax over
    the gathered K rows; the attention sink is a virtual key whose score is the
    per-head attn_sink value and whose value vector is zero, so -1e30 makes it
    a no-op.
  * "DeepSeek-V4 Attention: Query, Cache Write and History Addressing"
    (akiyangdev.github.io), section 1: MQA with one KV head, positions count
    from zero (position 6 -> sequence length 7); section 3: the current token
    is written to the SWA cache before attention and the backend passes k=v;
    section 4: req_pool_indices map a batch row to its request row, and
    cu_seqlens_q delimits each request's query rows; section 5: compress ratio
    0 reads SWA only, 4 adds the indexer's top-k compressed rows, 128 adds all
    compressed rows with no top-k; section 6: the output goes on to
    inverse-RoPE, so V keeps all 512 dims.
  * "DeepSeek-V4 and SGLang Day-0" (yhxrc.cn), "What V4 changed": every layer
    pairs a 128-token sliding window with C4 (4:1 compression, top-512 sparse)
    or C128 (128:1 compression, dense).

The oracle also states the cache write that precedes the step: a new key row
(512 bf16 values after RoPE) is stored at its request's slot of a paged pool,
packed to FP8 when the pool holds packed rows ("DeepSeek-V4 Attention: Query,
Cache Write and History Addressing", section 3: the current token's
representation is written into its SWA slot before the attention backend
reads the cache; "SGLang DeepSeek-V4 Attention Test Capability Matrix",
"Input And Config Coverage" and "Reference Implementation Notes": the
production pack-and-store path writes packed FP8 nope + BF16 rope rows, 584
bytes per token, into the SWA and extra pools).

It also states the top-k selection that produces the C4 index lists: for each
query token, the indices of the k best of its indexer scores ("DeepSeek-V4 and
SGLang Day-0", kernel list: at 1M context the indexer keeps the top 512 of
256K candidate compressed rows, done by a radix select).

Readings where the pages are silent (each is also listed in the design notes):
  R1 the current token is inside its own window: keys are positions
     max(0, p - window + 1) .. p;
  R2 the window and the compressed set are both attended, with no dedup;
  R3 a token at position p sees n_c(p) = (p + 1) // ratio compressed rows;
  R4 C4 indices are logical per-request compressed-row numbers, resolved
     through the extra page table with 256 rows per page; a negative index is
     an absent slot; an index >= n_c(p), or a page id outside the pool, is an
     invalid slot: it is skipped and reported;
  R5 the sink is a raw logit (not multiplied by scale);
  R6 lse is the natural log of the full denominator, sink included;
  R7 packed FP8 rows are [448 e4m3 nope][64 bf16 rope][7 fp32 scales], one
     scale per 64 nope values, stride 608 bytes;
  R8 e4m3 is the OCP FP8 E4M3 format (bias 7, subnormals, no infinities,
     S.1111.111 is NaN).
  R9 in a verify (or extend) call, request b's query rows are its last
     qlen_b positions, in order, and each sees keys up to its own position
     ("DeepSeek-V4 Attention: Query, Cache Write and History Addressing",
     section 4: cu_seqlens and positions);
  R10 req_pool_indices maps a batch row to its page-table row (same page,
     section 4, req_pool_indices = [5, 9]); without it the map is the
     identity;
  R11 the result is unique up to rounding: only the order of the sums is
     free;
  R12 the softmax scale is 1 / sqrt(512), the head dimension.
  R13 the packer's scale of a 64-value nope block is amax / 448 in float32
     (1 when the block is all zero) and each code is the e4m3 value nearest
     to value / scale in float32 (ties to even; beyond 448 it saturates); the
     quantisation decision is taken in float32, the precision the writer
     computes in;
  R14 a new row goes to pool row page_table[r][i // 256] * 256 + i % 256 of
     its request row r, where i is its logical row number (the token position
     for the SWA pool, the compressed-row number for an extra pool); a row
     whose request row, logical page or physical page is outside the tables
     or the pool is not written and is reported.
  R15 top-k selection: scores are float32; a row's candidates are its first
     `length` scores; they are ranked by value (-0 below +0, inputs finite),
     equal values by lower index first; the output is the k best indices in
     ascending index order, padded with -1 when length < k.

Parity pins: every function here is pinned by the CPU tests against something
other than itself (closed forms, brute force, textbook softmax, library e4m3
decode, the pages' worked request-mapping example); no function is unpinned.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# Page size of every paged pool ("Input And Config Coverage": page_size 256 is
# hard-asserted by the backend).
PAGE_SIZE = 256
HEAD_DIM = 512
NOPE_DIM = 448
ROPE_DIM = 64
FP8_BLOCK = 64
FP8_ROW_BYTES = 608

# Error bits the oracle reports (same meaning the library documents; the values
# are restated here, not shared).
ERR_SWA_PAGE = 1
ERR_EXTRA_PAGE = 2
ERR_INDEX_RANGE = 4
ERR_TOKEN_POSITION = 8
ERR_STORE_ROW = 128


# --------------------------------------------------------------------------
# Request coordinates
# --------------------------------------------------------------------------
def token_coordinates(seq_lens, cu_seqlens_q=None):
    """Return (request row, 0-based position) for every packed query token.

    Decode (cu_seqlens_q is None): token b belongs to request b and sits at
    position seq_lens[b] - 1 ("DeepSeek-V4 Attention: Query, Cache Write and
    History Addressing", section 1: positions=[6,6] with seq_lens=[7,7]).

    Verify / extend: cu_seqlens_q[b] .. cu_seqlens_q[b+1] are request b's query
    rows (section 4: extend lengths [6,3] give [0,6,9]); they are the last
    qlen_b positions of the request, so row i sits at
    seq_lens[b] - qlen_b + (i - cu_seqlens_q[b]).
    """
    seq_lens = [int(x) for x in np.asarray(seq_lens).reshape(-1)]
    if cu_seqlens_q is None:
        reqs = list(range(len(seq_lens)))
        pos = [s - 1 for s in seq_lens]
        return np.array(reqs, dtype=np.int64), np.array(pos, dtype=np.int64)
    cu = [int(x) for x in np.asarray(cu_seqlens_q).reshape(-1)]
    reqs, pos = [], []
    for b in range(len(seq_lens)):
        qlen = cu[b + 1] - cu[b]
        for i in range(qlen):
            reqs.append(b)
            pos.append(seq_lens[b] - qlen + i)
    return np.array(reqs, dtype=np.int64), np.array(pos, dtype=np.int64)


def physical_row(page_table, req_row, logical, num_pages):
    """Pool row holding logical row `logical` of request row `req_row`.

    A page table row lists the physical page of each logical page; a page holds
    PAGE_SIZE consecutive logical rows.  Returns -1 when the page id is not a
    page of the pool (or the logical page is past the table's width).
    """
    lp = logical // PAGE_SIZE
    if lp < 0 or lp >= page_table.shape[1]:
        return -1
    page = int(page_table[req_row, lp])
    if page < 0 or page >= num_pages:
        return -1
    return page * PAGE_SIZE + (logical % PAGE_SIZE)


def swa_positions(pos, window):
    """Window keys of a token at position pos (reading R1): the last `window`
    positions up to and including pos ("DeepSeek-V4 and SGLang Day-0", "What
    V4 changed": a 128-token sliding window)."""
    first = max(0, pos - window + 1)
    return list(range(first, pos + 1))


def visible_compressed(pos, ratio):
    """Number of compressed rows a token at position pos can see (reading R3)."""
    return (pos + 1) // ratio


@dataclass
class Resolved:
    """Rows one token attends to, in slot order: window slots, then extra."""
    rows: list = field(default_factory=list)      # physical row or -1 per slot
    from_extra: list = field(default_factory=list)  # slot belongs to the extra pool
    errors: int = 0


def resolve_token(b, pos, *, window, ratio, swa_page_table, swa_num_pages,
                  extra_page_table=None, extra_num_pages=0, topk_row=None):
    """Resolve one token's key slots to physical pool rows.

    Window slots come from the SWA page table; extra slots come from the
    compressed pool's page table: C4 takes the token's given index list
    (section 5: the indexer's top-k indices limit the compressed-side reads),
    C128 takes every visible compressed row (cmp_sparse_indices is None).
    """
    res = Resolved()
    if pos < 0:
        res.errors |= ERR_TOKEN_POSITION
        return res
    for j in swa_positions(pos, window):
        r = physical_row(swa_page_table, b, j, swa_num_pages)
        if r < 0:
            res.errors |= ERR_SWA_PAGE
        res.rows.append(r)
        res.from_extra.append(False)
    if ratio == 0:
        return res
    n_c = visible_compressed(pos, ratio)
    if ratio == 4:
        idx_list = [int(x) for x in topk_row]
    elif ratio == 128:
        idx_list = list(range(n_c))
    else:
        raise ValueError(f"invalid compress ratio {ratio}")
    for idx in idx_list:
        if idx < 0:
            r = -1                       # absent slot: not an error
        elif idx >= n_c:
            r = -1
            res.errors |= ERR_INDEX_RANGE
        else:
            r = physical_row(extra_page_table, b, idx, extra_num_pages)
            if r < 0:
                res.errors |= ERR_EXTRA_PAGE
        res.rows.append(r)
        res.from_extra.append(True)
    return res


# --------------------------------------------------------------------------
# Exact widening of stored values
# --------------------------------------------------------------------------
def bf16_bits_to_f64(bits):
    """bf16 bit patterns (uint16) -> float64, exactly: a bf16 value is the top
    half of the float32 with the same sign, exponent and leading mantissa bits."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def e4m3_to_f64(codes):
    """OCP FP8 E4M3 codes (uint8) -> float64 (reading R8).

    Layout S.EEEE.MMM, exponent bias 7.  E = 0 encodes subnormals
    M/8 * 2^(1-7); E = 15 with M = 7 is NaN; every other code is
    (1 + M/8) * 2^(E-7).  The largest finite value is 448.
    """
    codes = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(codes & 0x80, -1.0, 1.0)
    e = (codes >> 3) & 0xF
    m = codes & 0x7
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** (1 - 7)
    val = np.where(e == 0, sub, normal) * sign
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return val.astype(np.float64)


def unpack_fp8_rows(raw):
    """Packed FP8 KV rows (uint8 [n, >= 604]) -> float64 [n, 512] (reading R7).

    Bytes 0..447 are e4m3 nope values, bytes 448..575 are 64 little-endian
    bf16 rope values, bytes 576..603 are 7 little-endian float32 scales; nope
    value d is e4m3(byte d) * scale[d // 64] ("Input And Config Coverage":
    packed FP8 nope + BF16 rope).
    """
    raw = np.ascontiguousarray(np.asarray(raw, dtype=np.uint8))
    n = raw.shape[0]
    nope = e4m3_to_f64(raw[:, :NOPE_DIM])
    scales = raw[:, NOPE_DIM + 2 * ROPE_DIM: NOPE_DIM + 2 * ROPE_DIM + 4 * (NOPE_DIM // FP8_BLOCK)]
    scales = np.ascontiguousarray(scales).view('<f4').astype(np.float64).reshape(n, NOPE_DIM // FP8_BLOCK)
    nope = nope * np.repeat(scales, FP8_BLOCK, axis=1)
    rope_bits = np.ascontiguousarray(raw[:, NOPE_DIM:NOPE_DIM + 2 * ROPE_DIM]).view('<u2')
    rope = bf16_bits_to_f64(rope_bits)
    return np.concatenate([nope, rope], axis=1)


def e4m3_from_f32(x):
    """float32 values -> OCP FP8 E4M3 codes (uint8), rounding to nearest with
    ties to even and saturating to +-448 (readings R8, R13).

    A magnitude a >= 2^-6 is normal: a = (1 + m/8) * 2^e with the 3-bit
    mantissa m = round((a / 2^e - 1) * 8); a carry (m = 8) moves to the next
    binade.  Below 2^-6 the step is 2^-9 and the code is round(a / 2^-9)
    (a result of 8 is the smallest normal, code 8).  Values past 448 after
    rounding become 448.  The sign is the sign bit of the input (so -0.0 and
    negative values that round to zero give 0x80).  NaN gives 0x7F.
    """
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).astype(np.float64)
    sign = np.where(np.signbit(x), 0x80, 0x00).astype(np.int64)
    fin = np.where(np.isfinite(a), a, 1.0)
    _, ex = np.frexp(fin)                        # fin = f * 2^ex, f in [0.5, 1)
    e = ex.astype(np.int64) - 1                  # fin in [2^e, 2^(e+1))
    m = np.rint((fin / np.exp2(e.astype(np.float64)) - 1.0) * 8.0).astype(np.int64)
    carry = m == 8
    e = np.where(carry, e + 1, e)
    m = np.where(carry, 0, m)
    normal_code = ((e + 7) << 3) | m
    sub_code = np.rint(np.minimum(fin, 1.0) / 2.0 ** -9).astype(np.int64)   # 0 .. 8 below 2^-6
    code = np.where(a >= 2.0 ** -6, normal_code, sub_code)
    code = np.where((a >= 2.0 ** -6) & ((e > 8) | ((e == 8) & (m == 7))), 0x7E, code)
    code = np.where(np.isinf(a), 0x7E, code)
    code = code | sign
    code = np.where(np.isnan(a), 0x7F, code)
    return code.astype(np.uint8)


def pack_fp8_rows(bits):
    """bf16 rows (uint16 bit patterns [n, 512]) -> packed FP8 rows (uint8
    [n, 608]) in the layout of reading R7, quantised as reading R13.

    Per 64-value nope block b: amax = max |x|, scale = amax / 448 in float32
    (1.0 for an all-zero block), code = e4m3(x / scale) in float32.  The 64
    rope values keep their bf16 bits; the 7 scales are stored as float32;
    bytes 604..607 are zero.
    """
    bits = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    n = bits.shape[0]
    x = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)        # exact
    nope = x[:, :NOPE_DIM].reshape(n, NOPE_DIM // FP8_BLOCK, FP8_BLOCK)
    amax = np.max(np.abs(nope), axis=2)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    codes = e4m3_from_f32((nope / scale[:, :, None]).astype(np.float32))
    out = np.zeros((n, FP8_ROW_BYTES), dtype=np.uint8)
    out[:, :NOPE_DIM] = codes.reshape(n, NOPE_DIM)
    out[:, NOPE_DIM:NOPE_DIM + 2 * ROPE_DIM] = bits[:, NOPE_DIM:].astype("<u2").view(np.uint8)
    out[:, NOPE_DIM + 2 * ROPE_DIM:NOPE_DIM + 2 * ROPE_DIM + 4 * (NOPE_DIM // FP8_BLOCK)] = \
        scale.astype("<f4").view(np.uint8).reshape(n, 4 * (NOPE_DIM // FP8_BLOCK))
    return out


def kv_store(pool, bits, req_rows, positions, page_table, kv_format):
    """Write new key rows into a paged pool (readings R7, R13, R14).

    pool: uint16 [rows, 512] (bf16) or uint8 [rows, 608] (packed FP8);
    bits: uint16 [n, 512] bf16 bit patterns of the new rows; req_rows[i] is
    the page-table row of row i's request and positions[i] its logical row
    number.  Returns (new pool, OR of ERR_* bits); rows that cannot be placed
    are skipped and reported as ERR_STORE_ROW.
    """
    out = np.array(pool, copy=True)
    bits = np.asarray(bits, dtype=np.uint16)
    if kv_format == "fp8":
        packed = pack_fp8_rows(bits)
    elif kv_format != "bf16":
        raise ValueError(f"unknown kv format {kv_format}")
    num_pages = out.shape[0] // PAGE_SIZE
    errors = 0
    for i in range(bits.shape[0]):
        r = int(req_rows[i])
        dest = -1
        if 0 <= r < page_table.shape[0]:
            dest = physical_row(page_table, r, int(positions[i]), num_pages)
        if dest < 0:
            errors |= ERR_STORE_ROW
            continue
        out[dest] = packed[i] if kv_format == "fp8" else bits[i]
    return out, errors


def topk_indices(scores, lengths, k):
    """Top-k selection for every row (reading R15).

    scores: float32 [rows, >= max(lengths)]; lengths[r] candidates in row r.
    Returns int32 [rows, k]: for each row, the indices of its k best scores
    (by value, -0.0 ranked below +0.0, ties to the lower index), in
    ascending index order, then -1 padding.
    """
    scores = np.asarray(scores, dtype=np.float32)
    out = np.full((scores.shape[0], k), -1, dtype=np.int32)
    for r in range(scores.shape[0]):
        n = int(lengths[r])
        row = scores[r, :n]
        # the plain definition: sort the candidates by (value descending,
        # index ascending) and keep the first k; -0.0 sorts below +0.0
        order = sorted(range(n), key=lambda i: (-float(row[i]), 0 if np.signbit(row[i]) and row[i] == 0 else -1, i))
        best = sorted(order[:k])
        out[r, :len(best)] = best
    return out


def pool_rows_f64(pool, rows, kv_format):
    """Widen the given physical rows of a pool to float64 [len(rows), 512]."""
    rows = np.asarray(rows, dtype=np.int64)
    if kv_format == "bf16":
        return bf16_bits_to_f64(pool[rows])
    if kv_format == "fp8":
        return unpack_fp8_rows(pool[rows])
    raise ValueError(f"unknown kv format {kv_format}")


# --------------------------------------------------------------------------
# Attention with a sink
# --------------------------------------------------------------------------
def attend(q, keys, sink, scale):
    """Softmax attention of H heads over n shared key rows, with a sink.

    q [H, D], keys [n, D] (also the values), sink [H]: float64.
    The sink is an extra key with score sink[h] and a zero value
    ("Reference Implementation Notes", attention-sink correction), so it adds
    exp(sink[h]) to the denominator only.  Max-shifted in float64.
    Returns out [H, D] and lse [H] (natural log, sink included).
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64).reshape(-1, q.shape[1])
    sink = np.asarray(sink, dtype=np.float64)
    if keys.shape[0] == 0:
        return np.zeros_like(q), sink.copy()
    s = scale * (q @ keys.T)                                  # [H, n]
    m = np.maximum(s.max(axis=1), sink)                       # [H]
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m[:, None])
    denom = np.exp(sink - m) + e.sum(axis=1)
    out = (e @ keys) / denom[:, None]
    lse = m + np.log(denom)
    return out, lse


# --------------------------------------------------------------------------
# The whole step
# --------------------------------------------------------------------------
@dataclass
class OracleResult:
    out: np.ndarray          # [T, H, D] float64
    lse: np.ndarray          # [T, H] float64
    rows: list               # per token: list of physical rows (-1 = skipped)
    errors: int              # OR of the ERR_* bits met


def dsv4_attention(q_bits, sink, scale, seq_lens, *, window, swa_pool, swa_page_table,
                   kv_format="bf16", compress_ratio=0, extra_pool=None,
                   extra_page_table=None, topk_idx=None, cu_seqlens_q=None,
                   req_pool_indices=None, tokens=None):
    """Hybrid sparse MQA attention for packed query tokens.

    q_bits: uint16 [T, H, 512] bf16 bit patterns.  sink: float32 [H].
    swa_pool / extra_pool: uint16 [rows, 512] (bf16) or uint8 [rows, 608]
    (packed FP8).  Page tables: int32 [request rows, pages].  topk_idx: int32
    [T, topk] for compress_ratio 4.  req_pool_indices (optional) maps batch row
    b to its page-table row (section 4: req_pool_indices=[5,9]).
    tokens: optional subset of token ids to evaluate (the rest stay zero).
    """
    if compress_ratio not in (0, 4, 128):
        raise ValueError(f"invalid compress ratio {compress_ratio}")
    q_bits = np.asarray(q_bits)
    T, H, D = q_bits.shape
    reqs, poss = token_coordinates(seq_lens, cu_seqlens_q)
    if len(reqs) != T:
        raise ValueError("token count does not match cu_seqlens_q / seq_lens")
    sink64 = np.asarray(sink, dtype=np.float32).astype(np.float64)
    out = np.zeros((T, H, D), dtype=np.float64)
    lse = np.zeros((T, H), dtype=np.float64)
    rows_all = [[] for _ in range(T)]
    errors = 0
    swa_np = swa_pool.shape[0] // PAGE_SIZE
    ex_np = 0 if extra_pool is None else extra_pool.shape[0] // PAGE_SIZE
    sel = range(T) if tokens is None else tokens
    for t in sel:
        b = int(reqs[t])
        table_row = b if req_pool_indices is None else int(req_pool_indices[b])
        res = resolve_token(
            table_row, int(poss[t]), window=window, ratio=compress_ratio,
            swa_page_table=swa_page_table, swa_num_pages=swa_np,
            extra_page_table=extra_page_table, extra_num_pages=ex_np,
            topk_row=None if topk_idx is None else topk_idx[t])
        errors |= res.errors
        rows_all[t] = res.rows
        swa_rows = [r for r, x in zip(res.rows, res.from_extra) if not x and r >= 0]
        ext_rows = [r for r, x in zip(res.rows, res.from_extra) if x and r >= 0]
        parts = []
        if swa_rows:
            parts.append(pool_rows_f64(swa_pool, swa_rows, kv_format))
        if ext_rows:
            parts.append(pool_rows_f64(extra_pool, ext_rows, kv_format))
        keys = np.concatenate(parts, axis=0) if parts else np.zeros((0, D))
        qf = bf16_bits_to_f64(q_bits[t])
        out[t], lse[t] = attend(qf, keys, sink64, scale)
    return OracleResult(out=out, lse=lse, rows=rows_all, errors=errors)
