"""Checks that tie the float64 oracle to things other than itself.

Each pin_* function raises AssertionError when the oracle disagrees with a
closed form, a brute-force evaluation, a library routine, or the worked
request-mapping example printed on "DeepSeek-V4 Attention: Query, Cache Write
and History Addressing" (sections 1 and 4).  The pins are plain functions so
that the mutation tests can run all of them against a deliberately broken
oracle and see at least one fail.
"""
from __future__ import annotations

import math
import os
from dataclasses import replace

import numpy as np
import scipy.special
import torch

from oracle import dsv4_oracle as O
from hybrid_sparse_mqa_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers
def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = line.split("=", 1)
            vals[k.strip()] = [int(x) for x in v.split()]
    return vals


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    assert err <= tol * scale, f"{what}: max err {err:.3e} > {tol:.1e}"


def _torch_bf16_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _torch_fp8_rows_to_f64(raw):
    """Library decode of packed rows: torch's float8_e4m3fn widening for the
    codes, numpy byte views for the scales and rope."""
    raw = np.ascontiguousarray(raw)
    n = raw.shape[0]
    codes = torch.from_numpy(raw[:, :448].copy()).view(torch.float8_e4m3fn).double().numpy()
    scales = raw[:, 576:604].copy().view("<f4").astype(np.float64)
    nope = codes * np.repeat(scales, 64, axis=1)
    rope = _torch_bf16_to_f64(raw[:, 448:576].copy().view("<u2"))
    return np.concatenate([nope, rope], axis=1).reshape(n, 512)


def small_inputs(kind, *, kv_format="bf16", qlen=1, seed=0, heads=2, seq_lens=None):
    """Tiny inputs that still cross a page boundary and the window edge."""
    base = dict(swa=0, c4=4, c128=128)[kind]
    if seq_lens is None:
        seq_lens = dict(swa=(300, 7, 257), c4=(700, 515, 90), c128=(640, 255, 129))[kind]
    return synth.make_inputs(
        synth.Workload(f"pin_{kind}", batch=len(seq_lens), heads=heads, ratio=base,
                       seq_lens=tuple(seq_lens), qlen=qlen, topk=16, kv_format=kv_format,
                       decoy_pages=2, seed=seed),
        device="cpu")


def run_oracle(inp, **kw):
    args = inp.oracle_kwargs()
    args.update(kw)
    return O.dsv4_attention(**args)


# ------------------------------------------------------- brute force
def brute_force_token(inp, t, heads=None):
    """Dense attention over the request's whole logical history with an
    explicit boolean mask, in pure Python floats.  Independent of the oracle:
    coordinates are re-derived, pages are walked forwards (physical page ->
    logical rows), stored values are widened by torch."""
    kw = inp.oracle_kwargs()
    seq = [int(x) for x in kw["seq_lens"]]
    cu = kw["cu_seqlens_q"]
    # request and position of token t
    if cu is None:
        b, p = t, seq[t] - 1
    else:
        b = max(i for i in range(len(seq)) if int(cu[i]) <= t)
        qlen = int(cu[b + 1]) - int(cu[b])
        p = seq[b] - qlen + (t - int(cu[b]))
    row = b if kw["req_pool_indices"] is None else int(kw["req_pool_indices"][b])
    ratio, window = kw["compress_ratio"], kw["window"]

    def widen(pool, rows):
        if kw["kv_format"] == "bf16":
            return _torch_bf16_to_f64(pool[rows])
        return _torch_fp8_rows_to_f64(pool[rows])

    def forward_map(table):
        m = {}
        for lp, page in enumerate(table[row]):
            if page >= 0:
                for off in range(256):
                    m[lp * 256 + off] = int(page) * 256 + off
        return m

    keys, mask = [], []
    swa_map = forward_map(kw["swa_page_table"])
    for j in range(0, p + 1):
        keys.append(("swa", swa_map[j]) if (p - j) < window else None)
        mask.append((p - j) < window)
    if ratio:
        ex_map = forward_map(kw["extra_page_table"])
        n_total = seq[b] // ratio
        chosen = None
        if ratio == 4:
            chosen = {int(x) for x in kw["topk_idx"][t] if int(x) >= 0}
        for i in range(n_total):
            visible = (i + 1) * ratio <= p + 1
            on = visible and (chosen is None or i in chosen)
            keys.append(("ex", ex_map[i]) if on else None)
            mask.append(on)
    vals = []
    for k, on in zip(keys, mask):
        if not on:
            continue
        pool = kw["swa_pool"] if k[0] == "swa" else kw["extra_pool"]
        vals.append(widen(pool, [k[1]])[0].tolist())
    qv = _torch_bf16_to_f64(kw["q_bits"][t])
    H = qv.shape[0]
    heads = range(H) if heads is None else heads
    scale = kw["scale"]
    sink = [float(np.float32(x)) for x in kw["sink"]]
    out, lse = {}, {}
    for h in heads:
        qh = qv[h].tolist()
        logits = [scale * sum(a * c for a, c in zip(qh, v)) for v in vals]
        mx = max(logits + [sink[h]])
        w = [math.exp(x - mx) for x in logits]
        den = sum(w) + math.exp(sink[h] - mx)
        out[h] = [sum(w[j] * vals[j][d] for j in range(len(vals))) / den for d in range(512)]
        lse[h] = mx + math.log(den)
    return out, lse, len(vals)


# ------------------------------------------------------------ pins
def pin_e4m3_spec():
    v = O.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    assert v[0x00] == 0.0 and v[0x80] == 0.0 and math.copysign(1, v[0x80]) < 0
    assert v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9
    assert v[0x08] == 2.0 ** -6
    assert v[0x38] == 1.0 and v[0x3C] == 1.5 and v[0xB8] == -1.0
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert math.isnan(v[0x7F]) and math.isnan(v[0xFF])
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(v))
    assert np.array_equal(ref[~nan], v[~nan])


def pin_bf16_exact():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint32).astype(np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]          # drop inf / NaN patterns
    assert np.array_equal(O.bf16_bits_to_f64(bits), _torch_bf16_to_f64(bits))


def pin_fp8_unpack_closed_form():
    raw = np.zeros((1, 608), dtype=np.uint8)
    raw[0, :448] = 0x38                                   # e4m3 1.0
    raw[0, 576:604] = np.arange(1, 8, dtype="<f4").view(np.uint8)
    raw[0, 448:576] = np.full(64, 0xBF80, dtype="<u2").view(np.uint8)   # bf16 -1.0
    got = O.unpack_fp8_rows(raw)[0]
    want = np.concatenate([np.repeat(np.arange(1, 8, dtype=np.float64), 64), -np.ones(64)])
    assert np.array_equal(got, want)


def pin_fp8_unpack_roundtrip():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(64, 512, generator=g) * 0.5).to(torch.bfloat16)
    raw = O.pack_fp8_rows(x.view(torch.int16).numpy().view(np.uint16))
    got = O.unpack_fp8_rows(raw)
    xf = x.double().numpy()
    scales = raw[:, 576:604].copy().view("<f4").astype(np.float64)
    step = np.repeat(scales, 64, axis=1)
    err = np.abs(got[:, :448] - xf[:, :448])
    # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 for normals, absolute
    # error <= half the subnormal step 2^-10 * scale below the normal range
    assert np.all(err <= np.abs(xf[:, :448]) * 2.0 ** -4 + step * 2.0 ** -10 + 1e-300)
    assert np.array_equal(got[:, 448:], xf[:, 448:])
    assert np.array_equal(got, _torch_fp8_rows_to_f64(raw))


def _torch_e4m3(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def _torch_pack_fp8(bits):
    """The packer of reading R13 written with torch's float32 arithmetic and
    its float8_e4m3fn cast (which rounds to nearest even; no value here
    reaches its NaN range at 464 and above)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    n = bits.shape[0]
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float()
    nope = x[:, :448].reshape(n, 7, 64)
    amax = nope.abs().amax(dim=2)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    out = np.zeros((n, 608), dtype=np.uint8)
    out[:, :448] = (nope / scale[:, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(n, 448).numpy()
    out[:, 448:576] = bits[:, 448:].view(np.uint8).reshape(n, 128)
    out[:, 576:604] = scale.numpy().astype("<f4").view(np.uint8).reshape(n, 28)
    return out


def _bf16_bits(x):
    """float32 values that are exact in bf16 -> their bf16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert np.all((x.view(np.uint32) & 0xFFFF) == 0)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def pin_e4m3_encode_library():
    # every finite bf16 value below the saturation edge, random float32 values
    # over the whole range, and the exact midpoints between neighbouring e4m3
    # values (ties go to the even code), against torch's float8_e4m3fn cast
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = (b.astype(np.uint32) << np.uint32(16)).view(np.float32)
    parts = [f[np.isfinite(f)]]
    rng = np.random.default_rng(7)
    parts.append((rng.standard_normal(20000) * np.exp2(rng.uniform(-14, 9, 20000))).astype(np.float32))
    dec = O.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))          # 0 .. 448, increasing
    mids = (dec[:-1] + dec[1:]) / 2
    assert np.array_equal(mids.astype(np.float32).astype(np.float64), mids)   # exact in float32
    parts += [mids.astype(np.float32), -mids.astype(np.float32)]
    x = np.concatenate(parts)
    x = x[np.abs(x) < 464]
    assert np.array_equal(O.e4m3_from_f32(x), _torch_e4m3(x))


def pin_e4m3_encode_closed_form():
    codes = np.arange(256, dtype=np.uint8)
    finite = (codes & 0x7F) != 0x7F
    vals = O.e4m3_to_f64(codes[finite]).astype(np.float32)
    assert np.array_equal(O.e4m3_from_f32(vals), codes[finite])       # each finite code encodes its value
    sat = np.array([464.0, 470.0, 1.0e6, np.inf, -500.0, -np.inf], dtype=np.float32)
    assert O.e4m3_from_f32(sat).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert O.e4m3_from_f32(np.array([np.nan], dtype=np.float32)).tolist() == [0x7F]
    # half the smallest subnormal rounds to (signed) zero, 1.5 of it to 2 steps
    tiny = np.array([2.0 ** -10, -2.0 ** -10, 1.5 * 2.0 ** -9], dtype=np.float32)
    assert O.e4m3_from_f32(tiny).tolist() == [0x00, 0x80, 0x02]


def pin_fp8_pack_closed_form():
    # block b < 6 holds 448 * 2^-b and -224 * 2^-b: scale 2^-b exactly, codes
    # 0x7E (448) and 0xF6 (-224); block 6 is all zero: scale 1, codes 0; the
    # rope keeps its bits; the last four bytes are zero
    x = np.zeros((1, 512), dtype=np.float32)
    want = np.zeros(448, dtype=np.uint8)
    for blk in range(6):
        x[0, 64 * blk] = 448.0 * 2.0 ** -blk
        x[0, 64 * blk + 1] = -224.0 * 2.0 ** -blk
        want[64 * blk], want[64 * blk + 1] = 0x7E, 0xF6
    x[0, 448:] = np.arange(-32, 32, dtype=np.float32) / 8.0
    bits = _bf16_bits(x)
    raw = O.pack_fp8_rows(bits)[0]
    assert raw.shape == (608,)
    assert np.array_equal(raw[:448], want)
    assert np.array_equal(raw[448:576], bits[0, 448:].astype("<u2").view(np.uint8))
    assert raw[576:604].copy().view("<f4").tolist() == [1.0, 0.5, 0.25, 0.125, 0.0625, 0.03125, 1.0]
    assert raw[604:].tolist() == [0, 0, 0, 0]


def pin_fp8_pack_library():
    # random rows with blocks of very different magnitudes (down into the
    # subnormal codes), zero blocks and negative zeros, against torch
    g = torch.Generator().manual_seed(11)
    x = torch.randn(96, 512, generator=g) * 0.5
    mag = torch.exp2(torch.randint(-20, 6, (96, 8), generator=g).float())
    x = x * mag.repeat_interleave(64, dim=1)
    x[5, 64:128] = 0.0
    x[6, :] = -0.0
    x[7, 0:64] = torch.tensor([1e-30] + [0.0] * 63)
    bits = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.pack_fp8_rows(bits), _torch_pack_fp8(bits))


def pin_kv_store_round_trip():
    # The worked example's requests (request-pool rows 5 and 9): store the
    # prefill rows and the decode step's new rows, then read every stored
    # position back through the attention oracle (a one-key window and no
    # sink returns that key exactly); rows that cannot be placed are skipped
    # and reported, and nothing else in the pool changes.
    g = _golden("request_mapping.txt")
    rows5, rows9 = g["req_pool_indices"]
    page_table = np.full((10, 4), -1, dtype=np.int32)
    page_table[rows5] = [6, 1, 3, -1]
    page_table[rows9] = [0, 7, -1, 2]
    req, pos = [], []
    for b, p in zip(g["prefill.requests"], g["prefill.positions"]):
        req.append(g["req_pool_indices"][b])
        pos.append(p)
    for b, p in zip(g["decode.requests"], g["decode.positions"]):
        req.append(g["req_pool_indices"][b])
        pos.append(p)
    req += [rows5, rows9, rows9]
    pos += [511, 256, 1000]                       # logical pages 1, 1 and 3
    bad_req = [rows5, rows9, 3, 10, rows5]
    bad_pos = [-1, 520, 0, 0, 1024]               # negative, unmapped page, empty row, no row, past the table
    rng = np.random.default_rng(5)
    n = len(req) + len(bad_req)
    vals = (rng.standard_normal((n, 512)) * 0.5).astype(np.float32)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    req_all = np.array(req + bad_req, dtype=np.int32)
    pos_all = np.array(pos + bad_pos, dtype=np.int32)
    for fmt in ("bf16", "fp8"):
        width = 512 if fmt == "bf16" else 608
        dtype = np.uint16 if fmt == "bf16" else np.uint8
        pool = rng.integers(0, 200, size=(8 * 256, width)).astype(dtype)
        new, err = O.kv_store(pool, bits, req_all, pos_all, page_table, fmt)
        assert err == O.ERR_STORE_ROW
        changed = np.nonzero(np.any(new != pool, axis=1))[0]
        assert len(changed) <= len(req)
        for i, (r, p) in enumerate(zip(req, pos)):
            res = O.dsv4_attention(np.zeros((1, 1, 512), dtype=np.uint16), np.array([-np.inf], np.float32), 1.0,
                                   [p + 1], window=1, swa_pool=new, swa_page_table=page_table, kv_format=fmt,
                                   req_pool_indices=[r])
            want = O.bf16_bits_to_f64(bits[i]) if fmt == "bf16" else O.unpack_fp8_rows(O.pack_fp8_rows(bits[i:i + 1]))[0]
            assert res.errors == 0 and np.array_equal(res.out[0, 0], want), (fmt, r, p)
        _, err = O.kv_store(pool, bits[:len(req)], req_all[:len(req)], pos_all[:len(req)], page_table, fmt)
        assert err == 0


def pin_topk_library():
    # rows without repeated values: the selected set is torch.topk's; rows
    # with repeats: the selected values are torch.topk's (as a multiset)
    g = torch.Generator().manual_seed(23)
    rows, n, k = 6, 3000, 128
    x = torch.randn(rows, n, generator=g)
    x[3] = torch.randint(-20, 20, (n,), generator=g).float()         # many repeats
    x[4, :] = torch.linspace(-3, 3, n)
    lengths = [n, n, 2000, n, n, 700]
    got = O.topk_indices(x.numpy(), lengths, k)
    for r in range(rows):
        m = lengths[r]
        vals, idx = torch.topk(x[r, :m], min(k, m))
        sel = got[r][got[r] >= 0]
        assert list(sel) == sorted(sel) and len(sel) == min(k, m)
        assert np.array_equal(np.sort(x[r, sel].numpy()), np.sort(vals.numpy()))
        if r != 3:
            assert set(sel.tolist()) == set(idx.tolist())


def pin_topk_closed_form():
    # equal scores go to the lower index; fewer candidates than k pad with -1;
    # +0.0 ranks above -0.0; a rising row keeps its last k
    assert O.topk_indices(np.zeros((1, 10), np.float32), [10], 4).tolist() == [[0, 1, 2, 3]]
    assert O.topk_indices(np.ones((1, 10), np.float32), [3], 5).tolist() == [[0, 1, 2, -1, -1]]
    z = np.array([[-0.0, 0.0, -0.0, 0.0, -1.0]], dtype=np.float32)
    assert O.topk_indices(z, [5], 3).tolist() == [[0, 1, 3]]
    assert O.topk_indices(np.arange(50, dtype=np.float32)[None], [50], 5).tolist() == [[45, 46, 47, 48, 49]]
    s = np.array([[0.5, -0.0, 0.0, 2.0, 2.0, -1.0, 0.0, 7.0]], np.float32)
    assert O.topk_indices(s, [8], 4).tolist() == [[0, 3, 4, 7]]
    assert O.topk_indices(s, [8], 6).tolist() == [[0, 2, 3, 4, 6, 7]]
    assert O.topk_indices(s, [0], 2).tolist() == [[-1, -1]]


def pin_token_coordinates_golden():
    g = _golden("request_mapping.txt")
    req, pos = O.token_coordinates(g["decode.seq_lens"])
    assert pos.tolist() == g["decode.positions"] and req.tolist() == g["decode.requests"]
    req, pos = O.token_coordinates(g["decode.seq_lens"], g["decode.cu_seqlens_q"])
    assert pos.tolist() == g["decode.positions"] and req.tolist() == g["decode.requests"]
    cu = np.concatenate([[0], np.cumsum(g["prefill.extend_lens"])]).tolist()
    assert cu == g["prefill.cu_seqlens_q"]
    req, pos = O.token_coordinates(g["prefill.seq_lens"], cu)
    assert pos.tolist() == g["prefill.positions"] and req.tolist() == g["prefill.requests"]


def pin_req_pool_indices_golden():
    g = _golden("request_mapping.txt")
    inp = synth.make_inputs("swa_tiny")            # req_pool_indices = (5, 9)
    assert inp.req_pool_indices.tolist() == g["req_pool_indices"]
    res = run_oracle(inp)
    table = inp.swa_page_table.numpy()
    for b, r in enumerate(g["req_pool_indices"]):
        want = [int(table[r, 0]) * 256 + j for j in range(g["decode.positions"][b] + 1)]
        assert res.rows[b] == want, (b, res.rows[b][:4], want[:4])


def pin_softmax_without_sink():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal((4, 512)), rng.standard_normal((37, 512))
    out, lse = O.attend(q, k, np.full(4, -np.inf), 0.044)
    s = 0.044 * q @ k.T
    _close(out, scipy.special.softmax(s, axis=1) @ k, 1e-12, "softmax")
    _close(lse, scipy.special.logsumexp(s, axis=1), 1e-12, "logsumexp")
    out2, _ = O.attend(q, k, np.full(4, -1e30), 0.044)     # the pages' no-op sink value
    _close(out2, out, 1e-12, "sink -1e30")


def pin_identical_keys_closed_form():
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal((3, 512)), rng.standard_normal(512)
    sink = np.array([0.0, 1.5, -2.0])
    for n in (1, 5, 130):
        out, lse = O.attend(q, np.tile(k, (n, 1)), sink, 0.05)
        s = 0.05 * q @ k
        den = n * np.exp(s) + np.exp(sink)
        _close(out, (n * np.exp(s) / den)[:, None] * k[None, :], 1e-12, f"identical n={n}")
        _close(lse, np.log(den), 1e-12, f"identical lse n={n}")


def pin_attend_brute_force():
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal((3, 8)), rng.standard_normal((5, 8))
    sink = np.array([0.3, -1.0, 2.0])
    out, lse = O.attend(q, k, sink, 0.7)
    for h in range(3):
        e = [math.exp(0.7 * sum(q[h, d] * k[j, d] for d in range(8))) for j in range(5)]
        den = sum(e) + math.exp(sink[h])
        for d in range(8):
            assert abs(out[h, d] - sum(e[j] * k[j, d] for j in range(5)) / den) < 1e-12
        assert abs(lse[h] - math.log(den)) < 1e-12
    out0, lse0 = O.attend(q, np.zeros((0, 8)), sink, 0.7)   # no keys: only the sink
    assert np.all(out0 == 0) and np.array_equal(lse0, sink)


def _pin_step_brute(kind, kv_format, qlen, tokens):
    inp = small_inputs(kind, kv_format=kv_format, qlen=qlen)
    res = run_oracle(inp)
    assert res.errors == 0
    for t in tokens:
        out, lse, n = brute_force_token(inp, t)
        assert n == sum(1 for r in res.rows[t] if r >= 0)
        for h in out:
            _close(res.out[t, h], out[h], 1e-10, f"{kind} t={t} h={h}")
            assert abs(res.lse[t, h] - lse[h]) < 1e-10


def pin_swa_brute():
    _pin_step_brute("swa", "bf16", 1, [0, 1, 2])


def pin_c4_brute():
    _pin_step_brute("c4", "bf16", 1, [0, 1, 2])


def pin_c128_brute():
    _pin_step_brute("c128", "bf16", 1, [0, 1, 2])


def pin_verify_brute():
    _pin_step_brute("c4", "bf16", 3, [0, 2, 4, 8])
    _pin_step_brute("c128", "bf16", 2, [0, 1, 3, 5])


def pin_fp8_brute():
    _pin_step_brute("c4", "fp8", 2, [0, 3])
    _pin_step_brute("swa", "fp8", 1, [2])


def pin_index_permutation_invariance():
    inp = small_inputs("c4", seed=5)
    base = run_oracle(inp)
    g = torch.Generator().manual_seed(6)
    perm = torch.stack([r[torch.randperm(r.shape[0], generator=g)] for r in inp.topk_idx])
    inp2 = replace(inp, topk_idx=perm)
    _close(run_oracle(inp2).out, base.out, 1e-12, "index permutation")


def pin_page_permutation_invariance():
    for kind in ("swa", "c4"):
        inp = small_inputs(kind, seed=7)
        base = run_oracle(inp)
        g = torch.Generator().manual_seed(8)

        def relabel(pool, table):
            n = pool.shape[0] // 256
            perm = torch.randperm(n, generator=g)            # old page -> new page
            newpool = torch.empty_like(pool)
            newpool.view(n, 256, -1)[perm] = pool.view(n, 256, -1)
            t = table.clone()
            t[t >= 0] = perm[t[t >= 0].long()].to(torch.int32)
            return newpool, t
        sp, st = relabel(inp.swa_pool, inp.swa_page_table)
        kw = dict(swa_pool=sp, swa_page_table=st)
        if inp.extra_pool is not None:
            ep, et = relabel(inp.extra_pool, inp.extra_page_table)
            kw.update(extra_pool=ep, extra_page_table=et)
        res = run_oracle(replace(inp, **kw))
        assert np.array_equal(res.out, base.out), kind


def pin_verify_causality():
    inp = small_inputs("c128", qlen=3, seed=9, seq_lens=(400, 260))
    base = run_oracle(inp)
    # request 0's query rows sit at positions 397, 398, 399: overwrite the
    # window row of position 399 and check token 0 and 1 do not move
    table = inp.swa_page_table
    pool = inp.swa_pool.clone()
    prow = int(table[0, 399 // 256]) * 256 + 399 % 256
    pool[prow] = (pool[prow].float() + 3.0).to(pool.dtype)
    res = run_oracle(replace(inp, swa_pool=pool))
    assert np.array_equal(res.out[:2], base.out[:2])
    assert not np.allclose(res.out[2], base.out[2])


def pin_c4_all_rows_equals_dense():
    # request lengths <= 4 * 16 rows so n_c(p) <= topk for ratio 4
    inp = small_inputs("c4", seq_lens=(60, 33), seed=10)
    idx = torch.full_like(inp.topk_idx, -1)
    for t in range(inp.T):
        n_c = int(inp.seq_lens[t]) // 4
        idx[t, :n_c] = torch.arange(n_c, dtype=torch.int32)
    c4 = run_oracle(replace(inp, topk_idx=idx))
    # dense attention over the window rows followed by every compressed row
    kw = inp.oracle_kwargs()
    table = kw["extra_page_table"]
    for t in range(inp.T):
        p = int(inp.seq_lens[t]) - 1
        rows = [int(table[t, i // 256]) * 256 + i % 256 for i in range((p + 1) // 4)]
        win = c4.rows[t][: min(p + 1, 128)]
        keys = np.concatenate([O.bf16_bits_to_f64(kw["swa_pool"][win]),
                               O.bf16_bits_to_f64(kw["extra_pool"][rows])])
        out, lse = O.attend(O.bf16_bits_to_f64(kw["q_bits"][t]), keys,
                            kw["sink"].astype(np.float64), kw["scale"])
        _close(c4.out[t], out, 1e-12, "c4 all rows")
        _close(c4.lse[t], lse, 1e-12, "c4 all rows lse")


def pin_error_reporting():
    inp = small_inputs("c4", seed=11)
    t = inp.swa_page_table.clone()
    t[0, 699 // 256] = inp.swa_pool.shape[0] // 256          # page id past the pool
    idx = inp.topk_idx.clone()
    idx[1, 0] = (515 // 4)                                    # n_c(514) = 128: out of range
    idx[1, 1] = -1                                            # absent: not an error
    res = run_oracle(replace(inp, swa_page_table=t, topk_idx=idx))
    assert res.errors == (O.ERR_SWA_PAGE | O.ERR_INDEX_RANGE)
    assert res.rows[1][min(515, 128)] == -1 and res.rows[1][min(515, 128) + 1] == -1
    ok = run_oracle(inp)
    assert ok.errors == 0


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
