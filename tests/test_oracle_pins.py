"""The oracle against its pins, and the pins against plausible oracle mistakes."""
import numpy as np
import pytest

from oracle import dsv4_oracle as O
from tests import _pins


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# Each mutant is a plausible mistake in the oracle; at least one pin must fail.
def _m_window_short(pos, window):
    return list(range(max(0, pos - window + 2), pos + 1))


def _m_window_excludes_self(pos, window):
    return list(range(max(0, pos - window), pos))


def _m_visible_floor(pos, ratio):
    return pos // ratio


def _m_sink_scaled(q, keys, sink, scale):
    return _ATTEND(q, keys, np.asarray(sink, dtype=np.float64) * scale, scale)


def _m_sink_dropped(q, keys, sink, scale):
    out, lse = _ATTEND(q, keys, np.full(np.shape(sink), -np.inf), scale)
    return out, lse


def _m_lse_without_sink(q, keys, sink, scale):
    out, _ = _ATTEND(q, keys, sink, scale)
    _, lse = _ATTEND(q, keys, np.full(np.shape(sink), -np.inf), scale)
    return out, lse


def _m_value_without_rope(q, keys, sink, scale):
    out, lse = _ATTEND(q, keys, sink, scale)
    k = np.array(keys, dtype=np.float64).reshape(-1, np.shape(q)[1])
    if k.shape[0]:
        k[:, 448:] = 0.0
        s = scale * (np.asarray(q) @ np.asarray(keys).reshape(-1, np.shape(q)[1]).T)
        m = np.maximum(s.max(axis=1), sink)
        e = np.exp(s - m[:, None])
        out = (e @ k) / (np.exp(np.asarray(sink) - m) + e.sum(axis=1))[:, None]
    return out, lse


def _m_e4m3_bias8(codes):
    return _E4M3(codes) * 0.5


def _m_scale_index_mod(raw):
    raw = np.ascontiguousarray(np.asarray(raw, dtype=np.uint8))
    n = raw.shape[0]
    nope = O.e4m3_to_f64(raw[:, :448])
    sc = raw[:, 576:604].copy().view("<f4").astype(np.float64).reshape(n, 7)
    nope = nope * sc[:, np.arange(448) % 7]
    rope = O.bf16_bits_to_f64(raw[:, 448:576].copy().view("<u2"))
    return np.concatenate([nope, rope], axis=1)


def _m_page_offset(page_table, req_row, logical, num_pages):
    lp = logical // 256
    if lp < 0 or lp >= page_table.shape[1]:
        return -1
    page = int(page_table[req_row, lp])
    if page < 0 or page >= num_pages:
        return -1
    return page * 256 + lp


def _m_verify_shift(seq_lens, cu_seqlens_q=None):
    req, pos = _COORD(seq_lens, cu_seqlens_q)
    if cu_seqlens_q is not None:
        pos = pos + 1
    return req, pos


def _m_decode_shift(seq_lens, cu_seqlens_q=None):
    req, pos = _COORD(seq_lens, cu_seqlens_q)
    return req, (pos + 1 if cu_seqlens_q is None else pos)


def _m_e4m3_truncate(x):
    # rounds toward zero instead of to nearest
    x = np.asarray(x, dtype=np.float32)
    codes = _ENC(x)
    up = O.e4m3_to_f64(codes & 0x7F) > np.abs(x.astype(np.float64))
    return np.where(up & ((codes & 0x7F) > 0), codes - 1, codes).astype(np.uint8)


def _m_pack_scale_447(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    n = bits.shape[0]
    x = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    nope = x[:, :448].reshape(n, 7, 64)
    amax = np.max(np.abs(nope), axis=2)
    scale = np.where(amax > 0, amax / np.float32(447.0), np.float32(1.0)).astype(np.float32)
    out = _PACK(bits)
    out[:, :448] = O.e4m3_from_f32((nope / scale[:, :, None]).astype(np.float32)).reshape(n, 448)
    out[:, 576:604] = scale.astype("<f4").view(np.uint8).reshape(n, 28)
    return out


def _m_pack_rope_dropped(bits):
    out = _PACK(bits)
    out[:, 448:576] = 0
    return out


def _m_store_ignores_page(pool, bits, req_rows, positions, page_table, kv_format):
    # writes logical row i of request row r at r * 256 + i % 256
    out = np.array(pool, copy=True)
    packed = O.pack_fp8_rows(bits) if kv_format == "fp8" else np.asarray(bits, dtype=np.uint16)
    err = 0
    for i in range(len(req_rows)):
        r, p = int(req_rows[i]), int(positions[i])
        if not (0 <= r < page_table.shape[0]) or O.physical_row(page_table, r, p, out.shape[0] // 256) < 0:
            err |= O.ERR_STORE_ROW
            continue
        out[(r * 256 + p % 256) % out.shape[0]] = packed[i]
    return out, err


def _m_topk_ties_high(scores, lengths, k):
    # equal scores go to the higher index
    scores = np.asarray(scores, dtype=np.float32)
    out = np.full((scores.shape[0], k), -1, dtype=np.int32)
    for r in range(scores.shape[0]):
        n = int(lengths[r])
        order = sorted(range(n), key=lambda i: (-float(scores[r, i]), -i))
        best = sorted(order[:k])
        out[r, :len(best)] = best
    return out


def _m_topk_score_order(scores, lengths, k):
    # the best indices in score order instead of index order
    out = _TOPK(scores, lengths, k)
    scores = np.asarray(scores, dtype=np.float32)
    for r in range(out.shape[0]):
        sel = out[r][out[r] >= 0]
        out[r, :len(sel)] = sel[np.argsort(-scores[r, sel], kind="stable")]
    return out


def _m_topk_zero_equal(scores, lengths, k):
    # -0.0 and +0.0 treated as equal
    scores = np.asarray(scores, dtype=np.float32)
    out = np.full((scores.shape[0], k), -1, dtype=np.int32)
    for r in range(scores.shape[0]):
        n = int(lengths[r])
        order = sorted(range(n), key=lambda i: (-float(scores[r, i]), i))
        best = sorted(order[:k])
        out[r, :len(best)] = best
    return out


def _m_topk_ignores_length(scores, lengths, k):
    return _TOPK(scores, [np.asarray(scores).shape[1]] * len(lengths), k)


_ATTEND = O.attend
_TOPK = O.topk_indices
_E4M3 = O.e4m3_to_f64
_ENC = O.e4m3_from_f32
_PACK = O.pack_fp8_rows
_COORD = O.token_coordinates

MUTANTS = {
    "window_short": ("swa_positions", _m_window_short),
    "window_excludes_self": ("swa_positions", _m_window_excludes_self),
    "visible_floor": ("visible_compressed", _m_visible_floor),
    "sink_scaled": ("attend", _m_sink_scaled),
    "sink_dropped": ("attend", _m_sink_dropped),
    "lse_without_sink": ("attend", _m_lse_without_sink),
    "value_without_rope": ("attend", _m_value_without_rope),
    "e4m3_bias8": ("e4m3_to_f64", _m_e4m3_bias8),
    "scale_index_mod": ("unpack_fp8_rows", _m_scale_index_mod),
    "page_offset": ("physical_row", _m_page_offset),
    "verify_shift": ("token_coordinates", _m_verify_shift),
    "decode_shift": ("token_coordinates", _m_decode_shift),
    "e4m3_truncate": ("e4m3_from_f32", _m_e4m3_truncate),
    "pack_scale_447": ("pack_fp8_rows", _m_pack_scale_447),
    "pack_rope_dropped": ("pack_fp8_rows", _m_pack_rope_dropped),
    "store_ignores_page": ("kv_store", _m_store_ignores_page),
    "topk_ties_high": ("topk_indices", _m_topk_ties_high),
    "topk_score_order": ("topk_indices", _m_topk_score_order),
    "topk_zero_equal": ("topk_indices", _m_topk_zero_equal),
    "topk_ignores_length": ("topk_indices", _m_topk_ignores_length),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    caught = []
    for pin in _pins.ALL_PINS:
        try:
            pin()
        except (AssertionError, KeyError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
