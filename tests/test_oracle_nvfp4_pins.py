"""Pins of the NVFP4 single-head oracle ("flashinfer.sdsa.indexer_scores":
NVFP4 query [rows, 64] and key_cache [pages, 64, 64] of E2M1 values two to a
byte, E4M3 query_scales [rows, 8] and key_scales [pages, 64, 8], a scale per
16 values).  Each pin checks the oracle against something other than its own
code: the published E2M1 table, torch's E4M3 cast, exact rational
arithmetic, the separately pinned bf16 oracle, and hand-computed cases."""
import json
import os
from fractions import Fraction

import numpy as np
import torch

import oracle
from sparse_attention_indexer_logits_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_values.json")


def e2m1_table():
    d = json.load(open(GOLDEN))
    return np.array(d["values"], dtype=np.float64)


def e4m3_torch(codes) -> np.ndarray:
    t = torch.from_numpy(np.asarray(codes, dtype=np.uint8).copy()).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def dequant_rows(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """[n, 64] packed bytes and [n, 8] scale codes -> [n, 128] values, from the
    golden E2M1 table and torch's E4M3 cast (low nibble = even element)."""
    tab = e2m1_table()
    codes = np.empty((packed.shape[0], 128), dtype=np.int64)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    return tab[codes] * np.repeat(e4m3_torch(scales), 16, axis=1)


def run(p, mc=None):
    return oracle.indexer_scores_nvfp4(p.query, p.query_scales, p.key_view(), p.page_stride_bytes,
                                       p.scale_view(), p.scale_page_stride_bytes, p.block_table,
                                       p.context_lengths, p.requests,
                                       p.max_context if mc is None else mc)


def test_e2m1_decode_matches_the_published_table():
    tab = e2m1_table()
    got = np.array([oracle.e2m1_decode(c) for c in range(16)])
    assert np.array_equal(got, tab) and np.array_equal(np.signbit(got), np.signbit(tab))


def test_e2m1_values_are_exact_e4m3_values():
    """Library cross-check: every E2M1 magnitude survives torch's E4M3 cast
    unchanged, and the cast's codes decode back through the oracle's E4M3."""
    tab = e2m1_table()
    t = torch.from_numpy(tab.astype(np.float32)).to(torch.float8_e4m3fn)
    assert np.array_equal(t.to(torch.float64).numpy(), tab)
    codes = t.view(torch.uint8).numpy()
    assert all(oracle.e4m3_decode(int(c)) == v for c, v in zip(codes, tab))


def test_reduces_to_the_bf16_oracle_on_dequantised_inputs():
    """Every NVFP4 value (at most 6 significant bits, |v| <= 2688) is exact in
    bf16, so the bf16 oracle on the dequantised rows gives the same scores
    bit for bit."""
    p = W.indexer_nvfp4(3, seed=61, groups=6, max_context=300, min_zero=1, fused=False,
                        page_pad_bytes=32, scale_pad_bytes=8, poison=False)
    s4, m4 = run(p)
    q = dequant_rows(p.query, p.query_scales)
    kb = p.key_view()[:p.num_pages * p.page_stride_bytes].reshape(p.num_pages, -1)[:, :4096]
    sb = p.scale_view()[:p.num_pages * p.scale_page_stride_bytes].reshape(p.num_pages, -1)[:, :512]
    k = dequant_rows(kb.reshape(-1, 64), sb.reshape(-1, 8))          # [pages*64, 128]
    assert np.array_equal(W.to_bf16(q.astype(np.float32)).view(np.uint16).astype(np.uint32) << 16,
                          q.astype(np.float32).view(np.uint32))       # exact in bf16
    qb = W.to_bf16(q.astype(np.float32))
    kc = W.to_bf16(k.astype(np.float32)).reshape(p.num_pages, -1).view(np.uint8)
    s16, m16 = oracle.indexer_scores_bf16(qb, kc, 128 * 64 * 2, p.block_table, p.context_lengths,
                                          p.requests, p.max_context)
    assert np.array_equal(np.isnan(s4), np.isnan(s16))
    w = ~np.isnan(s4)
    assert np.array_equal(s4[w], s16[w]) and np.array_equal(m4[w], m16[w])


def test_brute_force_rationals():
    p = W.indexer_nvfp4(1, seed=62, groups=2, max_context=70, lo=60, hi=70, min_zero=0,
                        poison=False)
    s, _ = run(p)
    tab = [Fraction(v) for v in e2m1_table()]
    def val(byte_row, scale_row, d):
        code = (byte_row[d // 2] >> 4) if d & 1 else (byte_row[d // 2] & 0xF)
        return tab[code] * Fraction(float(e4m3_torch([scale_row[d // 16]])[0]))
    kv, sv = p.key_view(), p.scale_view()
    for g in range(2):
        for k in (0, 1, 63, int(p.context_lengths[g]) - 1):
            page = int(p.block_table[g, k // 64])
            kr = kv[page * p.page_stride_bytes + (k % 64) * 64:][:64]
            ks = sv[page * p.scale_page_stride_bytes + (k % 64) * 8:][:8]
            want = sum(val(p.query[g], p.query_scales[g], d) * val(kr, ks, d) for d in range(128))
            assert Fraction(s[g, k]) == want


def test_scales_factor_out():
    """Raising every key scale's exponent by one (code + 8) doubles every
    score exactly; the same for the query scales."""
    p = W.indexer_nvfp4(2, seed=63, groups=4, max_context=200, min_zero=1, poison=False,
                        fused=False)
    s0, _ = run(p)
    p.scale_buf = p.scale_buf + np.uint8(8)
    s1, _ = run(p)
    p.query_scales = p.query_scales + np.uint8(8)
    s2, _ = run(p)
    w = ~np.isnan(s0)
    assert np.array_equal(s1[w], 2 * s0[w]) and np.array_equal(s2[w], 4 * s0[w])


def test_nibble_order_by_hand():
    """Query element 0 = 1.0 (low nibble of byte 0 = code 2, scale 1.0) and
    every other element 0: the score is key element 0 = E2M1(low nibble of
    the key's byte 0) * the key's scale 0; moving the 1.0 to the high nibble
    selects key element 1 instead.  (Which nibble holds the even element is
    a reading, and not an observable one: both operands share it and the two
    elements of a byte share a scale, so swapping it leaves every score
    unchanged.  The pin checks that one position meets the same position.)"""
    p = W.indexer_nvfp4(1, seed=64, groups=1, max_context=64, lo=64, hi=64, min_zero=0,
                        poison=False)
    p.query[:] = 0
    p.query_scales[:] = 0x38                       # E4M3 1.0
    p.query[0, 0] = 0x02
    s_lo, _ = run(p)
    p.query[0, 0] = 0x20
    s_hi, _ = run(p)
    tab = e2m1_table()
    kv, sv = p.key_view(), p.scale_view()
    page = int(p.block_table[0, 0])
    for k in range(64):
        b0 = kv[page * p.page_stride_bytes + k * 64]
        sc = e4m3_torch([sv[page * p.scale_page_stride_bytes + k * 8]])[0]
        assert s_lo[0, k] == tab[b0 & 0xF] * sc
        assert s_hi[0, k] == tab[b0 >> 4] * sc


def test_untouched_past_lengths_and_empty_groups():
    p = W.indexer_nvfp4(2, seed=65, groups=5, max_context=256, min_zero=2, poison=True)
    s, _ = run(p)
    for g in range(5):
        L = min(int(p.context_lengths[g]), 256)
        rows = s[2 * g:2 * g + 2]
        assert np.isnan(rows[:, L:]).all()
        assert not np.isnan(rows[:, :L]).any()
