"""Exact brute-force restatement of the oracle for tiny inputs.

TEST INFRASTRUCTURE ONLY: used by the oracle's pin tests, never by the GPU
path.  Written independently of ``oracle.c`` (different language, exact
rational arithmetic with ``fractions.Fraction``) so that an indexing, sign or
operand mistake in either one shows up as a disagreement.

Sources: FlashInfer documentation, "flashinfer.attn_scores" (math block, the
two bullets on the per-head rectifier and on the per-token scale s_p, the
note on row order) and "flashinfer.sdsa.indexer_scores" (one head: plain dot
product), and the MXFP4 variant (the paragraph after the two bullets).
"""
from __future__ import annotations

import struct
from fractions import Fraction

HEAD_DIM = 128
BLOCK_KEYS = 64
KEY_BYTES = BLOCK_KEYS * HEAD_DIM


def e4m3_exact(code: int):
    """Exact value of an E4M3FN code as a Fraction (None for NaN).

    Sign bit 7; exponent bits 6..3, bias 7; mantissa bits 2..0.  Exponent 0
    is subnormal: (m/8) * 2^-6.  0x7F / 0xFF are NaN."""
    sign = -1 if code & 0x80 else 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return None
    if e == 0:
        return sign * Fraction(m, 8) * Fraction(1, 2 ** 6)
    scale = Fraction(2) ** (e - 7)
    return sign * (1 + Fraction(m, 8)) * scale


def bf16_exact(bits: int) -> Fraction:
    """Exact value of a bfloat16 pattern: the binary32 whose upper half it is."""
    (f,) = struct.unpack("<f", struct.pack("<I", (bits & 0xFFFF) << 16))
    return Fraction(f)


def fp8_logits(q, kv_fused, weights, seq_lens, block_table, next_n):
    """Dict ``{(row, p): (logit, mag)}`` of every written logit, both exact
    Fractions.

    ``mag`` is the size of the terms the logit is made of,
    ``|s_p| * sum_h |w[row,h]| * |q[row,h] . k_p|``, the quantity the
    parity tolerance is measured against (1e-3 times it, plus 1e-6).  ``q``: nested lists / arrays of e4m3 codes
    ``[batch*next_n][H][128]``; ``kv_fused``: per block a bytes-like of 8448
    bytes; ``weights`` fp32 values ``[batch*next_n][H]``;
    ``block_table[b][j]`` physical block."""
    res = {}
    for b, L in enumerate(seq_lens):
        for t in range(next_n):
            row = b * next_n + t
            for p in range(int(L)):
                blk = bytes(kv_fused[int(block_table[b][p // BLOCK_KEYS])])
                key = blk[(p % BLOCK_KEYS) * HEAD_DIM:(p % BLOCK_KEYS + 1) * HEAD_DIM]
                (s,) = struct.unpack_from("<f", blk, KEY_BYTES + 4 * (p % BLOCK_KEYS))
                total, terms = Fraction(0), Fraction(0)
                for h, wv in enumerate(weights[row]):
                    x = sum(e4m3_exact(int(a)) * e4m3_exact(int(c))
                            for a, c in zip(q[row][h], key))
                    total += Fraction(float(wv)) * max(x, Fraction(0))
                    terms += abs(Fraction(float(wv))) * abs(x)
                res[(row, p)] = (Fraction(s) * total, abs(Fraction(s)) * terms)
    return res


def bf16_scores(query, key_pages, block_table, context_lengths, requests, group_size):
    """Dict ``{(row, k): Fraction}``; ``key_pages[P]`` is a ``[64][128]`` array
    of bf16 bit patterns for page ``P``."""
    res = {}
    for g, L in enumerate(context_lengths):
        for r in range(g * group_size, (g + 1) * group_size):
            for k in range(int(L)):
                page = key_pages[int(block_table[int(requests[g])][k // BLOCK_KEYS])]
                key = page[k % BLOCK_KEYS]
                res[(r, k)] = sum(bf16_exact(int(a)) * bf16_exact(int(c))
                                  for a, c in zip(query[r], key))
    return res


def e2m1_exact(code: int) -> Fraction:
    """Exact value of a 4-bit E2M1 code: sign bit 3, exponent bits 2..1 (bias
    1), mantissa bit 0; exponent 0 is subnormal, (m/2) * 2^0."""
    sign = -1 if code & 0x8 else 1
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return sign * Fraction(m, 2)
    return sign * (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)


def e8m0_exact(code: int):
    """Exact value of an E8M0 scale byte, 2^(code - 127) (None for 0xFF)."""
    return None if code == 0xFF else Fraction(2) ** (code - 127)


def _mx_row(packed, scales):
    """128 exact values of a packed MXFP4 row (element d: byte d/2, low
    nibble for even d, times scale d/32)."""
    out = []
    for d in range(HEAD_DIM):
        byte = int(packed[d // 2])
        code = byte & 0xF if d % 2 == 0 else byte >> 4
        out.append(e2m1_exact(code) * e8m0_exact(int(scales[d // 32])))
    return out


def mxfp4_logits(q, q_sf, kv, weights, seq_lens, block_table, next_n):
    """Dict ``{(row, p): (Fraction logit, Fraction sum_h |w| |q.k|)}`` of
    every written MXFP4 logit ("flashinfer.attn_scores": the fp4 variant, no
    per-position factor).  ``kv``: per block a bytes-like of 4352 bytes, 64
    rows of 64 code bytes then 64 x 4 scale bytes."""
    res = {}
    for b, L in enumerate(seq_lens):
        for t in range(next_n):
            row = b * next_n + t
            qv = [_mx_row(q[row][h], q_sf[row][h]) for h in range(len(weights[row]))]
            for p in range(int(L)):
                blk = bytes(kv[int(block_table[b][p // BLOCK_KEYS])])
                r = p % BLOCK_KEYS
                kv_row = _mx_row(blk[r * 64:(r + 1) * 64], blk[4096 + 4 * r:4096 + 4 * r + 4])
                total, mag = Fraction(0), Fraction(0)
                for h, wv in enumerate(weights[row]):
                    x = sum(a * c for a, c in zip(qv[h], kv_row))
                    total += Fraction(float(wv)) * (x if x > 0 else 0)
                    mag += abs(Fraction(float(wv))) * abs(x)
                res[(row, p)] = (total, mag)
    return res
