"""Exact brute-force restatement of the oracle for tiny inputs.

TEST INFRASTRUCTURE ONLY: used by the oracle's pin tests, never by the GPU
path.  Written independently of ``oracle.c`` (different language, exact
rational arithmetic with ``fractions.Fraction``) so that an indexing, sign or
operand mistake in either one shows up as a disagreement.

Sources: FlashInfer documentation, "flashinfer.attn_scores" (math block, the
two bullets on the per-head rectifier and on the per-token scale s_p, the
note on row order) and "flashinfer.sdsa.indexer_scores" (one head: plain dot
product).
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
    """Dict ``{(row, p): Fraction}`` of every written logit.

    ``q``: nested lists / arrays of e4m3 codes ``[batch*next_n][H][128]``;
    ``kv_fused``: per block a bytes-like of 8448 bytes; ``weights`` fp32
    values ``[batch*next_n][H]``; ``block_table[b][j]`` physical block."""
    res = {}
    for b, L in enumerate(seq_lens):
        for t in range(next_n):
            row = b * next_n + t
            for p in range(int(L)):
                blk = bytes(kv_fused[int(block_table[b][p // BLOCK_KEYS])])
                key = blk[(p % BLOCK_KEYS) * HEAD_DIM:(p % BLOCK_KEYS + 1) * HEAD_DIM]
                (s,) = struct.unpack_from("<f", blk, KEY_BYTES + 4 * (p % BLOCK_KEYS))
                total = Fraction(0)
                for h, wv in enumerate(weights[row]):
                    x = sum(e4m3_exact(int(a)) * e4m3_exact(int(c))
                            for a, c in zip(q[row][h], key))
                    total += Fraction(float(wv)) * max(x, Fraction(0))
                res[(row, p)] = Fraction(s) * total
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
