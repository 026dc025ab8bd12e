"""Pins of the top-k selection oracle.  The pages name the selection step
(the logits are what the indexer uses to choose KV tokens to keep) but fix
neither k nor the order of equal values; the readings are: each row's k
largest logits among its meaningful positions, value-descending in float32
bit order, equal values by ascending position, -1 / -inf padding.  The pins
check the oracle against a plain Python sort of (value, position) pairs and
against invariants any correct top-k must satisfy."""
import math
import struct

import numpy as np

import oracle


def bit_key(v) -> int:
    b = struct.unpack("<I", struct.pack("<f", float(v)))[0]
    return (~b & 0xFFFFFFFF) if b >> 31 else (b | 0x80000000)


def brute(row_vals, lim, k):
    cand = sorted(range(lim), key=lambda p: (-bit_key(row_vals[p]), p))[:k]
    return cand + [-1] * (k - len(cand))


def test_matches_a_plain_sort_with_ties_and_specials():
    g = np.random.default_rng(7)
    seq_lens = np.array([37, 0, 5, 64], dtype=np.int32)
    n, mc, k = 2, 60, 8
    x = g.integers(-3, 4, size=(8, mc)).astype(np.float32)           # many ties
    x[0, 3] = np.inf; x[0, 4] = -np.inf; x[0, 5] = -0.0; x[0, 6] = 0.0
    x[6, 10] = np.nan
    idx, val = oracle.topk_logits(x, seq_lens, n, mc, k)
    for r in range(8):
        b, t = divmod(r, n)
        lim = min(seq_lens[b] - n + t + 1, mc) if seq_lens[b] > 0 else 0
        want = brute(x[r], max(lim, 0), k)
        assert idx[r].tolist() == want, r
        for i, p in enumerate(want):
            if p < 0:
                assert val[r, i] == -np.inf
            else:
                assert val[r, i].tobytes() == x[r, p].tobytes()


def test_invariants_on_random_rows():
    g = np.random.default_rng(8)
    seq_lens = g.integers(0, 300, size=6).astype(np.int32)
    n, mc, k = 3, 256, 40
    x = (g.standard_normal((18, mc)) * 4).round(1).astype(np.float32)
    idx, val = oracle.topk_logits(x, seq_lens, n, mc, k)
    for r in range(18):
        b, t = divmod(r, n)
        lim = min(int(seq_lens[b]) - n + t + 1, mc) if seq_lens[b] > 0 else 0
        lim = max(lim, 0)
        sel = [int(p) for p in idx[r] if p >= 0]
        assert len(sel) == min(k, lim) and len(set(sel)) == len(sel)
        assert all(0 <= p < lim for p in sel)
        v = [bit_key(x[r, p]) for p in sel]
        assert all(v[i] > v[i + 1] or (v[i] == v[i + 1] and sel[i] < sel[i + 1])
                   for i in range(len(v) - 1))
        rest = [p for p in range(lim) if p not in set(sel)]
        if sel and rest:
            worst = (v[-1], -sel[-1])
            assert all((bit_key(x[r, p]), -p) < worst for p in rest)
        assert all(math.isinf(val[r, i]) and val[r, i] < 0 for i in range(len(sel), k))
