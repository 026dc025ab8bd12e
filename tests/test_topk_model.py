"""A CPU model of the top-k kernel's index arithmetic (csrc/topk.cu), checked
on the GPU tests' inputs.  The model restates the kernel's steps in numpy:
the radix select with its early stop at k + 256 keys, the per-digit bins,
the places every CTA stores its keys at, and the ranks the receiving CTA
gives them.  The invariants it checks are those a wrong index on the GPU
would break silently:

* every store into another CTA's shared memory lands inside its k + 256
  entries, and no two keys land on one entry;
* the bins are at most 256, ascending in key;
* the ranks are a permutation of 0 .. (keys sorted) - 1;
* the first K ranks are the oracle's answer, bit for bit.

This is not the oracle (which is a plain sort) and shares no code with the
CUDA path; it is a model of the kernel's design, kept beside its tests."""
import numpy as np
import pytest

import oracle
from sparse_attention_indexer_logits_gb300 import workloads as W

SLICES = 8          # CTAs per row
CAP_EXTRA = 256     # keys past K the select may leave for the sort
BINS = 256


def order_keys(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.uint64)
    return np.where(b & 0x80000000, (~b) & 0xFFFFFFFF, b | 0x80000000)


def radix_select(keys: np.ndarray, K: int, cap: int):
    """8 bits a pass from the top; stops once the keys at or above the bin's
    lower edge are at most `cap`.  Returns (prefix, need, sort_all, h1,
    passes)."""
    prefix, mask, need = 0, 0, K
    h1 = np.bincount((keys >> 24).astype(np.int64), minlength=256)
    for passes, shift in enumerate((24, 16, 8, 0), start=1):
        sel = (keys & mask) == prefix
        h = np.bincount(((keys[sel] >> shift) & 255).astype(np.int64), minlength=256)
        above = np.concatenate([np.cumsum(h[::-1])[::-1][1:], [0]])   # keys in higher bins
        b = int(np.nonzero(above + h >= need)[0].max())
        need -= int(above[b])
        prefix |= b << shift
        mask |= 255 << shift
        if K - need + int(h[b]) <= cap:
            return prefix, need, True, h1, passes, int(h[b])
    return prefix, need, False, h1, 4, 0


def digit_tables(keys, lo, cand, h1, any_keys):
    """Per top-8-bit digit: its share of the bins, their power-of-two width
    and first bin; a key's bin is first[d] + ((key - base[d]) >> width[d])."""
    dlo = int(lo >> 24) if any_keys else 256
    c = np.zeros(256, np.int64)
    c[dlo + 1:] = h1[dlo + 1:]
    if dlo < 256:
        c[dlo] = cand - c[dlo + 1:].sum()
    nz = int((c > 0).sum())
    kmax = int(keys.max()) if keys.size else 0
    used = np.zeros(256, np.int64)
    base = np.zeros(256, np.int64)
    width = np.zeros(256, np.int64)
    for d in np.nonzero(c > 0)[0]:
        share = max(1, int(c[d]) * (BINS - nz) // cand)
        base[d] = max(int(lo), int(d) << 24)
        last = min(kmax, (int(d) << 24) | 0xFFFFFF) - int(base[d])
        w = 0
        if last >= share:
            w = last.bit_length() - share.bit_length()
            w += 1 if (last >> w) >= share else 0
        width[d], used[d] = w, (last >> w) + 1
    first = np.concatenate([[0], np.cumsum(used)[:-1]])
    assert used.sum() <= BINS
    return first, base, width, used


def model_row(bits: np.ndarray, lim: int, k: int):
    out_i = np.full(k, -1, np.int64)
    out_v = np.full(k, 0xFF800000, np.uint64)
    K = min(k, lim)
    if K == 0:
        return out_i, out_v, None
    keys = order_keys(bits[:lim])
    cap = k + CAP_EXTRA
    prefix, need, sort_all, h1, passes, bin_count = radix_select(keys, K, cap)
    T = prefix
    any_keys = sort_all or T != 0xFFFFFFFF
    lo = T if sort_all else T + 1
    cand = K - need + bin_count if sort_all else K - need
    first, base, width, used = digit_tables(keys, lo, cand, h1, any_keys)

    chunk = -(-lim // SLICES)
    pos = np.arange(lim)
    slice_of = pos // chunk
    take = (keys >= lo) if any_keys else np.zeros(lim, bool)
    d = (keys >> 24).astype(np.int64)
    binv = np.where(take, first[d] + ((keys - base[d].astype(np.uint64)) >> width[d].astype(np.uint64)), -1)
    binv = binv.astype(np.int64)
    assert (binv[take] >= first[d[take]]).all() and (binv[take] < (first + used)[d[take]]).all()
    # bins ascend with the key
    tk = keys[take]
    o = np.argsort(tk, kind="stable")
    assert (np.diff(binv[take][o]) >= 0).all()

    hs = np.zeros((SLICES, BINS), np.int64)
    np.add.at(hs, (slice_of[take], binv[take]), 1)
    m = hs.sum(0)
    total = int(m.sum())
    assert total == cand
    above = np.concatenate([np.cumsum(m[::-1])[::-1][1:], [0]])
    target = -(-total // SLICES)
    owner = np.minimum(SLICES - 1, above // target) if target else np.zeros(BINS, np.int64)
    before = np.cumsum(hs, axis=0) - hs                     # this slice's bins in the slices before
    # the stores: slice r's keys of bin b at owner[b]'s entry
    # above[b] - owner[b]*target + before[r, b] + slot
    ti = np.nonzero(take)[0]
    tb, tr = binv[ti], slice_of[ti]
    grp = tr * BINS + tb
    order = np.argsort(grp, kind="stable")
    slot = np.empty_like(order)
    _, starts, counts = np.unique(grp[order], return_index=True, return_counts=True)
    slot[order] = np.arange(order.size) - np.repeat(starts, counts)
    idx = above[tb] - owner[tb] * target + before[tr, tb] + slot
    assert (idx >= 0).all() and (idx < cap).all()
    dest = owner[tb] * cap + idx
    assert np.unique(dest).size == dest.size                 # no entry written twice

    # receivers: an entry's rank is the keys in higher bins plus the entries
    # of its bin that come before it (key descending, position ascending)
    packed = (keys[ti] << np.uint64(32)) | (np.uint64(0xFFFFFFFF) - ti.astype(np.uint64))
    o = np.lexsort((~packed, tb))                            # by bin, descending within
    rank = np.empty(ti.size, np.int64)
    sorted_b = tb[o]
    _, bstart, bcount = np.unique(sorted_b, return_index=True, return_counts=True)
    within = np.arange(o.size) - np.repeat(bstart, bcount)
    rank[o] = above[sorted_b] + within
    assert np.array_equal(np.sort(rank), np.arange(total))

    keep = rank < K
    out_i[rank[keep]] = ti[keep]
    out_v[rank[keep]] = keys[ti[keep]]
    if not sort_all:
        eq = np.nonzero(keys == T)[0][:need]                  # position order over the slices
        out_i[K - need + np.arange(eq.size)] = eq
        out_v[K - need + np.arange(eq.size)] = T
    vb = np.where(out_v & 0x80000000, out_v & 0x7FFFFFFF, (~out_v) & 0xFFFFFFFF)
    vb = np.where(out_i >= 0, vb, 0xFF800000)
    return out_i, vb, (passes, sort_all, int(idx.max()) + 1 if idx.size else 0)


def run_model(x, seq_lens, next_n, max_context, k):
    rows = x.shape[0]
    bits = x.view(np.uint32)
    gi = np.zeros((rows, k), np.int64)
    gv = np.zeros((rows, k), np.uint64)
    info = []
    for r in range(rows):
        b, t = divmod(r, next_n)
        L = int(seq_lens[b])
        lim = max(0, min(L - next_n + t + 1, max_context)) if L > 0 else 0
        gi[r], gv[r], inf = model_row(bits[r], lim, k)
        info.append(inf)
    ri, rv = oracle.topk_logits(x, seq_lens, next_n, max_context, k)
    assert np.array_equal(gi, ri)
    assert np.array_equal(gv.astype(np.uint32), rv.view(np.uint32))
    return [i for i in info if i is not None]


@pytest.mark.parametrize("next_n,k", [(1, 1), (1, 7), (2, 64), (3, 333), (4, 1024)])
def test_model_matches_oracle(next_n, k):
    x, sl = W.topk_logits_input(6, next_n, 3000, seed=500 + k, lo=0, hi=3000)
    run_model(x, sl, next_n, 3000, k)


def test_model_ties_and_short_rows():
    x, sl = W.topk_logits_input(5, 2, 2500, seed=510, distinct=5, lo=1000)
    run_model(x, sl, 2, 2500, 600)
    x, sl = W.topk_logits_input(6, 1, 512, seed=511, lo=0, hi=40)
    sl[0] = 0
    run_model(x, sl, 1, 512, 100)


def test_model_exact_threshold_path():
    x, sl = W.topk_logits_input(4, 2, 4000, seed=521, distinct=3, lo=3000)
    info = run_model(x, sl, 2, 4000, 1500)
    assert any(not s for _, s, _ in info) and any(s for _, s, _ in info)


def test_model_third_pass_stop():
    x, sl = W.topk_logits_input(4, 1, 4000, seed=522, lo=3000, narrow=True, specials=False)
    info = run_model(x, sl, 1, 4000, 300)
    assert all(p == 3 and s for p, s, _ in info)


def test_model_decode_rows_stop_after_two_passes():
    x, sl = W.topk_logits_input(8, 1, 32768, seed=513, lo=1024, specials=False)
    info = run_model(x, sl, 1, 32768, 2048)
    assert all(p == 2 and s for p, s, _ in info)


def test_model_largest_k_and_clip():
    x, sl = W.topk_logits_input(3, 1, 8192, seed=512, lo=6000)
    run_model(x, sl, 1, 5000, 4096)
