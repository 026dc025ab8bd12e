"""Pins of the MXFP4 paged-logits oracle ("flashinfer.attn_scores": the math
block, its two bullets and the paragraph after them -- MXFP4 block scales
folded into the dequantised values, one per 32-element group on both
operands, two FP4 values per q byte, 64 heads of 128, no per-position
factor).  Each pin checks the oracle against something other than its own
code: the published E8M0 and E2M1 tables, torch's E4M3 cast, the
separately pinned fp8 oracle on inputs both formats hold exactly, and an
exact rational restatement (``oracle/brute.py``) on scales far outside E4M3."""
import functools
import json
import os

import numpy as np
import torch

import oracle
from oracle import brute
from sparse_attention_indexer_logits_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def e2m1_table():
    d = json.load(open(os.path.join(GOLDEN, "e2m1_values.json")))
    return np.array(d["values"], dtype=np.float64)


def e8m0_table():
    d = json.load(open(os.path.join(GOLDEN, "e8m0_values.json")))
    return d["codes"], [float.fromhex(v) if v != "nan" else float("nan") for v in d["values"]]


def mx_values(packed: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """[..., 64] packed bytes and [..., 4] E8M0 codes -> [..., 128] values,
    from the golden E2M1 table (low nibble = even element) and the golden
    E8M0 rule checked below (2^(code - 127))."""
    tab = e2m1_table()
    codes = np.empty(packed.shape[:-1] + (128,), dtype=np.int64)
    codes[..., 0::2] = packed & 0xF
    codes[..., 1::2] = packed >> 4
    scale = np.ldexp(1.0, sf.astype(np.int64) - 127)
    return tab[codes] * np.repeat(scale, 32, axis=-1)


def to_e4m3_exact(values: np.ndarray) -> np.ndarray:
    """E4M3 bytes of values that E4M3 holds exactly (asserted with torch's
    cast, a library routine)."""
    t = torch.from_numpy(values.astype(np.float32)).to(torch.float8_e4m3fn)
    assert np.array_equal(t.to(torch.float64).numpy(), values), "value not exact in e4m3"
    return t.view(torch.uint8).numpy()


def as_fp8_problem(p: W.Mxfp4Problem):
    """The same logits problem in the fp8 layout: e4m3 q and keys holding the
    dequantised MXFP4 values, every per-token scale 1.0."""
    q8 = to_e4m3_exact(mx_values(p.q, p.q_sf))
    codes = p.kv[:, :W.MXFP4_BLOCK_CODE_BYTES].reshape(p.num_blocks, 64, 64)
    sf = p.kv[:, W.MXFP4_BLOCK_CODE_BYTES:].reshape(p.num_blocks, 64, 4)
    k8 = to_e4m3_exact(mx_values(codes, sf))
    kv8 = np.empty((p.num_blocks, W.BLOCK_BYTES), dtype=np.uint8)
    kv8[:, :W.BLOCK_KEY_BYTES] = k8.reshape(p.num_blocks, -1)
    kv8[:, W.BLOCK_KEY_BYTES:] = np.ones((p.num_blocks, 64), dtype="<f4").view(np.uint8)
    return q8, kv8


def small(seed, lo_exp, hi_exp, next_n=2):
    g = W.rng(seed)
    return W.mxfp4_problem("pin", [150, 0, 64, 7], next_n, seed, g=g, poison=False,
                           lo_exp=lo_exp, hi_exp=hi_exp)


def test_e8m0_decode_matches_the_published_table():
    codes, values = e8m0_table()
    for c, v in zip(codes, values):
        got = oracle.e8m0_decode(c)
        assert (np.isnan(v) and np.isnan(got)) or got == v, (c, got, v)


def test_unit_scales_reduce_to_the_fp8_oracle():
    """All scales 2^0: MXFP4 logits equal the fp8 logits of the same E2M1
    values in E4M3 with s_p = 1, bit for bit (both sums exact per head)."""
    p = small(21, 0, 0)
    q8, kv8 = as_fp8_problem(p)
    got, _ = oracle.fp4_paged_mqa_logits(p.q, p.q_sf, p.kv, p.weights, p.seq_lens,
                                         p.block_table, p.next_n, p.max_context)
    ref, _ = oracle.fp8_paged_mqa_logits(q8.reshape(-1, 64, 128), kv8, p.weights, p.seq_lens,
                                         p.block_table, p.next_n, p.max_context)
    assert np.array_equal(got, ref, equal_nan=True)
    assert np.isfinite(got).sum() == 2 * (150 + 64 + 7)


def test_group_scales_reduce_to_the_fp8_oracle():
    """Scales 2^-3 .. 2^3 per 32-value group on both operands: every value
    stays exact in E4M3, so the fp8 oracle on those values gives the same
    logits.  Pins the scale format, the 32-value grouping, where q's and each
    key's scales sit, the 4352-byte block and the paging."""
    for seed in (22, 23):
        p = small(seed, -3, 3)
        q8, kv8 = as_fp8_problem(p)
        got, _ = oracle.fp4_paged_mqa_logits(p.q, p.q_sf, p.kv, p.weights, p.seq_lens,
                                             p.block_table, p.next_n, p.max_context)
        ref, _ = oracle.fp8_paged_mqa_logits(q8.reshape(-1, 64, 128), kv8, p.weights,
                                             p.seq_lens, p.block_table, p.next_n, p.max_context)
        assert np.array_equal(got, ref, equal_nan=True), seed


def test_scale_is_homogeneous_per_query_row():
    """Raising every scale of one q row (all heads) by one binade doubles
    that row's logits (relu and the weighted sum are positively homogeneous)
    and leaves the other rows alone."""
    p = small(24, -2, 2)
    base, _ = oracle.fp4_paged_mqa_logits(p.q, p.q_sf, p.kv, p.weights, p.seq_lens,
                                          p.block_table, p.next_n, p.max_context)
    sf = p.q_sf.copy()
    sf[1] += 1
    got, _ = oracle.fp4_paged_mqa_logits(p.q, sf, p.kv, p.weights, p.seq_lens, p.block_table,
                                         p.next_n, p.max_context)
    assert np.array_equal(got[1], 2 * base[1], equal_nan=True)
    assert np.array_equal(np.delete(got, 1, 0), np.delete(base, 1, 0), equal_nan=True)


def test_negative_weights_and_unwritten_places():
    """The rectifier acts per head before the weighted sum, so negative
    weights give negative logits; rows of an empty request and positions
    past a request's length are never written (NaN here)."""
    p = small(25, -1, 1)
    out, mag = oracle.fp4_paged_mqa_logits(p.q, p.q_sf, p.kv, p.weights, p.seq_lens,
                                           p.block_table, p.next_n, p.max_context)
    n = p.next_n
    assert np.isnan(out[1 * n:2 * n]).all()                  # seq_len 0
    assert np.isnan(out[3 * n:4 * n, 7:]).all() and np.isfinite(out[3 * n:4 * n, :7]).all()
    assert (out[np.isfinite(out)] < 0).any() and (out[np.isfinite(out)] > 0).any()
    fin = np.isfinite(out)
    assert (np.abs(out[fin]) <= mag[fin]).all()


@functools.lru_cache(maxsize=1)
def _wide_problem_and_exact():
    # scales 2^-40 .. 2^40 on both operands: far outside what E4M3 holds
    p = W.mxfp4_problem("wide", [9, 5], 1, seed=26, poison=False, lo_exp=-40, hi_exp=40)
    exact = brute.mxfp4_logits(p.q, p.q_sf, p.kv, p.weights, p.seq_lens, p.block_table, 1)
    return p, exact


def test_brute_force_rationals_with_wide_scales():
    """Against an exact rational restatement (another language, no shared
    code) on scales spread over 80 binades: every written logit within
    fp64 rounding of the exact one (the 128-term sums are no longer exact
    there), and the error scale matches."""
    p, exact = _wide_problem_and_exact()
    out, mag = oracle.fp4_paged_mqa_logits(p.q, p.q_sf, p.kv, p.weights, p.seq_lens,
                                           p.block_table, 1, p.max_context)
    assert len(exact) == int(np.isfinite(out).sum()) == 14
    for (row, pos), (val, m) in exact.items():
        assert abs(out[row, pos] - float(val)) <= 2.0 ** -40 * float(m), (row, pos)
        assert abs(mag[row, pos] - float(m)) <= 2.0 ** -40 * float(m), (row, pos)
