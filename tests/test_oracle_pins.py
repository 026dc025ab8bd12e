"""Pins for the CPU oracle: checks against facts fixed by the pages and by
mathematics, never against the oracle itself or the GPU path.

Sources: FlashInfer documentation, "flashinfer.attn_scores" (math block, the
per-head rectifier bullet, the s_p bullet, the note on rows and empty
requests, "Scheduling and Setup") and "flashinfer.sdsa.indexer_scores".
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from sparse_attention_indexer_logits_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _kv_blocks(keys_codes, scales):
    """Assemble kv_fused bytes from per-block key codes [nb,64,128] and scales [nb,64]."""
    nb = keys_codes.shape[0]
    kv = np.zeros((nb, W.BLOCK_BYTES), dtype=np.uint8)
    kv[:, :W.BLOCK_KEY_BYTES] = keys_codes.reshape(nb, -1)
    kv[:, W.BLOCK_KEY_BYTES:] = np.asarray(scales, dtype="<f4").view(np.uint8).reshape(nb, -1)
    return kv


# ------------------------------------------------------------ number formats

def test_e4m3_decode_all_codes_match_torch():
    """All 256 codes against torch's float8_e4m3fn -> float32 cast (a library routine)."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_decode(c) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_e4m3_decode_hand_values():
    g = _golden("e4m3_values.json")
    for code, val in g["values"].items():
        got = oracle.e4m3_decode(int(code))
        assert got == val and np.signbit(got) == np.signbit(val), (code, got, val)
        assert brute.e4m3_exact(int(code)) == val
    for code in g["nan_codes"]:
        assert np.isnan(oracle.e4m3_decode(code))
        assert brute.e4m3_exact(code) is None


def test_bf16_decode_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    sample = np.concatenate([np.arange(0, 65536, 97), [0x0001, 0x7F7F, 0x8000, 0xFF80, 0x3F80]])
    for b in sample:
        got = oracle.bf16_decode(int(b))
        if np.isnan(ref[b]):
            assert np.isnan(got)
        else:
            assert got == ref[b]


# ------------------------------------------------------------ fp8 logits: pins

def _relu_problem(case):
    q = np.zeros((1, 2, 128), dtype=np.uint8)
    q[0, 0, 0] = 0x38          # e4m3 1.0: q[0] = e_0
    q[0, 1, 1] = 0x38          # q[1] = e_1
    keys = np.zeros((1, 64, 128), dtype=np.uint8)
    keys[0, 0, 0] = case["k0_code"]
    keys[0, 0, 1] = case["k1_code"]
    kv = _kv_blocks(keys, np.ones((1, 64), dtype=np.float32))
    w = np.array([case["w"]], dtype=np.float32)
    return q, kv, w


def test_relu_is_per_head_before_weighted_sum():
    """Counterexamples where sum_h w relu(x_h) differs from relu(sum_h w x_h)."""
    for case in _golden("relu_per_head.json")["cases"]:
        q, kv, w = _relu_problem(case)
        out, _ = oracle.fp8_paged_mqa_logits(q, kv, w, [1], [[0]], next_n=1)
        assert out[0, 0] == case["logit"]
        assert out[0, 0] != case["relu_of_sum"]
        b = brute.fp8_logits(q, kv, w, [1], [[0]], 1)
        assert float(b[(0, 0)][0]) == case["logit"]


def test_closed_form_one_hot_q_constant_k():
    g = _golden("closed_form.json")
    cf = g["one_hot"]
    codes = {float(k): v for k, v in g["e4m3_codes"].items()}
    H = cf["num_heads"]
    q = np.zeros((1, H, 128), dtype=np.uint8)
    for h, a in enumerate(cf["a"]):
        q[0, h, h] = codes[a]
    keys = np.zeros((1, 64, 128), dtype=np.uint8)
    scales = np.ones((1, 64), dtype=np.float32)
    for p, (c, s) in enumerate(zip(cf["c"], cf["s"])):
        keys[0, p, :] = codes[c]
        scales[0, p] = s
    kv = _kv_blocks(keys, scales)
    w = np.array([cf["w"]], dtype=np.float32)
    L = len(cf["c"])
    out, _ = oracle.fp8_paged_mqa_logits(q, kv, w, [L], [[0]], next_n=1)
    assert out[0, :L].tolist() == cf["logits"]

    ao = g["all_ones_q"]
    q = np.full((1, 1, 128), codes[1.0], dtype=np.uint8)
    keys = np.zeros((1, 64, 128), dtype=np.uint8)
    for p, c in enumerate(ao["c"]):
        keys[0, p, :] = codes[c]
    kv = _kv_blocks(keys, np.array([ao["s"] + [1.0] * (64 - len(ao["s"]))], dtype=np.float32))
    out, _ = oracle.fp8_paged_mqa_logits(q, kv, np.array([ao["w"]], np.float32),
                                         [len(ao["c"])], [[0]], next_n=1)
    assert out[0, :len(ao["c"])].tolist() == ao["logits"]


def test_closed_form_random_multislot_rows():
    """Random one-hot q per (row, head), constant keys: the logit is a scalar
    closed form, and row b*next_n+t must use slot t's q and weights."""
    g = W.rng(11)
    B, n, H = 3, 3, 5
    vals = np.array([0.5, 1.0, 2.0, -1.0, -2.0, 4.0, -0.25, 0.25])
    a = g.choice(vals, size=(B * n, H))
    c = g.choice(vals, size=(B, 130))
    s = g.uniform(0.5, 2.0, size=(B, 130)).astype(np.float32)
    w = g.standard_normal((B * n, H)).astype(np.float32)
    dims = g.integers(0, 128, size=(B * n, H))
    q = np.zeros((B * n, H, 128), dtype=np.uint8)
    for r in range(B * n):
        for h in range(H):
            q[r, h, dims[r, h]] = W.to_e4m3(np.array([a[r, h]]))[0]
    seq_lens = np.array([130, 65, 3], dtype=np.int32)
    nb = 3
    keys = np.zeros((B * nb, 64, 128), dtype=np.uint8)
    scales = np.ones((B * nb, 64), dtype=np.float32)
    bt = np.arange(B * nb, dtype=np.int32).reshape(B, nb)[:, ::-1].copy()   # reversed pages
    for b in range(B):
        for p in range(seq_lens[b]):
            blk = bt[b, p // 64]
            keys[blk, p % 64, :] = W.to_e4m3(np.array([c[b, p]]))[0]
            scales[blk, p % 64] = s[b, p]
    kv = _kv_blocks(keys, scales)
    out, _ = oracle.fp8_paged_mqa_logits(q, kv, w, seq_lens, bt, next_n=n, max_context=130)
    for b in range(B):
        for t in range(n):
            r = b * n + t
            for p in range(seq_lens[b]):
                x = a[r] * c[b, p]
                exp = float(s[b, p]) * float(np.sum(w[r].astype(np.float64) * np.maximum(x, 0)))
                assert out[r, p] == pytest.approx(exp, rel=1e-12, abs=1e-300)


@pytest.mark.parametrize("seed,n,H,lens", [
    (21, 1, 2, [130, 1]),
    (22, 2, 3, [64, 70]),
    (23, 4, 1, [5, 0, 66]),
    (24, 3, 4, [129]),
])
def test_oracle_matches_exact_brute_force(seed, n, H, lens):
    p = W.fp8_problem("brute", lens, n, H, seed, poison=True, extra_blocks=1)
    out, mag = oracle.fp8_paged_mqa_logits(p.q, p.kv_fused, p.weights, p.seq_lens,
                                           p.block_table, next_n=n, max_context=p.max_context)
    ref = brute.fp8_logits(p.q, p.kv_fused, p.weights, p.seq_lens, p.block_table, n)
    written = oracle.fp8_written_mask(p.seq_lens, n, p.max_context)
    assert written.sum() == len(ref)
    for (r, pos), (val, m) in ref.items():
        v = float(val)
        assert abs(out[r, pos] - v) <= 1e-12 * max(abs(v), 1e-30), (r, pos, out[r, pos], v)
        # the tolerance scale of every fp8 parity check, to the same precision
        assert m > 0 and abs(mag[r, pos] - float(m)) <= 1e-12 * float(m), (r, pos, mag[r, pos], m)
    assert np.isnan(out[~written]).all()
    assert np.isnan(mag[~written]).all()


def test_scale_factors_out():
    """s_p is uniform over the key: doubling every s_p doubles every logit
    exactly; s_p = 1 reduces to the unscaled definition (brute force)."""
    p = W.fp8_problem("scale", [200, 77], 2, 4, 31, poison=False)
    base, _ = oracle.fp8_paged_mqa_logits(p.q, p.kv_fused, p.weights, p.seq_lens,
                                          p.block_table, next_n=2)
    kv2 = p.kv_fused.copy()
    s = kv2[:, W.BLOCK_KEY_BYTES:].view("<f4")
    s *= 2
    dbl, _ = oracle.fp8_paged_mqa_logits(p.q, kv2, p.weights, p.seq_lens, p.block_table, next_n=2)
    m = ~np.isnan(base)
    assert np.array_equal(dbl[m], 2 * base[m])
    kv1 = p.kv_fused.copy()
    kv1[:, W.BLOCK_KEY_BYTES:].view("<f4")[:] = 1.0
    one, _ = oracle.fp8_paged_mqa_logits(p.q[:2], kv1, p.weights[:2], [70],
                                         p.block_table[:1], next_n=2, max_context=70)
    ref = brute.fp8_logits(p.q[:2], kv1, p.weights[:2], [70], p.block_table[:1], 2)
    for (r, pos), (v, _) in ref.items():
        assert one[r, pos] == pytest.approx(float(v), rel=1e-12)


def test_page_permutation_invariance():
    """Paging is pure indirection: moving physical blocks and rewriting the
    block table leaves every logit bit-identical."""
    p = W.fp8_problem("perm", [300, 1, 190, 64], 2, 8, 41, poison=True, extra_blocks=3)
    out1, _ = oracle.fp8_paged_mqa_logits(p.q, p.kv_fused, p.weights, p.seq_lens,
                                          p.block_table, next_n=2)
    g = W.rng(42)
    perm = g.permutation(p.num_blocks)          # new position of old block i
    kv2 = np.empty_like(p.kv_fused)
    kv2[perm] = p.kv_fused
    bt2 = perm[p.block_table].astype(np.int32)
    out2, _ = oracle.fp8_paged_mqa_logits(p.q, kv2, p.weights, p.seq_lens, bt2, next_n=2)
    assert np.array_equal(out1.view(np.uint64), out2.view(np.uint64))


def test_empty_requests_and_tail_untouched():
    """seq_lens[b] == 0 leaves the request's rows as they were; positions past
    seq_lens[b] are never written."""
    p = W.fp8_problem("sent", [0, 70, 0, 5], 2, 4, 51, poison=True)
    mc = 128
    sentinel = np.frombuffer(np.uint64(0x7FF8DEADBEEF0001).tobytes(), dtype=np.float64)[0]
    out = np.full((p.batch * 2, mc), sentinel)
    oracle.fp8_paged_mqa_logits(p.q, p.kv_fused, p.weights, p.seq_lens, p.block_table,
                                next_n=2, max_context=mc, out=out)
    written = oracle.fp8_written_mask(p.seq_lens, 2, mc)
    bits = out.view(np.uint64)
    assert (bits[~written] == 0x7FF8DEADBEEF0001).all()
    assert np.isfinite(out[written]).all()      # poison rows past the length never leak in
    assert written[2:4].sum() == 140 and written[0:2].sum() == 0


def test_valid_mask_per_slot_limit():
    """Row b*next_n+t is meaningful for p <= seq_lens[b] - next_n + t."""
    m = oracle.fp8_valid_mask([10, 3], 4, 12)
    assert m.shape == (8, 12)
    assert [int(r.sum()) for r in m] == [7, 8, 9, 10, 0, 1, 2, 3]


# ------------------------------------------------------------ bf16 indexer scores

def test_bf16_scores_equal_numpy_matmul():
    """One head, no weight, no ReLU: scores are the query rows times the
    gathered keys; numpy's float64 matmul is exact here (bf16 products are
    exact and 128-term sums of them fit in fp64)."""
    p = W.indexer(group_size=3, seed=61, groups=6, max_context=300, num_requests=3,
                  shared_requests=True, min_zero=1, page_pad_bytes=48)
    out, mag = oracle.indexer_scores_bf16(p.query, p.key_cache, p.page_stride_bytes,
                                          p.block_table, p.context_lengths, p.requests,
                                          p.max_context)
    qf = torch.from_numpy(p.query.view(np.int16)).view(torch.bfloat16).double().numpy()
    keys = torch.from_numpy(p.key_pages().view(np.int16)).view(torch.bfloat16).double().numpy()
    G = p.group_size
    for g in range(p.groups):
        L = int(p.context_lengths[g])
        rows = slice(g * G, (g + 1) * G)
        if L == 0:
            assert np.isnan(out[rows]).all()
            continue
        pages = p.block_table[p.requests[g], :(L + 63) // 64]
        K = keys[pages].reshape(-1, 128)[:L]
        ref = qf[rows] @ K.T
        assert np.array_equal(out[rows, :L], ref)
        assert np.isnan(out[rows, L:]).all()
        assert np.array_equal(mag[rows, :L], np.abs(qf[rows]) @ np.abs(K).T)


def test_bf16_scores_match_exact_brute_force():
    p = W.indexer(group_size=2, seed=62, groups=3, max_context=140, min_zero=1)
    out, _ = oracle.indexer_scores_bf16(p.query, p.key_cache, p.page_stride_bytes,
                                        p.block_table, p.context_lengths, p.requests,
                                        p.max_context)
    ref = brute.bf16_scores(p.query, p.key_pages(), p.block_table, p.context_lengths,
                            p.requests, p.group_size)
    assert len(ref) == int(np.isfinite(out).sum())
    for (r, k), v in ref.items():
        assert out[r, k] == float(v)


# ------------------------------------------------------------ schedule

def test_schedule_golden():
    for case in _golden("schedule.json")["cases"]:
        meta, total = oracle.schedule(case["seq_lens"], case["num_ctas"])
        assert total == case["total"]
        assert meta.tolist() == case["meta"]


@pytest.mark.parametrize("seed", range(6))
def test_schedule_partitions_blocks(seed):
    """Brute force: enumerating the blocks of every range reproduces each
    (request, block) exactly once, in order, range sizes within one."""
    g = W.rng(100 + seed)
    B = int(g.integers(1, 40))
    lens = g.integers(0, 700, size=B)
    lens[g.random(B) < 0.3] = 0
    G = int(g.integers(1, 50))
    meta, total = oracle.schedule(lens, G)
    flat = [(b, j) for b in range(B) for j in range((int(lens[b]) + 63) // 64)]
    assert total == len(flat)
    index = {bj: i for i, bj in enumerate(flat)}
    index[(B, 0)] = total
    starts = [index[tuple(m)] for m in meta.tolist()]
    assert starts[0] == 0 and starts[-1] == total
    sizes = np.diff(starts)
    assert (sizes >= 0).all() and sizes.max() - sizes.min() <= 1
    assert sizes.max() == -(-total // G)
