"""GPU parity of pml_topk_logits with the top-k oracle, bit for bit (indices
and selected values): k from 1 to 4096, ties (few distinct values), rows
with fewer candidates than k, empty requests, next_n 1..4, special values
(+-inf, signed zeros, NaN), max_context clipping, and a decode-sized batch
(64 rows x 32768, k = 2048).  Further cases steer the kernel down each of
its paths: the radix select stopping after the first, second or third pass,
the exact threshold with the tied keys placed by position, and slices too
long for registers (from shared memory, and from global memory).  The
inputs are synthetic logits from the seeded generator, not outputs of the
logits kernel."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_indexer_logits_gb300 as pml
from sparse_attention_indexer_logits_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run(x, seq_lens, next_n, max_context, k, with_values=True):
    dx = torch.from_numpy(x).cuda()
    ds = torch.from_numpy(seq_lens).cuda()
    vals = torch.empty((x.shape[0], k), dtype=torch.float32, device="cuda") if with_values else None
    idx, vals = pml.pml_topk_logits(dx, ds, next_n, max_context, k, values=vals)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), None if vals is None else vals.cpu().numpy()


def check(x, seq_lens, next_n, max_context, k):
    gi, gv = run(x, seq_lens, next_n, max_context, k)
    ri, rv = oracle.topk_logits(x, seq_lens, next_n, max_context, k)
    assert np.array_equal(gi, ri), f"first differing row {np.argwhere((gi != ri).any(1))[0][0]}"
    assert np.array_equal(gv.view(np.uint32), rv.view(np.uint32))


@pytest.mark.parametrize("next_n,k", [(1, 1), (1, 7), (2, 64), (3, 333), (4, 1024)])
def test_matches_oracle(next_n, k):
    x, sl = W.topk_logits_input(6, next_n, 3000, seed=500 + k, lo=0, hi=3000)
    check(x, sl, next_n, 3000, k)


def test_ties_decided_by_position():
    x, sl = W.topk_logits_input(5, 2, 2500, seed=510, distinct=5, lo=1000)
    check(x, sl, 2, 2500, 600)


def test_fewer_candidates_than_k_and_empty_requests():
    x, sl = W.topk_logits_input(6, 1, 512, seed=511, lo=0, hi=40)
    sl[0] = 0
    check(x, sl, 1, 512, 100)


def test_max_context_clip_and_largest_k():
    x, sl = W.topk_logits_input(3, 1, 8192, seed=512, lo=6000)
    check(x, sl, 1, 5000, 4096)


def test_decode_sized_batch():
    x, sl = W.topk_logits_input(64, 1, 32768, seed=513, lo=1024, specials=False)
    check(x, sl, 1, 32768, 2048)


def test_indices_only():
    x, sl = W.topk_logits_input(4, 1, 1000, seed=514)
    gi, _ = run(x, sl, 1, 1000, 50, with_values=False)
    ri, _ = oracle.topk_logits(x, sl, 1, 1000, 50)
    assert np.array_equal(gi, ri)


def test_exact_threshold_with_ties_placed_by_position():
    # three levels, k = 1500 of 3000-4000: the keys equal to the threshold
    # outnumber k + 256, so the select runs all four passes; the keys above
    # it go through the bins, the tied ones take the last places by position
    x, sl = W.topk_logits_input(4, 2, 4000, seed=521, distinct=3, lo=3000)
    check(x, sl, 2, 4000, 1500)


def test_select_stops_after_the_third_pass():
    # values that agree in their top 16 bits: the second pass cannot narrow
    # the candidates, the third can
    x, sl = W.topk_logits_input(4, 1, 4000, seed=522, lo=3000, narrow=True, specials=False)
    check(x, sl, 1, 4000, 300)


def test_long_rows_sliced_into_shared_memory():
    # 36000 positions: slices of 4500 keys, beyond the registers' 4096
    x, sl = W.topk_logits_input(4, 1, 36000, seed=523, lo=33000)
    check(x, sl, 1, 36000, 2048)


def test_long_rows_read_from_global_memory():
    # 70000 positions: slices of 8750 keys, beyond the shared-memory copy
    x, sl = W.topk_logits_input(3, 1, 70000, seed=524, lo=60000)
    check(x, sl, 1, 70000, 1024)
