"""The allocation-free logits entry point against the regular one.

pml_fp8_paged_mqa_logits_noalloc serves callers that cannot obtain device
memory of their own (plugins inside a runtime that owns every allocation,
serving loops under a pool that forbids raw cudaMalloc): it keeps the per-CTA
schedule in a fixed array inside the library instead of a caller buffer.
These tests call it through the C ABI twice in a row, on different problems
and grid sizes, and require the same logits as the regular two-step call
(pml_schedule into a caller buffer, then pml_fp8_paged_mqa_logits), within the
tolerance the other parity tests use.  This file is collected last so that a
run stopping at the first failure has run every other test first.
"""
import numpy as np
import pytest
import torch

import sparse_attention_indexer_logits_gb300 as pml
from sparse_attention_indexer_logits_gb300 import workloads as W
from tests import helpers as Hh

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _build():
    import __graft_entry__
    __graft_entry__.build()
    yield


def _regular(d, num_ctas):
    p = d.p
    out = Hh.dev_tensor(W.sentinel_f32((p.batch * p.next_n, p.max_context)))
    meta = pml.pml_schedule(d.seq_lens, num_ctas, p.next_n)
    pml.pml_fp8_paged_mqa_logits(d.q, d.kv, d.w, d.seq_lens, d.bt, out, p.max_context, p.next_n,
                                 schedule_meta=meta, num_ctas=num_ctas)
    return out


def _noalloc(d, num_ctas):
    p = d.p
    out = Hh.dev_tensor(W.sentinel_f32((p.batch * p.next_n, p.max_context)))
    pml.pml_fp8_paged_mqa_logits_noalloc(d.q, d.kv, d.w, d.seq_lens, d.bt, out, p.max_context,
                                         p.next_n, num_ctas=num_ctas)
    return out


def test_noalloc_matches_regular_entry_point_twice_in_a_row():
    pml.pml_device_status(clear=True)
    cases = [
        (W.fp8_problem("na1", [1000, 0, 37, 2049, 130, 64], 2, 64, seed=71), 152),
        (W.fp8_problem("na2", [3000, 5, 0, 700], 1, 32, seed=72), 40),
    ]
    for p, num_ctas in cases:
        d = Hh.Fp8Device(p)
        ref = _regular(d, num_ctas)
        got = _noalloc(d, num_ctas)
        torch.cuda.synchronize()
        ref_np, got_np = ref.cpu().numpy(), got.cpu().numpy()
        # same tolerance as the parity tests, against the oracle and each other
        Hh.check_fp8(p, got_np)
        written = ref_np.view(np.uint32) != W.SENTINEL_BITS
        assert np.array_equal(written, got_np.view(np.uint32) != W.SENTINEL_BITS)
        err = np.abs(got_np[written].astype(np.float64) - ref_np[written])
        assert (err <= Hh.FP8_REL * np.abs(ref_np[written]) + Hh.ABS).all()
    assert pml.pml_device_status(clear=True) == 0


def test_noalloc_default_grid_and_limit():
    p = W.decode(seed=73, batch=8, lo=1, hi=4000)
    d = Hh.Fp8Device(p)
    got = _noalloc(d, 0).cpu().numpy()
    Hh.check_fp8(p, got)
    limit = pml.lib().pml_noalloc_max_ctas()
    assert limit == 1024
    out = Hh.dev_tensor(W.sentinel_f32((p.batch, p.max_context)))
    with pytest.raises(pml.PmlError):
        pml.pml_fp8_paged_mqa_logits_noalloc(d.q, d.kv, d.w, d.seq_lens, d.bt, out, p.max_context,
                                             p.next_n, num_ctas=limit + 1)
    torch.cuda.synchronize()
    assert (out.cpu().numpy().view(np.uint32) == W.SENTINEL_BITS).all()
