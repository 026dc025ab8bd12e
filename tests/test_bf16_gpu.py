"""GPU parity of pml_indexer_scores_bf16 against the CPU oracle, through the
C ABI: group sizes 1..8, lengths with zeros and ragged tails, shared and
private requests, padded page strides, garbage request entries for empty
groups, max_context clipping, and the full-size workload (256 groups,
lengths U[0, 65536]) on sampled groups."""
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
    pml.pml_device_status(clear=True)
    yield


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 8])
def test_group_sizes(G):
    p = W.indexer(group_size=G, seed=300 + G, groups=9, max_context=1100, min_zero=2)
    Hh.check_bf16(p, Hh.run_bf16(p))
    assert pml.pml_device_status(clear=True) == 0


def test_shared_requests_and_padded_pages():
    p = W.indexer(group_size=4, seed=310, groups=12, max_context=900, num_requests=3,
                  shared_requests=True, page_pad_bytes=16 * 7, min_zero=3)
    Hh.check_bf16(p, Hh.run_bf16(p))
    assert pml.pml_device_status(clear=True) == 0


def test_max_context_clip():
    p = W.indexer(group_size=2, seed=311, groups=5, max_context=700, min_zero=0, lo=300)
    got = Hh.run_bf16(p, max_context=256)
    Hh.check_bf16(p, got, max_context=256)


def test_single_row():
    p = W.indexer(group_size=1, seed=312, groups=1, max_context=200, min_zero=0, lo=130)
    Hh.check_bf16(p, Hh.run_bf16(p))


def test_all_groups_empty():
    p = W.indexer(group_size=3, seed=313, groups=4, max_context=128, min_zero=4)
    got = Hh.run_bf16(p)
    assert (got.view(np.uint32) == W.SENTINEL_BITS).all()
    assert pml.pml_device_status(clear=True) == 0


@pytest.mark.parametrize("G", [1, 8])
def test_full_size_sampled(G):
    """256 groups, lengths U[0, 65536] with forced zeros, scores [rows, 65536]."""
    p = W.indexer(group_size=G)
    d = Hh.Bf16Device(p)
    s = d.run()
    torch.cuda.synchronize()
    got = s.cpu().numpy()
    lens = np.repeat(p.context_lengths, G)
    col = np.arange(p.max_context)[None, :]
    written = col < lens[:, None]
    assert np.isfinite(got[written]).all()
    assert (got[~written].view(np.uint32) == W.SENTINEL_BITS).all()
    order = np.argsort(p.context_lengths)
    sample = [int(order[-1]), int(order[len(order) // 2]), int(order[0])]
    Hh.check_bf16(p, got, groups=sample)
    assert pml.pml_device_status(clear=True) == 0
