"""pml_schedule on the GPU equals the oracle's schedule bit for bit."""
import numpy as np
import pytest

import oracle
import sparse_attention_indexer_logits_gb300 as pml
from sparse_attention_indexer_logits_gb300 import workloads as W
from tests import helpers as Hh

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _build():
    import __graft_entry__
    __graft_entry__.build()
    yield


@pytest.mark.parametrize("seed", range(8))
def test_random_schedules(seed):
    g = W.rng(500 + seed)
    B = int(g.integers(1, 3000))
    lens = g.integers(0, 70000, size=B).astype(np.int32)
    lens[g.random(B) < 0.2] = 0
    for G in (1, 5, 152, int(g.integers(1, 2000))):
        got = pml.pml_schedule(Hh.dev_tensor(lens), G).cpu().numpy()
        ref, _ = oracle.schedule(lens, G)
        assert np.array_equal(got, ref), (B, G)


def _blocks_per_cta(meta, seq_lens):
    """Blocks each CTA's range holds, read off the GPU schedule: the global
    index of each (request, block) start, differenced."""
    nb = (np.maximum(seq_lens.astype(np.int64), 0) + 63) // 64
    prefix = np.concatenate([[0], np.cumsum(nb)])
    starts = prefix[meta[:, 0]] + meta[:, 1]
    return np.diff(starts), int(prefix[-1])


def test_workload_schedules():
    for p in (W.tiny(), W.decode(), W.mtp(4), W.skewed()):
        for G in (148, 152, 304):
            got = pml.pml_schedule(Hh.dev_tensor(p.seq_lens), G, p.next_n).cpu().numpy()
            ref, total = oracle.schedule(p.seq_lens, G)
            assert np.array_equal(got, ref)
            # load balance of the persistent grid, on the GPU's own output:
            # every CTA holds floor(T/G) or ceil(T/G) blocks, T in all
            sizes, t = _blocks_per_cta(got, p.seq_lens)
            assert t == total and int(sizes.sum()) == total
            assert sizes.max() <= -(-total // G) and sizes.min() >= total // G, (G, sizes.min(),
                                                                                 sizes.max())


def test_empty_and_zero_batches():
    for lens in ([0], [0, 0, 0], [64], [1] * 300):
        lens = np.array(lens, dtype=np.int32)
        for G in (1, 3, 152):
            got = pml.pml_schedule(Hh.dev_tensor(lens), G).cpu().numpy()
            ref, _ = oracle.schedule(lens, G)
            assert np.array_equal(got, ref)
