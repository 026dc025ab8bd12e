"""GPU parity of pml_indexer_scores_nvfp4 against the CPU oracle, through the
C ABI ("flashinfer.sdsa.indexer_scores", NVFP4 forms): group sizes 1..8,
fused (keys then scales in one page) and separate caches, scale pages only
8-byte aligned, padded key pages, garbage request entries for empty groups,
max_context clipping, an out-of-range page, every E4M3 scale code (zeros,
subnormals, negatives, NaN) on either operand, and the full-size workload
(256 groups, lengths U[0, 65536]) on sampled groups.

Tolerance: |gpu - oracle| <= 1e-3 * sum_d |q_d k_d| + 1e-6, the bf16 path's
bound.  (Every product of two dequantised values is exact in fp32; only the
fp32 accumulation rounds.)  A score the oracle finds NaN -- a NaN scale on
either side reaches every score of its row or key -- must be NaN."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_indexer_logits_gb300 as pml
from sparse_attention_indexer_logits_gb300 import workloads as W
from tests.helpers import ABS, BF16_REL, dev_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _build():
    import __graft_entry__
    __graft_entry__.build()
    pml.pml_device_status(clear=True)
    yield


class Nvfp4Device:
    def __init__(self, p: W.Nvfp4Problem):
        self.p = p
        self.q = dev_tensor(p.query)
        self.qs = dev_tensor(p.query_scales)
        self.kb = dev_tensor(p.key_buf)
        self.sb = self.kb if p.fused else dev_tensor(p.scale_buf)
        self.bt = dev_tensor(p.block_table)
        self.cl = dev_tensor(p.context_lengths)
        self.req = dev_tensor(p.requests)

    def run(self, max_context=None, block_table=None):
        p = self.p
        mc = p.max_context if max_context is None else max_context
        scores = dev_tensor(W.sentinel_f32((p.rows, mc)))
        pml.pml_indexer_scores_nvfp4(self.q, self.qs, self.kb[p.key_off:], p.page_stride_bytes,
                                     self.sb[p.scale_off:], p.scale_page_stride_bytes, p.num_pages,
                                     self.bt if block_table is None else block_table, self.cl,
                                     self.req, scores, mc)
        torch.cuda.synchronize()
        return scores.cpu().numpy()


def check(p: W.Nvfp4Problem, got: np.ndarray, max_context=None, groups=None):
    mc = p.max_context if max_context is None else max_context
    G = p.group_size
    rows = np.arange(p.rows) if groups is None else \
        (np.asarray(groups)[:, None] * G + np.arange(G)[None, :]).reshape(-1)
    gsel = np.arange(p.groups) if groups is None else np.asarray(groups)
    ref, mag = oracle.indexer_scores_nvfp4(p.query[rows], p.query_scales[rows], p.key_view(),
                                           p.page_stride_bytes, p.scale_view(),
                                           p.scale_page_stride_bytes, p.block_table,
                                           p.context_lengths[gsel], p.requests[gsel], mc)
    g = got[rows]
    lens = np.minimum(np.repeat(p.context_lengths[gsel], G), mc)
    written = np.arange(mc)[None, :] < lens[:, None]
    nan = written & np.isnan(ref)
    fin = written & ~nan
    err = np.abs(g.astype(np.float64) - np.where(fin, ref, 0.0))
    bound = BF16_REL * np.where(fin, mag, 0.0) + ABS
    bad = fin & ~(err <= bound)
    assert not bad.any(), (f"{int(bad.sum())} of {int(fin.sum())} scores outside tolerance; first "
                           f"{np.argwhere(bad)[0]}: gpu {g[bad][0]!r} oracle {ref[bad][0]!r}")
    assert np.isnan(g[nan]).all(), f"{int((~np.isnan(g[nan])).sum())} scores should be NaN"
    assert (g[~written].view(np.uint32) == W.SENTINEL_BITS).all(), "unwritten entry modified"
    return int(nan.sum()), int(fin.sum())


@pytest.mark.parametrize("G", [1, 2, 3, 5, 8])
def test_group_sizes(G):
    p = W.indexer_nvfp4(G, seed=400 + G, groups=9, max_context=1100, min_zero=2)
    check(p, Nvfp4Device(p).run())
    assert pml.pml_device_status(clear=True) == 0


@pytest.mark.parametrize("page_pad,scale_pad", [(0, 0), (16, 8), (48, 24)])
def test_separate_caches_and_strides(page_pad, scale_pad):
    """Key pages 16-byte multiples apart, scale pages 8-byte multiples (an odd
    multiple of 8 too: the scale copies need only 8-byte alignment)."""
    p = W.indexer_nvfp4(4, seed=410 + page_pad + scale_pad, groups=7, max_context=900,
                        min_zero=1, fused=False, page_pad_bytes=page_pad,
                        scale_pad_bytes=scale_pad)
    check(p, Nvfp4Device(p).run())
    assert pml.pml_device_status(clear=True) == 0


def test_fused_padded_pages_and_max_context_clip():
    p = W.indexer_nvfp4(2, seed=420, groups=6, max_context=800, min_zero=0, lo=300,
                        page_pad_bytes=32)
    check(p, Nvfp4Device(p).run(max_context=320), max_context=320)


def test_all_groups_empty():
    p = W.indexer_nvfp4(3, seed=421, groups=4, max_context=128, min_zero=4)
    got = Nvfp4Device(p).run()
    assert (got.view(np.uint32) == W.SENTINEL_BITS).all()
    assert pml.pml_device_status(clear=True) == 0


def test_out_of_range_page_is_flagged():
    p = W.indexer_nvfp4(1, seed=422, groups=3, max_context=200, min_zero=0, lo=100, poison=False)
    d = Nvfp4Device(p)
    bt = p.block_table.copy()
    bt[1, 0] = p.num_pages + 5
    pml.pml_device_status(clear=True)
    d.run(block_table=dev_tensor(bt))
    assert pml.pml_device_status(clear=True) & pml.STATUS_BAD_BLOCK


@pytest.mark.parametrize("G,fused", [(8, True), (3, False)])
def test_every_scale_code(G, fused):
    """Scale bytes uniform over all 256 E4M3 codes for queries and keys: the
    MMA reads scales without their sign, so negative ones are applied to the
    codes; NaN scales make their rows' or keys' scores NaN."""
    p = W.indexer_nvfp4(G, seed=430 + G, groups=10, max_context=1500, min_zero=1, lo=200,
                        fused=fused, scales="all")
    nans, finite = check(p, Nvfp4Device(p).run())
    assert nans > 0 and finite > 0
    assert pml.pml_device_status(clear=True) == 0


@pytest.mark.parametrize("G", [2, 8])
def test_negative_scales(G):
    """Every scale of both operands negative (the sign bits flip the codes of
    their blocks on the way to the tensor cores)."""
    p = W.indexer_nvfp4(G, seed=440 + G, groups=8, max_context=1300, min_zero=1,
                        scales="negative")
    check(p, Nvfp4Device(p).run())
    assert pml.pml_device_status(clear=True) == 0


def test_one_negative_key_block():
    """A single negative scale block in one key among positive ones."""
    p = W.indexer_nvfp4(4, seed=450, groups=3, max_context=400, min_zero=0, lo=300,
                        poison=False)
    page = int(p.block_table[1, 2])
    at = p.scale_off + page * p.scale_page_stride_bytes + 37 * 8 + 5   # key 37, block 5
    p.scale_buf[at] |= 0x80
    got = Nvfp4Device(p).run()
    check(p, got)


@pytest.mark.parametrize("G", [1, 8])
def test_full_size_sampled(G):
    """256 groups, lengths U[0, 65536] with forced zeros, scores [rows, 65536]."""
    p = W.indexer_nvfp4(G)
    got = Nvfp4Device(p).run()
    lens = np.repeat(p.context_lengths, G)
    written = np.arange(p.max_context)[None, :] < lens[:, None]
    assert np.isfinite(got[written]).all()
    assert (got[~written].view(np.uint32) == W.SENTINEL_BITS).all()
    order = np.argsort(p.context_lengths)
    check(p, got, groups=[int(order[-1]), int(order[len(order) // 2]), int(order[0])])
    assert pml.pml_device_status(clear=True) == 0
