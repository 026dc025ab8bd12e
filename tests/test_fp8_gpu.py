"""GPU parity of pml_fp8_paged_mqa_logits against the CPU oracle, through the
C ABI (ctypes binding).

Cases span several 128-key tiles with ragged tails, every supported head
count and next_n, empty requests, lengths below next_n, a max_context below
the longest request, explicit schedules, many grid sizes, page permutation,
CUDA-graph replay with changed inputs, and the full-size decode / MTP /
skewed workloads on sampled requests.
"""
import numpy as np
import pytest
import torch

import oracle
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


def _status_clean():
    assert pml.pml_device_status(clear=True) == 0


def test_tiny_config():
    """batch 2, next_n 1, 8 heads, lengths {100, 37}, four shuffled blocks."""
    p = W.tiny()
    Hh.check_fp8(p, Hh.run_fp8(p))
    _status_clean()


@pytest.mark.parametrize("H", [8, 16, 32, 64])
@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_heads_and_slots(H, n):
    g = W.rng(1000 + H + n)
    lens = g.integers(1, 700, size=5)
    lens[1] = 0
    lens[2] = 128          # exactly one full tile
    lens[3] = 64 * 3 + 1   # ragged tail: two tiles, the second with one key
    p = W.fp8_problem(f"hn_{H}_{n}", lens, n, H, seed=2000 + H + n, extra_blocks=2)
    Hh.check_fp8(p, Hh.run_fp8(p))
    _status_clean()


def test_small_decode_many_tiles():
    p = W.decode(seed=11, batch=8, lo=1, hi=3000)
    Hh.check_fp8(p, Hh.run_fp8(p))


@pytest.mark.parametrize("n", [2, 4])
def test_small_mtp(n):
    p = W.mtp(next_n=n, seed=12 + n, batch=6, lo=1, hi=2500)
    Hh.check_fp8(p, Hh.run_fp8(p))


def test_lengths_below_next_n_and_single_keys():
    p = W.fp8_problem("short", [1, 2, 3, 0, 4, 65, 63], 4, 64, seed=13)
    Hh.check_fp8(p, Hh.run_fp8(p))


def test_all_requests_empty():
    p = W.fp8_problem("empty", [0, 0, 0], 2, 32, seed=14, max_context=64)
    got = Hh.run_fp8(p)
    assert (got.view(np.uint32) == W.SENTINEL_BITS).all()
    _status_clean()


@pytest.mark.parametrize("num_ctas", [1, 2, 3, 7, 64, 152, 300])
def test_grid_sizes_bit_identical(num_ctas):
    """Any persistent grid size gives the same logits (each key's arithmetic
    is independent of which CTA does it); explicit schedules agree with the
    in-kernel one bit for bit."""
    p = W.fp8_problem("grid", [1000, 0, 37, 2049, 130, 64], 2, 64, seed=15)
    d = Hh.Fp8Device(p)
    base = d.run().cpu().numpy()
    Hh.check_fp8(p, base)
    other = d.run(num_ctas=num_ctas).cpu().numpy()
    assert np.array_equal(base.view(np.uint32), other.view(np.uint32))
    meta = pml.pml_schedule(d.seq_lens, num_ctas, p.next_n)
    with_meta = d.run(num_ctas=num_ctas, schedule_meta=meta).cpu().numpy()
    assert np.array_equal(base.view(np.uint32), with_meta.view(np.uint32))


def test_page_permutation_bit_identical():
    p = W.fp8_problem("perm", [700, 1, 390, 64, 0, 257], 3, 32, seed=16, extra_blocks=5)
    base = Hh.run_fp8(p)
    g = W.rng(17)
    perm = g.permutation(p.num_blocks)
    kv2 = np.empty_like(p.kv_fused)
    kv2[perm] = p.kv_fused
    p2 = W.Fp8Problem(p.name, p.seed, p.next_n, p.num_heads, p.q, kv2, p.weights, p.seq_lens,
                      perm[p.block_table].astype(np.int32), p.max_context)
    assert np.array_equal(base.view(np.uint32), Hh.run_fp8(p2).view(np.uint32))


def test_max_context_below_longest_request():
    """Positions at or past max_context are neither computed nor written."""
    p = W.fp8_problem("mc", [300, 90, 1000], 2, 16, seed=18)
    mc = 200
    got = Hh.run_fp8(p, max_context=mc)
    Hh.check_fp8(p, got, max_context=mc)


def test_strided_out_and_block_table():
    """Row strides of out and block_table larger than their widths."""
    p = W.fp8_problem("strided", [500, 77], 2, 64, seed=19)
    d = Hh.Fp8Device(p)
    big = Hh.dev_tensor(W.sentinel_f32((p.batch * 2, p.max_context + 61)))
    out_view = big[:, :p.max_context]
    bt_big = torch.zeros((p.batch, p.block_table.shape[1] + 3), dtype=torch.int32, device="cuda")
    bt_big[:, :p.block_table.shape[1]] = d.bt
    d.bt = bt_big[:, :p.block_table.shape[1]]
    d.run(out=out_view)
    torch.cuda.synchronize()
    full = big.cpu().numpy()
    Hh.check_fp8(p, np.ascontiguousarray(full[:, :p.max_context]))
    assert (full[:, p.max_context:].view(np.uint32) == W.SENTINEL_BITS).all()


def test_scale_doubling_doubles_logits_exactly():
    p = W.fp8_problem("scale2", [400, 129], 1, 64, seed=20, poison=False)
    base = Hh.run_fp8(p)
    kv2 = p.kv_fused.copy()
    kv2[:, W.BLOCK_KEY_BYTES:].view("<f4")[:] *= 2
    p2 = W.Fp8Problem(p.name, p.seed, 1, 64, p.q, kv2, p.weights, p.seq_lens, p.block_table,
                      p.max_context)
    dbl = Hh.run_fp8(p2)
    written = oracle.fp8_written_mask(p.seq_lens, 1, p.max_context)
    assert np.array_equal(dbl[written], 2 * base[written])


def test_bad_block_index_is_flagged_not_read():
    """A block_table entry outside the cache sets PML_STATUS_BAD_BLOCK and is
    replaced by block 0; nothing faults."""
    p = W.fp8_problem("badblk", [130], 1, 8, seed=21)
    d = Hh.Fp8Device(p)
    bt = p.block_table.copy()
    bt[0, 1] = p.num_blocks + 1000
    d.bt = Hh.dev_tensor(bt)
    pml.pml_device_status(clear=True)
    d.run()
    assert pml.pml_device_status(clear=True) & pml.STATUS_BAD_BLOCK


def test_graph_replay_with_changed_inputs():
    """Schedule + logits captured once in a CUDA graph; the contents of
    seq_lens, q, weights and block_table change between replays."""
    B, n, H = 6, 2, 64
    g = W.rng(22)
    lens_a = g.integers(1, 900, size=B).astype(np.int32)
    lens_b = g.integers(0, 1500, size=B).astype(np.int32)
    width = W.blocks_for(1500)
    need_a = sum(W.blocks_for(x) for x in lens_a)
    need_b = sum(W.blocks_for(x) for x in lens_b)
    pool = max(need_a, need_b)
    # the same pool size for both, so one cache buffer serves both
    pa = W.fp8_problem("graph_a", lens_a, n, H, seed=23, bt_width=width, max_context=1500,
                       extra_blocks=pool - need_a)
    pb = W.fp8_problem("graph_b", lens_b, n, H, seed=24, bt_width=width, max_context=1500,
                       extra_blocks=pool - need_b)
    assert pb.num_blocks == pa.num_blocks
    d = Hh.Fp8Device(pa)
    num_ctas = 40
    meta = torch.empty((num_ctas + 1, 2), dtype=torch.int32, device="cuda")
    out = Hh.dev_tensor(W.sentinel_f32((B * n, 1500)))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pml.pml_schedule(d.seq_lens, num_ctas, n, schedule_meta=meta)
        d.run(max_context=1500, num_ctas=num_ctas, schedule_meta=meta, out=out)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pml.pml_schedule(d.seq_lens, num_ctas, n, schedule_meta=meta)
        d.run(max_context=1500, num_ctas=num_ctas, schedule_meta=meta, out=out)
    for prob in (pa, pb, pa):
        out.copy_(Hh.dev_tensor(W.sentinel_f32((B * n, 1500))))
        for dst, src in ((d.q, prob.q), (d.kv, prob.kv_fused), (d.w, prob.weights),
                         (d.seq_lens, prob.seq_lens), (d.bt, prob.block_table)):
            dst.copy_(Hh.dev_tensor(src))
        graph.replay()
        torch.cuda.synchronize()
        Hh.check_fp8(prob, out.cpu().numpy(), max_context=1500)
    _status_clean()


# ------------------------------------------------------------------ full sizes

def _full_size_sampled(p, sample):
    d = Hh.Fp8Device(p)
    out = d.run()
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    written = oracle.fp8_written_mask(p.seq_lens, p.next_n, p.max_context)
    assert np.isfinite(got[written]).all()
    assert (got[~written].view(np.uint32) == W.SENTINEL_BITS).all()
    sp = Hh.sub_problem(p, sample)
    n = p.next_n
    rows = (np.asarray(sample)[:, None] * n + np.arange(n)[None, :]).reshape(-1)
    Hh.check_fp8(sp, np.ascontiguousarray(got[rows]))
    _status_clean()


def test_full_decode_sampled():
    """Decode: batch 64, next_n 1, 64 heads, lengths U[1024, 32768]."""
    p = W.decode()
    _full_size_sampled(p, [0, 17, 40, 63])


@pytest.mark.parametrize("n", [2, 4])
def test_full_mtp_sampled(n):
    """MTP verify: batch 32, 64 heads, lengths U[8192, 65536]."""
    p = W.mtp(next_n=n)
    _full_size_sampled(p, [3, 31])


@pytest.mark.parametrize("order", ["shuffled", "first", "last"])
def test_full_skewed(order):
    """One 131072-token request, three empty, twelve short: empty rows stay
    untouched and the long request is checked in full."""
    p = W.skewed(order=order)
    long_idx = int(np.argmax(p.seq_lens))
    short_idx = int(np.argsort(p.seq_lens)[-2])
    _full_size_sampled(p, [long_idx, short_idx])
