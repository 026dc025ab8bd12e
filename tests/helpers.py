"""Shared helpers for the GPU parity tests: upload seeded inputs, call the
library through its C ABI binding, and compare with the oracle.

Tolerances:
* fp8 logits: |gpu - oracle| <= 1e-3 * s_p * sum_h |w| |q.k| + 1e-6 at every
  meaningful position (p <= seq_lens[b] - next_n + t).
* bf16 scores: |gpu - oracle| <= 1e-3 * sum_d |q_d k_d| + 1e-6.
* Everything the library must not write keeps its sentinel bit pattern.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_attention_indexer_logits_gb300 as pml
from sparse_attention_indexer_logits_gb300 import workloads as W

FP8_REL = 1e-3
BF16_REL = 1e-3
ABS = 1e-6


def dev_tensor(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


class Fp8Device:
    """A problem's inputs resident on the GPU."""

    def __init__(self, p: W.Fp8Problem):
        self.p = p
        self.q = dev_tensor(p.q)
        self.kv = dev_tensor(p.kv_fused)
        self.w = dev_tensor(p.weights)
        self.seq_lens = dev_tensor(p.seq_lens)
        self.bt = dev_tensor(p.block_table)

    def run(self, max_context=None, num_ctas=0, schedule_meta=None, out=None):
        p = self.p
        mc = p.max_context if max_context is None else max_context
        if out is None:
            out = dev_tensor(W.sentinel_f32((p.batch * p.next_n, mc)))
        pml.pml_fp8_paged_mqa_logits(self.q, self.kv, self.w, self.seq_lens, self.bt, out, mc,
                                     p.next_n, schedule_meta=schedule_meta, num_ctas=num_ctas)
        return out


def run_fp8(p: W.Fp8Problem, **kw) -> np.ndarray:
    d = Fp8Device(p)
    out = d.run(**kw)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def oracle_fp8(p: W.Fp8Problem, max_context=None):
    mc = p.max_context if max_context is None else max_context
    return oracle.fp8_paged_mqa_logits(p.q, p.kv_fused, p.weights, p.seq_lens, p.block_table,
                                       next_n=p.next_n, max_context=mc)


def check_fp8(p: W.Fp8Problem, got: np.ndarray, ref=None, mag=None, max_context=None):
    """Tolerance over meaningful positions, finiteness over written ones,
    untouched sentinel everywhere else."""
    mc = p.max_context if max_context is None else max_context
    if ref is None:
        ref, mag = oracle_fp8(p, mc)
    n = p.next_n
    valid = oracle.fp8_valid_mask(p.seq_lens, n, mc)
    written = oracle.fp8_written_mask(p.seq_lens, n, mc)
    assert got.shape == ref.shape
    err = np.abs(got.astype(np.float64) - np.where(written, ref, 0.0))
    bound = FP8_REL * np.nan_to_num(mag) + ABS
    bad = valid & ~(err <= bound)
    if bad.any():
        r, c = np.argwhere(bad)[0]
        raise AssertionError(
            f"{int(bad.sum())} of {int(valid.sum())} logits outside tolerance; first at "
            f"row {r} pos {c}: gpu {got[r, c]!r} oracle {ref[r, c]!r} bound {bound[r, c]!r}")
    assert np.isfinite(got[written]).all(), "a written logit is not finite"
    untouched = got[~written].view(np.uint32) == W.SENTINEL_BITS
    assert untouched.all(), f"{int((~untouched).sum())} unwritten positions were modified"


def sub_problem(p: W.Fp8Problem, idx) -> W.Fp8Problem:
    """The same cache restricted to requests ``idx`` (for oracle sampling at full size)."""
    idx = np.asarray(idx)
    n = p.next_n
    rows = (idx[:, None] * n + np.arange(n)[None, :]).reshape(-1)
    return W.Fp8Problem(p.name + "_sub", p.seed, n, p.num_heads, p.q[rows], p.kv_fused,
                        p.weights[rows], p.seq_lens[idx], p.block_table[idx], p.max_context)


class Bf16Device:
    def __init__(self, p: W.Bf16Problem):
        self.p = p
        self.query = dev_tensor(p.query.view(np.int16)).view(torch.bfloat16)
        self.kc = dev_tensor(p.key_cache)
        self.bt = dev_tensor(p.block_table)
        self.cl = dev_tensor(p.context_lengths)
        self.req = dev_tensor(p.requests)

    def run(self, max_context=None, scores=None):
        p = self.p
        mc = p.max_context if max_context is None else max_context
        if scores is None:
            scores = dev_tensor(W.sentinel_f32((p.rows, mc)))
        pml.pml_indexer_scores_bf16(self.query, self.kc, p.page_stride_bytes, p.num_pages, self.bt,
                                    self.cl, self.req, scores, mc)
        return scores


def run_bf16(p: W.Bf16Problem, **kw) -> np.ndarray:
    d = Bf16Device(p)
    s = d.run(**kw)
    torch.cuda.synchronize()
    return s.cpu().numpy()


def check_bf16(p: W.Bf16Problem, got: np.ndarray, max_context=None, groups=None):
    """Compare (optionally only the listed groups) with the oracle."""
    mc = p.max_context if max_context is None else max_context
    G = p.group_size
    if groups is None:
        ref, mag = oracle.indexer_scores_bf16(p.query, p.key_cache, p.page_stride_bytes,
                                              p.block_table, p.context_lengths, p.requests, mc)
        got_rows = got
    else:
        groups = np.asarray(groups)
        rsel = (groups[:, None] * G + np.arange(G)[None, :]).reshape(-1)
        ref, mag = oracle.indexer_scores_bf16(p.query[rsel], p.key_cache, p.page_stride_bytes,
                                              p.block_table, p.context_lengths[groups],
                                              p.requests[groups], mc)
        got_rows = got[rsel]
    written = ~np.isnan(ref)
    err = np.abs(got_rows.astype(np.float64) - np.where(written, ref, 0.0))
    bound = BF16_REL * np.nan_to_num(mag) + ABS
    bad = written & ~(err <= bound)
    if bad.any():
        r, c = np.argwhere(bad)[0]
        raise AssertionError(f"{int(bad.sum())} scores outside tolerance; first at row {r} "
                             f"key {c}: gpu {got_rows[r, c]!r} oracle {ref[r, c]!r}")
    untouched = got_rows[~written].view(np.uint32) == W.SENTINEL_BITS
    assert untouched.all(), f"{int((~untouched).sum())} unwritten scores were modified"
