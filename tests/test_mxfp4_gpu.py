"""MXFP4 paged MQA logits on the GPU against the fp64 oracle
("flashinfer.attn_scores": the MXFP4 variant -- block scales per 32 values
folded into the dequantised operands, 64 heads of 128, bf16 output by
default).

The GPU path rewrites every row as E4M3 values times one power of two and
runs the fp8 logits engine, so its error bound is the fp8 one: each logit is
computed in fp32 from exact products, |gpu - oracle| <= 1e-3 * mag + 1e-6
(mag = sum_h |w| |q.k|), plus half a bf16 ulp (<= 2^-9 of the value, 2^-8
taken) for bf16 output.  Inputs whose group scales lie within 8 binades are
exact in E4M3 and must leave the status word clean; unwritten positions keep
their sentinel."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_indexer_logits_gb300 as pml
from sparse_attention_indexer_logits_gb300 import workloads as W

from tests.helpers import ABS, FP8_REL, dev_tensor

pytestmark = pytest.mark.gpu
BF16_OUT_REL = 2.0 ** -8
STATUS_FP4_INEXACT = 8


def run(p: W.Mxfp4Problem, dtype=torch.bfloat16, mc=None):
    mc = p.max_context if mc is None else mc
    rows = p.batch * p.next_n
    if dtype == torch.bfloat16:
        out = dev_tensor(W.sentinel_bf16_bits((rows, mc)).view(np.int16)).view(torch.bfloat16)
    else:
        out = dev_tensor(W.sentinel_f32((rows, mc)))
    pml.pml_device_status(clear=True)
    pml.pml_fp4_paged_mqa_logits(dev_tensor(p.q), dev_tensor(p.q_sf), dev_tensor(p.kv),
                                 dev_tensor(p.weights), dev_tensor(p.seq_lens),
                                 dev_tensor(p.block_table), out, mc, p.next_n)
    torch.cuda.synchronize()
    return out, pml.pml_device_status(clear=True)


def check(p: W.Mxfp4Problem, out: torch.Tensor, mc=None):
    mc = p.max_context if mc is None else mc
    ref, mag = oracle.fp4_paged_mqa_logits(p.q, p.q_sf, p.kv, p.weights, p.seq_lens,
                                           p.block_table, p.next_n, mc)
    bf16 = out.dtype == torch.bfloat16
    got = out.float().cpu().numpy().astype(np.float64)
    valid = oracle.fp8_valid_mask(p.seq_lens, p.next_n, mc)
    written = oracle.fp8_written_mask(p.seq_lens, p.next_n, mc)
    refw = np.where(written, ref, 0.0)
    rel = BF16_OUT_REL if bf16 else 0.0
    bound = FP8_REL * np.nan_to_num(mag) * (1 + rel) + ABS + rel * np.abs(refw)
    bad = valid & ~(np.abs(got - refw) <= bound)
    assert not bad.any(), f"{int(bad.sum())} of {int(valid.sum())} logits outside tolerance"
    assert np.isfinite(got[written]).all()
    if bf16:
        bits = out.view(torch.int16).cpu().numpy().view(np.uint16)
        assert (bits[~written] == W.SENTINEL_BF16_BITS).all(), "an unwritten position was modified"
    else:
        bits = out.cpu().numpy().view(np.uint32)
        assert (bits[~written] == W.SENTINEL_BITS).all(), "an unwritten position was modified"


@pytest.mark.parametrize("next_n", [1, 2, 3, 4])
def test_matches_oracle_bf16_out(next_n):
    p = W.mxfp4_problem(f"mx_n{next_n}", [1000, 0, 130, 64, 2049, 7], next_n, seed=60 + next_n)
    out, status = run(p)
    check(p, out)
    assert status == 0


def test_matches_oracle_fp32_out_and_max_context_clip():
    p = W.mxfp4_problem("mx_f32", [900, 300, 65, 1], 2, seed=65)
    out, status = run(p, torch.float32, mc=512)
    check(p, out, mc=512)
    assert status == 0


def test_decode_shape_batch8():
    """The decode shape (64 heads, lengths up to 32K) on 8 requests, every
    position checked."""
    p = W.mxfp4_decode(seed=66, batch=8)
    out, status = run(p)
    check(p, out)
    assert status == 0


def test_wide_scale_spread_is_flagged():
    """A key whose group scales are 12 binades apart and whose small group
    holds the smallest codes cannot be held in E4M3: the status word says so
    (the logits are still written, rounded)."""
    p = W.mxfp4_problem("mx_spread", [64], 1, seed=67, poison=False)
    at = W.MXFP4_BLOCK_CODE_BYTES + 5 * 4                # key 5's four scale bytes
    p.kv[0, at:at + 4] = [127 + 6, 127 - 6, 127, 127]
    p.kv[0, 5 * 64 + 16:5 * 64 + 32] = 0x11              # group 1 of key 5: codes 0.5
    out, status = run(p, torch.float32)
    assert status & STATUS_FP4_INEXACT
    assert torch.isfinite(out[0, :64]).all()
