"""fp8 logits with output_dtype = bfloat16 ("flashinfer.attn_scores": the
fp8 call's output_dtype option, float32 by default).

The kernel computes each logit in fp32 exactly as for fp32 output and rounds
it to the nearest bf16 (ties to even).  Against the fp64 oracle the bound is
the fp32 one plus that rounding: |gpu - oracle| <= 1e-3 * mag * (1 + 2^-8)
+ 1e-6 + 2^-8 * |oracle| (half a bf16 ulp is at most 2^-9 of the value; the
factor 2 is margin).  Unwritten positions keep a bf16 sentinel pattern."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_indexer_logits_gb300 as pml
from sparse_attention_indexer_logits_gb300 import workloads as W

from tests.helpers import ABS, FP8_REL, Fp8Device, dev_tensor, oracle_fp8

pytestmark = pytest.mark.gpu
BF16_OUT_REL = 2.0 ** -8


def run_bf16_out(d: Fp8Device, mc=None, num_ctas=0):
    p = d.p
    mc = p.max_context if mc is None else mc
    bits = dev_tensor(W.sentinel_bf16_bits((p.batch * p.next_n, mc)).view(np.int16))
    out = bits.view(torch.bfloat16)
    pml.pml_fp8_paged_mqa_logits_ex(d.q, d.kv, d.w, d.seq_lens, d.bt, out, mc, p.next_n,
                                    num_ctas=num_ctas)
    torch.cuda.synchronize()
    return out


def check_bf16_out(p, out: torch.Tensor, mc=None):
    mc = p.max_context if mc is None else mc
    ref, mag = oracle_fp8(p, mc)
    got = out.float().cpu().numpy().astype(np.float64)
    bits = out.view(torch.int16).cpu().numpy().view(np.uint16)
    valid = oracle.fp8_valid_mask(p.seq_lens, p.next_n, mc)
    written = oracle.fp8_written_mask(p.seq_lens, p.next_n, mc)
    refw = np.where(written, ref, 0.0)
    bound = FP8_REL * np.nan_to_num(mag) * (1 + BF16_OUT_REL) + ABS + BF16_OUT_REL * np.abs(refw)
    bad = valid & ~(np.abs(got - refw) <= bound)
    assert not bad.any(), f"{int(bad.sum())} of {int(valid.sum())} bf16 logits outside tolerance"
    assert np.isfinite(got[written]).all()
    assert (bits[~written] == W.SENTINEL_BF16_BITS).all(), "an unwritten position was modified"


@pytest.mark.parametrize("heads,next_n", [(8, 1), (64, 1), (32, 2), (64, 3), (64, 4)])
def test_bf16_output_matches_oracle(heads, next_n):
    p = W.fp8_problem(f"bf16out_h{heads}n{next_n}", [1000, 0, 130, 64, 2049, 7], next_n, heads,
                      seed=40 + heads + next_n)
    d = Fp8Device(p)
    check_bf16_out(p, run_bf16_out(d))


def test_bf16_output_is_the_fp32_output_rounded():
    """Same kernel, two output types: the bf16 logits are the fp32 ones rounded
    to nearest even, bit for bit (torch's fp32 -> bf16 cast rounds that way)."""
    p = W.fp8_problem("bf16out_round", [3000, 517, 64, 1], 2, 64, seed=47)
    d = Fp8Device(p)
    f32 = d.run()
    b16 = run_bf16_out(d)
    written = torch.from_numpy(oracle.fp8_written_mask(p.seq_lens, p.next_n, p.max_context))
    want = f32.to(torch.bfloat16).view(torch.int16).cpu()[written]
    have = b16.view(torch.int16).cpu()[written]
    assert torch.equal(want, have)


def test_bf16_output_keyword_wrapper_and_max_context():
    p = W.fp8_problem("bf16out_kw", [900, 300], 1, 16, seed=48)
    d = Fp8Device(p)
    mc = 512                                        # clips the longer request
    out = torch.full((p.batch, mc), float("-inf"), dtype=torch.bfloat16, device="cuda")
    bits = torch.from_numpy(W.sentinel_bf16_bits(out.shape).view(np.int16)).cuda()
    out.view(torch.int16).copy_(bits)
    pml.fp8_paged_mqa_logits(d.q, d.kv, d.w, d.seq_lens, d.bt, max_context=mc, out=out,
                             output_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    check_bf16_out(p, out, mc)
