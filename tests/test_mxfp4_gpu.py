"""MXFP4 paged MQA logits on the GPU against the fp64 oracle
("flashinfer.attn_scores": the MXFP4 variant -- block scales per 32 values
folded into the dequantised operands, 64 heads of 128, bf16 output by
default).

The GPU path gives every row (a key, or one head of a slot) a frame, its
largest E8M0 exponent, and hands the block-scaled tensor cores the codes as
stored with the scales relative to the frame, so each block's terms are exact
in fp32 and the frames are applied after the weighted sum.  Its bound is the
fp8 one: |gpu - oracle| <= 1e-3 * mag + 1e-6 (mag = sum_h |w| |q.k|), plus
half a bf16 ulp (<= 2^-9 of the value, 2^-8 taken) for bf16 output.  A logit
beyond the output type's range must be the infinity of its sign (either is
accepted within 2^-7 of the largest finite value).

The scale domain is the pages' whole one: E8M0 exponents over every finite
value (2^-127 .. 2^127), each row's four groups drawn independently.  Where
a key's and a query row's scale spreads add up to more than 124 binades
the products below 2^-124 of their frames may be dropped; the status word
says so (the complementary-spread case below), and inputs within that reach
must leave it clean."""
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
FP32_MAX = float(np.finfo(np.float32).max)
BF16_MAX = float.fromhex("0x1.fep127")


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
    with np.errstate(invalid="ignore", over="ignore"):
        close = np.abs(got - refw) <= bound
        top = BF16_MAX if bf16 else FP32_MAX
        beyond = np.abs(refw) > top
        edge = np.abs(np.abs(refw) - top) <= 2.0 ** -7 * top
        signed_inf = np.isinf(got) & (np.sign(got) == np.sign(refw))
    good = close | ((beyond | edge) & signed_inf)
    bad = valid & ~good
    assert not bad.any(), (f"{int(bad.sum())} of {int(valid.sum())} logits outside tolerance; "
                           f"first {np.argwhere(bad)[0]}: gpu {got[bad][0]!r} oracle {refw[bad][0]!r}")
    assert not np.isnan(got[written]).any()
    if bf16:
        bits = out.view(torch.int16).cpu().numpy().view(np.uint16)
        assert (bits[~written] == W.SENTINEL_BF16_BITS).all(), "an unwritten position was modified"
    else:
        bits = out.cpu().numpy().view(np.uint32)
        assert (bits[~written] == W.SENTINEL_BITS).all(), "an unwritten position was modified"
    return valid, beyond


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


@pytest.mark.parametrize("next_n", [1, 2, 4])
def test_scales_over_62_binades_exact(next_n):
    """Group scales 2^-31 .. 2^31 on both operands: the spreads add up to at
    most 124 binades, so every block term is exact and the status word stays
    clean."""
    p = W.mxfp4_problem(f"mx_w62_n{next_n}", [700, 129, 64, 1500], next_n, seed=70 + next_n,
                        lo_exp=-31, hi_exp=31)
    out, status = run(p, torch.float32)
    check(p, out)
    assert status == 0


@pytest.mark.parametrize("next_n,dtype", [(1, torch.float32), (3, torch.bfloat16)])
def test_scales_over_80_binades(next_n, dtype):
    """Group scales 2^-40 .. 2^40 on both operands, as the oracle's own pin."""
    p = W.mxfp4_problem(f"mx_w80_n{next_n}", [640, 200, 77], next_n, seed=75 + next_n,
                        lo_exp=-40, hi_exp=40)
    out, _ = run(p, dtype)
    check(p, out)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_shape_full_e8m0_range(dtype):
    """The decode shape with every finite E8M0 scale (2^-127 .. 2^127) drawn
    independently for each group of each query row and key: most logits lie
    beyond fp32 and must be the infinity of their sign; the rest are
    compared as usual."""
    p = W.mxfp4_decode(seed=80, batch=6, q_exp=(-127, 127), k_exp=(-127, 127))
    out, _ = run(p, dtype)
    valid, beyond = check(p, out)
    assert (valid & ~beyond).any() and (valid & beyond).any()


def test_wide_queries_narrow_keys():
    """Query rows over 2^-100 .. 2^20 (frames far apart across heads), keys
    narrow: logits in range, compared everywhere."""
    p = W.mxfp4_problem("mx_qwide", [500, 1100], 2, seed=82, q_exp=(-100, 20), k_exp=(-4, 4))
    out, _ = run(p, torch.float32)
    valid, beyond = check(p, out)
    assert not (valid & beyond).any()


def test_wide_keys_narrow_queries():
    """Keys over every finite E8M0 value, queries narrow."""
    p = W.mxfp4_problem("mx_kwide", [500, 1100], 1, seed=83, q_exp=(-4, 4), k_exp=(-127, 127))
    out, _ = run(p, torch.float32)
    check(p, out)


def test_keys_with_one_far_group():
    """Narrow scales except for a few keys with a group 30 binades below its
    row's frame, in one call: their relative scales reach far below the
    others' and stay exact."""
    p = W.mxfp4_problem("mx_mixed", [1024, 700], 1, seed=84, poison=False)
    for blk, key in ((p.block_table[0, 3], 5), (p.block_table[0, 9], 63), (p.block_table[1, 2], 0)):
        p.kv[blk, W.MXFP4_BLOCK_CODE_BYTES + 4 * key + 1] = 127 - 30
    out, status = run(p, torch.float32)
    check(p, out)
    assert status == 0


def test_nan_scale_rectifies_to_zero():
    """An E8M0 NaN scale makes its group NaN; every head's dot product with
    that key is NaN and rectifies to 0, so the logit is 0 (the oracle's
    reading of relu on NaN)."""
    p = W.mxfp4_problem("mx_nan", [128], 1, seed=85, poison=False)
    p.kv[p.block_table[0, 1], W.MXFP4_BLOCK_CODE_BYTES + 4 * 7 + 2] = W.E8M0_NAN   # key 71
    out, _ = run(p, torch.float32)
    check(p, out)
    assert float(out[0, 71]) == 0.0


def test_complementary_spreads_are_flagged():
    """Keys whose groups sit 2^+100 / 2^-100 and query rows the other way
    round: every group's product is of order one, but each operand's small
    groups lie 200 binades below its frame.  The status word says that such
    products may have been dropped, and nothing non-finite is written."""
    p = W.mxfp4_problem("mx_compl", [64], 1, seed=86, poison=False)
    sc = W.MXFP4_BLOCK_CODE_BYTES
    for key in range(64):
        p.kv[p.block_table[0, 0], sc + 4 * key: sc + 4 * key + 4] = [227, 27, 127, 127]
    p.q_sf[0, :, :] = [27, 227, 127, 127]
    out, status = run(p, torch.float32)
    assert status & STATUS_FP4_INEXACT
    assert torch.isfinite(out[0, :64]).all()
