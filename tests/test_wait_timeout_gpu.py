"""The fp8 kernel's bounded waits run out, on the GPU, without a fault or a
hang: every in-kernel wait gives up after a limit, records
PML_STATUS_WAIT_TIMEOUT, raises the CTA's abort flag, lets the copies and
MMAs already issued complete and returns.  The test entry point
pml_fp8_paged_mqa_logits_wait_test makes each CTA's producer leave one of
its stages unpublished with a 2 ms limit: the call must return promptly with
the status bit set, and the next regular call on the same device must match
the oracle.  Both register layouts of the kernel are covered (next_n 1, and
next_n 4 at 64 heads, whose warpgroups re-split their registers and inline
their waits)."""
import time

import numpy as np
import pytest
import torch

import sparse_attention_indexer_logits_gb300 as pml
from sparse_attention_indexer_logits_gb300 import workloads as W

from tests import helpers as Hh

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("next_n,heads,lens,drop", [
    (1, 64, [8192, 8192, 6000, 9000], 0),      # every CTA with work stops at its first stage
    (1, 64, [32768] * 8, 1),                   # ... at its second
    (4, 64, [4096, 3000, 5000], 0),
    (2, 16, [2048, 70, 4000], 0),
])
def test_dropped_stage_times_out_then_device_recovers(next_n, heads, lens, drop):
    p = W.fp8_problem(f"timeout_n{next_n}", lens, next_n, heads, seed=90 + next_n, poison=True)
    d = Hh.Fp8Device(p)
    out = Hh.dev_tensor(W.sentinel_f32((p.batch * next_n, p.max_context)))
    pml.pml_device_status(clear=True)
    t0 = time.perf_counter()
    pml.pml_fp8_paged_mqa_logits_wait_test(d.q, d.kv, d.w, d.seq_lens, d.bt, out, p.max_context,
                                           next_n, drop_stage=drop, wait_limit_us=2000)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    status = pml.pml_device_status(clear=True)
    assert status & pml.STATUS_WAIT_TIMEOUT, f"status {status:#x}"
    assert not status & pml.STATUS_BAD_BLOCK
    assert elapsed < 0.5, elapsed                # a few 2 ms limits, not a 1 s one
    # the same device, the same inputs, the regular call: parity with the oracle
    got = d.run()
    torch.cuda.synchronize()
    Hh.check_fp8(p, got.cpu().numpy())
    assert pml.pml_device_status(clear=True) == 0


def test_nothing_dropped_past_the_last_stage():
    """A stage number no CTA reaches changes nothing: the result is complete
    and the status word stays clean."""
    p = W.fp8_problem("timeout_none", [300, 64, 129], 1, 32, seed=95, poison=True)
    d = Hh.Fp8Device(p)
    out = Hh.dev_tensor(W.sentinel_f32((p.batch, p.max_context)))
    pml.pml_device_status(clear=True)
    pml.pml_fp8_paged_mqa_logits_wait_test(d.q, d.kv, d.w, d.seq_lens, d.bt, out, p.max_context, 1,
                                           drop_stage=10000, wait_limit_us=2000)
    torch.cuda.synchronize()
    assert pml.pml_device_status(clear=True) == 0
    Hh.check_fp8(p, out.cpu().numpy())
