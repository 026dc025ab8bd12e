"""The C ABI library builds, loads and exports every entry point that
include/pml.h declares; host-side helpers and argument checks behave as
documented.  No GPU: only calls that return before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from sparse_attention_indexer_logits_gb300 import _build
    _build.build()
    import sparse_attention_indexer_logits_gb300 as pml
    return pml.lib()


def _declared():
    names = set()
    for fname in os.listdir(os.path.join(ROOT, "include")):
        if fname.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fname)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(pml_\w+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert {"pml_schedule", "pml_fp8_paged_mqa_logits", "pml_indexer_scores_bf16"} <= names
    for n in sorted(names):
        assert hasattr(L, n), f"libpml.so does not export {n}"


def test_host_helpers(L):
    assert L.pml_version() >= 100
    assert L.pml_min_block_table_width(1) == 1
    assert L.pml_min_block_table_width(64) == 1
    assert L.pml_min_block_table_width(65) == 2
    assert L.pml_min_block_table_width(0) == 0
    assert L.pml_padded_seq_len(100) == 128
    assert L.pml_padded_seq_len(131072) == 131072
    assert L.pml_schedule_meta_elems(152) == 306
    for code in range(5):
        assert L.pml_error_string(code)


P = 0x10000  # a 16-byte aligned stand-in pointer value; never dereferenced


def _fp8(L, **over):
    args = dict(q=P, kv=P, nb=10, w=P, sl=P, bt=P, bt_stride=4, meta=None, num_ctas=0, out=P,
                out_stride=256, mc=256, batch=2, n=1, H=64)
    args.update(over)
    return L.pml_fp8_paged_mqa_logits(
        args["q"], args["kv"], args["nb"], args["w"], args["sl"], args["bt"], args["bt_stride"],
        args["meta"], args["num_ctas"], args["out"], args["out_stride"], args["mc"],
        args["batch"], args["n"], args["H"], None)


def test_fp8_argument_checks(L):
    assert _fp8(L, batch=0) == 0                      # nothing to do, no launch
    assert _fp8(L, q=None) == 1
    assert _fp8(L, out=None) == 1
    assert _fp8(L, n=0) == 2 and _fp8(L, n=5) == 2
    assert _fp8(L, H=48) == 2 and _fp8(L, H=128) == 2
    assert _fp8(L, nb=0) == 1
    assert _fp8(L, mc=0) == 1
    assert _fp8(L, out_stride=100) == 1               # row shorter than max_context
    assert _fp8(L, bt_stride=3) == 1                  # block table does not cover max_context
    assert _fp8(L, meta=P) == 1                       # a schedule needs its grid size
    assert _fp8(L, q=P + 8) == 3
    assert _fp8(L, kv=P + 4) == 3
    assert _fp8(L, w=P + 4) == 3
    assert _fp8(L, out=P + 2) == 3


def _fp8_ex(L, dtype, **over):
    args = dict(q=P, kv=P, nb=10, w=P, sl=P, bt=P, bt_stride=4, meta=None, num_ctas=0, out=P,
                out_stride=256, mc=256, batch=2, n=1, H=64)
    args.update(over)
    return L.pml_fp8_paged_mqa_logits_ex(
        args["q"], args["kv"], args["nb"], args["w"], args["sl"], args["bt"], args["bt_stride"],
        args["meta"], args["num_ctas"], args["out"], args["out_stride"], dtype, args["mc"],
        args["batch"], args["n"], args["H"], None)


def test_fp8_output_dtype_checks(L):
    assert _fp8_ex(L, 2) == 2 and _fp8_ex(L, -1) == 2  # only fp32 (0) and bf16 (1)
    assert _fp8_ex(L, 1, batch=0) == 0
    assert _fp8_ex(L, 1, out=P + 2, n=0) == 2          # shape checks still come first
    assert _fp8_ex(L, 1, out=P + 1) == 3               # bf16 out: 2-byte alignment
    assert _fp8_ex(L, 0, out=P + 2) == 3               # fp32 out: 4-byte alignment
    assert _fp8_ex(L, 1, out_stride=100) == 1


def _bf16(L, **over):
    a = dict(q=P, rows=8, kc=P, stride=16384, pages=4, bt=P, bt_stride=4, nreq=2, cl=P, req=P,
             groups=2, sc=P, sc_stride=256, mc=256)
    a.update(over)
    return L.pml_indexer_scores_bf16(a["q"], a["rows"], a["kc"], a["stride"], a["pages"], a["bt"],
                                     a["bt_stride"], a["nreq"], a["cl"], a["req"], a["groups"],
                                     a["sc"], a["sc_stride"], a["mc"], None)


def test_bf16_argument_checks(L):
    assert _bf16(L, rows=0, groups=0) == 0
    assert _bf16(L, rows=9) == 1                      # rows not a multiple of groups
    assert _bf16(L, rows=18) == 2                     # group of 9 rows
    assert _bf16(L, stride=16384 + 8) == 3            # page stride not a multiple of 16
    assert _bf16(L, stride=8192) == 1                 # pages would overlap
    assert _bf16(L, q=None) == 1
    assert _bf16(L, sc_stride=100) == 1
    assert _bf16(L, bt_stride=2) == 1
    assert _bf16(L, kc=P + 8) == 3


def _nvfp4(L, **over):
    a = dict(q=P, qs=P, rows=8, kc=P, stride=4096, ks=P, sstride=512, pages=4, bt=P,
             bt_stride=4, nreq=2, cl=P, req=P, groups=2, sc=P, sc_stride=256, mc=256)
    a.update(over)
    return L.pml_indexer_scores_nvfp4(a["q"], a["qs"], a["rows"], a["kc"], a["stride"], a["ks"],
                                      a["sstride"], a["pages"], a["bt"], a["bt_stride"], a["nreq"],
                                      a["cl"], a["req"], a["groups"], a["sc"], a["sc_stride"],
                                      a["mc"], None)


def test_nvfp4_argument_checks(L):
    assert _nvfp4(L, rows=0, groups=0) == 0
    assert _nvfp4(L, rows=9) == 1                     # rows not a multiple of groups
    assert _nvfp4(L, rows=18) == 2                    # group of 9 rows
    assert _nvfp4(L, qs=None) == 1 and _nvfp4(L, ks=None) == 1
    assert _nvfp4(L, stride=4096 + 8) == 3            # key pages a multiple of 16 apart
    assert _nvfp4(L, sstride=512 + 4) == 3            # scale pages a multiple of 8 apart
    assert _nvfp4(L, stride=2048) == 1                # key pages would overlap
    assert _nvfp4(L, sstride=256) == 1                # scale pages would overlap
    assert _nvfp4(L, q=P + 8) == 3 and _nvfp4(L, qs=P + 4) == 3
    assert _nvfp4(L, kc=P + 8) == 3 and _nvfp4(L, ks=P + 4) == 3
    assert _nvfp4(L, sc_stride=100) == 1 and _nvfp4(L, bt_stride=2) == 1


def _fp4(L, **over):
    a = dict(q=P, qsf=P, kv=P, nb=4, w=P, sl=P, bt=P, bt_stride=4, meta=None, ctas=0, out=P,
             out_stride=256, dt=1, mc=256, batch=2, n=1)
    a.update(over)
    return L.pml_fp4_paged_mqa_logits(a["q"], a["qsf"], a["kv"], a["nb"], a["w"], a["sl"], a["bt"],
                                      a["bt_stride"], a["meta"], a["ctas"], a["out"],
                                      a["out_stride"], a["dt"], a["mc"], a["batch"], a["n"], None)


def test_wait_test_argument_checks(L):
    def call(drop, limit):
        return L.pml_fp8_paged_mqa_logits_wait_test(P, P, 4, P, P, P, 4, P, 256, 256, 2, 1, 64,
                                                    drop, limit, None)
    assert call(-1, 1000) == 1                        # a stage to leave out is required
    assert call(0, 0) == 1 and call(0, 1000001) == 1  # limit 1 us .. 1 s


def test_fp4_argument_checks(L):
    assert _fp4(L, batch=0) == 0
    assert _fp4(L, dt=7) == 2                         # output type
    assert _fp4(L, n=0) == 2 and _fp4(L, n=5) == 2
    assert _fp4(L, batch=70000) == 2
    assert _fp4(L, qsf=None) == 1 and _fp4(L, kv=None) == 1 and _fp4(L, w=None) == 1
    assert _fp4(L, out_stride=100) == 1 and _fp4(L, bt_stride=2) == 1
    assert _fp4(L, q=P + 8) == 3 and _fp4(L, kv=P + 8) == 3
    # query scales and weights arrive by bulk copies: 16-byte aligned
    assert _fp4(L, qsf=P + 4) == 3 and _fp4(L, w=P + 4) == 3
    assert _fp4(L, out=P + 1) == 3                    # bf16 out on a 2-byte boundary
    assert _fp4(L, dt=0, out=P + 2) == 3              # fp32 out on a 4-byte boundary
    assert _fp4(L, meta=P, ctas=0) == 1               # a schedule without its CTA count
    assert _fp4(L, meta=P + 2, ctas=4) == 3


def test_topk_argument_checks(L):
    def topk(**o):
        a = dict(x=P, xs=256, sl=P, batch=2, n=1, mc=256, k=16, idx=P, ids=16, val=None, vs=0)
        a.update(o)
        return L.pml_topk_logits(a["x"], a["xs"], a["sl"], a["batch"], a["n"], a["mc"], a["k"],
                                 a["idx"], a["ids"], a["val"], a["vs"], None)
    assert topk(batch=0) == 0
    assert topk(k=0) == 2 and topk(k=4097) == 2
    assert topk(x=None) == 1 and topk(idx=None) == 1
    assert topk(xs=100) == 1 and topk(ids=8) == 1
    assert topk(val=P, vs=8) == 1
    assert topk(x=P + 2) == 3 and topk(idx=P + 1) == 3


def test_schedule_argument_checks(L):
    assert L.pml_schedule(P, 4, 1, 0, P, None) == 1
    assert L.pml_schedule(P, 4, 1, 8, None, None) == 1
    assert L.pml_schedule(P, 4, 0, 8, P, None) == 2


def test_product_path_does_not_reach_the_oracle():
    """The library package imports nothing from oracle/."""
    pkg = os.path.join(ROOT, "sparse_attention_indexer_logits_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "oracle.c" not in text, f
