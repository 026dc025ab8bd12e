"""Plain fp64 CPU oracle for paged MQA logits and single-head indexer scores.

TEST INFRASTRUCTURE ONLY.  This package is the checker the GPU path is
compared against: only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import it.  It shares no code with the CUDA
library (``sparse_attention_indexer_logits_gb300``) and imports nothing from
it.

The arithmetic lives in ``oracle.c`` (plain loops, fp64, exact e4m3/bf16
decode, optional pthreads over requests); this module compiles it with gcc and
wraps it with ctypes.  ``brute.py`` holds a second, exact (``fractions``)
implementation for tiny inputs that pins the C code.

Sources: FlashInfer documentation, "flashinfer.attn_scores" (math block,
bullets, note, "Scheduling and Setup") and "flashinfer.sdsa.indexer_scores"
(body and parameter list).  Every function below states which passage it
follows.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np

HEAD_DIM = 128
BLOCK_KEYS = 64
BLOCK_KEY_BYTES = BLOCK_KEYS * HEAD_DIM
BLOCK_BYTES = BLOCK_KEY_BYTES + BLOCK_KEYS * 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, -O2)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_decode.restype = ctypes.c_double
    lib.orc_bf16_decode.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_decode.restype = ctypes.c_double
    lib.orc_schedule.argtypes = [P, ctypes.c_int, ctypes.c_int, P]
    lib.orc_schedule.restype = i64
    lib.orc_fp8_paged_mqa_logits.argtypes = [
        P, P, i64, P, P, P, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        P, P, i64, ctypes.c_int, ctypes.c_int,
    ]
    lib.orc_fp8_paged_mqa_logits.restype = ctypes.c_int
    lib.orc_indexer_scores_bf16.argtypes = [
        P, ctypes.c_int, P, i64, P, i64, P, P, ctypes.c_int, P, P, i64,
        ctypes.c_int, ctypes.c_int,
    ]
    lib.orc_indexer_scores_bf16.restype = ctypes.c_int
    lib.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e2m1_decode.restype = ctypes.c_double
    lib.orc_indexer_scores_nvfp4.argtypes = [
        P, P, ctypes.c_int, P, i64, P, i64, P, i64, P, P, ctypes.c_int, P, P, i64,
        ctypes.c_int, ctypes.c_int,
    ]
    lib.orc_indexer_scores_nvfp4.restype = ctypes.c_int
    lib.orc_e8m0_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e8m0_decode.restype = ctypes.c_double
    lib.orc_fp4_paged_mqa_logits.argtypes = [
        P, P, P, i64, P, P, P, i64, ctypes.c_int, ctypes.c_int, P, P, i64, ctypes.c_int,
        ctypes.c_int,
    ]
    lib.orc_fp4_paged_mqa_logits.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Run the oracle functions against another build of ``oracle.c`` (the
    pin tests use this to show that a planted mistake fails a pin)."""
    global _lib
    saved = _load()
    _lib = _bind(path)
    try:
        yield
    finally:
        _lib = saved


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def default_threads() -> int:
    return os.cpu_count() or 1


def e4m3_decode(code: int) -> float:
    """Value of an E4M3FN byte (OCP 8-bit float: bias 7, 0x7F/0xFF NaN)."""
    return _load().orc_e4m3_decode(int(code) & 0xFF)


def e2m1_decode(code: int) -> float:
    """Value of a 4-bit E2M1 code (OCP FP4: bias 1, one mantissa bit)."""
    return _load().orc_e2m1_decode(int(code) & 0xF)


def e8m0_decode(code: int) -> float:
    """Value of an E8M0 scale byte (OCP MX shared scale: 2^(code - 127),
    0xFF NaN)."""
    return float(_load().orc_e8m0_decode(code))


def bf16_decode(bits: int) -> float:
    """Value of a bfloat16 bit pattern (the upper half of a binary32)."""
    return _load().orc_bf16_decode(int(bits) & 0xFFFF)


def schedule(seq_lens, num_ctas: int):
    """Persistent CTA work assignment ("flashinfer.attn_scores", "Scheduling
    and Setup": a per-call CTA work assignment, a function of ``seq_lens``).

    Returns ``(meta, total)``: ``meta`` int32 ``[num_ctas + 1, 2]`` with the
    (request, block) where each CTA's contiguous range of 64-key blocks starts
    (``(batch, 0)`` for a start at the end), and ``total`` = number of blocks.
    """
    sl = _c(seq_lens, np.int32)
    meta = np.zeros((num_ctas + 1, 2), dtype=np.int32)
    total = _load().orc_schedule(_ptr(sl), int(sl.shape[0]), int(num_ctas), _ptr(meta))
    return meta, int(total)


def fp8_paged_mqa_logits(q, kv_fused, weights, seq_lens, block_table, next_n: int,
                         max_context: int | None = None, out=None, with_mag: bool = True,
                         nthreads: int | None = None):
    """fp64 logits ``out[b*next_n+t, p] = s_p * sum_h w[t,h] * relu(q[t,h].k_p)``
    ("flashinfer.attn_scores": math block, first and second bullets, note).

    ``q`` uint8 e4m3 ``[batch*next_n, H, 128]``; ``kv_fused`` uint8
    ``[num_blocks, 8448]`` (64x128 e4m3 keys, then 64 fp32 scales);
    ``weights`` fp32 ``[batch*next_n, H]``; ``seq_lens`` int32 ``[batch]``;
    ``block_table`` int32 ``[batch, width]``.  Positions ``p < seq_lens[b]``
    are written; every other entry of ``out`` (fp64, NaN-filled if not given)
    is left as it was.  Returns ``(out, mag)``; ``mag`` holds
    ``|s_p| * sum_h |w| * |q.k|`` at the written places (else NaN).
    """
    q = _c(q, np.uint8)
    kv = _c(kv_fused, np.uint8).reshape(-1, BLOCK_BYTES)
    w = _c(weights, np.float32)
    sl = _c(seq_lens, np.int32)
    bt = _c(block_table, np.int32)
    batch = sl.shape[0]
    H = q.shape[1]
    assert q.shape == (batch * next_n, H, HEAD_DIM), q.shape
    assert w.shape == (batch * next_n, H)
    if bt.ndim == 1:
        bt = bt.reshape(batch, -1)
    if max_context is None:
        max_context = int(max(1, sl.max(initial=0)))
    if out is None:
        out = np.full((batch * next_n, max_context), np.nan, dtype=np.float64)
    assert out.dtype == np.float64 and out.flags.c_contiguous
    mag = np.full(out.shape, np.nan, dtype=np.float64) if with_mag else None
    rc = _load().orc_fp8_paged_mqa_logits(
        _ptr(q), _ptr(kv), kv.shape[0], _ptr(w), _ptr(sl), _ptr(bt), bt.shape[1], batch,
        next_n, H, _ptr(out), _ptr(mag) if mag is not None else None, out.shape[1],
        max_context, nthreads or default_threads(),
    )
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out, mag


MXFP4_BLOCK_BYTES = BLOCK_KEYS * (HEAD_DIM // 2 + HEAD_DIM // 32)   # 4352


def fp4_paged_mqa_logits(q, q_sf, kv, weights, seq_lens, block_table, next_n: int,
                         max_context: int | None = None, out=None, with_mag: bool = True,
                         nthreads: int | None = None):
    """fp64 MXFP4 logits ``out[b*next_n+t, p] = sum_h w[t,h] * relu(q[t,h].k_p)``
    over dequantised values, no per-position factor ("flashinfer.attn_scores":
    math block, first and second bullets, the paragraph after them).

    ``q`` uint8 ``[batch*next_n, 64, 64]`` (E2M1 two to a byte, low nibble
    first), ``q_sf`` uint8 E8M0 ``[batch*next_n, 64, 4]`` (one per 32
    values), ``kv`` uint8 ``[num_blocks, 4352]`` (64 keys x 64 code bytes,
    then 64 x 4 scale bytes), ``weights`` fp32 ``[batch*next_n, 64]``.
    Written places and ``mag`` as for ``fp8_paged_mqa_logits`` (``mag`` =
    ``sum_h |w| * |q.k|``)."""
    q = _c(q, np.uint8)
    q_sf = _c(q_sf, np.uint8)
    kv = _c(kv, np.uint8).reshape(-1, MXFP4_BLOCK_BYTES)
    w = _c(weights, np.float32)
    sl = _c(seq_lens, np.int32)
    bt = _c(block_table, np.int32)
    batch = sl.shape[0]
    assert q.shape == (batch * next_n, 64, HEAD_DIM // 2), q.shape
    assert q_sf.shape == (batch * next_n, 64, HEAD_DIM // 32), q_sf.shape
    assert w.shape == (batch * next_n, 64)
    if bt.ndim == 1:
        bt = bt.reshape(batch, -1)
    if max_context is None:
        max_context = int(max(1, sl.max(initial=0)))
    if out is None:
        out = np.full((batch * next_n, max_context), np.nan, dtype=np.float64)
    assert out.dtype == np.float64 and out.flags.c_contiguous
    mag = np.full(out.shape, np.nan, dtype=np.float64) if with_mag else None
    rc = _load().orc_fp4_paged_mqa_logits(
        _ptr(q), _ptr(q_sf), _ptr(kv), kv.shape[0], _ptr(w), _ptr(sl), _ptr(bt), bt.shape[1],
        batch, next_n, _ptr(out), _ptr(mag) if mag is not None else None, out.shape[1],
        max_context, nthreads or default_threads(),
    )
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out, mag


def indexer_scores_bf16(query, key_cache, page_stride_bytes: int, block_table, context_lengths,
                        requests, max_context: int, out=None, with_mag: bool = True,
                        nthreads: int | None = None):
    """fp64 single-head scores ``scores[r, k] = query[r] . key_k`` for ``k``
    below the group's length ("flashinfer.sdsa.indexer_scores": body, and the
    ``block_table``, ``context_lengths``, ``requests`` and ``scores``
    parameters).  Groups are uniform: group ``g`` is rows
    ``[g*G, (g+1)*G)``, ``G = rows / groups``.

    ``query`` uint16 (bf16 bits) ``[rows, 128]``; ``key_cache`` raw bytes, page
    ``P`` at byte ``P*page_stride_bytes`` holding 64x128 bf16.  Entries past a
    group's length are left as they were.  Returns ``(scores, mag)``, ``mag``
    = ``sum_d |q_d k_d|``.
    """
    qy = _c(query, np.uint16)
    kc = _c(np.asarray(key_cache).view(np.uint8), np.uint8).reshape(-1)
    bt = _c(block_table, np.int32)
    cl = _c(context_lengths, np.int32)
    rq = _c(requests, np.int32)
    rows = qy.shape[0]
    if out is None:
        out = np.full((rows, max_context), np.nan, dtype=np.float64)
    assert out.dtype == np.float64 and out.flags.c_contiguous
    mag = np.full(out.shape, np.nan, dtype=np.float64) if with_mag else None
    rc = _load().orc_indexer_scores_bf16(
        _ptr(qy), rows, _ptr(kc), int(page_stride_bytes), _ptr(bt), bt.shape[1], _ptr(cl),
        _ptr(rq), cl.shape[0], _ptr(out), _ptr(mag) if mag is not None else None,
        out.shape[1], max_context, nthreads or default_threads(),
    )
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out, mag


def indexer_scores_nvfp4(query, query_scales, key_cache, page_stride_bytes: int, key_scales,
                         scale_page_stride_bytes: int, block_table, context_lengths, requests,
                         max_context: int, out=None, with_mag: bool = True,
                         nthreads: int | None = None):
    """fp64 single-head scores over NVFP4 queries and keys
    ("flashinfer.sdsa.indexer_scores": the NVFP4 forms of ``query``,
    ``key_cache``, ``query_scales`` and ``key_scales``).  Element ``d`` of a
    row is the E2M1 code in byte ``d//2`` (low nibble for even ``d``) times the
    row's E4M3 scale ``d//16``; a score is the plain dot product of the
    dequantised query row and key.  Groups are uniform as in
    ``indexer_scores_bf16``.

    ``query`` uint8 ``[rows, 64]``, ``query_scales`` uint8 ``[rows, 8]``;
    ``key_cache`` / ``key_scales`` raw bytes, page ``P`` at byte
    ``P*page_stride_bytes`` (64x64 packed bytes) and
    ``P*scale_page_stride_bytes`` (64x8 scale bytes).  Returns
    ``(scores, mag)``, ``mag`` = ``sum_d |q_d k_d|``; entries past a group's
    length are left as they were.
    """
    qy = _c(query, np.uint8)
    qs = _c(query_scales, np.uint8)
    kc = _c(np.asarray(key_cache).view(np.uint8), np.uint8).reshape(-1)
    ks = _c(np.asarray(key_scales).view(np.uint8), np.uint8).reshape(-1)
    bt = _c(block_table, np.int32)
    cl = _c(context_lengths, np.int32)
    rq = _c(requests, np.int32)
    rows = qy.shape[0]
    assert qy.shape[1] == 64 and qs.shape == (rows, 8)
    if out is None:
        out = np.full((rows, max_context), np.nan, dtype=np.float64)
    assert out.dtype == np.float64 and out.flags.c_contiguous
    mag = np.full(out.shape, np.nan, dtype=np.float64) if with_mag else None
    rc = _load().orc_indexer_scores_nvfp4(
        _ptr(qy), _ptr(qs), rows, _ptr(kc), int(page_stride_bytes), _ptr(ks),
        int(scale_page_stride_bytes), _ptr(bt), bt.shape[1], _ptr(cl), _ptr(rq), cl.shape[0],
        _ptr(out), _ptr(mag) if mag is not None else None, out.shape[1], max_context,
        nthreads or default_threads(),
    )
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out, mag


def fp8_valid_mask(seq_lens, next_n: int, max_context: int) -> np.ndarray:
    """Positions where row ``b*next_n+t`` is meaningful: ``p <= seq_lens[b] -
    next_n + t`` ("flashinfer.attn_scores", note)."""
    sl = np.asarray(seq_lens, dtype=np.int64)
    t = np.arange(next_n)
    lim = (sl[:, None] - next_n + t[None, :]).reshape(-1)          # inclusive limit per row
    p = np.arange(max_context)
    return p[None, :] <= lim[:, None]


def fp8_written_mask(seq_lens, next_n: int, max_context: int) -> np.ndarray:
    """Positions the fp8 path writes: ``p < seq_lens[b]`` (nothing for empty
    requests)."""
    sl = np.repeat(np.asarray(seq_lens, dtype=np.int64), next_n)
    return np.arange(max_context)[None, :] < sl[:, None]


def _order_key(values: np.ndarray) -> np.ndarray:
    """Unsigned keys whose order is the order of the float32 values they come
    from (negative values have their bits inverted, the rest their sign bit
    set): -NaN < -inf < ... < -0 < +0 < ... < +inf < +NaN."""
    bits = np.ascontiguousarray(values, dtype=np.float32).view(np.uint32)
    neg = (bits >> np.uint32(31)).astype(bool)
    return np.where(neg, ~bits, bits | np.uint32(0x80000000)).astype(np.uint32)


def topk_logits(logits, seq_lens, next_n: int, max_context: int, k: int):
    """The indexer's selection over paged MQA logits ("flashinfer.attn_scores",
    intro: the logits are what a sparse-attention indexer uses to choose which
    KV tokens to keep; the note: row b*next_n+t is meaningful for positions
    0 .. seq_lens[b]-next_n+t).  For each row, the k positions with the
    largest logits among p <= min(seq_lens[b]-next_n+t, max_context-1), in
    descending order of value (float32 bit order, see ``_order_key``), equal
    values in ascending position; fewer candidates than k leave the remaining
    slots as index -1 and value -inf.  Rows of empty requests have no
    candidates.  Returns ``(indices int32 [rows, k], values float32 [rows, k])``.
    """
    x = np.asarray(logits, dtype=np.float32)
    sl = np.asarray(seq_lens, dtype=np.int64)
    rows = sl.shape[0] * next_n
    idx = np.full((rows, k), -1, dtype=np.int32)
    val = np.full((rows, k), -np.inf, dtype=np.float32)
    for r in range(rows):
        b, t = divmod(r, next_n)
        lim = min(int(sl[b]) - next_n + t + 1, max_context) if sl[b] > 0 else 0
        if lim <= 0:
            continue
        keys = _order_key(x[r, :lim]).astype(np.int64)
        pos = np.arange(lim)
        order = np.lexsort((pos, -keys))[:k]         # key descending, then position
        idx[r, :order.shape[0]] = order
        val[r, :order.shape[0]] = x[r, order]
    return idx, val
