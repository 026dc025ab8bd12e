"""Paged MQA logits for the sparse-attention indexer, GB300-native (sm_103a).

Thin Python binding over the C ABI of ``libpml.so`` (``include/pml.h``):
argument marshalling only -- every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and the current
stream.  There is no CPU fallback: if the library is missing or cannot be
loaded, every call raises.

Entry points (same names as the C ABI):

* ``pml_schedule`` -- the persistent per-CTA work assignment
  ("flashinfer.attn_scores", "Scheduling and Setup").
* ``pml_fp8_paged_mqa_logits`` -- ``out[b*n+t, p] = s_p * sum_h w * relu(q.k_p)``
  over an fp8 paged ``kv_fused`` cache ("flashinfer.attn_scores").
* ``pml_fp8_paged_mqa_logits_ex`` -- the same with the ``output_dtype``
  option (fp32 or bf16 logits).
* ``pml_indexer_scores_bf16`` -- the single-head bf16 case
  ("flashinfer.sdsa.indexer_scores").
* ``pml_indexer_scores_nvfp4`` -- the same over NVFP4 queries and keys.
* ``pml_topk_logits`` -- the indexer's selection: each row's k largest
  logits among its meaningful positions.
* ``pml_fp4_paged_mqa_logits`` -- the MXFP4 variant of the logits (64
  heads, E2M1 codes with E8M0 scales per 32 values, bf16 out by default).

``fp8_paged_mqa_logits`` / ``indexer_scores`` wrap them with the pages'
keyword style (``out=``, ``schedule_meta=``, ``scores=``).
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "PmlError", "lib", "library_path", "pml_schedule", "pml_fp8_paged_mqa_logits",
    "pml_fp8_paged_mqa_logits_ex",
    "pml_indexer_scores_bf16", "pml_indexer_scores_nvfp4", "pml_topk_logits",
    "pml_fp4_paged_mqa_logits",
    "pml_fp8_paged_mqa_logits_noalloc", "pml_fp8_paged_mqa_logits_wait_test",
    "pml_device_status",
    "pml_default_num_ctas", "pml_min_block_table_width", "pml_padded_seq_len", "pml_schedule_meta_elems",
    "fp8_paged_mqa_logits", "indexer_scores", "compute_paged_mqa_logits_schedule",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libpml.so")
_lib = None

STATUS_WAIT_TIMEOUT = 1
STATUS_BAD_BLOCK = 2
STATUS_BAD_REQUEST = 4


class PmlError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = lib().pml_error_string(code).decode()
        if code == 4:
            msg += f" (cudaError {lib().pml_last_cuda_error()})"
        super().__init__(f"{what}: {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded library (built by ``__graft_entry__.build()`` or
    ``sparse_attention_indexer_logits_gb300._build.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(
                f"libpml.so not found at {library_path}: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(library_path)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.pml_version.restype = i32
        L.pml_error_string.argtypes = [i32]
        L.pml_error_string.restype = ctypes.c_char_p
        L.pml_last_cuda_error.restype = i32
        L.pml_default_num_ctas.argtypes = [i32]
        L.pml_default_num_ctas.restype = i32
        for name in ("pml_schedule_meta_elems", "pml_min_block_table_width", "pml_padded_seq_len"):
            getattr(L, name).argtypes = [i32]
            getattr(L, name).restype = i32
        L.pml_schedule.argtypes = [P, i32, i32, i32, P, P]
        L.pml_schedule.restype = i32
        L.pml_fp8_paged_mqa_logits.argtypes = [P, P, i64, P, P, P, i64, P, i32, P, i64, i32, i32,
                                               i32, i32, P]
        L.pml_fp8_paged_mqa_logits.restype = i32
        L.pml_fp8_paged_mqa_logits_ex.argtypes = [P, P, i64, P, P, P, i64, P, i32, P, i64, i32, i32,
                                                  i32, i32, i32, P]
        L.pml_fp8_paged_mqa_logits_ex.restype = i32
        L.pml_indexer_scores_bf16.argtypes = [P, i32, P, i64, i64, P, i64, i32, P, P, i32, P, i64,
                                              i32, P]
        L.pml_indexer_scores_bf16.restype = i32
        L.pml_indexer_scores_nvfp4.argtypes = [P, P, i32, P, i64, P, i64, i64, P, i64, i32, P, P,
                                               i32, P, i64, i32, P]
        L.pml_indexer_scores_nvfp4.restype = i32
        L.pml_topk_logits.argtypes = [P, i64, P, i32, i32, i32, i32, P, i64, P, i64, P]
        L.pml_topk_logits.restype = i32
        L.pml_fp4_paged_mqa_logits.argtypes = [P, P, P, i64, P, P, P, i64, P, i32, P, i64, i32,
                                               i32, i32, i32, P]
        L.pml_fp4_paged_mqa_logits.restype = i32
        L.pml_fp8_paged_mqa_logits_wait_test.argtypes = [P, P, i64, P, P, P, i64, P, i64, i32, i32,
                                                         i32, i32, i32, i64, P]
        L.pml_fp8_paged_mqa_logits_wait_test.restype = i32
        L.pml_fp8_paged_mqa_logits_noalloc.argtypes = [P, P, i64, P, P, P, i64, i32, P, i64, i32,
                                                       i32, i32, i32, P]
        L.pml_fp8_paged_mqa_logits_noalloc.restype = i32
        L.pml_noalloc_max_ctas.restype = i32
        L.pml_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), i32]
        L.pml_device_status.restype = i32
        _lib = L
    return _lib


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, what: str):
    if rc != 0:
        raise PmlError(rc, what)


def _cuda(t: torch.Tensor, name: str, contiguous: bool = True):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ---------------------------------------------------------------- helpers

def pml_default_num_ctas(device: int | None = None) -> int:
    d = torch.cuda.current_device() if device is None else device
    return lib().pml_default_num_ctas(d)


def pml_min_block_table_width(max_seq_len: int) -> int:
    return lib().pml_min_block_table_width(max_seq_len)


def pml_padded_seq_len(max_seq_len: int) -> int:
    return lib().pml_padded_seq_len(max_seq_len)


def pml_schedule_meta_elems(num_ctas: int) -> int:
    return lib().pml_schedule_meta_elems(num_ctas)


def pml_device_status(clear: bool = False) -> int:
    """Sticky device status bits (synchronises the device)."""
    v = ctypes.c_uint(0)
    _check(lib().pml_device_status(ctypes.byref(v), int(clear)), "pml_device_status")
    return v.value


# ---------------------------------------------------------------- C ABI calls

def pml_schedule(seq_lens: torch.Tensor, num_ctas: int, next_n: int = 1,
                 schedule_meta: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Persistent schedule for ``num_ctas`` CTAs: int32 ``[num_ctas + 1, 2]``."""
    _cuda(seq_lens, "seq_lens")
    if schedule_meta is None:
        schedule_meta = torch.empty((num_ctas + 1, 2), dtype=torch.int32, device=seq_lens.device)
    _cuda(schedule_meta, "schedule_meta")
    if schedule_meta.numel() < 2 * (num_ctas + 1) or schedule_meta.dtype != torch.int32:
        raise ValueError("schedule_meta must be int32 with (num_ctas + 1) * 2 elements")
    _check(lib().pml_schedule(_ptr(seq_lens), seq_lens.numel(), next_n, num_ctas,
                              _ptr(schedule_meta), _stream(stream)), "pml_schedule")
    return schedule_meta


def pml_fp8_paged_mqa_logits(q: torch.Tensor, kv_fused: torch.Tensor, weights: torch.Tensor,
                             seq_lens: torch.Tensor, block_table: torch.Tensor, out: torch.Tensor,
                             max_context: int, next_n: int, schedule_meta: torch.Tensor | None = None,
                             num_ctas: int = 0, stream=None) -> torch.Tensor:
    """``out[b*next_n+t, p] = s_p * sum_h weights[b*next_n+t,h] * relu(q[b*next_n+t,h].k_p)``.

    q: e4m3 (or uint8) ``[batch*next_n, H, 128]``; kv_fused: uint8
    ``[num_blocks, 8448]``; weights: fp32 ``[batch*next_n, H]``; seq_lens:
    int32 ``[batch]``; block_table: int32 ``[batch, width]`` (row stride used);
    out: fp32 ``[batch*next_n, >= max_context]`` (row stride used)."""
    for t, nm in ((q, "q"), (kv_fused, "kv_fused"), (weights, "weights"), (seq_lens, "seq_lens")):
        _cuda(t, nm)
    _cuda(block_table, "block_table", contiguous=False)
    _cuda(out, "out", contiguous=False)
    if block_table.stride(-1) != 1 or out.stride(-1) != 1:
        raise ValueError("block_table and out need unit stride in their last dimension")
    if q.dim() != 3 or q.shape[2] != 128 or q.element_size() != 1:
        raise ValueError("q must be [batch*next_n, heads, 128] with 1-byte elements")
    if weights.dtype != torch.float32 or out.dtype != torch.float32:
        raise ValueError("weights and out must be float32")
    if seq_lens.dtype != torch.int32 or block_table.dtype != torch.int32:
        raise ValueError("seq_lens and block_table must be int32")
    batch = seq_lens.numel()
    H = q.shape[1]
    if q.shape[0] != batch * next_n or tuple(weights.shape) != (batch * next_n, H):
        raise ValueError("q / weights rows must be batch*next_n")
    if kv_fused.numel() % 8448 != 0:
        raise ValueError("kv_fused must hold whole 8448-byte blocks")
    if out.shape[0] < batch * next_n or out.shape[1] < max_context:
        raise ValueError("out too small")
    _check(lib().pml_fp8_paged_mqa_logits(
        _ptr(q), _ptr(kv_fused), kv_fused.numel() // 8448, _ptr(weights), _ptr(seq_lens),
        _ptr(block_table), block_table.stride(0), _ptr(schedule_meta), num_ctas, _ptr(out),
        out.stride(0), max_context, batch, next_n, H, _stream(stream)),
        "pml_fp8_paged_mqa_logits")
    return out


_OUT_DTYPES = {torch.float32: 0, torch.bfloat16: 1}


def pml_fp8_paged_mqa_logits_ex(q: torch.Tensor, kv_fused: torch.Tensor, weights: torch.Tensor,
                                seq_lens: torch.Tensor, block_table: torch.Tensor,
                                out: torch.Tensor, max_context: int, next_n: int,
                                schedule_meta: torch.Tensor | None = None, num_ctas: int = 0,
                                stream=None) -> torch.Tensor:
    """``pml_fp8_paged_mqa_logits`` writing ``out`` in its own dtype: fp32, or
    bf16 (the fp32 logit rounded to nearest even)."""
    if out.dtype not in _OUT_DTYPES:
        raise ValueError("out must be float32 or bfloat16")
    for t, nm in ((q, "q"), (kv_fused, "kv_fused"), (weights, "weights"), (seq_lens, "seq_lens")):
        _cuda(t, nm)
    _cuda(block_table, "block_table", contiguous=False)
    _cuda(out, "out", contiguous=False)
    if block_table.stride(-1) != 1 or out.stride(-1) != 1:
        raise ValueError("block_table and out need unit stride in their last dimension")
    if q.dim() != 3 or q.shape[2] != 128 or q.element_size() != 1:
        raise ValueError("q must be [batch*next_n, heads, 128] with 1-byte elements")
    if weights.dtype != torch.float32:
        raise ValueError("weights must be float32")
    if seq_lens.dtype != torch.int32 or block_table.dtype != torch.int32:
        raise ValueError("seq_lens and block_table must be int32")
    batch = seq_lens.numel()
    H = q.shape[1]
    if q.shape[0] != batch * next_n or tuple(weights.shape) != (batch * next_n, H):
        raise ValueError("q / weights rows must be batch*next_n")
    if kv_fused.numel() % 8448 != 0:
        raise ValueError("kv_fused must hold whole 8448-byte blocks")
    if out.shape[0] < batch * next_n or out.shape[1] < max_context:
        raise ValueError("out too small")
    _check(lib().pml_fp8_paged_mqa_logits_ex(
        _ptr(q), _ptr(kv_fused), kv_fused.numel() // 8448, _ptr(weights), _ptr(seq_lens),
        _ptr(block_table), block_table.stride(0), _ptr(schedule_meta), num_ctas, _ptr(out),
        out.stride(0), _OUT_DTYPES[out.dtype], max_context, batch, next_n, H, _stream(stream)),
        "pml_fp8_paged_mqa_logits_ex")
    return out


def pml_indexer_scores_bf16(query: torch.Tensor, key_cache: torch.Tensor, page_stride_bytes: int,
                            num_pages: int, block_table: torch.Tensor,
                            context_lengths: torch.Tensor, requests: torch.Tensor,
                            scores: torch.Tensor, max_context: int, stream=None) -> torch.Tensor:
    """``scores[r, k] = query[r] . key_k`` for ``k`` below the group's length.

    query: bf16 ``[rows, 128]``; key_cache: any CUDA tensor whose storage holds
    ``num_pages`` pages ``page_stride_bytes`` apart; block_table int32
    ``[requests, width]``; context_lengths / requests int32 ``[groups]``;
    scores fp32 ``[rows, >= max_context]``."""
    for t, nm in ((query, "query"), (context_lengths, "context_lengths"), (requests, "requests")):
        _cuda(t, nm)
    _cuda(key_cache, "key_cache", contiguous=False)
    _cuda(block_table, "block_table", contiguous=False)
    _cuda(scores, "scores", contiguous=False)
    if block_table.stride(-1) != 1 or scores.stride(-1) != 1:
        raise ValueError("block_table and scores need unit stride in their last dimension")
    if query.dtype != torch.bfloat16 or query.dim() != 2 or query.shape[1] != 128:
        raise ValueError("query must be bf16 [rows, 128]")
    if scores.dtype != torch.float32 or scores.shape[1] < max_context:
        raise ValueError("scores must be float32 [rows, >= max_context]")
    _check(lib().pml_indexer_scores_bf16(
        _ptr(query), query.shape[0], _ptr(key_cache), page_stride_bytes, num_pages,
        _ptr(block_table), block_table.stride(0), block_table.shape[0], _ptr(context_lengths),
        _ptr(requests), context_lengths.numel(), _ptr(scores), scores.stride(0), max_context,
        _stream(stream)), "pml_indexer_scores_bf16")
    return scores


def pml_topk_logits(logits: torch.Tensor, seq_lens: torch.Tensor, next_n: int, max_context: int,
                    k: int, indices: torch.Tensor | None = None,
                    values: torch.Tensor | None = None, stream=None):
    """Each row's ``k`` largest logits among positions ``p <= seq_lens[b] -
    next_n + t`` (and ``< max_context``), descending, equal values by
    position; -1 / -inf past the candidates.  Returns ``(indices, values)``;
    ``values`` only if given."""
    _cuda(logits, "logits", contiguous=False)
    _cuda(seq_lens, "seq_lens")
    if logits.dtype != torch.float32 or logits.stride(-1) != 1:
        raise ValueError("logits must be float32 with unit last stride")
    if seq_lens.dtype != torch.int32:
        raise ValueError("seq_lens must be int32")
    rows = seq_lens.numel() * next_n
    if indices is None:
        indices = torch.empty((rows, k), dtype=torch.int32, device=logits.device)
    _cuda(indices, "indices", contiguous=False)
    if values is not None:
        _cuda(values, "values", contiguous=False)
    _check(lib().pml_topk_logits(
        _ptr(logits), logits.stride(0), _ptr(seq_lens), seq_lens.numel(), next_n, max_context, k,
        _ptr(indices), indices.stride(0), _ptr(values), values.stride(0) if values is not None else 0,
        _stream(stream)), "pml_topk_logits")
    return indices, values


def pml_indexer_scores_nvfp4(query: torch.Tensor, query_scales: torch.Tensor,
                             key_cache: torch.Tensor, page_stride_bytes: int,
                             key_scales: torch.Tensor, scale_page_stride_bytes: int,
                             num_pages: int, block_table: torch.Tensor,
                             context_lengths: torch.Tensor, requests: torch.Tensor,
                             scores: torch.Tensor, max_context: int, stream=None) -> torch.Tensor:
    """``scores[r, k] = query[r] . key_k`` over NVFP4 rows: 64 bytes of E2M1
    codes (two to a byte) and 8 E4M3 scales per row, one per 16 values.

    query uint8 ``[rows, 64]``, query_scales uint8 ``[rows, 8]``; key_cache /
    key_scales: CUDA tensors whose storage holds ``num_pages`` pages of 64x64
    code bytes ``page_stride_bytes`` apart and of 64x8 scale bytes
    ``scale_page_stride_bytes`` apart (they may view one buffer); the rest as
    ``pml_indexer_scores_bf16``."""
    for t, nm in ((query, "query"), (query_scales, "query_scales"), (context_lengths, "context_lengths"),
                  (requests, "requests")):
        _cuda(t, nm)
    for t, nm in ((key_cache, "key_cache"), (key_scales, "key_scales"), (block_table, "block_table"),
                  (scores, "scores")):
        _cuda(t, nm, contiguous=False)
    if query.element_size() != 1 or query.dim() != 2 or query.shape[1] != 64:
        raise ValueError("query must be uint8 [rows, 64]")
    if query_scales.element_size() != 1 or tuple(query_scales.shape) != (query.shape[0], 8):
        raise ValueError("query_scales must be uint8 [rows, 8]")
    if scores.dtype != torch.float32 or scores.stride(-1) != 1 or block_table.stride(-1) != 1:
        raise ValueError("scores must be float32 with unit last stride; block_table unit stride")
    _check(lib().pml_indexer_scores_nvfp4(
        _ptr(query), _ptr(query_scales), query.shape[0], _ptr(key_cache), int(page_stride_bytes),
        _ptr(key_scales), int(scale_page_stride_bytes), int(num_pages), _ptr(block_table),
        block_table.stride(0), block_table.shape[0], _ptr(context_lengths), _ptr(requests),
        context_lengths.numel(), _ptr(scores), scores.stride(0), max_context, _stream(stream)),
        "pml_indexer_scores_nvfp4")
    return scores


def pml_fp4_paged_mqa_logits(q: torch.Tensor, q_sf: torch.Tensor, kv_cache: torch.Tensor,
                             weights: torch.Tensor, seq_lens: torch.Tensor,
                             block_table: torch.Tensor, out: torch.Tensor, max_context: int,
                             next_n: int, schedule_meta: torch.Tensor | None = None,
                             num_ctas: int = 0, stream=None) -> torch.Tensor:
    """MXFP4 logits ``out[b*next_n+t, p] = sum_h w[t,h] * relu(q[t,h] . k_p)``.

    q uint8 ``[batch*next_n, 64, 64]`` (E2M1 two to a byte), q_sf uint8
    ``[batch*next_n, 64, 4]`` (E8M0, one per 32 values), kv_cache uint8
    ``[num_blocks, 4352]`` (64 keys x 64 code bytes, then 64 x 4 scales),
    weights fp32 ``[batch*next_n, 64]``; out bf16 or fp32 ``[batch*next_n,
    >= max_context]``."""
    for t, nm in ((q, "q"), (q_sf, "q_sf"), (kv_cache, "kv_cache"), (weights, "weights"),
                  (seq_lens, "seq_lens")):
        _cuda(t, nm)
    _cuda(block_table, "block_table", contiguous=False)
    _cuda(out, "out", contiguous=False)
    if out.dtype not in _OUT_DTYPES or out.stride(-1) != 1 or block_table.stride(-1) != 1:
        raise ValueError("out must be bf16 or float32 with unit last stride; block_table unit stride")
    batch = seq_lens.numel()
    if tuple(q.shape) != (batch * next_n, 64, 64) or tuple(q_sf.shape) != (batch * next_n, 64, 4):
        raise ValueError("q must be uint8 [batch*next_n, 64, 64], q_sf uint8 [batch*next_n, 64, 4]")
    _check(lib().pml_fp4_paged_mqa_logits(
        _ptr(q), _ptr(q_sf), _ptr(kv_cache), kv_cache.numel() // 4352, _ptr(weights),
        _ptr(seq_lens), _ptr(block_table), block_table.stride(0), _ptr(schedule_meta), num_ctas,
        _ptr(out), out.stride(0), _OUT_DTYPES[out.dtype], max_context, batch, next_n,
        _stream(stream)), "pml_fp4_paged_mqa_logits")
    return out


def pml_fp8_paged_mqa_logits_wait_test(q: torch.Tensor, kv_fused: torch.Tensor,
                                       weights: torch.Tensor, seq_lens: torch.Tensor,
                                       block_table: torch.Tensor, out: torch.Tensor,
                                       max_context: int, next_n: int, drop_stage: int,
                                       wait_limit_us: int, stream=None) -> torch.Tensor:
    """Test support (no counterpart on the pages): the fp32 fp8 logits call in
    which every CTA's producer leaves its stage ``drop_stage`` unpublished and
    every in-kernel wait gives up after ``wait_limit_us``, so that the
    kernel's timeout path runs: PML_STATUS_WAIT_TIMEOUT is set and the call
    returns with those CTAs' logits incomplete."""
    for t, nm in ((q, "q"), (kv_fused, "kv_fused"), (weights, "weights"), (seq_lens, "seq_lens")):
        _cuda(t, nm)
    _cuda(block_table, "block_table", contiguous=False)
    _cuda(out, "out", contiguous=False)
    if out.dtype != torch.float32 or out.stride(-1) != 1 or block_table.stride(-1) != 1:
        raise ValueError("out must be float32; out and block_table need unit last stride")
    batch = seq_lens.numel()
    _check(lib().pml_fp8_paged_mqa_logits_wait_test(
        _ptr(q), _ptr(kv_fused), kv_fused.numel() // 8448, _ptr(weights), _ptr(seq_lens),
        _ptr(block_table), block_table.stride(0), _ptr(out), out.stride(0), max_context, batch,
        next_n, q.shape[1], drop_stage, wait_limit_us, _stream(stream)),
        "pml_fp8_paged_mqa_logits_wait_test")
    return out


def pml_fp8_paged_mqa_logits_noalloc(q: torch.Tensor, kv_fused: torch.Tensor,
                                     weights: torch.Tensor, seq_lens: torch.Tensor,
                                     block_table: torch.Tensor, out: torch.Tensor, max_context: int,
                                     next_n: int, num_ctas: int = 0, stream=None) -> torch.Tensor:
    """Same result as ``pml_fp8_paged_mqa_logits`` with a GPU-computed schedule
    kept in the library's own fixed device array (no device allocation by the
    library; see include/pml.h for the sharing rules).  Arguments as there."""
    for t, nm in ((q, "q"), (kv_fused, "kv_fused"), (weights, "weights"), (seq_lens, "seq_lens")):
        _cuda(t, nm)
    _cuda(block_table, "block_table", contiguous=False)
    _cuda(out, "out", contiguous=False)
    batch = seq_lens.numel()
    _check(lib().pml_fp8_paged_mqa_logits_noalloc(
        _ptr(q), _ptr(kv_fused), kv_fused.numel() // 8448, _ptr(weights), _ptr(seq_lens),
        _ptr(block_table), block_table.stride(0), num_ctas, _ptr(out), out.stride(0), max_context,
        batch, next_n, q.shape[1], _stream(stream)), "pml_fp8_paged_mqa_logits_noalloc")
    return out


# ---------------------------------------------------------------- pages' keyword style

def compute_paged_mqa_logits_schedule(seq_lens: torch.Tensor, next_n: int = 1,
                                      num_ctas: int | None = None) -> torch.Tensor:
    """Build a schedule once to pass back via ``schedule_meta=`` (valid while
    the contents of ``seq_lens`` are unchanged)."""
    n = pml_default_num_ctas(seq_lens.device.index) if num_ctas is None else num_ctas
    return pml_schedule(seq_lens, n, next_n)


def fp8_paged_mqa_logits(q, kv_fused, weights, seq_lens, block_table, *, max_context=None,
                         schedule_meta=None, out=None, num_ctas=None, output_dtype=None):
    """Keyword-style wrapper.  ``out`` is allocated (filled with -inf, of
    ``output_dtype``: float32 by default, or bfloat16) only when not given;
    rows of empty requests and positions past each request's length are never
    written."""
    batch = seq_lens.numel()
    next_n = q.shape[0] // max(batch, 1)
    if max_context is None:
        max_context = block_table.shape[1] * 64
    if out is None:
        out = torch.full((q.shape[0], max_context), float("-inf"),
                         dtype=output_dtype or torch.float32, device=q.device)
    elif output_dtype is not None and out.dtype != output_dtype:
        raise ValueError("out and output_dtype disagree")
    if num_ctas is None:
        num_ctas = (schedule_meta.numel() // 2 - 1) if schedule_meta is not None else 0
    return pml_fp8_paged_mqa_logits_ex(q, kv_fused, weights, seq_lens, block_table, out,
                                       max_context, next_n, schedule_meta=schedule_meta,
                                       num_ctas=num_ctas)


def indexer_scores(query, key_cache, block_table, context_lengths, *, requests, scores,
                   page_stride_bytes=None, num_pages=None):
    """Keyword-style wrapper for ``key_cache`` given as ``[pages, 64, 128]``
    (possibly a strided view with any page stride that is a multiple of 16 B)."""
    if page_stride_bytes is None:
        page_stride_bytes = key_cache.stride(0) * key_cache.element_size()
    if num_pages is None:
        num_pages = key_cache.shape[0]
    return pml_indexer_scores_bf16(query, key_cache, page_stride_bytes, num_pages, block_table,
                                   context_lengths, requests, scores, scores.shape[1])
