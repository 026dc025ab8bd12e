"""Seeded synthetic inputs for paged MQA logits and single-head indexer scores.

This module only draws inputs: random numbers, their encoding into e4m3 /
bf16 bytes, and the paged-cache layout.  It holds none of the logits
arithmetic, so both the GPU library's tests and the CPU oracle can take their
inputs from it.

Generators are ``numpy.random.Generator(PCG64(seed))``; the drawing order per
fp8 problem is: sequence lengths -> physical page permutation -> q -> keys ->
per-token scales -> weights.

Layouts (the paged-cache reading of "flashinfer.attn_scores", second bullet,
and "flashinfer.sdsa.indexer_scores", ``key_cache`` parameter):

* ``kv_fused`` uint8 ``[num_blocks, 8448]``: per block 64 keys x 128 e4m3
  bytes, row-major, then 64 little-endian fp32 per-token scales.
* ``q`` uint8 e4m3 ``[batch*next_n, H, 128]``, ``weights`` fp32
  ``[batch*next_n, H]``, row ``b*next_n + t``.
* ``block_table`` int32 ``[batch, width]``; entries past a request's last
  block, and key rows past its length in its last block, hold a poison page /
  poison bytes (e4m3 NaN, NaN scale) when ``poison`` is set, so that reading
  them would show up in the output.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128
BLOCK_KEYS = 64
BLOCK_KEY_BYTES = BLOCK_KEYS * HEAD_DIM        # 8192
BLOCK_BYTES = BLOCK_KEY_BYTES + BLOCK_KEYS * 4  # 8448
E4M3_MAX = 448.0
E4M3_NAN = 0x7F
SENTINEL_BITS = 0x7FC0DEAD                     # a quiet-NaN payload used to pre-fill outputs


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_e4m3(x: np.ndarray) -> np.ndarray:
    """Round to E4M3FN (nearest-even, saturating at +-448) and return the bytes."""
    t = torch.from_numpy(np.clip(np.asarray(x, dtype=np.float32), -E4M3_MAX, E4M3_MAX))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def to_bf16(x: np.ndarray) -> np.ndarray:
    """Round to bfloat16 (nearest-even) and return the uint16 bit patterns."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def blocks_for(seq_len: int) -> int:
    return (max(int(seq_len), 0) + BLOCK_KEYS - 1) // BLOCK_KEYS


def sentinel_f32(shape) -> np.ndarray:
    return np.full(shape, SENTINEL_BITS, dtype=np.uint32).view(np.float32)


SENTINEL_BF16_BITS = 0x7FDE                    # a bf16 NaN payload for bf16 outputs


def sentinel_bf16_bits(shape) -> np.ndarray:
    """uint16 bit patterns of a bf16 array pre-filled with the sentinel."""
    return np.full(shape, SENTINEL_BF16_BITS, dtype=np.uint16)


@dataclass
class Fp8Problem:
    name: str
    seed: int
    next_n: int
    num_heads: int
    q: np.ndarray            # uint8 [B*n, H, 128]
    kv_fused: np.ndarray     # uint8 [num_blocks, 8448]
    weights: np.ndarray      # float32 [B*n, H]
    seq_lens: np.ndarray     # int32 [B]
    block_table: np.ndarray  # int32 [B, width]
    max_context: int
    info: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.kv_fused.shape[0])

    @property
    def positions(self) -> int:
        return int(np.maximum(self.seq_lens, 0).sum())

    def algorithmic_bytes(self, out_bytes: int = 4) -> int:
        """Bytes the method must move once: every valid key (128 e4m3 + one fp32
        scale), one block-table entry per block, each request's q rows and
        weights and its length, and the logits it writes (out_bytes each: 4
        for fp32, 2 for bf16)."""
        n, H = self.next_n, self.num_heads
        total = 0
        for L in self.seq_lens.tolist():
            if L <= 0:
                total += 4
                continue
            total += L * (HEAD_DIM + 4) + blocks_for(L) * 4 + n * H * (HEAD_DIM + 4) + 4
            total += n * L * out_bytes
        return total

    def algorithmic_flops(self) -> int:
        return int(2 * self.next_n * self.num_heads * HEAD_DIM * self.positions)


def fp8_problem(name: str, seq_lens, next_n: int, num_heads: int, seed: int, *,
                poison: bool = True, extra_blocks: int = 0, bt_width: int | None = None,
                max_context: int | None = None, g: np.random.Generator | None = None,
                block_table: np.ndarray | None = None, num_blocks: int | None = None
                ) -> Fp8Problem:
    """Build an fp8 paged problem for the given lengths.

    The physical pool holds every request's blocks (plus ``extra_blocks``
    unused ones and, with ``poison``, one poison block at the end), placed in
    a random order; ``block_table`` may instead be given explicitly together
    with ``num_blocks``."""
    g = g or rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = seq_lens.shape[0]
    nbs = [blocks_for(L) for L in seq_lens.tolist()]
    need = sum(nbs)
    width = bt_width or max(1, max(nbs, default=1))
    if block_table is None:
        pool = need + extra_blocks
        perm = g.permutation(pool).astype(np.int32)
        num_blocks = pool + (1 if poison else 0)
        poison_block = pool if poison else 0
        bt = np.full((B, width), poison_block, dtype=np.int32)
        off = 0
        for b, nb in enumerate(nbs):
            bt[b, :nb] = perm[off:off + nb]
            off += nb
    else:
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        assert num_blocks is not None
        width = bt.shape[1]
    rows = B * next_n
    q = to_e4m3(g.standard_normal((rows, num_heads, HEAD_DIM), dtype=np.float32))
    keys = to_e4m3(g.standard_normal((num_blocks, BLOCK_KEYS, HEAD_DIM), dtype=np.float32))
    scales = g.uniform(0.5, 2.0, size=(num_blocks, BLOCK_KEYS)).astype(np.float32)
    weights = (g.standard_normal((rows, num_heads), dtype=np.float32)
               / np.float32(np.sqrt(num_heads))).astype(np.float32)
    if poison:
        # key rows past each request's length inside its last block, and any
        # physical block no request uses, are e4m3 NaN with a NaN scale
        used = np.zeros(num_blocks, dtype=bool)
        for b, (L, nb) in enumerate(zip(seq_lens.tolist(), nbs)):
            used[bt[b, :nb]] = True
            if nb and L % BLOCK_KEYS:
                last = bt[b, nb - 1]
                keys[last, L % BLOCK_KEYS:, :] = E4M3_NAN
                scales[last, L % BLOCK_KEYS:] = np.nan
        keys[~used] = E4M3_NAN
        scales[~used] = np.nan
    kv = np.empty((num_blocks, BLOCK_BYTES), dtype=np.uint8)
    kv[:, :BLOCK_KEY_BYTES] = keys.reshape(num_blocks, BLOCK_KEY_BYTES)
    kv[:, BLOCK_KEY_BYTES:] = scales.astype("<f4").view(np.uint8).reshape(num_blocks, -1)
    mc = max_context or max(1, int(seq_lens.max(initial=0)))
    return Fp8Problem(name, seed, next_n, num_heads, q, kv, weights, seq_lens, bt, mc)


# ---------------------------------------------------------------- presets

def tiny(seed: int = 0) -> Fp8Problem:
    """batch 2, next_n 1, 8 heads, lengths {100, 37}, block_table a random
    permutation of 4 physical blocks (two per request)."""
    g = rng(seed)
    seq_lens = np.array([100, 37], dtype=np.int32)
    bt = g.permutation(4).astype(np.int32).reshape(2, 2)
    p = fp8_problem("tiny", seq_lens, 1, 8, seed, g=g, block_table=bt, num_blocks=4, poison=False)
    return p


def decode(seed: int = 1, batch: int = 64, lo: int = 1024, hi: int = 32768,
           num_heads: int = 64, poison: bool = True) -> Fp8Problem:
    """Decode: next_n 1, 64 heads, lengths uniform on [lo, hi]."""
    g = rng(seed)
    seq_lens = g.integers(lo, hi, size=batch, endpoint=True).astype(np.int32)
    return fp8_problem(f"decode_b{batch}", seq_lens, 1, num_heads, seed, g=g, poison=poison)


def mtp(next_n: int = 4, seed: int | None = None, batch: int = 32, lo: int = 8192,
        hi: int = 65536, num_heads: int = 64, poison: bool = True) -> Fp8Problem:
    """Multi-token-prediction verify: next_n 2 or 4, lengths uniform on [lo, hi]."""
    seed = seed if seed is not None else (2 if next_n == 4 else 3)
    g = rng(seed)
    seq_lens = g.integers(lo, hi, size=batch, endpoint=True).astype(np.int32)
    return fp8_problem(f"mtp{next_n}_b{batch}", seq_lens, next_n, num_heads, seed, g=g,
                       poison=poison)


def skewed(seed: int = 4, order: str = "shuffled", long_len: int = 131072,
           num_heads: int = 64, lo: int = 512, hi: int = 4096) -> Fp8Problem:
    """16 requests: one of ``long_len`` tokens, three empty, twelve uniform on
    [lo, hi]; ``order`` is "shuffled", "first" (long request first) or "last"."""
    g = rng(seed)
    rest = g.integers(lo, hi, size=12, endpoint=True).astype(np.int32)
    lens = np.concatenate([[long_len], [0, 0, 0], rest]).astype(np.int32)
    if order == "shuffled":
        lens = lens[g.permutation(lens.shape[0])]
    elif order == "last":
        lens = np.concatenate([lens[1:], lens[:1]])
    return fp8_problem(f"skewed_{order}", lens, 1, num_heads, seed, g=g)


# ---------------------------------------------------------------- bf16 indexer

@dataclass
class Bf16Problem:
    name: str
    seed: int
    group_size: int
    query: np.ndarray            # uint16 bf16 bits [rows, 128]
    key_cache: np.ndarray        # uint8 [num_pages, page_stride_bytes]
    page_stride_bytes: int
    block_table: np.ndarray      # int32 [requests, width]
    context_lengths: np.ndarray  # int32 [groups]
    requests: np.ndarray         # int32 [groups]
    max_context: int
    info: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return int(self.query.shape[0])

    @property
    def groups(self) -> int:
        return int(self.context_lengths.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.key_cache.shape[0])

    @property
    def positions(self) -> int:
        return int(np.maximum(self.context_lengths, 0).sum())

    def key_pages(self) -> np.ndarray:
        """The keys as a uint16 ``[pages, 64, 128]`` view (bf16 bits)."""
        return (self.key_cache[:, :BLOCK_KEYS * HEAD_DIM * 2].copy()
                .view(np.uint16).reshape(-1, BLOCK_KEYS, HEAD_DIM))

    def algorithmic_bytes(self) -> int:
        G = self.group_size
        total = self.rows * HEAD_DIM * 2
        for L in self.context_lengths.tolist():
            if L > 0:
                total += L * HEAD_DIM * 2 + G * L * 4 + blocks_for(L) * 4
        return total

    def algorithmic_flops(self) -> int:
        return int(2 * HEAD_DIM * self.group_size * self.positions)


def indexer(group_size: int, seed: int = 5, groups: int = 256, max_context: int = 65536,
            num_requests: int | None = None, min_zero: int = 8, page_pad_bytes: int = 0,
            shared_requests: bool = False, lo: int = 0, hi: int | None = None,
            poison: bool = True) -> Bf16Problem:
    """Single-head bf16 indexer problem: ``groups`` groups of ``group_size``
    consecutive query rows, lengths uniform on [lo, hi] (default [0,
    max_context]) with at least ``min_zero`` forced zeros.

    With ``shared_requests`` groups map to a random request among
    ``num_requests`` (each long enough for its longest group); otherwise each
    group has a request of its own.  Pages are ``64*128*2 + page_pad_bytes``
    bytes apart; the pad bytes and every unused page hold bf16 NaN when
    ``poison`` is set.  Groups of length 0 get a garbage ``requests`` entry
    (the pages allow any value there)."""
    g = rng(seed)
    hi = max_context if hi is None else hi
    lens = g.integers(lo, hi, size=groups, endpoint=True).astype(np.int32)
    if min_zero:
        lens[g.choice(groups, size=min(min_zero, groups), replace=False)] = 0
    rows = groups * group_size
    if shared_requests:
        R = num_requests or 64
        req = g.integers(0, R, size=groups).astype(np.int32)
        need = np.zeros(R, dtype=np.int64)
        for gi in range(groups):
            need[req[gi]] = max(need[req[gi]], blocks_for(lens[gi]))
    else:
        R = groups
        req = np.arange(groups, dtype=np.int32)
        need = np.array([blocks_for(L) for L in lens.tolist()], dtype=np.int64)
    width = max(1, (max_context + BLOCK_KEYS - 1) // BLOCK_KEYS)
    pool = int(need.sum())
    perm = g.permutation(pool).astype(np.int32)
    num_pages = pool + (1 if poison else 0)
    bt = np.full((R, width), pool if poison else 0, dtype=np.int32)
    off = 0
    for r in range(R):
        bt[r, :need[r]] = perm[off:off + need[r]]
        off += int(need[r])
    query = to_bf16(g.standard_normal((rows, HEAD_DIM), dtype=np.float32))
    keys = to_bf16(g.standard_normal((num_pages, BLOCK_KEYS, HEAD_DIM), dtype=np.float32))
    stride = BLOCK_KEYS * HEAD_DIM * 2 + page_pad_bytes
    assert stride % 16 == 0
    kc = np.empty((num_pages, stride), dtype=np.uint8)
    if poison:
        keys[pool:] = 0x7FC0
        kc[:, BLOCK_KEYS * HEAD_DIM * 2:] = 0xFF
    kc[:, :BLOCK_KEYS * HEAD_DIM * 2] = keys.reshape(num_pages, -1).view(np.uint8)
    # a group of length 0 reads nothing, so its request entry may hold any value
    req = req.copy()
    req[lens == 0] = np.int32(-123456789)
    return Bf16Problem(f"indexer_g{group_size}", seed, group_size, query, kc, stride, bt, lens,
                       req, max_context)


# ---------------------------------------------------------------- NVFP4 indexer

NVFP4_ROW_BYTES = HEAD_DIM // 2        # 64: two E2M1 codes per byte
NVFP4_SCALES = HEAD_DIM // 16          # 8 E4M3 scales per row
NVFP4_PAGE_KEY_BYTES = BLOCK_KEYS * NVFP4_ROW_BYTES    # 4096
NVFP4_PAGE_SCALE_BYTES = BLOCK_KEYS * NVFP4_SCALES     # 512
E4M3_NAN = 0x7F


@dataclass
class Nvfp4Problem:
    """Single-head indexer problem over NVFP4 queries and keys.  Keys of page
    P start at byte ``key_off + P*page_stride_bytes`` of ``key_buf`` (64 rows
    of 64 packed bytes); their scales at ``scale_off + P*scale_page_stride_bytes``
    of ``scale_buf`` (64 rows of 8 E4M3 bytes).  With ``fused`` the two are one
    buffer holding each page's keys and then its scales."""
    name: str
    seed: int
    group_size: int
    query: np.ndarray            # uint8 [rows, 64]
    query_scales: np.ndarray     # uint8 [rows, 8]
    key_buf: np.ndarray          # uint8 flat
    key_off: int
    page_stride_bytes: int
    scale_buf: np.ndarray        # uint8 flat (the same array as key_buf when fused)
    scale_off: int
    scale_page_stride_bytes: int
    num_pages: int
    block_table: np.ndarray      # int32 [requests, width]
    context_lengths: np.ndarray  # int32 [groups]
    requests: np.ndarray         # int32 [groups]
    max_context: int
    fused: bool = False

    @property
    def rows(self) -> int:
        return int(self.query.shape[0])

    @property
    def groups(self) -> int:
        return int(self.context_lengths.shape[0])

    @property
    def positions(self) -> int:
        return int(np.maximum(self.context_lengths, 0).sum())

    def key_view(self) -> np.ndarray:
        return self.key_buf[self.key_off:]

    def scale_view(self) -> np.ndarray:
        return self.scale_buf[self.scale_off:]

    def algorithmic_bytes(self) -> int:
        G = self.group_size
        total = self.rows * (NVFP4_ROW_BYTES + NVFP4_SCALES)
        for L in self.context_lengths.tolist():
            if L > 0:
                total += L * (NVFP4_ROW_BYTES + NVFP4_SCALES) + G * L * 4 + blocks_for(L) * 4
        return total

    def algorithmic_flops(self) -> int:
        return int(2 * HEAD_DIM * self.group_size * self.positions)


def random_e4m3_scales(g: np.random.Generator, shape, lo_exp: int = -3, hi_exp: int = 3):
    """Random positive normal E4M3 codes with exponents in [lo_exp, hi_exp]
    (bias 7) and any mantissa: the bytes directly, no rounding involved."""
    e = g.integers(lo_exp + 7, hi_exp + 7, size=shape, endpoint=True)
    m = g.integers(0, 7, size=shape, endpoint=True)
    return ((e << 3) | m).astype(np.uint8)


def indexer_nvfp4(group_size: int, seed: int = 6, groups: int = 256, max_context: int = 65536,
                  min_zero: int = 8, lo: int = 0, hi: int | None = None, fused: bool = True,
                  page_pad_bytes: int = 0, scale_pad_bytes: int = 0,
                  poison: bool = True, scales: str = "positive") -> Nvfp4Problem:
    """NVFP4 single-head problem: ``groups`` groups of ``group_size`` query rows,
    one request each, lengths uniform on [lo, hi] with at least ``min_zero``
    forced zeros.  E2M1 codes are uniform over all 16 values (bytes uniform on
    0..255).  ``scales``: "positive" -- random positive E4M3 codes between
    2^-3 and 2^3; "negative" -- the same codes with the sign bit set; "all" --
    bytes uniform on 0..255 (every E4M3 code: zeros, subnormals, negatives and
    the two NaNs), for queries and keys alike.
    ``fused``: one buffer of pages of [4096 key bytes][512 scale bytes]
    (+ ``page_pad_bytes``); otherwise separate key and scale buffers, pages
    4096 + ``page_pad_bytes`` and 512 + ``scale_pad_bytes`` bytes apart.  With
    ``poison`` every pad byte and the spare page's scales are E4M3 NaN, so a
    read outside a group's pages shows up as a NaN score."""
    g = rng(seed)
    hi = max_context if hi is None else hi
    lens = g.integers(lo, hi, size=groups, endpoint=True).astype(np.int32)
    if min_zero:
        lens[g.choice(groups, size=min(min_zero, groups), replace=False)] = 0
    rows = groups * group_size
    need = np.array([blocks_for(L) for L in lens.tolist()], dtype=np.int64)
    width = max(1, (max_context + BLOCK_KEYS - 1) // BLOCK_KEYS)
    pool = int(need.sum())
    perm = g.permutation(pool).astype(np.int32)
    num_pages = pool + (1 if poison else 0)
    bt = np.full((groups, width), pool if poison else 0, dtype=np.int32)
    off = 0
    for r in range(groups):
        bt[r, :need[r]] = perm[off:off + need[r]]
        off += int(need[r])
    def draw_scales(shape):
        if scales == "all":
            return g.integers(0, 255, size=shape, endpoint=True).astype(np.uint8)
        sc = random_e4m3_scales(g, shape)
        return sc | np.uint8(0x80) if scales == "negative" else sc

    assert scales in ("positive", "negative", "all")
    query = g.integers(0, 255, size=(rows, NVFP4_ROW_BYTES), endpoint=True).astype(np.uint8)
    qscales = draw_scales((rows, NVFP4_SCALES))
    keys = g.integers(0, 255, size=(num_pages, NVFP4_PAGE_KEY_BYTES), endpoint=True).astype(np.uint8)
    kscales = draw_scales((num_pages, NVFP4_PAGE_SCALE_BYTES))
    if poison:
        kscales[pool:] = E4M3_NAN
    fill = E4M3_NAN if poison else 0
    if fused:
        stride = NVFP4_PAGE_KEY_BYTES + NVFP4_PAGE_SCALE_BYTES + page_pad_bytes
        assert stride % 16 == 0
        buf = np.full((num_pages, stride), fill, dtype=np.uint8)
        buf[:, :NVFP4_PAGE_KEY_BYTES] = keys
        buf[:, NVFP4_PAGE_KEY_BYTES:NVFP4_PAGE_KEY_BYTES + NVFP4_PAGE_SCALE_BYTES] = kscales
        flat = buf.reshape(-1)
        p = Nvfp4Problem(f"nvfp4_g{group_size}", seed, group_size, query, qscales, flat, 0, stride,
                         flat, NVFP4_PAGE_KEY_BYTES, stride, num_pages, bt, lens, None,
                         max_context, fused=True)
    else:
        kstride = NVFP4_PAGE_KEY_BYTES + page_pad_bytes
        sstride = NVFP4_PAGE_SCALE_BYTES + scale_pad_bytes
        assert kstride % 16 == 0 and sstride % 8 == 0
        kb = np.full((num_pages, kstride), fill, dtype=np.uint8)
        kb[:, :NVFP4_PAGE_KEY_BYTES] = keys
        sb = np.full((num_pages, sstride), fill, dtype=np.uint8)
        sb[:, :NVFP4_PAGE_SCALE_BYTES] = kscales
        p = Nvfp4Problem(f"nvfp4_g{group_size}", seed, group_size, query, qscales,
                         kb.reshape(-1), 0, kstride, sb.reshape(-1), 0, sstride, num_pages, bt,
                         lens, None, max_context, fused=False)
    req = np.arange(groups, dtype=np.int32)
    req[lens == 0] = np.int32(-123456789)     # a group of length 0 may name any request
    p.requests = req
    return p


# ---------------------------------------------------------------- top-k input

def topk_logits_input(batch: int, next_n: int, max_context: int, seed: int = 9,
                      lo: int = 0, hi: int | None = None, distinct: int | None = None,
                      specials: bool = True, narrow: bool = False):
    """Synthetic logits rows [batch*next_n, max_context] and seq_lens for the
    top-k selection: values ~N(0, 4) (or ``distinct`` levels only, for many
    ties; or, ``narrow``, 1 + j * 2^-23 for j uniform below 2^15: values that
    agree in their top 16 bits), seq_lens uniform on [lo, hi] (default [0,
    max_context]); with ``specials`` some rows carry +-inf, signed zeros and a
    NaN."""
    g = rng(seed)
    hi = max_context if hi is None else hi
    seq_lens = g.integers(lo, hi, size=batch, endpoint=True).astype(np.int32)
    rows = batch * next_n
    if distinct:
        x = g.integers(-distinct // 2, distinct - distinct // 2, size=(rows, max_context))
        x = x.astype(np.float32)
    elif narrow:
        j = g.integers(0, 1 << 15, size=(rows, max_context)).astype(np.uint32)
        x = (np.uint32(0x3F800000) + j).view(np.float32)
    else:
        x = (g.standard_normal((rows, max_context), dtype=np.float32) * 4).astype(np.float32)
    if specials and rows > 0 and max_context >= 8:
        r = g.integers(0, rows, size=4)
        x[r[0], :4] = [np.inf, -np.inf, -0.0, 0.0]
        x[r[1], 1] = np.nan
        x[r[2], 2] = -np.nan
        x[r[3], 3] = np.float32(3.4e38)
    return x, seq_lens


@dataclass
class TopkProblem:
    """Synthetic logits rows for the top-k selection, shaped like a decode
    step's output (batch rows of max_context positions)."""
    name: str
    logits: np.ndarray        # float32 [batch*rows_per_request, max_context]
    seq_lens: np.ndarray      # int32 [batch]
    rows_per_request: int     # next_n of the logits
    max_context: int
    k: int

    @property
    def candidates(self) -> np.ndarray:
        n = self.rows_per_request
        sl = np.repeat(self.seq_lens.astype(np.int64), n)
        t = np.tile(np.arange(n), self.seq_lens.shape[0])
        lim = np.where(sl > 0, np.minimum(sl - n + t + 1, self.max_context), 0)
        return np.maximum(lim, 0)

    @property
    def positions(self) -> int:
        return int(self.candidates.sum())

    def algorithmic_bytes(self) -> int:
        """Each candidate logit read once, k indices written per row."""
        return int(self.candidates.sum() * 4 + self.logits.shape[0] * self.k * 4)

    def algorithmic_flops(self) -> int:
        return 0


def topk_decode(seed: int = 13, k: int = 2048) -> TopkProblem:
    """64 rows of 32768 logits with decode lengths U[1024, 32768], k = 2048."""
    x, sl = topk_logits_input(64, 1, 32768, seed=seed, lo=1024, hi=32768, specials=False)
    return TopkProblem("topk_decode", x, sl, 1, 32768, k)


# ---------------------------------------------------------------- MXFP4 logits
#
# The MXFP4 variant of the paged logits ("flashinfer.attn_scores", the
# paragraphs after the math block): q and keys hold E2M1 codes two to a byte
# with one E8M0 scale byte per 32 values; 64 heads, head_dim 128.  A KV block
# is 64 keys x 64 code bytes followed by 64 x 4 scale bytes.

MXFP4_ROW_BYTES = HEAD_DIM // 2                                   # 64
MXFP4_ROW_SCALES = HEAD_DIM // 32                                 # 4
MXFP4_BLOCK_CODE_BYTES = BLOCK_KEYS * MXFP4_ROW_BYTES              # 4096
MXFP4_BLOCK_BYTES = MXFP4_BLOCK_CODE_BYTES + BLOCK_KEYS * MXFP4_ROW_SCALES   # 4352
MXFP4_HEADS = 64
E8M0_NAN = 0xFF


@dataclass
class Mxfp4Problem:
    name: str
    seed: int
    next_n: int
    q: np.ndarray            # uint8 [B*n, 64, 64] packed E2M1
    q_sf: np.ndarray         # uint8 [B*n, 64, 4] E8M0
    kv: np.ndarray           # uint8 [num_blocks, 4352]
    weights: np.ndarray      # float32 [B*n, 64]
    seq_lens: np.ndarray     # int32 [B]
    block_table: np.ndarray  # int32 [B, width]
    max_context: int

    num_heads = MXFP4_HEADS

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.kv.shape[0])

    @property
    def positions(self) -> int:
        return int(np.maximum(self.seq_lens, 0).sum())

    def algorithmic_bytes(self, out_bytes: int = 2) -> int:
        """Bytes moved once: every valid key (64 code + 4 scale bytes), one
        block-table entry per block, each request's q rows, scales and weights
        and its length, and the logits written (bf16 by default)."""
        n, H = self.next_n, MXFP4_HEADS
        total = 0
        for L in self.seq_lens.tolist():
            if L <= 0:
                total += 4
                continue
            total += L * (MXFP4_ROW_BYTES + MXFP4_ROW_SCALES) + blocks_for(L) * 4
            total += n * H * (MXFP4_ROW_BYTES + MXFP4_ROW_SCALES + 4) + 4 + n * L * out_bytes
        return total

    def algorithmic_flops(self) -> int:
        """Multiply-adds of the dot products: 2 * n * H * 128 per position."""
        return int(2 * self.next_n * MXFP4_HEADS * HEAD_DIM * np.maximum(self.seq_lens, 0).sum())


def random_e8m0(g: np.random.Generator, shape, lo_exp: int = -4, hi_exp: int = 4) -> np.ndarray:
    """E8M0 scale bytes for 2^lo_exp .. 2^hi_exp (bias 127), drawn as bytes."""
    return (127 + g.integers(lo_exp, hi_exp, size=shape, endpoint=True)).astype(np.uint8)


def mxfp4_problem(name: str, seq_lens, next_n: int, seed: int, *, poison: bool = True,
                  g: np.random.Generator | None = None, block_table: np.ndarray | None = None,
                  num_blocks: int | None = None, max_context: int | None = None,
                  lo_exp: int = -4, hi_exp: int = 4, q_exp: tuple | None = None,
                  k_exp: tuple | None = None) -> Mxfp4Problem:
    """An MXFP4 paged problem.  Drawing order: page permutation -> q codes ->
    q scales -> key codes -> key scales -> weights.  Code bytes are uniform on
    0..255 (every E2M1 code, -0 included).  Scale exponents are uniform on
    ``q_exp`` / ``k_exp`` (inclusive (lo, hi) pairs, both ``(lo_exp, hi_exp)``
    unless given; (-127, 127) is every finite E8M0 value).  With ``poison``,
    key rows past a request's length and blocks no request uses carry NaN
    (0xFF) scales."""
    q_exp = q_exp or (lo_exp, hi_exp)
    k_exp = k_exp or (lo_exp, hi_exp)
    g = g or rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = seq_lens.shape[0]
    nbs = [blocks_for(L) for L in seq_lens.tolist()]
    need = sum(nbs)
    if block_table is None:
        perm = g.permutation(need).astype(np.int32)
        num_blocks = need + (1 if poison else 0)
        width = max(1, max(nbs, default=1))
        bt = np.full((B, width), need if poison else 0, dtype=np.int32)
        off = 0
        for b, nb in enumerate(nbs):
            bt[b, :nb] = perm[off:off + nb]
            off += nb
    else:
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        assert num_blocks is not None
    rows = B * next_n
    H = MXFP4_HEADS
    q = g.integers(0, 256, size=(rows, H, MXFP4_ROW_BYTES), dtype=np.uint8)
    q_sf = random_e8m0(g, (rows, H, MXFP4_ROW_SCALES), *q_exp)
    codes = g.integers(0, 256, size=(num_blocks, BLOCK_KEYS, MXFP4_ROW_BYTES), dtype=np.uint8)
    k_sf = random_e8m0(g, (num_blocks, BLOCK_KEYS, MXFP4_ROW_SCALES), *k_exp)
    weights = (g.standard_normal((rows, H), dtype=np.float32) / np.float32(8.0)).astype(np.float32)
    if poison:
        used = np.zeros(num_blocks, dtype=bool)
        for b, (L, nb) in enumerate(zip(seq_lens.tolist(), nbs)):
            used[bt[b, :nb]] = True
            if nb and L % BLOCK_KEYS:
                k_sf[bt[b, nb - 1], L % BLOCK_KEYS:, :] = E8M0_NAN
        k_sf[~used] = E8M0_NAN
    kv = np.empty((num_blocks, MXFP4_BLOCK_BYTES), dtype=np.uint8)
    kv[:, :MXFP4_BLOCK_CODE_BYTES] = codes.reshape(num_blocks, -1)
    kv[:, MXFP4_BLOCK_CODE_BYTES:] = k_sf.reshape(num_blocks, -1)
    mc = max_context or max(1, int(seq_lens.max(initial=0)))
    return Mxfp4Problem(name, seed, next_n, q, q_sf, kv, weights, seq_lens, bt, mc)


def mxfp4_decode(seed: int = 7, batch: int = 64, lo: int = 1024, hi: int = 32768,
                 next_n: int = 1, poison: bool = True, **scales) -> Mxfp4Problem:
    """MXFP4 decode: 64 heads, lengths uniform on [lo, hi] (the fp8 decode
    shape with the MXFP4 cache); ``scales`` as for ``mxfp4_problem``."""
    g = rng(seed)
    seq_lens = g.integers(lo, hi, size=batch, endpoint=True).astype(np.int32)
    return mxfp4_problem(f"mxfp4_decode_b{batch}", seq_lens, next_n, seed, g=g, poison=poison,
                         **scales)
