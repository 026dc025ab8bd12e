/*
 * pml -- paged MQA logits for the sparse-attention indexer, on GB300 (sm_103a).
 *
 * C ABI of libpml.so.  All tensor arguments are DEVICE pointers owned by the
 * caller; the library never allocates, frees or synchronises, and enqueues all
 * work on `stream` (a cudaStream_t passed as void*; NULL is the legacy default
 * stream).  Every entry point is one or two kernel launches with no host
 * round-trip, so it can be captured in a CUDA graph.
 *
 * Return value: PML_OK (0) or one of the PML_ERR_* codes.  Only conditions the
 * host can see are reported synchronously (null or misaligned pointers, shapes
 * outside the supported set, a CUDA launch error); nothing is launched when a
 * check fails.  Problems only the device can see -- a block-table entry outside
 * the cache, a bounded wait that ran out -- set bits of a sticky per-device
 * status word (pml_device_status) and the offending access is skipped.
 *
 * Sources: FlashInfer documentation pages "flashinfer.attn_scores" (the
 * definition, the output contract, "Scheduling and Setup") and
 * "flashinfer.sdsa.indexer_scores" (the single-head case and its arguments).
 */
#ifndef PML_H
#define PML_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    PML_OK = 0,
    PML_ERR_INVALID_ARG = 1,  /* null pointer, negative size, inconsistent sizes */
    PML_ERR_UNSUPPORTED = 2,  /* next_n, num_heads or group size outside the supported set */
    PML_ERR_ALIGNMENT = 3,    /* a pointer or stride not aligned as stated below */
    PML_ERR_CUDA = 4          /* a CUDA call failed; see pml_last_cuda_error() */
};

/* Device status bits (see pml_device_status). */
#define PML_STATUS_WAIT_TIMEOUT 1u  /* an in-kernel wait exceeded its limit; that CTA stopped early */
#define PML_STATUS_BAD_BLOCK 2u     /* a block_table entry was outside [0, num_blocks) */
#define PML_STATUS_BAD_REQUEST 4u   /* a group's request was outside [0, num_requests) */
#define PML_STATUS_FP4_INEXACT 8u   /* MXFP4 scales so far apart that tiny products may have been dropped (see pml_fp4_paged_mqa_logits) */

/* Version of this ABI (major*100 + minor). */
int pml_version(void);

/* Static description of an error code. */
const char* pml_error_string(int code);

/* The cudaError_t of the last PML_ERR_CUDA returned on this host thread. */
int pml_last_cuda_error(void);

/* Default persistent grid size for `device`: its SM count (0 on error). */
int pml_default_num_ctas(int device);

/* Number of int32 elements of a schedule for `num_ctas` CTAs: (num_ctas+1)*2. */
int pml_schedule_meta_elems(int num_ctas);

/* Block-table width that covers `max_seq_len` keys: ceil(max_seq_len / 64).
 * ("flashinfer.attn_scores", "Scheduling and Setup": min_block_table_width.) */
int pml_min_block_table_width(int max_seq_len);

/* `max_seq_len` rounded up to whole 64-key blocks.  (Same section:
 * padded_seq_len.) */
int pml_padded_seq_len(int max_seq_len);

/*
 * pml_schedule -- the persistent CTA work assignment
 * ("flashinfer.attn_scores", "Scheduling and Setup").
 *
 * Request b owns ceil(seq_lens[b]/64) blocks of 64 keys (none if
 * seq_lens[b] <= 0).  All blocks, in request order, are cut into num_ctas
 * contiguous ranges whose sizes differ by at most one, the first
 * (total mod num_ctas) one block longer.  schedule_meta (device, int32
 * [num_ctas+1][2], written) receives for each range the (request,
 * block-within-request) where it starts; a start at the end and the closing
 * entry are (batch, 0).
 *
 * The schedule depends on seq_lens and num_ctas only (next_n is accepted for
 * the pages' signature and must be 1..4).  A schedule is valid only while the
 * contents of seq_lens are unchanged: recompute it whenever they change,
 * including on every graph replay in which they change.
 */
int pml_schedule(const int32_t* seq_lens, int batch, int next_n, int num_ctas,
                 int32_t* schedule_meta, void* stream);

/*
 * pml_fp8_paged_mqa_logits ("flashinfer.attn_scores": math block, the two
 * bullets under it, the note on the output contract).
 *
 *   out[b*next_n + t, p] = s_p * sum_h weights[b*next_n + t, h]
 *                                     * relu( q[b*next_n + t, h, :] . k_p )
 *
 * for every request b with seq_lens[b] > 0, slot t < next_n and position
 * p < min(seq_lens[b], max_context); the rectifier acts per head, before the
 * weighted sum, and weights may be negative.  Key p of request b is row p%64
 * of physical block block_table[b*bt_stride + p/64]; s_p is that row's scale.
 * Row b*next_n+t is meaningful only for p <= seq_lens[b] - next_n + t; later
 * positions below seq_lens[b] are written but carry no meaning (callers mask).
 * Nothing else in `out` is written: not positions >= seq_lens[b], and not the
 * rows of requests with seq_lens[b] == 0 (pre-fill `out` to read them).
 *
 * q            e4m3 [batch*next_n, num_heads, 128], contiguous, 16-byte aligned
 * kv_fused     [num_blocks][8448] bytes, 16-byte aligned: per block 64 keys x
 *              128 e4m3 (row-major, 8192 B), then 64 little-endian fp32
 *              per-token scales (256 B)
 * weights      fp32 [batch*next_n, num_heads], contiguous, 16-byte aligned
 * seq_lens     int32 [batch]; contents are trusted (not checked)
 * block_table  int32 [batch, bt_stride]; entries below ceil(min(seq_lens[b],
 *              max_context)/64) must be in [0, num_blocks) (others are never
 *              read); an entry outside is replaced by 0 and flagged
 *              PML_STATUS_BAD_BLOCK
 * schedule_meta  NULL (each CTA computes its range on the GPU) or the output
 *              of pml_schedule for the same seq_lens and num_ctas
 * num_ctas     persistent grid size; 0 = pml_default_num_ctas (only allowed
 *              with schedule_meta == NULL)
 * out          fp32 [batch*next_n, out_stride], 4-byte aligned;
 *              out_stride >= max_context
 * max_context  >= 1, and ceil(max_context/64) <= bt_stride
 * next_n       1..4;  num_heads  8, 16, 32 or 64 (head dim fixed at 128)
 */
int pml_fp8_paged_mqa_logits(const uint8_t* q, const uint8_t* kv_fused, int64_t num_blocks,
                             const float* weights, const int32_t* seq_lens,
                             const int32_t* block_table, int64_t bt_stride,
                             const int32_t* schedule_meta, int num_ctas, float* out,
                             int64_t out_stride, int max_context, int batch, int next_n,
                             int num_heads, void* stream);

/* Output element types of pml_fp8_paged_mqa_logits_ex. */
#define PML_DTYPE_FLOAT32 0
#define PML_DTYPE_BFLOAT16 1

/*
 * pml_fp8_paged_mqa_logits_ex -- pml_fp8_paged_mqa_logits with the pages'
 * output_dtype option ("flashinfer.attn_scores": the paragraph comparing the
 * two variants -- the fp8 call exposes acc_dtype and output_dtype, output
 * float32 by default).
 *
 * output_dtype  PML_DTYPE_FLOAT32: `out` is fp32, exactly as
 *               pml_fp8_paged_mqa_logits (which is this call with that value);
 *               PML_DTYPE_BFLOAT16: `out` is bf16 [batch*next_n, out_stride]
 *               (2-byte aligned), each logit the fp32 result rounded to
 *               nearest even.  The accumulator is fp32 in both cases (the
 *               tensor cores' f32 accumulation; no other acc_dtype is
 *               offered).  Other values return PML_ERR_UNSUPPORTED.
 * All other arguments, the written region and the errors are those of
 * pml_fp8_paged_mqa_logits; out_stride counts elements of the output type.
 */
int pml_fp8_paged_mqa_logits_ex(const uint8_t* q, const uint8_t* kv_fused, int64_t num_blocks,
                                const float* weights, const int32_t* seq_lens,
                                const int32_t* block_table, int64_t bt_stride,
                                const int32_t* schedule_meta, int num_ctas, void* out,
                                int64_t out_stride, int output_dtype, int max_context, int batch,
                                int next_n, int num_heads, void* stream);

/*
 * pml_indexer_scores_bf16 ("flashinfer.sdsa.indexer_scores": body and the
 * query, key_cache, block_table, context_lengths, requests and scores
 * parameters).
 *
 *   scores[r, k] = query[r, :] . key_k      (one head: no weight, no ReLU)
 *
 * Query rows come in `groups` uniform groups of G = rows/groups consecutive
 * rows (1 <= G <= 8); group g owns rows [g*G, (g+1)*G), has
 * context_lengths[g] keys and reads the pages of block-table row
 * requests[g].  For k < min(context_lengths[g], max_context) the score is
 * written; later entries are not written, and a group of length <= 0 reads
 * nothing (its requests entry may hold any value).
 *
 * query          bf16 [rows, 128], contiguous, 16-byte aligned
 * key_cache      page P starts at byte P*page_stride_bytes and holds 64 keys x
 *                128 bf16 (row-major); base 16-byte aligned;
 *                page_stride_bytes a multiple of 16 and >= 16384
 * block_table    int32 [num_requests, bt_stride]; read entries must be in
 *                [0, num_pages) (else replaced by 0, PML_STATUS_BAD_BLOCK)
 * requests       int32 [groups]; read entries must be in [0, num_requests)
 *                (else replaced by 0, PML_STATUS_BAD_REQUEST)
 * scores         fp32 [rows, scores_stride], scores_stride >= max_context
 * max_context    >= 1, and ceil(max_context/64) <= bt_stride
 */
int pml_indexer_scores_bf16(const uint16_t* query, int rows, const uint16_t* key_cache,
                            int64_t page_stride_bytes, int64_t num_pages,
                            const int32_t* block_table, int64_t bt_stride, int num_requests,
                            const int32_t* context_lengths, const int32_t* requests, int groups,
                            float* scores, int64_t scores_stride, int max_context, void* stream);

/*
 * pml_indexer_scores_nvfp4 ("flashinfer.sdsa.indexer_scores": the NVFP4 forms
 * of query, key_cache, query_scales and key_scales).
 *
 *   scores[r, k] = q_r . k_k       (dequantised values; one head, no weight,
 *                                   no rectifier)
 *
 * A row of 128 values is 64 bytes of E2M1 codes, two to a byte (element d in
 * byte d/2; the low nibble holds the even element), and 8 E4M3 scale codes,
 * scale j applying to elements 16j .. 16j+15: value = E2M1(code) * E4M3(scale).
 * Every E4M3 code is accepted (negative scales negate their block; 0x7F and
 * 0xFF are NaN and make every score of their row or key NaN).  Groups,
 * lengths, requests, the written region and the status bits are those of
 * pml_indexer_scores_bf16.  Every product of two values is exact in fp32
 * (the block-scaled tensor cores take codes and scales as stored); only the
 * sums round.
 *
 * query           uint8 [rows, 64], 16-byte aligned
 * query_scales    uint8 [rows, 8] (E4M3), 8-byte aligned
 * key_cache       page P's 64 keys x 64 bytes start at byte P*page_stride_bytes;
 *                 base 16-byte aligned, page_stride_bytes a multiple of 16 and
 *                 >= 4096
 * key_scales      page P's 64 keys x 8 scale bytes start at byte
 *                 P*scale_page_stride_bytes; base 8-byte aligned,
 *                 scale_page_stride_bytes a multiple of 8 and >= 512 (the two
 *                 may be views of one cache holding each page's keys and then
 *                 its scales)
 * num_pages       pages in both (block_table entries must be below it)
 * scores          fp32 [rows, scores_stride], scores_stride >= max_context
 */
int pml_indexer_scores_nvfp4(const uint8_t* query, const uint8_t* query_scales, int rows,
                             const uint8_t* key_cache, int64_t page_stride_bytes,
                             const uint8_t* key_scales, int64_t scale_page_stride_bytes,
                             int64_t num_pages, const int32_t* block_table, int64_t bt_stride,
                             int num_requests, const int32_t* context_lengths,
                             const int32_t* requests, int groups, float* scores,
                             int64_t scores_stride, int max_context, void* stream);

/*
 * pml_fp8_paged_mqa_logits_wait_test -- test support; the pages have no
 * counterpart.  The fp32 fp8 logits call with the in-kernel schedule, in which
 * every CTA's producer leaves its stage number drop_stage (counted from 0
 * within the CTA) unpublished, and every wait inside the kernel gives up after
 * wait_limit_us microseconds instead of one second.  The roles waiting on the
 * missing stage run out of time: the CTA records PML_STATUS_WAIT_TIMEOUT,
 * raises its abort flag so that its other roles stop waiting, lets the copies
 * and MMAs it issued complete, frees its tensor memory and returns.  Logits of
 * the CTAs that stopped are incomplete.  It exists so that the tests can run
 * the kernel's timeout path on the GPU without a fault or a hang: the call
 * returns, the status word says what happened, and the device stays usable
 * for the next call.
 *
 * Arguments as pml_fp8_paged_mqa_logits (fp32 out, no schedule_meta, default
 * CTA count).  Returns PML_ERR_INVALID_ARG for drop_stage < 0 or
 * wait_limit_us outside 1 .. 1000000, else as pml_fp8_paged_mqa_logits.
 */
int pml_fp8_paged_mqa_logits_wait_test(const uint8_t* q, const uint8_t* kv_fused,
                                       int64_t num_blocks, const float* weights,
                                       const int32_t* seq_lens, const int32_t* block_table,
                                       int64_t bt_stride, float* out, int64_t out_stride,
                                       int max_context, int batch, int next_n, int num_heads,
                                       int drop_stage, int64_t wait_limit_us, void* stream);

/*
 * pml_fp4_paged_mqa_logits -- the MXFP4 variant ("flashinfer.attn_scores":
 * the math block, its two bullets and the paragraph after them: MXFP4 block
 * scales folded into the dequantised values, one per 32-element group on
 * both operands; two FP4 values per q byte; 64 heads of 128 only; no
 * per-position factor; default output bf16).
 *
 *   out[b*next_n + t, p] = sum_h w[t,h] * relu(q[t,h] . k_p)
 *
 * over values code * 2^(e - 127): code an E2M1 value (element d of a row in
 * byte d/2, low nibble for even d), e the row's E8M0 scale byte d/32.
 * Written region and schedule as pml_fp8_paged_mqa_logits.
 *
 * q          [batch*next_n, 64, 64] packed E2M1, 16-byte aligned
 * q_sf       [batch*next_n, 64, 4] E8M0, 16-byte aligned
 * kv_cache   [num_blocks][4352] bytes, 16-byte aligned: per block 64 keys x
 *            64 code bytes (4096 B), then 64 x 4 E8M0 scale bytes (256 B)
 * weights    fp32 [batch*next_n, 64], 16-byte aligned
 * out        output_dtype PML_DTYPE_BFLOAT16 (the pages' default) or
 *            PML_DTYPE_FLOAT32, [batch*next_n, out_stride], aligned to its
 *            element
 * batch      <= 65535; next_n 1..4; other arguments, the written region and
 *            the schedule as pml_fp8_paged_mqa_logits (next_n 3 and 4 run
 *            as two passes over the cache, slots 0-1 then the rest, each
 *            its own launch on `stream`)
 *
 * Method: every row (a key, or one head of one query slot) has a frame
 * 2^(E - 127), E its largest group exponent.  The block-scaled tensor cores
 * take the codes as stored and each group's scale relative to its row's
 * frame (2^(e - E), at most 1), so every product of a key group and a query
 * group is exact in fp32 and only the sums round; the key's and the query
 * rows' frames are applied afterwards, the rows' folded into the head weights
 * relative to the slot's largest one.  So each logit is its exact value up
 * to fp32 rounding of the sums -- a logit beyond the output type's range is
 * +-inf -- except where a key's and a query row's scale spreads together
 * exceed 124 binades, when products smaller than 2^-124 of the two rows'
 * frames may be rounded or dropped (a group more than 127 binades below its
 * row's frame is dropped), or a head's largest scale lies more than 100
 * binades below the slot's largest: both set PML_STATUS_FP4_INEXACT.  An
 * E8M0 NaN scale (0xFF) makes its group NaN, and a NaN dot product is
 * rectified to 0.
 */
int pml_fp4_paged_mqa_logits(const uint8_t* q, const uint8_t* q_sf, const uint8_t* kv_cache,
                             int64_t num_blocks, const float* weights, const int32_t* seq_lens,
                             const int32_t* block_table, int64_t bt_stride,
                             const int32_t* schedule_meta, int num_ctas, void* out,
                             int64_t out_stride, int output_dtype, int max_context, int batch,
                             int next_n, void* stream);

/*
 * pml_topk_logits -- the indexer's selection over the logits
 * ("flashinfer.attn_scores", intro: the logits are what a sparse-attention
 * indexer uses to choose which KV tokens to keep; note: row b*next_n+t is
 * meaningful for positions 0 .. seq_lens[b]-next_n+t).  The pages fix neither
 * k nor the order of equal values; this call's definition:
 *
 *   indices[r, 0..k) = the k positions p < min(seq_lens[b]-next_n+t+1,
 *   max_context) with the largest logits[r, p], r = b*next_n+t, in descending
 *   order of value -- the float32 bit order, -NaN < -inf < ... < -0 < +0 < ...
 *   < +inf < +NaN -- equal values in ascending position; slots past the
 *   number of candidates hold -1 (values: -inf).  Requests with
 *   seq_lens[b] <= 0 have no candidates.
 *
 * logits    fp32 [batch*next_n, logits_stride], logits_stride >= max_context
 *           (only candidate positions are read)
 * indices   int32 [batch*next_n, indices_stride], indices_stride >= k (written)
 * values    NULL, or fp32 [batch*next_n, values_stride] (written: the
 *           selected logits, bit for bit)
 * k         1 .. 4096 (else PML_ERR_UNSUPPORTED); next_n >= 1
 */
int pml_topk_logits(const float* logits, int64_t logits_stride, const int32_t* seq_lens, int batch,
                    int next_n, int max_context, int k, int32_t* indices, int64_t indices_stride,
                    float* values, int64_t values_stride, void* stream);

/*
 * pml_fp8_paged_mqa_logits_noalloc -- the two-step call (pml_schedule, then
 * pml_fp8_paged_mqa_logits with that schedule) for callers that cannot
 * allocate device memory.  The documentation pages have no counterpart: it
 * exists for this library's users.
 *
 * Who needs it: code that only receives the buffers it works on and has no
 * way to obtain more device memory -- a plugin inside a host runtime that owns
 * all allocations, a serving loop running under a memory pool that forbids
 * raw cudaMalloc (which also synchronises the device), or a C caller with no
 * allocator at hand.  The regular two-step path needs such a caller to find
 * room for the (num_ctas+1)*2 int32 schedule; here the schedule lives in a
 * fixed array inside the library's own device memory (8200 bytes, held on
 * every device that loads the library until the process exits).
 *
 * Arguments and results are those of pml_fp8_paged_mqa_logits without
 * schedule_meta.  num_ctas: 0 = pml_default_num_ctas (capped at the limit),
 * at most pml_noalloc_max_ctas() = 1024; larger values return
 * PML_ERR_INVALID_ARG and launch nothing.  Nothing is allocated or freed: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *
 * The first call on a device looks up the array's device address with that
 * device current (cudaGetSymbolAddress); make that first call before any
 * stream capture.  A failure there returns PML_ERR_CUDA.
 *
 * All calls share the one array, which keeps the last call's schedule; each
 * call rewrites every entry it reads, so nothing needs clearing.  Calls whose
 * work overlaps on the GPU (different streams, no ordering between them) race
 * on the array: order them, or use the regular entry points with separate
 * buffers.  If the logits launch is rejected after the schedule was written,
 * the only side effect is the rewritten array.
 */
int pml_fp8_paged_mqa_logits_noalloc(const uint8_t* q, const uint8_t* kv_fused,
                                     int64_t num_blocks, const float* weights,
                                     const int32_t* seq_lens, const int32_t* block_table,
                                     int64_t bt_stride, int num_ctas, float* out,
                                     int64_t out_stride, int max_context, int batch, int next_n,
                                     int num_heads, void* stream);

/* Largest num_ctas pml_fp8_paged_mqa_logits_noalloc accepts (1024). */
int pml_noalloc_max_ctas(void);

/* Read (and, if clear != 0, reset) the current device's sticky status word.
 * Synchronises with the device (waits for all work queued so far). */
int pml_device_status(unsigned int* status, int clear);

#ifdef __cplusplus
}
#endif

#endif /* PML_H */
