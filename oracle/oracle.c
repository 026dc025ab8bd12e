/*
 * Plain fp64 CPU oracle for the sparse-attention indexer's paged MQA logits.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker that the GPU path is
 * compared against.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or constant
 * with the CUDA library and includes nothing from it.
 *
 * Sources (FlashInfer documentation pages):
 *  - "flashinfer.attn_scores", intro and math block: the definition
 *        logits[t, p] = sum_h w[t,h] * relu(q[t,h] . k_p)
 *  - same page, first bullet: the rectifier is applied per head, before the
 *    weighted sum; weights may be negative, so the result may be negative.
 *  - same page, second bullet: the fp8 variant multiplies by the per-token
 *    FP32 KV scale s_p held in the trailing scale region of each kv_fused
 *    block.
 *  - same page, note: output row b*next_n + t; row t is meaningful for
 *    positions 0 .. seq_lens[b] - next_n + t; a request with seq_lens[b] == 0
 *    is skipped and its rows are never written.
 *  - same page, "Scheduling and Setup": a per-call CTA work assignment that is
 *    a function of seq_lens (and next_n) only.
 *  - "flashinfer.sdsa.indexer_scores": the single-head case, a plain dot
 *    product of a query row with each key below its group's length; later
 *    entries are not written.
 *
 * Readings (the pages leave these open):
 *  - kv_fused block = 64 keys x 128 e4m3 bytes (row-major, 8192 B) followed by
 *    64 little-endian fp32 scales (256 B): 8448 B per block.
 *  - e4m3 is the E4M3FN flavour: bias 7, no infinities, 0x7F/0xFF are NaN.
 *  - fp8: positions p >= seq_lens[b] are not written (stricter than "may never
 *    be written").
 *  - indexer_scores: groups are uniform, group g = rows [g*G, (g+1)*G) with
 *    G = rows / groups.
 *  - NVFP4 indexer_scores ("flashinfer.sdsa.indexer_scores": the query,
 *    key_cache, query_scales and key_scales parameters): element d of a
 *    128-value row is the E2M1 code in byte d/2, low nibble for even d, high
 *    nibble for odd d; its value is that code times the E4M3 scale number
 *    d/16 of the row (query_scales [rows][8], key_scales [pages][64][8]).
 *    No per-tensor scale appears in that call.
 *  - MXFP4 paged MQA logits ("flashinfer.attn_scores", second bullet and the
 *    paragraph after it: MXFP4 block scales folded into the dequantised
 *    values, one scale per 32-element group on both operands, two FP4 values
 *    per q byte, num_heads 64 and head_dim 128 only, no per-position factor):
 *    the scales are the OCP MX shared-scale format E8M0 (value 2^(e - 127),
 *    0xFF NaN), one per 32 values (sf_vec_size 32); element d of a row is the
 *    E2M1 code in byte d/2 (low nibble for even d) times scale d/32 of the
 *    row; q [batch*next_n][64][64] bytes with q_sf [batch*next_n][64][4]; a
 *    KV block (is_kv_sf_interleaved false) is 64 keys x 64 code bytes
 *    (4096 B) followed by 64 x 4 scale bytes (256 B): 4352 B per block, the
 *    same keys-then-scales order as the fp8 kv_fused block.
 *
 * MXFP4 arithmetic: a term is a product of two E2M1 values (at most 2
 * significant bits each) and two powers of two, exact in fp64; the 128-term
 * sum is exact too unless the group scales of the two rows put terms more
 * than ~45 binary orders apart.
 *
 * Arithmetic: every product of two e4m3 values is a multiple of 2^-18 below
 * 2^18 in magnitude, and every product of two bf16 values has at most 16
 * significant bits, so the 128-term dot products are exact in fp64 in any
 * order; so is an NVFP4 dot product, whose terms are products of four values
 * of at most 4 significant bits each, between 2^-40 and 2^23.  The only roundings are the fp64 products w*relu(x), the fp64 sum
 * over heads and the final product with s_p.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_HEAD_DIM 128
#define ORC_BLOCK_KEYS 64
#define ORC_BLOCK_KEY_BYTES (ORC_BLOCK_KEYS * ORC_HEAD_DIM)
#define ORC_BLOCK_BYTES (ORC_BLOCK_KEY_BYTES + ORC_BLOCK_KEYS * 4)

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* OCP 8-bit float E4M3 ("FN" variant): 1 sign bit, 4 exponent bits with bias
 * 7, 3 mantissa bits.  Exponent field 0 encodes subnormals m * 2^-9; the code
 * with all exponent and mantissa bits set (0x7F / 0xFF) is NaN; there is no
 * infinity, so the largest finite value is 1.75 * 2^8 = 448. */
double orc_e4m3_decode(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);             /* m/8 * 2^(1-7) */
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* OCP 4-bit float E2M1: 1 sign bit (bit 3), 2 exponent bits with bias 1, 1
 * mantissa bit.  Exponent field 0 encodes the subnormal m * 0.5; there are no
 * infinities or NaNs, so the magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double orc_e2m1_decode(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 0x3;
    int m = code & 0x1;
    double mag = e == 0 ? 0.5 * m : ldexp(1.0 + m / 2.0, e - 1);
    return sign ? -mag : mag;
}

/* OCP MX shared scale E8M0: an unsigned biased exponent, value 2^(e - 127);
 * 0xFF is NaN. */
double orc_e8m0_decode(uint8_t code)
{
    if (code == 0xFF) return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* bfloat16 is the upper half of an IEEE binary32 value. */
double orc_bf16_decode(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float orc_load_f32_le(const uint8_t* p)
{
    uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
                 ((uint32_t)p[3] << 24);
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------ */
/* Work schedule                                                       */
/* ------------------------------------------------------------------ */

/* The persistent schedule: request b owns nb_b = ceil(seq_lens[b]/64) KV
 * blocks; the blocks of all requests, in request order, are numbered
 * 0 .. T-1 and cut into num_ctas contiguous ranges whose sizes differ by at
 * most one (the first T mod num_ctas ranges get the extra block).  meta[2i],
 * meta[2i+1] is the (request, block-within-request) where range i starts;
 * a start at T (an empty range at the end) and the closing entry i = num_ctas
 * are (batch, 0).  Empty requests own no blocks, so a start never names one.
 * Returns T. */
int64_t orc_schedule(const int32_t* seq_lens, int batch, int num_ctas, int32_t* meta)
{
    int64_t total = 0;
    for (int b = 0; b < batch; ++b) {
        int32_t L = seq_lens[b] > 0 ? seq_lens[b] : 0;
        total += (L + ORC_BLOCK_KEYS - 1) / ORC_BLOCK_KEYS;
    }
    int64_t base = total / num_ctas, extra = total % num_ctas;
    for (int i = 0; i <= num_ctas; ++i) {
        int64_t start = (int64_t)i * base + (i < extra ? i : extra);
        /* find b with P[b] <= start < P[b+1] by a linear walk */
        int64_t prefix = 0;
        int b = 0;
        for (; b < batch; ++b) {
            int32_t L = seq_lens[b] > 0 ? seq_lens[b] : 0;
            int64_t nb = (L + ORC_BLOCK_KEYS - 1) / ORC_BLOCK_KEYS;
            if (start < prefix + nb) break;
            prefix += nb;
        }
        meta[2 * i] = b;
        meta[2 * i + 1] = (b < batch) ? (int32_t)(start - prefix) : 0;
    }
    return total;
}

/* ------------------------------------------------------------------ */
/* fp8 paged MQA logits                                                */
/* ------------------------------------------------------------------ */

typedef struct {
    const uint8_t* q;
    const uint8_t* kv_fused;
    int64_t num_blocks;
    const float* weights;
    const int32_t* seq_lens;
    const int32_t* block_table;
    int64_t bt_stride;
    int batch, next_n, num_heads;
    double* out;
    double* mag;
    int64_t out_stride;
    int max_context;
    double e4m3[256];
    int next_request;         /* shared work counter, guarded by lock */
    pthread_mutex_t lock;
    int status;
} orc_fp8_job;

static void orc_fp8_request(orc_fp8_job* J, int b)
{
    const int n = J->next_n, H = J->num_heads;
    const int32_t L = J->seq_lens[b];
    double x[256];
    if (L <= 0) return;                                  /* rows never written */
    for (int t = 0; t < n; ++t) {
        const int64_t row = (int64_t)b * n + t;
        const uint8_t* qrow = J->q + row * H * ORC_HEAD_DIM;
        const float* w = J->weights + row * H;
        for (int p = 0; p < L && p < J->max_context; ++p) {
            /* paging: logical block p/64 of request b lives in physical block
             * block_table[b, p/64]; key p is row p%64 of that block, and its
             * scale is the (p%64)-th fp32 of the block's trailing region. */
            const int64_t phys = J->block_table[(int64_t)b * J->bt_stride + p / ORC_BLOCK_KEYS];
            const uint8_t* blk = J->kv_fused + phys * ORC_BLOCK_BYTES;
            const uint8_t* k = blk + (p % ORC_BLOCK_KEYS) * ORC_HEAD_DIM;
            const double s = (double)orc_load_f32_le(blk + ORC_BLOCK_KEY_BYTES + 4 * (p % ORC_BLOCK_KEYS));
            double acc = 0.0, bound = 0.0;
            for (int h = 0; h < H; ++h) {
                double dot = 0.0;
                for (int d = 0; d < ORC_HEAD_DIM; ++d)
                    dot += J->e4m3[qrow[h * ORC_HEAD_DIM + d]] * J->e4m3[k[d]];
                x[h] = dot;
            }
            for (int h = 0; h < H; ++h) {
                double r = x[h] > 0.0 ? x[h] : 0.0;        /* relu per head */
                acc += (double)w[h] * r;                   /* then weight and sum */
                bound += fabs((double)w[h]) * fabs(x[h]);
            }
            J->out[row * J->out_stride + p] = s * acc;     /* times s_p */
            if (J->mag) J->mag[row * J->out_stride + p] = fabs(s) * bound;
        }
    }
}

static void* orc_fp8_worker(void* arg)
{
    orc_fp8_job* J = (orc_fp8_job*)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int b = J->next_request++;
        pthread_mutex_unlock(&J->lock);
        if (b >= J->batch) break;
        orc_fp8_request(J, b);
    }
    return NULL;
}

static int orc_run_threads(void* (*fn)(void*), void* job, int nthreads)
{
    if (nthreads <= 1) {
        fn(job);
        return 0;
    }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return -1;
    int started = 0;
    for (int i = 0; i < nthreads; ++i)
        if (pthread_create(&th[started], NULL, fn, job) == 0) ++started;
    if (started == 0) fn(job);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    return 0;
}

/* logits for every request with seq_lens[b] > 0, every slot t < next_n and
 * every position p < min(seq_lens[b], max_context), written to
 * out[(b*next_n + t) * out_stride + p] in fp64.  Nothing else in out is
 * touched.  If mag is not NULL it receives, at the same places,
 * |s_p| * sum_h |w[t,h]| * |q[t,h] . k_p|, the scale of the rounding error a
 * float implementation may make.  Returns 0, or -1 on bad arguments. */
int orc_fp8_paged_mqa_logits(const uint8_t* q, const uint8_t* kv_fused, int64_t num_blocks,
                             const float* weights, const int32_t* seq_lens,
                             const int32_t* block_table, int64_t bt_stride, int batch,
                             int next_n, int num_heads, double* out, double* mag,
                             int64_t out_stride, int max_context, int nthreads)
{
    if (!q || !kv_fused || !weights || !seq_lens || !block_table || !out) return -1;
    if (next_n < 1 || num_heads < 1 || num_heads > 256 || batch < 0) return -1;
    orc_fp8_job J;
    memset(&J, 0, sizeof J);
    J.q = q; J.kv_fused = kv_fused; J.num_blocks = num_blocks; J.weights = weights;
    J.seq_lens = seq_lens; J.block_table = block_table; J.bt_stride = bt_stride;
    J.batch = batch; J.next_n = next_n; J.num_heads = num_heads; J.out = out; J.mag = mag;
    J.out_stride = out_stride; J.max_context = max_context;
    for (int c = 0; c < 256; ++c) J.e4m3[c] = orc_e4m3_decode((uint8_t)c);
    pthread_mutex_init(&J.lock, NULL);
    orc_run_threads(orc_fp8_worker, &J, nthreads);
    pthread_mutex_destroy(&J.lock);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Single-head bf16 indexer scores                                     */
/* ------------------------------------------------------------------ */

typedef struct {
    const uint16_t* query;
    int rows;
    const uint8_t* key_cache;
    int64_t page_stride_bytes;
    const int32_t* block_table;
    int64_t bt_stride;
    const int32_t* context_lengths;
    const int32_t* requests;
    int groups;
    double* scores;
    double* mag;
    int64_t scores_stride;
    int max_context;
    int next_group;
    pthread_mutex_t lock;
} orc_bf16_job;

static void orc_bf16_group(orc_bf16_job* J, int g)
{
    const int G = J->rows / J->groups;
    const int32_t len = J->context_lengths[g];
    if (len <= 0) return;                           /* reads nothing, writes nothing */
    const int32_t req = J->requests[g];
    for (int r = g * G; r < (g + 1) * G; ++r) {
        const uint16_t* qr = J->query + (int64_t)r * ORC_HEAD_DIM;
        for (int k = 0; k < len && k < J->max_context; ++k) {
            const int64_t page = J->block_table[(int64_t)req * J->bt_stride + k / ORC_BLOCK_KEYS];
            const uint8_t* kp = J->key_cache + page * J->page_stride_bytes +
                                (int64_t)(k % ORC_BLOCK_KEYS) * ORC_HEAD_DIM * 2;
            double dot = 0.0, bound = 0.0;
            for (int d = 0; d < ORC_HEAD_DIM; ++d) {
                uint16_t kb = (uint16_t)(kp[2 * d] | (kp[2 * d + 1] << 8));
                double prod = orc_bf16_decode(qr[d]) * orc_bf16_decode(kb);
                dot += prod;
                bound += fabs(prod);
            }
            J->scores[(int64_t)r * J->scores_stride + k] = dot;
            if (J->mag) J->mag[(int64_t)r * J->scores_stride + k] = bound;
        }
    }
}

static void* orc_bf16_worker(void* arg)
{
    orc_bf16_job* J = (orc_bf16_job*)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int g = J->next_group++;
        pthread_mutex_unlock(&J->lock);
        if (g >= J->groups) break;
        orc_bf16_group(J, g);
    }
    return NULL;
}

/* scores[r, k] = query[r] . key k of the group's request, for every group g
 * with context_lengths[g] > 0, rows r of group g and k < min(length,
 * max_context), in fp64.  key_cache is addressed in bytes: page P starts at
 * P * page_stride_bytes and holds 64 keys of 128 little-endian bf16.  If mag
 * is not NULL it receives sum_d |query[r,d] * key[k,d]| at the same places.
 * Returns 0, or -1 on bad arguments. */
int orc_indexer_scores_bf16(const uint16_t* query, int rows, const uint8_t* key_cache,
                            int64_t page_stride_bytes, const int32_t* block_table,
                            int64_t bt_stride, const int32_t* context_lengths,
                            const int32_t* requests, int groups, double* scores, double* mag,
                            int64_t scores_stride, int max_context, int nthreads)
{
    if (!query || !key_cache || !block_table || !context_lengths || !requests || !scores)
        return -1;
    if (groups <= 0 || rows % groups != 0) return -1;
    orc_bf16_job J;
    memset(&J, 0, sizeof J);
    J.query = query; J.rows = rows; J.key_cache = key_cache;
    J.page_stride_bytes = page_stride_bytes; J.block_table = block_table;
    J.bt_stride = bt_stride; J.context_lengths = context_lengths; J.requests = requests;
    J.groups = groups; J.scores = scores; J.mag = mag; J.scores_stride = scores_stride;
    J.max_context = max_context;
    pthread_mutex_init(&J.lock, NULL);
    orc_run_threads(orc_bf16_worker, &J, nthreads);
    pthread_mutex_destroy(&J.lock);
    return 0;
}

/* ------------------------------------------------------------------ */
/* NVFP4 indexer scores                                                */
/* ------------------------------------------------------------------ */

typedef struct {
    const uint8_t* query;          /* [rows][64] packed E2M1 */
    const uint8_t* query_scales;   /* [rows][8] E4M3 */
    int rows;
    const uint8_t* key_cache;      /* page P at P * page_stride_bytes: [64][64] packed */
    int64_t page_stride_bytes;
    const uint8_t* key_scales;     /* page P at P * scale_page_stride_bytes: [64][8] E4M3 */
    int64_t scale_page_stride_bytes;
    const int32_t* block_table;
    int64_t bt_stride;
    const int32_t* context_lengths;
    const int32_t* requests;
    int groups;
    double* scores;
    double* mag;
    int64_t scores_stride;
    int max_context;
    int next_group;
    double e2m1[16];
    double e4m3[256];
    pthread_mutex_t lock;
} orc_nvfp4_job;

/* Value of element d of a packed row with its eight per-16 scales. */
static double orc_nvfp4_value(const orc_nvfp4_job* J, const uint8_t* packed,
                              const uint8_t* scales, int d)
{
    const uint8_t byte = packed[d / 2];
    const uint8_t code = (d & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
    return J->e2m1[code] * J->e4m3[scales[d / 16]];
}

static void orc_nvfp4_group(orc_nvfp4_job* J, int g)
{
    const int G = J->rows / J->groups;
    const int32_t len = J->context_lengths[g];
    if (len <= 0) return;                           /* reads nothing, writes nothing */
    const int32_t req = J->requests[g];
    for (int r = g * G; r < (g + 1) * G; ++r) {
        const uint8_t* qp = J->query + (int64_t)r * (ORC_HEAD_DIM / 2);
        const uint8_t* qs = J->query_scales + (int64_t)r * (ORC_HEAD_DIM / 16);
        for (int k = 0; k < len && k < J->max_context; ++k) {
            const int64_t page = J->block_table[(int64_t)req * J->bt_stride + k / ORC_BLOCK_KEYS];
            const int key = k % ORC_BLOCK_KEYS;
            const uint8_t* kp = J->key_cache + page * J->page_stride_bytes +
                                (int64_t)key * (ORC_HEAD_DIM / 2);
            const uint8_t* ks = J->key_scales + page * J->scale_page_stride_bytes +
                                (int64_t)key * (ORC_HEAD_DIM / 16);
            double dot = 0.0, bound = 0.0;
            for (int d = 0; d < ORC_HEAD_DIM; ++d) {
                const double prod = orc_nvfp4_value(J, qp, qs, d) * orc_nvfp4_value(J, kp, ks, d);
                dot += prod;
                bound += fabs(prod);
            }
            J->scores[(int64_t)r * J->scores_stride + k] = dot;
            if (J->mag) J->mag[(int64_t)r * J->scores_stride + k] = bound;
        }
    }
}

static void* orc_nvfp4_worker(void* arg)
{
    orc_nvfp4_job* J = (orc_nvfp4_job*)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int g = J->next_group++;
        pthread_mutex_unlock(&J->lock);
        if (g >= J->groups) break;
        orc_nvfp4_group(J, g);
    }
    return NULL;
}

/* scores[r, k] = (dequantised query row r) . (dequantised key k of the
 * group's request), in fp64, for every group g with context_lengths[g] > 0,
 * rows r of group g and k < min(length, max_context); nothing else is
 * written.  Dequantisation: element d = E2M1 code (byte d/2, low nibble for
 * even d) times the row's E4M3 scale d/16.  If mag is not NULL it receives
 * sum_d |q_d * k_d| at the same places.  Returns 0, or -1 on bad arguments. */
int orc_indexer_scores_nvfp4(const uint8_t* query, const uint8_t* query_scales, int rows,
                             const uint8_t* key_cache, int64_t page_stride_bytes,
                             const uint8_t* key_scales, int64_t scale_page_stride_bytes,
                             const int32_t* block_table, int64_t bt_stride,
                             const int32_t* context_lengths, const int32_t* requests, int groups,
                             double* scores, double* mag, int64_t scores_stride, int max_context,
                             int nthreads)
{
    if (!query || !query_scales || !key_cache || !key_scales || !block_table ||
        !context_lengths || !requests || !scores)
        return -1;
    if (groups <= 0 || rows % groups != 0) return -1;
    orc_nvfp4_job J;
    memset(&J, 0, sizeof J);
    J.query = query; J.query_scales = query_scales; J.rows = rows;
    J.key_cache = key_cache; J.page_stride_bytes = page_stride_bytes;
    J.key_scales = key_scales; J.scale_page_stride_bytes = scale_page_stride_bytes;
    J.block_table = block_table; J.bt_stride = bt_stride;
    J.context_lengths = context_lengths; J.requests = requests; J.groups = groups;
    J.scores = scores; J.mag = mag; J.scores_stride = scores_stride; J.max_context = max_context;
    for (int c = 0; c < 16; ++c) J.e2m1[c] = orc_e2m1_decode((uint8_t)c);
    for (int c = 0; c < 256; ++c) J.e4m3[c] = orc_e4m3_decode((uint8_t)c);
    pthread_mutex_init(&J.lock, NULL);
    orc_run_threads(orc_nvfp4_worker, &J, nthreads);
    pthread_mutex_destroy(&J.lock);
    return 0;
}

/* ------------------------------------------------------------------ */
/* MXFP4 paged MQA logits                                              */
/* ------------------------------------------------------------------ */

#define ORC_FP4_HEADS 64
#define ORC_FP4_ROW_BYTES (ORC_HEAD_DIM / 2)                     /* 64 */
#define ORC_FP4_ROW_SCALES (ORC_HEAD_DIM / 32)                   /* 4 */
#define ORC_FP4_BLOCK_CODE_BYTES (ORC_BLOCK_KEYS * ORC_FP4_ROW_BYTES)
#define ORC_FP4_BLOCK_BYTES (ORC_FP4_BLOCK_CODE_BYTES + ORC_BLOCK_KEYS * ORC_FP4_ROW_SCALES)

typedef struct {
    const uint8_t* q;
    const uint8_t* q_sf;
    const uint8_t* kv;
    int64_t num_blocks;
    const float* weights;
    const int32_t* seq_lens;
    const int32_t* block_table;
    int64_t bt_stride;
    int batch, next_n;
    double* out;
    double* mag;
    int64_t out_stride;
    int max_context;
    int next_request;
    pthread_mutex_t lock;
} orc_fp4_job;

/* Value of element d of a packed MXFP4 row with its four per-32 scales. */
static double orc_mxfp4_value(const uint8_t* packed, const uint8_t* scales, int d)
{
    const uint8_t byte = packed[d / 2];
    const uint8_t code = (d % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
    return orc_e2m1_decode(code) * orc_e8m0_decode(scales[d / 32]);
}

static void orc_fp4_request(orc_fp4_job* J, int b)
{
    const int n = J->next_n, H = ORC_FP4_HEADS;
    const int32_t L = J->seq_lens[b];
    double qv[ORC_FP4_HEADS][ORC_HEAD_DIM], kv[ORC_HEAD_DIM], x[ORC_FP4_HEADS];
    if (L <= 0) return;                                  /* rows never written */
    for (int t = 0; t < n; ++t) {
        const int64_t row = (int64_t)b * n + t;
        for (int h = 0; h < H; ++h)
            for (int d = 0; d < ORC_HEAD_DIM; ++d)
                qv[h][d] = orc_mxfp4_value(J->q + (row * H + h) * ORC_FP4_ROW_BYTES,
                                           J->q_sf + (row * H + h) * ORC_FP4_ROW_SCALES, d);
        const float* w = J->weights + row * H;
        for (int p = 0; p < L && p < J->max_context; ++p) {
            /* paging as for fp8: key p is row p%64 of physical block
             * block_table[b, p/64]; its 4 scales are the (p%64)-th group of 4
             * bytes after the block's 4096 code bytes */
            const int64_t phys = J->block_table[J->bt_stride * (int64_t)b + p / ORC_BLOCK_KEYS];
            const uint8_t* blk = J->kv + phys * ORC_FP4_BLOCK_BYTES;
            const uint8_t* k = blk + (p % ORC_BLOCK_KEYS) * ORC_FP4_ROW_BYTES;
            const uint8_t* ks = blk + ORC_FP4_BLOCK_CODE_BYTES + (p % ORC_BLOCK_KEYS) * ORC_FP4_ROW_SCALES;
            for (int d = 0; d < ORC_HEAD_DIM; ++d) kv[d] = orc_mxfp4_value(k, ks, d);
            double sum = 0.0, err = 0.0;
            for (int h = 0; h < H; ++h) {
                double dot = 0.0;
                for (int d = 0; d < ORC_HEAD_DIM; ++d) dot += qv[h][d] * kv[d];
                x[h] = dot;
            }
            for (int h = 0; h < H; ++h) {
                const double rl = x[h] > 0.0 ? x[h] : 0.0;  /* relu per head */
                sum += (double)w[h] * rl;                   /* then weight and sum */
                err += fabs((double)w[h]) * fabs(x[h]);
            }
            J->out[row * J->out_stride + p] = sum;          /* no per-position factor */
            if (J->mag) J->mag[row * J->out_stride + p] = err;
        }
    }
}

static void* orc_fp4_worker(void* arg)
{
    orc_fp4_job* J = (orc_fp4_job*)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int b = J->next_request++;
        pthread_mutex_unlock(&J->lock);
        if (b >= J->batch) break;
        orc_fp4_request(J, b);
    }
    return NULL;
}

/* MXFP4 logits out[(b*next_n + t) * out_stride + p] = sum_h w[t,h] *
 * relu(q[t,h] . k_p) over dequantised values, for every request with
 * seq_lens[b] > 0, every slot t < next_n and every p < min(seq_lens[b],
 * max_context); nothing else in out is touched.  mag (optional) receives
 * sum_h |w[t,h]| * |q[t,h] . k_p|.  Returns 0, or -1 on bad arguments. */
int orc_fp4_paged_mqa_logits(const uint8_t* q, const uint8_t* q_sf, const uint8_t* kv,
                             int64_t num_blocks, const float* weights, const int32_t* seq_lens,
                             const int32_t* block_table, int64_t bt_stride, int batch, int next_n,
                             double* out, double* mag, int64_t out_stride, int max_context,
                             int nthreads)
{
    if (!q || !q_sf || !kv || !weights || !seq_lens || !block_table || !out) return -1;
    if (next_n < 1 || batch < 0) return -1;
    orc_fp4_job J;
    memset(&J, 0, sizeof J);
    J.q = q; J.q_sf = q_sf; J.kv = kv; J.num_blocks = num_blocks; J.weights = weights;
    J.seq_lens = seq_lens; J.block_table = block_table; J.bt_stride = bt_stride;
    J.batch = batch; J.next_n = next_n; J.out = out; J.mag = mag;
    J.out_stride = out_stride; J.max_context = max_context;
    pthread_mutex_init(&J.lock, NULL);
    orc_run_threads(orc_fp4_worker, &J, nthreads);
    pthread_mutex_destroy(&J.lock);
    return 0;
}
