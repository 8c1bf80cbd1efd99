/*
 * Oracle for paged decode attention, cache write and block copy.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the package smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library: it is a plain, slow, fp64 restatement of what the pages
 * define, written so that it can be checked against them by eye.
 *
 * Sources (page title, section):
 *  - "KV cache: la memoria de trabajo que sostiene la inferencia LLM",
 *    "El mecanismo en sí (en cristiano)": the new token's query is multiplied
 *    against the keys of all previous tokens, normalised with a softmax, and
 *    the values are weighted by it.
 *  - "Cómo funciona realmente vLLM (y por qué lo necesitas)", "PagedAttention: la paginación del
 *    sistema operativo aplicada a la GPU": paging changes only how the K/V of
 *    a sequence are addressed, never the attention arithmetic.
 *  - "PagedAttention por dentro", "El modelo de bloques" and "La tabla de
 *    páginas (block table)": a block holds K and V of 16 consecutive tokens of
 *    one sequence; token t of a sequence lives in the physical block listed at
 *    position floor(t / 16) of the sequence's block table.
 *  - same page, "La tabla de páginas (block table)": a new token is written into the slot
 *    of its block (cache write).
 *  - same page, "Copy-on-write para sampling paralelo": on divergence only the
 *    last shared block is copied (block copy).
 *  - "PagedAttention por dentro", "Sliding window attention": a model with a
 *    window of W tokens attends only to the last W tokens of its context.
 *  - "KV cache: la memoria de trabajo que sostiene la inferencia LLM", "Trucos para que el cuaderno sea más fino":
 *    under GQA query heads share K/V in groups; query head h reads KV head
 *    floor(h / (Hq / Hkv)).
 *
 * Layout (the pages do not fix one; this is the library's documented layout):
 *   key_cache / value_cache : [num_blocks][num_kv_heads][block_size][head_dim]
 *   query                   : [num_seqs][num_q_heads][head_dim]
 *   block_tables            : int32 [num_seqs][max_blocks]
 *   context_lens            : int32 [num_seqs]
 *   slot_mapping            : int64 [num_tokens], slot = block * block_size + offset,
 *                             a negative slot means "no write"
 * Element types: dtype 0 = float32, dtype 1 = bfloat16 (raw 16-bit patterns),
 * dtype 2 = FP8 E4M3 codes (K/V pools only, each KV head with its own scale:
 * the stored value is code_value * scale[kv_head]).  The pages name FP8
 * caches ("KV cache: la memoria de trabajo que sostiene la inferencia LLM",
 * "Trucos para que el cuaderno sea más fino": quantising the cache to FP8
 * halves it); the format itself is the E4M3 ("E4M3FN") encoding of the OCP
 * 8-bit floating point specification.
 * Every element is widened exactly to double before any arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PAO_OK 0
#define PAO_ERR_ARG 1
#define PAO_ERR_INDEX 2
#define PAO_ERR_NOMEM 3

/* Value of an E4M3 code: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits; exponent field 0 holds subnormals (m * 2^-9); S.1111.111 is NaN; there
 * are no infinities (the largest finite value is 1.75 * 2^8 = 448). */
double pao_e4m3_value(uint8_t code)
{
    const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Nearest integer to y >= 0, halfway cases to the even integer. */
static double round_half_even(double y)
{
    double fl = floor(y);
    double diff = y - fl;
    if (diff > 0.5)
        return fl + 1.0;
    if (diff < 0.5)
        return fl;
    return fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
}

/* E4M3 code of a float: the nearest E4M3 value (ties to an even mantissa);
 * magnitudes of 448 or more give +-448 (saturation); NaN gives 0x7F. */
uint8_t pao_e4m3_encode(float x)
{
    if (x != x)
        return 0x7F;
    const int sign = signbit(x) ? 1 : 0;
    const double a = fabs((double)x);
    uint8_t mag;
    if (a >= 448.0) {
        mag = 0x7E;
    } else if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9 (8 of them reach the smallest normal) */
        const int n = (int)round_half_even(a * 512.0);
        mag = (uint8_t)(n == 8 ? (1 << 3) : n);
    } else {
        int e2;
        (void)frexp(a, &e2);              /* a = f * 2^e2, f in [0.5, 1) */
        int E = e2 - 1;                   /* a in [2^E, 2^(E+1)) */
        int n = (int)round_half_even(a / ldexp(1.0, E - 3));   /* 8 .. 16 */
        if (n == 16) {
            E += 1;
            n = 8;
        }
        mag = (uint8_t)(((E + 7) << 3) | (n - 8));
    }
    return (uint8_t)((sign << 7) | mag);
}

/* Widen one stored element to double.  bfloat16 is the upper half of an IEEE
 * binary32, so shifting its 16 bits up by 16 gives the float exactly. */
static double widen(const void *base, int64_t idx, int dtype)
{
    if (dtype == 0) {
        return (double)((const float *)base)[idx];
    } else if (dtype == 1) {
        uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    } else {
        return pao_e4m3_value(((const uint8_t *)base)[idx]);
    }
}

/* Attention of one query row over positions [first, last) of sequence b's
 * paged context (KV head kvh).  Two passes over the scores (maximum, then
 * normalised weights), exactly the textbook softmax(q K^T * scale) V with the
 * K/V rows gathered through the block table in logical token order.  The
 * query row starts at element qbase of `query`. */
static int attend_span(double *out, const void *query, int64_t qbase, int q_dtype,
                       const void *key_cache, const void *value_cache, int kv_dtype,
                       const float *k_scales, const float *v_scales,
                       const int32_t *block_tables, int b, int kvh, int first, int last,
                       int num_kv_heads, int head_dim, int block_size, int max_blocks,
                       int num_blocks, double scale)
{
    int d, t;

    for (d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    if (last <= first)
        return PAO_OK;
    if (first < 0 || (int64_t)last > (int64_t)max_blocks * block_size)
        return PAO_ERR_INDEX;

    double *score = (double *)malloc(sizeof(double) * (size_t)last);
    int64_t *row = (int64_t *)malloc(sizeof(int64_t) * (size_t)last);
    if (!score || !row) {
        free(score);
        free(row);
        return PAO_ERR_NOMEM;
    }

    /* Gather: logical token t -> (physical block, offset inside it). */
    for (t = first; t < last; ++t) {
        int logical_block = t / block_size;
        int offset = t % block_size;
        int32_t phys = block_tables[(int64_t)b * max_blocks + logical_block];
        if (phys < 0 || phys >= num_blocks) {
            free(score);
            free(row);
            return PAO_ERR_INDEX;
        }
        row[t] = (((int64_t)phys * num_kv_heads + kvh) * block_size + offset) * head_dim;
    }

    /* Stored K/V values are code_value * per-head scale for FP8 pools. */
    const double ks = k_scales ? (double)k_scales[kvh] : 1.0;
    const double vs = v_scales ? (double)v_scales[kvh] : 1.0;

    /* Scores s_t = scale * <q, k_t>. */
    for (t = first; t < last; ++t) {
        double dot = 0.0;
        for (d = 0; d < head_dim; ++d)
            dot += widen(query, qbase + d, q_dtype) * (widen(key_cache, row[t] + d, kv_dtype) * ks);
        score[t] = scale * dot;
    }

    /* Softmax: subtract the maximum, exponentiate, normalise. */
    double mx = score[first];
    for (t = first + 1; t < last; ++t)
        if (score[t] > mx)
            mx = score[t];
    double denom = 0.0;
    for (t = first; t < last; ++t)
        denom += exp(score[t] - mx);

    /* Output: the softmax-weighted sum of the value rows. */
    for (t = first; t < last; ++t) {
        double w = exp(score[t] - mx) / denom;
        for (d = 0; d < head_dim; ++d)
            out[d] += w * (widen(value_cache, row[t] + d, kv_dtype) * vs);
    }

    free(score);
    free(row);
    return PAO_OK;
}

/* Decode: query head h of sequence b attends to its whole context [0, L), or
 * with a window of W tokens to [L - W, L). */
static int attend_one(double *out, const void *query, int q_dtype, const void *key_cache,
                      const void *value_cache, int kv_dtype, const float *k_scales,
                      const float *v_scales, const int32_t *block_tables,
                      const int32_t *context_lens, int b, int h, int num_q_heads,
                      int num_kv_heads, int head_dim, int block_size, int max_blocks,
                      int num_blocks, double scale, int window)
{
    const int group = num_q_heads / num_kv_heads;
    const int L = context_lens[b];
    if (L < 0 || (int64_t)L > (int64_t)max_blocks * block_size)
        return PAO_ERR_INDEX;
    /* With a window of W tokens only positions [L - W, L) take part. */
    const int first = (window > 0 && L > window) ? L - window : 0;
    const int64_t qbase = ((int64_t)b * num_q_heads + h) * head_dim;
    return attend_span(out, query, qbase, q_dtype, key_cache, value_cache, kv_dtype, k_scales,
                       v_scales, block_tables, b, h / group, first, L, num_kv_heads, head_dim,
                       block_size, max_blocks, num_blocks, scale);
}

/*
 * Paged decode attention.
 *   out : double; [num_seqs][num_q_heads][head_dim] when sel == NULL,
 *         otherwise [n_sel][head_dim] for the (b, h) pairs listed in sel
 *         (sel holds 2 * n_sel int32 values: b0, h0, b1, h1, ...).
 *   q_dtype, kv_dtype : element types of the query and of the pools; for
 *         FP8 pools k_scales / v_scales hold one scale per KV head (NULL = 1).
 *   window : 0 = the whole context; W > 0 = only the last W tokens.
 *   num_threads : OpenMP threads over (b, h) pairs; 1 = serial.
 * Returns 0, or a nonzero code for bad arguments or an out-of-range table
 * entry (the oracle never reads outside the pools).
 */
int pao_paged_decode_ex(double *out, const void *query, int q_dtype, const void *key_cache,
                        const void *value_cache, int kv_dtype, const float *k_scales,
                        const float *v_scales, const int32_t *block_tables,
                        const int32_t *context_lens, int num_seqs, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, int max_blocks,
                        int num_blocks, double scale, const int32_t *sel, int n_sel,
                        int num_threads, int window)
{
    if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens)
        return PAO_ERR_ARG;
    if (q_dtype < 0 || q_dtype > 1 || kv_dtype < 0 || kv_dtype > 2)
        return PAO_ERR_ARG;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks < 0 || num_blocks < 0)
        return PAO_ERR_ARG;
    if (num_q_heads % num_kv_heads != 0)
        return PAO_ERR_ARG;

    const int64_t n_pairs = sel ? (int64_t)n_sel : (int64_t)num_seqs * num_q_heads;
    int status = PAO_OK;
    int64_t i;
    (void)num_threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads > 0 ? num_threads : 1)
#endif
    for (i = 0; i < n_pairs; ++i) {
        int b, h;
        if (sel) {
            b = sel[2 * i];
            h = sel[2 * i + 1];
        } else {
            b = (int)(i / num_q_heads);
            h = (int)(i % num_q_heads);
        }
        int rc;
        if (b < 0 || b >= num_seqs || h < 0 || h >= num_q_heads)
            rc = PAO_ERR_ARG;
        else
            rc = attend_one(out + i * head_dim, query, q_dtype, key_cache, value_cache, kv_dtype,
                            k_scales, v_scales, block_tables, context_lens, b, h, num_q_heads,
                            num_kv_heads, head_dim, block_size, max_blocks, num_blocks, scale,
                            window);
        if (rc != PAO_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
            status = rc;
        }
    }
    return status;
}

/* Paged decode attention with query and pools of one element type (0 or 1). */
int pao_paged_decode(double *out, const void *query, const void *key_cache,
                     const void *value_cache, int dtype,
                     const int32_t *block_tables, const int32_t *context_lens,
                     int num_seqs, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, int max_blocks,
                     int num_blocks, double scale, const int32_t *sel,
                     int n_sel, int num_threads)
{
    if (dtype != 0 && dtype != 1)
        return PAO_ERR_ARG;
    return pao_paged_decode_ex(out, query, dtype, key_cache, value_cache, dtype, NULL, NULL,
                               block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                               head_dim, block_size, max_blocks, num_blocks, scale, sel, n_sel,
                               num_threads, 0);
}

/*
 * Cache write: each new token i whose slot s_i is not negative has its K and V
 * rows (all KV heads) copied into offset s_i % block_size of physical block
 * s_i / block_size.  key / value are [num_tokens][num_kv_heads][head_dim].
 * Tokens are applied in index order.
 */
int pao_cache_write(void *key_cache, void *value_cache, const void *key,
                    const void *value, const int64_t *slot_mapping,
                    int num_tokens, int num_kv_heads, int head_dim,
                    int block_size, int num_blocks, int elem_bytes)
{
    if (!key_cache || !value_cache || !key || !value || (!slot_mapping && num_tokens > 0))
        return PAO_ERR_ARG;
    const int64_t row_bytes = (int64_t)head_dim * elem_bytes;
    int i, kvh;
    for (i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0)
            continue;
        if (s >= (int64_t)num_blocks * block_size)
            return PAO_ERR_INDEX;
        int64_t blk = s / block_size;
        int64_t off = s % block_size;
        for (kvh = 0; kvh < num_kv_heads; ++kvh) {
            int64_t dst = ((blk * num_kv_heads + kvh) * block_size + off) * row_bytes;
            int64_t src = ((int64_t)i * num_kv_heads + kvh) * row_bytes;
            memcpy((char *)key_cache + dst, (const char *)key + src, (size_t)row_bytes);
            memcpy((char *)value_cache + dst, (const char *)value + src, (size_t)row_bytes);
        }
    }
    return PAO_OK;
}

/*
 * Cache write into FP8 pools: every element x of a new token's bfloat16 K (V)
 * row is quantised to the E4M3 code of the float32 quotient x / scale[kv_head]
 * (IEEE single-precision division, then pao_e4m3_encode) and stored at the
 * token's slot, as pao_cache_write does for unquantised rows.
 */
int pao_cache_write_fp8(uint8_t *key_cache, uint8_t *value_cache, const uint16_t *key,
                        const uint16_t *value, const int64_t *slot_mapping, int num_tokens,
                        int num_kv_heads, int head_dim, int block_size, int num_blocks,
                        const float *k_scales, const float *v_scales)
{
    if (!key_cache || !value_cache || !key || !value || !k_scales || !v_scales ||
        (!slot_mapping && num_tokens > 0))
        return PAO_ERR_ARG;
    int i, kvh, d;
    for (i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0)
            continue;
        if (s >= (int64_t)num_blocks * block_size)
            return PAO_ERR_INDEX;
        int64_t blk = s / block_size;
        int64_t off = s % block_size;
        for (kvh = 0; kvh < num_kv_heads; ++kvh) {
            int64_t dst = ((blk * num_kv_heads + kvh) * block_size + off) * head_dim;
            int64_t src = ((int64_t)i * num_kv_heads + kvh) * head_dim;
            for (d = 0; d < head_dim; ++d) {
                float kx = (float)widen(key, src + d, 1);
                float vx = (float)widen(value, src + d, 1);
                float kq = kx / k_scales[kvh];
                float vq = vx / v_scales[kvh];
                key_cache[dst + d] = pao_e4m3_encode(kq);
                value_cache[dst + d] = pao_e4m3_encode(vq);
            }
        }
    }
    return PAO_OK;
}

/*
 * Block copy (copy-on-write), "PagedAttention por dentro", "Copy-on-write para
 * sampling paralelo": a sequence about to write into a block it shares gets a
 * copy of that one block in a block taken from the pool, and only the copy
 * changes.  Each pair (src, dst) of the list is one such copy: the whole
 * physical block dst of both pools becomes block src as it was before the
 * call.  Since every copy on the pages goes into a freshly taken block, no copy
 * of a list writes a block that another copy of the same list reads or
 * writes; a list is read that way, pair by pair:
 *   - a pair with an index outside [0, num_blocks) is skipped;
 *   - a pair with src == dst changes nothing (it is not "live");
 *   - a live pair whose dst is the src or the dst of another live pair is
 *     skipped (it would overwrite what the other reads, or what it writes);
 *   - every other live pair is copied.
 * The copied pairs then touch disjoint destinations that no copied pair
 * reads, so copying them one after another in list order gives the same
 * pools as copying them all at once from the pools before the call.
 * *skipped receives 1 when some pair was skipped, else 0.
 * pairs holds 2 * num_pairs int32 values: src0, dst0, src1, dst1, ...
 */
int pao_block_copy(void *key_cache, void *value_cache, const int32_t *pairs,
                   int num_pairs, int num_kv_heads, int head_dim,
                   int block_size, int num_blocks, int elem_bytes, int *skipped)
{
    if (!key_cache || !value_cache || !skipped || (!pairs && num_pairs > 0) || num_pairs < 0)
        return PAO_ERR_ARG;
    const int64_t block_bytes = (int64_t)num_kv_heads * block_size * head_dim * elem_bytes;
    char *live = (char *)calloc((size_t)num_pairs + 1, 1);
    if (!live)
        return PAO_ERR_NOMEM;
    *skipped = 0;
    int p, q;
    for (p = 0; p < num_pairs; ++p) {
        int32_t src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            *skipped = 1;
            continue;
        }
        live[p] = src != dst;
    }
    for (p = 0; p < num_pairs; ++p) {
        if (!live[p])
            continue;
        int32_t src = pairs[2 * p], dst = pairs[2 * p + 1];
        int clash = 0;
        for (q = 0; q < num_pairs; ++q)
            if (q != p && live[q] && (pairs[2 * q] == dst || pairs[2 * q + 1] == dst))
                clash = 1;
        if (clash) {
            *skipped = 1;
            continue;
        }
        memcpy((char *)key_cache + dst * block_bytes, (const char *)key_cache + src * block_bytes,
               (size_t)block_bytes);
        memcpy((char *)value_cache + dst * block_bytes,
               (const char *)value_cache + src * block_bytes, (size_t)block_bytes);
    }
    free(live);
    return PAO_OK;
}

/* Threads OpenMP would use by default (1 when built without OpenMP). */
int pao_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Chunked (paged) prefill ("PagedAttention por dentro", section "Chunked
 * prefill integrado con paged KV": prefill is cut into chunks that run over
 * the same paged KV cache as decode).  Sequence b brings a chunk of
 * T_b = query_start[b+1] - query_start[b] new tokens whose K/V are already in
 * the pools; its context then holds L_b = context_lens[b] tokens, the chunk
 * being the last T_b of them.  Query row i of the chunk sits at position
 * p = L_b - T_b + i and attends causally ("KV cache: la memoria de trabajo",
 * "El mecanismo en sí (en cristiano)": a token looks at itself and the tokens
 * before it) to positions [0, p], or with a window of W tokens to
 * [p + 1 - W, p].
 *   query : [total_tokens][num_q_heads][head_dim], row query_start[b] + i for
 *           token i of sequence b; out likewise, in double.
 *   query_start : int32 [num_seqs + 1], non-decreasing, query_start[0] = 0.
 */
int pao_paged_prefill(double *out, const void *query, int q_dtype, const void *key_cache,
                      const void *value_cache, int kv_dtype, const float *k_scales,
                      const float *v_scales, const int32_t *block_tables,
                      const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      int max_blocks, int num_blocks, double scale, int window, int num_threads)
{
    if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens ||
        !query_start)
        return PAO_ERR_ARG;
    if (q_dtype < 0 || q_dtype > 1 || kv_dtype < 0 || kv_dtype > 2)
        return PAO_ERR_ARG;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks < 0 || num_blocks < 0 || window < 0)
        return PAO_ERR_ARG;
    if (num_q_heads % num_kv_heads != 0 || query_start[0] != 0)
        return PAO_ERR_ARG;
    int b;
    for (b = 0; b < num_seqs; ++b) {
        const int T = query_start[b + 1] - query_start[b];
        if (T < 0 || T > context_lens[b])
            return PAO_ERR_ARG;
    }
    const int group = num_q_heads / num_kv_heads;
    const int64_t rows = (int64_t)query_start[num_seqs] * num_q_heads;
    int status = PAO_OK;
    int64_t r;
    (void)num_threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 16) num_threads(num_threads > 0 ? num_threads : 1)
#endif
    for (r = 0; r < rows; ++r) {
        const int64_t tok = r / num_q_heads;
        const int h = (int)(r % num_q_heads);
        int sb = 0;
        while (query_start[sb + 1] <= tok)   /* the sequence that owns this token */
            ++sb;
        const int T = query_start[sb + 1] - query_start[sb];
        const int L = context_lens[sb];
        const int p = L - T + (int)(tok - query_start[sb]);
        const int first = (window > 0 && p + 1 > window) ? p + 1 - window : 0;
        int rc = attend_span(out + r * head_dim, query, r * head_dim, q_dtype, key_cache,
                             value_cache, kv_dtype, k_scales, v_scales, block_tables, sb,
                             h / group, first, p + 1, num_kv_heads, head_dim, block_size,
                             max_blocks, num_blocks, scale);
        if (rc != PAO_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
            status = rc;
        }
    }
    return status;
}
