/*
 * pkv_oracle.c -- CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the paged decode-attention path computes.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.  It
 * shares no code, header, table or constant with the CUDA library and the
 * product path never calls it.
 *
 * Arithmetic is IEEE fp64 over the exact values of the bf16 inputs.  Nothing
 * is blocked, fused or reordered beyond the definition:
 *
 *   Attention(Q, K, V) = softmax((Q K^T / sqrt(d_k)) + causal_mask) V
 *     -- "Transformer inference mechanics", What Q, K, and V do in causal
 *        attention (per-head decoder attention and the causal mask);
 *        "Transformer and attention intuition", Q, K, V -- and why they force
 *        a cache.
 *
 * The KV cache holds K[1..t], V[1..t] per layer and gains the new token's K/V
 * each step ("Transformer inference mechanics", What the KV cache stores per
 * layer).  It is stored in fixed-size blocks reached through a per-request
 * block table that maps logical positions to physical blocks ("Inference
 * Engines", The Breakthrough, PagedAttention paragraph; CS336 lecture-10
 * notes, PagedAttention (vLLM)).  Query heads share K/V heads in contiguous
 * groups (GQA; MQA is one group, MHA one head per group) ("Transformer
 * inference mechanics", MHA versus MQA versus GQA).
 *
 * Readings where the pages leave a detail open (each is also listed with the
 * design notes):
 *   - cache layout [num_blocks][n_kv][block_size][head_dim];
 *   - query head h reads KV head h / (n_q / n_kv);
 *   - context_lens[b] counts every resident token including the q_len new
 *     ones, and new token i sits at position ctx - q_len + i, seeing keys at
 *     positions <= its own (the causal mask);
 *   - a row that sees no key (ctx == 0, or ctx < q_len) outputs zeros;
 *   - sliding window W > 0: the query at position pos sees only positions
 *     pos - W + 1 .. pos (its own and the W - 1 before it; CS336 lecture-10
 *     notes, Local attention & sparse variants); W = 0 means no window;
 *   - the softmax is evaluated as max, then sum of exp(s - max): subtracting
 *     the row maximum leaves softmax unchanged and keeps exp finite;
 *   - an 8-bit KV cache ("Efficient inference", Quantization: fewer bytes per
 *     weight -- the KV cache may be stored in low precision, dequantised
 *     through a scale; CS336 lecture-10 notes, Quantization & pruning:
 *     bf16 -> fp8) holds e4m3 codes with one scale per KV head for K and one
 *     for V: the cached value is code_value * scale.  Its layout is
 *     [num_blocks][n_kv][2][block_size][head_dim]: for every (block, KV
 *     head) the K rows, then the V rows;  A new value x is stored
 *     as the e4m3 code nearest to x / scale, the division taken in fp32 and
 *     ties going to the even code; quotients beyond the largest finite e4m3
 *     (448) store +-448;
 *   - the same 8-bit cache may instead carry one scale per (block, KV head)
 *     for K and one for V, kept in [num_blocks][n_kv][4] fp32 (K scale, V
 *     scale, two reserved words), so that a scale follows the values of its
 *     own block.  The appending side sets them as written out at
 *     oracle_kv_append_fp8_block.
 *
 * Parallelism: one OpenMP loop over independent (sequence, KV head) units.
 * Each unit is computed by one thread, start to finish, in sequential order,
 * so the result does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening: a bf16 is the top 16 bits of an fp32. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * e4m3 (the 8-bit float of the OCP FP8 format, E4M3 variant): sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits.  Exponent field 0 holds the
 * subnormals m/8 * 2^-6; S.1111.111 is NaN; there is no infinity, so the
 * largest finite magnitude is 1.75 * 2^8 = 448.
 */
static double e4m3_value(uint8_t code)
{
    const int e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7)
        return NAN;
    const double mag = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return (code & 0x80) ? -mag : mag;
}

/*
 * The e4m3 code nearest to x, ties to the even code, magnitudes that would
 * round past 448 (infinities included) saturating to 448, NaN to 0x7F.  Codes grow with magnitude
 * one ulp at a time (code 8 = 2^-6 follows subnormal 7/8 * 2^-6), so with
 * 2^e <= |x| < 2^(e+1) the code is 8(e + 7) + rint(|x| / 2^(e-3)) - 8, and
 * below 2^-6 it is rint(|x| * 2^9); rint rounds half to even.
 */
static uint8_t e4m3_code(float x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    long code;
    if (a >= 448.0) {
        code = 0x7E; /* the largest finite code, for infinities too */
    } else if (a < ldexp(1.0, -6)) {
        code = (long)rint(ldexp(a, 9));
    } else {
        int e2;
        (void)frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1): 2^(e2-1) <= a < 2^e2 */
        const int e = e2 - 1;
        code = 8L * (e + 7) + (long)rint(ldexp(a, 3 - e)) - 8;
    }
    return (uint8_t)(sign | code); /* below 448 the code is at most 0x7E */
}

void oracle_e4m3_encode(const float *x, long n, uint8_t *codes)
{
    for (long i = 0; i < n; ++i)
        codes[i] = e4m3_code(x[i]);
}

void oracle_e4m3_decode(const uint8_t *codes, long n, double *x)
{
    for (long i = 0; i < n; ++i)
        x[i] = e4m3_value(codes[i]);
}

/*
 * A KV cache as the attention reads it: bf16 bit patterns in separate K and V
 * caches [num_blocks][n_kv][block_size][head_dim], or e4m3 codes in one cache
 * [num_blocks][n_kv][2][block_size][head_dim] (K rows, then V rows) with one
 * dequantisation scale per KV head (k_scale[g], v_scale[g]).
 */
typedef struct {
    const uint16_t *k16, *v16; /* bf16 caches, or NULL */
    const uint8_t *kv8;        /* e4m3 cache, or NULL */
    const float *k_scale, *v_scale;
    const float *blk_scales;   /* e4m3 cache with per-(block, head) scales, or NULL */
} cache_view;

/*
 * Copy sequence b's logical keys and values for KV head g into dense
 * K[ctx][d], V[ctx][d] by walking its block table: logical token t lives in
 * physical block block_tables[b][t / block_size] at offset t % block_size.
 * Returns 0, or -1 if a block index the walk needs is outside [0, num_blocks).
 */
static int gather_sequence(const cache_view *c, const int32_t *table_row, int ctx, int g,
                           int n_kv, int head_dim, int block_size, int num_blocks,
                           double *K, double *V)
{
    for (int t = 0; t < ctx; ++t) {
        int blk = table_row[t / block_size];
        int off = t % block_size;
        if (blk < 0 || blk >= num_blocks)
            return -1;
        size_t base = (((size_t)blk * n_kv + g) * block_size + off) * head_dim;
        /* e4m3: K row of (blk, g, off) and the V row block_size rows after it */
        size_t kbase8 = ((((size_t)blk * n_kv + g) * 2) * block_size + off) * head_dim;
        size_t vbase8 = kbase8 + (size_t)block_size * head_dim;
        /* the scales of this token's values: its physical block's, or its head's */
        const double ks = c->blk_scales ? (double)c->blk_scales[((size_t)blk * n_kv + g) * 4 + 0]
                          : c->kv8      ? (double)c->k_scale[g] : 0.0;
        const double vs = c->blk_scales ? (double)c->blk_scales[((size_t)blk * n_kv + g) * 4 + 1]
                          : c->kv8      ? (double)c->v_scale[g] : 0.0;
        for (int e = 0; e < head_dim; ++e) {
            if (c->kv8) {
                K[(size_t)t * head_dim + e] = e4m3_value(c->kv8[kbase8 + e]) * ks;
                V[(size_t)t * head_dim + e] = e4m3_value(c->kv8[vbase8 + e]) * vs;
            } else {
                K[(size_t)t * head_dim + e] = bf16_value(c->k16[base + e]);
                V[(size_t)t * head_dim + e] = bf16_value(c->v16[base + e]);
            }
        }
    }
    return 0;
}

/*
 * out[b][i][h][:] for all b, query tokens i, query heads h (fp64).
 * q: [num_seqs][q_len][n_q][head_dim] bf16 bits.  window: 0 for full causal
 * attention, W > 0 for a sliding window of W positions.  Returns 0 on
 * success, 1 on bad shape arguments, 2 if a block table or context length is
 * invalid.
 */
static int paged_attn(const uint16_t *q, const cache_view *cache,
                      const int32_t *block_tables, const int32_t *context_lens,
                      int num_seqs, int q_len, int n_q, int n_kv, int head_dim,
                      int block_size, int max_blocks_per_seq, int num_blocks,
                      double scale, int window, double *out)
{
    if (num_seqs < 0 || q_len < 1 || n_q < 1 || n_kv < 1 || n_q % n_kv != 0 ||
        head_dim < 1 || block_size < 1 || max_blocks_per_seq < 0 || num_blocks < 0 ||
        window < 0)
        return 1;
    const int G = n_q / n_kv;
    int status = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (long unit = 0; unit < (long)num_seqs * n_kv; ++unit) {
        const int b = (int)(unit / n_kv);
        const int g = (int)(unit % n_kv);
        const int ctx = context_lens[b];
        if (ctx < 0 || (long)ctx > (long)max_blocks_per_seq * block_size) {
#pragma omp atomic write
            status = 2;
            continue;
        }
        double *K = (double *)malloc(sizeof(double) * ((size_t)ctx * head_dim + 1));
        double *V = (double *)malloc(sizeof(double) * ((size_t)ctx * head_dim + 1));
        double *s = (double *)malloc(sizeof(double) * ((size_t)ctx + 1));
        double *acc = (double *)malloc(sizeof(double) * (size_t)head_dim);
        if (gather_sequence(cache, block_tables + (size_t)b * max_blocks_per_seq, ctx, g,
                            n_kv, head_dim, block_size, num_blocks, K, V) != 0) {
#pragma omp atomic write
            status = 2;
        } else {
            for (int i = 0; i < q_len; ++i) {
                /* New token i sits at position ctx - q_len + i and sees keys
                 * first..pos (first = 0, or pos - window + 1 with a window). */
                const long pos = (long)ctx - q_len + i;
                const int nvis = pos < 0 ? 0 : (int)(pos + 1 < ctx ? pos + 1 : ctx);
                const long first_l = window > 0 ? pos - window + 1 : 0;
                const int first = first_l < 0 ? 0 : (int)first_l;
                for (int h = g * G; h < (g + 1) * G; ++h) {
                    const uint16_t *qrow = q + (((size_t)b * q_len + i) * n_q + h) * head_dim;
                    double *orow = out + (((size_t)b * q_len + i) * n_q + h) * head_dim;
                    for (int e = 0; e < head_dim; ++e)
                        acc[e] = 0.0;
                    if (nvis <= first) {
                        for (int e = 0; e < head_dim; ++e)
                            orow[e] = 0.0;
                        continue;
                    }
                    /* scores s_t = scale * q . K_t */
                    double mx = -INFINITY;
                    for (int t = first; t < nvis; ++t) {
                        double dot = 0.0;
                        for (int e = 0; e < head_dim; ++e)
                            dot += bf16_value(qrow[e]) * K[(size_t)t * head_dim + e];
                        s[t] = scale * dot;
                        if (s[t] > mx)
                            mx = s[t];
                    }
                    /* softmax weights and the weighted sum of values */
                    double denom = 0.0;
                    for (int t = first; t < nvis; ++t) {
                        double w = exp(s[t] - mx);
                        denom += w;
                        for (int e = 0; e < head_dim; ++e)
                            acc[e] += w * V[(size_t)t * head_dim + e];
                    }
                    for (int e = 0; e < head_dim; ++e)
                        orow[e] = acc[e] / denom;
                }
            }
        }
        free(K);
        free(V);
        free(s);
        free(acc);
    }
    return status;
}

int oracle_paged_attn(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                      const int32_t *block_tables, const int32_t *context_lens,
                      int num_seqs, int q_len, int n_q, int n_kv, int head_dim,
                      int block_size, int max_blocks_per_seq, int num_blocks,
                      double scale, int window, double *out)
{
    const cache_view c = {k_cache, v_cache, NULL, NULL, NULL, NULL};
    return paged_attn(q, &c, block_tables, context_lens, num_seqs, q_len, n_q, n_kv, head_dim,
                      block_size, max_blocks_per_seq, num_blocks, scale, window, out);
}

/* The same attention over an e4m3 cache: K_t = code * k_scale[g], V_t = code * v_scale[g]. */
int oracle_paged_attn_fp8(const uint16_t *q, const uint8_t *kv_cache,
                          const float *k_scale, const float *v_scale,
                          const int32_t *block_tables, const int32_t *context_lens,
                          int num_seqs, int q_len, int n_q, int n_kv, int head_dim,
                          int block_size, int max_blocks_per_seq, int num_blocks,
                          double scale, int window, double *out)
{
    const cache_view c = {NULL, NULL, kv_cache, k_scale, v_scale, NULL};
    return paged_attn(q, &c, block_tables, context_lens, num_seqs, q_len, n_q, n_kv, head_dim,
                      block_size, max_blocks_per_seq, num_blocks, scale, window, out);
}

/*
 * The same attention over an e4m3 cache with one scale per (physical block,
 * KV head): token t of sequence b in KV head g decodes as code * s, s the K
 * (or V) scale of kv_scales[block_tables[b][t / block_size]][g].
 */
int oracle_paged_attn_fp8_block(const uint16_t *q, const uint8_t *kv_cache,
                                const float *kv_scales, const int32_t *block_tables,
                                const int32_t *context_lens, int num_seqs, int q_len, int n_q,
                                int n_kv, int head_dim, int block_size, int max_blocks_per_seq,
                                int num_blocks, double scale, int window, double *out)
{
    const cache_view c = {NULL, NULL, kv_cache, NULL, NULL, kv_scales};
    return paged_attn(q, &c, block_tables, context_lens, num_seqs, q_len, n_q, n_kv, head_dim,
                      block_size, max_blocks_per_seq, num_blocks, scale, window, out);
}

/*
 * Attention of one query row restricted to the logical key range
 * [t_begin, t_end) (further cut by the causal limit), returned as the three
 * quantities that FlashAttention's online softmax keeps per row: the running
 * maximum m, the running sum l = sum_t exp(s_t - m) and the unnormalised
 * output o = sum_t exp(s_t - m) V_t.  An empty range gives m = -inf, l = 0,
 * o = 0.  ("Efficient inference", FlashAttention: exact attention without
 * the matrix -- partial results from different key blocks are rescaled and
 * combined exactly; CS336 lecture-10 notes, PagedAttention (vLLM), where
 * FlashDecoding splits the context.)
 * Output rows are laid out like the full output: [num_seqs][q_len][n_q].
 */
int oracle_attn_partial(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_tables, const int32_t *context_lens,
                        int num_seqs, int q_len, int n_q, int n_kv, int head_dim,
                        int block_size, int max_blocks_per_seq, int num_blocks,
                        double scale, int t_begin, int t_end,
                        double *o, double *m, double *l)
{
    if (num_seqs < 0 || q_len < 1 || n_q < 1 || n_kv < 1 || n_q % n_kv != 0 ||
        head_dim < 1 || block_size < 1 || t_begin < 0 || t_end < t_begin)
        return 1;
    const int G = n_q / n_kv;
    for (int b = 0; b < num_seqs; ++b) {
        const int ctx = context_lens[b];
        if (ctx < 0 || (long)ctx > (long)max_blocks_per_seq * block_size)
            return 2;
        for (int i = 0; i < q_len; ++i) {
            const long pos = (long)ctx - q_len + i;
            long hi = pos + 1 < ctx ? pos + 1 : ctx;
            if (hi > t_end)
                hi = t_end;
            for (int h = 0; h < n_q; ++h) {
                const int g = h / G;
                const size_t row = ((size_t)b * q_len + i) * n_q + h;
                const uint16_t *qrow = q + row * head_dim;
                double *orow = o + row * head_dim;
                for (int e = 0; e < head_dim; ++e)
                    orow[e] = 0.0;
                double mx = -INFINITY;
                for (long t = t_begin; t < hi; ++t) {
                    int blk = block_tables[(size_t)b * max_blocks_per_seq + t / block_size];
                    if (blk < 0 || blk >= num_blocks)
                        return 2;
                    size_t base = (((size_t)blk * n_kv + g) * block_size + t % block_size) * head_dim;
                    double dot = 0.0;
                    for (int e = 0; e < head_dim; ++e)
                        dot += bf16_value(qrow[e]) * bf16_value(k_cache[base + e]);
                    if (scale * dot > mx)
                        mx = scale * dot;
                }
                double sum = 0.0;
                for (long t = t_begin; t < hi; ++t) {
                    int blk = block_tables[(size_t)b * max_blocks_per_seq + t / block_size];
                    size_t base = (((size_t)blk * n_kv + g) * block_size + t % block_size) * head_dim;
                    double dot = 0.0;
                    for (int e = 0; e < head_dim; ++e)
                        dot += bf16_value(qrow[e]) * bf16_value(k_cache[base + e]);
                    double w = exp(scale * dot - mx);
                    sum += w;
                    for (int e = 0; e < head_dim; ++e)
                        orow[e] += w * bf16_value(v_cache[base + e]);
                }
                m[row] = mx;
                l[row] = sum;
            }
        }
    }
    return 0;
}

/*
 * Combine nsplit partial results of the same rows into the final output:
 * M = max_s m_s, w_s = exp(m_s - M), out = sum_s w_s o_s / sum_s w_s l_s.
 * A partial with l_s == 0 (empty range, m_s = -inf) gets weight 0; a row whose
 * partials are all empty outputs zeros.  Layouts: o [nsplit][rows][head_dim],
 * m and l [nsplit][rows], out [rows][head_dim].
 * ("Efficient inference", FlashAttention: running maximum and running sum,
 * partial results rescaled and combined exactly.)
 */
void oracle_lse_merge(int nsplit, long rows, int head_dim, const double *o,
                      const double *m, const double *l, double *out)
{
    for (long r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int s = 0; s < nsplit; ++s)
            if (l[(size_t)s * rows + r] > 0.0 && m[(size_t)s * rows + r] > M)
                M = m[(size_t)s * rows + r];
        double denom = 0.0;
        for (int e = 0; e < head_dim; ++e)
            out[(size_t)r * head_dim + e] = 0.0;
        if (M == -INFINITY)
            continue;
        for (int s = 0; s < nsplit; ++s) {
            double ls = l[(size_t)s * rows + r];
            if (ls <= 0.0)
                continue;
            double w = exp(m[(size_t)s * rows + r] - M);
            denom += w * ls;
            for (int e = 0; e < head_dim; ++e)
                out[(size_t)r * head_dim + e] += w * o[((size_t)s * rows + r) * head_dim + e];
        }
        for (int e = 0; e < head_dim; ++e)
            out[(size_t)r * head_dim + e] /= denom;
    }
}

/*
 * Write each new token's K and V rows into its cache slot: slot s names
 * physical block s / block_size, offset s % block_size.  Slots < 0 and slots
 * >= num_blocks * block_size are skipped; every other cache byte is left as
 * it was.  The copy is of the bf16 bits.  ("Transformer inference
 * mechanics", What the KV cache stores per layer: "+ new K/V for t+1";
 * "Transformer and attention intuition": the cache is appended to on every
 * decode step.)
 * k_new, v_new: [num_tokens][n_kv][head_dim]; caches: [num_blocks][n_kv][block_size][head_dim].
 */
int oracle_kv_append(const uint16_t *k_new, const uint16_t *v_new, const int32_t *slot_mapping,
                     int num_tokens, int n_kv, int head_dim, int block_size, int num_blocks,
                     uint16_t *k_cache, uint16_t *v_cache)
{
    if (num_tokens < 0 || n_kv < 1 || head_dim < 1 || block_size < 1 || num_blocks < 0)
        return 1;
    for (int i = 0; i < num_tokens; ++i) {
        long slot = slot_mapping[i];
        if (slot < 0 || slot >= (long)num_blocks * block_size)
            continue;
        long blk = slot / block_size;
        long off = slot % block_size;
        for (int g = 0; g < n_kv; ++g) {
            size_t dst = (((size_t)blk * n_kv + g) * block_size + off) * head_dim;
            size_t src = ((size_t)i * n_kv + g) * head_dim;
            memcpy(k_cache + dst, k_new + src, sizeof(uint16_t) * head_dim);
            memcpy(v_cache + dst, v_new + src, sizeof(uint16_t) * head_dim);
        }
    }
    return 0;
}

/*
 * The same append into an e4m3 cache (layout as above: K rows, then V rows
 * of each (block, KV head)): the code stored for value x of KV head g is
 * e4m3_code(x / k_scale[g]) (v_scale[g] for V), the quotient rounded to fp32
 * first -- quantise via a scale ("Efficient inference", Quantization:
 * fewer bytes per weight; CS336 lecture-10 notes, Quantization & pruning).
 */
int oracle_kv_append_fp8(const uint16_t *k_new, const uint16_t *v_new,
                         const int32_t *slot_mapping, int num_tokens, int n_kv, int head_dim,
                         int block_size, int num_blocks, const float *k_scale,
                         const float *v_scale, uint8_t *kv_cache)
{
    if (num_tokens < 0 || n_kv < 1 || head_dim < 1 || block_size < 1 || num_blocks < 0)
        return 1;
    for (int i = 0; i < num_tokens; ++i) {
        long slot = slot_mapping[i];
        if (slot < 0 || slot >= (long)num_blocks * block_size)
            continue;
        long blk = slot / block_size;
        long off = slot % block_size;
        for (int g = 0; g < n_kv; ++g) {
            size_t kdst = ((((size_t)blk * n_kv + g) * 2) * block_size + off) * head_dim;
            size_t vdst = kdst + (size_t)block_size * head_dim;
            size_t src = ((size_t)i * n_kv + g) * head_dim;
            for (int e = 0; e < head_dim; ++e) {
                const float kq = (float)bf16_value(k_new[src + e]) / k_scale[g];
                const float vq = (float)bf16_value(v_new[src + e]) / v_scale[g];
                kv_cache[kdst + e] = e4m3_code(kq);
                kv_cache[vdst + e] = e4m3_code(vq);
            }
        }
    }
    return 0;
}

/*
 * The quantising append into an e4m3 cache with per-(block, KV head) scales
 * (layouts as for oracle_paged_attn_fp8_block).  Quantise and dequantise
 * through a scale ("Efficient inference", Quantization: fewer bytes per
 * weight; CS336 lecture-10 notes, Quantization & pruning), here one scale per
 * block so that it follows the values of the block.  For every block B that
 * receives tokens in this call and every KV head, separately for K and V:
 *   - R = the call's tokens whose slots fall in B, o_min their lowest offset;
 *     the rows below o_min are the block's resident rows;
 *   - s_old = the stored scale if o_min > 0, else 0 (a block written from
 *     offset 0 starts over); scale 0 means "no value but zeros so far";
 *   - a = the largest finite |x| over R's rows (non-finite values are stored
 *     as they encode: NaN as the NaN code, infinities saturated);
 *   - s_new = s_old if a == 0, else the larger of s_old and 2^e, the smallest
 *     power of two with e >= -126 and a <= 448 * 2^e;
 *   - if s_new > s_old > 0, each resident row code c becomes
 *     E(fp32(fp32(value(c) * s_old) / s_new)) -- with powers of two exact
 *     except where the smaller value falls below the normal e4m3 range;
 *   - each token of R, in call order, writes E(fp32(x / s_new)) at its
 *     offset (E(x) itself when s_new == 0); a later token wins on a shared
 *     offset;
 *   - the scale entry becomes s_new (its two reserved words 0).
 * E is e4m3_code.  Slots outside [0, num_blocks * block_size) are skipped.
 */
int oracle_kv_append_fp8_block(const uint16_t *k_new, const uint16_t *v_new,
                               const int32_t *slot_mapping, int num_tokens, int n_kv,
                               int head_dim, int block_size, int num_blocks,
                               uint8_t *kv_cache, float *kv_scales)
{
    if (num_tokens < 0 || n_kv < 1 || head_dim < 1 || block_size < 1 || num_blocks < 0)
        return 1;
    const long nslots = (long)num_blocks * block_size;
    /* The tokens of each block, in call order: head[B] is the first, next[i] the
     * one after token i (-1 ends a list). */
    int *head = (int *)malloc(sizeof(int) * ((size_t)num_blocks + 1));
    int *tail = (int *)malloc(sizeof(int) * ((size_t)num_blocks + 1));
    int *next = (int *)malloc(sizeof(int) * ((size_t)num_tokens + 1));
    if (!head || !tail || !next) {
        free(head);
        free(tail);
        free(next);
        return 3;
    }
    for (long b = 0; b < num_blocks; ++b)
        head[b] = tail[b] = -1;
    for (int i = 0; i < num_tokens; ++i) {
        next[i] = -1;
        const long slot = slot_mapping[i];
        if (slot < 0 || slot >= nslots)
            continue;
        const long blk = slot / block_size;
        if (head[blk] < 0)
            head[blk] = i;
        else
            next[tail[blk]] = i;
        tail[blk] = i;
    }
    for (int i = 0; i < num_tokens; ++i) {
        const long slot = slot_mapping[i];
        if (slot < 0 || slot >= nslots || head[slot / block_size] != i)
            continue; /* each block once, at the first of its tokens */
        const long blk = slot / block_size;
        long o_min = block_size;
        for (int j = i; j >= 0; j = next[j])
            if (slot_mapping[j] % block_size < o_min)
                o_min = slot_mapping[j] % block_size;
        for (int g = 0; g < n_kv; ++g) {
            for (int which = 0; which < 2; ++which) { /* 0: K, 1: V */
                const uint16_t *src = which == 0 ? k_new : v_new;
                float *sc = kv_scales + ((size_t)blk * n_kv + g) * 4;
                uint8_t *rows = kv_cache +
                                (((size_t)blk * n_kv + g) * 2 + which) * (size_t)block_size * head_dim;
                const float s_old = o_min > 0 ? sc[which] : 0.0f;
                double a = 0.0;
                for (int j = i; j >= 0; j = next[j])
                    for (int e = 0; e < head_dim; ++e) {
                        const double x = bf16_value(src[((size_t)j * n_kv + g) * head_dim + e]);
                        if (isfinite(x) && fabs(x) > a)
                            a = fabs(x);
                    }
                float s_new = s_old;
                if (a > 0.0) {
                    int e = -126;
                    while (ldexp(448.0, e) < a)
                        ++e;
                    const float s_req = (float)ldexp(1.0, e);
                    if (s_req > s_new)
                        s_new = s_req;
                }
                if (s_new > s_old && s_old > 0.0f) {
                    for (long r = 0; r < o_min; ++r)
                        for (int e = 0; e < head_dim; ++e) {
                            uint8_t *cp = rows + (size_t)r * head_dim + e;
                            const float v = (float)e4m3_value(*cp) * s_old;
                            *cp = e4m3_code(v / s_new);
                        }
                }
                for (int j = i; j >= 0; j = next[j])
                    for (int e = 0; e < head_dim; ++e) {
                        const float x = (float)bf16_value(src[((size_t)j * n_kv + g) * head_dim + e]);
                        rows[(size_t)(slot_mapping[j] % block_size) * head_dim + e] =
                            e4m3_code(s_new > 0.0f ? x / s_new : x);
                    }
                sc[which] = s_new;
            }
            kv_scales[((size_t)blk * n_kv + g) * 4 + 2] = 0.0f;
            kv_scales[((size_t)blk * n_kv + g) * 4 + 3] = 0.0f;
        }
    }
    free(head);
    free(tail);
    free(next);
    return 0;
}

/*
 * Copy whole physical blocks: for each pair, block dst of both caches becomes
 * a bit copy of block src (all KV heads).  Pairs with an id outside
 * [0, num_blocks) or src == dst are skipped.  This is the copy of
 * copy-on-write block sharing (CS336 lecture-10 notes, PagedAttention (vLLM):
 * a shared block is split only when generations diverge).
 */
int oracle_copy_blocks(const int32_t *pairs, int num_pairs, int num_blocks, int n_kv,
                       int head_dim, int block_size, uint16_t *k_cache, uint16_t *v_cache)
{
    if (num_pairs < 0 || num_blocks < 0 || n_kv < 1 || head_dim < 1 || block_size < 1)
        return 1;
    const size_t per_block = (size_t)n_kv * block_size * head_dim;
    for (int p = 0; p < num_pairs; ++p) {
        const int src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks || src == dst)
            continue;
        memcpy(k_cache + (size_t)dst * per_block, k_cache + (size_t)src * per_block,
               sizeof(uint16_t) * per_block);
        memcpy(v_cache + (size_t)dst * per_block, v_cache + (size_t)src * per_block,
               sizeof(uint16_t) * per_block);
    }
    return 0;
}

/*
 * KV-cache bytes M_kv = 2 * L * n_kv * d_h * (s * b) * p, with s * b given as
 * the number of resident tokens ("Inference Engines", The Mathematics;
 * "Efficient inference", Key ideas).  Returns -1 on a negative argument.
 */
int64_t oracle_kv_bytes(int layers, int n_kv, int head_dim, int elem_bytes, int64_t tokens)
{
    if (layers < 0 || n_kv < 0 || head_dim < 0 || elem_bytes < 0 || tokens < 0)
        return -1;
    return (int64_t)2 * layers * n_kv * head_dim * elem_bytes * tokens;
}
