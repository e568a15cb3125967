/*
 * pa_oracle.c -- plain, slow, obviously-correct CPU definition of paged
 * attention and of the two paged-cache copy operations, in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header or constant with the CUDA library, and it never calls it.
 *
 * Sources (page titles; sections as printed on the pages):
 *  [EVOL]  blog "PagedAttention origin and evolution" (PagedAttention的起源与演进),
 *          sec. 3.2.1 "块管理机制" (block pool layout [num_blocks, block_size,
 *          num_heads, head_dim], separate K and V pools) and sec. 3.2.2
 *          "PagedAttention的前向传播" (per-request gather through the block
 *          table until the -1 sentinel, truncation to context_len, Q K^T /
 *          sqrt(head_dim), softmax over keys, weights times V).
 *  [VLLM4] tutorial chapter "4. PagedAttention机制：vLLM的核心创新",
 *          section "PagedAttention的注意力计算" (the pseudocode: for each
 *          query, for each logical block, physical = block_table[logical],
 *          score every token, softmax, weighted sum of values).
 *  [DW5]   study notes "DataWhale组队学习笔记--llm-algo-leetcode(五)",
 *          "代码实现" (KVCacheManager.get_physical_cache: concatenate the
 *          physical blocks of the table and cut to seq_len).
 *
 * Readings where the pages are silent or garbled (each also listed in the
 * design notes):
 *  - causal mask for a multi-query chunk is aligned to the END of the
 *    context: query i of Lq sees keys 0 .. ctx-Lq+i (for Lq == ctx this is
 *    the [EVOL] 3.2.2 lower-triangular mask; for Lq == 1 it is plain decode);
 *  - the product is per head: scores_h = scale * q_h . K_h (the [EVOL]
 *    transpose is shape-inconsistent as printed);
 *  - softmax is over all visible keys of one (query, head) row; subtracting
 *    the row maximum is the usual exact rewrite;
 *  - only ceil(ctx/block_size) table entries are read; an entry outside
 *    [0, num_blocks) among them is an error; ctx == 0 gives a zero row;
 *  - negative slots in a cache write are padding and are skipped;
 *    duplicate slots, overlapping copy pairs are rejected.
 *
 * All floating point is IEEE binary64 with plain left-to-right summation.
 * fp16 inputs arrive as raw bit patterns and are decoded exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum {
    ORACLE_OK = 0,
    ORACLE_BAD_ARG = 1,       /* a size or pointer makes no sense */
    ORACLE_BAD_BLOCK = 2,     /* a needed block-table entry is out of range */
    ORACLE_BAD_CONTEXT = 3,   /* ctx < 0 or more keys than the table holds */
    ORACLE_BAD_SLOT = 4,      /* slot beyond the pool */
    ORACLE_DUP_SLOT = 5,      /* two tokens written to the same slot */
    ORACLE_BAD_PAIR = 6,      /* copy pair out of range or overlapping */
};

/* IEEE-754 binary16 -> binary64, exact.  1 sign bit, 5 exponent bits
 * (bias 15), 10 fraction bits.  Exponent 0: subnormal, value = frac * 2^-24.
 * Exponent 31: infinity (frac 0) or NaN.  Otherwise (1024 + frac) * 2^(e-25). */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)frac, -24);
    else if (e == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), e - 25);
    return sign ? -mag : mag;
}

/* Element (blk, tok, head, d) of a pool laid out [num_blocks, bs, H, D]. */
static double pool_at(const uint16_t *pool, int64_t blk, int tok, int head,
                      int d, int bs, int H, int D)
{
    int64_t idx = (((blk * bs + tok) * (int64_t)H + head) * D) + d;
    return oracle_half_to_double(pool[idx]);
}

/*
 * One output row: the query row q[0..D) of head `head` attends to logical
 * keys 0 .. n_keys-1 of one sequence whose block table is `table`.
 *   key j lives in physical block table[j / bs], token slot j % bs;
 *   s_j = scale * sum_d q[d] * K[j][d];
 *   w_j = exp(s_j - max_k s_k);  out[d] = sum_j w_j V[j][d] / sum_j w_j.
 * n_keys == 0 gives a zero row.
 */
int oracle_attend_row(const uint16_t *q_row, const uint16_t *k_cache,
                      const uint16_t *v_cache, const int32_t *table,
                      int table_len, int n_keys, int H, int head, int D,
                      int bs, int64_t num_blocks, double scale, double *out)
{
    if (n_keys < 0 || D <= 0 || bs <= 0 || head < 0 || head >= H)
        return ORACLE_BAD_ARG;
    if ((int64_t)n_keys > (int64_t)table_len * bs)
        return ORACLE_BAD_CONTEXT;
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    if (n_keys == 0)
        return ORACLE_OK;

    int n_blocks_used = (n_keys + bs - 1) / bs;
    for (int lb = 0; lb < n_blocks_used; ++lb)
        if (table[lb] < 0 || (int64_t)table[lb] >= num_blocks)
            return ORACLE_BAD_BLOCK;

    double *q = (double *)malloc(sizeof(double) * (size_t)D);
    double *s = (double *)malloc(sizeof(double) * (size_t)n_keys);
    if (!q || !s) {
        free(q);
        free(s);
        return ORACLE_BAD_ARG;
    }
    for (int d = 0; d < D; ++d)
        q[d] = oracle_half_to_double(q_row[d]);

    /* scores */
    for (int j = 0; j < n_keys; ++j) {
        int64_t blk = table[j / bs];
        int tok = j % bs;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += q[d] * pool_at(k_cache, blk, tok, head, d, bs, H, D);
        s[j] = scale * dot;
    }
    /* softmax over the row */
    double m = s[0];
    for (int j = 1; j < n_keys; ++j)
        if (s[j] > m)
            m = s[j];
    double z = 0.0;
    for (int j = 0; j < n_keys; ++j) {
        s[j] = exp(s[j] - m);
        z += s[j];
    }
    /* weighted sum of V */
    for (int j = 0; j < n_keys; ++j) {
        int64_t blk = table[j / bs];
        int tok = j % bs;
        double w = s[j] / z;
        for (int d = 0; d < D; ++d)
            out[d] += w * pool_at(v_cache, blk, tok, head, d, bs, H, D);
    }
    free(q);
    free(s);
    return ORACLE_OK;
}

/* Decode: q[B,H,D], one query per sequence, attending to all context_lens[b]
 * keys.  out[B,H,D] in fp64. */
int oracle_decode(const uint16_t *q, const uint16_t *k_cache,
                  const uint16_t *v_cache, const int32_t *block_tables,
                  const int32_t *context_lens, int B, int H, int D, int bs,
                  int64_t num_blocks, int max_blocks_per_seq, double scale,
                  double *out)
{
    if (B < 0 || H <= 0 || D <= 0 || bs <= 0 || max_blocks_per_seq < 0)
        return ORACLE_BAD_ARG;
    for (int b = 0; b < B; ++b) {
        int ctx = context_lens[b];
        if (ctx < 0)
            return ORACLE_BAD_CONTEXT;
        for (int h = 0; h < H; ++h) {
            int rc = oracle_attend_row(
                q + ((int64_t)b * H + h) * D, k_cache, v_cache,
                block_tables + (int64_t)b * max_blocks_per_seq,
                max_blocks_per_seq, ctx, H, h, D, bs, num_blocks, scale,
                out + ((int64_t)b * H + h) * D);
            if (rc != ORACLE_OK)
                return rc;
        }
    }
    return ORACLE_OK;
}

/* Chunked prefill: q[B,H,Lq,D] are the last Lq positions of each sequence's
 * context_lens[b] keys.  Query i sees keys 0 .. ctx-Lq+i (end-aligned causal
 * mask).  ctx < Lq is an error.  out[B,H,Lq,D] in fp64. */
int oracle_prefill(const uint16_t *q, const uint16_t *k_cache,
                   const uint16_t *v_cache, const int32_t *block_tables,
                   const int32_t *context_lens, int B, int H, int Lq, int D,
                   int bs, int64_t num_blocks, int max_blocks_per_seq,
                   double scale, double *out)
{
    if (B < 0 || H <= 0 || Lq < 0 || D <= 0 || bs <= 0)
        return ORACLE_BAD_ARG;
    for (int b = 0; b < B; ++b) {
        int ctx = context_lens[b];
        if (ctx < Lq)
            return ORACLE_BAD_CONTEXT;
        for (int h = 0; h < H; ++h)
            for (int i = 0; i < Lq; ++i) {
                int64_t row = (((int64_t)b * H + h) * Lq + i) * D;
                int rc = oracle_attend_row(
                    q + row, k_cache, v_cache,
                    block_tables + (int64_t)b * max_blocks_per_seq,
                    max_blocks_per_seq, ctx - Lq + i + 1, H, h, D, bs,
                    num_blocks, scale, out + row);
                if (rc != ORACLE_OK)
                    return rc;
            }
    }
    return ORACLE_OK;
}

/* Cache write: for each token t with slot_mapping[t] >= 0, copy the H*D
 * values k[t] into k_cache viewed as [num_blocks*bs, H, D] at row slot, and
 * the same for v.  Bit patterns are copied unchanged. */
int oracle_kv_cache_write(const uint16_t *k, const uint16_t *v,
                          const int64_t *slot_mapping, int T, int H, int D,
                          int bs, int64_t num_blocks, uint16_t *k_cache,
                          uint16_t *v_cache)
{
    if (T < 0 || H <= 0 || D <= 0 || bs <= 0)
        return ORACLE_BAD_ARG;
    int64_t n_slots = num_blocks * bs;
    int64_t row = (int64_t)H * D;
    for (int t = 0; t < T; ++t) {
        if (slot_mapping[t] >= n_slots)
            return ORACLE_BAD_SLOT;
        for (int u = 0; u < t; ++u)
            if (slot_mapping[t] >= 0 && slot_mapping[u] == slot_mapping[t])
                return ORACLE_DUP_SLOT;
    }
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        for (int64_t e = 0; e < row; ++e) {
            k_cache[slot * row + e] = k[(int64_t)t * row + e];
            v_cache[slot * row + e] = v[(int64_t)t * row + e];
        }
    }
    return ORACLE_OK;
}

/* Block copy (copy-on-write): for each pair (src, dst), physical block dst
 * of both pools becomes a copy of block src (all bs*H*D values).  Pairs must
 * be in range, destinations distinct, and no destination may also be a
 * source; src == dst is a no-op. */
int oracle_block_copy(uint16_t *k_cache, uint16_t *v_cache,
                      const int64_t *pairs, int N, int H, int D, int bs,
                      int64_t num_blocks)
{
    if (N < 0 || H <= 0 || D <= 0 || bs <= 0)
        return ORACLE_BAD_ARG;
    for (int i = 0; i < N; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks)
            return ORACLE_BAD_PAIR;
    }
    for (int i = 0; i < N; ++i) {
        int64_t dst = pairs[2 * i + 1];
        if (pairs[2 * i] == dst)
            continue; /* no-op pair */
        for (int u = 0; u < N; ++u) {
            int64_t us = pairs[2 * u], ud = pairs[2 * u + 1];
            if (u == i || us == ud)
                continue;
            if (ud == dst || us == dst) /* shared destination, or dst read by another pair */
                return ORACLE_BAD_PAIR;
        }
    }
    int64_t blk = (int64_t)bs * H * D;
    for (int i = 0; i < N; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src == dst)
            continue;
        memcpy(k_cache + dst * blk, k_cache + src * blk, sizeof(uint16_t) * (size_t)blk);
        memcpy(v_cache + dst * blk, v_cache + src * blk, sizeof(uint16_t) * (size_t)blk);
    }
    return ORACLE_OK;
}

/* Gather to contiguous ([DW5] get_physical_cache): out[j] = pool row of
 * logical key j for j < seq_len, for one head, as fp64 [seq_len, D]. */
int oracle_gather(const uint16_t *pool, const int32_t *table, int table_len,
                  int seq_len, int H, int head, int D, int bs,
                  int64_t num_blocks, double *out)
{
    if (seq_len < 0 || (int64_t)seq_len > (int64_t)table_len * bs)
        return ORACLE_BAD_CONTEXT;
    for (int j = 0; j < seq_len; ++j) {
        int64_t blk = table[j / bs];
        if (blk < 0 || blk >= num_blocks)
            return ORACLE_BAD_BLOCK;
        for (int d = 0; d < D; ++d)
            out[(int64_t)j * D + d] = pool_at(pool, blk, j % bs, head, d, bs, H, D);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------
 * FP8 (e4m3) KV storage -- the "mixed-precision KV storage" of the blog
 * "PagedAttention origin and evolution", sec. 2.3, read as: each (token,
 * head) row of K and of V is stored as D e4m3 codes plus one fp32 scale,
 * value = code * scale, scale = max|row| / 448 (448 is the largest finite
 * e4m3 value), a zero row gets scale 1.
 *
 * e4m3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 fraction
 * bits, no infinities; S.1111.111 is NaN; the largest finite value is
 * S.1111.110 = 1.75 * 2^8 = 448; exponent 0 is subnormal: frac * 2^-9.
 * ------------------------------------------------------------------------ */
double oracle_e4m3_to_double(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int frac = c & 7;
    double mag;
    if (e == 15 && frac == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)frac, -9);
    else
        mag = ldexp((double)(8 + frac), e - 10);
    return sign ? -mag : mag;
}

/* Round a float to the nearest e4m3 value, ties to even, saturating to
 * +-448.  Works on the exact binary value of x: every e4m3 value is exactly
 * representable in double, so the nearest one is found by comparing
 * distances to the two neighbours below and above |x|. */
uint8_t oracle_e4m3_from_float(float x)
{
    if (x != x)
        return 0x7f;
    int sign = signbit(x) ? 1 : 0;
    double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)((sign << 7) | 0x7e);
    /* largest code whose magnitude is <= a */
    int lo = 0;
    for (int c = 0; c <= 0x7e; ++c)
        if (oracle_e4m3_to_double((uint8_t)c) <= a)
            lo = c;
    int hi = lo < 0x7e ? lo + 1 : lo;
    double dlo = a - oracle_e4m3_to_double((uint8_t)lo);
    double dhi = oracle_e4m3_to_double((uint8_t)hi) - a;
    int pick;
    if (dlo < dhi)
        pick = lo;
    else if (dhi < dlo)
        pick = hi;
    else
        pick = (lo & 1) ? hi : lo; /* tie: even fraction (last bit 0) */
    return (uint8_t)((sign << 7) | pick);
}

/* Quantizing cache write: like oracle_kv_cache_write, but each (token, head)
 * row is stored as e4m3 codes into k8/v8 [num_blocks, bs, H, D] with its
 * fp32 scale in ks/vs [num_blocks, H, bs].  The scale and the quotient are
 * IEEE single-precision divisions. */
static void quantize_row(const uint16_t *x, int D, uint8_t *codes, float *scale)
{
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float v = (float)fabs(oracle_half_to_double(x[d]));
        if (v > amax)
            amax = v;
    }
    float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int d = 0; d < D; ++d) {
        float v = (float)oracle_half_to_double(x[d]);
        codes[d] = oracle_e4m3_from_float(v / s);
    }
    *scale = s;
}

int oracle_kv_cache_write_fp8(const uint16_t *k, const uint16_t *v,
                              const int64_t *slot_mapping, int T, int H, int D,
                              int bs, int64_t num_blocks, uint8_t *k8,
                              uint8_t *v8, float *ks, float *vs)
{
    if (T < 0 || H <= 0 || D <= 0 || bs <= 0)
        return ORACLE_BAD_ARG;
    int64_t n_slots = num_blocks * bs;
    for (int t = 0; t < T; ++t) {
        if (slot_mapping[t] >= n_slots)
            return ORACLE_BAD_SLOT;
        for (int u = 0; u < t; ++u)
            if (slot_mapping[t] >= 0 && slot_mapping[u] == slot_mapping[t])
                return ORACLE_DUP_SLOT;
    }
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t blk = slot / bs, off = slot % bs;
        for (int h = 0; h < H; ++h) {
            int64_t src = ((int64_t)t * H + h) * D;
            int64_t dst = (slot * H + h) * D;
            int64_t si = (blk * H + h) * bs + off;
            quantize_row(k + src, D, k8 + dst, ks + si);
            quantize_row(v + src, D, v8 + dst, vs + si);
        }
    }
    return ORACLE_OK;
}

/* Decode over an e4m3 cache: key j of head h is e4m3(k8[...]) * ks[...],
 * dequantized exactly in double; then the same definition as
 * oracle_attend_row. */
int oracle_decode_fp8(const uint16_t *q, const uint8_t *k8, const uint8_t *v8,
                      const float *ks, const float *vs,
                      const int32_t *block_tables, const int32_t *context_lens,
                      int B, int H, int D, int bs, int64_t num_blocks,
                      int max_blocks_per_seq, double scale, double *out)
{
    if (B < 0 || H <= 0 || D <= 0 || bs <= 0 || max_blocks_per_seq < 0)
        return ORACLE_BAD_ARG;
    for (int b = 0; b < B; ++b) {
        int n = context_lens[b];
        const int32_t *table = block_tables + (int64_t)b * max_blocks_per_seq;
        if (n < 0 || (int64_t)n > (int64_t)max_blocks_per_seq * bs)
            return ORACLE_BAD_CONTEXT;
        for (int lb = 0; lb < (n + bs - 1) / bs; ++lb)
            if (table[lb] < 0 || (int64_t)table[lb] >= num_blocks)
                return ORACLE_BAD_BLOCK;
        for (int h = 0; h < H; ++h) {
            double *o = out + ((int64_t)b * H + h) * D;
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            if (n == 0)
                continue;
            double *s = (double *)malloc(sizeof(double) * (size_t)n);
            if (!s)
                return ORACLE_BAD_ARG;
            const uint16_t *qr = q + ((int64_t)b * H + h) * D;
            for (int j = 0; j < n; ++j) {
                int64_t blk = table[j / bs];
                int off = j % bs;
                const uint8_t *kr = k8 + ((blk * bs + off) * H + h) * D;
                double kscale = (double)ks[(blk * H + h) * bs + off];
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += oracle_half_to_double(qr[d]) * (oracle_e4m3_to_double(kr[d]) * kscale);
                s[j] = scale * dot;
            }
            double m = s[0];
            for (int j = 1; j < n; ++j)
                if (s[j] > m)
                    m = s[j];
            double z = 0.0;
            for (int j = 0; j < n; ++j) {
                s[j] = exp(s[j] - m);
                z += s[j];
            }
            for (int j = 0; j < n; ++j) {
                int64_t blk = table[j / bs];
                int off = j % bs;
                const uint8_t *vr = v8 + ((blk * bs + off) * H + h) * D;
                double vscale = (double)vs[(blk * H + h) * bs + off];
                double w = s[j] / z;
                for (int d = 0; d < D; ++d)
                    o[d] += w * (oracle_e4m3_to_double(vr[d]) * vscale);
            }
            free(s);
        }
    }
    return ORACLE_OK;
}
