/*
 * pagedkv_oracle.c -- plain, slow CPU oracle for decode-phase paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU
 * baseline legs of bench.py may load this library.  The product (the CUDA
 * library under paged_kv_cache_97_gb300/) never includes, links or calls it,
 * and this file includes nothing from the product: the two share no code.
 *
 * Everything is written as the plain definition of what the pages describe,
 * in fp64 for floating point, with no blocking or fusion beyond what that
 * definition states:
 *
 *   - slot mapping through a block table
 *       (“让 Agent 跑得快：LLM 推理服务”, §五 “Block 级管理的优雅性”: a block
 *        table maps each request's logical blocks to physical blocks of a
 *        shared pool; §二: blocks hold 16 tokens by default)
 *   - appending the new token's K/V into its slot (bf16 bit copy, or an int8
 *       or FP8 E4M3 code under a per-(block, KV head) scale)
 *       (same page, §一 “KV Cache”: decode computes the new token's Q, attends
 *        over cached K/V and appends the new K/V; §五 “共享前缀”: only the
 *        current decode token writes; pool layout [num_blocks, block_size,
 *        num_heads, head_dim] from “LLM 推理引擎深度解析”, §2.1 PagedKVCache)
 *   - attention for one query token: gather the sequence's blocks into
 *       contiguous K and V, then the three-pass safe softmax
 *       (“LLM 推理优化技术全景”, 在线 Softmax: max pass, sum pass, divide pass)
 *   - the online (m, l) recurrence, written as that page states it, with the
 *       output kept normalised after every block (self-check only)
 *   - per-partition partials and their log-sum-exp merge (self-check of the
 *       split-K reading of “Flash Attention v2 的改进”: parallelism along the
 *       sequence with the rescale deferred to the end)
 *
 * GQA head mapping (“让 Agent 跑得快”, framework table: 32 query heads share
 * 8 KV heads): query head h reads KV head h / (num_q_heads / num_kv_heads).
 *
 * Return codes: 0 = ok, 1 = invalid argument, 4 = an index (block id, slot,
 * sequence length) out of range; the affected output rows are set to zero.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_INVALID 1
#define OR_INDEX 4

/* bf16 is the upper half of an IEEE fp32; widen exactly. */
static float bf16_to_float(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------------ */
/* Slot mapping: slot = block_tables[s][p / bs] * bs + p % bs.              */
/* ------------------------------------------------------------------------ */

/* Token i belongs to sequence seq_idx[i] (or i when seq_idx is NULL) and sits
 * at 0-based position positions[i].  A negative position yields slot -1.  A
 * position past the table, or a table entry outside [0, num_blocks), yields
 * slot -1 and the return value OR_INDEX. */
int oracle_token_slots(const int32_t *block_tables, int max_blocks_per_seq,
                       const int32_t *seq_idx, const int32_t *positions,
                       int num_tokens, int block_size, int num_blocks,
                       int64_t *slots)
{
    if (!block_tables || !positions || !slots || block_size <= 0 ||
        max_blocks_per_seq <= 0 || num_tokens < 0)
        return OR_INVALID;
    int rc = OR_OK;
    for (int i = 0; i < num_tokens; ++i) {
        int s = seq_idx ? seq_idx[i] : i;
        int p = positions[i];
        slots[i] = -1;
        if (p < 0)
            continue;
        int logical = p / block_size;
        if (logical >= max_blocks_per_seq) {
            rc = OR_INDEX;
            continue;
        }
        int32_t physical = block_tables[(int64_t)s * max_blocks_per_seq + logical];
        if (physical < 0 || physical >= num_blocks) {
            rc = OR_INDEX;
            continue;
        }
        slots[i] = (int64_t)physical * block_size + (p % block_size);
    }
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Append (reshape_and_cache).                                              */
/* ------------------------------------------------------------------------ */

/* Element (slot, head, e) of a pool laid out [num_blocks, block_size,
 * num_kv_heads, head_dim]; slot = block * block_size + row. */
static int64_t pool_index(int64_t slot, int block_size, int num_kv_heads,
                          int head_dim, int head, int e)
{
    int64_t block = slot / block_size;
    int64_t row = slot % block_size;
    return ((block * block_size + row) * num_kv_heads + head) * head_dim + e;
}

/* k, v: bf16 bits [num_tokens, num_kv_heads, head_dim].  Copies each element's
 * bits into the token's slot.  Slots < 0 are skipped; slots >= num_blocks *
 * block_size are skipped and reported. */
int oracle_append_bf16(const uint16_t *k, const uint16_t *v, uint16_t *k_cache,
                       uint16_t *v_cache, const int64_t *slots, int num_tokens,
                       int num_blocks, int block_size, int num_kv_heads,
                       int head_dim)
{
    if (!k || !v || !k_cache || !v_cache || !slots)
        return OR_INVALID;
    int rc = OR_OK;
    int64_t capacity = (int64_t)num_blocks * block_size;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slots[i];
        if (slot < 0)
            continue;
        if (slot >= capacity) {
            rc = OR_INDEX;
            continue;
        }
        for (int h = 0; h < num_kv_heads; ++h)
            for (int e = 0; e < head_dim; ++e) {
                int64_t src = ((int64_t)i * num_kv_heads + h) * head_dim + e;
                int64_t dst = pool_index(slot, block_size, num_kv_heads, head_dim, h, e);
                k_cache[dst] = k[src];
                v_cache[dst] = v[src];
            }
    }
    return rc;
}

/* The int8 code of value x under scale s, decided in fp32:
 *   code = clamp(round_half_even(x / s), -127, 127), NaN -> 0, s == 0 -> s = 1.
 * The fp32 quotient is the IEEE-rounded one (no contraction); nearbyintf uses
 * the default rounding mode, ties to even. */
static int8_t quantize_int8(float x, float s)
{
    if (s == 0.0f)
        s = 1.0f;
    float r = nearbyintf(x / s);
    if (r != r)
        return 0;
    if (r > 127.0f)
        return 127;
    if (r < -127.0f)
        return -127;
    return (int8_t)(int)r;
}

int oracle_quantize_int8(float x, float s) { return (int)quantize_int8(x, s); }

/* FP8 E4M3 (the 8-bit float named beside E5M2 in “LLM 推理优化技术全景”,
 * Flash Attention v3, and used for the KV cache in “让 Agent 跑得快”, §四
 * “FP8 量化”): bit 7 sign, bits 6..3 exponent field E (bias 7), bits 2..0
 * mantissa M.  E = 0: subnormal, M/8 * 2^-6.  Otherwise (1 + M/8) * 2^(E-7).
 * The one pattern with E = 15 and M = 7 is NaN; there is no infinity, so the
 * largest finite value is (1 + 6/8) * 2^8 = 448. */
double oracle_fp8_value(int code)
{
    int c = code & 0xFF;
    int e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    double mag = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return (c & 0x80) ? -mag : mag;
}

/* The E4M3 code of value x under scale s: the fp32 quotient x / s (as for
 * int8; s == 0 -> 1), rounded to the nearest finite E4M3 value with ties to
 * the even code (even mantissa), magnitudes above 448 saturating to 448 (the
 * reading this library takes, as int8 clamps to 127), NaN -> 0x7F.  The sign
 * is kept, so negative values that round to zero give 0x80.  Found by
 * comparing the quotient with every finite non-negative code. */
static uint8_t quantize_fp8(float x, float s)
{
    if (s == 0.0f)
        s = 1.0f;
    float r = x / s;
    if (r != r)
        return 0x7F;
    uint8_t sign = signbit(r) ? 0x80 : 0x00;
    double a = fabs((double)r);
    if (a >= 448.0)
        return sign | 0x7E;
    int best = 0;
    double best_d = a;
    for (int c = 1; c <= 0x7E; ++c) {
        double d = fabs(oracle_fp8_value(c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return sign | (uint8_t)best;
}

int oracle_quantize_fp8(float x, float s) { return (int)quantize_fp8(x, s); }

/* int8 codes as bytes, for the shared 8-bit append below. */
static uint8_t quantize_int8_byte(float x, float s) { return (uint8_t)quantize_int8(x, s); }

/* As oracle_append_bf16, but stores 8-bit codes under k_scale / v_scale,
 * which are fp32 [num_blocks, num_kv_heads]: the scale of the slot's block. */
static int append_codes(const uint16_t *k, const uint16_t *v, uint8_t *k_cache,
                        uint8_t *v_cache, const float *k_scale, const float *v_scale,
                        const int64_t *slots, int num_tokens, int num_blocks,
                        int block_size, int num_kv_heads, int head_dim,
                        uint8_t (*code)(float, float))
{
    if (!k || !v || !k_cache || !v_cache || !k_scale || !v_scale || !slots)
        return OR_INVALID;
    int rc = OR_OK;
    int64_t capacity = (int64_t)num_blocks * block_size;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slots[i];
        if (slot < 0)
            continue;
        if (slot >= capacity) {
            rc = OR_INDEX;
            continue;
        }
        int64_t block = slot / block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            float ks = k_scale[block * num_kv_heads + h];
            float vs = v_scale[block * num_kv_heads + h];
            for (int e = 0; e < head_dim; ++e) {
                int64_t src = ((int64_t)i * num_kv_heads + h) * head_dim + e;
                int64_t dst = pool_index(slot, block_size, num_kv_heads, head_dim, h, e);
                k_cache[dst] = code(bf16_to_float(k[src]), ks);
                v_cache[dst] = code(bf16_to_float(v[src]), vs);
            }
        }
    }
    return rc;
}

int oracle_append_int8(const uint16_t *k, const uint16_t *v, int8_t *k_cache,
                       int8_t *v_cache, const float *k_scale,
                       const float *v_scale, const int64_t *slots,
                       int num_tokens, int num_blocks, int block_size,
                       int num_kv_heads, int head_dim)
{
    return append_codes(k, v, (uint8_t *)k_cache, (uint8_t *)v_cache, k_scale, v_scale, slots,
                        num_tokens, num_blocks, block_size, num_kv_heads, head_dim,
                        quantize_int8_byte);
}

int oracle_append_fp8(const uint16_t *k, const uint16_t *v, uint8_t *k_cache,
                      uint8_t *v_cache, const float *k_scale,
                      const float *v_scale, const int64_t *slots,
                      int num_tokens, int num_blocks, int block_size,
                      int num_kv_heads, int head_dim)
{
    return append_codes(k, v, k_cache, v_cache, k_scale, v_scale, slots, num_tokens,
                        num_blocks, block_size, num_kv_heads, head_dim, quantize_fp8);
}

/* ------------------------------------------------------------------------ */
/* Attention.                                                               */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q;       /* bf16 [batch, num_q_heads, head_dim] */
    const void *k_cache;     /* bf16 bits, int8 or E4M3 [num_blocks, bs, Hkv, d] */
    const void *v_cache;
    const float *k_scale;    /* [num_blocks, Hkv] for 8-bit pools */
    const float *v_scale;
    int kv_kind;             /* 0 bf16, 1 int8, 2 E4M3 */
    const int32_t *block_tables; /* [batch, max_blocks] */
    int max_blocks;
    const int32_t *seq_lens;     /* [batch], including the appended token */
    int batch, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size;
    double scale;
    /* Multi-token queries (NULL for one query token per sequence): the
     * query tokens of sequence b are q rows query_start[b] ..
     * query_start[b + 1] - 1, the last n_b = query_start[b + 1] -
     * query_start[b] tokens of the sequence, in order. */
    const int32_t *query_start;  /* [batch + 1] */
    int num_tokens;
} attn_problem;

/* Value of element e of the token at logical position t of sequence b, KV
 * head hk, from the K (which = 0) or V (which = 1) pool, widened to fp64.
 * int8 and E4M3 codes are multiplied by their block's scale in fp64. */
static double pool_value(const attn_problem *P, int which, int32_t block,
                         int row, int hk, int e)
{
    int64_t idx = (((int64_t)block * P->block_size + row) * P->num_kv_heads + hk) *
                      P->head_dim + e;
    if (P->kv_kind != 0) {
        const float *s = which ? P->v_scale : P->k_scale;
        double sc = (double)s[(int64_t)block * P->num_kv_heads + hk];
        if (P->kv_kind == 2) {
            const uint8_t *c = (const uint8_t *)(which ? P->v_cache : P->k_cache);
            return oracle_fp8_value(c[idx]) * sc;
        }
        const int8_t *c = (const int8_t *)(which ? P->v_cache : P->k_cache);
        return (double)c[idx] * sc;
    }
    const uint16_t *c = (const uint16_t *)(which ? P->v_cache : P->k_cache);
    return (double)bf16_to_float(c[idx]);
}

/* Check a sequence's length and table entries.  Returns 0 when every logical
 * block the sequence uses names a physical block of the pool. */
static int check_sequence(const attn_problem *P, int b)
{
    int L = P->seq_lens[b];
    if (L <= 0 || (int64_t)L > (int64_t)P->max_blocks * P->block_size)
        return OR_INDEX;
    int nblk = (L + P->block_size - 1) / P->block_size;
    for (int j = 0; j < nblk; ++j) {
        int32_t p = P->block_tables[(int64_t)b * P->max_blocks + j];
        if (p < 0 || p >= P->num_blocks)
            return OR_INDEX;
    }
    return OR_OK;
}

/* Gather the first L tokens of sequence b, KV head hk, into contiguous fp64
 * K[L][d] and V[L][d]: token t lives in physical block
 * block_tables[b][t / bs], row t % bs. */
static void gather_kv(const attn_problem *P, int b, int hk, int L, double *K, double *V)
{
    int d = P->head_dim, bs = P->block_size;
    for (int t = 0; t < L; ++t) {
        int32_t block = P->block_tables[(int64_t)b * P->max_blocks + t / bs];
        for (int e = 0; e < d; ++e) {
            K[(int64_t)t * d + e] = pool_value(P, 0, block, t % bs, hk, e);
            V[(int64_t)t * d + e] = pool_value(P, 1, block, t % bs, hk, e);
        }
    }
}

/* s_t = scale * sum_e q_e K_t,e for the first L gathered tokens, q being
 * row qrow of the query tensor [rows, d]. */
static void scores(const attn_problem *P, int64_t qrow, int L, const double *K, double *s)
{
    int d = P->head_dim;
    const uint16_t *q = P->q + qrow * d;
    for (int t = 0; t < L; ++t) {
        double acc = 0.0;
        for (int e = 0; e < d; ++e)
            acc += (double)bf16_to_float(q[e]) * K[(int64_t)t * d + e];
        s[t] = P->scale * acc;
    }
}

/* Three-pass safe softmax attention for query row qrow over the first L
 * tokens:
 *   pass 1: m = max_t s_t
 *   pass 2: Z = sum_t exp(s_t - m)
 *   pass 3: o = sum_t exp(s_t - m) / Z * V_t                           */
static void three_pass_row(const attn_problem *P, int64_t qrow, int L, const double *K,
                           const double *V, double *s, double *o)
{
    int d = P->head_dim;
    scores(P, qrow, L, K, s);
    double m = -INFINITY;
    for (int t = 0; t < L; ++t)
        if (s[t] > m)
            m = s[t];
    double Z = 0.0;
    for (int t = 0; t < L; ++t)
        Z += exp(s[t] - m);
    for (int e = 0; e < d; ++e)
        o[e] = 0.0;
    for (int t = 0; t < L; ++t) {
        double w = exp(s[t] - m) / Z;
        for (int e = 0; e < d; ++e)
            o[e] += w * V[(int64_t)t * d + e];
    }
}

/* Online softmax over the sequence's logical blocks, as the recurrence is
 * written in “LLM 推理优化技术全景”, 在线 Softmax:
 *   m_new = max(m_old, max S_j)
 *   l_new = l_old * exp(m_old - m_new) + sum exp(S_j - m_new)
 *   O_new = O_old * l_old * exp(m_old - m_new) / l_new
 *           + sum exp(S_j - m_new) V_j / l_new
 * with m = -inf, l = 0, O = 0 before the first block, and the chunk S_j being
 * one block of block_size tokens (the last one ragged). */
static void online_row(const attn_problem *P, int64_t qrow, int L, const double *K,
                       const double *V, double *s, double *o)
{
    int d = P->head_dim, bs = P->block_size;
    scores(P, qrow, L, K, s);
    double m_old = -INFINITY, l_old = 0.0;
    for (int e = 0; e < d; ++e)
        o[e] = 0.0;
    double *num = (double *)calloc((size_t)d, sizeof(double));
    for (int t0 = 0; t0 < L; t0 += bs) {
        int t1 = t0 + bs < L ? t0 + bs : L;
        double mj = -INFINITY;
        for (int t = t0; t < t1; ++t)
            if (s[t] > mj)
                mj = s[t];
        double m_new = m_old > mj ? m_old : mj;
        double carry = (l_old == 0.0) ? 0.0 : exp(m_old - m_new);
        double sum = 0.0;
        for (int e = 0; e < d; ++e)
            num[e] = 0.0;
        for (int t = t0; t < t1; ++t) {
            double p = exp(s[t] - m_new);
            sum += p;
            for (int e = 0; e < d; ++e)
                num[e] += p * V[(int64_t)t * d + e];
        }
        double l_new = l_old * carry + sum;
        for (int e = 0; e < d; ++e)
            o[e] = o[e] * l_old * carry / l_new + num[e] / l_new;
        m_old = m_new;
        l_old = l_new;
    }
    free(num);
}

/* Per-partition partials of row (b, h): partition i covers logical tokens
 * [i*part, min((i+1)*part, L)) and holds
 *   m_i = max s,  l_i = sum exp(s - m_i),  acc_i = sum exp(s - m_i) V
 * (acc_i unnormalised).  Partials are written to ml[i][2] and acc[i][d]. */
static void partial_row(const attn_problem *P, int b, int h, const double *K,
                        const double *V, double *s, int part, double *ml,
                        double *acc)
{
    int L = P->seq_lens[b], d = P->head_dim;
    scores(P, (int64_t)b * P->num_q_heads + h, L, K, s);
    int np = (L + part - 1) / part;
    for (int i = 0; i < np; ++i) {
        int t0 = i * part, t1 = (i + 1) * part < L ? (i + 1) * part : L;
        double m = -INFINITY;
        for (int t = t0; t < t1; ++t)
            if (s[t] > m)
                m = s[t];
        double l = 0.0;
        double *a = acc + (int64_t)i * d;
        for (int e = 0; e < d; ++e)
            a[e] = 0.0;
        for (int t = t0; t < t1; ++t) {
            double p = exp(s[t] - m);
            l += p;
            for (int e = 0; e < d; ++e)
                a[e] += p * V[(int64_t)t * d + e];
        }
        ml[2 * i] = m;
        ml[2 * i + 1] = l;
    }
}

/* ------------------------------------------------------------------------ */
/* Row scheduling over host threads.                                        */
/* ------------------------------------------------------------------------ */

enum { MODE_THREE_PASS = 0, MODE_ONLINE = 1 };

typedef struct {
    const attn_problem *P;
    const int32_t *rows;  /* pairs (b, h); NULL = every (b, h) */
    int n_rows;
    int mode;
    double *out;          /* [n_rows, d] */
    int next;             /* shared work counter */
    int status;
    pthread_mutex_t lock;
} row_job;

/* Multi-token queries: the sequence b of query token j (query_start[b] <= j <
 * query_start[b + 1]) and the number of tokens it attends: with n_b query
 * tokens, token i = j - query_start[b] sits at position L_b - n_b + i and
 * attends positions 0 .. L_b - n_b + i (causal: its own and the earlier ones).
 * OR_INDEX when the offsets are not non-decreasing from 0 to num_tokens or
 * n_b exceeds L_b. */
static int multi_token_row(const attn_problem *P, int j, int *b_out, int *L_out)
{
    const int32_t *qs = P->query_start;
    if (qs[0] != 0 || qs[P->batch] != P->num_tokens || j < 0 || j >= P->num_tokens)
        return OR_INDEX;
    for (int b = 0; b < P->batch; ++b) {
        if (qs[b + 1] < qs[b])
            return OR_INDEX;
        if (j < qs[b + 1]) {
            int n = qs[b + 1] - qs[b], L = P->seq_lens[b];
            if (n > L)
                return OR_INDEX;
            *b_out = b;
            *L_out = L - n + (j - qs[b]) + 1;
            return OR_OK;
        }
    }
    return OR_INDEX;
}

static int take_row(row_job *J)
{
    pthread_mutex_lock(&J->lock);
    int r = J->next < J->n_rows ? J->next++ : -1;
    pthread_mutex_unlock(&J->lock);
    return r;
}

static void *row_worker(void *arg)
{
    row_job *J = (row_job *)arg;
    const attn_problem *P = J->P;
    int d = P->head_dim;
    int64_t cap = (int64_t)P->max_blocks * P->block_size;
    double *K = (double *)malloc((size_t)cap * d * sizeof(double));
    double *V = (double *)malloc((size_t)cap * d * sizeof(double));
    double *s = (double *)malloc((size_t)cap * sizeof(double));
    for (int r; (r = take_row(J)) >= 0;) {
        /* The row's sequence b, query head h, query-tensor row and the
         * number of tokens it attends (L_b, or pos + 1 for a multi-token
         * query at position pos). */
        int b = -1, h, L = 0;
        int64_t qrow = 0;
        if (P->query_start) {
            int j = r / P->num_q_heads;
            h = r % P->num_q_heads;
            int ok = 0;
            if (multi_token_row(P, j, &b, &L) == OR_OK) {
                qrow = (int64_t)j * P->num_q_heads + h;
                ok = 1;
            }
            if (!ok)
                b = -1;
        } else {
            if (J->rows) {
                b = J->rows[2 * r];
                h = J->rows[2 * r + 1];
            } else {
                b = r / P->num_q_heads;
                h = r % P->num_q_heads;
            }
            if (b >= 0 && b < P->batch) {
                L = P->seq_lens[b];
                qrow = (int64_t)b * P->num_q_heads + h;
            }
        }
        double *o = J->out + (int64_t)r * d;
        if (b < 0 || b >= P->batch || h < 0 || h >= P->num_q_heads ||
            check_sequence(P, b) != OR_OK) {
            for (int e = 0; e < d; ++e)
                o[e] = 0.0;
            pthread_mutex_lock(&J->lock);
            J->status = OR_INDEX;
            pthread_mutex_unlock(&J->lock);
            continue;
        }
        int hk = h / (P->num_q_heads / P->num_kv_heads);
        gather_kv(P, b, hk, L, K, V);
        if (J->mode == MODE_ONLINE)
            online_row(P, qrow, L, K, V, s, o);
        else
            three_pass_row(P, qrow, L, K, V, s, o);
    }
    free(K);
    free(V);
    free(s);
    return NULL;
}

static int run_job(attn_problem *P, const int32_t *rows, int n_rows, int mode,
                   double *out, int num_threads);

/* Listed rows (pairs (b, h)), or every (b, h) when rows is NULL. */
static int run_rows(attn_problem *P, const int32_t *rows, int n_rows, int mode,
                    double *out, int num_threads)
{
    return run_job(P, rows, rows ? n_rows : P->batch * P->num_q_heads, mode, out, num_threads);
}

/* Every (query token, head) row of a multi-token problem. */
static int run_rows_n(attn_problem *P, int n_rows, int mode, double *out, int num_threads)
{
    return run_job(P, NULL, n_rows, mode, out, num_threads);
}

static int valid_problem(const attn_problem *P)
{
    if (!P->q || !P->k_cache || !P->v_cache || !P->block_tables || !P->seq_lens)
        return 0;
    if (P->kv_kind != 0 && (!P->k_scale || !P->v_scale))
        return 0;
    if (P->batch < 0 || P->num_q_heads <= 0 || P->num_kv_heads <= 0 ||
        P->num_q_heads % P->num_kv_heads || P->head_dim <= 0 ||
        P->block_size <= 0 || P->max_blocks <= 0 || P->num_blocks <= 0)
        return 0;
    return 1;
}

static int run_job(attn_problem *P, const int32_t *rows, int n_rows, int mode,
                   double *out, int num_threads)
{
    if (!valid_problem(P) || !out)
        return OR_INVALID;
    row_job J;
    J.P = P;
    J.rows = rows;
    J.n_rows = n_rows;
    J.mode = mode;
    J.out = out;
    J.next = 0;
    J.status = OR_OK;
    pthread_mutex_init(&J.lock, NULL);
    if (num_threads < 1)
        num_threads = 1;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)num_threads);
    for (int i = 0; i < num_threads; ++i)
        pthread_create(&tid[i], NULL, row_worker, &J);
    for (int i = 0; i < num_threads; ++i)
        pthread_join(tid[i], NULL);
    free(tid);
    pthread_mutex_destroy(&J.lock);
    return J.status;
}

/* Attention for the listed query rows (pairs (b, h) in rows[2*n_rows], or
 * every (b, h) in b-major order when rows is NULL), fp64 output [n, d].
 * mode 0 = three-pass softmax (the oracle), 1 = online recurrence. */
int oracle_paged_attention(double *out, const uint16_t *q, const void *k_cache,
                           const void *v_cache, const float *k_scale,
                           const float *v_scale, int kv_kind,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *seq_lens, int batch, int num_q_heads,
                           int num_kv_heads, int head_dim, int num_blocks,
                           int block_size, double scale, const int32_t *rows,
                           int n_rows, int mode, int num_threads)
{
    attn_problem P = {q, k_cache, v_cache, k_scale, v_scale, kv_kind,
                      block_tables, max_blocks_per_seq, seq_lens, batch,
                      num_q_heads, num_kv_heads, head_dim, num_blocks,
                      block_size, scale, NULL, 0};
    return run_rows(&P, rows, n_rows, mode, out, num_threads);
}

/* Partials of one query row (b, h) over partitions of `part` tokens:
 * ml[np][2] = (m_i, l_i), acc[np][d]; returns the partition count np, or a
 * negative value on error. */
int oracle_attention_partials(double *ml, double *acc, const uint16_t *q,
                              const void *k_cache, const void *v_cache,
                              const float *k_scale, const float *v_scale,
                              int kv_kind, const int32_t *block_tables,
                              int max_blocks_per_seq, const int32_t *seq_lens,
                              int batch, int num_q_heads, int num_kv_heads,
                              int head_dim, int num_blocks, int block_size,
                              double scale, int b, int h, int part)
{
    attn_problem P = {q, k_cache, v_cache, k_scale, v_scale, kv_kind,
                      block_tables, max_blocks_per_seq, seq_lens, batch,
                      num_q_heads, num_kv_heads, head_dim, num_blocks,
                      block_size, scale, NULL, 0};
    if (!valid_problem(&P) || part <= 0 || b < 0 || b >= batch || h < 0 ||
        h >= num_q_heads)
        return -OR_INVALID;
    if (check_sequence(&P, b) != OR_OK)
        return -OR_INDEX;
    int L = seq_lens[b], d = head_dim;
    double *K = (double *)malloc((size_t)L * d * sizeof(double));
    double *V = (double *)malloc((size_t)L * d * sizeof(double));
    double *s = (double *)malloc((size_t)L * sizeof(double));
    gather_kv(&P, b, h / (num_q_heads / num_kv_heads), seq_lens[b], K, V);
    partial_row(&P, b, h, K, V, s, part, ml, acc);
    free(K);
    free(V);
    free(s);
    return (L + part - 1) / part;
}

/* Log-sum-exp merge of np partials (natural-log domain):
 *   M = max_i m_i,  w_i = exp(m_i - M),  o = sum_i w_i acc_i / sum_i w_i l_i */
void oracle_lse_merge(const double *ml, const double *acc, int np, int head_dim,
                      double *out)
{
    double M = -INFINITY;
    for (int i = 0; i < np; ++i)
        if (ml[2 * i] > M)
            M = ml[2 * i];
    double den = 0.0;
    for (int e = 0; e < head_dim; ++e)
        out[e] = 0.0;
    for (int i = 0; i < np; ++i) {
        double w = exp(ml[2 * i] - M);
        den += w * ml[2 * i + 1];
        for (int e = 0; e < head_dim; ++e)
            out[e] += w * acc[(int64_t)i * head_dim + e];
    }
    for (int e = 0; e < head_dim; ++e)
        out[e] /= den;
}

/* Attention of multi-token queries (speculative verification, chunked
 * prefill: “让 Agent 跑得快”, §六 投机解码 -- the target model scores the
 * gamma draft tokens in one parallel pass instead of gamma decode steps).
 * Sequence b has n_b = query_start[b + 1] - query_start[b] query tokens,
 * already appended, the last n_b of its seq_lens[b] tokens; query token i
 * (q row query_start[b] + i) at position L_b - n_b + i attends, causally,
 * positions 0 .. L_b - n_b + i.  q: bf16 [num_tokens, Hq, d]; out fp64
 * [num_tokens, Hq, d], rows of bad sequences (length, table, offsets)
 * zeroed with return value OR_INDEX.  mode as for oracle_paged_attention. */
int oracle_paged_attention_multi(double *out, const uint16_t *q, const void *k_cache,
                                 const void *v_cache, const float *k_scale,
                                 const float *v_scale, int kv_kind,
                                 const int32_t *block_tables, int max_blocks_per_seq,
                                 const int32_t *seq_lens, const int32_t *query_start,
                                 int batch, int num_tokens, int num_q_heads,
                                 int num_kv_heads, int head_dim, int num_blocks,
                                 int block_size, double scale, int mode, int num_threads)
{
    if (!query_start || num_tokens < 0)
        return OR_INVALID;
    attn_problem P = {q, k_cache, v_cache, k_scale, v_scale, kv_kind,
                      block_tables, max_blocks_per_seq, seq_lens, batch,
                      num_q_heads, num_kv_heads, head_dim, num_blocks,
                      block_size, scale, query_start, num_tokens};
    return run_rows_n(&P, num_tokens * num_q_heads, mode, out, num_threads);
}
