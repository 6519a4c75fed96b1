/*
 * pa_oracle.c -- plain float64 CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library,
 * its Python binding) may include, link or call this file; only the tests,
 * the smoke check and the CPU-baseline leg of the benchmark use it.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * What it computes, and where that is defined (page title + section):
 *
 *  [P1] "feat: add paged-attention monolithic decode-only AR foundation"
 *       (lucebox pull 555), sections Summary and Validation: one decode step
 *       of attention, one query token per head, K/V rows gathered through a
 *       per-sequence block table of fixed-size blocks; GQA (one K/V head
 *       serves a group of query heads); F16 / Q8_0 / Q4_0 K/V; Q quantised
 *       once per step to q8_1 for the quantised-K dot products; context split
 *       into partitions whose normalised partials are merged by a stable
 *       split-softmax (log-sum-exp) merge; empty sequences supported.
 *  [P4] "fix(paged-attention): use 64-bit pool offsets in the fused decode
 *       kernels" (mlxcel issue 2153), sections Current Behavior and Proposed
 *       Solution: the pool row offset ((row * block_size + slot) * stride +
 *       kv_head * dim), widened to 64 bits before the multiply.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - softmax scale is supplied by the caller (1/sqrt(D) in every workload);
 *    no soft-cap, ALiBi, sinks or window;
 *  - query head h reads K/V head h / G, G = Hq / Hkv (consecutive query heads
 *    share a K/V head);
 *  - Q4_0 block (18 bytes): f16 d, then 16 bytes qs; element j < 16 is the low
 *    nibble of qs[j], element j + 16 the high nibble; value (nibble - 8) * d;
 *  - Q8_0 block (34 bytes): f16 d, then 32 int8 q; value q * d;
 *  - q8_1 block (36 bytes): f16 d, f16 s, then 32 int8 q; value q * d; the
 *    quantiser works in float32: amax = max|x|, d = amax / 127, q =
 *    clamp(roundf(x / d), -127, 127) (roundf: half away from zero; x / d an
 *    IEEE float division), d = q = 0 for an all-zero block; stored d =
 *    f16_rn(d), s = f16_rn(d * sum(q));
 *  - for F16 K the query is used unquantised (float32 widened to float64);
 *  - an empty sequence (length 0) gives an all-zero output;
 *  - a block-table entry outside [0, n_pool_blocks) is a corrupt table: the
 *    oracle refuses with OR_ERR_CORRUPT and writes nothing for that unit.
 *
 * Everything below is written as loops over the definition, in float64,
 * without blocking, fusion or reordering beyond what the definition states.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F16 0
#define OR_Q8_0 1
#define OR_Q4_0 2

#define OR_OK 0
#define OR_ERR_INVALID (-1)
#define OR_ERR_NOMEM (-2)
#define OR_ERR_CORRUPT (-5)

/* ---------------------------------------------------------------- formats */

/* IEEE binary16 bits -> double (exact). */
double or_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* float -> IEEE binary16 bits, round to nearest, ties to even. */
uint16_t or_float_to_half_rn(float xf)
{
    double x = (double)xf;
    uint16_t sign = 0;
    if (isnan(x))
        return 0x7e00;
    if (signbit(x)) {
        sign = 0x8000;
        x = -x;
    }
    if (x >= 65520.0) /* half-way between 65504 and 2^16 rounds to even: inf */
        return sign | 0x7c00;
    if (x < ldexp(1.0, -14)) {
        /* subnormal range: a multiple of 2^-24; rint() rounds ties to even */
        double m = rint(ldexp(x, 24));
        return sign | (uint16_t)m; /* m == 1024 encodes the smallest normal */
    }
    int k;
    frexp(x, &k);   /* x = f * 2^k, f in [0.5, 1) */
    int E = k - 1;  /* x in [2^E, 2^(E+1)) */
    double m = rint(ldexp(x, 10 - E)); /* in [1024, 2048] */
    if (m >= 2048.0) {
        m = 1024.0;
        E += 1;
    }
    if (E + 15 >= 31)
        return sign | 0x7c00;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)m - 1024));
}

static uint16_t rd16(const uint8_t *p)
{
    return (uint16_t)(p[0] | (p[1] << 8)); /* little-endian, as stored */
}

uint64_t or_row_bytes(int type, uint32_t D)
{
    switch (type) {
    case OR_F16: return 2ull * D;
    case OR_Q8_0: return (uint64_t)(D / 32) * 34ull;
    case OR_Q4_0: return (uint64_t)(D / 32) * 18ull;
    default: return 0;
    }
}

/* Dequantise one K or V row of D values into out[D]. */
void or_dequant_row(int type, const uint8_t *row, uint32_t D, double *out)
{
    if (type == OR_F16) {
        for (uint32_t i = 0; i < D; ++i)
            out[i] = or_half_to_double(rd16(row + 2 * i));
    } else if (type == OR_Q8_0) {
        for (uint32_t b = 0; b < D / 32; ++b) {
            const uint8_t *blk = row + 34 * b;
            double d = or_half_to_double(rd16(blk));
            for (int j = 0; j < 32; ++j)
                out[32 * b + j] = (double)(int8_t)blk[2 + j] * d;
        }
    } else if (type == OR_Q4_0) {
        for (uint32_t b = 0; b < D / 32; ++b) {
            const uint8_t *blk = row + 18 * b;
            double d = or_half_to_double(rd16(blk));
            for (int j = 0; j < 16; ++j) {
                int lo = blk[2 + j] & 0x0f;
                int hi = blk[2 + j] >> 4;
                out[32 * b + j] = (double)(lo - 8) * d;
                out[32 * b + j + 16] = (double)(hi - 8) * d;
            }
        }
    }
}

/* q8_1 quantiser: n_rows rows of D float32 values -> n_rows * D/32 blocks of
 * 36 bytes.  All arithmetic in float32, exactly as the definition states. */
int or_quantize_q8_1(const float *x, uint8_t *out, int64_t n_rows, uint32_t D)
{
    if (D == 0 || D % 32 != 0 || n_rows < 0)
        return OR_ERR_INVALID;
    int64_t n_blocks = n_rows * (int64_t)(D / 32);
    for (int64_t bi = 0; bi < n_blocks; ++bi) {
        const float *xb = x + 32 * bi;
        uint8_t *ob = out + 36 * bi;
        float amax = 0.0f;
        for (int j = 0; j < 32; ++j) {
            float a = fabsf(xb[j]);
            if (a > amax)
                amax = a;
        }
        float d = amax / 127.0f;
        int sum = 0;
        int8_t q[32];
        for (int j = 0; j < 32; ++j) {
            int v = 0;
            if (amax != 0.0f) {
                float r = roundf(xb[j] / d);
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                v = (int)r;
            }
            q[j] = (int8_t)v;
            sum += v;
        }
        if (amax == 0.0f)
            d = 0.0f;
        uint16_t d16 = or_float_to_half_rn(d);
        uint16_t s16 = or_float_to_half_rn(d * (float)sum);
        ob[0] = (uint8_t)(d16 & 0xff);
        ob[1] = (uint8_t)(d16 >> 8);
        ob[2] = (uint8_t)(s16 & 0xff);
        ob[3] = (uint8_t)(s16 >> 8);
        memcpy(ob + 4, q, 32);
    }
    return OR_OK;
}

/* Pool-row quantisers of the K/V append step ("feat: add paged-attention
 * monolithic decode-only AR foundation" (lucebox pull 555), Summary: the new
 * token's K/V rows are written into the pool next to which the paging
 * metadata stays resident; the block formats are those above).  The pages
 * give the formats, not the rounding, so this takes the ggml reference
 * convention, every step in float32 in this order:
 *  Q8_0: amax = max|x|; d = amax / 127; id = 1 / d (0 when d is 0);
 *        q = clamp(roundf(x * id), -127, 127); stored f16_rn(d).
 *  Q4_0: m = the first value of largest magnitude, with its sign; d = m / -8;
 *        id = 1 / d (0 when d is 0); nib = min(15, floor(x * id + 8.5));
 *        stored f16_rn(d), value j < 16 in the low half of byte j, value
 *        j + 16 in its high half.
 *  F16:  f16_rn(x).
 * out receives or_row_bytes(type, D) bytes. */
int or_quantize_row(int type, const float *x, uint32_t D, uint8_t *out)
{
    if (D == 0 || D % 32 != 0)
        return OR_ERR_INVALID;
    if (type == OR_F16) {
        for (uint32_t i = 0; i < D; ++i) {
            uint16_t h = or_float_to_half_rn(x[i]);
            out[2 * i] = (uint8_t)(h & 0xff);
            out[2 * i + 1] = (uint8_t)(h >> 8);
        }
        return OR_OK;
    }
    for (uint32_t b = 0; b < D / 32; ++b) {
        const float *xb = x + 32 * b;
        if (type == OR_Q8_0) {
            uint8_t *ob = out + 34 * b;
            float amax = 0.0f;
            for (int j = 0; j < 32; ++j) {
                float a = fabsf(xb[j]);
                if (a > amax)
                    amax = a;
            }
            float d = amax / 127.0f;
            float id = d > 0.0f ? 1.0f / d : 0.0f;
            for (int j = 0; j < 32; ++j) {
                float t = xb[j] * id;
                float r = roundf(t);
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                ob[2 + j] = (uint8_t)(int8_t)(int)r;
            }
            uint16_t d16 = or_float_to_half_rn(d);
            ob[0] = (uint8_t)(d16 & 0xff);
            ob[1] = (uint8_t)(d16 >> 8);
        } else if (type == OR_Q4_0) {
            uint8_t *ob = out + 18 * b;
            /* the first of equal magnitudes wins, so an all-zero block takes
               x[0] itself (its sign included) */
            float m = xb[0], amax = fabsf(xb[0]);
            for (int j = 1; j < 32; ++j) {
                float a = fabsf(xb[j]);
                if (a > amax) {
                    amax = a;
                    m = xb[j];
                }
            }
            float d = m / -8.0f;
            float id = d != 0.0f ? 1.0f / d : 0.0f;
            uint8_t nib[32];
            for (int j = 0; j < 32; ++j) {
                float t = xb[j] * id;
                t = t + 8.5f;
                float f = floorf(t);
                if (f > 15.0f) f = 15.0f;
                if (f < 0.0f) f = 0.0f;
                nib[j] = (uint8_t)(int)f;
            }
            uint16_t d16 = or_float_to_half_rn(d);
            ob[0] = (uint8_t)(d16 & 0xff);
            ob[1] = (uint8_t)(d16 >> 8);
            for (int j = 0; j < 16; ++j)
                ob[2 + j] = (uint8_t)(nib[j] | (nib[j + 16] << 4));
        } else {
            return OR_ERR_INVALID;
        }
    }
    return OR_OK;
}

/* Dequantise one q8_1 row (D/32 blocks) into out[D]: q * d. */
void or_dequant_q8_1_row(const uint8_t *blocks, uint32_t D, double *out)
{
    for (uint32_t b = 0; b < D / 32; ++b) {
        const uint8_t *blk = blocks + 36 * b;
        double d = or_half_to_double(rd16(blk));
        for (int j = 0; j < 32; ++j)
            out[32 * b + j] = (double)(int8_t)blk[4 + j] * d;
    }
}

/* Byte offset of the row (block, slot, kv_head) in a token-major pool
 * [n_blocks][block_size][hkv][row_bytes]; 64-bit before any multiply. */
uint64_t or_row_offset(int64_t block, uint32_t slot, uint32_t kv_head,
                       uint32_t block_size, uint32_t hkv, uint64_t row_bytes)
{
    uint64_t token_slot = (uint64_t)block * (uint64_t)block_size + (uint64_t)slot;
    return (token_slot * (uint64_t)hkv + (uint64_t)kv_head) * row_bytes;
}

/* --------------------------------------------------------------- attention */

typedef struct {
    const uint8_t *k_pool;
    const uint8_t *v_pool;
    uint64_t n_pool_blocks;
    const int32_t *block_table; /* [n_seqs][table_stride] */
    uint32_t table_stride;
    const int32_t *seq_lens;    /* [n_seqs] */
    const float *q;             /* [n_seqs][q_tokens][hq][d] float32 */
    double scale;
    uint32_t n_seqs, hq, hkv, d, block_size;
    int32_t k_type, v_type;
    uint32_t q_tokens;          /* query tokens per sequence (0 is read as 1) */
} or_args;

/* Query rows.  With T query tokens per sequence ("TensorFold pull 1418",
 * What: several query rows of a sequence -- a prompt chunk or a verify window
 * -- attend over the same paged cache), query row u is token i = u % T of
 * sequence s = u / T, at position L_s - T + i, and attends causally to the
 * keys 0 .. L_s - T + i: its length is L_s - T + 1 + i (none when that is not
 * positive).  T = 1 is the one-token decode step. */
static uint32_t n_tokens(const or_args *a) { return a->q_tokens > 1 ? a->q_tokens : 1; }

static uint32_t row_len(const or_args *a, uint32_t u)
{
    uint32_t T = n_tokens(a);
    int64_t L = (int64_t)a->seq_lens[u / T] - (int64_t)(T - 1 - u % T);
    return L > 0 ? (uint32_t)L : 0;
}

static int check_args(const or_args *a)
{
    if (!a || !a->k_pool || !a->v_pool || !a->block_table || !a->seq_lens || !a->q)
        return OR_ERR_INVALID;
    if (a->hkv == 0 || a->hq % a->hkv != 0 || a->d == 0 || a->d % 32 != 0 ||
        a->block_size == 0)
        return OR_ERR_INVALID;
    if (or_row_bytes(a->k_type, a->d) == 0 || or_row_bytes(a->v_type, a->d) == 0)
        return OR_ERR_INVALID;
    return OR_OK;
}

/* The query row that the dot products use: fp32 Q for F16 K, otherwise the
 * dequantised q8_1 quantisation of Q (quantised here by the oracle itself). */
static void query_row(const or_args *a, uint32_t u, uint32_t h, double *qhat)
{
    const float *qr = a->q + ((uint64_t)u * a->hq + h) * a->d;
    if (a->k_type == OR_F16) {
        for (uint32_t i = 0; i < a->d; ++i)
            qhat[i] = (double)qr[i];
    } else {
        uint8_t *blocks = (uint8_t *)malloc((size_t)(a->d / 32) * 36);
        or_quantize_q8_1(qr, blocks, 1, a->d);
        or_dequant_q8_1_row(blocks, a->d, qhat);
        free(blocks);
    }
}

/* Resolve token t of the sequence of query row u to the byte offset of its
 * kv_head row; -1 on a table entry outside the pool. */
static int token_row(const or_args *a, uint32_t u, uint32_t t, uint32_t g,
                     uint64_t row_bytes, uint64_t *off)
{
    uint32_t s = u / n_tokens(a);
    int32_t blk = a->block_table[(uint64_t)s * a->table_stride + t / a->block_size];
    if (blk < 0 || (uint64_t)blk >= a->n_pool_blocks)
        return -1;
    *off = or_row_offset(blk, t % a->block_size, g, a->block_size, a->hkv, row_bytes);
    return 0;
}

/* Scores s_t = scale * <qhat, khat_t> for t in [t0, t1). */
static int scores(const or_args *a, uint32_t s, uint32_t h, const double *qhat,
                  uint32_t t0, uint32_t t1, double *sc, double *row)
{
    uint32_t g = h / (a->hq / a->hkv);
    uint64_t krb = or_row_bytes(a->k_type, a->d);
    for (uint32_t t = t0; t < t1; ++t) {
        uint64_t off;
        if (token_row(a, s, t, g, krb, &off))
            return OR_ERR_CORRUPT;
        or_dequant_row(a->k_type, a->k_pool + off, a->d, row);
        double acc = 0.0;
        for (uint32_t i = 0; i < a->d; ++i)
            acc += qhat[i] * row[i];
        sc[t - t0] = a->scale * acc;
    }
    return OR_OK;
}

/* One (query row, query head) unit: out[d] = sum_t softmax(s)_t * vhat_t. */
static int decode_unit(const or_args *a, uint32_t s, uint32_t h, double *out)
{
    uint32_t L = row_len(a, s);
    uint32_t D = a->d;
    for (uint32_t i = 0; i < D; ++i)
        out[i] = 0.0;
    if (L == 0)
        return OR_OK; /* empty sequence: zero output */
    double *qhat = (double *)malloc(sizeof(double) * D);
    double *row = (double *)malloc(sizeof(double) * D);
    double *sc = (double *)malloc(sizeof(double) * L);
    if (!qhat || !row || !sc) {
        free(qhat); free(row); free(sc);
        return OR_ERR_NOMEM;
    }
    query_row(a, s, h, qhat);
    int rc = scores(a, s, h, qhat, 0, L, sc, row);
    if (rc == OR_OK) {
        double mx = -INFINITY;
        for (uint32_t t = 0; t < L; ++t)
            if (sc[t] > mx) mx = sc[t];
        double z = 0.0;
        for (uint32_t t = 0; t < L; ++t) {
            sc[t] = exp(sc[t] - mx);
            z += sc[t];
        }
        uint32_t g = h / (a->hq / a->hkv);
        uint64_t vrb = or_row_bytes(a->v_type, D);
        for (uint32_t t = 0; t < L; ++t) {
            uint64_t off;
            token_row(a, s, t, g, vrb, &off);
            or_dequant_row(a->v_type, a->v_pool + off, D, row);
            double p = sc[t] / z;
            for (uint32_t i = 0; i < D; ++i)
                out[i] += p * row[i];
        }
    }
    free(qhat); free(row); free(sc);
    return rc;
}

/* Partitioned form of the same unit: partitions of part_tokens tokens each
 * give (m_p, l_p, o_p) with o_p normalised; they are combined by the
 * log-sum-exp merge.  Algebraically identical to decode_unit. */
static int decode_unit_partitioned(const or_args *a, uint32_t s, uint32_t h,
                                   uint32_t part_tokens, double *out)
{
    uint32_t L = row_len(a, s);
    uint32_t D = a->d;
    for (uint32_t i = 0; i < D; ++i)
        out[i] = 0.0;
    if (L == 0)
        return OR_OK;
    uint32_t n_parts = (L + part_tokens - 1) / part_tokens;
    double *qhat = (double *)malloc(sizeof(double) * D);
    double *row = (double *)malloc(sizeof(double) * D);
    double *sc = (double *)malloc(sizeof(double) * part_tokens);
    double *m = (double *)malloc(sizeof(double) * n_parts);
    double *l = (double *)malloc(sizeof(double) * n_parts);
    double *o = (double *)calloc((size_t)n_parts * D, sizeof(double));
    int rc = OR_OK;
    if (!qhat || !row || !sc || !m || !l || !o) {
        rc = OR_ERR_NOMEM;
        goto done;
    }
    query_row(a, s, h, qhat);
    uint32_t g = h / (a->hq / a->hkv);
    uint64_t vrb = or_row_bytes(a->v_type, D);
    for (uint32_t p = 0; p < n_parts; ++p) {
        uint32_t t0 = p * part_tokens;
        uint32_t t1 = t0 + part_tokens < L ? t0 + part_tokens : L;
        rc = scores(a, s, h, qhat, t0, t1, sc, row);
        if (rc != OR_OK)
            goto done;
        double mx = -INFINITY;
        for (uint32_t t = t0; t < t1; ++t)
            if (sc[t - t0] > mx) mx = sc[t - t0];
        double lp = 0.0;
        double *op = o + (size_t)p * D;
        for (uint32_t t = t0; t < t1; ++t) {
            double w = exp(sc[t - t0] - mx);
            lp += w;
            uint64_t off;
            token_row(a, s, t, g, vrb, &off);
            or_dequant_row(a->v_type, a->v_pool + off, D, row);
            for (uint32_t i = 0; i < D; ++i)
                op[i] += w * row[i];
        }
        for (uint32_t i = 0; i < D; ++i)
            op[i] /= lp;
        m[p] = mx;
        l[p] = lp;
    }
    /* merge: M = max m_p, w_p = l_p exp(m_p - M), O = sum w_p o_p / sum w_p */
    double M = -INFINITY;
    for (uint32_t p = 0; p < n_parts; ++p)
        if (m[p] > M) M = m[p];
    double wsum = 0.0;
    for (uint32_t p = 0; p < n_parts; ++p) {
        double w = l[p] * exp(m[p] - M);
        wsum += w;
        for (uint32_t i = 0; i < D; ++i)
            out[i] += w * o[(size_t)p * D + i];
    }
    for (uint32_t i = 0; i < D; ++i)
        out[i] /= wsum;
done:
    free(qhat); free(row); free(sc); free(m); free(l); free(o);
    return rc;
}

/* ---------------------------------------------------------- thread driver */

typedef struct {
    const or_args *a;
    const int32_t *units; /* pairs (query row, head) */
    int64_t n_units;
    uint32_t part_tokens; /* 0 = single pass */
    double *out;          /* [n_units][d] */
    int64_t next;
    int rc;
    pthread_mutex_t mu;
} job_t;

static void *worker(void *arg)
{
    job_t *j = (job_t *)arg;
    for (;;) {
        pthread_mutex_lock(&j->mu);
        int64_t u = j->next++;
        pthread_mutex_unlock(&j->mu);
        if (u >= j->n_units)
            break;
        uint32_t s = (uint32_t)j->units[2 * u];
        uint32_t h = (uint32_t)j->units[2 * u + 1];
        double *o = j->out + (size_t)u * j->a->d;
        int rc;
        if (s >= j->a->n_seqs * n_tokens(j->a) || h >= j->a->hq)
            rc = OR_ERR_INVALID;
        else if (j->part_tokens)
            rc = decode_unit_partitioned(j->a, s, h, j->part_tokens, o);
        else
            rc = decode_unit(j->a, s, h, o);
        if (rc != OR_OK) {
            pthread_mutex_lock(&j->mu);
            if (j->rc == OR_OK) j->rc = rc;
            pthread_mutex_unlock(&j->mu);
        }
    }
    return NULL;
}

/* Decode the listed (query row, head) units (the query row is the sequence
 * when there is one query token); part_tokens = 0 for the single-pass
 * definition, otherwise the partitioned form with that partition length. */
int or_decode_units(const or_args *a, const int32_t *units, int64_t n_units,
                    uint32_t part_tokens, double *out, int n_threads)
{
    int rc = check_args(a);
    if (rc != OR_OK)
        return rc;
    if (n_threads < 1)
        n_threads = 1;
    job_t j;
    j.a = a; j.units = units; j.n_units = n_units; j.part_tokens = part_tokens;
    j.out = out; j.next = 0; j.rc = OR_OK;
    pthread_mutex_init(&j.mu, NULL);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    int started = 0;
    for (int i = 0; i < n_threads; ++i)
        if (pthread_create(&th[i], NULL, worker, &j) == 0)
            started++;
        else
            break;
    if (started == 0)
        worker(&j);
    for (int i = 0; i < started; ++i)
        pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&j.mu);
    return j.rc;
}

/* ----------------------------------------------------------------- merge */

/* Merge of stored partials ([P1] Summary: partials stored normalised in f16,
 * combined by a stable split-softmax merge).  For each of n_units rows:
 * n_live partials, each an f16 row o_p (already divided by l_p), a running
 * max m_p in the log2 domain (scores pre-multiplied by log2 e) and a sum
 * l_p = sum_t 2^(s_t - m_p).  O = sum_p w_p o_p / sum_p w_p with
 * w_p = l_p 2^(m_p - M), M = max over partials with l_p > 0; partials with
 * l_p == 0 are dead and skipped; no live partial gives O = 0.
 * Layout: o [n_units][n_parts][d] f16 bits, ml [n_units][n_parts][2] float. */
int or_merge(const uint16_t *o, const float *ml, const int32_t *n_live,
             int64_t n_units, uint32_t n_parts, uint32_t d, double *out)
{
    for (int64_t u = 0; u < n_units; ++u) {
        double *ou = out + (size_t)u * d;
        for (uint32_t i = 0; i < d; ++i)
            ou[i] = 0.0;
        int32_t nl = n_live[u];
        if (nl < 0 || (uint32_t)nl > n_parts)
            return OR_ERR_INVALID;
        double M = -INFINITY;
        for (int32_t p = 0; p < nl; ++p) {
            const float *mlp = ml + ((size_t)u * n_parts + p) * 2;
            if (mlp[1] > 0.0f && (double)mlp[0] > M)
                M = (double)mlp[0];
        }
        if (M == -INFINITY)
            continue;
        double wsum = 0.0;
        for (int32_t p = 0; p < nl; ++p) {
            const float *mlp = ml + ((size_t)u * n_parts + p) * 2;
            if (!(mlp[1] > 0.0f))
                continue;
            double w = (double)mlp[1] * exp2((double)mlp[0] - M);
            wsum += w;
            const uint16_t *op = o + ((size_t)u * n_parts + p) * d;
            for (uint32_t i = 0; i < d; ++i)
                ou[i] += w * or_half_to_double(op[i]);
        }
        for (uint32_t i = 0; i < d; ++i)
            ou[i] /= wsum;
    }
    return OR_OK;
}

/* max |Vhat| over the live rows the listed (seq, head) units read: the scale
 * of the accuracy gate (max|err| <= tol * max|V| over the live tokens). */
int or_vmax_units(const or_args *a, const int32_t *units, int64_t n_units, double *vmax)
{
    int rc = check_args(a);
    if (rc != OR_OK)
        return rc;
    double *row = (double *)malloc(sizeof(double) * a->d);
    if (!row)
        return OR_ERR_NOMEM;
    uint64_t vrb = or_row_bytes(a->v_type, a->d);
    double mx = 0.0;
    for (int64_t u = 0; u < n_units; ++u) {
        uint32_t s = (uint32_t)units[2 * u], h = (uint32_t)units[2 * u + 1];
        if (s >= a->n_seqs * n_tokens(a) || h >= a->hq) {
            free(row);
            return OR_ERR_INVALID;
        }
        uint32_t g = h / (a->hq / a->hkv);
        int32_t L = (int32_t)row_len(a, s);
        for (int32_t t = 0; t < L; ++t) {
            uint64_t off;
            if (token_row(a, s, (uint32_t)t, g, vrb, &off)) {
                free(row);
                return OR_ERR_CORRUPT;
            }
            or_dequant_row(a->v_type, a->v_pool + off, a->d, row);
            for (uint32_t i = 0; i < a->d; ++i)
                if (fabs(row[i]) > mx) mx = fabs(row[i]);
        }
    }
    free(row);
    *vmax = mx;
    return OR_OK;
}
