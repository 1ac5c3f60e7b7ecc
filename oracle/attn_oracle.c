/*
 * attn_oracle.c -- fp64 CPU oracle for causal scaled dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or table with the CUDA library.
 *
 * What it computes (the method's plain definition, in double precision):
 *   "Profiling in PyTorch (Part 3)" retelling, section "Naive Attention",
 *   five-step list and the NaiveCausalAttention listing:
 *     1. scores = Q . K^T
 *     2. scores = scores * scale
 *     3. scores[j > i] = -inf            (causal mask; the diagonal is kept)
 *     4. attn = softmax(scores) over keys
 *     5. out = attn . V
 *   An optional block mask drops whole 128 x 128 (query tile, key tile) blocks
 *   as well -- the block-sparse attention the ai-manual.ru article gives as a
 *   reason for custom kernels (sections 4 and 7): key j is masked for query i
 *   when block_mask[h][i / 128][j / 128] == 0, h = 0 for a mask shared by all
 *   heads, else the query head.
 *   and the definition Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V from
 *   the ainews.cool article, section "technical deep dive".
 *   The fully-masked-row convention (output 0 instead of NaN) follows the
 *   same retelling's description of the SDPA math backend's _safe_softmax
 *   (section "The Math Backend").  It cannot arise for causal, Sq == Sk.
 *
 * The log-sum-exp output (natural log of sum_j exp(s_j), s_j the scaled and
 * masked scores) is not on the pages; it is the usual companion output of a
 * fused attention forward and is defined here as written above.
 *
 * The oracle works one query row at a time, so the [S,S] score matrix is
 * never held; within a row it performs the five steps in the order above,
 * each as its own loop.  A library primitive is not needed.
 *
 * Inputs are bf16 bit patterns (uint16) in [B,H,S,D] contiguous layout, the
 * same bits the GPU receives.  Widening bf16 -> double is exact.  A second
 * entry point takes FP8 E4M3 bit patterns (uint8) with one descale factor per
 * tensor (value = decoded code * descale, in double): the FP8 attention that
 * the ai-manual.ru article mentions for newer GPUs (section 6, "FP8 and BF16").
 *
 * Parity pins (tests/test_oracle_pins.py): library softmax / SDPA in float64,
 * closed forms (causal row 0, Q = 0 means, S = 1), key-shift and linearity
 * invariants, a hand-derived worked example, and row sums.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 bit pattern -> double.  A bf16 value is the top half of an IEEE-754
 * binary32, so shifting the 16 bits up gives the float exactly. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* FP8 E4M3 (the "fn" variant: no infinities) bit pattern -> double, exactly:
 * sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 holds the
 * subnormals m/8 * 2^-6; S.1111.111 is NaN. */
static double e4m3_bits_to_double(uint8_t b) {
    const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

enum { FMT_BF16 = 0, FMT_E4M3 = 1 };

typedef struct {
    const void *t[3];        /* q, k, v */
    int format;              /* FMT_BF16 or FMT_E4M3 */
    double descale[3];       /* FMT_E4M3: value = decoded code * descale */
    int B, Hq, Hkv, S, D;
    double scale;
    int causal;
    const uint8_t *block_mask; /* NULL, or [mask_heads][nt][nt], nt = ceil(S / 128) */
    int mask_heads;            /* 1 (shared by all heads) or Hq */
    const int64_t *rows; /* flat query-row ids, or NULL for all rows */
    int64_t nrows;
    double *out; /* [nrows, D] */
    double *lse; /* [nrows]    */
    int64_t begin, end;
    int status;
} oracle_job_t;

/* Element idx of tensor `which` (0 q, 1 k, 2 v) as a double. */
static double elem(const oracle_job_t *J, int which, int64_t idx) {
    if (J->format == FMT_BF16) return bf16_bits_to_double(((const uint16_t *)J->t[which])[idx]);
    return e4m3_bits_to_double(((const uint8_t *)J->t[which])[idx]) * J->descale[which];
}

/*
 * One query row: flat id r = (b*Hq + hq)*S + i.
 * GQA head mapping: contiguous groups of G = Hq/Hkv query heads share one
 * key/value head, hkv = hq / G (the grouped-query strategy named in the
 * ainews.cool strategy table; with Hkv == Hq it is plain multi-head).
 */
static void oracle_one_row(const oracle_job_t *J, int64_t r, double *s,
                           double *o_row, double *lse_out) {
    const int S = J->S, D = J->D;
    const int64_t i = r % S;
    const int64_t bh = r / S;
    const int64_t b = bh / J->Hq;
    const int64_t hq = bh % J->Hq;
    const int64_t G = J->Hq / J->Hkv;
    const int64_t hkv = hq / G;

    const int64_t qi = (bh * S + i) * (int64_t)D;              /* q_i */
    const int64_t kb = ((b * J->Hkv + hkv) * S) * (int64_t)D;  /* k_0 of this head */
    const int64_t vb = ((b * J->Hkv + hkv) * S) * (int64_t)D;  /* v_0 of this head */

    /* Step 1: scores_j = sum_d q_id * k_jd. */
    for (int64_t j = 0; j < S; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += elem(J, 0, qi + d) * elem(J, 1, kb + j * D + d);
        s[j] = acc;
    }
    /* Step 2: scale (multiply by the caller's scale). */
    for (int64_t j = 0; j < S; ++j) s[j] = s[j] * J->scale;
    /* Step 3: causal mask, keys after the query position get -inf. */
    if (J->causal)
        for (int64_t j = i + 1; j < S; ++j) s[j] = -INFINITY;
    /* ... and keys in a dropped block of the block mask. */
    if (J->block_mask) {
        const int64_t nt = (S + 127) / 128;
        const uint8_t *mrow = J->block_mask + ((J->mask_heads == 1 ? 0 : hq) * nt + i / 128) * nt;
        for (int64_t j = 0; j < S; ++j)
            if (mrow[j / 128] == 0) s[j] = -INFINITY;
    }
    /* Step 4: softmax over keys, max-subtracted ("safe") form. */
    double m = -INFINITY;
    for (int64_t j = 0; j < S; ++j)
        if (s[j] > m) m = s[j];
    if (m == -INFINITY) { /* every key masked: output 0, LSE -inf */
        for (int d = 0; d < D; ++d) o_row[d] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < S; ++j) {
        s[j] = exp(s[j] - m); /* exp(-inf) == 0 */
        l += s[j];
    }
    for (int64_t j = 0; j < S; ++j) s[j] = s[j] / l;
    /* Step 5: out_d = sum_j attn_j * v_jd. */
    for (int d = 0; d < D; ++d) o_row[d] = 0.0;
    for (int64_t j = 0; j < S; ++j) {
        if (s[j] == 0.0) continue; /* masked key contributes nothing */
        for (int d = 0; d < D; ++d) o_row[d] += s[j] * elem(J, 2, vb + j * D + d);
    }
    *lse_out = m + log(l);
}

static void *oracle_worker(void *arg) {
    oracle_job_t *J = (oracle_job_t *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)J->S);
    if (!s) {
        J->status = 1;
        return NULL;
    }
    for (int64_t n = J->begin; n < J->end; ++n) {
        int64_t r = J->rows ? J->rows[n] : n;
        oracle_one_row(J, r, s, J->out + n * (int64_t)J->D, J->lse + n);
    }
    free(s);
    J->status = 0;
    return NULL;
}

static int run_rows(const void *q, const void *k, const void *v, int format, const double descale[3],
                    int B, int Hq, int Hkv, int S, int D, float scale, int causal,
                    const uint8_t *block_mask, int mask_heads,
                    const int64_t *rows, int64_t nrows, double *out, double *lse, int nthreads) {
    if (!q || !k || !v || !out || !lse) return 1;
    if (block_mask && mask_heads != 1 && mask_heads != Hq) return 1;
    if (B < 1 || Hq < 1 || Hkv < 1 || S < 1 || D < 1 || Hq % Hkv != 0) return 1;
    const int64_t total = (int64_t)B * Hq * S;
    if (!rows && nrows != total) return 1;
    if (rows)
        for (int64_t n = 0; n < nrows; ++n)
            if (rows[n] < 0 || rows[n] >= total) return 1;
    if (nrows == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nrows) nthreads = (int)nrows;

    oracle_job_t *jobs = (oracle_job_t *)calloc((size_t)nthreads, sizeof(oracle_job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return 1;
    }
    int status = 0;
    for (int t = 0; t < nthreads; ++t) {
        oracle_job_t *J = &jobs[t];
        J->t[0] = q; J->t[1] = k; J->t[2] = v;
        J->format = format;
        for (int w = 0; w < 3; ++w) J->descale[w] = descale[w];
        J->B = B; J->Hq = Hq; J->Hkv = Hkv; J->S = S; J->D = D;
        J->scale = (double)scale;
        J->causal = causal ? 1 : 0;
        J->block_mask = block_mask; J->mask_heads = mask_heads;
        J->rows = rows; J->nrows = nrows;
        J->out = out; J->lse = lse;
        J->begin = nrows * t / nthreads;
        J->end = nrows * (t + 1) / nthreads;
        J->status = 1;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, oracle_worker, &jobs[t]) != 0) break;
        started = t;
    }
    /* threads that failed to start: run their share here */
    oracle_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
    for (int t = started + 1; t < nthreads; ++t) oracle_worker(&jobs[t]);
    for (int t = 0; t < nthreads; ++t) status |= jobs[t].status;
    free(jobs);
    free(tid);
    return status;
}

/*
 * oracle_attn_rows -- O and LSE for selected query rows (or all rows).
 *
 *   q [B,Hq,S,D], k/v [B,Hkv,S,D]: bf16 bit patterns, contiguous.
 *   rows: nrows flat ids (b*Hq + hq)*S + i, or NULL for every row in order
 *         (then nrows must equal B*Hq*S).
 *   out:  double [nrows, D];  lse: double [nrows] (natural log).
 *   nthreads: worker threads (>= 1).
 * Returns 0 on success, 1 on a bad argument or allocation failure.
 */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Hq,
                     int Hkv, int S, int D, float scale, int causal, const int64_t *rows,
                     int64_t nrows, double *out, double *lse, int nthreads) {
    const double one[3] = {1.0, 1.0, 1.0};
    return run_rows(q, k, v, FMT_BF16, one, B, Hq, Hkv, S, D, scale, causal, NULL, 1, rows, nrows,
                    out, lse, nthreads);
}

/*
 * oracle_attn_rows_masked -- oracle_attn_rows plus a block mask: uint8
 * [mask_heads][nt][nt], nt = ceil(S / 128), mask_heads 1 or Hq; 0 drops the
 * block.  Rows left without any key give O = 0 and LSE = -inf.
 */
int oracle_attn_rows_masked(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Hq,
                            int Hkv, int S, int D, float scale, int causal,
                            const uint8_t *block_mask, int mask_heads, const int64_t *rows,
                            int64_t nrows, double *out, double *lse, int nthreads) {
    const double one[3] = {1.0, 1.0, 1.0};
    if (!block_mask) return 1;
    return run_rows(q, k, v, FMT_BF16, one, B, Hq, Hkv, S, D, scale, causal, block_mask,
                    mask_heads, rows, nrows, out, lse, nthreads);
}

/*
 * oracle_attn_rows_e4m3 -- the same for FP8 E4M3 inputs (uint8 bit patterns);
 * the value of an element is its decoded code times the descale of its tensor.
 */
int oracle_attn_rows_e4m3(const uint8_t *q, const uint8_t *k, const uint8_t *v, float q_descale,
                          float k_descale, float v_descale, int B, int Hq, int Hkv, int S, int D,
                          float scale, int causal, const int64_t *rows, int64_t nrows,
                          double *out, double *lse, int nthreads) {
    const double ds[3] = {(double)q_descale, (double)k_descale, (double)v_descale};
    return run_rows(q, k, v, FMT_E4M3, ds, B, Hq, Hkv, S, D, scale, causal, NULL, 1, rows, nrows,
                    out, lse, nthreads);
}

/* Decodes n E4M3 codes to doubles (exposed so the decoding can be pinned). */
void oracle_e4m3_decode(const uint8_t *codes, int64_t n, double *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_bits_to_double(codes[i]);
}
