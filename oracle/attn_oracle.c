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
 *   heads, else the query head.  An optional element mask (the arbitrary
 *   masks of the same sections) drops single (query, key) pairs: key j is
 *   masked for query i when bit j % 8 of byte j / 8 of row i of the mask is
 *   0, rows 16 * ceil(S / 128) bytes apart, one bit matrix shared by all
 *   heads or one per query head.  The masks combine: a key is visible only
 *   when every mask given keeps it.
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
 * The gradients of the same function (dQ, dK, dV for an upstream dO) are
 * defined and computed at the end of this file (oracle_attn_bwd).
 *
 * Parity pins (tests/test_oracle_pins.py): library softmax / SDPA in float64,
 * closed forms (causal row 0, Q = 0 means, S = 1), key-shift and linearity
 * invariants, a hand-derived worked example, and row sums.  The gradients:
 * central finite differences of the forward oracle on double inputs, torch's
 * float64 autograd, closed forms (dQ of causal row 0, column sums of dK and
 * dV, dV for Q = 0) and invariants (key shift, linearity in dO).
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

/* Element formats: bf16 bit patterns (the GPU's inputs), E4M3 codes, or
 * plain doubles (used by the finite-difference pins of the gradients). */
enum { FMT_BF16 = 0, FMT_E4M3 = 1, FMT_F64 = 2 };

typedef struct {
    const void *t[4];        /* q, k, v, and dO for the gradients */
    int format;              /* FMT_BF16, FMT_E4M3 or FMT_F64 */
    double descale[4];       /* FMT_E4M3: value = decoded code * descale */
    int B, Hq, Hkv, S, D;
    double scale;
    int causal;
    const uint8_t *block_mask; /* NULL, or [mask_heads][nt][nt], nt = ceil(S / 128) */
    int mask_heads;            /* 1 (shared by all heads) or Hq */
    const uint8_t *keep_bits;  /* NULL, or [keep_heads][S][16 * nt] bytes, bit j % 8 of byte j / 8 keeps key j */
    int keep_heads;            /* 1 (shared by all heads) or Hq */
    int dropout_p8;            /* 0: no dropout; else weights dropped with probability p8 / 256 */
    uint64_t dropout_seed;     /* Philox key (two 32-bit words) */
    uint64_t dropout_offset;   /* fourth Philox counter word, < 2^32 */
    const int64_t *rows; /* flat query-row ids, or NULL for all rows */
    int64_t nrows;
    double *out; /* [nrows, D] */
    double *lse; /* [nrows]    */
    int64_t begin, end;
    int status;
} oracle_job_t;

/* Element idx of tensor `which` (0 q, 1 k, 2 v, 3 dO) as a double. */
static double elem(const oracle_job_t *J, int which, int64_t idx) {
    if (J->format == FMT_BF16) return bf16_bits_to_double(((const uint16_t *)J->t[which])[idx]);
    if (J->format == FMT_F64) return ((const double *)J->t[which])[idx];
    return e4m3_bits_to_double(((const uint8_t *)J->t[which])[idx]) * J->descale[which];
}

/*
 * Steps 1-4 for one query row, flat id r = (b*Hq + hq)*S + i: on return s[j]
 * holds the attention weight of key j (0 where masked) and *lse_out the
 * log-sum-exp of the scaled, masked scores (-inf when every key is masked,
 * and then every weight is 0).
 * GQA head mapping: contiguous groups of G = Hq/Hkv query heads share one
 * key/value head, hkv = hq / G (the grouped-query strategy named in the
 * ainews.cool strategy table; with Hkv == Hq it is plain multi-head).
 */
static void attn_weights(const oracle_job_t *J, int64_t r, double *s, double *lse_out) {
    const int S = J->S, D = J->D;
    const int64_t i = r % S;
    const int64_t bh = r / S;
    const int64_t b = bh / J->Hq;
    const int64_t hq = bh % J->Hq;
    const int64_t G = J->Hq / J->Hkv;
    const int64_t hkv = hq / G;

    const int64_t qi = (bh * S + i) * (int64_t)D;              /* q_i */
    const int64_t kb = ((b * J->Hkv + hkv) * S) * (int64_t)D;  /* k_0 of this head */

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
    /* ... and keys whose bit in the element mask is 0. */
    if (J->keep_bits) {
        const int64_t row_bytes = 16 * ((S + 127) / 128);
        const uint8_t *krow = J->keep_bits + ((J->keep_heads == 1 ? 0 : hq) * (int64_t)S + i) * row_bytes;
        for (int64_t j = 0; j < S; ++j)
            if (((krow[j / 8] >> (j % 8)) & 1) == 0) s[j] = -INFINITY;
    }
    /* Step 4: softmax over keys, max-subtracted ("safe") form. */
    double m = -INFINITY;
    for (int64_t j = 0; j < S; ++j)
        if (s[j] > m) m = s[j];
    if (m == -INFINITY) { /* every key masked: all weights 0, LSE -inf */
        for (int64_t j = 0; j < S; ++j) s[j] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < S; ++j) {
        s[j] = exp(s[j] - m); /* exp(-inf) == 0 */
        l += s[j];
    }
    for (int64_t j = 0; j < S; ++j) s[j] = s[j] / l;
    *lse_out = m + log(l);
}

/*
 * Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
 * easy as 1, 2, 3", SC 2011), the 32-bit-word variant: ten rounds of
 *   (x0, x1, x2, x3) <- (hi(M1 x2) ^ x1 ^ k0, lo(M1 x2), hi(M0 x0) ^ x3 ^ k1, lo(M0 x0))
 * with 32 x 32 -> 64-bit products split into high and low words, and the key
 * bumped by the Weyl constants (golden ratio, sqrt(3) - 1) after every round.
 */
static void philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    const uint64_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3], k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = M0 * (uint64_t)x0;
        const uint64_t p1 = M1 * (uint64_t)x2;
        const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        x0 = hi1 ^ x1 ^ k0;
        x1 = lo1;
        x2 = hi0 ^ x3 ^ k1;
        x3 = lo0;
        k0 += W0;
        k1 += W1;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/*
 * Dropout of the attention weights (the fused dropout the ai-manual.ru
 * article names in section 6, "Dropout"; the weights are dropped after the
 * softmax and the kept ones scaled by 1 / (1 - p), as in
 * scaled_dot_product_attention).  The random draw is Philox4x32-10 with
 * counter {j / 16, i, b*Hq + hq, offset} and key {seed mod 2^32, seed / 2^32}:
 * its 16 output bytes (word 0 first, each word little-endian) give keys
 * j = 16*(j/16) + 0..15 of query row i.  Key j is kept when its byte is
 * >= p8 (probability 1 - p8/256) and then scaled by 256 / (256 - p8).
 */
static int dropout_keeps(const oracle_job_t *J, int64_t bh, int64_t i, int64_t j) {
    const uint32_t ctr[4] = {(uint32_t)(j / 16), (uint32_t)i, (uint32_t)bh, (uint32_t)J->dropout_offset};
    const uint32_t key[2] = {(uint32_t)(J->dropout_seed & 0xFFFFFFFFu), (uint32_t)(J->dropout_seed >> 32)};
    uint32_t out[4];
    philox4x32_10(ctr, key, out);
    const int byte = (int)((out[(j % 16) / 4] >> (8 * (j % 4))) & 0xFF);
    return byte >= J->dropout_p8;
}

/* One query row of the forward pass: steps 1-4, then step 5. */
static void oracle_one_row(const oracle_job_t *J, int64_t r, double *s,
                           double *o_row, double *lse_out) {
    const int S = J->S, D = J->D;
    const int64_t i = r % S;
    const int64_t b = (r / S) / J->Hq;
    const int64_t hkv = ((r / S) % J->Hq) / (J->Hq / J->Hkv);
    const int64_t vb = ((b * J->Hkv + hkv) * S) * (int64_t)D;  /* v_0 of this head */
    attn_weights(J, r, s, lse_out);
    /* Optional dropout of the weights (the LSE is that of the kept softmax). */
    if (J->dropout_p8 > 0) {
        const double keep_scale = 256.0 / (256.0 - (double)J->dropout_p8);
        for (int64_t j = 0; j < S; ++j) {
            if (s[j] == 0.0) continue;
            s[j] = dropout_keeps(J, r / S, i, j) ? s[j] * keep_scale : 0.0;
        }
    }
    /* Step 5: out_d = sum_j attn_j * v_jd (every weight 0 when all keys are masked). */
    for (int d = 0; d < D; ++d) o_row[d] = 0.0;
    for (int64_t j = 0; j < S; ++j) {
        if (s[j] == 0.0) continue; /* masked key contributes nothing */
        for (int d = 0; d < D; ++d) o_row[d] += s[j] * elem(J, 2, vb + j * D + d);
    }
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

static int run_rows_dropout(const void *q, const void *k, const void *v, int format,
                            const double descale[3], int B, int Hq, int Hkv, int S, int D,
                            float scale, int causal, const uint8_t *block_mask, int mask_heads,
                            const uint8_t *keep_bits, int keep_heads, int dropout_p8, uint64_t seed,
                            uint64_t offset, const int64_t *rows, int64_t nrows, double *out,
                            double *lse, int nthreads) {
    if (!q || !k || !v || !out || !lse) return 1;
    if (block_mask && mask_heads != 1 && mask_heads != Hq) return 1;
    if (keep_bits && keep_heads != 1 && keep_heads != Hq) return 1;
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
        J->t[0] = q; J->t[1] = k; J->t[2] = v; J->t[3] = NULL;
        J->format = format;
        for (int w = 0; w < 3; ++w) J->descale[w] = descale[w];
        J->descale[3] = 1.0;
        J->B = B; J->Hq = Hq; J->Hkv = Hkv; J->S = S; J->D = D;
        J->scale = (double)scale;
        J->causal = causal ? 1 : 0;
        J->block_mask = block_mask; J->mask_heads = mask_heads;
        J->keep_bits = keep_bits; J->keep_heads = keep_heads;
        J->dropout_p8 = dropout_p8;
        J->dropout_seed = seed; J->dropout_offset = offset;
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

static int run_rows(const void *q, const void *k, const void *v, int format, const double descale[3],
                    int B, int Hq, int Hkv, int S, int D, float scale, int causal,
                    const uint8_t *block_mask, int mask_heads,
                    const int64_t *rows, int64_t nrows, double *out, double *lse, int nthreads) {
    return run_rows_dropout(q, k, v, format, descale, B, Hq, Hkv, S, D, scale, causal, block_mask,
                            mask_heads, NULL, 1, 0, 0, 0, rows, nrows, out, lse, nthreads);
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
 * oracle_attn_rows_keep -- oracle_attn_rows plus an element mask: keep_bits
 * uint8 [keep_heads][S][16 * ceil(S / 128)], keep_heads 1 or Hq; bit j % 8 of
 * byte j / 8 of row i keeps key j for query i.  block_mask (optional, NULL
 * for none) as in oracle_attn_rows_masked.  Rows left without any key give
 * O = 0 and LSE = -inf.
 */
int oracle_attn_rows_keep(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Hq,
                          int Hkv, int S, int D, float scale, int causal, const uint8_t *keep_bits,
                          int keep_heads, const uint8_t *block_mask, int mask_heads,
                          const int64_t *rows, int64_t nrows, double *out, double *lse,
                          int nthreads) {
    const double one[3] = {1.0, 1.0, 1.0};
    if (!keep_bits) return 1;
    return run_rows_dropout(q, k, v, FMT_BF16, one, B, Hq, Hkv, S, D, scale, causal, block_mask,
                            block_mask ? mask_heads : 1, keep_bits, keep_heads, 0, 0, 0, rows,
                            nrows, out, lse, nthreads);
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

/*
 * oracle_attn_rows_f64 -- oracle_attn_rows on double inputs (no rounding of
 * the inputs at all); the finite-difference pins of the gradients use it.
 */
int oracle_attn_rows_f64(const double *q, const double *k, const double *v, int B, int Hq, int Hkv,
                         int S, int D, float scale, int causal, const int64_t *rows, int64_t nrows,
                         double *out, double *lse, int nthreads) {
    const double one[3] = {1.0, 1.0, 1.0};
    return run_rows(q, k, v, FMT_F64, one, B, Hq, Hkv, S, D, scale, causal, NULL, 1, rows, nrows,
                    out, lse, nthreads);
}

/* ======================================================================
 * Gradients (backward pass).
 *
 * The ai-manual.ru article (section 6, "gradients and backward") warns that
 * the fused backward pass is the hard part to get right; the pages give no
 * formula, so the oracle is the plain definition: the gradients of the
 * forward function above with respect to Q, K and V for an upstream gradient
 * dO of the output.  With P_ij the attention weight of key j for query i
 * (steps 1-4; 0 where masked) and O_i = sum_j P_ij V_j, differentiating
 * steps 5, 4 and 1-2 in turn gives, per query head:
 *   dV_j    = sum_i P_ij dO_i
 *   dP_ij   = dO_i . V_j
 *   delta_i = sum_k P_ik dP_ik
 *   dS_ij   = P_ij (dP_ij - delta_i)          (softmax Jacobian applied to dP)
 *   dQ_i    = scale * sum_j dS_ij K_j
 *   dK_j    = scale * sum_i dS_ij Q_i
 * and a key/value head's dK and dV add up the contributions of every query
 * head of its group.  Masked pairs have P_ij = 0, hence dS_ij = 0.  With
 * dropout (oracle_attn_bwd_dropout) the output uses P_ij Z_ij s instead of
 * P_ij, so dV_j = sum_i P_ij Z_ij s dO_i and dP_ij = Z_ij s (dO_i . V_j).
 *
 * Work per selected key/value head (b, hkv): pass 1, one query row at a time
 * (any order, rows independent), stores the rows of P and dS of all G query
 * heads of the group and writes dQ and delta; pass 2, one key at a time,
 * sums dK_j and dV_j over query heads and rows in ascending order, so the
 * result does not depend on the number of threads.
 * ====================================================================== */
typedef struct {
    const oracle_job_t *J;
    int64_t b, hkv, G;
    double *P, *dS;            /* [G*S][S] rows of weights and score gradients */
    double *dq, *dk, *dv;      /* [G][S][D], [S][D], [S][D] of this head */
    double *delta;             /* [G][S] */
    int pass;
    int64_t begin, end;
    int status;
} bwd_job_t;

/* Pass 1 for row n = g*S + i of the group: P, dP, delta, dS, dQ. */
static void bwd_row(const bwd_job_t *W, int64_t n, double *dP) {
    const oracle_job_t *J = W->J;
    const int S = J->S, D = J->D;
    const int64_t g = n / S, i = n % S;
    const int64_t hq = W->hkv * W->G + g;
    const int64_t bh = W->b * J->Hq + hq;
    const int64_t qo = (bh * S + i) * (int64_t)D;                   /* q_i and dO_i */
    const int64_t kvb = ((W->b * J->Hkv + W->hkv) * S) * (int64_t)D; /* k_0, v_0 */
    double *p = W->P + n * S, *ds = W->dS + n * S;
    double lse;
    attn_weights(J, bh * S + i, p, &lse);
    /* dP_ij = dO_i . V_j (only where P_ij != 0: elsewhere dS_ij = 0 anyway). */
    for (int64_t j = 0; j < S; ++j) {
        dP[j] = 0.0;
        if (p[j] == 0.0) continue;
        for (int d = 0; d < D; ++d) dP[j] += elem(J, 3, qo + d) * elem(J, 2, kvb + j * D + d);
    }
    /* With dropout the output uses the weights P_ij Z_ij s (Z_ij the keep
     * decision, s = 256 / (256 - p8)), so the gradient reaching P_ij is
     * Z_ij s (dO_i . V_j). */
    if (J->dropout_p8 > 0) {
        const double keep_scale = 256.0 / (256.0 - (double)J->dropout_p8);
        for (int64_t j = 0; j < S; ++j)
            if (p[j] != 0.0) dP[j] = dropout_keeps(J, bh, i, j) ? dP[j] * keep_scale : 0.0;
    }
    /* delta_i = sum_k P_ik dP_ik. */
    double delta = 0.0;
    for (int64_t j = 0; j < S; ++j) delta += p[j] * dP[j];
    /* dS_ij = P_ij (dP_ij - delta_i). */
    for (int64_t j = 0; j < S; ++j) ds[j] = p[j] * (dP[j] - delta);
    /* dQ_i = scale * sum_j dS_ij K_j. */
    double *dq = W->dq + n * (int64_t)D;
    for (int d = 0; d < D; ++d) dq[d] = 0.0;
    for (int64_t j = 0; j < S; ++j) {
        if (ds[j] == 0.0) continue;
        for (int d = 0; d < D; ++d) dq[d] += ds[j] * elem(J, 1, kvb + j * D + d);
    }
    for (int d = 0; d < D; ++d) dq[d] *= J->scale;
    W->delta[n] = delta;
}

/* Pass 2 for key j: dK_j and dV_j summed over the group's query heads and rows. */
static void bwd_key(const bwd_job_t *W, int64_t j) {
    const oracle_job_t *J = W->J;
    const int S = J->S, D = J->D;
    double *dk = W->dk + j * (int64_t)D, *dv = W->dv + j * (int64_t)D;
    for (int d = 0; d < D; ++d) dk[d] = dv[d] = 0.0;
    for (int64_t g = 0; g < W->G; ++g) {
        const int64_t bh = W->b * J->Hq + W->hkv * W->G + g;
        for (int64_t i = 0; i < S; ++i) {
            const double pij = W->P[(g * S + i) * S + j], dsij = W->dS[(g * S + i) * S + j];
            if (pij == 0.0) continue;
            /* dV takes the weight the output used: dropped or scaled with dropout. */
            double wij = pij;
            if (J->dropout_p8 > 0)
                wij = dropout_keeps(J, bh, i, j) ? pij * (256.0 / (256.0 - (double)J->dropout_p8)) : 0.0;
            const int64_t qo = (bh * S + i) * (int64_t)D;
            for (int d = 0; d < D; ++d) {
                dv[d] += wij * elem(J, 3, qo + d);
                dk[d] += dsij * elem(J, 0, qo + d);
            }
        }
    }
    for (int d = 0; d < D; ++d) dk[d] *= J->scale;
}

static void *bwd_worker(void *arg) {
    bwd_job_t *W = (bwd_job_t *)arg;
    double *dP = NULL;
    if (W->pass == 1 && !(dP = (double *)malloc(sizeof(double) * (size_t)W->J->S))) {
        W->status = 1;
        return NULL;
    }
    for (int64_t n = W->begin; n < W->end; ++n) {
        if (W->pass == 1)
            bwd_row(W, n, dP);
        else
            bwd_key(W, n);
    }
    free(dP);
    W->status = 0;
    return NULL;
}

/* Runs pass `pass` over [0, count) on nthreads threads; 0 on success. */
static int bwd_parallel(const bwd_job_t *proto, int pass, int64_t count, int nthreads) {
    if (nthreads > count) nthreads = (int)count;
    if (nthreads < 1) nthreads = 1;
    bwd_job_t *jobs = (bwd_job_t *)calloc((size_t)nthreads, sizeof(bwd_job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return 1;
    }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].pass = pass;
        jobs[t].begin = count * t / nthreads;
        jobs[t].end = count * (t + 1) / nthreads;
        jobs[t].status = 1;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, bwd_worker, &jobs[t]) != 0) break;
        started = t;
    }
    bwd_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
    for (int t = started + 1; t < nthreads; ++t) bwd_worker(&jobs[t]);
    int status = 0;
    for (int t = 0; t < nthreads; ++t) status |= jobs[t].status;
    free(jobs);
    free(tid);
    return status;
}

/*
 * oracle_attn_bwd -- dQ, dK, dV and delta for selected key/value heads.
 *
 *   q, dout [B,Hq,S,D], k, v [B,Hkv,S,D]: bf16 bit patterns (f64_inputs == 0)
 *        or doubles (f64_inputs != 0), contiguous.
 *   kv_heads: n_kv_heads flat ids b*Hkv + hkv, or NULL for all of them in
 *        order (then n_kv_heads must be B*Hkv).
 *   dq: double [n_kv_heads][G][S][D] -- the G = Hq/Hkv query heads of each
 *       selected key/value head (with every head selected: [B,Hq,S,D]);
 *   dk, dv: double [n_kv_heads][S][D];  delta: double [n_kv_heads][G][S].
 * Returns 0 on success, 1 on a bad argument or allocation failure.
 */
static int bwd_run(const void *q, const void *k, const void *v, const void *dout, int f64_inputs,
                   int B, int Hq, int Hkv, int S, int D, float scale, int causal,
                   const uint8_t *block_mask, int mask_heads, const uint8_t *keep_bits,
                   int keep_heads, int dropout_p8, uint64_t seed, uint64_t offset,
                   const int64_t *kv_heads, int64_t n_kv_heads, double *dq, double *dk,
                   double *dv, double *delta, int nthreads) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv || !delta) return 1;
    if (B < 1 || Hq < 1 || Hkv < 1 || S < 1 || D < 1 || Hq % Hkv != 0) return 1;
    if (!kv_heads && n_kv_heads != (int64_t)B * Hkv) return 1;
    if (kv_heads)
        for (int64_t n = 0; n < n_kv_heads; ++n)
            if (kv_heads[n] < 0 || kv_heads[n] >= (int64_t)B * Hkv) return 1;
    oracle_job_t J;
    memset(&J, 0, sizeof J);
    J.t[0] = q; J.t[1] = k; J.t[2] = v; J.t[3] = dout;
    J.format = f64_inputs ? FMT_F64 : FMT_BF16;
    for (int w = 0; w < 4; ++w) J.descale[w] = 1.0;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.S = S; J.D = D;
    J.scale = (double)scale;
    J.causal = causal ? 1 : 0;
    if (block_mask && mask_heads != 1 && mask_heads != Hq) return 1;
    J.block_mask = block_mask;
    J.mask_heads = block_mask ? mask_heads : 1;
    if (keep_bits && keep_heads != 1 && keep_heads != Hq) return 1;
    J.keep_bits = keep_bits;
    J.keep_heads = keep_bits ? keep_heads : 1;
    if (dropout_p8 < 0 || dropout_p8 > 255) return 1;
    if (dropout_p8 > 0 && offset > 0xFFFFFFFFull) return 1;  /* a 32-bit counter word */
    J.dropout_p8 = dropout_p8;
    J.dropout_seed = seed;
    J.dropout_offset = offset;
    const int64_t G = Hq / Hkv;
    double *P = (double *)malloc(sizeof(double) * (size_t)(G * S) * (size_t)S);
    double *dS = (double *)malloc(sizeof(double) * (size_t)(G * S) * (size_t)S);
    if (!P || !dS) {
        free(P);
        free(dS);
        return 1;
    }
    int status = 0;
    for (int64_t n = 0; n < n_kv_heads && !status; ++n) {
        const int64_t flat = kv_heads ? kv_heads[n] : n;
        bwd_job_t W;
        memset(&W, 0, sizeof W);
        W.J = &J;
        W.b = flat / Hkv;
        W.hkv = flat % Hkv;
        W.G = G;
        W.P = P;
        W.dS = dS;
        W.dq = dq + n * G * S * (int64_t)D;
        W.dk = dk + n * S * (int64_t)D;
        W.dv = dv + n * S * (int64_t)D;
        W.delta = delta + n * G * S;
        status |= bwd_parallel(&W, 1, G * S, nthreads);
        if (!status) status |= bwd_parallel(&W, 2, S, nthreads);
    }
    free(P);
    free(dS);
    return status;
}

/*
 * oracle_attn_rows_dropout -- oracle_attn_rows with dropout of the attention
 * weights: drop probability p8 / 256 (0 <= p8 < 256), Philox4x32-10 key
 * seed and counter word offset (< 2^32); see dropout_keeps for which weights
 * are dropped.
 */
int oracle_attn_rows_dropout(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Hq,
                             int Hkv, int S, int D, float scale, int causal, int p8, uint64_t seed,
                             uint64_t offset, const int64_t *rows, int64_t nrows, double *out,
                             double *lse, int nthreads) {
    const double one[3] = {1.0, 1.0, 1.0};
    if (p8 < 0 || p8 > 255) return 1;
    if (p8 > 0 && offset > 0xFFFFFFFFull) return 1;  /* a 32-bit counter word */
    return run_rows_dropout(q, k, v, FMT_BF16, one, B, Hq, Hkv, S, D, scale, causal, NULL, 1, NULL,
                            1, p8, seed, offset, rows, nrows, out, lse, nthreads);
}

/* Philox4x32-10 of one counter block (exposed so the generator can be pinned). */
void oracle_philox4x32(const uint32_t *ctr, const uint32_t *key, uint32_t *out) {
    philox4x32_10(ctr, key, out);
}

int oracle_attn_bwd(const void *q, const void *k, const void *v, const void *dout, int f64_inputs,
                    int B, int Hq, int Hkv, int S, int D, float scale, int causal,
                    const int64_t *kv_heads, int64_t n_kv_heads, double *dq, double *dk,
                    double *dv, double *delta, int nthreads) {
    return bwd_run(q, k, v, dout, f64_inputs, B, Hq, Hkv, S, D, scale, causal, NULL, 1, NULL, 1, 0,
                   0, 0, kv_heads, n_kv_heads, dq, dk, dv, delta, nthreads);
}

/*
 * oracle_attn_bwd_masked -- oracle_attn_bwd for the block-masked attention
 * (the weights of steps 1-4 include the block mask, so the same derivative
 * applies; a row without any visible key has all weights 0, hence dQ = 0 for
 * it and no contribution to dK or dV).
 */
int oracle_attn_bwd_masked(const void *q, const void *k, const void *v, const void *dout,
                           int f64_inputs, int B, int Hq, int Hkv, int S, int D, float scale,
                           int causal, const uint8_t *block_mask, int mask_heads,
                           const int64_t *kv_heads, int64_t n_kv_heads, double *dq, double *dk,
                           double *dv, double *delta, int nthreads) {
    if (!block_mask) return 1;
    return bwd_run(q, k, v, dout, f64_inputs, B, Hq, Hkv, S, D, scale, causal, block_mask,
                   mask_heads, NULL, 1, 0, 0, 0, kv_heads, n_kv_heads, dq, dk, dv, delta, nthreads);
}

/*
 * oracle_attn_bwd_keep -- oracle_attn_bwd for the element-masked attention of
 * oracle_attn_rows_keep (block_mask optional).  Masked pairs have weight 0,
 * so the same derivative applies.
 */
int oracle_attn_bwd_keep(const void *q, const void *k, const void *v, const void *dout,
                         int f64_inputs, int B, int Hq, int Hkv, int S, int D, float scale,
                         int causal, const uint8_t *keep_bits, int keep_heads,
                         const uint8_t *block_mask, int mask_heads, const int64_t *kv_heads,
                         int64_t n_kv_heads, double *dq, double *dk, double *dv, double *delta,
                         int nthreads) {
    if (!keep_bits) return 1;
    return bwd_run(q, k, v, dout, f64_inputs, B, Hq, Hkv, S, D, scale, causal, block_mask,
                   mask_heads, keep_bits, keep_heads, 0, 0, 0, kv_heads, n_kv_heads, dq, dk, dv,
                   delta, nthreads);
}

/*
 * oracle_attn_bwd_dropout -- oracle_attn_bwd for the attention with dropout of
 * oracle_attn_rows_dropout (same p8, seed, offset): the output uses the
 * weights P_ij Z_ij s, so dV_j = sum_i P_ij Z_ij s dO_i, the gradient reaching
 * P_ij is Z_ij s (dO_i . V_j), and delta_i = sum_j P_ij Z_ij s (dO_i . V_j)
 * = dO_i . O_i; the rest as without dropout.
 */
int oracle_attn_bwd_dropout(const void *q, const void *k, const void *v, const void *dout,
                            int f64_inputs, int B, int Hq, int Hkv, int S, int D, float scale,
                            int causal, int p8, uint64_t seed, uint64_t offset,
                            const int64_t *kv_heads, int64_t n_kv_heads, double *dq, double *dk,
                            double *dv, double *delta, int nthreads) {
    return bwd_run(q, k, v, dout, f64_inputs, B, Hq, Hkv, S, D, scale, causal, NULL, 1, NULL, 1, p8,
                   seed, offset, kv_heads, n_kv_heads, dq, dk, dv, delta, nthreads);
}

/*
 * oracle_attn_rows_ex -- every forward variant at once: inputs as bf16 bit
 * patterns (format 0) or E4M3 codes with per-tensor descales (format 1); an
 * optional block mask and optional keep bits (NULL for none; the masks
 * combine); dropout of the weights with p8 > 0 (seed, offset as in dropout_keeps).
 */
int oracle_attn_rows_ex(const void *q, const void *k, const void *v, int format, float q_descale,
                        float k_descale, float v_descale, int B, int Hq, int Hkv, int S, int D,
                        float scale, int causal, const uint8_t *block_mask, int mask_heads,
                        const uint8_t *keep_bits, int keep_heads, int p8, uint64_t seed,
                        uint64_t offset, const int64_t *rows, int64_t nrows, double *out,
                        double *lse, int nthreads) {
    const double ds[3] = {(double)q_descale, (double)k_descale, (double)v_descale};
    const double one[3] = {1.0, 1.0, 1.0};
    if (format != FMT_BF16 && format != FMT_E4M3) return 1;
    if (p8 < 0 || p8 > 255) return 1;
    if (p8 > 0 && offset > 0xFFFFFFFFull) return 1;  /* a 32-bit counter word */
    return run_rows_dropout(q, k, v, format, format == FMT_E4M3 ? ds : one, B, Hq, Hkv, S, D, scale,
                            causal, block_mask, block_mask ? mask_heads : 1, keep_bits,
                            keep_bits ? keep_heads : 1, p8, seed, offset, rows, nrows, out, lse,
                            nthreads);
}

/*
 * oracle_attn_bwd_ex -- the gradients of oracle_attn_rows_ex's bf16 (or
 * double) variants: optional block mask, optional keep bits and dropout.
 */
int oracle_attn_bwd_ex(const void *q, const void *k, const void *v, const void *dout, int f64_inputs,
                       int B, int Hq, int Hkv, int S, int D, float scale, int causal,
                       const uint8_t *block_mask, int mask_heads, const uint8_t *keep_bits,
                       int keep_heads, int p8, uint64_t seed, uint64_t offset,
                       const int64_t *kv_heads, int64_t n_kv_heads, double *dq, double *dk,
                       double *dv, double *delta, int nthreads) {
    return bwd_run(q, k, v, dout, f64_inputs, B, Hq, Hkv, S, D, scale, causal, block_mask,
                   block_mask ? mask_heads : 1, keep_bits, keep_bits ? keep_heads : 1, p8, seed, offset,
                   kv_heads, n_kv_heads, dq, dk, dv, delta, nthreads);
}
