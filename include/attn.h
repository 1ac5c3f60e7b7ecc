/*
 * attn.h -- C ABI of libattn: causal scaled dot-product attention on GB300
 * (sm_103a).
 *
 * Entry points: the forward (attn_fwd; FP8 inputs attn_fwd_fp8; block masks
 * attn_fwd_block_masked; per-pair keep bits attn_fwd_elem_masked; dropout of
 * the weights attn_fwd_dropout; their combinations attn_fwd_ex), the matching
 * gradients (attn_bwd, attn_bwd_block_masked, attn_bwd_elem_masked,
 * attn_bwd_dropout, attn_bwd_ex), the output
 * projection of the attention output (attn_out_proj), status helpers
 * (attn_sync_status, attn_selftest_wait_timeout, attn_status_string,
 * attn_version), and the forward's work order for inspection
 * (attn_fwd_schedule).
 *
 * The operation (one output row per query position i of every batch b and
 * query head hq) is the five-step naive causal attention that the
 * "Profiling in PyTorch (Part 3)" retelling lists in its section "Naive
 * Attention":
 *     1. S = Q K^T      2. S = S * scale      3. S[j > i] = -inf
 *     4. P = softmax(S) over keys              5. O = P V
 * with scale = 1/sqrt(head_dim) in the pages' usage (the NaiveCausalAttention
 * listing in that section; the ai-manual.ru article, section 1, divides by
 * sqrt(D), which is the same up to one fp32 rounding).  The library computes
 * it in one fused pass that never stores S or P in global memory (the
 * tiled online-softmax idea the same retelling describes for FlashAttention-2,
 * section "The Flash Backend").
 *
 * Additionally the row log-sum-exp  LSE_i = ln sum_j exp(S_ij)  (S after steps
 * 2 and 3) is written, in fp32, natural log.  The pages do not define it; it
 * is the usual companion output of a fused attention forward.
 *
 * Threading: every entry point may be called from any host thread.  The only
 * internal state is per-device setup (capability check, SM count, kernel
 * attributes; done once per device) and a least-recently-used cache of 64
 * encoded TMA descriptors, keyed by device, address, element size, extents and
 * box -- every input of the encode, so a hit is exactly what a fresh encode
 * would give, including for a buffer freed and reallocated at the same
 * address -- and a least-recently-used cache of the forward kernel's work
 * order for 32 shapes (attn_fwd_schedule; a pure function of the shape and
 * the SM count; the first call with a new shape spends up to about 0.2 ms of
 * host time building it), each guarded by a mutex.  The work runs on the calling thread's
 * current device (cudaGetDevice), which must hold every buffer; its primary
 * context is bound to the thread on entry, so a thread that has made no CUDA
 * call yet (an autograd engine's worker, say) can call too.
 *
 * Device status word: kernels whose bounded waits run out record it in one
 * word per device (read and cleared by attn_sync_status).  It is shared by
 * every stream and caller on that device.
 */
#ifndef LIBATTN_ATTN_H_
#define LIBATTN_ATTN_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes of every entry point. */
typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* NULL pointer, non-positive size, Hq % Hkv != 0, bad scale */
    ATTN_ERR_UNSUPPORTED = 2, /* head_dim not 64 or 128, or device not compute capability 10.3 */
    ATTN_ERR_MISALIGNED = 3,  /* a tensor pointer not 16-byte aligned (TMA requirement) */
    ATTN_ERR_DEVICE = 4,      /* a CUDA runtime/driver query failed */
    ATTN_ERR_LAUNCH = 5,      /* the kernel launch itself failed */
    ATTN_ERR_TIMEOUT = 6      /* a device-side wait ran past its limit (read by attn_sync_status) */
} attn_status_t;

/* Input formats of attn_options_t. */
enum { ATTN_INPUT_BF16 = 0, ATTN_INPUT_E4M3 = 1 };

/*
 * attn_options_t -- the optional features of attn_fwd_ex / attn_bwd_ex, each
 * as documented for its own entry point, combinable in one call:
 *   input_format      ATTN_INPUT_BF16, or ATTN_INPUT_E4M3 (attn_fwd_fp8's codes
 *                     with q_descale, k_descale, v_descale; forward only).
 *   block_mask, mask_heads   as attn_fwd_block_masked (NULL: none).
 *   keep_bits, keep_heads    as attn_fwd_elem_masked (NULL: none).
 *   dropout_p, seed, offset  as attn_fwd_dropout (dropout_p = 0: none).
 * Supported together: bf16 inputs with any combination of the block mask,
 * keep bits and dropout (forward and backward); E4M3 inputs with either or
 * both masks (forward only, D = 128).  E4M3 with dropout, and E4M3 in the
 * backward, return ATTN_ERR_UNSUPPORTED.
 */
typedef struct {
    int input_format;
    float q_descale, k_descale, v_descale;
    const unsigned char *block_mask;
    int mask_heads;
    const unsigned char *keep_bits;
    int keep_heads;
    float dropout_p;
    unsigned long long seed, offset;
} attn_options_t;

/*
 * attn_fwd -- O = softmax(mask(Q K^T * scale)) V  and  LSE, on the GPU.
 *
 * Arguments (all tensors live in device memory of the current CUDA device and
 * are owned by the caller; the library keeps no reference after the call):
 *   q     bf16 [B, Hq,  S, D] contiguous (row-major, D fastest).
 *   k     bf16 [B, Hkv, S, D] contiguous.
 *   v     bf16 [B, Hkv, S, D] contiguous.
 *   out   bf16 [B, Hq,  S, D] contiguous; written.  Must not alias q, k or v.
 *   lse   fp32 [B, Hq,  S] contiguous; written; may be NULL to skip it.
 *   B, Hq, Hkv, S   batch, query heads, key/value heads, sequence length (>= 1).
 *         Hq % Hkv == 0.  Query head hq reads key/value head hq / (Hq / Hkv)
 *         (grouped-query attention; Hkv == Hq is plain multi-head, Hkv == 1
 *         is multi-query).
 *   D     head dimension: 64 or 128.
 *   scale finite and > 0; the scores are multiplied by it (usually 1/sqrt(D)).
 *         Zero, negative or non-finite: ATTN_ERR_INVALID_ARG.
 *   causal  non-zero: key j is masked for query i when j > i (query and key
 *         positions share one index, Sq == Sk == S).  Zero: no mask.
 *   stream  CUDA stream (cudaStream_t, passed as void*) the work is enqueued
 *         on; NULL means the legacy default stream.
 *
 * Every pointer must be 16-byte aligned.  The call is asynchronous: it
 * returns once the kernel is enqueued and does not synchronise.  On an
 * argument error nothing is launched.  Output rows are written for
 * i < S only; nothing outside out[0 .. B*Hq*S*D) and lse[0 .. B*Hq*S) is
 * written.  Results are deterministic: repeated calls give the same bits.
 *
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED,
 * ATTN_ERR_MISALIGNED, ATTN_ERR_DEVICE or ATTN_ERR_LAUNCH.
 */
int attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
             int B, int Hq, int Hkv, int S, int D, float scale, int causal, void *stream);

/*
 * attn_fwd_block_masked -- attn_fwd plus a block mask that drops whole
 * 128 x 128 blocks of (query tile, key tile): the block-sparse attention the
 * ai-manual.ru article gives as a reason to write custom kernels (sections 4
 * and 7).  Key j is masked for query i when
 *     block_mask[h][i / 128][j / 128] == 0
 * on top of the causal mask when causal != 0.
 *
 *   block_mask  device memory, uint8 [mask_heads][nt][nt] with nt = ceil(S / 128),
 *               contiguous; non-zero keeps the block.  Read-only, caller-owned.
 *   mask_heads  1 (one mask for every batch entry and head) or Hq (one per
 *               query head, shared across the batch).
 * Blocks that are dropped are neither loaded nor computed.  A query whose keys
 * are all masked gets O = 0 and LSE = -inf (the safe-softmax convention of
 * the "Profiling in PyTorch (Part 3)" retelling, section "The Math Backend").
 * Other arguments, errors and rules as attn_fwd; ATTN_ERR_INVALID_ARG also for
 * a NULL mask or mask_heads not 1 or Hq.  The mask contents are not checked
 * against the shape: the caller guarantees mask_heads * nt * nt bytes.
 */
int attn_fwd_block_masked(const void *q, const void *k, const void *v, void *out, float *lse,
                          int B, int Hq, int Hkv, int S, int D, float scale, int causal,
                          const unsigned char *block_mask, int mask_heads, void *stream);

/*
 * attn_fwd_dropout -- attn_fwd with dropout of the attention weights, fused
 * into the kernel (the fused SDPA dropout the ai-manual.ru article describes
 * in section 6, "Dropout"): after the softmax each weight is dropped with
 * probability p and the kept ones are scaled by 1 / (1 - p).
 *
 *   dropout_p   0 <= p < 1, rounded to p8 / 256 with p8 = round(256 p), and
 *               p8 <= 255 (ATTN_ERR_INVALID_ARG otherwise); p8 = 0 is attn_fwd.
 *               Kept weights are scaled by 256 / (256 - p8).
 *   seed     the 64-bit Philox4x32-10 key {low 32 bits, high 32 bits}.
 *   offset   a 32-bit counter word (0 <= offset < 2^32, ATTN_ERR_INVALID_ARG
 *            otherwise): calls with different offsets draw independent masks.
 * Which weights are dropped: key j of query row i of head b*Hq + hq is kept
 * when byte (j mod 16) of Philox4x32-10(counter {j / 16, i, b*Hq + hq,
 * offset}, key {seed mod 2^32, seed / 2^32}) -- the four 32-bit output words
 * in order, each little-endian -- is >= p8 (Philox4x32-10: Salmon et al.,
 * "Parallel random numbers: as easy as 1, 2, 3", SC 2011).  The same call
 * with the same seed and offset drops the same weights.  LSE is that of the
 * undropped softmax.  Other arguments, errors and rules as attn_fwd (bf16
 * inputs).
 */
int attn_fwd_dropout(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                     int Hq, int Hkv, int S, int D, float scale, int causal, float dropout_p,
                     unsigned long long seed, unsigned long long offset, void *stream);

/*
 * attn_fwd_fp8 -- the same attention with FP8 E4M3 inputs and per-tensor
 * descale factors (the FP8 attention the ai-manual.ru article mentions for
 * newer GPUs, section 6 "FP8 and BF16").
 *
 *   q, k, v  E4M3 codes (one byte each, the OCP "fn" encoding), layouts as in
 *            attn_fwd: q [B,Hq,S,D], k and v [B,Hkv,S,D], contiguous.  Element
 *            value = decoded code * its tensor's descale.
 *   q_descale, k_descale, v_descale   finite and > 0.
 *   out      bf16 [B,Hq,S,D]; lse fp32 [B,Hq,S] or NULL; scale, causal, stream
 *            as in attn_fwd.
 *   D        128 only (ATTN_ERR_UNSUPPORTED otherwise).
 *
 * Scores accumulate in fp32 from the exact products of the codes; the
 * probabilities that multiply V are rounded to E4M3 (round to nearest even),
 * the row sums and LSE use the unrounded fp32 probabilities.  Same alignment,
 * asynchrony and error rules as attn_fwd.
 */
int attn_fwd_fp8(const void *q, const void *k, const void *v, float q_descale, float k_descale,
                 float v_descale, void *out, float *lse, int B, int Hq, int Hkv, int S, int D,
                 float scale, int causal, void *stream);

/*
 * attn_fwd_elem_masked -- attn_fwd plus an element mask that drops single
 * (query, key) pairs: the arbitrary masks the ai-manual.ru article gives,
 * with block-sparse ones, as a reason to write custom kernels (sections 4 and
 * 7).  Key j is masked for query i of head h when
 *     (keep_bits[h][i][j / 8] >> (j % 8)) & 1 == 0
 * on top of the causal mask when causal != 0, and on top of an optional block
 * mask (as in attn_fwd_block_masked).
 *
 *   keep_bits   device memory, uint8 [keep_heads][S][16 * ceil(S / 128)],
 *               contiguous and 16-byte aligned: row i holds one bit per key,
 *               16 bytes per 128 keys (bits past key S - 1 are ignored).
 *               Read-only, caller-owned.
 *   keep_heads  1 (one mask for every batch entry and head) or Hq (one per
 *               query head, shared across the batch).
 *   block_mask  NULL, or uint8 [mask_heads][nt][nt] as in attn_fwd_block_masked;
 *               blocks it drops are neither loaded nor computed.  Without it
 *               every block within the causal bound is computed, so callers
 *               whose element mask leaves whole blocks empty should pass the
 *               matching block mask too.
 *   mask_heads  1 or Hq (ignored when block_mask is NULL).
 * A query whose keys are all masked gets O = 0 and LSE = -inf.  Other
 * arguments, errors and rules as attn_fwd; ATTN_ERR_INVALID_ARG also for a
 * NULL keep_bits or keep_heads / mask_heads not 1 or Hq, ATTN_ERR_MISALIGNED
 * for keep_bits not 16-byte aligned.  The caller guarantees the sizes above.
 */
int attn_fwd_elem_masked(const void *q, const void *k, const void *v, void *out, float *lse,
                         int B, int Hq, int Hkv, int S, int D, float scale, int causal,
                         const unsigned char *keep_bits, int keep_heads,
                         const unsigned char *block_mask, int mask_heads, void *stream);

/*
 * attn_fwd_ex -- attn_fwd with the options above (opts NULL: attn_fwd).
 * Errors as the entry points of the features used.
 */
int attn_fwd_ex(const void *q, const void *k, const void *v, void *out, float *lse, int B, int Hq,
                int Hkv, int S, int D, float scale, int causal, const attn_options_t *opts,
                void *stream);

/*
 * attn_bwd -- gradients of attn_fwd's output: dQ, dK, dV for an upstream
 * gradient dO.  The pages give no formula (the ai-manual.ru article, section 6,
 * only warns that the fused backward pass is hard to get right); this is the
 * derivative of the forward:
 *     P_ij = exp(scale * q_i . k_j - LSE_i)  (0 for masked pairs),
 *     dP_ij = dO_i . V_j,  delta_i = dO_i . O_i,  dS_ij = P_ij (dP_ij - delta_i),
 *     dQ_i = scale * sum_j dS_ij K_j,  dK_j = scale * sum_i dS_ij Q_i,
 *     dV_j = sum_i P_ij dO_i,
 * with dK and dV of a key/value head summed over its group's query heads.
 *
 *   q, k, v, scale, B, Hq, Hkv, S, D, causal   exactly as passed to attn_fwd.
 *   out      bf16 [B,Hq,S,D]: attn_fwd's output O.
 *   dout     bf16 [B,Hq,S,D]: the upstream gradient dO.
 *   lse      fp32 [B,Hq,S]: attn_fwd's LSE (required here).
 *   delta    fp32 [B,Hq,S], written: delta_i = dO_i . O_i (the kernels'
 *            row term; callers may read it).
 *   dq       bf16 [B,Hq,S,D], written.
 *   dk, dv   bf16 [B,Hkv,S,D], written.
 * Every pointer is device memory owned by the caller; the bf16 tensors must be
 * 16-byte aligned, lse and delta 4-byte aligned.  The outputs (delta, dq, dk,
 * dv) may overlap neither the inputs nor each other (ATTN_ERR_INVALID_ARG).
 * Two kernels run on `stream` (dQ and delta, then dK and dV); the call is
 * asynchronous and allocates nothing.  Other errors as attn_fwd.
 */
int attn_bwd(const void *q, const void *k, const void *v, const void *out, const void *dout,
             const float *lse, float *delta, void *dq, void *dk, void *dv, int B, int Hq, int Hkv,
             int S, int D, float scale, int causal, void *stream);

/*
 * attn_bwd_block_masked -- attn_bwd for attn_fwd_block_masked: the gradients of
 * the block-masked attention, with the same block_mask and mask_heads as the
 * forward call (see attn_fwd_block_masked).  Dropped tiles are neither loaded
 * nor computed; query rows that see no key (LSE = -inf, O = 0) get dQ = 0
 * and contribute nothing to dK and dV.  ATTN_ERR_INVALID_ARG also for a NULL
 * mask or mask_heads not 1 or Hq; otherwise as attn_bwd.
 */
int attn_bwd_block_masked(const void *q, const void *k, const void *v, const void *out,
                          const void *dout, const float *lse, float *delta, void *dq, void *dk,
                          void *dv, int B, int Hq, int Hkv, int S, int D, float scale, int causal,
                          const unsigned char *block_mask, int mask_heads, void *stream);

/*
 * attn_bwd_elem_masked -- attn_bwd for the element-masked attention of
 * attn_fwd_elem_masked (same keep_bits, keep_heads, block_mask, mask_heads;
 * out and lse from that call).  Masked pairs have weight 0, so they add
 * nothing to any gradient; a query without any visible key gets dQ = 0 and
 * delta = 0.  Arguments, errors and rules as attn_bwd and
 * attn_fwd_elem_masked.
 */
int attn_bwd_elem_masked(const void *q, const void *k, const void *v, const void *out,
                         const void *dout, const float *lse, float *delta, void *dq, void *dk,
                         void *dv, int B, int Hq, int Hkv, int S, int D, float scale, int causal,
                         const unsigned char *keep_bits, int keep_heads,
                         const unsigned char *block_mask, int mask_heads, void *stream);

/*
 * attn_bwd_dropout -- attn_bwd for the attention with dropout of
 * attn_fwd_dropout (same dropout_p, seed, offset; out and lse from that
 * call).  With Z_ij the keep decision of attn_fwd_dropout and s = 256 /
 * (256 - p8) the output uses the weights P_ij Z_ij s, so
 *     dV_j = sum_i P_ij Z_ij s dO_i,   dP_ij = Z_ij s (dO_i . V_j),
 *     delta_i = dO_i . O_i,            dS_ij = P_ij (dP_ij - delta_i),
 * and dQ, dK as in attn_bwd.  The keep decisions are regenerated from the
 * same counter-based generator, not stored.  Arguments, errors and rules as
 * attn_bwd and attn_fwd_dropout (dropout_p rounds to p8 = round(256 p) <= 255;
 * p8 = 0 is attn_bwd).
 */
int attn_bwd_dropout(const void *q, const void *k, const void *v, const void *out,
                     const void *dout, const float *lse, float *delta, void *dq, void *dk, void *dv,
                     int B, int Hq, int Hkv, int S, int D, float scale, int causal, float dropout_p,
                     unsigned long long seed, unsigned long long offset, void *stream);

/*
 * attn_bwd_ex -- the gradients of attn_fwd_ex's output for the same options
 * (bf16 inputs, every combination of block mask, keep bits and dropout;
 * opts NULL: attn_bwd).  E4M3 inputs: ATTN_ERR_UNSUPPORTED.
 */
int attn_bwd_ex(const void *q, const void *k, const void *v, const void *out, const void *dout,
                const float *lse, float *delta, void *dq, void *dk, void *dv, int B, int Hq, int Hkv,
                int S, int D, float scale, int causal, const attn_options_t *opts, void *stream);

/*
 * attn_out_proj -- the layer's output projection applied to attention's
 * output where it lies (the "output projection" operator the ainews.cool
 * article profiles right after attention, per-operator table):
 *     Y[b, s, e] = sum_{h, d} O[b, h, s, d] * W[e, h*D + d] + bias[e],
 * i.e. the heads of each position laid side by side, times W^T.
 *
 *   out    bf16 [B, H, S, D]: attn_fwd's output, read in place (no transpose).
 *   w      bf16 [E, H*D], row-major (the weight of a linear layer with H*D
 *          inputs and E outputs).
 *   bias   fp32 [E], or NULL for none.
 *   y      bf16 [B, S, E], written.
 *   D      64 or 128; E a multiple of 8 (ATTN_ERR_UNSUPPORTED otherwise).
 * out, w and y 16-byte aligned, bias 4-byte aligned; y may overlap nothing
 * else.  fp32 accumulation, one rounding to bf16 at the end.  One kernel on
 * `stream`, asynchronous; allocates nothing.  Errors as attn_fwd.
 */
int attn_out_proj(const void *out, const void *w, const float *bias, void *y, int B, int H, int S,
                  int D, int E, void *stream);

/*
 * attn_sync_status -- synchronise `stream` and report device-side failures of
 * the attention kernels enqueued on this device since the last call.
 *
 * Every wait inside the kernels is bounded in time; a wait that runs out sets
 * a per-device status word and makes the kernel exit cleanly (it never traps).
 * This call waits for `stream`, reads and clears that word, and returns
 * ATTN_OK, ATTN_ERR_TIMEOUT, or ATTN_ERR_DEVICE if the synchronisation itself
 * failed.  The word is one per device, not per stream: a timeout left by a
 * kernel on another stream of the same device is reported (and cleared) here
 * too, and outputs of a kernel that timed out are only partly written.
 */
int attn_sync_status(void *stream);

/*
 * attn_selftest_wait_timeout -- launch one tiny kernel that waits on an
 * mbarrier nobody arrives at, with a limit of `limit_us` microseconds
 * (1 .. 1000000).  The wait must give up, set the status word and let the
 * kernel return; attn_sync_status then reports ATTN_ERR_TIMEOUT.  It exists so
 * the bounded-wait path is exercised without faulting or hanging a GPU.
 * Returns ATTN_OK once launched, ATTN_ERR_INVALID_ARG for a bad limit.
 */
int attn_selftest_wait_timeout(int limit_us, void *stream);

/* Human-readable name of a return code (static storage; never NULL). */
const char *attn_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int attn_version(void);

/*
 * attn_fwd_schedule -- the order in which the forward kernel's `num_ctas`
 * persistent CTAs take their work units, for inspection and tests; the pages
 * have no counterpart (it is this library's scheduling, not part of the
 * method).  A unit is one flat head bh = b*Hq + hq (0 <= bh < batch_heads)
 * and one pair of query tiles m (tiles 2m and 2m+1 of num_q_tiles =
 * ceil(S / 128)), numbered u = (npairs - 1 - m) * batch_heads + bh with
 * npairs = ceil(num_q_tiles / 2).  On ATTN_OK, CTA c runs
 * order[start[c]] .. order[start[c + 1] - 1] in turn: `start` receives
 * num_ctas + 1 entries and `order` batch_heads * npairs (caller-owned host
 * arrays).  Units go out head block by head block (16 query heads), the
 * heaviest pair of a block first, each to the CTA that frees up first under
 * a cost of its tile products (causal != 0: a pair's tiles need key tiles up
 * to their diagonal).  Pure host computation: no device, no stream.
 * The block-masked forwards (a block mask given) always use the arithmetic
 * order, whose CTAs get equal unit counts whatever the mask keeps.
 * Returns ATTN_ERR_INVALID_ARG for a null array or a size <= 0, and
 * ATTN_ERR_UNSUPPORTED when the forward does not use a table for the shape:
 * fewer than two units per CTA, or more than the table holds (4096 units,
 * 160 CTAs).  The forward then uses its arithmetic order (round r: units
 * rG .. rG+G-1 for G CTAs, even rounds by CTA index, odd rounds reversed).
 */
int attn_fwd_schedule(int batch_heads, int num_q_tiles, int causal, int num_ctas, unsigned short *order,
                      unsigned short *start);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* LIBATTN_ATTN_H_ */
