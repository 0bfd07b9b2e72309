/*
 * attn_skip -- softmax-threshold block skipping inside a FlashAttention-style
 * online-softmax tile loop, for one NVIDIA GB300 (sm_103a).
 *
 * Method: the web page "BLASST：一个标量阈值实现的动态块稀疏注意力（MLSys 2026）"
 * (BLASST, arXiv 2512.12087).  For query tile i and KV block j, after the
 * running max is updated to m_i^(j), the block is skipped when
 *
 *        rowmax(S_ij) - m_i^(j) < ln(lambda)          (section "BLASST 的判定准则", Eq. 5)
 *
 * holds for every row of the tile (section "判定本身：几乎零成本的秘密"); a
 * skipped block costs no exponentials, no P.V product and -- in decode -- no
 * value load (sections "Prefill 内核：砍计算", "Decode 内核：砍带宽").  Q.K^T
 * is always computed: it is the only source of the block max.
 *
 * Conventions shared by every call
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    allocates no device memory and keeps no state between calls except one
 *    device error word per GPU.  Layouts are dense row-major (C order).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Arguments are validated on the host before any launch;
 *    on a validation error nothing is launched and no output is written.
 *  - Scores are s = scale * <q, k>; scale <= 0 selects 1/sqrt(dk).  LSE outputs
 *    are natural-log log-sum-exp of the scaled scores of the kept keys.
 *  - lambda in [0, 1).  lambda = 0 disables skipping (dense attention).
 *    The library evaluates ln(lambda) once on the host in double precision and
 *    compares in the log domain in fp32 (section "BLASST 的判定准则": one
 *    subtraction and one compare per element, no exponential).
 *  - Skip bitmaps are uint32 words; bit (j % 32) of word (j / 32) of a unit's
 *    row is 1 when block j was skipped.  Blocks a unit does not traverse (causal
 *    blocks above the diagonal, positions past the end of a split) read 0.
 *    Every word of every unit is written, so the buffer needs no clearing.
 *  - Pointers must be 16-byte aligned.
 *
 * Status codes: ATTN_EINVAL for a null pointer, a non-positive size, Hq not a
 * multiple of Hkv, lambda outside [0,1) or NaN, or a misaligned pointer;
 * ATTN_EUNSUPPORTED for a valid combination the library has no kernel for;
 * ATTN_ECUDA for a launch or CUDA runtime error (the CUDA error is cleared);
 * ATTN_ETIMEOUT when a device-side bounded wait gave up, ATTN_EINTERNAL when a
 * kernel found its dynamic shared memory placed off the 1024-byte boundary its
 * swizzled tiles need and returned without work (both reported by
 * attn_skip_last_device_error).
 */
#ifndef ATTN_SKIP_H
#define ATTN_SKIP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_EINVAL = 1,
  ATTN_EUNSUPPORTED = 2,
  ATTN_ECUDA = 3,
  ATTN_ETIMEOUT = 4,
  ATTN_EINTERNAL = 5
} attn_status;

typedef enum { ATTN_BF16 = 0, ATTN_F32 = 1 } attn_dtype;

/* Samplers of the sampled decode output (attn_skip_santa_decode). */
typedef enum {
  ATTN_SANTA_IID = 0,   /* S independent draws from the attention weights        */
  ATTN_SANTA_SYS = 1,   /* one offset, S equally spaced thresholds (systematic)  */
  ATTN_SANTA_STRAT = 2  /* one draw inside each of S equal-mass strata           */
} attn_santa_mode;

/*
 * Causal (or full) GQA prefill with block skipping.
 *
 * Defines: the online-softmax loop of section "铺垫：FlashAttention 的在线 softmax"
 * (Eqs. 2-4) with the skip test of Eq. 5, KV blocks visited in ascending
 * order; a query tile of Br rows skips block j only if all its valid rows
 * vote skip.  Causal masking is top-left with equal query and key length:
 * key c is visible to row r iff c <= r.
 *
 *  q          [B, Hq,  T, dk]  (dt)
 *  k          [B, Hkv, T, dk]  (dt)   query head h reads KV head h / (Hq/Hkv)
 *  v          [B, Hkv, T, dv]  (dt)
 *  o          [B, Hq,  T, dv]  (dt)   written: softmax over the kept keys times V
 *  lse        [B, Hq,  T]      fp32   written
 *  skip_bits  [B, Hq, ceil(T/Br), ceil(ceil(T/Bc)/32)] uint32, written
 *
 * Kernels built: dt = ATTN_BF16 with dk = dv = 128, Br = Bc = 128 (tcgen05
 * tensor-core path, fp32 accumulation, P rounded to bf16 for the P.V product);
 * dt = ATTN_F32 with dk = dv in {32, 64}, Br, Bc in {64, 128} (CUDA-core path).
 * Anything else returns ATTN_EUNSUPPORTED.
 */
attn_status attn_skip_prefill(const void *q, const void *k, const void *v, attn_dtype dt, int B,
                              int Hq, int Hkv, int T, int dk, int dv, float scale, double lambda,
                              int Br, int Bc, int causal, void *o, float *lse,
                              uint32_t *skip_bits, void *stream);

/*
 * The same prefill with its inputs and outputs in host memory: Q, K, V are
 * copied in and O, LSE copied back, overlapped with the computation.  The
 * B * Hkv KV heads (flattened, batch-major) are split into n_groups
 * contiguous groups; group g's copies in run on copy_in_stream while group
 * g - 1 is computed on `stream` and group g - 2's results are copied back on
 * copy_out_stream (each group is attn_skip_prefill on its own query heads and
 * KV heads, so the results are bit-identical to one attn_skip_prefill call).
 *
 * Defines: as attn_skip_prefill; the pipelining is not on the pages (it moves
 * data to and from the device, not any step of the method).
 *
 *  q_host, k_host, v_host  host, the layouts of q, k, v of attn_skip_prefill;
 *                          page-locked memory lets the copies run
 *                          asynchronously (pageable memory still works, the
 *                          copies then stall the host)
 *  q_dev, k_dev, v_dev     device staging of the same shapes, written
 *  o_dev, lse_dev, skip_bits  device outputs as for attn_skip_prefill
 *  o_host, lse_host        host outputs, same layouts as o, lse; written when
 *                          `stream` has reached the end of the call's work
 *  n_groups                1 .. B*Hkv (0 picks min(8, B*Hkv))
 *  stream                  computation; the call's work (copies included) is
 *                          complete when `stream` reaches the point of the call
 *  copy_in_stream, copy_out_stream  streams of the two copy directions; NULL
 *                          uses `stream` (no overlap in that direction).
 * Every pointer is caller-owned.  The call creates 2 * n_groups + 1 CUDA
 * events and releases them before it returns (their last records complete
 * later, as CUDA allows).  Errors: those of attn_skip_prefill, EINVAL for a
 * null host or staging pointer or n_groups out of range; argument errors are
 * found before anything is enqueued.
 */
attn_status attn_skip_prefill_from_host(
    const void *q_host, const void *k_host, const void *v_host, void *q_dev, void *k_dev,
    void *v_dev, attn_dtype dt, int B, int Hq, int Hkv, int T, int dk, int dv, float scale,
    double lambda, int Br, int Bc, int causal, void *o_dev, float *lse_dev, uint32_t *skip_bits,
    void *o_host, float *lse_host, int n_groups, void *stream, void *copy_in_stream,
    void *copy_out_stream);

/*
 * Prefill restricted to an explicit block set per query tile, composed with
 * the threshold test: the consumer side of a block-selection stage such as the
 * SparDA page's InfLLM-V2 access set B_init u B_local u B_topk (section 2.1).
 * Blocks outside a tile's set are not traversed -- no Q.K^T, no running-max
 * update, no value load -- and read 0 in skip_bits; inside the set the loop and
 * the skip test are those of attn_skip_prefill, blocks visited in ascending
 * order.  A row whose tile set holds no visible key gets O = 0, LSE = -inf.
 *
 *  block_set  [B, Hq, ceil(T/Br), ceil(ceil(T/Bc)/32)] uint32 (device): bit
 *             (j % 32) of word (j / 32) = block j is in the tile's set; bits
 *             of blocks a causal tile does not reach are ignored
 *  other arguments and outputs as for attn_skip_prefill; same kernels built.
 */
attn_status attn_skip_prefill_blocks(const void *q, const void *k, const void *v, attn_dtype dt,
                                     int B, int Hq, int Hkv, int T, int dk, int dv, float scale,
                                     double lambda, int Br, int Bc, int causal,
                                     const uint32_t *block_set, void *o, float *lse,
                                     uint32_t *skip_bits, void *stream);

/*
 * Batched variable-length causal (or full) prefill, one threshold per sequence.
 *
 * Defines: section "λ = a/L：反比关系的直觉与依据" -- the threshold that keeps
 * a target sparsity falls as a / L with the context length L, so a batch of
 * sequences of different lengths takes one lambda per sequence (e.g.
 * lambda[s] = a / L_s, or alpha * exp(beta * S) / L_s from the calibration
 * model); each sequence is the loop of attn_skip_prefill on its own tokens.
 *
 *  cu_seqlens [n_seq + 1] int32 (device): sequence s holds tokens
 *             [cu_seqlens[s], cu_seqlens[s+1]); cu_seqlens[0] = 0,
 *             nondecreasing, last = total; lengths <= max_seqlen; a length
 *             of 0 is allowed
 *  lambda     [n_seq] fp32 (device), each in [0, 1); 0 = dense; ln(lambda)
 *             is taken on the device in fp32
 *  q          [total, Hq, dk] token-major (device); k [total, Hkv, dk];
 *             v [total, Hkv, dv]
 *  o          [total, Hq, dv] (same dtype as q)
 *  lse        [Hq, total] fp32, natural log
 *  skip_bits  [n_seq, Hq, n_t, ceil(n_t / 32)] uint32, n_t =
 *             ceil(max_seqlen / Br): tile t of sequence s in row (s, h, t);
 *             rows of tiles a sequence does not have read 0
 *  scale      as for attn_skip_prefill
 *
 * Host checks as for attn_skip_prefill (EINVAL also for a null cu_seqlens
 * or lambda, n_seq <= 0, max_seqlen < 0 or total < 0; cu_seqlens and lambda
 * need only 4-byte alignment).  Kernels built: bf16, dk = dv = 128,
 * Br = Bc = 128 (else ATTN_EUNSUPPORTED).  The device arrays are checked by
 * the kernel: a sequence whose bounds are out of range is treated as empty,
 * a lambda outside [0, 1) as 0, and attn_skip_last_device_error then returns
 * ATTN_EINVAL.  max_seqlen = 0 launches nothing; total = 0 (every sequence
 * empty; q, k, v, o, lse may then be NULL) only zeroes skip_bits.
 */
attn_status attn_skip_prefill_varlen(const void *q, const void *k, const void *v, attn_dtype dt,
                                     int n_seq, const int32_t *cu_seqlens, int max_seqlen,
                                     int total, int Hq, int Hkv, int dk, int dv, float scale,
                                     const float *lambda, int Br, int Bc, int causal, void *o,
                                     float *lse, uint32_t *skip_bits, void *stream);

/*
 * Split-KV decode, one query token per sequence, with block skipping.
 *
 * Defines: section "Decode 内核：砍带宽" -- scores of a batch of KV blocks are
 * computed first, the skip decisions are taken for the batch in block order,
 * and values are loaded only for the kept blocks.  The G = Hq/Hkv query heads
 * that share a KV head form one group and skip a block only if all of them
 * vote skip.  The cache of each (b, KV head) is split into n_splits ranges of
 * whole blocks, split s owning blocks [floor(s*nb/n), floor((s+1)*nb/n)) with
 * nb = ceil(L/Bc); each split restarts its running max (FlashDecoding).
 *
 *  q          [B, Hq, dk]                      (dt)
 *  k          key c of (b, hk) at k + ((b*Hkv + hk)*L + c) * k_row_stride   (dt)
 *  v          value c at v + ((b*Hkv + hk)*L + c) * v_row_stride            (dt)
 *             (an absorbed-MLA latent cache passes v == k: values are the
 *             first dv columns of each key row)
 *  o_part     [B, Hq, n_splits, dv]  fp32, written (0 for an empty split)
 *  lse_part   [B, Hq, n_splits]      fp32, written (-inf for an empty split)
 *  skip_bits  [B, Hkv, n_splits, ceil(bps/32)] uint32 with bps = ceil(nb/n_splits);
 *             bit p of split s is block floor(s*nb/n_splits) + p
 *
 * Kernels built: dt = ATTN_BF16, dk = dv = 128, Bc = 128, G in {1, 2, 4, 8},
 * k_row_stride = v_row_stride = 128 (tcgen05 path with the G heads padded to
 * the 128 MMA rows; memory bound; P rounded to bf16 for P.V); and the
 * absorbed-MLA shape dt = ATTN_BF16, Hkv = 1, Hq = 128, dk = 576, dv = 512,
 * v == k, k_row_stride = v_row_stride = 576, Bc = 64 (tcgen05 path, the 128
 * heads as one M = 128 tile; a skipped block saves its exponentials and its
 * P.V product, its value bytes being the key bytes already read).
 */
attn_status attn_skip_decode(const void *q, const void *k, const void *v, attn_dtype dt, int B,
                             int Hq, int Hkv, int L, int dk, int dv, int64_t k_row_stride,
                             int64_t v_row_stride, float scale, double lambda, int Bc,
                             int n_splits, float *o_part, float *lse_part, uint32_t *skip_bits,
                             void *stream);

/*
 * Split-KV decode with per-head decisions: each of the G query heads sharing a
 * KV head takes Eq. 5 for itself (a block it skips adds nothing to its
 * output), instead of the group skipping a block only when all G agree.  A
 * block's values are read when any head of the group keeps it, so the bytes
 * read equal the group-AND call's; only each head's approximation changes.
 * For G = 1 the two calls coincide.
 *
 *  skip_bits  [B, Hq, n_splits, ceil(bps/32)] uint32: per query head
 *  other arguments and outputs as for attn_skip_decode.
 *
 * Kernels built: the GQA shape of attn_skip_decode (dt = ATTN_BF16, dk = dv =
 * 128, Bc = 128, G in {1, 2, 4, 8}, row strides 128) and its absorbed-MLA
 * shape (128 heads over one 576-column latent row, v == k, dv = 512, Bc = 64)
 * for splits of at most 2048 blocks; anything else returns ATTN_EUNSUPPORTED.
 * With MLA's 128 heads on one latent head, per-head decisions reach sparsity
 * that the group AND (a block skipped only when all 128 agree) cannot.
 */
attn_status attn_skip_decode_per_head(const void *q, const void *k, const void *v, attn_dtype dt,
                                      int B, int Hq, int Hkv, int L, int dk, int dv,
                                      int64_t k_row_stride, int64_t v_row_stride, float scale,
                                      double lambda, int Bc, int n_splits, float *o_part,
                                      float *lse_part, uint32_t *skip_bits, void *stream);

/*
 * Split-KV decode with block skipping over an FP8 (E4M3) key/value cache.
 *
 * Defines: the loop of attn_skip_decode (section "Decode 内核：砍带宽": decide
 * from the scores, read values only for kept blocks) over a cache of E4M3
 * codes (OCP FP8 E4M3: bias 7, max 448, S.1111.111 = NaN) with one fp32
 * scale per (sequence, KV head) for keys and for values:
 * key row = k_scale[b,h] * E4M3(k), value row = v_scale[b,h] * E4M3(v).
 * The BLASST page evaluates FP8/NVFP4-quantised models but fixes no cache
 * format; halving the cache bytes halves the time of this bandwidth-bound
 * loop.
 *
 *  q          [B, Hq, dk] bf16 (device).  The products are E4M3 x E4M3, so
 *             each query head enters as the pair hi + lo of E4M3 values of
 *             q * 2^e (2^e the largest power of two with max|q| 2^e <= 256),
 *             both rounded to nearest even: exact for every element within
 *             about 2^-10 of the head's largest, and otherwise off by at most
 *             2^-10 / 2^e, which moves a score by at most
 *             scale * k_scale * 2^-10 / 2^e * sum_d |E4M3(k_d)|
 *  k, v       [B, Hkv, L, d] uint8 E4M3 codes (device), row strides in bytes
 *             (multiples of 16); no NaN codes
 *  k_scale, v_scale [B, Hkv] fp32 (device)
 *  outputs, bitmap layout, merge, lambda, scale: as attn_skip_decode
 *  (o_part already multiplied by v_scale; attn_skip_decode_combine merges)
 *
 * Kernels built: dk = dv = 128, Bc = 128, Hq/Hkv in {1, 2, 4, 8}; P is
 * rounded to fp16 for the P.V product, accumulation in fp32.  EINVAL as for
 * attn_skip_decode (also for a null or misaligned scale pointer).
 */
attn_status attn_skip_decode_fp8(const void *q, const void *k, const void *v, const float *k_scale,
                                 const float *v_scale, int B, int Hq, int Hkv, int L, int dk,
                                 int dv, int64_t k_row_stride, int64_t v_row_stride, float scale,
                                 double lambda, int Bc, int n_splits, float *o_part,
                                 float *lse_part, uint32_t *skip_bits, void *stream);

/*
 * Split-KV decode with block skipping over an NVFP4 key/value cache.
 *
 * Defines: the loop of attn_skip_decode (section "Decode 内核：砍带宽") over a
 * cache in the NVFP4 layout (the BLASST page evaluates NVFP4-quantised models,
 * section "更大模型、MLA 与组合性", and fixes no format): per row, E2M1 codes
 * (OCP MX FP4: +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}) two per byte, element 2i in
 * the low nibble; one E4M3 block scale per 16 consecutive elements; one fp32
 * scale per (sequence, KV head) for keys and one for values:
 * row element = scale[b,h] * E4M3(block scale) * E2M1(code).  The key scale
 * is folded into the score scale, the value scale multiplies the outputs.
 *
 *  q          [B, Hq, dk] bf16 (device).  The key products are fp16 x fp16,
 *             so each query head enters as fp16(q * 2^e), 2^e the largest
 *             power of two with max|q| 2^e <= 2^15: exact for every element
 *             not below about 2^-31 of the head's largest, and otherwise off
 *             by at most 2^-25 / 2^e
 *  k4, v4     [B, Hkv, L, d/2] uint8 packed E2M1 codes (device), row strides
 *             in bytes (multiples of 16, at least d/2)
 *  k_bs, v_bs [B, Hkv, L, d/16] uint8 E4M3 block scales (device, dense)
 *  k_scale, v_scale [B, Hkv] fp32 (device)
 *  outputs, bitmap layout, merge, lambda, scale: as attn_skip_decode
 *  (o_part already multiplied by v_scale; attn_skip_decode_combine merges)
 *
 * Codes and block scales are widened exactly to fp16 on the chip (an E2M1
 * value times an E4M3 scale is an fp16 normal number); P is rounded to fp16
 * for the P.V product, accumulation in fp32.  No NaN block-scale codes.
 * Kernels built: dk = dv = 128, Bc = 128, Hq/Hkv in {1, 2, 4, 8}.  EINVAL
 * as for attn_skip_decode_fp8 (also for a null or misaligned block-scale
 * pointer).
 */
attn_status attn_skip_decode_nvfp4(const void *q, const void *k4, const void *v4,
                                   const uint8_t *k_bs, const uint8_t *v_bs,
                                   const float *k_scale, const float *v_scale, int B, int Hq,
                                   int Hkv, int L, int dk, int dv, int64_t k_row_stride,
                                   int64_t v_row_stride, float scale, double lambda, int Bc,
                                   int n_splits, float *o_part, float *lse_part,
                                   uint32_t *skip_bits, void *stream);

/*
 * Merge of decode split partials by log-sum-exp (FlashDecoding):
 * LSE = ln sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) * O_s.
 * Splits with LSE_s = -inf weigh zero.
 *
 *  o_part [B, Hq, n_splits, dv] fp32,  lse_part [B, Hq, n_splits] fp32
 *  o      [B, Hq, dv] (out_dt),       lse      [B, Hq] fp32
 */
attn_status attn_skip_decode_combine(const float *o_part, const float *lse_part, int B, int Hq,
                                     int n_splits, int dv, attn_dtype out_dt, void *o,
                                     float *lse, void *stream);

/*
 * Threshold calibration (section "校准算法：一次前向，一个指数模型", Algorithm 2):
 * the block statistic that Eq. 5 compares with ln(lambda) does not depend on
 * lambda (the running max advances on every traversed block, skipped or not),
 * so one pass over the scores gives the sparsity for every candidate lambda.
 *
 * The two *_margins calls run the same kernels as attn_skip_prefill /
 * attn_skip_decode in a statistics mode: every block is treated as skipped (no
 * value load, no exponential, no P.V product) and, per traversed block,
 *
 *     margin = max over the unit's rows of (rowmax(S_ij) - m_new)   (natural log, <= 0)
 *
 * is written; the block is skipped at lambda iff margin < ln(lambda).  A unit
 * is a prefill query tile (rows = its valid query rows) or a decode (b, KV
 * head, split) (rows = its G query heads).  -inf: no row has a visible key in
 * the block; NaN: block not traversed (causal blocks above the diagonal,
 * positions past a split's last block).  No other output is written.
 *
 *  prefill: q, k as for attn_skip_prefill (no value tensor);
 *           margin [B, Hq, ceil(T/Br), ceil(T/Bc)] fp32 (device)
 *  decode:  q, k as for attn_skip_decode (no value tensor; dk = 576 selects
 *           the absorbed-MLA shape with dv = 512);
 *           margin [B, Hkv, n_splits, ceil(ceil(L/Bc)/n_splits)] fp32 (device)
 *
 * Same kernels built, same status codes as the corresponding calls.
 */
attn_status attn_skip_prefill_margins(const void *q, const void *k, attn_dtype dt, int B, int Hq,
                                      int Hkv, int T, int dk, float scale, int Br, int Bc,
                                      int causal, float *margin, void *stream);
attn_status attn_skip_decode_margins(const void *q, const void *k, attn_dtype dt, int B, int Hq,
                                     int Hkv, int L, int dk, int64_t k_row_stride, float scale,
                                     int Bc, int n_splits, float *margin, void *stream);

/*
 * Host-side helpers (host memory, synchronous, no GPU work).
 *
 * attn_skip_sparsity_at: fraction of the n margins' traversed entries (NaN
 * entries are ignored) that lambda skips, i.e. margin < ln(lambda); 0 for
 * lambda = 0 and for an array with no traversed entry; -1 for invalid input.
 *
 * attn_skip_lambda_for_sparsity: a lambda in [0, 1) that skips the fraction
 * `target` of the traversed entries: ln(lambda) is placed halfway between the
 * largest skipped and the smallest kept statistic.  A statistic of 0 (some row
 * found a new max in the block) is never skipped by any lambda < 1, so a target
 * above the fraction of negative statistics returns the lambda that skips all
 * of them.  ATTN_EINVAL for a null pointer, n <= 0, a target outside [0, 1]
 * or no traversed entry.
 *
 * attn_skip_fit_lambda_model: least-squares fit of the section's exponential
 * model lambda * L = alpha * exp(beta * s) to n >= 2 calibration points
 * (L_i, s_i, lambda_i), on ln(lambda * L) = ln(alpha) + beta * s.  ATTN_EINVAL
 * for null pointers, n < 2, a non-positive L or lambda, or all s equal.
 *
 * attn_skip_lambda_for_target: lambda = alpha * exp(beta * S) / L for a target
 * sparsity S at context length L (the section's inference-time rule), capped
 * below 1; 0 for alpha <= 0 or L <= 0.
 */
double attn_skip_sparsity_at(const float *margin, int64_t n, double lambda);
attn_status attn_skip_lambda_for_sparsity(const float *margin, int64_t n, double target,
                                          double *lambda);
attn_status attn_skip_fit_lambda_model(const double *L, const double *sparsity,
                                       const double *lambda, int n, double *alpha, double *beta);
double attn_skip_lambda_for_target(double alpha, double beta, double sparsity, double L);

/*
 * Sampled decode output: the web page "Stochastic Sparse Attention for
 * Memory-Bound Inference" (SANTA), section "关键设计".  The softmax weights
 * p_i of a decode query over its L keys form a categorical distribution; with
 * the cumulative weights F_i = p_0 + ... + p_i, the inverse CDF of a threshold
 * T in [0, 1) is the smallest i with F_i > T, and
 *
 *     o = (1/S) * sum_{m<S} V[J_m],   J_m = inverse CDF of T_m,
 *
 * is an unbiased estimate of sum_i p_i V_i that reads S value rows instead of
 * L.  Thresholds ("SANTA 无偏估计 + Stratified/Systematic 降方差"):
 *   ATTN_SANTA_SYS:    T_m = (m + u[b,h]) / S     (the page's offset U ~
 *                      Unif[0, 1/S) is u / S; one draw per head)
 *   ATTN_SANTA_STRAT:  T_m = (m + u[b,h,m]) / S  (one draw per stratum)
 *   ATTN_SANTA_IID:    T_m = u[b,h,m]            (independent draws; sorted on
 *                      the device, idx[b,h,m] is still the index of draw m)
 * The caller draws u (uniform in [0, 1)); a value outside [0, 1) still yields
 * an in-range key index, but not the estimator.
 *
 * Schedule (item "S²ANTA-prop"): pass 1 streams the keys once per KV head and
 * writes every key's score (log2-scaled, fp32) to the `scores` stash and one
 * (max, sum of 2^(score - max)) pair per key tile and query head to
 * `tile_stats`; pass 2, per query head, turns the tile sums into the CDF at
 * the tile boundaries, gives each tile the thresholds that fall inside it,
 * places them on keys with the tile's running sum, and gathers the sampled
 * value rows.  A tile that receives no threshold costs no value read and no
 * second read of its scores.  Tile t holds the 128-key blocks
 * [floor(t*n_b/n_tiles), floor((t+1)*n_b/n_tiles)), n_b = ceil(L/128).
 *
 *  q           [B, Hq, dk]              bf16 (device)
 *  k, v        [B, Hkv, L, 128]         bf16 (device), row strides 128
 *  u           [B, Hq] (SYS) or [B, Hq, S] (STRAT, IID) fp32 (device)
 *  scores      [B, Hq, n_b * 128] fp32  (device, caller-owned workspace;
 *              keys past L hold -inf)
 *  tile_stats  [B, Hq, n_tiles, 2] fp32 (device, caller-owned workspace)
 *  o           [B, Hq, 128]             out_dt (device)
 *  idx         [B, Hq, S] int32         sample indices J_m (device) or NULL
 * Index decisions are taken in fp32: a threshold within rounding of a CDF
 * boundary may land on either neighbour.
 *
 * Kernels built: dt = ATTN_BF16, dk = dv = 128, row strides 128, G = Hq/Hkv
 * in {1, 2, 4, 8}, S <= 2048, n_tiles <= 1024, at most 16 blocks (2048 keys)
 * per tile; other valid combinations return ATTN_EUNSUPPORTED.  EINVAL for a
 * null required pointer, a non-positive size or count, Hq % Hkv != 0, a
 * stride below the head size, an unknown mode or dtype, or a misaligned
 * pointer.  Both workspaces are fully written before they are read.
 *
 * attn_skip_santa_workspace: the two workspace sizes, in floats.
 */
attn_status attn_skip_santa_workspace(int B, int Hq, int L, int n_tiles, size_t *scores_floats,
                                      size_t *stats_floats);
attn_status attn_skip_santa_decode(const void *q, const void *k, const void *v, attn_dtype dt,
                                   int B, int Hq, int Hkv, int L, int dk, int dv,
                                   int64_t k_row_stride, int64_t v_row_stride, float scale,
                                   int n_samples, attn_santa_mode mode, const float *u,
                                   int n_tiles, float *scores, float *tile_stats,
                                   attn_dtype out_dt, void *o, int32_t *idx, void *stream);

/*
 * attn_skip_santa_decode without caller workspaces.  The pages have no
 * counterpart: this is a convenience of this library for callers that cannot
 * allocate device memory when they decode (a host runtime whose plugin
 * interface passes only input and output pointers, an engine that reserved
 * all its device memory up front, a loop that cannot take the device-wide
 * synchronisation of cudaMalloc / cudaFree).
 *
 * Same arguments, meaning and results as attn_skip_santa_decode, minus
 * `scores` and `tile_stats`: both workspaces live in one fixed array in the
 * library's device memory (16.25 MiB, held on every device that loads the
 * library until the process exits).  The call allocates nothing: no
 * cudaMalloc, cudaFree or allocating library routine.
 *
 * Limits: B * Hq * ceil(L / 128) * 128 <= 4,194,304 (e.g. B = 4, Hq = 32,
 * L = 32768) and B * Hq * n_tiles * 2 <= 65,536; beyond either the call
 * returns ATTN_EINVAL before any CUDA call.  The other checks are those of
 * attn_skip_santa_decode.
 *
 * Set-up: every call looks up the array's device address with
 * cudaGetSymbolAddress in the context current on the calling thread (`stream`
 * must belong to its device); no address is kept between calls, so a
 * cudaDeviceReset or another context on the same device is followed
 * correctly.  The first call in a context can load the library's device code;
 * make that first call before any stream capture.  ATTN_ECUDA if the look-up
 * fails.
 *
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents.  Nothing in it needs clearing (the score pass writes both
 * parts in full before the sampling pass reads them), but two calls that
 * overlap on the GPU (different streams, or concurrent host threads without
 * ordering) race on it and both results are then undefined: order such calls
 * on one stream or with events.
 */
attn_status attn_skip_santa_decode_noalloc(const void *q, const void *k, const void *v,
                                           attn_dtype dt, int B, int Hq, int Hkv, int L, int dk,
                                           int dv, int64_t k_row_stride, int64_t v_row_stride,
                                           float scale, int n_samples, attn_santa_mode mode,
                                           const float *u, int n_tiles, attn_dtype out_dt,
                                           void *o, int32_t *idx, void *stream);

/*
 * Diagnostic: launches one small CTA that allocates TMEM and then waits, with
 * the same bounded wait as every kernel, on an mbarrier phase that nothing
 * completes.  After the 1 s limit the wait gives up, the CTA raises its abort
 * flag, frees its TMEM and exits, and the device error word records the
 * timeout, so a following attn_skip_last_device_error returns ATTN_ETIMEOUT
 * and the context stays usable.  Exercises the failure path without a fault.
 */
attn_status attn_skip_selftest_wait_timeout(void *stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word: ATTN_ETIMEOUT if a kernel gave up a bounded wait since the last read,
 * ATTN_EINVAL if a kernel found a device-side argument out of range (the
 * varlen lengths and thresholds), ATTN_EINTERNAL if a kernel found its shared
 * memory misaligned, ATTN_ECUDA on a CUDA error, else ATTN_OK.
 */
attn_status attn_skip_last_device_error(void *stream);

/* Static, human-readable name of a status code. */
const char *attn_skip_status_string(attn_status s);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_SKIP_H */
