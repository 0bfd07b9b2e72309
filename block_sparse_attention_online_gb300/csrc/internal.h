// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
// Not part of the public ABI.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn_skip {

// Bits of the device error word.
enum : unsigned {
  kErrTimeout = 1u,  // a bounded mbarrier / flag wait gave up
  kErrBadArg = 2u,   // a device-side argument (a varlen length or threshold) was out of range
  kErrLayout = 4u,   // the dynamic shared-memory base was not 1024-byte aligned
};

struct PrefillArgs {
  const void *q, *k, *v;
  void *o;
  float *lse;
  uint32_t *bits;
  int B, Hq, Hkv, T, dk, dv, Br, Bc, causal;
  int n_t, n_b, words;  // tiles, blocks, bitmap words per tile
  float scale;          // natural-log scale applied to q.k
  float ln_lambda;      // -inf when lambda == 0
  unsigned *err;        // device error word
  // Statistics mode: margin [B,Hq,n_t,n_b] receives each traversed block's
  // statistic max_r(rowmax_r - m_new_r) (natural log; NaN = not traversed),
  // every block is treated as skipped, and o, lse, bits are not written.
  float *margin;
  int stats_only;
  // Explicit block set: [B,Hq,n_t,words] bit masks, bit j = block j is
  // traversed (within the causal range); null = every block.
  const uint32_t *block_set;
  // Variable-length batch: B sequences packed token-major, sequence b at
  // tokens [cu_seqlens[b], cu_seqlens[b+1]) of q [total,Hq,128], k and v
  // [total,Hkv,128] and o [total,Hq,128]; lse [Hq,total]; threshold
  // lambda_seq[b]; T = the longest length.  Null cu_seqlens = fixed length.
  const int32_t *cu_seqlens;
  const float *lambda_seq;
  int total;
};

struct DecodeArgs {
  const void *q, *k, *v;
  float *o_part, *lse_part;
  uint32_t *bits;
  int B, Hq, Hkv, L, dk, dv, Bc, n_splits;
  int64_t k_row_stride, v_row_stride;
  int n_b, bps, words;  // blocks, blocks per split (max), bitmap words per split
  float scale;
  float ln_lambda;
  unsigned *err;
  // Statistics mode: margin [B,Hkv,n_splits,bps] receives each block's
  // statistic over the query heads of the KV head (NaN past a split's last
  // block); every block is treated as skipped; o_part, lse_part, bits unused.
  float *margin;
  int stats_only;
  // Per-head decisions: bits [B,Hq,n_splits,words], each query head decides
  // for itself (the GQA kernel only).
  int per_head;
  // FP8 (E4M3) cache: k and v hold codes; one fp32 scale per (b, KV head)
  // for keys (multiplies the scores) and values (multiplies the outputs).
  const float *k_scale, *v_scale;
  // NVFP4 cache: k and v hold packed E2M1 codes [.., L, d/2], k_bs and v_bs
  // the E4M3 block scales [B,Hkv,L,d/16] (one per 16 elements of a row).
  const uint8_t *k_bs, *v_bs;
};

// Sampled decode output (SANTA estimator).
enum : int { kSantaIid = 0, kSantaSys = 1, kSantaStrat = 2 };

struct SantaArgs {
  const void *q, *k, *v;     // bf16 [B,Hq,128], [B,Hkv,L,128], [B,Hkv,L,128]
  const float *u;            // [B,Hq] (systematic) or [B,Hq,S] (stratified), in [0,1)
  float *scores;             // [B,Hq,n_b*128] stash: log2-scaled scores, -inf past L
  float *tile_stats;         // [B,Hq,n_tiles] (max, sum) pairs
  void *o;                   // [B,Hq,128] fp32 or bf16
  int32_t *idx;              // [B,Hq,S] sample indices, or null
  int B, Hq, Hkv, L, n_b, n_tiles, bps, S, mode, out_bf16;
  float scale;
  unsigned *err;
};

struct CombineArgs {
  const float *o_part, *lse_part;
  void *o;
  float *lse;
  int B, Hq, n_splits, dv;
  int out_bf16;
};

cudaError_t launch_prefill_f32(const PrefillArgs &a, cudaStream_t s);
cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t s);
cudaError_t launch_decode_bf16(const DecodeArgs &a, cudaStream_t s);
cudaError_t launch_mla_decode(const DecodeArgs &a, cudaStream_t s);
cudaError_t launch_mla_cluster(const DecodeArgs &a, cudaStream_t s);
int mla_cluster_max_bps();
cudaError_t launch_decode_fp8(const DecodeArgs &a, cudaStream_t s);
cudaError_t launch_decode_nvfp4(const DecodeArgs &a, cudaStream_t s);
cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s);
cudaError_t launch_selftest_wait(unsigned *err, cudaStream_t s);
cudaError_t launch_santa_decode(const SantaArgs &a, cudaStream_t s);
size_t santa_sample_smem_bytes(int n_tiles, int S);

}  // namespace attn_skip
