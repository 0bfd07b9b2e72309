// C-ABI entry points: host-side validation, the log-domain threshold, the
// device error word, dispatch to the kernels, and the host-side threshold
// calibration helpers.  No entry point allocates device memory.
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include "../../include/attn_skip.h"
#include "internal.h"

namespace attn_skip {
namespace {

// One error word per device (a kernel that gives up a bounded wait ORs a bit in).
__device__ unsigned g_error_word;

// Device address of g_error_word in the context current on this thread,
// looked up on every call (a host-side table read once the module is loaded):
// a cached address would go stale after cudaDeviceReset or when another
// context is made current on the same device.
cudaError_t error_word(unsigned **out) {
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_error_word);
  if (e != cudaSuccess) return e;
  *out = (unsigned *)p;
  return cudaSuccess;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool lambda_ok(double lambda) { return lambda >= 0.0 && lambda < 1.0; }  // false for NaN

float ln_lambda(double lambda) {
  return lambda > 0.0 ? (float)log(lambda) : -INFINITY;
}

attn_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  cudaGetLastError();  // clear a sticky launch error so the caller can continue
  return ATTN_ECUDA;
}

}  // namespace
}  // namespace attn_skip

using namespace attn_skip;

namespace attn_skip {
namespace {

// Shared by attn_skip_prefill and attn_skip_prefill_margins: validation of
// the common arguments, the argument block, and dispatch.  `o`, `lse`,
// `bits` are null in statistics mode.
attn_status prefill_common(PrefillArgs &a, const void *q, const void *k, const void *v,
                           attn_dtype dt, int B, int Hq, int Hkv, int T, int dk, int dv,
                           float scale, double lambda, int Br, int Bc, int causal,
                           cudaStream_t s) {
  if (!q || !k || !v) return ATTN_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || dk <= 0 || dv <= 0 || Br <= 0 || Bc <= 0)
    return ATTN_EINVAL;
  if (Hq % Hkv != 0 || !lambda_ok(lambda) || !(scale == scale)) return ATTN_EINVAL;
  if (dt != ATTN_BF16 && dt != ATTN_F32) return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return ATTN_EINVAL;
  const long n_t = (T + (long)Br - 1) / Br, n_b = (T + (long)Bc - 1) / Bc;
  if ((long)B * Hq * n_t > 0x7fffffffL || (long)B * Hq * n_t * n_b > 0x7fffffffffffL)
    return ATTN_EUNSUPPORTED;
  a.q = q; a.k = k; a.v = v;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.T = T; a.dk = dk; a.dv = dv; a.Br = Br; a.Bc = Bc;
  a.causal = causal ? 1 : 0;
  a.n_t = (int)n_t; a.n_b = (int)n_b; a.words = (int)((n_b + 31) / 32);
  a.scale = scale > 0.f ? scale : (float)(1.0 / sqrt((double)dk));
  a.ln_lambda = ln_lambda(lambda);
  cudaError_t e = error_word(&a.err);
  if (e != cudaSuccess) return from_cuda(e);
  if (dt == ATTN_F32) {
    if (dk != dv || (dk != 32 && dk != 64) || (Br != 64 && Br != 128) || (Bc != 64 && Bc != 128))
      return ATTN_EUNSUPPORTED;
    return from_cuda(launch_prefill_f32(a, s));
  }
  if (dk != 128 || dv != 128 || Br != 128 || Bc != 128) return ATTN_EUNSUPPORTED;
  e = launch_prefill_tc(a, s);
  if (e == cudaErrorNotYetImplemented) return ATTN_EUNSUPPORTED;
  return from_cuda(e);
}

// Shared by attn_skip_decode and attn_skip_decode_margins.
attn_status decode_common(DecodeArgs &a, const void *q, const void *k, const void *v,
                          attn_dtype dt, int B, int Hq, int Hkv, int L, int dk, int dv,
                          int64_t k_row_stride, int64_t v_row_stride, float scale,
                          double lambda, int Bc, int n_splits, cudaStream_t s) {
  if (!q || !k || !v) return ATTN_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || dk <= 0 || dv <= 0 || Bc <= 0 || n_splits <= 0)
    return ATTN_EINVAL;
  if (Hq % Hkv != 0 || !lambda_ok(lambda) || !(scale == scale)) return ATTN_EINVAL;
  if (k_row_stride < dk || v_row_stride < dv) return ATTN_EINVAL;
  if (dt != ATTN_BF16 && dt != ATTN_F32) return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return ATTN_EINVAL;
  const int G = Hq / Hkv;
  const long n_b = (L + (long)Bc - 1) / Bc;
  if ((long)B * Hkv * n_splits > 0x7fffffffL) return ATTN_EUNSUPPORTED;
  a.q = q; a.k = k; a.v = v;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.L = L; a.dk = dk; a.dv = dv; a.Bc = Bc;
  a.n_splits = n_splits; a.k_row_stride = k_row_stride; a.v_row_stride = v_row_stride;
  a.n_b = (int)n_b;
  a.bps = (int)((n_b + n_splits - 1) / n_splits);
  a.words = (a.bps + 31) / 32;
  a.scale = scale > 0.f ? scale : (float)(1.0 / sqrt((double)dk));
  a.ln_lambda = ln_lambda(lambda);
  cudaError_t e = error_word(&a.err);
  if (e != cudaSuccess) return from_cuda(e);
  if (dt == ATTN_BF16 && dk == 128 && dv == 128 && Bc == 128 && k_row_stride == 128 &&
      v_row_stride == 128 && (G == 1 || G == 2 || G == 4 || G == 8))
    return from_cuda(launch_decode_bf16(a, s));
  // Absorbed MLA: one latent head of 576 columns, values = its first 512 columns.
  // Per-head decisions run in the cluster kernel (splits of up to its block
  // count).
  if (dt == ATTN_BF16 && dk == 576 && dv == 512 && v == k && k_row_stride == 576 &&
      v_row_stride == 576 && Bc == 64 && Hkv == 1 && Hq == 128) {
    if (a.per_head && (a.stats_only || a.bps > mla_cluster_max_bps())) return ATTN_EUNSUPPORTED;
    return from_cuda(launch_mla_decode(a, s));
  }
  return ATTN_EUNSUPPORTED;
}

}  // namespace
}  // namespace attn_skip

extern "C" attn_status attn_skip_prefill(const void *q, const void *k, const void *v,
                                         attn_dtype dt, int B, int Hq, int Hkv, int T, int dk,
                                         int dv, float scale, double lambda, int Br, int Bc,
                                         int causal, void *o, float *lse, uint32_t *skip_bits,
                                         void *stream) {
  if (!o || !lse || !skip_bits) return ATTN_EINVAL;
  if (!aligned16(o) || !aligned16(lse) || !aligned16(skip_bits)) return ATTN_EINVAL;
  PrefillArgs a{};
  a.o = o; a.lse = lse; a.bits = skip_bits;
  return prefill_common(a, q, k, v, dt, B, Hq, Hkv, T, dk, dv, scale, lambda, Br, Bc, causal,
                        (cudaStream_t)stream);
}

namespace attn_skip {
namespace {

// The argument checks of prefill_common and its choice of kernel, without a
// launch: ATTN_OK when prefill_common would launch.
attn_status prefill_check(const void *q, const void *k, const void *v, attn_dtype dt, int B,
                          int Hq, int Hkv, int T, int dk, int dv, float scale, double lambda,
                          int Br, int Bc) {
  if (!q || !k || !v) return ATTN_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || dk <= 0 || dv <= 0 || Br <= 0 || Bc <= 0)
    return ATTN_EINVAL;
  if (Hq % Hkv != 0 || !lambda_ok(lambda) || !(scale == scale)) return ATTN_EINVAL;
  if (dt != ATTN_BF16 && dt != ATTN_F32) return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return ATTN_EINVAL;
  const long n_t = (T + (long)Br - 1) / Br, n_b = (T + (long)Bc - 1) / Bc;
  if ((long)B * Hq * n_t > 0x7fffffffL || (long)B * Hq * n_t * n_b > 0x7fffffffffffL)
    return ATTN_EUNSUPPORTED;
  if (dt == ATTN_F32)
    return (dk != dv || (dk != 32 && dk != 64) || (Br != 64 && Br != 128) ||
            (Bc != 64 && Bc != 128))
               ? ATTN_EUNSUPPORTED
               : ATTN_OK;
  return (dk != 128 || dv != 128 || Br != 128 || Bc != 128) ? ATTN_EUNSUPPORTED : ATTN_OK;
}

}  // namespace
}  // namespace attn_skip

extern "C" attn_status attn_skip_prefill_from_host(
    const void *q_host, const void *k_host, const void *v_host, void *q_dev, void *k_dev,
    void *v_dev, attn_dtype dt, int B, int Hq, int Hkv, int T, int dk, int dv, float scale,
    double lambda, int Br, int Bc, int causal, void *o_dev, float *lse_dev, uint32_t *skip_bits,
    void *o_host, float *lse_host, int n_groups, void *stream, void *copy_in_stream,
    void *copy_out_stream) {
  if (!q_host || !k_host || !v_host || !o_host || !lse_host) return ATTN_EINVAL;
  if (!o_dev || !lse_dev || !skip_bits) return ATTN_EINVAL;
  if (!aligned16(o_dev) || !aligned16(lse_dev) || !aligned16(skip_bits)) return ATTN_EINVAL;
  attn_status st =
      prefill_check(q_dev, k_dev, v_dev, dt, B, Hq, Hkv, T, dk, dv, scale, lambda, Br, Bc);
  if (st != ATTN_OK) return st;
  const long rows = (long)B * Hkv;  // KV heads, batch-major
  if (n_groups == 0) n_groups = (int)(rows < 8 ? rows : 8);
  if (n_groups < 1 || n_groups > rows) return ATTN_EINVAL;
  const int G = Hq / Hkv;
  const size_t es = dt == ATTN_F32 ? 4 : 2;
  const long n_t = (T + (long)Br - 1) / Br, words = ((T + (long)Bc - 1) / Bc + 31) / 32;
  // Per KV head: its G query heads' rows of Q, O, LSE and the bitmap, its K and V.
  const size_t q_row = (size_t)G * T * dk * es, o_row = (size_t)G * T * dv * es;
  const size_t k_row = (size_t)T * dk * es, v_row = (size_t)T * dv * es;
  const size_t l_row = (size_t)G * T, b_row = (size_t)G * n_t * words;
  cudaStream_t s = (cudaStream_t)stream;
  cudaStream_t si = copy_in_stream ? (cudaStream_t)copy_in_stream : s;
  cudaStream_t so = copy_out_stream ? (cudaStream_t)copy_out_stream : s;
  // 8 groups of the T = 16384 prefill (32/8 heads) overlap 337 MB of copies
  // with the computation: 2.85 -> 1.49 ms per call against copies in, prefill,
  // copies out in sequence.
  // Events: [0] `stream` at the call (the staging buffers are free), then per
  // group its inputs in and its results computed, last the copies out done.
  const int n_ev = 2 * n_groups + 2;
  cudaEvent_t *ev = (cudaEvent_t *)calloc((size_t)n_ev, sizeof(cudaEvent_t));
  if (!ev) return ATTN_EINTERNAL;
  cudaError_t e = cudaSuccess;
  int made = 0;
  for (; made < n_ev && e == cudaSuccess; ++made)
    e = cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming);
  if (e != cudaSuccess) --made;  // the failed create made no event
  auto uc = [](const void *p, size_t off) { return (const char *)p + off; };
  auto um = [](void *p, size_t off) { return (char *)p + off; };
  if (e == cudaSuccess) e = cudaEventRecord(ev[0], s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(si, ev[0], 0);
  for (int g = 0; g < n_groups && e == cudaSuccess && st == ATTN_OK; ++g) {
    const long r0 = rows * g / n_groups, r1 = rows * (g + 1) / n_groups, nr = r1 - r0;
    cudaEvent_t in = ev[1 + 2 * g], done = ev[2 + 2 * g];
    e = cudaMemcpyAsync(um(q_dev, r0 * q_row), uc(q_host, r0 * q_row), nr * q_row,
                        cudaMemcpyHostToDevice, si);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(um(k_dev, r0 * k_row), uc(k_host, r0 * k_row), nr * k_row,
                          cudaMemcpyHostToDevice, si);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(um(v_dev, r0 * v_row), uc(v_host, r0 * v_row), nr * v_row,
                          cudaMemcpyHostToDevice, si);
    if (e == cudaSuccess) e = cudaEventRecord(in, si);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, in, 0);
    if (e != cudaSuccess) break;
    // This group as its own batch: nr "sequences" of one KV head and G query heads.
    PrefillArgs a{};
    a.o = um(o_dev, r0 * o_row);
    a.lse = lse_dev + r0 * l_row;
    a.bits = skip_bits + r0 * b_row;
    st = prefill_common(a, um(q_dev, r0 * q_row), um(k_dev, r0 * k_row), um(v_dev, r0 * v_row),
                        dt, (int)nr, G, 1, T, dk, dv, scale, lambda, Br, Bc, causal, s);
    if (st != ATTN_OK) break;
    e = cudaEventRecord(done, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(so, done, 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(um(o_host, r0 * o_row), uc(o_dev, r0 * o_row), nr * o_row,
                          cudaMemcpyDeviceToHost, so);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(lse_host + r0 * l_row, lse_dev + r0 * l_row,
                          nr * l_row * sizeof(float), cudaMemcpyDeviceToHost, so);
  }
  // `stream` reaches the end of the call once the last copy out has landed.
  if (e == cudaSuccess && st == ATTN_OK) e = cudaEventRecord(ev[n_ev - 1], so);
  if (e == cudaSuccess && st == ATTN_OK) e = cudaStreamWaitEvent(s, ev[n_ev - 1], 0);
  for (int i = 0; i < made; ++i) cudaEventDestroy(ev[i]);
  free(ev);
  if (st != ATTN_OK) return st;
  return e == cudaSuccess ? ATTN_OK : from_cuda(e);
}

extern "C" attn_status attn_skip_prefill_blocks(const void *q, const void *k, const void *v,
                                                attn_dtype dt, int B, int Hq, int Hkv, int T,
                                                int dk, int dv, float scale, double lambda,
                                                int Br, int Bc, int causal,
                                                const uint32_t *block_set, void *o, float *lse,
                                                uint32_t *skip_bits, void *stream) {
  if (!block_set || !o || !lse || !skip_bits) return ATTN_EINVAL;
  if (!aligned16(block_set) || !aligned16(o) || !aligned16(lse) || !aligned16(skip_bits))
    return ATTN_EINVAL;
  PrefillArgs a{};
  a.o = o; a.lse = lse; a.bits = skip_bits; a.block_set = block_set;
  return prefill_common(a, q, k, v, dt, B, Hq, Hkv, T, dk, dv, scale, lambda, Br, Bc, causal,
                        (cudaStream_t)stream);
}

extern "C" attn_status attn_skip_prefill_varlen(const void *q, const void *k, const void *v,
                                                attn_dtype dt, int n_seq,
                                                const int32_t *cu_seqlens, int max_seqlen,
                                                int total, int Hq, int Hkv, int dk, int dv,
                                                float scale, const float *lambda, int Br, int Bc,
                                                int causal, void *o, float *lse,
                                                uint32_t *skip_bits, void *stream) {
  if (!cu_seqlens || !lambda) return ATTN_EINVAL;
  if (n_seq <= 0 || max_seqlen < 0 || total < 0 || Hq <= 0 || Hkv <= 0 || dk <= 0 || dv <= 0 ||
      Br <= 0 || Bc <= 0)
    return ATTN_EINVAL;
  // With no token the tensors may be empty (null); the bitmap is needed
  // whenever there is a tile row.
  if (total > 0 && (!q || !k || !v || !o || !lse)) return ATTN_EINVAL;
  if (max_seqlen > 0 && !skip_bits) return ATTN_EINVAL;
  if (Hq % Hkv != 0 || !(scale == scale)) return ATTN_EINVAL;
  if (dt != ATTN_BF16 && dt != ATTN_F32) return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(skip_bits) || ((uintptr_t)cu_seqlens & 3u) || ((uintptr_t)lambda & 3u))
    return ATTN_EINVAL;
  if (dt != ATTN_BF16 || dk != 128 || dv != 128 || Br != 128 || Bc != 128)
    return ATTN_EUNSUPPORTED;
  const long n_t = (max_seqlen + 127L) / 128;
  if ((long)n_seq * Hq * n_t > 0x7fffffffL ||
      (long)Hq * ((total + 127L) / 128 + n_seq) > 0x7fffffffL)
    return ATTN_EUNSUPPORTED;
  if (n_t == 0) return ATTN_OK;  // every sequence is empty: no tile, no bitmap word
  if (total == 0)                 // every sequence is empty: only the bitmap to clear
    return from_cuda(cudaMemsetAsync(skip_bits, 0,
                                     (size_t)n_seq * Hq * n_t * ((n_t + 31) / 32) * 4,
                                     (cudaStream_t)stream));
  PrefillArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse; a.bits = skip_bits;
  a.B = n_seq; a.Hq = Hq; a.Hkv = Hkv; a.T = max_seqlen; a.dk = dk; a.dv = dv;
  a.Br = Br; a.Bc = Bc; a.causal = causal ? 1 : 0;
  a.n_t = (int)n_t; a.n_b = (int)n_t; a.words = (int)((n_t + 31) / 32);
  a.scale = scale > 0.f ? scale : (float)(1.0 / sqrt((double)dk));
  a.ln_lambda = -INFINITY;  // per sequence from lambda[]
  a.cu_seqlens = cu_seqlens; a.lambda_seq = lambda; a.total = total;
  cudaError_t e = error_word(&a.err);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(launch_prefill_tc(a, (cudaStream_t)stream));
}

extern "C" attn_status attn_skip_prefill_margins(const void *q, const void *k, attn_dtype dt,
                                                 int B, int Hq, int Hkv, int T, int dk,
                                                 float scale, int Br, int Bc, int causal,
                                                 float *margin, void *stream) {
  if (!margin || !aligned16(margin)) return ATTN_EINVAL;
  PrefillArgs a{};
  a.margin = margin;
  a.stats_only = 1;
  // No value is read in statistics mode; the key tensor stands in for it.
  return prefill_common(a, q, k, k, dt, B, Hq, Hkv, T, dk, dk, scale, 0.0, Br, Bc, causal,
                        (cudaStream_t)stream);
}

extern "C" attn_status attn_skip_decode(const void *q, const void *k, const void *v,
                                        attn_dtype dt, int B, int Hq, int Hkv, int L, int dk,
                                        int dv, int64_t k_row_stride, int64_t v_row_stride,
                                        float scale, double lambda, int Bc, int n_splits,
                                        float *o_part, float *lse_part, uint32_t *skip_bits,
                                        void *stream) {
  if (!o_part || !lse_part || !skip_bits) return ATTN_EINVAL;
  if (!aligned16(o_part) || !aligned16(lse_part) || !aligned16(skip_bits)) return ATTN_EINVAL;
  DecodeArgs a{};
  a.o_part = o_part; a.lse_part = lse_part; a.bits = skip_bits;
  return decode_common(a, q, k, v, dt, B, Hq, Hkv, L, dk, dv, k_row_stride, v_row_stride, scale,
                       lambda, Bc, n_splits, (cudaStream_t)stream);
}

extern "C" attn_status attn_skip_decode_per_head(const void *q, const void *k, const void *v,
                                                 attn_dtype dt, int B, int Hq, int Hkv, int L,
                                                 int dk, int dv, int64_t k_row_stride,
                                                 int64_t v_row_stride, float scale,
                                                 double lambda, int Bc, int n_splits,
                                                 float *o_part, float *lse_part,
                                                 uint32_t *skip_bits, void *stream) {
  if (!o_part || !lse_part || !skip_bits) return ATTN_EINVAL;
  if (!aligned16(o_part) || !aligned16(lse_part) || !aligned16(skip_bits)) return ATTN_EINVAL;
  DecodeArgs a{};
  a.o_part = o_part; a.lse_part = lse_part; a.bits = skip_bits; a.per_head = 1;
  return decode_common(a, q, k, v, dt, B, Hq, Hkv, L, dk, dv, k_row_stride, v_row_stride, scale,
                       lambda, Bc, n_splits, (cudaStream_t)stream);
}

extern "C" attn_status attn_skip_decode_margins(const void *q, const void *k, attn_dtype dt,
                                                int B, int Hq, int Hkv, int L, int dk,
                                                int64_t k_row_stride, float scale, int Bc,
                                                int n_splits, float *margin, void *stream) {
  if (!margin || !aligned16(margin)) return ATTN_EINVAL;
  DecodeArgs a{};
  a.margin = margin;
  a.stats_only = 1;
  // The value view is never read in statistics mode: the MLA layout (values =
  // the first 512 latent columns) or the key tensor itself.
  const int dv = dk == 576 ? 512 : dk;
  return decode_common(a, q, k, k, dt, B, Hq, Hkv, L, dk, dv, k_row_stride, k_row_stride, scale,
                       0.0, Bc, n_splits, (cudaStream_t)stream);
}

extern "C" attn_status attn_skip_decode_fp8(const void *q, const void *k, const void *v,
                                            const float *k_scale, const float *v_scale, int B,
                                            int Hq, int Hkv, int L, int dk, int dv,
                                            int64_t k_row_stride, int64_t v_row_stride,
                                            float scale, double lambda, int Bc, int n_splits,
                                            float *o_part, float *lse_part, uint32_t *skip_bits,
                                            void *stream) {
  if (!q || !k || !v || !k_scale || !v_scale || !o_part || !lse_part || !skip_bits)
    return ATTN_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || dk <= 0 || dv <= 0 || Bc <= 0 || n_splits <= 0)
    return ATTN_EINVAL;
  if (Hq % Hkv != 0 || !lambda_ok(lambda) || !(scale == scale)) return ATTN_EINVAL;
  if (k_row_stride < dk || v_row_stride < dv) return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_part) ||
      !aligned16(lse_part) || !aligned16(skip_bits) || ((uintptr_t)k_scale & 3u) ||
      ((uintptr_t)v_scale & 3u))
    return ATTN_EINVAL;
  const int G = Hq / Hkv;
  if (dk != 128 || dv != 128 || Bc != 128 || !(G == 1 || G == 2 || G == 4 || G == 8) ||
      (k_row_stride % 16) || (v_row_stride % 16))
    return ATTN_EUNSUPPORTED;
  const long n_b = (L + (long)Bc - 1) / Bc;
  if ((long)B * Hkv * n_splits > 0x7fffffffL) return ATTN_EUNSUPPORTED;
  DecodeArgs a{};
  a.q = q; a.k = k; a.v = v; a.k_scale = k_scale; a.v_scale = v_scale;
  a.o_part = o_part; a.lse_part = lse_part; a.bits = skip_bits;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.L = L; a.dk = dk; a.dv = dv; a.Bc = Bc;
  a.n_splits = n_splits; a.k_row_stride = k_row_stride; a.v_row_stride = v_row_stride;
  a.n_b = (int)n_b;
  a.bps = (int)((n_b + n_splits - 1) / n_splits);
  a.words = (a.bps + 31) / 32;
  a.scale = scale > 0.f ? scale : (float)(1.0 / sqrt((double)dk));
  a.ln_lambda = ln_lambda(lambda);
  cudaError_t e = error_word(&a.err);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(launch_decode_fp8(a, (cudaStream_t)stream));
}

extern "C" attn_status attn_skip_decode_nvfp4(const void *q, const void *k4, const void *v4,
                                              const uint8_t *k_bs, const uint8_t *v_bs,
                                              const float *k_scale, const float *v_scale, int B,
                                              int Hq, int Hkv, int L, int dk, int dv,
                                              int64_t k_row_stride, int64_t v_row_stride,
                                              float scale, double lambda, int Bc, int n_splits,
                                              float *o_part, float *lse_part,
                                              uint32_t *skip_bits, void *stream) {
  if (!q || !k4 || !v4 || !k_bs || !v_bs || !k_scale || !v_scale || !o_part || !lse_part ||
      !skip_bits)
    return ATTN_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || dk <= 0 || dv <= 0 || Bc <= 0 || n_splits <= 0)
    return ATTN_EINVAL;
  if (Hq % Hkv != 0 || !lambda_ok(lambda) || !(scale == scale)) return ATTN_EINVAL;
  if ((dk % 16) || (dv % 16) || k_row_stride < dk / 2 || v_row_stride < dv / 2)
    return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(k4) || !aligned16(v4) || !aligned16(k_bs) ||
      !aligned16(v_bs) || !aligned16(o_part) || !aligned16(lse_part) || !aligned16(skip_bits) ||
      ((uintptr_t)k_scale & 3u) || ((uintptr_t)v_scale & 3u))
    return ATTN_EINVAL;
  const int G = Hq / Hkv;
  if (dk != 128 || dv != 128 || Bc != 128 || !(G == 1 || G == 2 || G == 4 || G == 8) ||
      (k_row_stride % 16) || (v_row_stride % 16))
    return ATTN_EUNSUPPORTED;
  const long n_b = (L + (long)Bc - 1) / Bc;
  if ((long)B * Hkv * n_splits > 0x7fffffffL || (long)B * Hkv * L > 0x7fffffffL)
    return ATTN_EUNSUPPORTED;
  DecodeArgs a{};
  a.q = q; a.k = k4; a.v = v4; a.k_bs = k_bs; a.v_bs = v_bs;
  a.k_scale = k_scale; a.v_scale = v_scale;
  a.o_part = o_part; a.lse_part = lse_part; a.bits = skip_bits;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.L = L; a.dk = dk; a.dv = dv; a.Bc = Bc;
  a.n_splits = n_splits; a.k_row_stride = k_row_stride; a.v_row_stride = v_row_stride;
  a.n_b = (int)n_b;
  a.bps = (int)((n_b + n_splits - 1) / n_splits);
  a.words = (a.bps + 31) / 32;
  a.scale = scale > 0.f ? scale : (float)(1.0 / sqrt((double)dk));
  a.ln_lambda = ln_lambda(lambda);
  cudaError_t e = error_word(&a.err);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(launch_decode_nvfp4(a, (cudaStream_t)stream));
}

extern "C" attn_status attn_skip_decode_combine(const float *o_part, const float *lse_part, int B,
                                                int Hq, int n_splits, int dv, attn_dtype out_dt,
                                                void *o, float *lse, void *stream) {
  if (!o_part || !lse_part || !o || !lse) return ATTN_EINVAL;
  if (B <= 0 || Hq <= 0 || n_splits <= 0 || dv <= 0) return ATTN_EINVAL;
  if (out_dt != ATTN_BF16 && out_dt != ATTN_F32) return ATTN_EINVAL;
  if (!aligned16(o_part) || !aligned16(lse_part) || !aligned16(o) || !aligned16(lse))
    return ATTN_EINVAL;
  if (n_splits > 1024 || (long)B * Hq > 0x7fffffffL) return ATTN_EUNSUPPORTED;
  CombineArgs a{};
  a.o_part = o_part; a.lse_part = lse_part; a.o = o; a.lse = lse;
  a.B = B; a.Hq = Hq; a.n_splits = n_splits; a.dv = dv; a.out_bf16 = out_dt == ATTN_BF16;
  return from_cuda(launch_combine(a, (cudaStream_t)stream));
}

extern "C" attn_status attn_skip_santa_workspace(int B, int Hq, int L, int n_tiles,
                                                 size_t *scores_floats, size_t *stats_floats) {
  if (B <= 0 || Hq <= 0 || L <= 0 || n_tiles <= 0 || !scores_floats || !stats_floats)
    return ATTN_EINVAL;
  const size_t n_b = ((size_t)L + 127) / 128;
  *scores_floats = (size_t)B * Hq * n_b * 128;
  *stats_floats = (size_t)B * Hq * n_tiles * 2;
  return ATTN_OK;
}

extern "C" attn_status attn_skip_santa_decode(const void *q, const void *k, const void *v,
                                              attn_dtype dt, int B, int Hq, int Hkv, int L, int dk,
                                              int dv, int64_t k_row_stride, int64_t v_row_stride,
                                              float scale, int n_samples, attn_santa_mode mode,
                                              const float *u, int n_tiles, float *scores,
                                              float *tile_stats, attn_dtype out_dt, void *o,
                                              int32_t *idx, void *stream) {
  if (!q || !k || !v || !u || !scores || !tile_stats || !o) return ATTN_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || dk <= 0 || dv <= 0 || n_samples <= 0 ||
      n_tiles <= 0)
    return ATTN_EINVAL;
  if (Hq % Hkv != 0 || !(scale == scale) || k_row_stride < dk || v_row_stride < dv)
    return ATTN_EINVAL;
  if (mode != ATTN_SANTA_IID && mode != ATTN_SANTA_SYS && mode != ATTN_SANTA_STRAT)
    return ATTN_EINVAL;
  if ((dt != ATTN_BF16 && dt != ATTN_F32) || (out_dt != ATTN_BF16 && out_dt != ATTN_F32))
    return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(u) || !aligned16(scores) ||
      !aligned16(tile_stats) || !aligned16(o) || (idx && !aligned16(idx)))
    return ATTN_EINVAL;
  const int G = Hq / Hkv;
  const long n_b = (L + 127L) / 128;
  const long bps = (n_b + n_tiles - 1) / n_tiles;
  if (dt != ATTN_BF16 || dk != 128 || dv != 128 || k_row_stride != 128 || v_row_stride != 128 ||
      !(G == 1 || G == 2 || G == 4 || G == 8))
    return ATTN_EUNSUPPORTED;
  if (n_samples > 2048 || n_tiles > 1024 || bps > 16 || (long)B * Hkv * n_tiles > 0x7fffffffL ||
      (long)B * Hq > 0x7fffffffL)
    return ATTN_EUNSUPPORTED;
  if (santa_sample_smem_bytes(n_tiles, n_samples) > 200 * 1024) return ATTN_EUNSUPPORTED;
  SantaArgs a{};
  a.q = q; a.k = k; a.v = v; a.u = u; a.scores = scores; a.tile_stats = tile_stats;
  a.o = o; a.idx = idx;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.L = L; a.n_b = (int)n_b; a.n_tiles = n_tiles;
  a.bps = (int)bps; a.S = n_samples; a.mode = (int)mode; a.out_bf16 = out_dt == ATTN_BF16;
  a.scale = scale > 0.f ? scale : (float)(1.0 / sqrt((double)dk));
  cudaError_t e = error_word(&a.err);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(launch_santa_decode(a, (cudaStream_t)stream));
}

extern "C" attn_status attn_skip_selftest_wait_timeout(void *stream) {
  unsigned *err = nullptr;
  cudaError_t e = error_word(&err);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(launch_selftest_wait(err, (cudaStream_t)stream));
}

extern "C" attn_status attn_skip_last_device_error(void *stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return from_cuda(e);
  unsigned word = 0;
  e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word));
  if (e != cudaSuccess) return from_cuda(e);
  if (word) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return from_cuda(e);
    return (word & kErrTimeout)  ? ATTN_ETIMEOUT
           : (word & kErrBadArg) ? ATTN_EINVAL
           : (word & kErrLayout) ? ATTN_EINTERNAL
                                 : ATTN_ECUDA;
  }
  return ATTN_OK;
}

namespace attn_skip {
namespace {
int cmp_float(const void *x, const void *y) {
  const float a = *(const float *)x, b = *(const float *)y;
  return (a > b) - (a < b);
}
}  // namespace
}  // namespace attn_skip

extern "C" double attn_skip_sparsity_at(const float *margin, int64_t n, double lambda) {
  if (!margin || n < 0 || !(lambda >= 0.0 && lambda < 1.0)) return -1.0;
  const double ln_l = lambda > 0.0 ? log(lambda) : -INFINITY;
  int64_t trav = 0, skipped = 0;
  for (int64_t i = 0; i < n; ++i) {
    const float x = margin[i];
    if (x != x) continue;
    ++trav;
    if (lambda > 0.0 && (double)x < ln_l) ++skipped;
  }
  return trav ? (double)skipped / (double)trav : 0.0;
}

extern "C" attn_status attn_skip_lambda_for_sparsity(const float *margin, int64_t n,
                                                     double target, double *lambda) {
  if (!margin || !lambda || n <= 0 || !(target >= 0.0 && target <= 1.0)) return ATTN_EINVAL;
  // Traversed entries (NaN = not traversed), ascending; -inf sorts first.
  float *v = (float *)malloc(sizeof(float) * (size_t)n);
  if (!v) return ATTN_EINVAL;
  int64_t m = 0, neg = 0;
  for (int64_t i = 0; i < n; ++i) {
    const float x = margin[i];
    if (x != x) continue;
    v[m++] = x;
    if (x < 0.f) ++neg;  // a statistic of 0 (a row found a new max) is never skipped
  }
  if (m == 0) {
    free(v);
    return ATTN_EINVAL;
  }
  qsort(v, (size_t)m, sizeof(float), cmp_float);
  int64_t k = (int64_t)llround(target * (double)m);  // entries to skip
  if (k > neg) k = neg;                               // the most any lambda < 1 skips
  double ln_l;
  if (k == 0) {
    *lambda = 0.0;
    free(v);
    return ATTN_OK;
  }
  const double lo = v[k - 1];                   // largest skipped statistic
  const double hi = k < m ? (double)v[k] : 0.0;  // smallest kept one
  if (lo == -INFINITY) ln_l = hi == -INFINITY ? -1e30 : hi - 1.0;
  else ln_l = 0.5 * (lo + (hi < 0.0 ? hi : 0.0));
  free(v);
  *lambda = exp(ln_l);
  if (!(*lambda < 1.0)) *lambda = nextafter(1.0, 0.0);
  return ATTN_OK;
}

extern "C" double attn_skip_lambda_for_target(double alpha, double beta, double sparsity,
                                              double L) {
  if (!(alpha > 0.0) || !(L > 0.0) || !(sparsity == sparsity) || !(beta == beta)) return 0.0;
  const double lambda = alpha * exp(beta * sparsity) / L;
  return lambda < 1.0 ? lambda : nextafter(1.0, 0.0);
}

extern "C" attn_status attn_skip_fit_lambda_model(const double *L, const double *sparsity,
                                                  const double *lambda, int n, double *alpha,
                                                  double *beta) {
  if (!L || !sparsity || !lambda || !alpha || !beta || n < 2) return ATTN_EINVAL;
  // Least squares on ln(lambda * L) = ln(alpha) + beta * sparsity.
  double sx = 0, sy = 0, sxx = 0, sxy = 0;
  for (int i = 0; i < n; ++i) {
    if (!(L[i] > 0.0) || !(lambda[i] > 0.0) || !(sparsity[i] == sparsity[i])) return ATTN_EINVAL;
    const double x = sparsity[i], y = log(lambda[i] * L[i]);
    sx += x; sy += y; sxx += x * x; sxy += x * y;
  }
  const double den = n * sxx - sx * sx;
  if (!(fabs(den) > 1e-300)) return ATTN_EINVAL;  // all sparsities equal
  *beta = (n * sxy - sx * sy) / den;
  *alpha = exp((sy - *beta * sx) / n);
  return ATTN_OK;
}

extern "C" const char *attn_skip_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_EINVAL: return "invalid argument";
    case ATTN_EUNSUPPORTED: return "unsupported combination (no kernel built for it)";
    case ATTN_ECUDA: return "CUDA error";
    case ATTN_ETIMEOUT: return "device-side bounded wait timed out";
    case ATTN_EINTERNAL: return "kernel shared-memory layout misaligned (internal error)";
  }
  return "unknown status";
}
