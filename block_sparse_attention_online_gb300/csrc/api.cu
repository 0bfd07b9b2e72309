// C-ABI entry points: host-side validation, the log-domain threshold, the
// device error word, and dispatch to the kernels.  No entry point allocates
// device memory.
#include <math.h>
#include <stdint.h>

#include "../../include/attn_skip.h"
#include "internal.h"

namespace attn_skip {
namespace {

// One error word per device (a kernel that gives up a bounded wait ORs a bit in).
__device__ unsigned g_error_word;

constexpr int kMaxDevices = 64;
unsigned *g_err_ptr[kMaxDevices];

cudaError_t error_word(unsigned **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!g_err_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_error_word);
    if (e != cudaSuccess) return e;
    g_err_ptr[dev] = (unsigned *)p;
  }
  *out = g_err_ptr[dev];
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

extern "C" attn_status attn_skip_prefill(const void *q, const void *k, const void *v,
                                         attn_dtype dt, int B, int Hq, int Hkv, int T, int dk,
                                         int dv, float scale, double lambda, int Br, int Bc,
                                         int causal, void *o, float *lse, uint32_t *skip_bits,
                                         void *stream) {
  if (!q || !k || !v || !o || !lse || !skip_bits) return ATTN_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || dk <= 0 || dv <= 0 || Br <= 0 || Bc <= 0)
    return ATTN_EINVAL;
  if (Hq % Hkv != 0 || !lambda_ok(lambda) || !(scale == scale)) return ATTN_EINVAL;
  if (dt != ATTN_BF16 && dt != ATTN_F32) return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(skip_bits))
    return ATTN_EINVAL;
  const long n_t = (T + (long)Br - 1) / Br, n_b = (T + (long)Bc - 1) / Bc;
  if ((long)B * Hq * n_t > 0x7fffffffL) return ATTN_EUNSUPPORTED;

  PrefillArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse; a.bits = skip_bits;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.T = T; a.dk = dk; a.dv = dv; a.Br = Br; a.Bc = Bc;
  a.causal = causal ? 1 : 0;
  a.n_t = (int)n_t; a.n_b = (int)n_b; a.words = (int)((n_b + 31) / 32);
  a.scale = scale > 0.f ? scale : (float)(1.0 / sqrt((double)dk));
  a.ln_lambda = ln_lambda(lambda);
  cudaError_t e = error_word(&a.err);
  if (e != cudaSuccess) return from_cuda(e);
  cudaStream_t s = (cudaStream_t)stream;

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

extern "C" attn_status attn_skip_decode(const void *q, const void *k, const void *v,
                                        attn_dtype dt, int B, int Hq, int Hkv, int L, int dk,
                                        int dv, int64_t k_row_stride, int64_t v_row_stride,
                                        float scale, double lambda, int Bc, int n_splits,
                                        float *o_part, float *lse_part, uint32_t *skip_bits,
                                        void *stream) {
  if (!q || !k || !v || !o_part || !lse_part || !skip_bits) return ATTN_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || dk <= 0 || dv <= 0 || Bc <= 0 || n_splits <= 0)
    return ATTN_EINVAL;
  if (Hq % Hkv != 0 || !lambda_ok(lambda) || !(scale == scale)) return ATTN_EINVAL;
  if (k_row_stride < dk || v_row_stride < dv) return ATTN_EINVAL;
  if (dt != ATTN_BF16 && dt != ATTN_F32) return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_part) ||
      !aligned16(lse_part) || !aligned16(skip_bits))
    return ATTN_EINVAL;
  const int G = Hq / Hkv;
  const long n_b = (L + (long)Bc - 1) / Bc;
  if ((long)B * Hkv * n_splits > 0x7fffffffL) return ATTN_EUNSUPPORTED;

  DecodeArgs a{};
  a.q = q; a.k = k; a.v = v; a.o_part = o_part; a.lse_part = lse_part; a.bits = skip_bits;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.L = L; a.dk = dk; a.dv = dv; a.Bc = Bc;
  a.n_splits = n_splits; a.k_row_stride = k_row_stride; a.v_row_stride = v_row_stride;
  a.n_b = (int)n_b;
  a.bps = (int)((n_b + n_splits - 1) / n_splits);
  a.words = (a.bps + 31) / 32;
  a.scale = scale > 0.f ? scale : (float)(1.0 / sqrt((double)dk));
  a.ln_lambda = ln_lambda(lambda);
  cudaError_t e = error_word(&a.err);
  if (e != cudaSuccess) return from_cuda(e);
  cudaStream_t s = (cudaStream_t)stream;

  if (dt == ATTN_BF16 && dk == 128 && dv == 128 && Bc == 128 && k_row_stride == 128 &&
      v_row_stride == 128 && (G == 1 || G == 2 || G == 4 || G == 8))
    return from_cuda(launch_decode_bf16(a, s));
  // Absorbed MLA: one latent head of 576 columns, values = its first 512 columns.
  if (dt == ATTN_BF16 && dk == 576 && dv == 512 && v == k && k_row_stride == 576 &&
      v_row_stride == 576 && Bc == 64 && Hkv == 1 && Hq == 128)
    return from_cuda(launch_mla_decode(a, s));
  return ATTN_EUNSUPPORTED;
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
    return (word & kErrTimeout) ? ATTN_ETIMEOUT : ATTN_ECUDA;
  }
  return ATTN_OK;
}

extern "C" const char *attn_skip_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_EINVAL: return "invalid argument";
    case ATTN_EUNSUPPORTED: return "unsupported combination (no kernel built for it)";
    case ATTN_ECUDA: return "CUDA error";
    case ATTN_ETIMEOUT: return "device-side bounded wait timed out";
  }
  return "unknown status";
}
