// Merge of split-KV decode partials by log-sum-exp (FlashDecoding):
//   LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) * O_s,
// splits with LSE_s = -inf (no key) weighing zero.  One CTA per (sequence,
// query head); the per-split weights are computed once into shared memory.
#include <cuda_bf16.h>
#include <math.h>
#include "internal.h"

namespace attn_skip {
namespace {

constexpr int NT = 128;
constexpr int kMaxSplits = 1024;

__global__ void __launch_bounds__(NT) combine_kernel(const CombineArgs a) {
  __shared__ float w[kMaxSplits];
  __shared__ float s_lse;
  const int row = blockIdx.x;  // b * Hq + h
  const float *ls = a.lse_part + (size_t)row * a.n_splits;
  if (threadIdx.x < 32) {
    float M = -INFINITY;
    for (int s = threadIdx.x; s < a.n_splits; s += 32) M = fmaxf(M, ls[s]);
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float Z = 0.f;
    if (M != -INFINITY)
      for (int s = threadIdx.x; s < a.n_splits; s += 32) Z += (ls[s] == -INFINITY) ? 0.f : expf(ls[s] - M);
    for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
    const float lse = (M == -INFINITY) ? -INFINITY : M + logf(Z);
    for (int s = threadIdx.x; s < a.n_splits; s += 32)
      w[s] = (ls[s] == -INFINITY) ? 0.f : expf(ls[s] - lse);
    if (threadIdx.x == 0) s_lse = lse;
  }
  __syncthreads();
  const float *op = a.o_part + (size_t)row * a.n_splits * a.dv;
  for (int e = threadIdx.x; e < a.dv; e += NT) {
    float o = 0.f;
    for (int s = 0; s < a.n_splits; ++s) o = fmaf(w[s], op[(size_t)s * a.dv + e], o);
    if (a.out_bf16)
      ((__nv_bfloat16 *)a.o)[(size_t)row * a.dv + e] = __float2bfloat16_rn(o);
    else
      ((float *)a.o)[(size_t)row * a.dv + e] = o;
  }
  if (threadIdx.x == 0) a.lse[row] = s_lse;
}

}  // namespace

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s) {
  if (a.n_splits > kMaxSplits) return cudaErrorInvalidValue;
  combine_kernel<<<(unsigned)((long)a.B * a.Hq), NT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace attn_skip
