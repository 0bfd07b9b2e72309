// fp32 CUDA-core prefill with softmax-threshold block skipping.
//
// One CTA per (batch, query head, query tile), one thread per query row.  The
// loop is the online softmax of the BLASST page's section
// "铺垫：FlashAttention 的在线 softmax" (Eqs. 2-4) with the skip test of section
// "BLASST 的判定准则" (Eq. 5): per row a predicate, a warp vote, and an AND of
// the warp votes through shared memory (section "判定本身：几乎零成本的秘密").
// A skipped block costs neither its value load, nor its exponentials, nor its
// P.V accumulation.  This path serves fp32 inputs with head sizes 32/64.
#include <math.h>
#include "internal.h"

namespace attn_skip {
namespace {

template <int D, int BR, int BC>
__global__ void __launch_bounds__(BR) prefill_f32_kernel(const PrefillArgs a) {
  extern __shared__ __align__(16) float smem[];
  float *Ks = smem;               // [BC][D]
  float *Vs = Ks + BC * D;        // [BC][D]
  float *Ss = Vs + BC * D;        // [BR][BC + 1], one private row per thread
  __shared__ int warp_vote[BR / 32];
  __shared__ float warp_stat[BR / 32];

  const int unit = blockIdx.x;
  const int t = unit % a.n_t;
  const int h = (unit / a.n_t) % a.Hq;
  const int b = unit / (a.n_t * a.Hq);
  const int hk = h / (a.Hq / a.Hkv);
  const int r = threadIdx.x;
  const int row = t * BR + r;
  const bool valid = row < a.T;
  const int lane = r & 31, warp = r >> 5;

  const float *qg = (const float *)a.q + ((size_t)(b * a.Hq + h) * a.T) * D;
  const float *kg = (const float *)a.k + ((size_t)(b * a.Hkv + hk) * a.T) * D;
  const float *vg = (const float *)a.v + ((size_t)(b * a.Hkv + hk) * a.T) * D;

  float qr[D], acc[D];
#pragma unroll
  for (int i = 0; i < D; ++i) {
    qr[i] = valid ? qg[(size_t)row * D + i] : 0.f;
    acc[i] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int last_row = min(a.T, (t + 1) * BR) - 1;
  const int jmax = a.causal ? last_row / BC : a.n_b - 1;
  uint32_t *bits = a.bits ? a.bits + (size_t)unit * a.words : nullptr;
  uint32_t word = 0;
  int wcur = 0;  // next bitmap word to write
  float *Sr = Ss + r * (BC + 1);
  // Explicit block set (null = every block): blocks outside it are not traversed.
  const uint32_t *set = a.block_set ? a.block_set + (size_t)unit * a.words : nullptr;

  for (int j = 0; j <= jmax; ++j) {
    if (set && !((set[j >> 5] >> (j & 31)) & 1u)) {
      if (a.margin && r == 0) a.margin[(size_t)unit * a.n_b + j] = NAN;
      continue;
    }
    __syncthreads();  // the previous block's readers of Ks / Vs are done
    for (int i = r; i < BC * D / 4; i += BR) {
      const int c = (i * 4) / D, e = (i * 4) % D, key = j * BC + c;
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (key < a.T) kv = *reinterpret_cast<const float4 *>(kg + (size_t)key * D + e);
      *reinterpret_cast<float4 *>(Ks + c * D + e) = kv;
    }
    __syncthreads();

    // S_ij row, block row max (Eq. 2's rowmax) and the updated running max.
    float mt = -INFINITY;
    for (int c = 0; c < BC; ++c) {
      const int key = j * BC + c;
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < D; i += 4) {
        const float4 kv = *reinterpret_cast<const float4 *>(Ks + c * D + i);
        s = fmaf(qr[i], kv.x, s);
        s = fmaf(qr[i + 1], kv.y, s);
        s = fmaf(qr[i + 2], kv.z, s);
        s = fmaf(qr[i + 3], kv.w, s);
      }
      const bool vis = key < a.T && (!a.causal || key <= row);
      s = vis ? s * a.scale : -INFINITY;
      Sr[c] = s;
      mt = fmaxf(mt, s);
    }
    const float mnew = fmaxf(m, mt);
    // Eq. 5 against the updated max; a row with no visible key votes skip, and
    // rows past the end of the sequence do not take part (neutral vote).
    const float diff = (mt == -INFINITY) ? -INFINITY : mt - mnew;
    const bool vote = !valid || (diff < a.ln_lambda);
    const unsigned all = __all_sync(0xffffffffu, vote);
    if (lane == 0) warp_vote[warp] = (int)all;
    if (a.margin) {  // the block statistic: max over the tile's rows of rowmax - m_new
      float st = valid ? diff : -INFINITY;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) st = fmaxf(st, __shfl_xor_sync(0xffffffffu, st, o));
      if (lane == 0) warp_stat[warp] = st;
    }
    __syncthreads();
    bool skip = true;
#pragma unroll
    for (int w = 0; w < BR / 32; ++w) skip = skip && warp_vote[w];
    if (a.margin && r == 0) {
      float st = warp_stat[0];
#pragma unroll
      for (int w = 1; w < BR / 32; ++w) st = fmaxf(st, warp_stat[w]);
      a.margin[(size_t)unit * a.n_b + j] = st;
    }
    if (a.stats_only) skip = true;
    for (; wcur < (j >> 5); ++wcur) {  // earlier words are complete
      if (!a.stats_only && r == 0) bits[wcur] = word;
      word = 0;
    }
    if (skip) word |= 1u << (j & 31);

    if (!skip) {
      for (int i = r; i < BC * D / 4; i += BR) {
        const int c = (i * 4) / D, e = (i * 4) % D, key = j * BC + c;
        float4 vv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (key < a.T) vv = *reinterpret_cast<const float4 *>(vg + (size_t)key * D + e);
        *reinterpret_cast<float4 *>(Vs + c * D + e) = vv;
      }
      __syncthreads();
      // Eqs. 3-4: rescale the history to the new max and add this block.
      const float alpha = (m == -INFINITY) ? 0.f : expf(m - mnew);
      l *= alpha;
#pragma unroll
      for (int i = 0; i < D; ++i) acc[i] *= alpha;
      for (int c = 0; c < BC; ++c) {
        const float s = Sr[c];
        const float p = (s == -INFINITY) ? 0.f : expf(s - mnew);
        l += p;
#pragma unroll
        for (int i = 0; i < D; i += 4) {
          const float4 vv = *reinterpret_cast<const float4 *>(Vs + c * D + i);
          acc[i] = fmaf(p, vv.x, acc[i]);
          acc[i + 1] = fmaf(p, vv.y, acc[i + 1]);
          acc[i + 2] = fmaf(p, vv.z, acc[i + 2]);
          acc[i + 3] = fmaf(p, vv.w, acc[i + 3]);
        }
      }
    }
    m = mnew;  // unchanged on a skipped block (its row max is below m)
  }
  if (a.stats_only) {
    if (r == 0)
      for (int j = jmax + 1; j < a.n_b; ++j) a.margin[(size_t)unit * a.n_b + j] = NAN;
    return;
  }
  if (r == 0) {
    for (; wcur < a.words; ++wcur) {
      bits[wcur] = word;
      word = 0;
    }
  }
  if (a.margin && r == 0)
    for (int j = jmax + 1; j < a.n_b; ++j) a.margin[(size_t)unit * a.n_b + j] = NAN;
  if (valid) {
    float *og = (float *)a.o + ((size_t)(b * a.Hq + h) * a.T + row) * D;
    // (A row whose block set holds no visible key has no mass: O = 0, LSE = -inf.)
    const bool empty = !(l > 0.f);
    const float inv = empty ? 0.f : 1.f / l;
#pragma unroll
    for (int i = 0; i < D; ++i) og[i] = empty ? 0.f : acc[i] * inv;
    a.lse[(size_t)(b * a.Hq + h) * a.T + row] = empty ? -INFINITY : m + logf(l);
  }
}

template <int D, int BR, int BC>
cudaError_t launch(const PrefillArgs &a, cudaStream_t s) {
  const size_t smem = sizeof(float) * (2 * BC * D + BR * (BC + 1));
  cudaError_t e = cudaFuncSetAttribute(prefill_f32_kernel<D, BR, BC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long units = (long)a.B * a.Hq * a.n_t;
  prefill_f32_kernel<D, BR, BC><<<(unsigned)units, BR, smem, s>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const PrefillArgs &a, cudaStream_t s) {
  if (a.Br == 64 && a.Bc == 64) return launch<D, 64, 64>(a, s);
  if (a.Br == 64 && a.Bc == 128) return launch<D, 64, 128>(a, s);
  if (a.Br == 128 && a.Bc == 64) return launch<D, 128, 64>(a, s);
  return launch<D, 128, 128>(a, s);
}

}  // namespace

cudaError_t launch_prefill_f32(const PrefillArgs &a, cudaStream_t s) {
  return a.dk == 32 ? launch_d<32>(a, s) : launch_d<64>(a, s);
}

}  // namespace attn_skip
