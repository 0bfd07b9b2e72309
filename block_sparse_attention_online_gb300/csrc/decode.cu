// Split-KV decode with softmax-threshold block skipping (bf16 cache, d = 128).
//
// One CTA per (sequence, KV head, split).  The G query heads sharing the KV
// head are packed into the CTA, so each key byte is read once for all of them.
// Following the BLASST page's section "Decode 内核：砍带宽" (batched load
// scheduling), the CTA works on batches of NB consecutive KV blocks:
//   1. Q.K^T for the whole batch with 16-byte vector loads of K (always done --
//      it is the only source of the block maxima), scores to shared memory;
//   2. the skip decisions of the batch, taken in block order against the
//      running max (Eq. 5; a block is skipped only if all G heads vote skip);
//   3. exponentials, then value loads and P.V only for the kept blocks.
// The value loads of a batch are issued together, so skipping removes HBM
// traffic instead of leaving bubbles in a load pipeline.
#include <cuda_bf16.h>
#include <math.h>
#include "internal.h"

namespace attn_skip {
namespace {

constexpr int D = 128;         // head size (keys and values)
constexpr int BC = 128;        // keys per block
constexpr int NB = 4;          // blocks per decision batch
constexpr int NT = 256;        // threads per CTA
constexpr int NW = NT / 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int G>
__global__ void __launch_bounds__(NT, 2) decode_bf16_kernel(const DecodeArgs a) {
  // Scores (log2 domain, then P) during the loop; the cross-warp reduction of O
  // in the epilogue reuses the same storage.
  __shared__ __align__(16) float smem_f[G * (NW * D > NB * BC ? NW * D : NB * BC)];
  float (*S)[NB * BC] = reinterpret_cast<float (*)[NB * BC]>(smem_f);
  float (*red)[G][D] = reinterpret_cast<float (*)[G][D]>(smem_f);
  __shared__ float bmax[NB][G];
  __shared__ float lred[NW][G];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int unit = blockIdx.x;
  const int sp = unit % a.n_splits;
  const int hk = (unit / a.n_splits) % a.Hkv;
  const int b = unit / (a.n_splits * a.Hkv);
  const int j0 = (int)((long)sp * a.n_b / a.n_splits);
  const int j1 = (int)((long)(sp + 1) * a.n_b / a.n_splits);
  const float s2 = a.scale * kLog2e;          // scores kept in log2 units
  const float c2 = a.ln_lambda * kLog2e;      // ln(lambda) in log2 units (-inf if lambda = 0)

  const __nv_bfloat16 *kg =
      (const __nv_bfloat16 *)a.k + ((size_t)(b * a.Hkv + hk) * a.L) * a.k_row_stride;
  const __nv_bfloat16 *vg =
      (const __nv_bfloat16 *)a.v + ((size_t)(b * a.Hkv + hk) * a.L) * a.v_row_stride;
  uint32_t *bits = a.bits + (size_t)unit * a.words;

  // QK layout: 8 lanes per key, lane p holds dims [8p, 8p+8) and [64+8p, 64+8p+8).
  const int kq = lane >> 3, p = lane & 7;
  float qf[G][16];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const __nv_bfloat16 *qh = (const __nv_bfloat16 *)a.q + (size_t)(b * a.Hq + hk * G + g) * D;
    const uint4 lo = *reinterpret_cast<const uint4 *>(qh + 8 * p);
    const uint4 hi = *reinterpret_cast<const uint4 *>(qh + 64 + 8 * p);
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      qf[g][2 * i] = bf_lo(w[i]);
      qf[g][2 * i + 1] = bf_hi(w[i]);
    }
  }

  // PV layout: lane chunk c = tid % 16 owns value dims [8c, 8c+8); key slot ks = tid / 16.
  const int c = tid & 15, ks = tid >> 4;
  float acc[G][8];
  float lsum[G];
  float m[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    lsum[g] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
  }
  uint32_t word = 0;

  for (int jb = j0; jb < j1; jb += NB) {
    const int nblk = min(NB, j1 - jb);
    const int key0 = jb * BC;
    // ---- 1. scores of the batch ------------------------------------------
    constexpr int kSteps = NB * BC / (4 * NW);  // warp steps of 4 keys
#pragma unroll 1
    for (int i0 = 0; i0 < kSteps; i0 += 4) {
      uint4 kr[4][2];
      int kl[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        kl[u] = ((i0 + u) * NW + warp) * 4 + kq;
        const int key = key0 + kl[u];
        if (kl[u] < nblk * BC && key < a.L) {
          const __nv_bfloat16 *kr_p = kg + (size_t)key * a.k_row_stride;
          kr[u][0] = ldg_stream(kr_p + 8 * p);
          kr[u][1] = ldg_stream(kr_p + 64 + 8 * p);
        } else {
          kr[u][0] = make_uint4(0, 0, 0, 0);
          kr[u][1] = make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float dot[G];
#pragma unroll
        for (int g = 0; g < G; ++g) dot[g] = 0.f;
        const uint32_t w[8] = {kr[u][0].x, kr[u][0].y, kr[u][0].z, kr[u][0].w,
                               kr[u][1].x, kr[u][1].y, kr[u][1].z, kr[u][1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float x0 = bf_lo(w[i]), x1 = bf_hi(w[i]);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            dot[g] = fmaf(qf[g][2 * i], x0, dot[g]);
            dot[g] = fmaf(qf[g][2 * i + 1], x1, dot[g]);
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          dot[g] += __shfl_xor_sync(0xffffffffu, dot[g], 1);
          dot[g] += __shfl_xor_sync(0xffffffffu, dot[g], 2);
          dot[g] += __shfl_xor_sync(0xffffffffu, dot[g], 4);
        }
        const int key = key0 + kl[u];
        const bool vis = kl[u] < nblk * BC && key < a.L;
#pragma unroll
        for (int g = 0; g < G; ++g)
          if (p == (g & 7) && kl[u] < NB * BC) S[g][kl[u]] = vis ? dot[g] * s2 : -INFINITY;
      }
    }
    __syncthreads();

    // ---- 2. block maxima, then the decisions in block order --------------
    if (warp < nblk) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float x = -INFINITY;
#pragma unroll
        for (int i = 0; i < BC / 32; ++i) x = fmaxf(x, S[g][warp * BC + lane + 32 * i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
        if (lane == 0) bmax[warp][g] = x;
      }
    }
    __syncthreads();
    float m_prev[G];
#pragma unroll
    for (int g = 0; g < G; ++g) m_prev[g] = m[g];
    unsigned keep = 0;
    for (int jj = 0; jj < nblk; ++jj) {
      bool all_skip = true;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float mt = bmax[jj][g];
        const float mn = fmaxf(m[g], mt);
        const float diff = (mt == -INFINITY) ? -INFINITY : mt - mn;
        all_skip = all_skip && (diff < c2);
        m[g] = mn;
      }
      const int pos = jb + jj - j0;
      if (all_skip) word |= 1u << (pos & 31);
      else keep |= 1u << jj;
      if ((pos & 31) == 31 || jb + jj == j1 - 1) {
        if (tid == 0) bits[pos >> 5] = word;
        word = 0;
      }
    }
    if (keep == 0) {  // nothing kept: the running max did not move
      __syncthreads();
      continue;
    }

    // ---- 3. exponentials of the kept blocks (reference = max after the batch)
    float alpha[G];
#pragma unroll
    for (int g = 0; g < G; ++g) alpha[g] = (m_prev[g] == -INFINITY) ? 0.f : fast_exp2(m_prev[g] - m[g]);
    for (int idx = tid; idx < G * NB * BC; idx += NT) {
      const int g = idx / (NB * BC), kk = idx % (NB * BC);
      if ((keep >> (kk / BC)) & 1u) {
        const float sv = S[g][kk];
        S[g][kk] = (sv == -INFINITY) ? 0.f : fast_exp2(sv - m[g]);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      lsum[g] *= alpha[g];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[g][e] *= alpha[g];
    }
    __syncthreads();

    // ---- 4. value loads and P.V, kept blocks only ------------------------
    for (int jj = 0; jj < nblk; ++jj) {
      if (!((keep >> jj) & 1u)) continue;
      uint4 vr[BC / 16];
#pragma unroll
      for (int i = 0; i < BC / 16; ++i) {
        const int key = (jb + jj) * BC + ks + 16 * i;
        vr[i] = key < a.L ? ldg_stream(vg + (size_t)key * a.v_row_stride + 8 * c)
                          : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < BC / 16; ++i) {
        const int kk = jj * BC + ks + 16 * i;
        const uint32_t w[4] = {vr[i].x, vr[i].y, vr[i].z, vr[i].w};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pg = S[g][kk];
          lsum[g] += pg;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[g][2 * e] = fmaf(pg, bf_lo(w[e]), acc[g][2 * e]);
            acc[g][2 * e + 1] = fmaf(pg, bf_hi(w[e]), acc[g][2 * e + 1]);
          }
        }
      }
    }
    __syncthreads();  // S is overwritten by the next batch
  }

  // ---- epilogue: reduce over the 16 key slots ------------------------------
  __syncthreads();  // S is dead; its storage becomes the reduction buffer
#pragma unroll
  for (int g = 0; g < G; ++g) {
    lsum[g] += __shfl_xor_sync(0xffffffffu, lsum[g], 16);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], 16);
      if (lane < 16) red[warp][g][8 * c + e] = acc[g][e];
    }
    if (lane == 0) lred[warp][g] = lsum[g];
  }
  if (j1 > j0 && tid == 0) {
    const int last = j1 - 1 - j0;
    for (int w = (last >> 5) + 1; w < a.words; ++w) bits[w] = 0u;
  } else if (j1 == j0) {
    for (int w = tid; w < a.words; w += NT) bits[w] = 0u;
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += NT) {
    const int g = idx / D, e = idx % D;
    float o = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      o += red[w][g][e];
      l += lred[w][g];
    }
    const size_t row = (size_t)(b * a.Hq + hk * G + g) * a.n_splits + sp;
    if (j1 == j0) {
      a.o_part[row * D + e] = 0.f;
      if (e == 0) a.lse_part[row] = -INFINITY;
    } else {
      a.o_part[row * D + e] = o / l;
      if (e == 0) a.lse_part[row] = m[g] * kLn2 + logf(l);
    }
  }
}

template <int G>
cudaError_t launch(const DecodeArgs &a, cudaStream_t s) {
  const long units = (long)a.B * a.Hkv * a.n_splits;
  decode_bf16_kernel<G><<<(unsigned)units, NT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_bf16(const DecodeArgs &a, cudaStream_t s) {
  switch (a.Hq / a.Hkv) {
    case 1: return launch<1>(a, s);
    case 2: return launch<2>(a, s);
    case 4: return launch<4>(a, s);
    default: return launch<8>(a, s);
  }
}

}  // namespace attn_skip
