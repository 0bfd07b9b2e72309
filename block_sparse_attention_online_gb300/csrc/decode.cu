// Split-KV decode with softmax-threshold block skipping (bf16 cache, d = 128).
//
// One CTA per (sequence, KV head, split).  The G query heads sharing the KV
// head are packed into the CTA, so each key byte is read once for all of them.
// The BLASST page's decode kernel (section "Decode 内核：砍带宽") skips the value
// load of a skipped block and avoids a decide-then-load bubble by computing
// the scores of a batch of blocks before issuing the value loads of the
// survivors.  Here that batch is a sliding window:
//   * a K-producer warp streams whole 32 KB key blocks into a 4-stage shared
//     memory ring with bulk copies (every block: Q.K^T is never skipped);
//   * eight consumer warps compute the scores of block j from shared memory
//     (16-byte vector reads, fp32 FMA), reduce the block maxima and take the
//     decision of block j in order (Eq. 5 against the running max; all G
//     heads must vote skip);
//   * a V-producer warp loads the value block of each kept block as soon as
//     its decision is published;
//   * the consumers exponentiate block j-2 and accumulate P.V of block j-3,
//     so a kept block's value load has the score work of two blocks to land.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"
#include "tc_common.cuh"

namespace attn_skip {
namespace {

using namespace tc;

constexpr int D = 128;         // head size (keys and values)
constexpr int BC = 128;        // keys per block
constexpr int NKS = 4;         // key stages
constexpr int NVS = 2;         // value stages
constexpr int LAG = 2;         // exponentials of block j - LAG, P.V of block j - LAG - 1
constexpr int R = LAG + 3;     // score ring (see the reuse argument at the loop)
constexpr int NDEC = 8;        // decision ring
constexpr int NCW = 8;         // consumer warps
constexpr int NT = (NCW + 2) * 32;
constexpr int WARP_K = NCW, WARP_V = NCW + 1;
constexpr uint32_t BLK_BYTES = BC * D * 2;  // 32 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int G>
struct DecShared {
  uint64_t k_full[NKS], k_empty[NKS];
  uint64_t v_full[NVS], v_empty[NVS];
  uint64_t dec_full[NDEC], dec_empty[NDEC];
  uint64_t bar[2], fin;
  int dec[NDEC];
  float wmax[2][NCW][G];
  float mrow[R][G];               // running max after block (log2 units), slot block % R
  alignas(16) float S[R][BC][G];  // scores (log2 units), then P in place
  int abort;
};

template <int G>
constexpr uint32_t smem_bytes() {
  return (NKS + NVS) * BLK_BYTES + (uint32_t)sizeof(DecShared<G>);
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}

template <int G>
__global__ void __launch_bounds__(NT, 1) decode_bf16_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  DecShared<G> &sh = *reinterpret_cast<DecShared<G> *>(smem + (NKS + NVS) * BLK_BYTES);
  const uint32_t kring = smem_u32(smem), vring = kring + NKS * BLK_BYTES;
  volatile int *abort = &sh.abort;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int unit = blockIdx.x;
  const int sp = unit % a.n_splits;
  const int hk = (unit / a.n_splits) % a.Hkv;
  const int b = unit / (a.n_splits * a.Hkv);
  const int j0 = (int)((long)sp * a.n_b / a.n_splits);
  const int j1 = (int)((long)(sp + 1) * a.n_b / a.n_splits);
  const int nb = j1 - j0;
  const float sl2 = a.scale * kLog2e;      // raw score -> log2 units
  const float c2 = a.ln_lambda * kLog2e;   // ln(lambda) in log2 units (-inf if lambda = 0)
  const __nv_bfloat16 *kg = (const __nv_bfloat16 *)a.k + ((size_t)(b * a.Hkv + hk) * a.L) * D;
  const __nv_bfloat16 *vg = (const __nv_bfloat16 *)a.v + ((size_t)(b * a.Hkv + hk) * a.L) * D;
  uint32_t *bits = a.bits + (size_t)unit * a.words;

  if (nb == 0) {  // empty split: no key, zero weight in the merge
    for (int idx = tid; idx < G * D; idx += NT) {
      const size_t row = (size_t)(b * a.Hq + hk * G + idx / D) * a.n_splits + sp;
      a.o_part[row * D + idx % D] = 0.f;
      if (idx % D == 0) a.lse_part[row] = -INFINITY;
    }
    for (int w = tid; w < a.words; w += NT) bits[w] = 0u;
    return;
  }

  if (tid == 0) {
    for (int i = 0; i < NKS; ++i) {
      mbar_init(smem_u32(&sh.k_full[i]), 1);
      mbar_init(smem_u32(&sh.k_empty[i]), NCW);
    }
    for (int i = 0; i < NVS; ++i) {
      mbar_init(smem_u32(&sh.v_full[i]), 1);
      mbar_init(smem_u32(&sh.v_empty[i]), NCW);
    }
    for (int i = 0; i < NDEC; ++i) {
      mbar_init(smem_u32(&sh.dec_full[i]), 1);
      mbar_init(smem_u32(&sh.dec_empty[i]), 1);
    }
    mbar_init(smem_u32(&sh.bar[0]), NCW);
    mbar_init(smem_u32(&sh.bar[1]), NCW);
    mbar_init(smem_u32(&sh.fin), NCW);
    sh.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  auto block_keys = [&](int j) { return min(BC, a.L - (j0 + j) * BC); };

  if (warp == WARP_K) {
    // ---------------------------------------------------------- K producer --
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();  // the cache is streamed once
      int issued = 0;
      for (int j = 0; j < nb && !*abort; ++j) {
        const int s = j % NKS;
        if (j >= NKS &&
            !mbar_wait(smem_u32(&sh.k_empty[s]), ((j / NKS) - 1) & 1, abort, a.err, kErrTimeout))
          break;
        const uint32_t bytes = (uint32_t)block_keys(j) * D * 2;
        mbar_expect_tx(smem_u32(&sh.k_full[s]), bytes);
        bulk_load(kring + s * BLK_BYTES, kg + (size_t)(j0 + j) * BC * D, bytes,
                  smem_u32(&sh.k_full[s]), pol);
        ++issued;
      }
      for (int s = 0; s < NKS && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / NKS) * NKS;
        mbar_wait_drain(smem_u32(&sh.k_full[s]), (last / NKS) & 1);
      }
    }
    return;
  }
  if (warp == WARP_V) {
    // ---------------------------------------------------------- V producer --
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int vi = 0;
      for (int j = 0; j < nb && !*abort; ++j) {
        if (!mbar_wait(smem_u32(&sh.dec_full[j % NDEC]), (j / NDEC) & 1, abort, a.err,
                       kErrTimeout))
          break;
        const int keep = sh.dec[j % NDEC];
        mbar_arrive(smem_u32(&sh.dec_empty[j % NDEC]));
        if (!keep) continue;
        const int s = vi % NVS;
        if (vi >= NVS &&
            !mbar_wait(smem_u32(&sh.v_empty[s]), ((vi / NVS) - 1) & 1, abort, a.err, kErrTimeout))
          break;
        const uint32_t bytes = (uint32_t)block_keys(j) * D * 2;
        mbar_expect_tx(smem_u32(&sh.v_full[s]), bytes);
        bulk_load(vring + s * BLK_BYTES, vg + (size_t)(j0 + j) * BC * D, bytes,
                  smem_u32(&sh.v_full[s]), pol);
        ++vi;
      }
      for (int s = 0; s < NVS && s < vi; ++s) {
        const int last = s + ((vi - 1 - s) / NVS) * NVS;
        mbar_wait_drain(smem_u32(&sh.v_full[s]), (last / NVS) & 1);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers --
  // QK layout: 8 lanes per key, lane p holds dims [8p, 8p+8) and [64+8p, 64+8p+8);
  // a warp step covers 4 keys.
  const int kq = lane >> 3, p = lane & 7;
  uint64_t qp[G][8];  // packed fp32 pairs of the thread's 16 query dims, per head
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const __nv_bfloat16 *qh = (const __nv_bfloat16 *)a.q + (size_t)(b * a.Hq + hk * G + g) * D;
    const uint4 lo = *reinterpret_cast<const uint4 *>(qh + 8 * p);
    const uint4 hi = *reinterpret_cast<const uint4 *>(qh + 64 + 8 * p);
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) qp[g][i] = f2(bf_lo(w[i]), bf_hi(w[i]));
  }
  // PV layout: chunk c = tid % 16 owns value dims [8c, 8c+8); key slot ks = tid / 16.
  const int c = tid & 15, ks = tid >> 4;
  uint64_t acc2[G][4];  // packed output pairs (dims 8c+2e, 8c+2e+1)
  float lsum[G], ref[G], m[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    ref[g] = -INFINITY;
    lsum[g] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) acc2[g][e] = f2(0.f, 0.f);
  }
  uint32_t hist = 0;  // bit d: block (j - d) kept
  uint32_t word = 0;
  int vi = 0;
  bool ok = true;

  // Ring reuse: the score slot of block j (written before the barrier of
  // iteration j) last served the P.V of block j - R = j - LAG - 3 in iteration
  // j - 2, which every warp finished before the barrier of iteration j - 1.
  for (int j = 0; ok && j < nb + LAG + 1; ++j) {
    const int pb = j & 1;
    if (j < nb) {
      // ---- scores of block j ---------------------------------------------
      const int s = j % NKS, rs = j % R;
      if (!mbar_wait_warp(smem_u32(&sh.k_full[s]), (j / NKS) & 1, abort, a.err, kErrTimeout)) {
        ok = false;
        break;
      }
      const int keys = block_keys(j);
      const uint32_t kt = kring + s * BLK_BYTES;
      constexpr int NSTEP = BC / (4 * NCW);  // warp steps of 4 keys (= 4)
      float val[NSTEP * G];                    // partial dots, index step * G + g
#pragma unroll
      for (int step = 0; step < NSTEP; ++step) {
        const int kl = (step * NCW + warp) * 4 + kq;
        uint4 k0 = make_uint4(0, 0, 0, 0), k1 = make_uint4(0, 0, 0, 0);
        if (kl < keys) {
          k0 = lds128(kt + kl * (D * 2) + p * 16);
          k1 = lds128(kt + kl * (D * 2) + 128 + p * 16);
        }
        const uint32_t w[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
        uint64_t d2[G];
#pragma unroll
        for (int g = 0; g < G; ++g) d2[g] = f2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint64_t x = f2(bf_lo(w[i]), bf_hi(w[i]));
#pragma unroll
          for (int g = 0; g < G; ++g) d2[g] = f2_fma(qp[g][i], x, d2[g]);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float lo, hi;
          f2_split(d2[g], lo, hi);
          val[step * G + g] = lo + hi;
        }
      }
      // Sum over the 8 lanes of a key group.  Transposed butterfly: each level
      // exchanges half of the values, so after three levels lane p holds the
      // full dots v = p*G/2 + r (r < G/2) of step p/2, heads (p%2)*G/2 + r.
      float bm[G];
#pragma unroll
      for (int g = 0; g < G; ++g) bm[g] = -INFINITY;
      if constexpr (G >= 2) {
        float v1[2 * G], v2[G], v3[G / 2];
        const bool u1 = lane & 4, u2 = lane & 2, u3 = lane & 1;
#pragma unroll
        for (int i = 0; i < 2 * G; ++i) {
          const float x = val[i], y = val[i + 2 * G];
          v1[i] = (u1 ? y : x) + __shfl_xor_sync(0xffffffffu, u1 ? x : y, 4);
        }
#pragma unroll
        for (int i = 0; i < G; ++i) {
          const float x = v1[i], y = v1[i + G];
          v2[i] = (u2 ? y : x) + __shfl_xor_sync(0xffffffffu, u2 ? x : y, 2);
        }
#pragma unroll
        for (int i = 0; i < G / 2; ++i) {
          const float x = v2[i], y = v2[i + G / 2];
          v3[i] = (u3 ? y : x) + __shfl_xor_sync(0xffffffffu, u3 ? x : y, 1);
        }
        const int step = p >> 1, g0 = (p & 1) * (G / 2);
        const int kl = (step * NCW + warp) * 4 + kq;
        float hm[G / 2];
#pragma unroll
        for (int r = 0; r < G / 2; ++r) {
          const float sv = kl < keys ? v3[r] * sl2 : -INFINITY;
          sh.S[rs][kl][g0 + r] = sv;
          hm[r] = sv;
        }
        // block max per head: lanes with the same p%2 hold the same heads
#pragma unroll
        for (int r = 0; r < G / 2; ++r) {
          hm[r] = fmaxf(hm[r], __shfl_xor_sync(0xffffffffu, hm[r], 2));
          hm[r] = fmaxf(hm[r], __shfl_xor_sync(0xffffffffu, hm[r], 4));
          hm[r] = fmaxf(hm[r], __shfl_xor_sync(0xffffffffu, hm[r], 8));
          hm[r] = fmaxf(hm[r], __shfl_xor_sync(0xffffffffu, hm[r], 16));
        }
        if (lane < 2) {
#pragma unroll
          for (int r = 0; r < G / 2; ++r) sh.wmax[pb][warp][lane * (G / 2) + r] = hm[r];
        }
      } else {  // one head: plain butterfly over the 8 lanes
#pragma unroll
        for (int step = 0; step < NSTEP; ++step) {
          float x = val[step];
          x += __shfl_xor_sync(0xffffffffu, x, 1);
          x += __shfl_xor_sync(0xffffffffu, x, 2);
          x += __shfl_xor_sync(0xffffffffu, x, 4);
          const int kl = (step * NCW + warp) * 4 + kq;
          const float sv = kl < keys ? x * sl2 : -INFINITY;
          if (p == 0) sh.S[rs][kl][0] = sv;
          bm[0] = fmaxf(bm[0], sv);
        }
        bm[0] = fmaxf(bm[0], __shfl_xor_sync(0xffffffffu, bm[0], 8));
        bm[0] = fmaxf(bm[0], __shfl_xor_sync(0xffffffffu, bm[0], 16));
        if (lane == 0) sh.wmax[pb][warp][0] = bm[0];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.k_empty[s]));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh.bar[pb]));
    if (!mbar_wait_warp(smem_u32(&sh.bar[pb]), (j >> 1) & 1, abort, a.err, kErrTimeout)) {
      ok = false;
      break;
    }

    // ---- decision of block j (every thread takes it identically) -----------
    if (j < nb) {
      bool all_skip = true;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float mt = sh.wmax[pb][0][g];
#pragma unroll
        for (int w = 1; w < NCW; ++w) mt = fmaxf(mt, sh.wmax[pb][w][g]);
        const float mn = fmaxf(m[g], mt);
        const float diff = (mt == -INFINITY) ? -INFINITY : mt - mn;
        all_skip = all_skip && (diff < c2);
        m[g] = mn;
      }
      hist = (hist << 1) | (all_skip ? 0u : 1u);
      if (tid == 0) {
        // On a timeout the abort flag is raised and every later wait fails.
        if (j < NDEC || mbar_wait(smem_u32(&sh.dec_empty[j % NDEC]), ((j / NDEC) - 1) & 1, abort,
                                  a.err, kErrTimeout)) {
          sh.dec[j % NDEC] = all_skip ? 0 : 1;
          mbar_arrive(smem_u32(&sh.dec_full[j % NDEC]));
        }
#pragma unroll
        for (int g = 0; g < G; ++g) sh.mrow[j % R][g] = m[g];
        if (all_skip) word |= 1u << (j & 31);
        if ((j & 31) == 31 || j == nb - 1) {
          bits[j >> 5] = word;
          word = 0;
        }
      }
    } else {
      hist <<= 1;  // past the end: nothing to keep
    }

    // ---- P.V of block j - LAG - 1 (its P was written in the last iteration) -
    const int i1 = j - LAG - 1;
    if (i1 >= 0 && ((hist >> (LAG + 1)) & 1u)) {
      const int vs = vi % NVS;
      if (!mbar_wait_warp(smem_u32(&sh.v_full[vs]), (vi / NVS) & 1, abort, a.err, kErrTimeout)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float nr = sh.mrow[i1 % R][g];
        const float alpha = (ref[g] == -INFINITY) ? 0.f : ex2(ref[g] - nr);
        ref[g] = nr;
        lsum[g] *= alpha;
        const uint64_t a2 = f2(alpha, alpha);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc2[g][e] = f2_fma(acc2[g][e], a2, f2(0.f, 0.f));
      }
      const int keys = block_keys(i1);
      const uint32_t vt = vring + vs * BLK_BYTES;
#pragma unroll 4
      for (int kk = ks; kk < keys; kk += 16) {
        const uint4 v = lds128(vt + kk * (D * 2) + c * 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float pg[G];
        if constexpr (G == 4) {
          const float4 p4 = *reinterpret_cast<const float4 *>(&sh.S[i1 % R][kk][0]);
          pg[0] = p4.x;
          pg[1] = p4.y;
          pg[2] = p4.z;
          pg[3] = p4.w;
        } else {
#pragma unroll
          for (int g = 0; g < G; ++g) pg[g] = sh.S[i1 % R][kk][g];
        }
        uint64_t vx[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) vx[e] = f2(bf_lo(w[e]), bf_hi(w[e]));
#pragma unroll
        for (int g = 0; g < G; ++g) {
          lsum[g] += pg[g];
          const uint64_t pp = f2(pg[g], pg[g]);
#pragma unroll
          for (int e = 0; e < 4; ++e) acc2[g][e] = f2_fma(pp, vx[e], acc2[g][e]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.v_empty[vs]));
      ++vi;
    }

    // ---- exponentials of block j - LAG (in place; read after the next barrier)
    const int i2 = j - LAG;
    if (i2 >= 0 && ((hist >> LAG) & 1u)) {
      float nr[G];
#pragma unroll
      for (int g = 0; g < G; ++g) nr[g] = sh.mrow[i2 % R][g];
      float *Sv = &sh.S[i2 % R][0][0];
      for (int idx = tid; idx < BC * G; idx += NCW * 32) {
        const float sv = Sv[idx];
        Sv[idx] = (sv == -INFINITY) ? 0.f : ex2(sv - nr[idx % G]);
      }
    }
  }

  // ---- epilogue: reduce the 16 key slots ------------------------------------
  if (tid == 0) {
    for (int w = ((nb - 1) >> 5) + 1; w < a.words; ++w) bits[w] = 0u;
  }
  // Every key block was consumed, so the key ring is free for the reduction.
  float(*red)[G][D] = reinterpret_cast<float(*)[G][D]>(smem);
  float(*lred)[G] = reinterpret_cast<float(*)[G]>(smem + NCW * G * D * sizeof(float));
#pragma unroll
  for (int g = 0; g < G; ++g) {
    lsum[g] += __shfl_xor_sync(0xffffffffu, lsum[g], 16);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float lo, hi;
      f2_split(acc2[g][e], lo, hi);
      lo += __shfl_xor_sync(0xffffffffu, lo, 16);
      hi += __shfl_xor_sync(0xffffffffu, hi, 16);
      if (lane < 16) {
        red[warp][g][8 * c + 2 * e] = lo;
        red[warp][g][8 * c + 2 * e + 1] = hi;
      }
    }
    if (lane == 0) lred[warp][g] = lsum[g];
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&sh.fin));
  if (!mbar_wait_warp(smem_u32(&sh.fin), 0, abort, a.err, kErrTimeout) || !ok) return;
  for (int idx = tid; idx < G * D; idx += NCW * 32) {
    const int g = idx / D, e = idx % D;
    float o = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) {
      o += red[w][g][e];
      l += lred[w][g];
    }
    const size_t row = (size_t)(b * a.Hq + hk * G + g) * a.n_splits + sp;
    a.o_part[row * D + e] = o / l;
    if (e == 0) a.lse_part[row] = ref[g] * kLn2 + logf(l);
  }
}

template <int G>
cudaError_t launch(const DecodeArgs &a, cudaStream_t s) {
  constexpr uint32_t bytes = smem_bytes<G>();
  static_assert(bytes <= 227 * 1024, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(decode_bf16_kernel<G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  const long units = (long)a.B * a.Hkv * a.n_splits;
  decode_bf16_kernel<G><<<(unsigned)units, NT, bytes, s>>>(a);
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
