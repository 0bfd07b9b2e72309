// Sampled decode output (SANTA estimator, S²ANTA-prop schedule) for a bf16
// GQA cache with d = 128.
//
// Method: the web page "Stochastic Sparse Attention for Memory-Bound
// Inference" (SANTA), section "关键设计": the attention weights of a decode
// query form a categorical distribution over its keys, and the mean of the
// value rows at S inverse-CDF samples is an unbiased estimate of the output;
// stratified (one draw per equal-mass stratum) or systematic (one offset for
// a lattice of S thresholds) samples lower its variance.  The S²ANTA-prop
// item gives the GPU schedule: a first pass writes every key's score and one
// (max, sum) pair per key tile; a light global step turns the tile sums into
// the tile boundaries of the CDF and hands each tile its share of the
// samples; a second pass places each sample inside its tile and gathers only
// the sampled value rows, so a tile that gets no sample costs no value read.
//
// Pass 1 (santa_scores_kernel), one CTA per (sequence, KV head, key tile):
// the tensor core computes S^T = K_j Q^T with the block's 128 keys as the
// MMA rows (M = 128) and the G query heads of the KV head, padded to 16, as
// the columns (N = 16).  Each of the four score warps then holds one key per
// thread with the G heads' scores in G registers: the score stores are
// coalesced (32 consecutive keys per warp instruction) and the running
// (max, sum) of the tile is kept per thread and reduced once at the end.
//   warps 0-3  scores: TMEM -> registers, log2-scaled scores to the stash,
//              per-thread online (max, sum);
//   warp 4     TMA producer of K_j (6-stage ring of 32 KB tiles);
//   warp 5     S^T issuer (four 16-column TMEM buffers; allocates TMEM).
// Pass 2 (santa_sample_kernel), one CTA of 8 warps per (sequence, query head):
// tile weights and their prefix (the CDF at the tile boundaries), the tile of
// every threshold by bisection, then per tile that holds samples a warp
// builds the tile's running sum in shared memory and places its samples by
// bisection, and last the sampled value rows are gathered and averaged.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"
#include "tc_common.cuh"

namespace attn_skip {
namespace {

using namespace tc;

constexpr int D = 128;   // head size (keys and values)
constexpr int BC = 128;  // keys per block (MMA rows)
constexpr int NQ = 16;   // MMA columns: query heads of a KV head, padded
constexpr int NK = 6;    // key stages
constexpr int NS = 4;    // TMEM score buffers (16 columns each)
constexpr int NT1 = 6 * 32;
constexpr int WARP_K = 4, WARP_MMA = 5;  // warps 0-3: scores
constexpr uint32_t TILE_BYTES = BC * D * 2;      // 32 KB: 128 keys x 128 bf16
constexpr uint32_t HALF_BYTES = TILE_BYTES / 2;  // one 64-column swizzled box
constexpr uint32_t Q_BOX = NQ * 128;             // 16 rows x 128 bytes
constexpr uint32_t SMEM_K = 0;
constexpr uint32_t SMEM_Q = SMEM_K + NK * TILE_BYTES;
constexpr uint32_t SMEM_TILES = SMEM_Q + 2 * Q_BOX;
constexpr uint32_t TMEM_COLS = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t IDESC = idesc_bf16_f32(BC, NQ, 0);  // A = K_j, B = Q: both K-major

struct Shared1 {
  uint64_t k_full[NK], k_empty[NK];
  uint64_t s_full[NS], s_free[NS];
  float red_m[4][8], red_z[4][8];
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t SMEM1 = SMEM_TILES + ((sizeof(Shared1) + 127) / 128) * 128;
static_assert(SMEM1 <= 227 * 1024, "shared memory budget");

// K-major operand of 128-byte-swizzled boxes of 64 columns: k-step kk (16
// columns) is box kk/4 at 32-byte step kk%4; 8-row groups are 1024 bytes apart.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile) {
  return smem_desc_sw128(tile, 16u, 1024u);
}
__device__ __forceinline__ constexpr uint64_t kmajor_step(int kk, uint32_t box_bytes) {
  return (uint64_t)(((uint32_t)(kk >> 2) * box_bytes + (uint32_t)(kk & 3) * 32u) >> 4);
}

// 32 lanes x 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr)
      : "memory");
}

// Merge of two (max, sum-of-exp2-relative-to-max) pairs.
__device__ __forceinline__ void lse2_merge(float &m, float &z, float mo, float zo) {
  const float M = fmaxf(m, mo);
  z = (M == -INFINITY) ? 0.f : z * ex2(m - M) + zo * ex2(mo - M);
  m = M;
}

template <int G>
__global__ void __launch_bounds__(NT1, 1)
    santa_scores_kernel(const __grid_constant__ CUtensorMap tm_k, const SantaArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Shared1 &sh = *reinterpret_cast<Shared1 *>(smem_raw + SMEM_TILES);
  const uint32_t base = smem_u32(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (base & 1023u) {  // the swizzled layouts need a 1024-byte aligned base
    if (tid == 0) atomicOr(a.err, kErrLayout);
    return;
  }
  const int t = blockIdx.x % a.n_tiles;
  const int hk = (blockIdx.x / a.n_tiles) % a.Hkv;
  const int b = blockIdx.x / (a.n_tiles * a.Hkv);
  const int j0 = (int)((long)t * a.n_b / a.n_tiles);
  const int j1 = (int)((long)(t + 1) * a.n_b / a.n_tiles);
  const int nb = j1 - j0;
  const int zkv = b * a.Hkv + hk;
  const int h0 = b * a.Hq + hk * G;  // first query head (flat) of this KV head
  float2 *stats = reinterpret_cast<float2 *>(a.tile_stats);
  if (nb == 0) {  // a tile with no key: zero weight
    if (tid < G) stats[(size_t)(h0 + tid) * a.n_tiles + t] = make_float2(-INFINITY, 0.f);
    return;
  }
  volatile int *abort = &sh.abort;

  // Q (B operand): row g < G = query head h0 + g, rows G..15 zero; two
  // 128-byte-swizzled boxes of 64 columns (16-byte chunk c of row r at chunk
  // position c ^ (r % 8)).
  {
    const __nv_bfloat16 *qg = (const __nv_bfloat16 *)a.q + (size_t)h0 * D;
    for (int idx = tid; idx < NQ * (D / 8); idx += NT1) {
      const int r = idx / (D / 8), cc = idx % (D / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < G) v = *reinterpret_cast<const uint4 *>(qg + (size_t)r * D + cc * 8);
      const int box = cc >> 3, c = cc & 7;
      st_shared_v4(base + SMEM_Q + box * Q_BOX + r * 128 + ((c ^ (r & 7)) * 16), v.x, v.y, v.z,
                   v.w);
    }
    fence_proxy_async_smem();
  }
  if (tid == 0) {
    for (int i = 0; i < NK; ++i) {
      mbar_init(smem_u32(&sh.k_full[i]), 1);
      mbar_init(smem_u32(&sh.k_empty[i]), 1);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&sh.s_full[i]), 1);
      mbar_init(smem_u32(&sh.s_free[i]), 4);  // the four score warps
    }
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == WARP_MMA) tmem_alloc(smem_u32(&sh.tmem_base), TMEM_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  if (warp == WARP_K) {
    // ---------------------------------------------------------- K producer --
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      const uint64_t pol = policy_evict_first();  // the cache is streamed once
      int issued = 0;
      for (int j = 0; j < nb && !*abort; ++j) {
        const int s = j % NK;
        if (j >= NK &&
            !mbar_wait(smem_u32(&sh.k_empty[s]), ((j / NK) - 1) & 1, abort, a.err, kErrTimeout))
          break;
        const uint32_t dst = base + SMEM_K + s * TILE_BYTES;
        const int key0 = (j0 + j) * BC;
        mbar_expect_tx(smem_u32(&sh.k_full[s]), TILE_BYTES);
        tma_load_3d(dst, &tm_k, smem_u32(&sh.k_full[s]), 0, key0, zkv, pol);
        tma_load_3d(dst + HALF_BYTES, &tm_k, smem_u32(&sh.k_full[s]), 64, key0, zkv, pol);
        ++issued;
      }
      for (int s = 0; s < NK && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / NK) * NK;
        mbar_wait_drain(smem_u32(&sh.k_full[s]), (last / NK) & 1);
      }
    }
  } else if (warp == WARP_MMA) {
    // ---------------------------------------------------------- S^T issuer --
    if (lane == 0) {
      const uint64_t qdesc = kmajor_desc(base + SMEM_Q);
      for (int j = 0; j < nb; ++j) {
        const int s = j % NK, sb = j % NS;
        if (!mbar_wait(smem_u32(&sh.k_full[s]), (j / NK) & 1, abort, a.err, kErrTimeout)) break;
        if (j >= NS && !mbar_wait(smem_u32(&sh.s_free[sb]), ((j / NS) - 1) & 1, abort, a.err,
                                  kErrTimeout))
          break;
        fence_after_sync();
        const uint64_t kd = kmajor_desc(base + SMEM_K + s * TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(tmem + sb * NQ, kd + kmajor_step(kk, HALF_BYTES),
                      qdesc + kmajor_step(kk, Q_BOX), IDESC, kk > 0);
        mma_commit(smem_u32(&sh.s_full[sb]));
        mma_commit(smem_u32(&sh.k_empty[s]));
      }
    }
  } else {
    // -------------------------------------------------------------- scores --
    // Thread (warp w, lane l) owns key 32 w + l of every block (TMEM lane
    // 32 w + l) and the G heads' scores of that key.
    const float sl2 = a.scale * kLog2e;
    const size_t row = (size_t)a.n_b * BC;  // stash row of one query head
    float *sc = a.scores + (size_t)h0 * row;
    float m[G], z[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
      z[g] = 0.f;
    }
    for (int j = 0; j < nb; ++j) {
      const int sb = j % NS;
      if (!mbar_wait_warp(smem_u32(&sh.s_full[sb]), (j / NS) & 1, abort, a.err, kErrTimeout))
        break;
      fence_after_sync();
      uint32_t x[8];
      tmem_ld8(tmem + ((uint32_t)(32 * warp) << 16) + sb * NQ, x);
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.s_free[sb]));
      const int key = (j0 + j) * BC + 32 * warp + lane;
      const bool valid = key < a.L;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float xs = valid ? __uint_as_float(x[g]) * sl2 : -INFINITY;
        sc[(size_t)g * row + key] = xs;
        if (valid) {
          if (xs > m[g]) {
            z[g] = z[g] * ex2(m[g] - xs) + 1.f;
            m[g] = xs;
          } else {
            z[g] += ex2(xs - m[g]);
          }
        }
      }
    }
    // Tile (max, sum) per head: over the lanes, then over the four warps.
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m[g], o);
        const float zo = __shfl_xor_sync(0xffffffffu, z[g], o);
        lse2_merge(m[g], z[g], mo, zo);
      }
      if (lane == 0) {
        sh.red_m[warp][g] = m[g];
        sh.red_z[warp][g] = z[g];
      }
    }
    named_bar_sync(1, 128);
    if (tid < G) {
      float mm = sh.red_m[0][tid], zz = sh.red_z[0][tid];
      for (int w = 1; w < 4; ++w) lse2_merge(mm, zz, sh.red_m[w][tid], sh.red_z[w][tid]);
      stats[(size_t)(h0 + tid) * a.n_tiles + t] = make_float2(mm, zz);
    }
  }

  __syncwarp();
  fence_before_sync();
  __syncthreads();
  if (warp == WARP_MMA) {
    fence_after_sync();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ----------------------------------------------------------------- pass 2 --
constexpr int NT2 = 256;
constexpr int NW2 = NT2 / 32;

// Smallest index i in [0, n) of a nondecreasing shared array with
// x[i] > r (strict) or x[i] >= r; n when none.  `x` is indexed through
// `at(i)` so padded layouts can be searched.
template <typename F>
__device__ __forceinline__ int first_above(int n, float r, bool strict, F at) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const float v = at(mid);
    if (strict ? (v > r) : (v >= r)) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

// Shared memory of pass 2 (floats / ints):
//   P[n_tiles + 1]        CDF at the tile boundaries (unnormalised)
//   rr[S], tile_of[S]     each sample's tile and its offset inside the tile
//   idx_s[S]              sample indices
//   cdf[NW2][64]          per warp: the chunk starts and ends of a tile
//   grp[NW2][32][4]       per warp and lane: running sums at the 16-key group ends
//   red[NW2][D]           per-warp partial sums of the gathered rows
//   su[S2], sp[S2]        i.i.d. sampler: the draws sorted ascending and their
//                         sample numbers (S2 = S rounded up to a power of two)
// A few KB: several CTAs share an SM, so the (sequence, head) CTAs run in
// one wave.
__host__ __device__ inline int pow2_ceil(int S) {
  int p = 1;
  while (p < S) p <<= 1;
  return p;
}
__host__ __device__ inline size_t sample_smem_floats(int n_tiles, int S) {
  return (size_t)(n_tiles + 1) + 3 * (size_t)S + (size_t)NW2 * 64 + (size_t)NW2 * 32 * 4 +
         (size_t)NW2 * D + 2 * (size_t)pow2_ceil(S);
}

// Running sum of exp2(x - M) over the keys of one lane chunk (consecutive
// stash entries, a multiple of 4, at most kMaxChunk), added in key order;
// the sum after every group of kGroup keys goes to grp[0..].  The search
// below resumes from those group sums and adds the same terms in the same
// order, so a sample's key follows the chunk and group ends exactly.
constexpr int kGroup = 16;                      // keys per group (4 float4 loads)
constexpr int kMaxChunk = 64;                   // keys per lane chunk at most (16 blocks a tile)
constexpr int kGroups = kMaxChunk / kGroup;     // group sums per lane
constexpr int kChunkLoads = 4;                  // float4 loads in flight per lane (16 keys)

__device__ __forceinline__ float chunk_total(const float *src, int cl, float M, float *grp) {
  float run = 0.f;
  for (int i0 = 0; i0 < cl; i0 += 4 * kChunkLoads) {
    float4 x[kChunkLoads];
#pragma unroll
    for (int q = 0; q < kChunkLoads; ++q)
      if (i0 + 4 * q < cl) x[q] = __ldg(reinterpret_cast<const float4 *>(src + i0 + 4 * q));
#pragma unroll
    for (int q = 0; q < kChunkLoads; ++q) {
      if (i0 + 4 * q < cl) {
        run += ex2(x[q].x - M);
        run += ex2(x[q].y - M);
        run += ex2(x[q].z - M);
        run += ex2(x[q].w - M);
        if (((i0 + 4 * q + 4) % kGroup) == 0 || i0 + 4 * q + 4 == cl)
          grp[(i0 + 4 * q) / kGroup] = run;
      }
    }
  }
  return run;
}

// First key i of the chunk whose running sum, offset by `pl`, exceeds `r`
// (strict) or reaches it; cl when none.  The group sums `grp` of the chunk
// pick the group; only its (at most kGroup) keys are read again.
__device__ __forceinline__ int chunk_first_above(const float *src, int cl, float M, float pl,
                                                 float r, bool strict, const float *grp) {
  const int ng = (cl + kGroup - 1) / kGroup;
  int g = 0;
  while (g < ng && !(strict ? (pl + grp[g] > r) : (pl + grp[g] >= r))) ++g;
  if (g == ng) return cl;
  const int i0 = g * kGroup;
  float run = g > 0 ? grp[g - 1] : 0.f;
  float4 x[kGroup / 4];
#pragma unroll
  for (int q = 0; q < kGroup / 4; ++q)
    if (i0 + 4 * q < cl) x[q] = __ldg(reinterpret_cast<const float4 *>(src + i0 + 4 * q));
  int found = cl;
#pragma unroll
  for (int q = 0; q < kGroup / 4; ++q) {
    if (i0 + 4 * q < cl) {
      const float e[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        run += ex2(e[u] - M);
        const float v = pl + run;
        if (found == cl && (strict ? (v > r) : (v >= r))) found = i0 + 4 * q + u;
      }
    }
  }
  return found;
}

__global__ void __launch_bounds__(NT2, 4) santa_sample_kernel(const SantaArgs a) {
  extern __shared__ float sm[];
  const int T = a.n_tiles, S = a.S;
  float *P = sm;
  float *rr = P + T + 1;
  int *tile_of = reinterpret_cast<int *>(rr + S);
  int *idx_s = tile_of + S;
  float *cdf_all = reinterpret_cast<float *>(idx_s + S);
  float *grp_all = cdf_all + (size_t)NW2 * 64;
  float *red = grp_all + (size_t)NW2 * 32 * kGroups;
  float *su = red + (size_t)NW2 * D;
  int *sp = reinterpret_cast<int *>(su + pow2_ceil(S));
  __shared__ float sh_M, sh_Z;
  __shared__ int sh_tlast;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x;
  const int G = a.Hq / a.Hkv;
  const int b = bh / a.Hq, hk = (bh % a.Hq) / G;
  const float2 *st = reinterpret_cast<const float2 *>(a.tile_stats) + (size_t)bh * T;

  // ---- 1. tile weights w_t = sum_t 2^(max_t - M) and their prefix P --------
  if (warp == 0) {
    float M = -INFINITY;
    for (int t = lane; t < T; t += 32) M = fmaxf(M, st[t].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const int ct = (T + 31) / 32, t0 = min(T, lane * ct), t1 = min(T, t0 + ct);
    float sum = 0.f;
    int tlast = -1;
    for (int t = t0; t < t1; ++t) {
      const float2 s2 = st[t];
      const float w = (s2.x == -INFINITY) ? 0.f : s2.y * ex2(s2.x - M);
      sum += w;
      if (w > 0.f) tlast = t;
    }
    float incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    float run = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) run = 0.f;
    for (int t = t0; t < t1; ++t) {
      P[t] = run;
      const float2 s2 = st[t];
      run += (s2.x == -INFINITY) ? 0.f : s2.y * ex2(s2.x - M);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tlast = max(tlast, __shfl_xor_sync(0xffffffffu, tlast, o));
    const float total = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      P[T] = total;
      sh_M = M;
      sh_Z = total;
      sh_tlast = max(tlast, 0);
    }
  }
  __syncthreads();
  const float M = sh_M, Z = sh_Z;
  const int tlast = sh_tlast;

  // ---- 2. the tile of each threshold: largest t with P[t] <= T_m Z ----------
  // The steps below want the thresholds in ascending order (a tile's samples
  // are a contiguous range): the systematic and stratified thresholds come in
  // order; the i.i.d. draws are sorted first (bitonic, with their sample
  // numbers, so that each index is reported at its own sample).
  const bool iid = a.mode == kSantaIid;
  if (iid) {
    const int S2 = pow2_ceil(S);
    for (int i = tid; i < S2; i += NT2) {
      su[i] = i < S ? a.u[(size_t)bh * S + i] : INFINITY;
      sp[i] = i;
    }
    __syncthreads();
    for (int k2 = 2; k2 <= S2; k2 <<= 1) {
      for (int j2 = k2 >> 1; j2 > 0; j2 >>= 1) {
        for (int i = tid; i < S2; i += NT2) {
          const int o = i ^ j2;
          if (o > i && ((su[i] > su[o]) == ((i & k2) == 0))) {
            const float tu = su[i];
            su[i] = su[o];
            su[o] = tu;
            const int tp = sp[i];
            sp[i] = sp[o];
            sp[o] = tp;
          }
        }
        __syncthreads();
      }
    }
  }
  const float invS = 1.f / (float)S;
  for (int m = tid; m < S; m += NT2) {
    float R;
    if (iid) {
      R = su[m] * Z;
    } else {
      const float um = a.mode == kSantaSys ? a.u[bh] : a.u[(size_t)bh * S + m];
      R = ((float)m + um) * invS * Z;
    }
    int lo = 0, hi = T - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (P[mid] <= R) lo = mid;
      else hi = mid - 1;
    }
    const int t = min(lo, tlast);
    tile_of[m] = t;
    rr[m] = R - P[t];
    idx_s[m] = 0;
  }
  __syncthreads();

  // ---- 3. per tile holding samples: chunk sums and each sample's key ------
  // Lane l of the tile's warp owns a chunk of cl consecutive keys: the chunk
  // totals and their prefix over the lanes locate a sample's chunk; the
  // sample's lane then walks that chunk's running sum to its key.
  {
    float *pre = cdf_all + (size_t)warp * 64;  // chunk starts
    float *ends = pre + 32;                    // chunk ends
    float *grp = grp_all + (size_t)warp * 32 * kGroups;  // [lane][group] running sums
    const size_t row = (size_t)a.n_b * BC;
    for (int t = warp; t < T; t += NW2) {
      const int mlo = first_above(S, (float)t, false, [&](int i) { return (float)tile_of[i]; });
      const int mhi = first_above(S, (float)t, true, [&](int i) { return (float)tile_of[i]; });
      if (mlo >= mhi) continue;
      const int jb0 = (int)((long)t * a.n_b / T), jb1 = (int)((long)(t + 1) * a.n_b / T);
      const int k0 = jb0 * BC;
      const int cl = (jb1 - jb0) * (BC / 32);  // keys per lane in this tile (multiple of 4)
      if (cl == 0) continue;  // a tile with no key gets no sample unless the weights are NaN
      const float *tile_src = a.scores + (size_t)bh * row + k0;
      const float run = chunk_total(tile_src + (size_t)lane * cl, cl, M, grp + lane * kGroups);
      float incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      float p0 = __shfl_up_sync(0xffffffffu, incl, 1);
      if (lane == 0) p0 = 0.f;
      pre[lane] = p0;
      ends[lane] = p0 + run;
      __syncwarp();
      const float tot = ends[31];
      for (int m = mlo + lane; m < mhi; m += 32) {
        // Smallest key whose running sum exceeds the sample's offset; past the
        // tile's own total (rounding), the last key of positive weight.
        float r = rr[m];
        bool strict = true;
        int l = first_above(32, r, true, [&](int i) { return ends[i]; });
        if (l == 32) {
          r = tot;
          strict = false;
          l = first_above(32, r, false, [&](int i) { return ends[i]; });
          if (l == 32) l = 31;
        }
        int ii = chunk_first_above(tile_src + (size_t)l * cl, cl, M, pre[l], r, strict,
                                   grp + l * kGroups);
        if (ii >= cl) ii = cl - 1;
        idx_s[m] = max(0, min(k0 + l * cl + ii, a.L - 1));
      }
      __syncwarp();
    }
  }
  __syncthreads();

  // ---- 4. gather the sampled value rows ---------------------------------------
  const __nv_bfloat16 *vb = (const __nv_bfloat16 *)a.v + (size_t)(b * a.Hkv + hk) * a.L * D;
  // Up to kGather rows in flight per warp; added in sample order.
  constexpr int kGather = 8;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int m0 = warp; m0 < S; m0 += NW2 * kGather) {
    uint2 raw[kGather];
#pragma unroll
    for (int q = 0; q < kGather; ++q) {
      const int m = m0 + q * NW2;
      if (m < S)
        raw[q] = __ldg(reinterpret_cast<const uint2 *>(vb + (size_t)idx_s[m] * D + lane * 4));
    }
#pragma unroll
    for (int q = 0; q < kGather; ++q) {
      if (m0 + q * NW2 < S) {
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw[q].x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw[q].y));
        acc[0] += lo.x;
        acc[1] += lo.y;
        acc[2] += hi.x;
        acc[3] += hi.y;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) red[warp * D + lane * 4 + i] = acc[i];
  __syncthreads();
  if (tid < D) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NW2; ++w) s += red[w * D + tid];
    s *= invS;
    if (a.out_bf16)
      reinterpret_cast<__nv_bfloat16 *>(a.o)[(size_t)bh * D + tid] = __float2bfloat16_rn(s);
    else
      reinterpret_cast<float *>(a.o)[(size_t)bh * D + tid] = s;
  }
  if (a.idx)
    for (int m = tid; m < S; m += NT2) a.idx[(size_t)bh * S + (iid ? sp[m] : m)] = idx_s[m];
}

}  // namespace

size_t santa_sample_smem_bytes(int n_tiles, int S) {
  return sample_smem_floats(n_tiles, S) * sizeof(float);
}

cudaError_t launch_santa_decode(const SantaArgs &a, cudaStream_t s) {
  CUtensorMap mk;
  // [B*Hkv, L, 128] bf16; boxes of 64 columns x 128 keys; keys past L read as
  // zero (their scores are stashed as -inf).
  if (!make_map_bf16_3d(&mk, a.k, D, D, a.L, a.B * a.Hkv, BC)) return cudaErrorInvalidValue;
  const int G = a.Hq / a.Hkv;
  auto k1 = G == 1   ? santa_scores_kernel<1>
            : G == 2 ? santa_scores_kernel<2>
            : G == 4 ? santa_scores_kernel<4>
            : G == 8 ? santa_scores_kernel<8>
                     : nullptr;
  if (!k1) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM1);
  if (e != cudaSuccess) return e;
  const long units = (long)a.B * a.Hkv * a.n_tiles;
  k1<<<(unsigned)units, NT1, SMEM1, s>>>(mk, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem2 = santa_sample_smem_bytes(a.n_tiles, a.S);
  e = cudaFuncSetAttribute(santa_sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem2);
  if (e != cudaSuccess) return e;
  santa_sample_kernel<<<(unsigned)((long)a.B * a.Hq), NT2, smem2, s>>>(a);
  return cudaGetLastError();
}

}  // namespace attn_skip
