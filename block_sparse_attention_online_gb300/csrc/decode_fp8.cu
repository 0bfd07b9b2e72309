// Split-KV decode with softmax-threshold block skipping over an FP8 (E4M3)
// key/value cache (d = 128, Bc = 128), on the tensor cores.
//
// Method: the BLASST page, sections "BLASST 的判定准则" (Eq. 5) and "Decode 内核：
// 砍带宽": the scores of a block decide whether its values are read at all;
// the cache format is E4M3 codes with one fp32 scale per (sequence, KV head)
// for keys and for values (the page evaluates FP8/NVFP4 models and names no
// cache format; this is the plainest one).  Decode is bound by the cache
// bytes, so halving them halves the time of the same schedule -- provided
// shared memory, which every byte crosses, keeps up.
//
// The schedule is that of the bf16 decode kernel: the G query heads sharing
// a KV head are padded to the 128 rows of a tcgen05 MMA, one softmax warp
// holds each head's 128 scores in one thread (row maxima, votes and the group
// decision need no reduction across warps) and frees the S buffer as soon as
// the scores are in registers, P has two TMEM buffers, and values are loaded
// only for kept blocks, as soon as the decision exists.
//
// Keys stay E4M3 all the way: S = Q K^T is a kind::f8f6f4 product straight
// from the TMA tile.  The query is written once, exactly, as an E4M3 pair: per
// head, q 2^e (the largest power of two keeping the row within 256) = hi + lo
// with hi = E4M3(q 2^e) and lo = E4M3(q 2^e - hi), which for a bf16 row is
// exact except for elements below about 2^-10 of the row's largest; S = hi
// K^T + lo K^T (eight k-steps of 32 codes, fp32 accumulation) and 2^-e goes
// into the head's score scale.  Values are widened, exactly, to fp16 by
// converter warps (P is no E4M3 quantity: its small weights would vanish) and
// O += P V is a kind::f16 product with P in fp16.  Widening the keys as well
// would move three times their bytes through shared memory.  The key scale
// multiplies the scores (folded into the score scale), the value scale the
// split outputs.
//
// Warp roles (256 threads):
//   warp 0      softmax: lane g < G owns head g (TMEM lane g);
//   warp 1      TMA producer of the E4M3 key tiles (every block, 6 stages);
//   warp 2      Q.K^T issuer (A = the Q pair, B = the E4M3 key tile, both in
//               shared memory; allocates TMEM);
//   warp 3      TMA producer of the E4M3 value tiles of kept blocks (2 stages);
//   warp 4      P.V issuer (A = P from TMEM, B = fp16 V tile);
//   warps 5-7   value converters (follow the decisions; a third of each tile).
// TMEM columns: S buffers [0,256), P buffers [256,384), O [384,512).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "internal.h"
#include "tc_common.cuh"

namespace attn_skip {
namespace {

using namespace tc;

constexpr int D = 128;    // head size (keys and values)
constexpr int BC = 128;   // keys per block
constexpr int MR = 128;   // MMA rows (heads padded)
constexpr int NKF = 6;    // E4M3 key stages
constexpr int NVF = 2;    // E4M3 value stages
constexpr int NVH = 2;    // fp16 value stages
constexpr int NS = 2;     // TMEM S buffers
constexpr int NP = 2;     // TMEM P buffers
constexpr int NDEC = 8;   // decision ring
constexpr int NT = 8 * 32;
constexpr int WARP_K = 1, WARP_QK = 2, WARP_V = 3, WARP_PV = 4;  // warp 0: softmax
constexpr int WARP_VC = 5;                                        // three warps
constexpr int NVC = 3 * 32;                                       // converter threads
constexpr uint32_t F8_BYTES = BC * D;           // 16 KB: 128 rows x 128 codes
constexpr uint32_t H_BYTES = BC * D * 2;        // 32 KB: 128 keys x 128 fp16
constexpr uint32_t HALF_BYTES = H_BYTES / 2;    // one 64-column swizzled box
constexpr uint32_t SMEM_KF = 0;
constexpr uint32_t SMEM_Q = SMEM_KF + NKF * F8_BYTES;  // Q hi, then Q lo
constexpr uint32_t SMEM_VF = SMEM_Q + 2 * F8_BYTES;
constexpr uint32_t SMEM_VH = SMEM_VF + NVF * F8_BYTES;
constexpr uint32_t SMEM_TILES = SMEM_VH + NVH * H_BYTES;  // 224 KB
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_P = NS * BC;             // 256
constexpr uint32_t TMEM_O = TMEM_P + NP * (BC / 2);  // 384
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // exp reference may lag the max by 2^8
constexpr uint32_t IDESC_QK = idesc_e4m3_f32(MR, BC);    // E4M3 x E4M3, both K-major
constexpr uint32_t IDESC_PV = idesc_f16_f32(MR, D, 1);   // V tile: MN-major
constexpr uint32_t NEG_INF_BITS = 0xff800000u;
static_assert(TMEM_O + D == TMEM_COLS, "TMEM budget");

struct Shared {
  uint64_t kf_full[NKF], kf_empty[NKF];
  uint64_t vf_full[NVF], vf_empty[NVF];
  uint64_t vh_full[NVH], vh_empty[NVH];
  uint64_t s_full[NS], s_free[NS];
  uint64_t p_full[NP], p_free[NP];
  uint64_t pv_done[2];
  uint64_t dec_full[NDEC], dec_empty[NDEC];
  int dec[NDEC];
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t SMEM_ALLOC = SMEM_TILES + ((sizeof(Shared) + 127) / 128) * 128;
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");

// E4M3 tiles (the key tile, the two query tiles) as K-major operands of
// Q.K^T: one 128-byte-swizzled box of 128 codes x 128 rows; k-step kk (32
// codes) starts 32 bytes further, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t kmajor8_base(uint32_t tile) {
  return smem_desc_sw128(tile, 16u, 1024u);
}
__device__ __forceinline__ constexpr uint64_t kmajor8_step(int kk) {
  return (uint64_t)(((uint32_t)kk * 32u) >> 4);
}
// fp16 value tiles: two 128-byte-swizzled boxes of 64 columns, 128 rows each,
// as the MN-major B operand of P.V (rows are keys): 8-key groups 1024 bytes
// apart, the second 64-value half 16 KB further; k-step kk (16 keys) starts
// 2048 bytes further.
__device__ __forceinline__ uint64_t vmajor_base(uint32_t tile) {
  return smem_desc_sw128(tile, HALF_BYTES, 1024u);
}
__device__ __forceinline__ constexpr uint64_t vmajor_step(int kk) {
  return (uint64_t)(((uint32_t)kk * 2048u) >> 4);
}

// Two E4M3 codes -> an fp16 pair holding the code values times 2^-8, exactly
// (the 2^8 goes into the value scale): with the code in the high byte of a
// half word, the sign is already in place and the seven exponent / mantissa
// bits, shifted right by one, land on the fp16 exponent / mantissa with the
// exponent bias 7 read as 15 (subnormal codes become subnormal halves).
// `w` holds the codes at bits 8-15 and 24-31.  NaN codes are not expected.
__device__ __forceinline__ uint32_t e4m3_hi_bytes_to_f16x2(uint32_t w) {
  return (w & 0x80008000u) | ((w >> 1) & 0x3f803f80u);
}

// Chunk c (codes 16c..16c+15) of row r of an E4M3 tile (128 codes per row,
// 128-byte-swizzled: chunk c at chunk position c ^ (r % 8)) -> the same
// columns of row r of an fp16 tile of the values times 2^-8 (columns
// 64b..64b+63 in box b, 16-byte chunk c' of a box row at position c' ^ (r % 8)).
__device__ __forceinline__ void widen_chunk(uint32_t src_tile, uint32_t dst_tile, int r, int c) {
  const uint32_t sw = (uint32_t)(r & 7);
  uint32_t x[4];
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
               : "r"(src_tile + (uint32_t)r * 128u + (((uint32_t)c ^ sw) << 4)));
  uint32_t h[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[2 * i] = e4m3_hi_bytes_to_f16x2(__byte_perm(x[i], 0u, 0x1404));      // codes 0, 1
    h[2 * i + 1] = e4m3_hi_bytes_to_f16x2(__byte_perm(x[i], 0u, 0x3424));  // codes 2, 3
  }
  const uint32_t box = dst_tile + (uint32_t)r * 128u + (uint32_t)(c >> 2) * HALF_BYTES;
  const uint32_t c0 = (uint32_t)(2 * (c & 3));
  st_shared_v4(box + ((c0 ^ sw) << 4), h[0], h[1], h[2], h[3]);
  st_shared_v4(box + (((c0 + 1) ^ sw) << 4), h[4], h[5], h[6], h[7]);
}

__device__ __forceinline__ float chunk_max(const uint32_t (&s)[32]) {
  float m[11];
#pragma unroll
  for (int i = 0; i < 10; ++i)
    m[i] = fmax3(__uint_as_float(s[3 * i]), __uint_as_float(s[3 * i + 1]),
                 __uint_as_float(s[3 * i + 2]));
  m[10] = fmaxf(__uint_as_float(s[30]), __uint_as_float(s[31]));
  const float a = fmax3(m[0], m[1], m[2]), b = fmax3(m[3], m[4], m[5]);
  const float c = fmax3(m[6], m[7], m[8]), d = fmaxf(m[9], m[10]);
  return fmaxf(fmax3(a, b, c), d);
}

// P = exp2(s * sl2 - ref) for one 32-key chunk as 16 packed fp16 pairs, with
// the row sum accumulated in two packed fp32 pairs.
__device__ __forceinline__ void chunk_exp(const uint32_t (&s)[32], uint64_t sl2x2,
                                          uint64_t negref2, uint64_t (&acc)[2],
                                          uint32_t *pk) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float x0, x1;
    f2_split(f2_fma(f2(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), sl2x2,
                    negref2),
             x0, x1);
    const float p0 = ex2(x0), p1 = ex2(x1);
    acc[i & 1] = f2_add(acc[i & 1], f2(p0, p1));
    pk[i] = pack_f16x2(p0, p1);
  }
}

// Scores of keys at or past the cache end (the zero-filled tail of the last
// block) become -inf in TMEM before anything reads them.  Short and out of
// line: it runs once per sequence from a cold instruction cache.
__device__ __noinline__ void mask_tail_tmem(uint32_t sa, int lim) {
  uint32_t ninf[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) ninf[i] = NEG_INF_BITS;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    const int l = lim - 32 * c;
    if (l >= 32) continue;
    if (l <= 0) {
      tmem_st32(sa + 32 * c, ninf);
      continue;
    }
    uint32_t x[32];
    tmem_ld32(sa + 32 * c, x);
    tmem_wait_ld_regs(x);
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = i < l ? x[i] : NEG_INF_BITS;
    tmem_st32(sa + 32 * c, x);
  }
  tmem_wait_st();
}


// The query pair of head row r (r < G: query head hk*G + r) into the two
// E4M3 query tiles (128-byte-swizzled rows of 128 codes); other rows zero.
// Returns the row's exponent e (q 2^e = hi + lo, max |q| 2^e <= 256).
__device__ __forceinline__ int write_query_pair(const DecodeArgs &a, int b, int hk, int G, int r,
                                                uint32_t q_hi, uint32_t q_lo) {
  const uint32_t sw = (uint32_t)(r & 7);
  if (r >= G) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t off = (uint32_t)r * 128u + (((uint32_t)c ^ sw) << 4);
      st_shared_v4(q_hi + off, 0u, 0u, 0u, 0u);
      st_shared_v4(q_lo + off, 0u, 0u, 0u, 0u);
    }
    return 0;
  }
  // bf16 pairs of the row (low element first), 8 per 16-byte load.
  const uint4 *qr = reinterpret_cast<const uint4 *>((const __nv_bfloat16 *)a.q +
                                                    (size_t)(b * a.Hq + hk * G + r) * D);
  uint32_t amax_bits = 0;  // |bf16| bit patterns order like their values
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint4 v = __ldg(qr + i);
    amax_bits = max(amax_bits, max(v.x & 0x7fffu, (v.x >> 16) & 0x7fffu));
    amax_bits = max(amax_bits, max(v.y & 0x7fffu, (v.y >> 16) & 0x7fffu));
    amax_bits = max(amax_bits, max(v.z & 0x7fffu, (v.z >> 16) & 0x7fffu));
    amax_bits = max(amax_bits, max(v.w & 0x7fffu, (v.w >> 16) & 0x7fffu));
  }
  const float amax = __uint_as_float(amax_bits << 16);
  int ex = 0;
  const float fr = frexpf(amax > 0.f ? amax : 1.f, &ex);  // amax = fr * 2^ex
  const int qexp = amax > 0.f ? 8 - (fr == 0.5f ? ex - 1 : ex) : 0;  // 8 - ceil(log2 amax)
#pragma unroll 2
  for (int c = 0; c < 8; ++c) {  // codes 16c .. 16c+15: two 16-byte loads of bf16
    const uint4 v0 = __ldg(qr + 2 * c), v1 = __ldg(qr + 2 * c + 1);
    const uint32_t pr[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t wh = 0, wl = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t pair = pr[2 * w + (i >> 1)];
        const float q = __uint_as_float((i & 1) ? (pair & 0xffff0000u) : (pair << 16));
        const float x = ldexpf(q, qexp);      // exact
        const __nv_fp8_e4m3 h(x);             // nearest even
        const __nv_fp8_e4m3 l(x - (float)h);  // x - h is exact
        wh |= (uint32_t)h.__x << (8 * i);
        wl |= (uint32_t)l.__x << (8 * i);
      }
      hi[w] = wh;
      lo[w] = wl;
    }
    const uint32_t off = (uint32_t)r * 128u + (((uint32_t)c ^ sw) << 4);
    st_shared_v4(q_hi + off, hi[0], hi[1], hi[2], hi[3]);
    st_shared_v4(q_lo + off, lo[0], lo[1], lo[2], lo[3]);
  }
  return qexp;
}

__global__ void __launch_bounds__(NT, 1)
    decode_fp8_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Shared &sh = *reinterpret_cast<Shared *>(smem_raw + SMEM_TILES);
  const uint32_t base = smem_u32(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (base & 1023u) {  // the swizzled layouts need a 1024-byte aligned base
    if (tid == 0) atomicOr(a.err, kErrTimeout);
    return;
  }
  const int G = a.Hq / a.Hkv;
  const int unit = blockIdx.x;
  const int sp = unit % a.n_splits;
  const int hk = (unit / a.n_splits) % a.Hkv;
  const int b = unit / (a.n_splits * a.Hkv);
  const int j0 = (int)((long)sp * a.n_b / a.n_splits);
  const int j1 = (int)((long)(sp + 1) * a.n_b / a.n_splits);
  const int nb = j1 - j0;
  const int zkv = b * a.Hkv + hk;
  volatile int *abort = &sh.abort;

  if (nb == 0) {  // empty split: no key, zero weight in the merge
    for (int idx = tid; idx < G * D; idx += NT) {
      const size_t row = (size_t)(b * a.Hq + hk * G + idx / D) * a.n_splits + sp;
      a.o_part[row * D + idx % D] = 0.f;
      if (idx % D == 0) a.lse_part[row] = -INFINITY;
    }
    for (int idx = tid; idx < a.words; idx += NT) a.bits[(size_t)unit * a.words + idx] = 0u;
    return;
  }

  // The query pair (threads 0-127, one row each); thread g < G keeps its
  // head's exponent for the score scale.
  int qexp = 0;
  if (tid < MR) qexp = write_query_pair(a, b, hk, G, tid, base + SMEM_Q, base + SMEM_Q + F8_BYTES);
  fence_proxy_async_smem();  // visible to the tensor core
  if (tid == 0) {
    for (int i = 0; i < NKF; ++i) {
      mbar_init(smem_u32(&sh.kf_full[i]), 1);
      mbar_init(smem_u32(&sh.kf_empty[i]), 1);  // the Q.K^T commit
    }
    for (int i = 0; i < NVF; ++i) {
      mbar_init(smem_u32(&sh.vf_full[i]), 1);
      mbar_init(smem_u32(&sh.vf_empty[i]), 3);  // the three value converters
    }
    for (int i = 0; i < NVH; ++i) {
      mbar_init(smem_u32(&sh.vh_full[i]), 3);
      mbar_init(smem_u32(&sh.vh_empty[i]), 1);  // the P.V commit
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&sh.s_full[i]), 1);
      mbar_init(smem_u32(&sh.s_free[i]), 1);
    }
    for (int i = 0; i < NP; ++i) {
      mbar_init(smem_u32(&sh.p_full[i]), 1);
      mbar_init(smem_u32(&sh.p_free[i]), 1);
    }
    mbar_init(smem_u32(&sh.pv_done[0]), 1);
    mbar_init(smem_u32(&sh.pv_done[1]), 1);
    for (int i = 0; i < NDEC; ++i) {
      mbar_init(smem_u32(&sh.dec_full[i]), 1);
      // readers: the value producer, the P.V issuer, the three value converters
      mbar_init(smem_u32(&sh.dec_empty[i]), 5);
    }
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == WARP_QK) tmem_alloc(smem_u32(&sh.tmem_base), TMEM_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  if (warp == WARP_K) {
    // ------------------------------------------------- E4M3 key producer --
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      const uint64_t pol = policy_evict_first();  // the cache is streamed once
      int issued = 0;
      for (int j = 0; j < nb && !*abort; ++j) {
        const int f = j % NKF;
        if (j >= NKF &&
            !mbar_wait(smem_u32(&sh.kf_empty[f]), ((j / NKF) - 1) & 1, abort, a.err, kErrTimeout))
          break;
        mbar_expect_tx(smem_u32(&sh.kf_full[f]), F8_BYTES);
        tma_load_3d(base + SMEM_KF + f * F8_BYTES, &tm_k, smem_u32(&sh.kf_full[f]), 0,
                    (j0 + j) * BC, zkv, pol);
        ++issued;
      }
      for (int f = 0; f < NKF && f < issued; ++f) {
        const int last = f + ((issued - 1 - f) / NKF) * NKF;
        mbar_wait_drain(smem_u32(&sh.kf_full[f]), (last / NKF) & 1);
      }
    }
  } else if (warp == WARP_V) {
    // ----------------------------------------------- E4M3 value producer --
    if (lane == 0) {
      prefetch_tmap(&tm_v);
      const uint64_t pol = policy_evict_first();
      int vi = 0;
      for (int j = 0; j < nb && !*abort; ++j) {
        if (!mbar_wait(smem_u32(&sh.dec_full[j % NDEC]), (j / NDEC) & 1, abort, a.err,
                       kErrTimeout))
          break;
        const int keep = sh.dec[j % NDEC];
        mbar_arrive(smem_u32(&sh.dec_empty[j % NDEC]));
        if (!keep) continue;
        const int f = vi % NVF;
        if (vi >= NVF &&
            !mbar_wait(smem_u32(&sh.vf_empty[f]), ((vi / NVF) - 1) & 1, abort, a.err, kErrTimeout))
          break;
        mbar_expect_tx(smem_u32(&sh.vf_full[f]), F8_BYTES);
        tma_load_3d(base + SMEM_VF + f * F8_BYTES, &tm_v, smem_u32(&sh.vf_full[f]), 0,
                    (j0 + j) * BC, zkv, pol);
        ++vi;
      }
      for (int f = 0; f < NVF && f < vi; ++f) {
        const int last = f + ((vi - 1 - f) / NVF) * NVF;
        mbar_wait_drain(smem_u32(&sh.vf_full[f]), (last / NVF) & 1);
      }
    }
  } else if (warp >= WARP_VC) {
    // -------------------------------------------------- value converters --
    // Follow the decisions; chunks t, t + 96, ... (row = chunk / 8) of every
    // kept value tile.
    const int t0 = (warp - WARP_VC) * 32 + lane;
    int vi = 0;
    for (int j = 0; j < nb; ++j) {
      if (!mbar_wait_warp(smem_u32(&sh.dec_full[j % NDEC]), (j / NDEC) & 1, abort, a.err,
                          kErrTimeout))
        break;
      const int keep = sh.dec[j % NDEC];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.dec_empty[j % NDEC]));
      if (!keep) continue;
      const int f = vi % NVF, hs = vi % NVH;
      if (!mbar_wait_warp(smem_u32(&sh.vf_full[f]), (vi / NVF) & 1, abort, a.err, kErrTimeout))
        break;
      if (vi >= NVH && !mbar_wait_warp(smem_u32(&sh.vh_empty[hs]), ((vi / NVH) - 1) & 1, abort,
                                       a.err, kErrTimeout))
        break;
#pragma unroll 4
      for (int t = t0; t < BC * 8; t += NVC)
        widen_chunk(base + SMEM_VF + f * F8_BYTES, base + SMEM_VH + hs * H_BYTES, t >> 3, t & 7);
      fence_proxy_async_smem();  // the fp16 rows are visible to the tensor core
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sh.vf_empty[f]));
        mbar_arrive(smem_u32(&sh.vh_full[hs]));
      }
      ++vi;
    }
  } else if (warp == WARP_QK) {
    // -------------------------------------------------------- Q.K^T issuer --
    if (lane == 0) {
      const uint64_t qhi = kmajor8_base(base + SMEM_Q), qlo = kmajor8_base(base + SMEM_Q + F8_BYTES);
      for (int j = 0; j < nb; ++j) {
        const int f = j % NKF, sb = j % NS;
        if (!mbar_wait(smem_u32(&sh.kf_full[f]), (j / NKF) & 1, abort, a.err, kErrTimeout))
          break;
        // S buffer sb is free once the softmax warp has read block j - NS.
        if (j >= NS && !mbar_wait(smem_u32(&sh.s_free[sb]), ((j / NS) - 1) & 1, abort, a.err,
                                  kErrTimeout))
          break;
        fence_after_sync();
        const uint64_t kd = kmajor8_base(base + SMEM_KF + f * F8_BYTES);
        const uint32_t d_s = tmem + sb * BC;
        // S = hi K^T + lo K^T: four k-steps of 32 codes for each part.
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_f8f6f4_ss(d_s, (kk < 4 ? qhi : qlo) + kmajor8_step(kk & 3),
                        kd + kmajor8_step(kk & 3), IDESC_QK, kk > 0);
        mma_commit(smem_u32(&sh.s_full[sb]));
        mma_commit(smem_u32(&sh.kf_empty[f]));
      }
    }
  } else if (warp == WARP_PV) {
    // ---------------------------------------------------------- P.V issuer --
    if (lane == 0) {
      int kc = 0;
      for (int j = 0; j < nb && !*abort; ++j) {
        if (!mbar_wait(smem_u32(&sh.dec_full[j % NDEC]), (j / NDEC) & 1, abort, a.err,
                       kErrTimeout))
          break;
        const int keep = sh.dec[j % NDEC];
        mbar_arrive(smem_u32(&sh.dec_empty[j % NDEC]));
        if (!keep) continue;
        const int pb = kc % NP, hs = kc % NVH;
        if (!mbar_wait(smem_u32(&sh.p_full[pb]), (kc / NP) & 1, abort, a.err, kErrTimeout) ||
            !mbar_wait(smem_u32(&sh.vh_full[hs]), (kc / NVH) & 1, abort, a.err, kErrTimeout))
          break;
        fence_after_sync();
        // P (fp16 pairs): keys [0,128) in the 64 columns of P buffer pb.
        const uint32_t pt = tmem + TMEM_P + pb * (BC / 2);
        const uint64_t vd = vmajor_base(base + SMEM_VH + hs * H_BYTES);
#pragma unroll
        for (int kk = 0; kk < BC / 16; ++kk)
          mma_bf16_ts(tmem + TMEM_O, pt + kk * 8, vd + vmajor_step(kk), IDESC_PV,
                      (kc > 0 || kk > 0) ? 1u : 0u);
        mma_commit(smem_u32(&sh.vh_empty[hs]));
        mma_commit(smem_u32(&sh.p_free[pb]));
        mma_commit(smem_u32(&sh.pv_done[kc & 1]));
        ++kc;
      }
    }
  } else {
    // ------------------------------------------------------------- softmax --
    // Lane g < G: head g's row (TMEM lane g) over the block's 128 keys.
    const bool head = lane < G;
    uint32_t *bits = a.bits + (size_t)unit * a.words;
    // Raw score -> log2 units: the score scale, the key scale and 2^-e of the
    // head's query pair.
    const float sl2 = ldexpf(a.scale * __ldg(a.k_scale + zkv) * kLog2e, -qexp);
    const float c2 = a.ln_lambda * kLog2e;  // ln(lambda), log2 units
    float m2 = -INFINITY;    // running max of the split (log2 units)
    float mref = -INFINITY;  // exp reference (log2 units)
    float l = 0.f;           // row sum relative to mref
    int kc = 0;              // kept blocks
    uint32_t word = 0;
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      const int sb = j % NS;
      if (!mbar_wait_warp(smem_u32(&sh.s_full[sb]), (j / NS) & 1, abort, a.err, kErrTimeout)) {
        ok = false;
        break;
      }
      fence_after_sync();
      const uint32_t sa = tmem + sb * BC;  // lanes 0-31: this warp's TMEM quarter
      const int lim = a.L - (j0 + j) * BC;
      if (lim < BC) mask_tail_tmem(sa, lim);
      uint32_t x0[32], x1[32], x2[32], x3[32];
      tmem_ld32(sa, x0);
      tmem_ld32(sa + 32, x1);
      tmem_ld32(sa + 64, x2);
      tmem_ld32(sa + 96, x3);
      tmem_wait_ld_regs(x0);
      tmem_wait_ld_regs(x1);
      tmem_wait_ld_regs(x2);
      tmem_wait_ld_regs(x3);
      // The scores are in registers: the S buffer can take block j + NS.
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.s_free[sb]));
      const float mt =
          fmaxf(fmaxf(chunk_max(x0), chunk_max(x1)), fmaxf(chunk_max(x2), chunk_max(x3)));
      const float pm2 = mt * sl2;
      // With c < 0, "rowmax - m_new < c" is "rowmax - m_old < c" (a block
      // that raises the max fails both).  Every head must vote skip.
      const float diff = (mt == -INFINITY) ? -INFINITY : pm2 - m2;
      const bool skip = __all_sync(0xffffffffu, !head || diff < c2);
      if (lane == 0) {
        // On a timeout the abort flag is raised and every later wait fails.
        if (j < NDEC || mbar_wait(smem_u32(&sh.dec_empty[j % NDEC]), ((j / NDEC) - 1) & 1,
                                  abort, a.err, kErrTimeout)) {
          sh.dec[j % NDEC] = skip ? 0 : 1;
          mbar_arrive(smem_u32(&sh.dec_full[j % NDEC]));
        }
        if (skip) word |= 1u << (j & 31);
        if ((j & 31) == 31 || j == nb - 1) {
          bits[j >> 5] = word;
          word = 0;
        }
      }
      // The running max advances on every block (a skipped block leaves it unchanged).
      const float mnew = fmaxf(m2, pm2);
      m2 = mnew;
      if (skip) continue;
      bool rescale = false;
      float alpha = 1.f;
      if (mref == -INFINITY) {
        mref = mnew;
      } else if (mnew > mref + kRescaleLog2) {
        alpha = ex2(mref - mnew);
        mref = mnew;
        rescale = true;
      }
      const int pb = kc % NP;
      // P buffer pb last fed the P.V of kept block kc - NP.
      if (kc >= NP && !mbar_wait_warp(smem_u32(&sh.p_free[pb]), ((kc / NP) - 1) & 1, abort,
                                      a.err, kErrTimeout)) {
        ok = false;
        break;
      }
      fence_after_sync();
      const uint32_t pa = tmem + TMEM_P + pb * (BC / 2);
      const uint64_t sl2x2 = f2(sl2, sl2), negref2 = f2(-mref, -mref);
      uint64_t acc2[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
      {
        uint32_t pk[32];
        chunk_exp(x0, sl2x2, negref2, acc2, pk);
        chunk_exp(x1, sl2x2, negref2, acc2, pk + 16);
        tmem_st32(pa, pk);
        chunk_exp(x2, sl2x2, negref2, acc2, pk);
        chunk_exp(x3, sl2x2, negref2, acc2, pk + 16);
        tmem_st32(pa + 32, pk);
      }
      tmem_wait_st();
      float acc[4];
      f2_split(acc2[0], acc[0], acc[1]);
      f2_split(acc2[1], acc[2], acc[3]);
      l = l * alpha + ((acc[0] + acc[1]) + (acc[2] + acc[3]));
      // O rescale of the heads' rows once the previous P.V has landed.
      if (__any_sync(0xffffffffu, rescale) && kc >= 1) {
        if (!mbar_wait_warp(smem_u32(&sh.pv_done[(kc - 1) & 1]), ((kc - 1) >> 1) & 1, abort,
                            a.err, kErrTimeout)) {
          ok = false;
          break;
        }
        fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          const uint32_t oa = tmem + TMEM_O + c * 32;
          tmem_ld32(oa, o);
          tmem_wait_ld_regs(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(oa, o);
        }
        tmem_wait_st();
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.p_full[pb]));
      ++kc;
    }

    // ---- epilogue: O_s = v_scale * O / l and LSE_s = ref + ln l per head ----
    if (lane == 0)
      for (int w = ((nb - 1) >> 5) + 1; w < a.words; ++w) bits[w] = 0u;
    if (ok && kc > 0)
      ok = mbar_wait_warp(smem_u32(&sh.pv_done[(kc - 1) & 1]), ((kc - 1) >> 1) & 1, abort, a.err,
                          kErrTimeout);
    if (ok) {
      fence_after_sync();
      const float inv = __ldg(a.v_scale + zkv) * 256.f / l;  // values were widened times 2^-8
      const size_t row = (size_t)(b * a.Hq + hk * G + lane) * a.n_splits + sp;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + TMEM_O + c * 32, o);
        tmem_wait_ld_regs(o);
        if (head) {
          float4 *dst = reinterpret_cast<float4 *>(a.o_part + row * D + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            dst[q4] = make_float4(__uint_as_float(o[4 * q4]) * inv,
                                  __uint_as_float(o[4 * q4 + 1]) * inv,
                                  __uint_as_float(o[4 * q4 + 2]) * inv,
                                  __uint_as_float(o[4 * q4 + 3]) * inv);
        }
      }
      if (head) a.lse_part[row] = mref * kLn2 + logf(l);
    }
  }

  __syncwarp();
  fence_before_sync();
  __syncthreads();
  if (warp == WARP_QK) {
    fence_after_sync();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_decode_fp8(const DecodeArgs &a, cudaStream_t s) {
  CUtensorMap mk, mv;
  // [B*Hkv, L, 128] E4M3 codes with the caller's row stride (bytes); boxes of
  // 128 codes x 128 keys; keys past L read as zero (and are masked).
  if (!make_map_u8_3d(&mk, a.k, D, a.k_row_stride, a.L, a.B * a.Hkv, BC) ||
      !make_map_u8_3d(&mv, a.v, D, a.v_row_stride, a.L, a.B * a.Hkv, BC))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(decode_fp8_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  const long units = (long)a.B * a.Hkv * a.n_splits;
  decode_fp8_kernel<<<(unsigned)units, NT, SMEM_ALLOC, s>>>(mk, mv, a);
  return cudaGetLastError();
}

}  // namespace attn_skip
