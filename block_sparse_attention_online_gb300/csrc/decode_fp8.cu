// Split-KV decode with softmax-threshold block skipping over an FP8 (E4M3)
// key/value cache (d = 128, Bc = 128), on the tensor cores.
//
// Method: the BLASST page, sections "BLASST 的判定准则" (Eq. 5) and "Decode 内核：
// 砍带宽": the scores of a block decide whether its values are read at all;
// the cache format is E4M3 codes with one fp32 scale per (sequence, KV head)
// for keys and for values (the page evaluates FP8/NVFP4 models and names no
// cache format; this is the plainest one).  Decode is bound by the cache
// bytes, so halving them should halve the time -- provided the per-block work
// on the chip keeps up with half the bytes.
//
// Transposed products.  One CTA per (sequence, KV head, split).  The block's
// 128 keys are the MMA rows and the G <= 8 query heads sharing the KV head
// the columns (N = 16, padded):
//   S^T = K_j Q^T   kind::f8f6f4, A = the E4M3 key tile straight from TMA,
//                   B = the query as an exact E4M3 pair (below) stacked as
//                   32 rows (hi heads, then lo heads), 4 k-steps; the score
//                   threads add the two parts;
//   O^T += V_j^T P^T  kind::f16, A = the fp16 value tile (MN-major: d is the
//                   contiguous dimension), B = P^T (fp16, heads x keys).
// So every thread of the four score warps owns one key of the block and its G
// scores: a block costs G exponentials per thread for a kept block and one
// cross-warp reduction of G maxima per block, spread over all four SMSPs,
// and the tensor core computes 16 columns instead of 128 padded rows.
//
// The query: per head, q 2^e (the largest power of two keeping the row within
// 256) = hi + lo with hi = E4M3(q 2^e) and lo = E4M3(q 2^e - hi), exact for a
// bf16 row except for elements below about 2^-10 of its largest; S = hi K^T +
// lo K^T and 2^-e goes into the head's score scale with the key scale.  P is
// no E4M3 quantity (its small weights would vanish), so value tiles are
// widened, exactly, to fp16 by converter warps (the fp16 pattern of code x
// 2^-8; 2^8 goes into the value scale).
//
// Warp roles (512 threads):
//   warps 0-3   scores: thread = key 32w + lane of the block (TMEM lane);
//               maxima, votes, decision, exponentials, P^T, row sums, O^T
//               rescale, epilogue (thread = value dimension d);
//   warp 4      TMA producer of the E4M3 key tiles (every block; three stages
//               of two tiles);
//   warp 5      S^T issuer (allocates TMEM);
//   warp 6      TMA producer of the E4M3 value tiles of kept blocks;
//   warp 7      O^T issuer;
//   warps 8-15  value converters (follow the decisions).
// The decision ring holds 32 decisions and there are three P^T buffers, so
// the score warps run ahead of the value loads and their widening by up to
// three kept blocks; the value pipeline (load, widen, product) drains behind
// them.  Six key tiles (96 KB) keep enough bytes in flight to cover the load
// latency under a full GPU's traffic (~2.8 us measured); three E4M3 value
// stages give a kept block's value load the same lead when most blocks are
// kept.
// TMEM columns: S^T buffers [0,128) (32 each: the hi part, then the lo part), O^T
// [128,144).
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
constexpr int BC = 128;   // keys per block (MMA rows of S^T)
constexpr int NQ = 16;    // MMA columns: query heads, padded
constexpr int NKP = 3;    // E4M3 key stages of two blocks each (one barrier per pair)
constexpr int NVF = 3;    // E4M3 value stages
constexpr int NVH = 2;    // fp16 value stages
constexpr int NS = 4;     // TMEM S^T buffers (two pairs)
constexpr int NPT = 3;    // P^T buffers
constexpr int NDP = 16;   // decision ring, in block pairs
constexpr int NT = 16 * 32;
constexpr int WARP_K = 4, WARP_QK = 5, WARP_V = 6, WARP_PV = 7, WARP_VC = 8;  // 0-3: scores
constexpr int NVC = 8 * 32;                                                 // converter threads
constexpr uint32_t F8_BYTES = BC * D;         // 16 KB: 128 rows x 128 codes
constexpr uint32_t H_BYTES = BC * D * 2;      // 32 KB: 128 keys x 128 fp16
constexpr uint32_t HALF_BYTES = H_BYTES / 2;  // one 64-column swizzled box
constexpr uint32_t QT_BYTES = NQ * 128;       // 2 KB: 16 rows x 128 codes
constexpr uint32_t PT_BOX = NQ * 128;         // 2 KB: 16 heads x 64 fp16 keys
constexpr uint32_t SMEM_KF = 0;
constexpr uint32_t SMEM_VF = SMEM_KF + NKP * 2 * F8_BYTES;
constexpr uint32_t SMEM_VH = SMEM_VF + NVF * F8_BYTES;
constexpr uint32_t SMEM_Q = SMEM_VH + NVH * H_BYTES;  // Q hi, then Q lo
constexpr uint32_t SMEM_PT = SMEM_Q + 2 * QT_BYTES;   // NPT x two 64-key boxes
constexpr uint32_t SMEM_TILES = SMEM_PT + NPT * 2 * PT_BOX;  // 224 KB
// An S^T buffer holds K Q_hi^T in its first NQ columns and K Q_lo^T in the
// next NQ: one N = 2 NQ product per k-step instead of one per part.
constexpr int NSC = 2 * NQ;
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t TMEM_O = NS * NSC;  // 128
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // exp reference may lag the max by 2^8
// S^T: E4M3 x E4M3, both K-major.  O^T: fp16, A (V^T) MN-major, B (P^T) K-major.
constexpr uint32_t IDESC_QK = idesc_e4m3_f32(BC, NSC);
constexpr uint32_t IDESC_PV = idesc_f16_f32(D, NQ, 0) | (1u << 15);
static_assert(TMEM_O + NQ <= TMEM_COLS, "TMEM budget");
static_assert(NS == 4, "two pair buffers of two adjacent S^T buffers");
static_assert(NT >= NQ * 16, "16 threads per query row write the query pair");

struct Shared {
  uint64_t kf_full[NKP], kf_empty[NKP];
  uint64_t vf_full[NVF], vf_empty[NVF];
  uint64_t vh_full[NVH], vh_empty[NVH];
  uint64_t s_full[2], s_free[2];  // per pair buffer
  uint64_t p_full[NPT], p_free[NPT];
  uint64_t dec_full[NDP], dec_empty[NDP];
  uint64_t red_full[2];  // the four score warps' partial maxima of a block pair are in
  uint64_t l_full;       // the four score warps' row sums are in
  int dec[NDP][2];
  float red[2][4][16];  // per block pair (double buffered): per score warp, per head max
  float lsum[4][8];    // epilogue: per score warp, per head row sum
  float sl2[NQ];       // per head: raw score -> log2 units
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t SMEM_ALLOC = SMEM_TILES + ((sizeof(Shared) + 127) / 128) * 128;
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");

// K-major E4M3 / fp16 operands with 128-byte rows: one 128-byte-swizzled box,
// 8-row groups 1024 bytes apart; a k-step of 32 bytes (32 codes, 16 fp16).
__device__ __forceinline__ uint64_t kmajor_base(uint32_t tile) {
  return smem_desc_sw128(tile, 16u, 1024u);
}
// P^T (16 heads x 128 fp16 keys) as K-major B: k-step kk (16 keys) is box kk/4
// at 32-byte step kk%4.
__device__ __forceinline__ constexpr uint64_t pt_step(int kk) {
  return (uint64_t)(((uint32_t)(kk >> 2) * PT_BOX + (uint32_t)(kk & 3) * 32u) >> 4);
}
// fp16 value tile (rows are keys, two 128-byte-swizzled boxes of 64 d values)
// as the MN-major A operand V^T: the second 64-d half 16 KB further (LBO),
// 8-key groups 1024 bytes apart (SBO); k-step kk (16 keys) 2048 bytes further.
__device__ __forceinline__ uint64_t vmajor_base(uint32_t tile) {
  return smem_desc_sw128(tile, HALF_BYTES, 1024u);
}
__device__ __forceinline__ constexpr uint64_t vmajor_step(int kk) {
  return (uint64_t)(((uint32_t)kk * 2048u) >> 4);
}

// Maximum over the 32 lanes of the warp (one instruction on sm_100 family).
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// 32 lanes x 16 consecutive 32-bit columns (S^T or O^T rows of this warp's
// lane quarter): thread i receives the 16 columns of its lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
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

// The query pair into the two E4M3 query tiles (16 rows of 128 codes,
// 128-byte-swizzled), by threads 0-255: thread t takes row r = t / 16 (query
// head hk*G + r, zero for r >= G) and its 16-byte chunk t % 16 of bf16
// values, so the whole query is read in one round of coalesced loads.  Per
// row: e = 8 - ceil(log2 max|q|) (the largest power of two with max|q| 2^e <=
// 256), hi = E4M3(q 2^e), lo = E4M3(q 2^e - hi), both nearest even; sl2[r] =
// the row's score scale (scale * key scale * log2 e * 2^-e).
__device__ __forceinline__ void write_query_pair(const DecodeArgs &a, int b, int hk, int G, int zkv,
                                                 int t, uint32_t q_hi, uint32_t q_lo,
                                                 float *sl2) {
  const int r = t >> 4, c16 = t & 15;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (r < G)
    v = __ldg(reinterpret_cast<const uint4 *>((const __nv_bfloat16 *)a.q +
                                              (size_t)(b * a.Hq + hk * G + r) * D) + c16);
  const uint32_t pr[4] = {v.x, v.y, v.z, v.w};  // bf16 pairs, low element first
  uint32_t amax_bits = 0;  // |bf16| bit patterns order like their values
#pragma unroll
  for (int i = 0; i < 4; ++i)
    amax_bits = max(amax_bits, max(pr[i] & 0x7fffu, (pr[i] >> 16) & 0x7fffu));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1)  // the 16 threads of the row
    amax_bits = max(amax_bits, __shfl_xor_sync(0xffffffffu, amax_bits, o));
  const float amax = __uint_as_float(amax_bits << 16);
  int ex = 0;
  const float fr = frexpf(amax > 0.f ? amax : 1.f, &ex);  // amax = fr * 2^ex
  const int qexp = amax > 0.f ? 8 - (fr == 0.5f ? ex - 1 : ex) : 0;  // 8 - ceil(log2 amax)
  uint32_t hi[2], lo[2];
#pragma unroll
  for (int w = 0; w < 2; ++w) {
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
  const uint32_t off = (uint32_t)r * 128u + ((((uint32_t)c16 >> 1) ^ (uint32_t)(r & 7)) << 4) +
                       ((uint32_t)c16 & 1u) * 8u;
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(q_hi + off), "r"(hi[0]), "r"(hi[1])
               : "memory");
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(q_lo + off), "r"(lo[0]), "r"(lo[1])
               : "memory");
  if (c16 == 0) sl2[r] = ldexpf(a.scale * __ldg(a.k_scale + zkv) * kLog2e, -qexp);
}

template <int G>
__global__ void __launch_bounds__(NT, 1)
    decode_fp8_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Shared &sh = *reinterpret_cast<Shared *>(smem_raw + SMEM_TILES);
  const uint32_t base = smem_u32(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (base & 1023u) {  // the swizzled layouts need a 1024-byte aligned base
    if (tid == 0) atomicOr(a.err, kErrLayout);
    return;
  }
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

  // The query pair and each head's score scale; the P^T rows of the padding
  // heads are zeroed once.
  if (tid < NQ * 16)
    write_query_pair(a, b, hk, G, zkv, tid, base + SMEM_Q, base + SMEM_Q + QT_BYTES, sh.sl2);
  for (int idx = tid; idx < NPT * 2 * (NQ - 8) * 8; idx += NT) {  // rows 8..15, 16-byte chunks
    const int c = idx & 7, r = 8 + ((idx >> 3) & 7), box = idx >> 6;
    st_shared_v4(base + SMEM_PT + box * PT_BOX + r * 128 + c * 16, 0u, 0u, 0u, 0u);
  }
  if constexpr (G < 8) {
    for (int idx = tid; idx < NPT * 2 * (8 - G) * 8; idx += NT) {  // rows G..7
      const int c = idx & 7, r = G + (idx >> 3) % (8 - G), box = (idx >> 3) / (8 - G);
      st_shared_v4(base + SMEM_PT + box * PT_BOX + r * 128 + c * 16, 0u, 0u, 0u, 0u);
    }
  }
  fence_proxy_async_smem();  // visible to the tensor core
  if (tid == 0) {
    for (int i = 0; i < NKP; ++i) {
      mbar_init(smem_u32(&sh.kf_full[i]), 1);
      mbar_init(smem_u32(&sh.kf_empty[i]), 1);  // the S^T commit of the pair
    }
    for (int i = 0; i < NVF; ++i) {
      mbar_init(smem_u32(&sh.vf_full[i]), 1);
      mbar_init(smem_u32(&sh.vf_empty[i]), 8);  // the eight value converters
    }
    for (int i = 0; i < NVH; ++i) {
      mbar_init(smem_u32(&sh.vh_full[i]), 8);
      mbar_init(smem_u32(&sh.vh_empty[i]), 1);  // the O^T commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh.s_full[i]), 1);
      mbar_init(smem_u32(&sh.s_free[i]), 4);  // the four score warps
    }
    for (int i = 0; i < NPT; ++i) {
      mbar_init(smem_u32(&sh.p_full[i]), 4);  // the four score warps
      mbar_init(smem_u32(&sh.p_free[i]), 1);  // the O^T commit
    }
    for (int i = 0; i < NDP; ++i) {
      mbar_init(smem_u32(&sh.dec_full[i]), 1);
      // readers: the value producer, the O^T issuer, the eight value converters
      mbar_init(smem_u32(&sh.dec_empty[i]), 10);
    }
    mbar_init(smem_u32(&sh.red_full[0]), 4);
    mbar_init(smem_u32(&sh.red_full[1]), 4);
    mbar_init(smem_u32(&sh.l_full), 4);
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
      // Blocks in pairs: one stage (two tiles) and one barrier per pair.
      const int npair = (nb + 1) / 2;
      int issued = 0;
      for (int q = 0; q < npair && !*abort; ++q) {
        const int f = q % NKP;
        const int n = 2 * q + 1 < nb ? 2 : 1;
        if (q >= NKP &&
            !mbar_wait(smem_u32(&sh.kf_empty[f]), ((q / NKP) - 1) & 1, abort, a.err, kErrTimeout))
          break;
        mbar_expect_tx(smem_u32(&sh.kf_full[f]), n * F8_BYTES);
        for (int t = 0; t < n; ++t)
          tma_load_3d(base + SMEM_KF + (2 * f + t) * F8_BYTES, &tm_k, smem_u32(&sh.kf_full[f]), 0,
                      (j0 + 2 * q + t) * BC, zkv, pol);
        ++issued;
      }
      for (int f = 0; f < NKP && f < issued; ++f) {
        const int last = f + ((issued - 1 - f) / NKP) * NKP;
        mbar_wait_drain(smem_u32(&sh.kf_full[f]), (last / NKP) & 1);
      }
    }
  } else if (warp == WARP_V) {
    // ----------------------------------------------- E4M3 value producer --
    if (lane == 0) {
      prefetch_tmap(&tm_v);
      const uint64_t pol = policy_evict_first();
      int vi = 0;
      for (int j = 0; j < nb && !*abort; ++j) {
        const int q = j >> 1, ds = q % NDP;
        if (!(j & 1) && !mbar_wait(smem_u32(&sh.dec_full[ds]), (q / NDP) & 1, abort, a.err,
                                   kErrTimeout))
          break;
        const int keep = sh.dec[ds][j & 1];
        if ((j & 1) || j == nb - 1) mbar_arrive(smem_u32(&sh.dec_empty[ds]));  // pair read
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
    // Follow the decisions; chunks t, t + 256, ... (row = chunk / 8) of every
    // kept value tile.
    const int t0 = (warp - WARP_VC) * 32 + lane;
    int vi = 0;
    for (int j = 0; j < nb; ++j) {
      const int q = j >> 1, ds = q % NDP;
      if (!(j & 1) && !mbar_wait_warp(smem_u32(&sh.dec_full[ds]), (q / NDP) & 1, abort, a.err,
                                      kErrTimeout))
        break;
      const int keep = sh.dec[ds][j & 1];
      __syncwarp();
      if (lane == 0 && ((j & 1) || j == nb - 1)) mbar_arrive(smem_u32(&sh.dec_empty[ds]));
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
    // --------------------------------------------------------- S^T issuer --
    if (lane == 0) {
      // The query pair as one 32-row operand: hi in rows 0-15, lo in rows 16-31
      // (the two 2 KB tiles are adjacent, 8-row groups 1 KB apart).
      const uint64_t qd = kmajor_base(base + SMEM_Q);
      // Blocks in pairs: one key barrier, one S^T buffer barrier and two
      // commits per pair (a barrier wait between products costs about as
      // much as a product).
      const int npair = (nb + 1) / 2;
      for (int q = 0; q < npair; ++q) {
        const int f = q % NKP, pb = q & 1;
        const int n = 2 * q + 1 < nb ? 2 : 1;
        if (!mbar_wait(smem_u32(&sh.kf_full[f]), (q / NKP) & 1, abort, a.err, kErrTimeout))
          break;
        // Pair buffer pb is free once the score warps have read pair q - 2.
        if (q >= 2 && !mbar_wait(smem_u32(&sh.s_free[pb]), ((q >> 1) - 1) & 1, abort, a.err,
                                 kErrTimeout))
          break;
        fence_after_sync();
        for (int t = 0; t < n; ++t) {
          const uint64_t kd = kmajor_base(base + SMEM_KF + (2 * f + t) * F8_BYTES);
          // [K hi^T | K lo^T]: four k-steps of 32 codes; the score threads add
          // the two parts.
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8f6f4_ss(tmem + (2 * pb + t) * NSC, kd + ((uint64_t)kk * 2), qd + ((uint64_t)kk * 2),
                          IDESC_QK, kk > 0);
        }
        mma_commit(smem_u32(&sh.s_full[pb]));
        mma_commit(smem_u32(&sh.kf_empty[f]));
      }
    }
  } else if (warp == WARP_PV) {
    // --------------------------------------------------------- O^T issuer --
    if (lane == 0) {
      int kc = 0;
      for (int j = 0; j < nb && !*abort; ++j) {
        const int q = j >> 1, ds = q % NDP;
        if (!(j & 1) && !mbar_wait(smem_u32(&sh.dec_full[ds]), (q / NDP) & 1, abort, a.err,
                                   kErrTimeout))
          break;
        const int keep = sh.dec[ds][j & 1];
        if ((j & 1) || j == nb - 1) mbar_arrive(smem_u32(&sh.dec_empty[ds]));  // pair read
        if (!keep) continue;
        const int pb = kc % NPT, hs = kc % NVH;
        if (!mbar_wait(smem_u32(&sh.p_full[pb]), (kc / NPT) & 1, abort, a.err, kErrTimeout) ||
            !mbar_wait(smem_u32(&sh.vh_full[hs]), (kc / NVH) & 1, abort, a.err, kErrTimeout))
          break;
        fence_after_sync();
        const uint64_t vd = vmajor_base(base + SMEM_VH + hs * H_BYTES);
        const uint64_t pd = kmajor_base(base + SMEM_PT + pb * 2 * PT_BOX);
#pragma unroll
        for (int kk = 0; kk < BC / 16; ++kk)
          mma_bf16_ss(tmem + TMEM_O, vd + vmajor_step(kk), pd + pt_step(kk), IDESC_PV,
                      (kc > 0 || kk > 0) ? 1u : 0u);
        mma_commit(smem_u32(&sh.vh_empty[hs]));
        mma_commit(smem_u32(&sh.p_free[pb]));
        ++kc;
      }
    }
  } else {
    // ------------------------------------------------------------- scores --
    // Thread = key kidx of the block (TMEM lane of S^T); G scores per thread.
    // Every thread computes the same maxima, decisions and references from
    // the four warps' partial maxima, so the warps stay in step.
    const int kidx = warp * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    uint32_t *bits = a.bits + (size_t)unit * a.words;
    const float c2 = a.ln_lambda * kLog2e;  // ln(lambda), log2 units
    float sl2[G], m2[G], mref[G], l[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      sl2[g] = sh.sl2[g];
      m2[g] = -INFINITY;
      mref[g] = -INFINITY;
      l[g] = 0.f;
    }
    int kc = 0;
    uint32_t word = 0;
    bool ok = true;
    // Kept block: exponent references (rescaled lazily, as in the other
    // kernels), this key's P for every head into the next P^T buffer, the
    // per-thread row sums, an O^T rescale when a reference moved.
    auto kept = [&](const float (&s)[G], const float (&mnew)[G]) -> bool {
      bool rescale = false;
      float alpha[G], p[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        alpha[g] = 1.f;
        if (mref[g] == -INFINITY) {
          mref[g] = mnew[g];
        } else if (mnew[g] > mref[g] + kRescaleLog2) {
          alpha[g] = ex2(mref[g] - mnew[g]);
          mref[g] = mnew[g];
          rescale = true;
        }
        p[g] = ex2(s[g] - mref[g]);
        l[g] = l[g] * alpha[g] + p[g];
      }
      const int pb = kc % NPT;
      // P^T buffer pb last fed the O^T product of kept block kc - NPT.
      if (kc >= NPT && !mbar_wait_warp(smem_u32(&sh.p_free[pb]), ((kc / NPT) - 1) & 1, abort,
                                       a.err, kErrTimeout))
        return false;
      {
        // P^T[g][kidx] (fp16): box kidx / 64, row g, 16-byte chunk (kidx % 64) / 8
        // at chunk position chunk ^ (g % 8).
        const uint32_t box = base + SMEM_PT + (uint32_t)(pb * 2 + (kidx >> 6)) * PT_BOX;
        const uint32_t kk = (uint32_t)(kidx & 63);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const uint32_t addr = box + (uint32_t)g * 128u + ((((kk >> 3) ^ (uint32_t)g)) << 4) +
                                (kk & 7u) * 2u;
          const unsigned short hv = __half_as_ushort(__float2half_rn(p[g]));
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(hv) : "memory");
        }
      }
      // O^T rescale (columns g of this warp's lanes) once the previous product
      // has landed (its commit to the P^T buffer it read; the score warps may be
      // several kept blocks ahead, so a two-slot completion ring could alias);
      // the same decision in every thread.
      if (rescale && kc >= 1) {
        if (!mbar_wait_warp(smem_u32(&sh.p_free[(kc - 1) % NPT]), ((kc - 1) / NPT) & 1, abort,
                            a.err, kErrTimeout))
          return false;
        fence_after_sync();
        uint32_t o[16];
        tmem_ld16(lane_base + TMEM_O, o);
#pragma unroll
        for (int g = 0; g < G; ++g) o[g] = __float_as_uint(__uint_as_float(o[g]) * alpha[g]);
        tmem_st16(lane_base + TMEM_O, o);
        tmem_wait_st();
      }
      fence_proxy_async_smem();  // P^T is visible to the tensor core
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.p_full[pb]));
      ++kc;
      return true;
    };
    // Decisions of pair q (thread 0): published to the value pipeline together
    // (one barrier per pair); bitmap.
    auto publish = [&](int q, bool skip0, bool skip1, bool two) {
      const int ds = q % NDP;
      // On a timeout the abort flag is raised and every later wait fails.
      if (q < NDP || mbar_wait(smem_u32(&sh.dec_empty[ds]), ((q / NDP) - 1) & 1, abort, a.err,
                               kErrTimeout)) {
        sh.dec[ds][0] = skip0 ? 0 : 1;
        sh.dec[ds][1] = skip1 ? 0 : 1;
        mbar_arrive(smem_u32(&sh.dec_full[ds]));
      }
      for (int t = 0; t < (two ? 2 : 1); ++t) {
        const int jj = 2 * q + t;
        if (t ? skip1 : skip0) word |= 1u << (jj & 31);
        if ((jj & 31) == 31 || jj == nb - 1) {
          bits[jj >> 5] = word;
          word = 0;
        }
      }
    };
    // Blocks in pairs: both S^T buffers read at once (j even, so they are
    // adjacent), both blocks' partial maxima exchanged in one round.
    for (int j = 0; j < nb; j += 2) {
      const bool two = j + 1 < nb;
      const int q = j >> 1;  // pair index
      const int pb = q & 1, sb = 2 * pb;
      if (!mbar_wait_warp(smem_u32(&sh.s_full[pb]), (q >> 1) & 1, abort, a.err, kErrTimeout)) {
        ok = false;
        break;
      }
      fence_after_sync();
      uint32_t x[32], y[32];
      tmem_ld32(lane_base + sb * NSC, x);        // block j: hi part [0,16), lo part [16,32)
      tmem_ld32(lane_base + (sb + 1) * NSC, y);  // block j + 1 (unused when there is none)
      tmem_wait_ld_regs(x);
      tmem_wait_ld_regs(y);
      fence_before_sync();  // the scores are in registers: the S^T buffers are free
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.s_free[pb]));
      const bool v0 = (j0 + j) * BC + kidx < a.L;
      const bool v1 = two && (j0 + j + 1) * BC + kidx < a.L;
      float s0[G], s1[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        s0[g] = v0 ? (__uint_as_float(x[g]) + __uint_as_float(x[16 + g])) * sl2[g] : -INFINITY;
        s1[g] = v1 ? (__uint_as_float(y[g]) + __uint_as_float(y[16 + g])) * sl2[g] : -INFINITY;
        const float m0 = warp_max(s0[g]), m1 = warp_max(s1[g]);
        if (lane == 0) {
          sh.red[q & 1][warp][g] = m0;
          sh.red[q & 1][warp][8 + g] = m1;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.red_full[q & 1]));
      if (!mbar_wait_warp(smem_u32(&sh.red_full[q & 1]), (q >> 1) & 1, abort, a.err,
                          kErrTimeout)) {
        ok = false;
        break;
      }
      // Block maxima per head; with c < 0, "rowmax - m_new < c" is "rowmax -
      // m_old < c" (a block that raises the max fails both).  Every head must
      // vote skip.  Block j + 1 is tested against the max after block j.
      bool skip0 = true, skip1 = true;
      float mn0[G], mn1[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float b0 = fmaxf(fmaxf(sh.red[q & 1][0][g], sh.red[q & 1][1][g]),
                               fmaxf(sh.red[q & 1][2][g], sh.red[q & 1][3][g]));
        const float d0 = (b0 == -INFINITY) ? -INFINITY : b0 - m2[g];
        skip0 = skip0 && (d0 < c2);
        mn0[g] = fmaxf(m2[g], b0);
        const float b1 = fmaxf(fmaxf(sh.red[q & 1][0][8 + g], sh.red[q & 1][1][8 + g]),
                               fmaxf(sh.red[q & 1][2][8 + g], sh.red[q & 1][3][8 + g]));
        const float d1 = (b1 == -INFINITY) ? -INFINITY : b1 - mn0[g];
        skip1 = skip1 && (d1 < c2);
        mn1[g] = fmaxf(mn0[g], b1);
        m2[g] = two ? mn1[g] : mn0[g];  // the running max advances on every block
      }
      if (tid == 0) publish(q, skip0, skip1, two);
      if (!skip0 && !kept(s0, mn0)) {
        ok = false;
        break;
      }
      if (two && !skip1 && !kept(s1, mn1)) {
        ok = false;
        break;
      }
    }

    // ---- epilogue: O_s = v_scale * O / l and LSE_s = ref + ln l per head ----
    if (tid == 0)
      for (int w = ((nb - 1) >> 5) + 1; w < a.words; ++w) bits[w] = 0u;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float v = l[g];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) sh.lsum[warp][g] = v;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh.l_full));
    if (ok) ok = mbar_wait_warp(smem_u32(&sh.l_full), 0, abort, a.err, kErrTimeout);
    if (ok && kc > 0)  // the last product has landed
      ok = mbar_wait_warp(smem_u32(&sh.p_free[(kc - 1) % NPT]), ((kc - 1) / NPT) & 1, abort,
                          a.err, kErrTimeout);
    if (ok) {
      fence_after_sync();
      uint32_t o[16];
      tmem_ld16(lane_base + TMEM_O, o);  // thread = value dimension d = kidx
      const float vs = __ldg(a.v_scale + zkv) * 256.f;  // values were widened times 2^-8
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float lt = (sh.lsum[0][g] + sh.lsum[1][g]) + (sh.lsum[2][g] + sh.lsum[3][g]);
        const size_t row = (size_t)(b * a.Hq + hk * G + g) * a.n_splits + sp;
        a.o_part[row * D + kidx] = __uint_as_float(o[g]) * (vs / lt);
        if (tid == 0) a.lse_part[row] = mref[g] * kLn2 + logf(lt);
      }
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
  const int G = a.Hq / a.Hkv;
  auto kernel = G == 1   ? decode_fp8_kernel<1>
                : G == 2 ? decode_fp8_kernel<2>
                : G == 4 ? decode_fp8_kernel<4>
                : G == 8 ? decode_fp8_kernel<8>
                         : nullptr;
  if (!kernel) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  const long units = (long)a.B * a.Hkv * a.n_splits;
  kernel<<<(unsigned)units, NT, SMEM_ALLOC, s>>>(mk, mv, a);
  return cudaGetLastError();
}

}  // namespace attn_skip
