// Split-KV decode with softmax-threshold block skipping over an NVFP4
// key/value cache (d = 128, Bc = 128), on the tensor cores.
//
// Method: the BLASST page, sections "BLASST 的判定准则" (Eq. 5) and "Decode 内核：
// 砍带宽": the scores of a block decide whether its values are read at all.
// The cache format (the page evaluates NVFP4-quantised models and names no
// format): E2M1 codes two per byte (element 2i in the low nibble), one E4M3
// scale per 16 consecutive elements of a row, one fp32 scale per (sequence,
// KV head) for keys and one for values; a row element is
// head scale * E4M3(block scale) * E2M1(code).  A 128-key block is 8 KB of
// codes and 1 KB of block scales: a quarter of the bf16 cache's bytes.
//
// The block scales vary along the contracted dimension, so no E2M1 product
// can take them; both caches are widened, exactly, to fp16 on the chip: an
// E2M1 value has two significant bits and an E4M3 scale four, so their
// product (|x| in [2^-10, 2688]) is an fp16 normal number.  Keys go straight
// into TMEM (no shared-memory round trip), values into a shared-memory tile.
//
// Transposed products, one CTA per (sequence, KV head, split):
//   S^T = K_j Q^T     kind::f16, A = the widened key tile read from TMEM
//                     (the block's 128 keys are the MMA rows, lane = key),
//                     B = the query as fp16 after a power-of-two per-head
//                     scale 2^e (max|q| 2^e <= 2^15), exact for every bf16
//                     element not below ~2^-31 of the head's largest;
//   O^T += V_j^T P^T  kind::f16, A = the widened value tile (MN-major),
//                     B = P^T (fp16, heads x keys).
// Every thread of the four score warps owns one key of the block and its G
// scores, as in the E4M3-cache kernel.
//
// Warp roles (512 threads):
//   warps 0-3   scores: thread = key 32w + lane; maxima, votes, decision,
//               exponentials, P^T, row sums, O^T rescale, epilogue;
//   warp 4      key producer: TMA of the code tile (64-byte swizzle), the
//               block scales by cp.async from all 32 lanes;
//   warp 5      S^T issuer (allocates TMEM);
//   warp 6      value producer (kept blocks only), as warp 4;
//   warp 7      O^T issuer;
//   warps 8-11  key wideners: warp 8 + q owns TMEM lane quarter q, thread =
//               key row; codes and scales -> 64 columns of fp16 pairs;
//   warps 12-15 value wideners (follow the decisions).
// TMEM columns: widened key tiles [0,256) (64 each), S^T buffers [256,320)
// (16 each), O^T [320,336).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "internal.h"
#include "tc_common.cuh"

namespace attn_skip {
namespace {

using namespace tc;

constexpr int D = 128;    // head size (keys and values)
constexpr int BC = 128;   // keys per block (MMA rows of S^T)
constexpr int NQ = 16;    // MMA columns: query heads, padded
constexpr int NKF = 12;   // key code stages in shared memory (NKF / 2 block pairs)
constexpr int NKT = 4;    // widened key tiles in TMEM (NKT / 2 block pairs)
constexpr int NVF = 3;    // value code stages
constexpr int NVH = 2;    // widened (fp16) value tiles
constexpr int NS = 4;     // TMEM S^T buffers
constexpr int NPT = 3;    // P^T buffers
constexpr int NDP = 16;   // decision ring, in block pairs
constexpr int NT = 16 * 32;
constexpr int WARP_K = 4, WARP_QK = 5, WARP_V = 6, WARP_PV = 7, WARP_KW = 8, WARP_VW = 12;
constexpr int NVW = 4 * 32;                  // value widener threads
constexpr uint32_t CODE_ROW = D / 2;         // 64 bytes of codes per row
constexpr uint32_t SC_ROW = D / 16;          // 8 block scales per row
constexpr uint32_t CODE_BYTES = BC * CODE_ROW;  // 8 KB
constexpr uint32_t SC_BYTES = BC * SC_ROW;      // 1 KB
constexpr uint32_t H_BYTES = BC * D * 2;        // 32 KB: 128 keys x 128 fp16
constexpr uint32_t HALF_BYTES = H_BYTES / 2;    // one 64-column swizzled box
constexpr uint32_t QBOX = NQ * 128;             // 2 KB: 16 heads x 64 fp16
constexpr uint32_t SMEM_KC = 0;
constexpr uint32_t SMEM_VC = SMEM_KC + NKF * CODE_BYTES;
constexpr uint32_t SMEM_VH = SMEM_VC + NVF * CODE_BYTES;
constexpr uint32_t SMEM_KS = SMEM_VH + NVH * H_BYTES;
constexpr uint32_t SMEM_VS = SMEM_KS + NKF * SC_BYTES;
constexpr uint32_t SMEM_Q = SMEM_VS + NVF * SC_BYTES;  // two boxes
constexpr uint32_t SMEM_PT = SMEM_Q + 2 * QBOX;        // NPT x two 64-key boxes
constexpr uint32_t SMEM_TILES = SMEM_PT + NPT * 2 * QBOX;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_K = 0;                 // NKT x 64 columns
constexpr uint32_t TMEM_S = TMEM_K + NKT * 64; // NS x NQ columns
constexpr uint32_t TMEM_O = TMEM_S + NS * NQ;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // exp reference may lag the max by 2^8
// S^T: fp16, A (keys) from TMEM, B (query) K-major.  O^T: fp16, A (V^T)
// MN-major, B (P^T) K-major.
constexpr uint32_t IDESC_QK = idesc_f16_f32(BC, NQ, 0);
constexpr uint32_t IDESC_PV = idesc_f16_f32(D, NQ, 0) | (1u << 15);
static_assert(TMEM_O + NQ <= TMEM_COLS, "TMEM budget");
static_assert(NS == 4 && NKF % 2 == 0 && NKT % 2 == 0, "stages and buffers in block pairs");
static_assert(NT >= NQ * 16, "16 threads per query row write the query");
static_assert(SMEM_KC % 1024 == 0 && SMEM_VC % 1024 == 0 && SMEM_VH % 1024 == 0 &&
                  SMEM_Q % 1024 == 0 && SMEM_PT % 1024 == 0,
              "swizzled tiles on 1024-byte boundaries");

struct Shared {
  uint64_t kc_full[NKF / 2], kc_empty[NKF / 2];  // per pair stage
  uint64_t kt_full[NKT / 2], kt_empty[NKT / 2];  // per pair of TMEM tiles
  uint64_t vc_full[NVF], vc_empty[NVF];
  uint64_t vh_full[NVH], vh_empty[NVH];
  uint64_t s_full[2], s_free[2];  // per pair buffer
  uint64_t p_full[NPT], p_free[NPT];
  uint64_t dec_full[NDP], dec_empty[NDP];
  uint64_t red_full[2];  // the four score warps' partial maxima of a block pair are in
  uint64_t l_full;       // the four score warps' row sums are in
  int dec[NDP][2];
  float red[2][4][16];  // per block pair (double buffered): per score warp, per head max
  float lsum[4][8];     // epilogue: per score warp, per head row sum
  float sl2[NQ];        // per head: raw score -> log2 units
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t SMEM_ALLOC = SMEM_TILES + ((sizeof(Shared) + 127) / 128) * 128;
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");

// K-major fp16 operand with 128-byte rows of 64 elements (the query, P^T):
// two 128-byte-swizzled boxes of 16 rows, 8-row groups 1024 bytes apart;
// k-step kk (16 elements) is box kk / 4 at 32-byte step kk % 4.
__device__ __forceinline__ uint64_t kmajor_base(uint32_t tile) {
  return smem_desc_sw128(tile, 16u, 1024u);
}
__device__ __forceinline__ constexpr uint64_t box_step(int kk) {
  return (uint64_t)(((uint32_t)(kk >> 2) * QBOX + (uint32_t)(kk & 3) * 32u) >> 4);
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

__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

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

// 8-byte copy global -> shared through the L1-bypassing path; src_bytes = 0
// writes zeros and reads nothing.  Both addresses 8-byte aligned.
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
// Arrive on `bar` once this thread's earlier cp.async copies have landed
// (the arrival is one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Four E2M1 pairs (the bytes of w, element 2i in the low nibble) -> four fp16
// pairs (element 2i in the low half), each times the fp16 pair `s2`.
__device__ __forceinline__ void e2m1x8_scaled(uint32_t w, uint32_t s2, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t"
      "mul.rn.f16x2 %0, %0, %5;\n\t"
      "mul.rn.f16x2 %1, %1, %5;\n\t"
      "mul.rn.f16x2 %2, %2, %5;\n\t"
      "mul.rn.f16x2 %3, %3, %5;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w), "r"(s2));
}

// E4M3 block scale (byte `i` of the pair (lo, hi)) -> the fp16 pair (s, s).
__device__ __forceinline__ uint32_t e4m3_scale2(uint32_t lo, uint32_t hi, int i) {
  const uint32_t byte = ((i < 4 ? lo : hi) >> (8 * (i & 3))) & 0xffu;
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((unsigned short)(byte | (byte << 8))));
  return r;
}

// Code chunk c (bytes 16c..16c+15: elements 32c..32c+31) of row r of a code
// tile (64-byte rows, 64-byte swizzle: chunk c at chunk position
// c ^ ((r / 2) % 4)).
__device__ __forceinline__ uint4 ld_code_chunk(uint32_t tile, int r, int c) {
  uint4 x;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
               : "r"(tile + (uint32_t)r * CODE_ROW +
                     (((uint32_t)c ^ (((uint32_t)r >> 1) & 3u)) << 4)));
  return x;
}

// Widen value chunk t of a kept block: row r = t / 4, code chunk c = t % 4
// (32 elements, block scales 2c and 2c + 1) -> 64 bytes of the fp16 tile
// (box c / 2, 16-byte chunks 4 (c % 2) .. + 3 of the row, at chunk position
// chunk ^ (r % 8)).
__device__ __forceinline__ void widen_value_chunk(uint32_t codes, uint32_t scales,
                                                  uint32_t dst_tile, int t) {
  const int r = t >> 2, c = t & 3;
  const uint4 x = ld_code_chunk(codes, r, c);
  uint32_t sc;
  asm volatile("ld.shared.u16 %0, [%1];"
               : "=r"(sc)
               : "r"(scales + (uint32_t)r * SC_ROW + 2u * (uint32_t)c));
  const uint32_t s0 = e4m3_scale2(sc & 0xffu, 0u, 0);
  const uint32_t s1 = e4m3_scale2((sc >> 8) & 0xffu, 0u, 0);
  uint32_t h[16];
  e2m1x8_scaled(x.x, s0, *reinterpret_cast<uint32_t(*)[4]>(&h[0]));
  e2m1x8_scaled(x.y, s0, *reinterpret_cast<uint32_t(*)[4]>(&h[4]));
  e2m1x8_scaled(x.z, s1, *reinterpret_cast<uint32_t(*)[4]>(&h[8]));
  e2m1x8_scaled(x.w, s1, *reinterpret_cast<uint32_t(*)[4]>(&h[12]));
  const uint32_t sw = (uint32_t)(r & 7);
  const uint32_t row = dst_tile + (uint32_t)r * 128u + (uint32_t)(c >> 1) * HALF_BYTES;
  const uint32_t c0 = (uint32_t)(4 * (c & 1));
#pragma unroll
  for (int i = 0; i < 4; ++i)
    st_shared_v4(row + (((c0 + i) ^ sw) << 4), h[4 * i], h[4 * i + 1], h[4 * i + 2],
                 h[4 * i + 3]);
}

// The query as fp16 into the two query boxes (16 rows of 64 fp16, 128-byte
// swizzled), by threads 0-255: thread t takes row r = t / 16 (query head
// hk*G + r, zero for r >= G) and its 16-byte chunk t % 16 of bf16 values.
// Per row: e = 15 - ceil(log2 max|q|) (the largest power of two with max|q|
// 2^e <= 2^15), the row times 2^e rounded to fp16; sl2[r] = the row's score
// scale (scale * key scale * log2 e * 2^-e).
__device__ __forceinline__ void write_query(const DecodeArgs &a, int b, int hk, int G, int zkv,
                                            int t, uint32_t q_tile, float *sl2) {
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
  const int qexp = amax > 0.f ? 15 - (fr == 0.5f ? ex - 1 : ex) : 0;  // 15 - ceil(log2 amax)
  uint32_t h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    h[i] = pack_f16x2(ldexpf(__uint_as_float(pr[i] << 16), qexp),
                      ldexpf(__uint_as_float(pr[i] & 0xffff0000u), qexp));
  const uint32_t box = q_tile + (uint32_t)(c16 >> 3) * QBOX;
  st_shared_v4(box + (uint32_t)r * 128u + ((((uint32_t)c16 & 7u) ^ (uint32_t)(r & 7)) << 4), h[0],
               h[1], h[2], h[3]);
  if (c16 == 0) sl2[r] = ldexpf(a.scale * __ldg(a.k_scale + zkv) * kLog2e, -qexp);
}

// The scale rows of block `row0` .. row0 + 127 of (b, KV head) slice `zkv`
// into the 1 KB stage at `dst`, by the 32 lanes of a producer warp (rows
// lane, lane + 32, lane + 64, lane + 96; rows past L read as zero). The
// caller adds each lane's arrival on the stage barrier (cp_async_arrive).
__device__ __forceinline__ void load_scales(uint32_t dst, const uint8_t *sc, int zkv, int row0,
                                            int L, int lane) {
  const uint8_t *slice = sc + (size_t)zkv * L * SC_ROW;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = lane + 32 * i;
    const int row = row0 + r;
    const bool in = row < L;
    cp_async8(dst + (uint32_t)r * SC_ROW, slice + (size_t)(in ? row : L - 1) * SC_ROW,
              in ? 8u : 0u);
  }
}

template <int G>
__global__ void __launch_bounds__(NT, 1)
    decode_nvfp4_kernel(const __grid_constant__ CUtensorMap tm_k,
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

  // The query and each head's score scale; the P^T rows of the padding heads
  // are zeroed once.
  if (tid < NQ * 16) write_query(a, b, hk, G, zkv, tid, base + SMEM_Q, sh.sl2);
  for (int idx = tid; idx < NPT * 2 * (NQ - G) * 8; idx += NT) {  // rows G..15, 16-byte chunks
    const int c = idx & 7, r = G + (idx >> 3) % (NQ - G), box = (idx >> 3) / (NQ - G);
    st_shared_v4(base + SMEM_PT + box * QBOX + r * 128 + c * 16, 0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();  // visible to the tensor core
  if (tid == 0) {
    for (int i = 0; i < NKF / 2; ++i) {
      mbar_init(smem_u32(&sh.kc_full[i]), 1 + 32);  // TMA arrival + 32 cp.async lanes
      mbar_init(smem_u32(&sh.kc_empty[i]), 4);      // the four key wideners
    }
    for (int i = 0; i < NKT / 2; ++i) {
      mbar_init(smem_u32(&sh.kt_full[i]), 4);  // the four key wideners
      mbar_init(smem_u32(&sh.kt_empty[i]), 1);  // the S^T commit of the pair
    }
    for (int i = 0; i < NVF; ++i) {
      mbar_init(smem_u32(&sh.vc_full[i]), 1 + 32);
      mbar_init(smem_u32(&sh.vc_empty[i]), 4);  // the four value wideners
    }
    for (int i = 0; i < NVH; ++i) {
      mbar_init(smem_u32(&sh.vh_full[i]), 4);
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
      // readers: the value producer, the O^T issuer, the four value wideners
      mbar_init(smem_u32(&sh.dec_empty[i]), 6);
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
    // ------------------------------------------------------ key producer --
    if (lane == 0) prefetch_tmap(&tm_k);
    const uint64_t pol = policy_evict_first();  // the cache is streamed once
    // Blocks in pairs: stage f holds two blocks' codes and scales under one
    // barrier.
    const int npair = (nb + 1) / 2;
    int issued = 0;
    for (int q = 0; q < npair; ++q) {
      if (__any_sync(0xffffffffu, *abort)) break;  // one outcome for the warp
      const int f = q % (NKF / 2);
      const int n = 2 * q + 1 < nb ? 2 : 1;
      if (q >= NKF / 2 && !mbar_wait_warp(smem_u32(&sh.kc_empty[f]), ((q / (NKF / 2)) - 1) & 1,
                                          abort, a.err, kErrTimeout))
        break;
      if (lane == 0) {
        mbar_expect_tx(smem_u32(&sh.kc_full[f]), n * CODE_BYTES);
        for (int t = 0; t < n; ++t)
          tma_load_3d(base + SMEM_KC + (2 * f + t) * CODE_BYTES, &tm_k, smem_u32(&sh.kc_full[f]),
                      0, (j0 + 2 * q + t) * BC, zkv, pol);
      }
      for (int t = 0; t < n; ++t)
        load_scales(base + SMEM_KS + (2 * f + t) * SC_BYTES, a.k_bs, zkv, (j0 + 2 * q + t) * BC,
                    a.L, lane);
      cp_async_arrive(smem_u32(&sh.kc_full[f]));
      ++issued;
    }
    for (int f = 0; f < NKF / 2 && f < issued; ++f) {  // drain the copies in flight
      const int last = f + ((issued - 1 - f) / (NKF / 2)) * (NKF / 2);
      mbar_wait_drain(smem_u32(&sh.kc_full[f]), (last / (NKF / 2)) & 1);
    }
  } else if (warp == WARP_V) {
    // ---------------------------------------------------- value producer --
    if (lane == 0) prefetch_tmap(&tm_v);
    const uint64_t pol = policy_evict_first();
    int vi = 0;
    for (int j = 0; j < nb; ++j) {
      if (__any_sync(0xffffffffu, *abort)) break;  // one outcome for the warp
      const int q = j >> 1, ds = q % NDP;
      if (!(j & 1) && !mbar_wait_warp(smem_u32(&sh.dec_full[ds]), (q / NDP) & 1, abort, a.err,
                                      kErrTimeout))
        break;
      const int keep = sh.dec[ds][j & 1];
      __syncwarp();
      if (lane == 0 && ((j & 1) || j == nb - 1)) mbar_arrive(smem_u32(&sh.dec_empty[ds]));
      if (!keep) continue;
      const int f = vi % NVF;
      if (vi >= NVF && !mbar_wait_warp(smem_u32(&sh.vc_empty[f]), ((vi / NVF) - 1) & 1, abort,
                                       a.err, kErrTimeout))
        break;
      if (lane == 0) {
        mbar_expect_tx(smem_u32(&sh.vc_full[f]), CODE_BYTES);
        tma_load_3d(base + SMEM_VC + f * CODE_BYTES, &tm_v, smem_u32(&sh.vc_full[f]), 0,
                    (j0 + j) * BC, zkv, pol);
      }
      load_scales(base + SMEM_VS + f * SC_BYTES, a.v_bs, zkv, (j0 + j) * BC, a.L, lane);
      cp_async_arrive(smem_u32(&sh.vc_full[f]));
      ++vi;
    }
    for (int f = 0; f < NVF && f < vi; ++f) {
      const int last = f + ((vi - 1 - f) / NVF) * NVF;
      mbar_wait_drain(smem_u32(&sh.vc_full[f]), (last / NVF) & 1);
    }
  } else if (warp >= WARP_KW && warp < WARP_VW) {
    // ------------------------------------------------------ key wideners --
    // Thread = key row r of the block = TMEM lane r: its 64 bytes of codes
    // and 8 block scales -> 64 columns of fp16 pairs (element 2i low).
    const int r = (warp - WARP_KW) * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int npair = (nb + 1) / 2;
    for (int q = 0; q < npair; ++q) {
      const int f = q % (NKF / 2), kp = q % (NKT / 2);
      const int n = 2 * q + 1 < nb ? 2 : 1;
      if (!mbar_wait_warp(smem_u32(&sh.kc_full[f]), (q / (NKF / 2)) & 1, abort, a.err,
                          kErrTimeout))
        break;
      // TMEM tiles of pair kp last fed the S^T products of pair q - NKT / 2.
      if (q >= NKT / 2 && !mbar_wait_warp(smem_u32(&sh.kt_empty[kp]), ((q / (NKT / 2)) - 1) & 1,
                                          abort, a.err, kErrTimeout))
        break;
      fence_after_sync();
      for (int t = 0; t < n; ++t) {
        const uint32_t codes = base + SMEM_KC + (2 * f + t) * CODE_BYTES;
        uint32_t slo, shi;
        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];"
                     : "=r"(slo), "=r"(shi)
                     : "r"(base + SMEM_KS + (2 * f + t) * SC_BYTES + (uint32_t)r * SC_ROW));
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // elements 64 half .. + 63: columns 32 half ..
          const uint4 x0 = ld_code_chunk(codes, r, 2 * half);
          const uint4 x1 = ld_code_chunk(codes, r, 2 * half + 1);
          const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          uint32_t h[32];
#pragma unroll
          for (int qw = 0; qw < 8; ++qw)  // word qw: elements 8qw..8qw+7, block 4 half + qw/2
            e2m1x8_scaled(w[qw], e4m3_scale2(slo, shi, 4 * half + (qw >> 1)),
                          *reinterpret_cast<uint32_t(*)[4]>(&h[4 * qw]));
          tmem_st32(lane_addr + TMEM_K + (uint32_t)(2 * kp + t) * 64u + (uint32_t)half * 32u, h);
        }
      }
      tmem_wait_st();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sh.kc_empty[f]));
        mbar_arrive(smem_u32(&sh.kt_full[kp]));
      }
    }
  } else if (warp >= WARP_VW) {
    // ---------------------------------------------------- value wideners --
    // Follow the decisions; chunks t, t + 128, ... (row = chunk / 4) of every
    // kept value tile.
    const int t0 = (warp - WARP_VW) * 32 + lane;
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
      if (!mbar_wait_warp(smem_u32(&sh.vc_full[f]), (vi / NVF) & 1, abort, a.err, kErrTimeout))
        break;
      if (vi >= NVH && !mbar_wait_warp(smem_u32(&sh.vh_empty[hs]), ((vi / NVH) - 1) & 1, abort,
                                       a.err, kErrTimeout))
        break;
#pragma unroll 2
      for (int t = t0; t < BC * 4; t += NVW)
        widen_value_chunk(base + SMEM_VC + f * CODE_BYTES, base + SMEM_VS + f * SC_BYTES,
                          base + SMEM_VH + hs * H_BYTES, t);
      fence_proxy_async_smem();  // the fp16 rows are visible to the tensor core
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sh.vc_empty[f]));
        mbar_arrive(smem_u32(&sh.vh_full[hs]));
      }
      ++vi;
    }
  } else if (warp == WARP_QK) {
    // --------------------------------------------------------- S^T issuer --
    if (lane == 0) {
      const uint64_t qd = kmajor_base(base + SMEM_Q);
      // Blocks in pairs: one TMEM-tile barrier, one S^T buffer barrier and
      // two commits per pair (a barrier wait between products costs about as
      // much as a product).
      const int npair = (nb + 1) / 2;
      for (int q = 0; q < npair; ++q) {
        const int kp = q % (NKT / 2), pb = q & 1;
        const int n = 2 * q + 1 < nb ? 2 : 1;
        if (!mbar_wait(smem_u32(&sh.kt_full[kp]), (q / (NKT / 2)) & 1, abort, a.err,
                       kErrTimeout) ||
            // pair buffer pb is free once the score warps have read pair q - 2
            (q >= 2 && !mbar_wait(smem_u32(&sh.s_free[pb]), ((q >> 1) - 1) & 1, abort, a.err,
                                  kErrTimeout)))
          break;
        fence_after_sync();
        for (int t = 0; t < n; ++t) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_ts(tmem + TMEM_S + (2 * pb + t) * NQ, tmem + TMEM_K + (2 * kp + t) * 64 + kk * 8,
                        qd + box_step(kk), IDESC_QK, kk > 0);
        }
        mma_commit(smem_u32(&sh.s_full[pb]));
        mma_commit(smem_u32(&sh.kt_empty[kp]));
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
        const uint64_t pd = kmajor_base(base + SMEM_PT + pb * 2 * QBOX);
#pragma unroll
        for (int kk = 0; kk < BC / 16; ++kk)
          mma_bf16_ss(tmem + TMEM_O, vd + vmajor_step(kk), pd + box_step(kk), IDESC_PV,
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
    // Kept block: exponent references (rescaled lazily), this key's P for
    // every head into the next P^T buffer, the per-thread row sums, an O^T
    // rescale when a reference moved.
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
        const uint32_t box = base + SMEM_PT + (uint32_t)(pb * 2 + (kidx >> 6)) * QBOX;
        const uint32_t kk = (uint32_t)(kidx & 63);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const uint32_t addr = box + (uint32_t)g * 128u + ((((kk >> 3) ^ (uint32_t)g)) << 4) +
                                (kk & 7u) * 2u;
          const unsigned short hv = __half_as_ushort(__float2half_rn(p[g]));
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(hv) : "memory");
        }
      }
      // O^T rescale once the previous product has landed (its commit to the
      // P^T buffer it read); the same decision in every thread.
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
      uint32_t x[32];  // block j: columns [0,16); block j + 1: [16,32) (the adjacent buffer)
      tmem_ld32(lane_base + TMEM_S + sb * NQ, x);
      tmem_wait_ld_regs(x);
      fence_before_sync();  // the scores are in registers: the S^T buffers are free
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.s_free[pb]));
      const bool v0 = (j0 + j) * BC + kidx < a.L;
      const bool v1 = two && (j0 + j + 1) * BC + kidx < a.L;
      float s0[G], s1[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        s0[g] = v0 ? __uint_as_float(x[g]) * sl2[g] : -INFINITY;
        s1[g] = v1 ? __uint_as_float(x[NQ + g]) * sl2[g] : -INFINITY;
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
      const float vs = __ldg(a.v_scale + zkv);
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

cudaError_t launch_decode_nvfp4(const DecodeArgs &a, cudaStream_t s) {
  CUtensorMap mk, mv;
  // [B*Hkv, L, 64] bytes of E2M1 codes with the caller's row stride (bytes);
  // boxes of 64 bytes x 128 keys, 64-byte swizzle; keys past L read as zero.
  if (!make_map_u8_3d(&mk, a.k, CODE_ROW, a.k_row_stride, a.L, a.B * a.Hkv, BC,
                      CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map_u8_3d(&mv, a.v, CODE_ROW, a.v_row_stride, a.L, a.B * a.Hkv, BC,
                      CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  const int G = a.Hq / a.Hkv;
  auto kernel = G == 1   ? decode_nvfp4_kernel<1>
                : G == 2 ? decode_nvfp4_kernel<2>
                : G == 4 ? decode_nvfp4_kernel<4>
                : G == 8 ? decode_nvfp4_kernel<8>
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
