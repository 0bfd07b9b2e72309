// Split-KV decode with softmax-threshold block skipping over an NVFP4
// key/value cache (d = 128, Bc = 128), on warp-level tensor-core products.
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
// A decode block is a batched matrix-vector product (G <= 8 query heads
// against 128 keys) and HBM bound.  A tcgen05 product has 128 rows and takes
// about as long to issue whatever its width, so with G heads most of it is
// padding and the issue rate, not HBM, would set the pace.  Here every
// product is a warp-level m16n8k16 one (fp16 operands, fp32 accumulation)
// with its operands in registers:
//   S = K_j Q^T       A = 16 keys x 16 elements, widened from the codes in
//                     registers (cvt.e2m1x2 times the E4M3 block scale: an
//                     E2M1 value has two significant bits and an E4M3 scale
//                     four, so the product is an exact fp16 normal number);
//                     B = the query as fp16 after a power-of-two per-head
//                     scale 2^e (max|q| 2^e <= 2^15), exact for every bf16
//                     element not below ~2^-31 of the head's largest;
//                     C = 16 keys x 8 heads (heads past G are zero columns);
//   O^T += V_j^T P^T  A = 16 value dimensions x 16 keys from a widened fp16
//                     value tile (ldmatrix.trans), B = P^T (keys x heads,
//                     fp16) from shared memory, C = O^T held in registers.
// The contracted dimension of S is taken in a permuted order, the same for A
// and B (a dot product does not depend on the order of its terms): lane
// (g, q) = (lane / 4, lane % 4) holds elements 32q .. 32q + 31 of its key
// rows and of query head g, so one 16-byte load of a code row serves all
// eight k-steps of a block; in k-step kk, columns 2q, 2q + 1 are elements
// 32q + 4kk + {0, 1} (code byte 16q + 2kk) and columns 2q + 8, 2q + 9 are
// elements 32q + 4kk + {2, 3} (the next byte).
//
// One CTA per (sequence, KV head, split).  Warp roles (320 threads):
//   warps 0-3  scores: warp w owns keys 32w .. 32w + 31 of every block (two
//              16-key products per k-step); blocks in pairs: both blocks'
//              products, one exchange of the four warps' maxima per head, both
//              decisions (every head votes skip), exponentials, P^T, row sums;
//   warps 4-7  values: warp 4 + w owns value dimensions 32w .. 32w + 31 (two
//              16-row products per k-step) of O^T; it widens those columns
//              of every kept value tile into its own part of one fp16 tile,
//              then runs its products; rescales and the epilogue;
//   warp 8     key producer: TMA of the code tile, block scales by cp.async
//              from its 32 lanes (zero past L);
//   warp 9     value producer, kept blocks only.
// Two CTAs share an SM (105 KB of shared memory, <= 102 registers a thread),
// so one CTA's per-block latencies (loads, product chains, the score warps'
// exchange) overlap the other's.  Every other wait inside the loops is a
// bounded mbarrier wait, so a failed wait ends the roles' loops with an
// error status instead of a hang; the score warps' one named barrier is met
// equally often by all four (their loop runs to its end).
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
constexpr int BC = 128;   // keys per block
constexpr int NKF = 5;    // key stages (codes + block scales)
constexpr int NVF = 2;    // value code stages
constexpr int NP = 4;     // P^T buffers
constexpr int NDEC = 16;  // decision ring
constexpr int NSW = 4;    // score warps
constexpr int NVW = 4;    // value warps
constexpr int WARP_VAL = NSW, WARP_K = NSW + NVW, WARP_V = WARP_K + 1;
constexpr int NT = (WARP_V + 1) * 32;
constexpr int kScoreBarrier = 1;  // named barrier of the four score warps
constexpr uint32_t CODE_ROW = D / 2;            // 64 bytes of codes per row
constexpr uint32_t SC_ROW = D / 16;             // 8 block scales per row
constexpr uint32_t CODE_BYTES = BC * CODE_ROW;  // 8 KB
constexpr uint32_t SC_BYTES = BC * SC_ROW;      // 1 KB
constexpr uint32_t H_BYTES = BC * D * 2;        // 32 KB: 128 keys x 128 fp16
constexpr uint32_t HALF_BYTES = H_BYTES / 2;    // one 64-column box
// P^T buffer: 8 head rows of 128 fp16 keys, rows 272 bytes apart so that the
// eight rows of a fragment load fall in different banks.
constexpr uint32_t P_ROW = BC * 2 + 16;
constexpr uint32_t P_BYTES = 8 * P_ROW;
constexpr uint32_t SMEM_KC = 0;
constexpr uint32_t SMEM_VC = SMEM_KC + NKF * CODE_BYTES;
constexpr uint32_t SMEM_VH = SMEM_VC + NVF * CODE_BYTES;
constexpr uint32_t SMEM_KS = SMEM_VH + H_BYTES;
constexpr uint32_t SMEM_VS = SMEM_KS + NKF * SC_BYTES;
constexpr uint32_t SMEM_P = SMEM_VS + NVF * SC_BYTES;
constexpr uint32_t SMEM_TILES = SMEM_P + NP * P_BYTES;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // exp reference may lag the max by 2^8
static_assert(SMEM_VC % 1024 == 0 && SMEM_VH % 1024 == 0 && SMEM_P % 16 == 0,
              "swizzled TMA destinations and value tiles on 1024-byte boundaries");

struct Shared {
  uint64_t kc_full[NKF], kc_empty[NKF];
  uint64_t vc_full[NVF], vc_empty[NVF];
  uint64_t p_full[NP], p_free[NP];
  uint64_t dec_full[NDEC], dec_empty[NDEC];
  uint64_t l_full;       // the score warps' row sums are in
  int dec[NDEC];
  float red[2][NSW][16];  // per block pair (double buffered): per score warp, block, head max
  float alpha[NP][8];    // per P^T buffer: the heads' O^T rescale factors
  float lsum[NSW][8];    // epilogue: per score warp, per head row sum
  int abort;
};
constexpr uint32_t SMEM_ALLOC = SMEM_TILES + ((sizeof(Shared) + 127) / 128) * 128;
static_assert(2 * SMEM_ALLOC <= 226 * 1024, "shared memory budget: two CTAs per SM");

// D += A B for one m16n8k16 product (fp16 operands, fp32 accumulators).
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
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

// Two E4M3 block scales (the low two bytes of v: scale 0, scale 1) -> the
// fp16 pairs (s0, s0) and (s1, s1).
__device__ __forceinline__ void e4m3_scale_pairs(uint32_t v, uint32_t &s00, uint32_t &s11) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((unsigned short)(v & 0xffffu)));
  s00 = __byte_perm(r, r, 0x1010);
  s11 = __byte_perm(r, r, 0x3232);
}

// Code chunk c (bytes 16c..16c+15: elements 32c..32c+31) of row r of a value
// code tile (64-byte rows, 64-byte swizzle: chunk c at chunk position
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
// (box c / 2 of two 64-column boxes of 128-byte rows; 16-byte chunks
// 4 (c % 2) .. + 3 of the row, at chunk position chunk ^ (r % 8)).
__device__ __forceinline__ void widen_value_chunk(uint32_t codes, uint32_t scales,
                                                  uint32_t dst_tile, int t) {
  const int r = t >> 2, c = t & 3;
  const uint4 x = ld_code_chunk(codes, r, c);
  uint32_t sc;
  asm volatile("ld.shared.u16 %0, [%1];"
               : "=r"(sc)
               : "r"(scales + (uint32_t)r * SC_ROW + 2u * (uint32_t)c));
  uint32_t s0, s1;
  e4m3_scale_pairs(sc, s0, s1);
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

// The scale rows of block `row0` .. row0 + 127 of (b, KV head) slice `zkv`
// into the 1 KB stage at `dst`, by the 32 lanes of a producer warp (rows
// lane, lane + 32, lane + 64, lane + 96; rows past L read as zero).  The
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
__global__ void __launch_bounds__(NT, 2)
    decode_nvfp4_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Shared &sh = *reinterpret_cast<Shared *>(smem_raw + SMEM_TILES);
  const uint32_t base = smem_u32(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;  // fragment row group, thread in the group
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

  // The P^T rows of the heads past G stay zero (the products' padding columns).
  if constexpr (G < 8) {
    constexpr int kChunks = (int)(P_ROW / 16), kPad = (8 - G) * kChunks;
    for (int idx = tid; idx < NP * kPad; idx += NT) {
      const int buf = idx / kPad, r = G + (idx % kPad) / kChunks, c = (idx % kPad) % kChunks;
      st_shared_v4(base + SMEM_P + buf * P_BYTES + r * P_ROW + c * 16, 0u, 0u, 0u, 0u);
    }
  }
  if (tid == 0) {
    for (int i = 0; i < NKF; ++i) {
      mbar_init(smem_u32(&sh.kc_full[i]), 1 + 32);  // TMA arrival + 32 cp.async lanes
      mbar_init(smem_u32(&sh.kc_empty[i]), NSW);
    }
    for (int i = 0; i < NVF; ++i) {
      mbar_init(smem_u32(&sh.vc_full[i]), 1 + 32);
      mbar_init(smem_u32(&sh.vc_empty[i]), NVW);
    }
    for (int i = 0; i < NP; ++i) {
      mbar_init(smem_u32(&sh.p_full[i]), NSW);
      mbar_init(smem_u32(&sh.p_free[i]), NVW);
    }
    for (int i = 0; i < NDEC; ++i) {
      mbar_init(smem_u32(&sh.dec_full[i]), 1);
      mbar_init(smem_u32(&sh.dec_empty[i]), 1 + NVW);  // the value producer, the value warps
    }
    mbar_init(smem_u32(&sh.l_full), NSW);
    sh.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == WARP_K) {
    // ------------------------------------------------------ key producer --
    if (lane == 0) prefetch_tmap(&tm_k);
    const uint64_t pol = policy_evict_first();  // the cache is streamed once
    int issued = 0;
    for (int j = 0; j < nb; ++j) {
      if (__any_sync(0xffffffffu, *abort)) break;  // one outcome for the warp
      const int f = j % NKF;
      if (j >= NKF && !mbar_wait_warp(smem_u32(&sh.kc_empty[f]), ((j / NKF) - 1) & 1, abort,
                                      a.err, kErrTimeout))
        break;
      if (lane == 0) {
        mbar_expect_tx(smem_u32(&sh.kc_full[f]), CODE_BYTES);
        tma_load_3d(base + SMEM_KC + f * CODE_BYTES, &tm_k, smem_u32(&sh.kc_full[f]), 0,
                    (j0 + j) * BC, zkv, pol);
      }
      load_scales(base + SMEM_KS + f * SC_BYTES, a.k_bs, zkv, (j0 + j) * BC, a.L, lane);
      cp_async_arrive(smem_u32(&sh.kc_full[f]));
      ++issued;
    }
    for (int f = 0; f < NKF && f < issued; ++f) {  // drain the copies in flight
      const int last = f + ((issued - 1 - f) / NKF) * NKF;
      mbar_wait_drain(smem_u32(&sh.kc_full[f]), (last / NKF) & 1);
    }
  } else if (warp == WARP_V) {
    // ---------------------------------------------------- value producer --
    if (lane == 0) prefetch_tmap(&tm_v);
    const uint64_t pol = policy_evict_first();
    int vi = 0;
    for (int j = 0; j < nb; ++j) {
      if (__any_sync(0xffffffffu, *abort)) break;  // one outcome for the warp
      const int ds = j % NDEC;
      if (!mbar_wait_warp(smem_u32(&sh.dec_full[ds]), (j / NDEC) & 1, abort, a.err, kErrTimeout))
        break;
      const int keep = sh.dec[ds];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.dec_empty[ds]));
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
  } else if (warp >= WARP_VAL) {
    // ------------------------------------------------------------- values --
    // O^T rows (value dimensions) 32 vw + 16 mt + g and + 8, for mt = 0, 1;
    // columns (heads) 2q, 2q + 1.
    const int vw = warp - WARP_VAL;
    float o[2][2][4];  // [mt][even / odd k-steps][fragment]
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[mt][e][i] = 0.f;
    // ldmatrix row addresses: lane l gives row l % 8 of matrix l / 8, whose
    // keys are 8 further for matrices 2 and 3 and whose value dimensions are 8
    // further for matrices 1 and 3 (the A fragment's four registers).
    const int lm = lane >> 3, li = lane & 7;
    const int key_off = (lm >> 1) * 8 + li;  // key within the 16-key k-step
    uint32_t a_box[2], a_chunk[2];           // per mt: box and 16-byte chunk of the dimensions
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const int d0 = vw * 32 + mt * 16 + (lm & 1) * 8;
      a_box[mt] = (uint32_t)(d0 >> 6) * HALF_BYTES;
      a_chunk[mt] = (uint32_t)((d0 & 63) >> 3);
    }
    const uint32_t tile = base + SMEM_VH;
    bool ok = true;
    int kc = 0;
    for (int j = 0; j < nb; ++j) {
      const int ds = j % NDEC;
      if (!mbar_wait_warp(smem_u32(&sh.dec_full[ds]), (j / NDEC) & 1, abort, a.err,
                          kErrTimeout)) {
        ok = false;
        break;
      }
      const int keep = sh.dec[ds];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.dec_empty[ds]));
      if (!keep) continue;
      const int f = kc % NVF, pb = kc % NP;
      if (!mbar_wait_warp(smem_u32(&sh.vc_full[f]), (kc / NVF) & 1, abort, a.err, kErrTimeout)) {
        ok = false;
        break;
      }
      // This warp's value dimensions (code chunk vw) of all 128 keys into its
      // own columns of the fp16 tile, which only it reads: the previous
      // block's reads of them are done (its products have completed).
#pragma unroll
      for (int i = 0; i < 4; ++i)
        widen_value_chunk(base + SMEM_VC + f * CODE_BYTES, base + SMEM_VS + f * SC_BYTES, tile,
                          (lane + 32 * i) * 4 + vw);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.vc_empty[f]));  // the codes are read
      if (!mbar_wait_warp(smem_u32(&sh.p_full[pb]), (kc / NP) & 1, abort, a.err, kErrTimeout)) {
        ok = false;
        break;
      }
      const float al0 = sh.alpha[pb][2 * q], al1 = sh.alpha[pb][2 * q + 1];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          o[mt][e][0] *= al0;
          o[mt][e][1] *= al1;
          o[mt][e][2] *= al0;
          o[mt][e][3] *= al1;
        }
      const uint32_t pbuf = base + SMEM_P + pb * P_BYTES;
#pragma unroll
      for (int ks = 0; ks < BC / 16; ++ks) {
        // B = P^T: keys 16ks + 2q, +1 (b0) and 16ks + 8 + 2q, +1 (b1) of head g
        // (lanes 0-7 address the first 8 keys' rows, lanes 8-15 the next 8).
        uint32_t b0, b1;
        ldsm_x2(pbuf + (uint32_t)li * P_ROW + (uint32_t)(16 * ks + (lm & 1) * 8) * 2u, b0, b1);
        const int key = 16 * ks + key_off;
        const uint32_t row = tile + (uint32_t)key * 128u;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          uint32_t av[4];
          ldsm_x4_trans(row + a_box[mt] + ((a_chunk[mt] ^ (uint32_t)(key & 7)) << 4), av);
          mma16816(o[mt][ks & 1], av, b0, b1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.p_free[pb]));  // P^T is read
      ++kc;
    }
    // ---- epilogue: O_s = v_scale * O / l per head (the score warps' sums) ----
    if (ok) ok = mbar_wait_warp(smem_u32(&sh.l_full), 0, abort, a.err, kErrTimeout);
    if (ok) {
      const float vs = __ldg(a.v_scale + zkv);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int h = 2 * q + c;
        if (h < G) {
          const float lt = (sh.lsum[0][h] + sh.lsum[1][h]) + (sh.lsum[2][h] + sh.lsum[3][h]);
          const float sc = vs / lt;
          float *orow = a.o_part + ((size_t)(b * a.Hq + hk * G + h) * a.n_splits + sp) * D;
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            const int d0 = vw * 32 + mt * 16 + g;
            orow[d0] = (o[mt][0][c] + o[mt][1][c]) * sc;
            orow[d0 + 8] = (o[mt][0][2 + c] + o[mt][1][2 + c]) * sc;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------- scores --
    // Keys 32 warp + 16 mt + g and + 8 of each block, heads 2q, 2q + 1.
    // The query fragments (B) of all eight k-steps: head g, elements
    // 32q .. 32q + 31 as fp16 pairs after the head's power-of-two scale.
    uint32_t qb[16];
    float sl2h[2];  // raw score -> log2 units, heads 2q, 2q + 1
    {
      uint4 v[4] = {};
      if (g < G) {
        const uint4 *src = reinterpret_cast<const uint4 *>((const __nv_bfloat16 *)a.q +
                                                           (size_t)(b * a.Hq + hk * G + g) * D) +
                           4 * q;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = __ldg(src + i);
      }
      const uint32_t pr[16] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w,
                               v[2].x, v[2].y, v[2].z, v[2].w, v[3].x, v[3].y, v[3].z, v[3].w};
      uint32_t amax_bits = 0;  // |bf16| bit patterns order like their values
#pragma unroll
      for (int i = 0; i < 16; ++i)
        amax_bits = max(amax_bits, max(pr[i] & 0x7fffu, (pr[i] >> 16) & 0x7fffu));
      // The four lanes of head g hold its 128 elements.
      amax_bits = max(amax_bits, __shfl_xor_sync(0xffffffffu, amax_bits, 1));
      amax_bits = max(amax_bits, __shfl_xor_sync(0xffffffffu, amax_bits, 2));
      const float amax = __uint_as_float(amax_bits << 16);
      int ex = 0;
      const float fr = frexpf(amax > 0.f ? amax : 1.f, &ex);  // amax = fr * 2^ex
      const int qexp = amax > 0.f ? 15 - (fr == 0.5f ? ex - 1 : ex) : 0;  // 15 - ceil(log2 amax)
#pragma unroll
      for (int i = 0; i < 16; ++i)
        qb[i] = pack_f16x2(ldexpf(__uint_as_float(pr[i] << 16), qexp),
                           ldexpf(__uint_as_float(pr[i] & 0xffff0000u), qexp));
      const float kscale = a.scale * __ldg(a.k_scale + zkv) * kLog2e;
#pragma unroll
      for (int c = 0; c < 2; ++c)  // head 2q + c: its exponent is in lanes 4 (2q + c) ..
        sl2h[c] = ldexpf(kscale, -__shfl_sync(0xffffffffu, qexp, 4 * (2 * q + c)));
    }
    uint32_t *bits = a.bits + (size_t)unit * a.words;
    const float c2 = a.ln_lambda * kLog2e;  // ln(lambda), log2 units
    // Running max and exp reference of this thread's heads 2q, 2q + 1 (heads
    // past G vote skip and are never used).
    float m2[2] = {-INFINITY, -INFINITY}, mref[2] = {-INFINITY, -INFINITY};
    bool hv[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) hv[c] = 2 * q + c < G;
    float lp[2] = {0.f, 0.f};  // this thread's part of the row sums, heads 2q, 2q + 1
    int kc = 0;
    uint32_t word = 0;
    bool ok = true;
    // Blocks in pairs: both blocks' products, then one exchange of the four
    // warps' maxima and both decisions (block j + 1 is tested against the
    // running max after block j).
    for (int j = 0; j < nb; j += 2) {
      const int np = j + 1 < nb ? 2 : 1;
      const int pr = (j >> 1) & 1;  // exchange buffer of this pair
      float s[2][2][4];             // [block][mt][fragment]: scores in log2 units, -inf past L
#pragma unroll
      for (int t = 0; t < 2; ++t) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) s[t][mt][i] = -INFINITY;
        if ((t == 1 && np == 1) || !ok) break;
        const int jj = j + t, f = jj % NKF;
        if (!mbar_wait_warp(smem_u32(&sh.kc_full[f]), (jj / NKF) & 1, abort, a.err,
                            kErrTimeout)) {
          ok = false;
          break;
        }
        // Rows r and r + 8 of each 16-key product: code bytes 16q .. 16q + 15
        // (elements 32q .. 32q + 31) and their two block scales (2q, 2q + 1).
        const uint32_t codes = base + SMEM_KC + f * CODE_BYTES;
        const uint32_t scales = base + SMEM_KS + f * SC_BYTES;
        uint4 cw[2][2];
        uint32_t sw[2][2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int r = warp * 32 + mt * 16 + hr * 8 + g;
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(cw[mt][hr].x), "=r"(cw[mt][hr].y), "=r"(cw[mt][hr].z),
                           "=r"(cw[mt][hr].w)
                         : "r"(codes + (uint32_t)r * CODE_ROW + 16u * (uint32_t)q));
            asm volatile("ld.shared.u16 %0, [%1];"
                         : "=r"(sw[mt][hr])
                         : "r"(scales + (uint32_t)r * SC_ROW + 2u * (uint32_t)q));
          }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.kc_empty[f]));  // the stage is in registers
        // S, with two accumulators per product (even and odd k-steps) so that
        // the chains of dependent products are half as long.
        float acc[2][2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[mt][e][i] = 0.f;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          uint32_t s0[2], s1[2];  // per row (r, r + 8): scale pairs of blocks 2q, 2q + 1
          e4m3_scale_pairs(sw[mt][0], s0[0], s1[0]);
          e4m3_scale_pairs(sw[mt][1], s0[1], s1[1]);
          const uint32_t w0[4] = {cw[mt][0].x, cw[mt][0].y, cw[mt][0].z, cw[mt][0].w};
          const uint32_t w1[4] = {cw[mt][1].x, cw[mt][1].y, cw[mt][1].z, cw[mt][1].w};
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            // Word m: k-steps 2m (bytes 0, 1) and 2m + 1 (bytes 2, 3); elements
            // 32q + 8m .. + 7, block scale 2q for m < 2, 2q + 1 after.
            uint32_t h0[4], h1[4];
            e2m1x8_scaled(w0[m], m < 2 ? s0[0] : s1[0], h0);
            e2m1x8_scaled(w1[m], m < 2 ? s0[1] : s1[1], h1);
            const uint32_t a0[4] = {h0[0], h1[0], h0[1], h1[1]};
            const uint32_t a1[4] = {h0[2], h1[2], h0[3], h1[3]};
            mma16816(acc[mt][0], a0, qb[4 * m], qb[4 * m + 1]);
            mma16816(acc[mt][1], a1, qb[4 * m + 2], qb[4 * m + 3]);
          }
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int key = (j0 + jj) * BC + warp * 32 + mt * 16 + (i >> 1) * 8 + g;
            const float v = (acc[mt][0][i] + acc[mt][1][i]) * sl2h[i & 1];
            s[t][mt][i] = key < a.L ? v : -INFINITY;
          }
      }
      // This thread's maxima over its four keys of each block, heads 2q,
      // 2q + 1, then over the warp's row groups; the four warps' exchange.
      float mx[2][2];
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float m = fmaxf(fmaxf(s[t][0][c], s[t][0][2 + c]), fmaxf(s[t][1][c], s[t][1][2 + c]));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
          mx[t][c] = m;
        }
      if (g == 0) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          sh.red[pr][warp][8 * t + 2 * q] = mx[t][0];
          sh.red[pr][warp][8 * t + 2 * q + 1] = mx[t][1];
        }
      }
      // The four score warps meet on a named barrier once per pair, whatever
      // happened before: after a failed wait a warp skips the work but not
      // the barrier, so none waits for ever.  (A warp writes buffer pr again
      // two pairs later, after the next barrier, when every warp has read it.)
      named_bar_sync(kScoreBarrier, NSW * 32);
      if (!ok) continue;
      // Block maxima of this thread's heads; with c < 0, "rowmax - m_new < c"
      // is "rowmax - m_old < c" (a block that raises the max fails both).
      // Every head must vote skip: the four lanes of a row group hold all
      // eight heads, and every warp takes the same decisions.
      bool skip[2] = {true, true};
      float mnew[2][2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        bool mine = true;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int h = 8 * t + 2 * q + c;
          const float bm = fmaxf(fmaxf(sh.red[pr][0][h], sh.red[pr][1][h]),
                                 fmaxf(sh.red[pr][2][h], sh.red[pr][3][h]));
          const float d = (bm == -INFINITY) ? -INFINITY : bm - m2[c];
          mine = mine && (!hv[c] || d < c2);
          mnew[t][c] = fmaxf(m2[c], bm);
          if (t < np) m2[c] = mnew[t][c];  // the running max advances on every block
        }
        skip[t] = __all_sync(0xffffffffu, mine);
      }
      if (tid == 0) {
        for (int t = 0; t < np; ++t) {
          const int jj = j + t, ds = jj % NDEC;
          // On a timeout the abort flag is raised and every later wait fails.
          if (jj < NDEC || mbar_wait(smem_u32(&sh.dec_empty[ds]), ((jj / NDEC) - 1) & 1, abort,
                                     a.err, kErrTimeout)) {
            sh.dec[ds] = skip[t] ? 0 : 1;
            mbar_arrive(smem_u32(&sh.dec_full[ds]));
          }
          if (skip[t]) word |= 1u << (jj & 31);
          if ((jj & 31) == 31 || jj == nb - 1) {
            bits[jj >> 5] = word;
            word = 0;
          }
        }
      }
      // Kept blocks: exponent references (rescaled lazily; the factors go to
      // the value warps with P^T), P^T of this thread's keys, row sums.
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (t >= np || skip[t] || !ok) continue;
        const int pb = kc % NP;
        if (kc >= NP && !mbar_wait_warp(smem_u32(&sh.p_free[pb]), ((kc / NP) - 1) & 1, abort,
                                         a.err, kErrTimeout)) {
          ok = false;
          continue;
        }
        float alpha[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          alpha[c] = 1.f;
          if (mref[c] == -INFINITY) {
            mref[c] = mnew[t][c];
          } else if (mnew[t][c] > mref[c] + kRescaleLog2) {
            alpha[c] = ex2(mref[c] - mnew[t][c]);
            mref[c] = mnew[t][c];
          }
          lp[c] *= alpha[c];
        }
        if (warp == 0 && g == 0) {  // heads 2q, 2q + 1 (1 past G)
          sh.alpha[pb][2 * q] = hv[0] ? alpha[0] : 1.f;
          sh.alpha[pb][2 * q + 1] = hv[1] ? alpha[1] : 1.f;
        }
        const uint32_t pbuf = base + SMEM_P + pb * P_BYTES;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = i & 1, h = 2 * q + c;
            if (h < G) {
              const int key = warp * 32 + mt * 16 + (i >> 1) * 8 + g;
              const float p = ex2(s[t][mt][i] - mref[c]);
              lp[c] += p;
              const unsigned short hv16 = __half_as_ushort(__float2half_rn(p));
              asm volatile("st.shared.u16 [%0], %1;" ::"r"(pbuf + (uint32_t)h * P_ROW +
                                                          (uint32_t)key * 2u),
                           "h"(hv16)
                           : "memory");
            }
          }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.p_full[pb]));
        ++kc;
      }
    }
    // ---- epilogue: row sums per head to the value warps, LSE_s = ref + ln l ----
    if (tid == 0)
      for (int w = ((nb - 1) >> 5) + 1; w < a.words; ++w) bits[w] = 0u;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      lp[c] += __shfl_xor_sync(0xffffffffu, lp[c], 4);
      lp[c] += __shfl_xor_sync(0xffffffffu, lp[c], 8);
      lp[c] += __shfl_xor_sync(0xffffffffu, lp[c], 16);
    }
    if (g == 0) {
      sh.lsum[warp][2 * q] = lp[0];
      sh.lsum[warp][2 * q + 1] = lp[1];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh.l_full));
    if (ok) ok = mbar_wait_warp(smem_u32(&sh.l_full), 0, abort, a.err, kErrTimeout);
    if (ok && warp == 0 && g == 0) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int h = 2 * q + c;
        if (hv[c]) {
          const float lt = (sh.lsum[0][h] + sh.lsum[1][h]) + (sh.lsum[2][h] + sh.lsum[3][h]);
          a.lse_part[(size_t)(b * a.Hq + hk * G + h) * a.n_splits + sp] = mref[c] * kLn2 + logf(lt);
        }
      }
    }
  }

  __syncwarp();
  __syncthreads();
}

}  // namespace

cudaError_t launch_decode_nvfp4(const DecodeArgs &a, cudaStream_t s) {
  CUtensorMap mk, mv;
  // [B*Hkv, L, 64] bytes of E2M1 codes with the caller's row stride (bytes);
  // boxes of 64 bytes x 128 keys, keys past L read as zero.  Key tiles land
  // unswizzled (the score lanes' 16-byte loads at 16q of rows r, r + 1 of
  // each eight-lane phase meet no bank twice); value tiles with the 64-byte
  // swizzle (one widening thread per row chunk).
  if (!make_map_u8_3d(&mk, a.k, CODE_ROW, a.k_row_stride, a.L, a.B * a.Hkv, BC,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
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
