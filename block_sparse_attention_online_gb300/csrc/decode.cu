// Split-KV decode with softmax-threshold block skipping (bf16 cache, d = 128,
// Bc = 128), on the tensor cores.
//
// Method: the BLASST page, sections "BLASST 的判定准则" (Eq. 5) and "Decode 内核：
// 砍带宽" (in decode the skipped block's value load is the saving; the scores
// of a block decide whether its values are read at all).  One CTA per
// (sequence, KV head, split); the G query heads sharing the KV head are the
// rows of the products, so each key byte is read once for all of them and the
// decision of a block is the AND of the G heads' votes.
//
// The G heads are padded to the 128 rows of a tcgen05 MMA: the tensor core
// idles in decode anyway, and a full-width row per head puts each head's 128
// scores in one thread, so a block's row maxima, votes and decision need no
// reduction across warps.  Per block:
//   S_j   = Q K_j^T        (M 128 padded heads, N 128 keys, K 128; TMEM)
//   P_j   = exp2(S_j - ref) (bf16 pairs into a TMEM P buffer, kept blocks)
//   O    += P_j V_j        (A = P from TMEM, B = V_j from shared memory)
// Warp roles (160 threads):
//   warp 0  softmax: lane g < G owns head g.  Row max of S_j, vote, decision
//           (published to the producers and the P.V issuer), then for a kept
//           block P_j, its row sum and a lazy O rescale; epilogue;
//   warp 1  TMA producer of K_j (every block, 4-stage ring);
//   warp 2  Q.K^T issuer (two TMEM S buffers; also allocates TMEM);
//   warp 3  TMA producer of V_j for kept blocks only, issued as soon as the
//           block's decision is published (2-stage ring);
//   warp 4  P.V issuer.
// The softmax warp frees a block's S buffer as soon as the scores are in its
// registers (P lives in its own TMEM buffers), so the Q.K^T products of the
// next blocks, and with them the next decisions and value loads, run ahead
// while a kept block's value load is still in flight.
// TMEM columns: S buffers [0,256), P buffers [256,384), O [384,512).
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"
#include "tc_common.cuh"

namespace attn_skip {
namespace {

using namespace tc;

constexpr int D = 128;   // head size (keys and values)
constexpr int BC = 128;  // keys per block
constexpr int MR = 128;  // MMA rows (heads padded)
constexpr int NK = 4;    // key stages
constexpr int NV = 2;    // value stages
constexpr int NS = 2;    // TMEM S buffers
constexpr int NP = 2;    // TMEM P buffers
constexpr int NDEC = 8;  // decision ring
constexpr int NT = 5 * 32;
constexpr int WARP_K = 1, WARP_QK = 2, WARP_V = 3, WARP_PV = 4;  // warp 0: softmax
constexpr uint32_t TILE_BYTES = BC * D * 2;      // 32 KB: 128 rows x 128 bf16
constexpr uint32_t HALF_BYTES = TILE_BYTES / 2;  // one 64-column swizzled box
constexpr uint32_t SMEM_K = 0;
constexpr uint32_t SMEM_V = SMEM_K + NK * TILE_BYTES;
constexpr uint32_t SMEM_Q = SMEM_V + NV * TILE_BYTES;
constexpr uint32_t SMEM_TILES = SMEM_Q + TILE_BYTES;  // 224 KB
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_P = NS * BC;
constexpr uint32_t TMEM_O = TMEM_P + NP * (BC / 2);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // exp reference may lag the max by 2^8
constexpr uint32_t IDESC_QK = idesc_bf16_f32(MR, BC, 0);  // K_j: K-major
constexpr uint32_t IDESC_PV = idesc_bf16_f32(MR, D, 1);   // V_j: MN-major
constexpr uint32_t NEG_INF_BITS = 0xff800000u;

struct Shared {
  uint64_t k_full[NK], k_empty[NK];
  uint64_t v_full[NV], v_empty[NV];
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

// K-major 128 x 128 bf16 tile held as two 128-byte-swizzled boxes of 64
// columns: k-step kk (16 columns) is box kk/4 at 32-byte step kk%4; 8-row
// groups are 1024 bytes apart.
__device__ __forceinline__ uint64_t kmajor_base(uint32_t tile) {
  return smem_desc_sw128(tile, 16u, 1024u);
}
__device__ __forceinline__ constexpr uint64_t kmajor_step(int kk) {
  return (uint64_t)(((uint32_t)(kk >> 2) * HALF_BYTES + (uint32_t)(kk & 3) * 32u) >> 4);
}
// MN-major value tile: rows are keys (64 values per swizzled 128-byte row),
// 8-key groups 1024 bytes apart, the second 64-value half 16 KB further;
// k-step kk (16 keys) starts 2048 bytes further.
__device__ __forceinline__ uint64_t vmajor_base(uint32_t tile) {
  return smem_desc_sw128(tile, HALF_BYTES, 1024u);
}
__device__ __forceinline__ constexpr uint64_t vmajor_step(int kk) {
  return (uint64_t)(((uint32_t)kk * 2048u) >> 4);
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

// P = exp2(s * sl2 - ref) for one 32-key chunk as 16 packed bf16 pairs, with
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
    pk[i] = pack_bf16x2(p0, p1);
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

// PH: per-head decisions (each query head decides alone; the block's values
// are read when any head keeps it), compiled separately from the group-AND
// kernel.
template <bool PH>
__global__ void __launch_bounds__(NT, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Shared &sh = *reinterpret_cast<Shared *>(smem_raw + SMEM_TILES);
  const uint32_t base = smem_u32(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (base & 1023u) {  // the swizzled layouts need a 1024-byte aligned base
    if (tid == 0) atomicOr(a.err, kErrLayout);
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
  // Bitmap words of this unit (group mode) or of head lane g (per-head mode).
  auto bits_of = [&](int g) -> uint32_t * {
    if (!a.bits) return nullptr;
    return PH ? a.bits + ((size_t)(b * a.Hq + hk * G + g) * a.n_splits + sp) * a.words
              : a.bits + (size_t)unit * a.words;
  };
  volatile int *abort = &sh.abort;

  if (nb == 0) {  // empty split: no key, zero weight in the merge
    if (a.margin)
      for (int j = tid; j < a.bps; j += NT) a.margin[(size_t)unit * a.bps + j] = NAN;
    if (a.stats_only) return;
    for (int idx = tid; idx < G * D; idx += NT) {
      const size_t row = (size_t)(b * a.Hq + hk * G + idx / D) * a.n_splits + sp;
      a.o_part[row * D + idx % D] = 0.f;
      if (idx % D == 0) a.lse_part[row] = -INFINITY;
    }
    for (int idx = tid; idx < (PH ? G : 1) * a.words; idx += NT)
      bits_of(idx / a.words)[idx % a.words] = 0u;
    return;
  }

  // Q tile (A operand of Q.K^T): row g < G = query head hk*G + g, other rows
  // zero; K-major, two 128-byte-swizzled boxes of 64 columns (16-byte chunk c
  // of row r sits at chunk position c ^ (r % 8)).
  {
    const __nv_bfloat16 *qg = (const __nv_bfloat16 *)a.q + (size_t)(b * a.Hq + hk * G) * D;
    for (int idx = tid; idx < MR * (D / 8); idx += NT) {  // one 16-byte chunk each
      const int r = idx / (D / 8), cc = idx % (D / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < G) v = *reinterpret_cast<const uint4 *>(qg + (size_t)r * D + cc * 8);
      const int box = cc >> 3, c = cc & 7;
      st_shared_v4(base + SMEM_Q + box * HALF_BYTES + r * 128 + ((c ^ (r & 7)) * 16), v.x, v.y,
                   v.z, v.w);
    }
    fence_proxy_async_smem();  // visible to the tensor core
  }
  if (tid == 0) {
    for (int i = 0; i < NK; ++i) {
      mbar_init(smem_u32(&sh.k_full[i]), 1);
      mbar_init(smem_u32(&sh.k_empty[i]), 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(smem_u32(&sh.v_full[i]), 1);
      mbar_init(smem_u32(&sh.v_empty[i]), 1);
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
      mbar_init(smem_u32(&sh.dec_empty[i]), 2);  // V producer and P.V issuer
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
      // Drain: the last load issued into each slot has landed before exit.
      for (int s = 0; s < NK && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / NK) * NK;
        mbar_wait_drain(smem_u32(&sh.k_full[s]), (last / NK) & 1);
      }
    }
  } else if (warp == WARP_V) {
    // ---------------------------------------------------------- V producer --
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
        const int s = vi % NV;
        if (vi >= NV &&
            !mbar_wait(smem_u32(&sh.v_empty[s]), ((vi / NV) - 1) & 1, abort, a.err, kErrTimeout))
          break;
        const uint32_t dst = base + SMEM_V + s * TILE_BYTES;
        const int key0 = (j0 + j) * BC;
        mbar_expect_tx(smem_u32(&sh.v_full[s]), TILE_BYTES);
        tma_load_3d(dst, &tm_v, smem_u32(&sh.v_full[s]), 0, key0, zkv, pol);
        tma_load_3d(dst + HALF_BYTES, &tm_v, smem_u32(&sh.v_full[s]), 64, key0, zkv, pol);
        ++vi;
      }
      for (int s = 0; s < NV && s < vi; ++s) {
        const int last = s + ((vi - 1 - s) / NV) * NV;
        mbar_wait_drain(smem_u32(&sh.v_full[s]), (last / NV) & 1);
      }
    }
  } else if (warp == WARP_QK) {
    // -------------------------------------------------------- Q.K^T issuer --
    if (lane == 0) {
      const uint64_t qdesc = kmajor_base(base + SMEM_Q);
      for (int j = 0; j < nb; ++j) {
        const int s = j % NK, sb = j % NS;
        if (!mbar_wait(smem_u32(&sh.k_full[s]), (j / NK) & 1, abort, a.err, kErrTimeout)) break;
        // S buffer sb is free once the softmax warp has read block j - NS.
        if (j >= NS && !mbar_wait(smem_u32(&sh.s_free[sb]), ((j / NS) - 1) & 1, abort, a.err,
                                  kErrTimeout))
          break;
        fence_after_sync();
        const uint64_t kd = kmajor_base(base + SMEM_K + s * TILE_BYTES);
        const uint32_t d_s = tmem + sb * BC;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(d_s, qdesc + kmajor_step(kk), kd + kmajor_step(kk), IDESC_QK, kk > 0);
        mma_commit(smem_u32(&sh.s_full[sb]));
        mma_commit(smem_u32(&sh.k_empty[s]));
      }
    }
  } else if (warp == WARP_PV) {
    // ---------------------------------------------------------- P.V issuer --
    if (lane == 0) {
      int kc = 0, vi = 0;
      for (int j = 0; j < nb && !*abort; ++j) {
        if (!mbar_wait(smem_u32(&sh.dec_full[j % NDEC]), (j / NDEC) & 1, abort, a.err,
                       kErrTimeout))
          break;
        const int keep = sh.dec[j % NDEC];
        mbar_arrive(smem_u32(&sh.dec_empty[j % NDEC]));
        if (!keep) continue;
        const int pb = kc % NP, vs = vi % NV;
        if (!mbar_wait(smem_u32(&sh.p_full[pb]), (kc / NP) & 1, abort, a.err, kErrTimeout) ||
            !mbar_wait(smem_u32(&sh.v_full[vs]), (vi / NV) & 1, abort, a.err, kErrTimeout))
          break;
        fence_after_sync();
        // P (bf16 pairs): keys [0,128) in the 64 columns of P buffer pb.
        const uint32_t pt = tmem + TMEM_P + pb * (BC / 2);
        const uint64_t vd = vmajor_base(base + SMEM_V + vs * TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < BC / 16; ++kk)
          mma_bf16_ts(tmem + TMEM_O, pt + kk * 8, vd + vmajor_step(kk), IDESC_PV,
                      (kc > 0 || kk > 0) ? 1u : 0u);
        mma_commit(smem_u32(&sh.v_empty[vs]));
        mma_commit(smem_u32(&sh.p_free[pb]));
        mma_commit(smem_u32(&sh.pv_done[kc & 1]));
        ++kc;
        ++vi;
      }
    }
  } else {
    // ------------------------------------------------------------- softmax --
    // Lane g < G: head g's row (TMEM lane g) over the block's 128 keys.
    const bool head = lane < G;
    uint32_t *bits = bits_of(PH ? (head ? lane : 0) : 0);
    const float sl2 = a.scale * kLog2e;   // raw score -> log2 units
    const float c2 = a.ln_lambda * kLog2e;  // ln(lambda) in log2 units
    float m2 = -INFINITY;                 // running max of the split (log2 units)
    float mref = -INFINITY;               // exp reference (log2 units)
    float l = 0.f;                        // row sum relative to mref
    int kc = 0;                           // kept blocks
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
      // skip_h: this head leaves the block out; skip: nobody needs its values.
      const bool vote = !head || diff < c2;
      const bool skip_h = a.stats_only || (PH ? vote : __all_sync(0xffffffffu, vote));
      const bool skip = PH ? __all_sync(0xffffffffu, skip_h) : skip_h;
      if (a.margin) {
        // The block statistic: max over the heads of rowmax - m_new, where
        // rowmax - m_new = min(rowmax - m_old, 0) (log2 units).
        float st = (head && mt != -INFINITY) ? fminf(diff, 0.f) : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) st = fmaxf(st, __shfl_xor_sync(0xffffffffu, st, o));
        if (lane == 0) a.margin[(size_t)unit * a.bps + j] = st * kLn2;
      }
      if (lane == 0) {
        // On a timeout the abort flag is raised and every later wait fails.
        if (j < NDEC || mbar_wait(smem_u32(&sh.dec_empty[j % NDEC]), ((j / NDEC) - 1) & 1,
                                  abort, a.err, kErrTimeout)) {
          sh.dec[j % NDEC] = skip ? 0 : 1;
          mbar_arrive(smem_u32(&sh.dec_full[j % NDEC]));
        }
      }
      if (PH ? head : lane == 0) {
        if (skip_h) word |= 1u << (j & 31);
        if (!a.stats_only && ((j & 31) == 31 || j == nb - 1)) {
          bits[j >> 5] = word;
          word = 0;
        }
      }
      // The running max advances on every block (a skipped block leaves it
      // unchanged unless the statistics mode forced the skip).
      const float mnew = fmaxf(m2, pm2);
      m2 = mnew;
      if (skip) continue;
      bool rescale = false;
      float alpha = 1.f;
      if (!skip_h) {  // (per-head mode: a head that leaves the block out keeps its state)
        if (mref == -INFINITY) {
          mref = mnew;
        } else if (mnew > mref + kRescaleLog2) {
          alpha = ex2(mref - mnew);
          mref = mnew;
          rescale = true;
        }
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
      // A head that leaves the block out gets P = exp2(-inf) = 0 on its row.
      const float nref = skip_h ? -INFINITY : -mref;
      const uint64_t sl2x2 = f2(sl2, sl2), negref2 = f2(nref, nref);
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

    // ---- epilogue: O_s = O / l and LSE_s = ref + ln l per head ---------------
    if (PH ? head : lane == 0) {
      if (!a.stats_only)
        for (int w = ((nb - 1) >> 5) + 1; w < a.words; ++w) bits[w] = 0u;
    }
    if (lane == 0) {
      if (a.margin)
        for (int j = nb; j < a.bps; ++j) a.margin[(size_t)unit * a.bps + j] = NAN;
    }
    // (Statistics mode: every block was treated as skipped, kc == 0, no output.)
    if (ok && kc > 0)
      ok = mbar_wait_warp(smem_u32(&sh.pv_done[(kc - 1) & 1]), ((kc - 1) >> 1) & 1, abort, a.err,
                          kErrTimeout);
    if (ok && !a.stats_only) {
      fence_after_sync();
      const float inv = 1.f / l;
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

cudaError_t launch_decode_bf16(const DecodeArgs &a, cudaStream_t s) {
  CUtensorMap mk, mv;
  // [B*Hkv, L, 128] bf16 with the caller's row stride; boxes of 64 columns x
  // 128 keys; keys past L read as zero (and are masked).
  if (!make_map_bf16_3d(&mk, a.k, D, a.k_row_stride, a.L, a.B * a.Hkv, BC) ||
      !make_map_bf16_3d(&mv, a.v, D, a.v_row_stride, a.L, a.B * a.Hkv, BC))
    return cudaErrorInvalidValue;
  auto kernel = a.per_head ? decode_tc_kernel<true> : decode_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  const long units = (long)a.B * a.Hkv * a.n_splits;
  kernel<<<(unsigned)units, NT, SMEM_ALLOC, s>>>(mk, mv, a);
  return cudaGetLastError();
}

}  // namespace attn_skip
