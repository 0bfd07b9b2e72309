// Absorbed-MLA split-KV decode with softmax-threshold block skipping:
// 128 query heads share one latent cache row of 576 bf16 (512 latent + 64
// rope); the values are the first 512 columns of the same rows.  Bc = 64.
//
// The BLASST page notes that MLA decode can be compute-bound (section
// "Decode 内核：砍带宽", last paragraph), so here a skipped block saves the
// exponentials and the P.V product; its value bytes are the key bytes already
// staged for Q.K^T.  The 128 heads form one M = 128 tcgen05 tile.
//
// The latent values are large (the cache rows themselves), so P.V runs in
// fp16 rather than bf16: P is rounded to fp16 (values <= 2^8) and, once Q.K^T
// of a kept block has read it, the CTA's half of the value columns is
// converted in place from bf16 to fp16 (exact), for a 2^-11 rather than
// 2^-8 relative rounding of P.
//
// TMEM holds 512 fp32 columns and O alone is 128 x 512, so each (sequence,
// split) runs as two CTAs that own output columns [0,256) and [256,512).  Both
// compute the same S = Q K^T with the same instruction sequence, so their
// scores, decisions, running maxima and row sums are bit-identical; the CTA
// of half 0 writes the skip bits and the LSE.
//
// Per CTA (224 threads): warps 0-3 softmax (thread i owns head i = TMEM lane
// i), warp 4 TMA producer, warp 5 Q.K^T issuer, warp 6 P.V issuer.  With
// separate issuing threads a kept block's P.V, and with it the release of its
// latent slot, never waits behind the next block's Q.K^T (which waits for
// that block's load).
// Shared memory: Q dims [0,320) as five 128-byte-swizzled 64-column boxes
// (80 KB); a two-slot ring of latent blocks, each nine 64 x 64 boxes (72 KB).
// TMEM: Q dims [320,576) [0,128) (two bf16 per column, the MMA A operand),
// two S buffers [128,192) and [192,256) (P is written over its S), O half
// [256,512).
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"
#include "tc_common.cuh"

namespace attn_skip {
namespace {

using namespace tc;

constexpr int DK = 576, DV = 512, DVH = 256;
constexpr int H = 128;            // query heads (M)
constexpr int BN = 64;            // keys per block
constexpr int NCH = DK / 64;      // 64-column chunks of a latent row
constexpr int NCH_S = 5;          // chunks of Q kept in shared memory
constexpr int NCH_T = NCH - NCH_S;  // chunks of Q kept in TMEM
constexpr int NTHREADS = 224;
constexpr int WARP_TMA = 4, WARP_MMA = 5, WARP_PV = 6;
constexpr uint32_t QCH_BYTES = H * 64 * 2;   // 16 KB
constexpr uint32_t KCH_BYTES = BN * 64 * 2;  // 8 KB
constexpr uint32_t KBLK_BYTES = NCH * KCH_BYTES;  // 72 KB
constexpr uint32_t SMEM_Q = 0;
constexpr uint32_t SMEM_K = SMEM_Q + NCH_S * QCH_BYTES;  // 80 KB
constexpr uint32_t SMEM_TILES = SMEM_K + 2 * KBLK_BYTES;  // 224 KB
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_QT = 0, TMEM_S = 128, TMEM_O = 256;
constexpr int NDEC = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t IDESC_QK = idesc_bf16_f32(H, BN, 0);   // B = latent block, K-major
constexpr uint32_t IDESC_PV = idesc_f16_f32(H, DVH, 1);   // fp16 P x fp16 V (MN-major)
constexpr uint32_t NEG_INF_BITS = 0xff800000u;

struct Shared {
  uint64_t q_full, qt_ready;
  uint64_t k_full[2], k_empty[2];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2], pv_done[2];
  uint64_t dec_full[NDEC];
  uint64_t vote_full[2];
  int dec[NDEC];
  int vote[2][4];
  float wstat[2][4];  // statistics mode: per warp, max over its heads of rowmax - m_new
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t SMEM_ALLOC = SMEM_TILES + ((sizeof(Shared) + 127) / 128) * 128;
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");

__global__ void __launch_bounds__(NTHREADS, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_kv, const DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Shared &sh = *reinterpret_cast<Shared *>(smem_raw + SMEM_TILES);
  const uint32_t base = smem_u32(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (base & 1023u) {
    if (tid == 0) atomicOr(a.err, kErrLayout);
    return;
  }
  const int half = blockIdx.x & 1;
  const int us = blockIdx.x >> 1;  // b * n_splits + split
  const int sp = us % a.n_splits, b = us / a.n_splits;
  const int j0 = (int)((long)sp * a.n_b / a.n_splits);
  const int j1 = (int)((long)(sp + 1) * a.n_b / a.n_splits);
  const int nb = j1 - j0;
  uint32_t *bits = a.bits ? a.bits + (size_t)us * a.words : nullptr;
  volatile int *abort = &sh.abort;

  // Statistics mode: the half-0 CTA computes the statistics alone.
  if (a.stats_only && half == 1) return;
  if (nb == 0) {  // empty split
    if (a.margin)
      for (int j = tid; j < a.bps; j += NTHREADS) a.margin[(size_t)us * a.bps + j] = NAN;
    if (a.stats_only) return;
    for (int idx = tid; idx < H * DVH; idx += NTHREADS) {
      const int hh = idx / DVH, e = idx % DVH;
      const size_t row = (size_t)(b * a.Hq + hh) * a.n_splits + sp;
      a.o_part[row * DV + half * DVH + e] = 0.f;
      if (half == 0 && e == 0) a.lse_part[row] = -INFINITY;
    }
    if (half == 0)
      for (int w = tid; w < a.words; w += NTHREADS) bits[w] = 0u;
    return;
  }

  if (tid == 0) {
    mbar_init(smem_u32(&sh.q_full), 1);
    mbar_init(smem_u32(&sh.qt_ready), 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh.k_full[i]), 1);
      mbar_init(smem_u32(&sh.k_empty[i]), 2);  // Q.K^T commit + P.V commit (or skip)
      mbar_init(smem_u32(&sh.s_full[i]), 1);
      mbar_init(smem_u32(&sh.s_free[i]), 1);
      mbar_init(smem_u32(&sh.p_full[i]), 4);
      mbar_init(smem_u32(&sh.pv_done[i]), 1);
      mbar_init(smem_u32(&sh.vote_full[i]), 4);
    }
    for (int i = 0; i < NDEC; ++i) mbar_init(smem_u32(&sh.dec_full[i]), 1);
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == WARP_MMA) tmem_alloc(smem_u32(&sh.tmem_base), TMEM_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sh.tmem_base;
  const uint32_t kslot1 = base + SMEM_K + KBLK_BYTES;  // also stages the TMEM part of Q

  if (warp == WARP_TMA) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_kv);
      const uint64_t pol_q = policy_evict_first(), pol_kv = policy_evict_last();
      // Q: chunks [0,5) to their shared-memory home, chunks [5,9) staged in slot 1.
      mbar_expect_tx(smem_u32(&sh.q_full), NCH * QCH_BYTES);
      for (int c = 0; c < NCH; ++c) {
        const uint32_t dst = c < NCH_S ? base + SMEM_Q + c * QCH_BYTES
                                       : kslot1 + (c - NCH_S) * QCH_BYTES;
        tma_load_3d(dst, &tm_q, smem_u32(&sh.q_full), c * 64, 0, b, pol_q);
      }
      int issued = 0;
      for (int j = 0; j < nb && !*abort; ++j) {
        const int s = j & 1;
        // Slot 1 is free once the TMEM part of Q has been copied out of it.
        if (j == 1 && !mbar_wait(smem_u32(&sh.qt_ready), 0, abort, a.err, kErrTimeout)) break;
        if (j >= 2 &&
            !mbar_wait(smem_u32(&sh.k_empty[s]), ((j >> 1) - 1) & 1, abort, a.err, kErrTimeout))
          break;
        const uint32_t dst = base + SMEM_K + s * KBLK_BYTES;
        mbar_expect_tx(smem_u32(&sh.k_full[s]), KBLK_BYTES);
        for (int c = 0; c < NCH; ++c)
          tma_load_3d(dst + c * KCH_BYTES, &tm_kv, smem_u32(&sh.k_full[s]), c * 64,
                      (j0 + j) * BN, b, pol_kv);
        ++issued;
      }
      mbar_wait_drain(smem_u32(&sh.q_full), 0);
      for (int s = 0; s < 2 && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / 2) * 2;
        mbar_wait_drain(smem_u32(&sh.k_full[s]), (last >> 1) & 1);
      }
    }
  } else if (warp == WARP_MMA) {
    // -------------------------------------------------------- Q.K^T issuer --
    if (lane == 0) {
      bool ok = mbar_wait(smem_u32(&sh.q_full), 0, abort, a.err, kErrTimeout) &&
                mbar_wait(smem_u32(&sh.qt_ready), 0, abort, a.err, kErrTimeout);
      fence_after_sync();
      for (int j = 0; ok && j < nb; ++j) {
        const int s = j & 1;
        if (!mbar_wait(smem_u32(&sh.k_full[s]), (j >> 1) & 1, abort, a.err, kErrTimeout)) break;
        if (j >= 2 && !mbar_wait(smem_u32(&sh.s_free[s]), ((j >> 1) - 1) & 1, abort, a.err,
                                 kErrTimeout))
          break;
        fence_after_sync();
        const uint32_t kt = base + SMEM_K + s * KBLK_BYTES;
        const uint32_t d = tmem + TMEM_S + s * BN;
#pragma unroll 1
        for (int c = 0; c < NCH; ++c) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // B: 64 keys x 16 dims of chunk c (K-major, 32-byte step, 8-row groups 1 KB apart)
            const uint64_t bd = smem_desc_sw128(kt + c * KCH_BYTES + kk * 32, 16, 1024);
            const uint32_t acc = (c > 0 || kk > 0) ? 1u : 0u;
            if (c < NCH_S)
              mma_bf16_ss(d, smem_desc_sw128(base + SMEM_Q + c * QCH_BYTES + kk * 32, 16, 1024),
                          bd, IDESC_QK, acc);
            else
              mma_bf16_ts(d, tmem + TMEM_QT + (c - NCH_S) * 32 + kk * 8, bd, IDESC_QK, acc);
          }
        }
        mma_commit(smem_u32(&sh.s_full[s]));
        mma_commit(smem_u32(&sh.k_empty[s]));  // this block's Q.K^T has read the slot
      }
    }
  } else if (warp == WARP_PV) {
    // ---------------------------------------------------------- P.V issuer --
    if (lane == 0) {
      int kc = 0;
      for (int i = 0; i < nb && !*abort; ++i) {
        if (!mbar_wait(smem_u32(&sh.dec_full[i % NDEC]), (i / NDEC) & 1, abort, a.err,
                       kErrTimeout))
          break;
        const int s = i & 1;
        if (!sh.dec[i % NDEC]) {
          mbar_arrive(smem_u32(&sh.k_empty[s]));  // skipped: no value read
          continue;
        }
        if (!mbar_wait(smem_u32(&sh.p_full[kc & 1]), (kc >> 1) & 1, abort, a.err, kErrTimeout))
          break;
        fence_after_sync();
        // O_half += P (TMEM, 64 keys = 32 columns) x V_half (MN-major: keys are the
        // 128-byte rows of chunks 4*half..4*half+3, 8 KB apart).
        const uint32_t vt = base + SMEM_K + s * KBLK_BYTES + half * 4 * KCH_BYTES;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_bf16_ts(tmem + TMEM_O, tmem + TMEM_S + s * BN + kk * 8,
                      smem_desc_sw128(vt + kk * 2048, KCH_BYTES, 1024), IDESC_PV,
                      (kc > 0 || kk > 0) ? 1u : 0u);
        mma_commit(smem_u32(&sh.s_free[s]));
        mma_commit(smem_u32(&sh.pv_done[kc & 1]));
        mma_commit(smem_u32(&sh.k_empty[s]));
        ++kc;
      }
    }
  } else {
    // ------------------------------------------------------------ softmax --
    const int r = tid;  // head == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const float sl2 = a.scale * kLog2e;
    const float c2 = a.ln_lambda * kLog2e;
    bool ok = mbar_wait_warp(smem_u32(&sh.q_full), 0, abort, a.err, kErrTimeout);
    if (ok) {
      // Copy Q dims [320,576) of head r from the staging slot into TMEM.
#pragma unroll 1
      for (int c = 0; c < NCH_T; ++c) {
        const uint32_t rowp = kslot1 + c * QCH_BYTES + (uint32_t)r * 128u;
        uint32_t w[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint32_t x0, x1, x2, x3;
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                       : "r"(rowp + ((uint32_t)(q ^ (r & 7)) << 4)));
          w[4 * q] = x0;
          w[4 * q + 1] = x1;
          w[4 * q + 2] = x2;
          w[4 * q + 3] = x3;
        }
        tmem_st32(lane_base + TMEM_QT + c * 32, w);
      }
      tmem_wait_st();
    }
    fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh.qt_ready));

    float m2 = -INFINITY, mref = -INFINITY, l = 0.f;
    int kc = 0;
    uint32_t word = 0;
    for (int j = 0; ok && j < nb; ++j) {
      const int s = j & 1;
      if (!mbar_wait_warp(smem_u32(&sh.s_full[s]), (j >> 1) & 1, abort, a.err, kErrTimeout)) {
        ok = false;
        break;
      }
      fence_after_sync();
      const uint32_t sa = lane_base + TMEM_S + s * BN;
      uint32_t x[32], y[32];
      tmem_ld32(sa, x);
      tmem_ld32(sa + 32, y);
      tmem_wait_ld_regs(x);
      tmem_wait_ld_regs(y);
      const int keys = min(BN, a.L - (j0 + j) * BN);
      if (keys < BN) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (i >= keys) x[i] = NEG_INF_BITS;
          if (i + 32 >= keys) y[i] = NEG_INF_BITS;
        }
      }
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; i += 2)
        mt = fmax3(mt, fmaxf(__uint_as_float(x[i]), __uint_as_float(x[i + 1])),
                   fmaxf(__uint_as_float(y[i]), __uint_as_float(y[i + 1])));
      const float mt2 = mt * sl2;
      const float mnew = fmaxf(m2, mt2);
      const float diff = (mt == -INFINITY) ? -INFINITY : mt2 - mnew;
      const bool vote = diff < c2;  // Eq. 5; all 128 heads must agree
      const unsigned all = __all_sync(0xffffffffu, vote);
      const int vb = j & 1;
      if (lane == 0) sh.vote[vb][warp] = (int)all;
      if (a.margin) {  // the block statistic: max over the heads of rowmax - m_new
        float st = diff;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) st = fmaxf(st, __shfl_xor_sync(0xffffffffu, st, o));
        if (lane == 0) sh.wstat[vb][warp] = st;
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.vote_full[vb]));
      if (!mbar_wait_warp(smem_u32(&sh.vote_full[vb]), (j >> 1) & 1, abort, a.err,
                          kErrTimeout)) {
        ok = false;
        break;
      }
      const bool skip =
          a.stats_only || (sh.vote[vb][0] && sh.vote[vb][1] && sh.vote[vb][2] && sh.vote[vb][3]);
      if (a.margin && tid == 0 && half == 0)
        a.margin[(size_t)us * a.bps + j] =
            fmaxf(fmaxf(sh.wstat[vb][0], sh.wstat[vb][1]), fmaxf(sh.wstat[vb][2], sh.wstat[vb][3])) *
            kLn2;
      if (tid == 0) {
        if (skip) {
          fence_after_sync();
          fence_before_sync();
          mbar_arrive(smem_u32(&sh.s_free[s]));
        }
        sh.dec[j % NDEC] = skip ? 0 : 1;
        mbar_arrive(smem_u32(&sh.dec_full[j % NDEC]));
        if (half == 0 && !a.stats_only) {
          if (skip) word |= 1u << (j & 31);
          if ((j & 31) == 31 || j == nb - 1) {
            bits[j >> 5] = word;
            word = 0;
          }
        }
      }
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
      const uint64_t sl2x2 = f2(sl2, sl2), negref2 = f2(-mref, -mref);
      uint64_t acc2 = f2(0.f, 0.f);
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float e0, e1;
        f2_split(f2_fma(f2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1])), sl2x2,
                        negref2),
                 e0, e1);
        const float p0 = ex2(e0), p1 = ex2(e1);
        acc2 = f2_add(acc2, f2(p0, p1));
        pk[i] = pack_f16x2(p0, p1);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float e0, e1;
        f2_split(f2_fma(f2(__uint_as_float(y[2 * i]), __uint_as_float(y[2 * i + 1])), sl2x2,
                        negref2),
                 e0, e1);
        const float p0 = ex2(e0), p1 = ex2(e1);
        acc2 = f2_add(acc2, f2(p0, p1));
        pk[16 + i] = pack_f16x2(p0, p1);
      }
      tmem_st32(sa, pk);  // P over 64 keys -> the first 32 columns of S_j
      // This CTA's value columns of the block (chunks 4*half..4*half+3, 32 KB),
      // bf16 -> fp16 in place; Q.K^T of this block has completed (s_full).
      {
        const uint32_t vt = base + SMEM_K + s * KBLK_BYTES + half * 4 * KCH_BYTES;
#pragma unroll 4
        for (int i = 0; i < (4 * KCH_BYTES / 16) / 128; ++i) {
          const uint32_t addr = vt + (uint32_t)(tid + 128 * i) * 16u;
          uint32_t w0, w1, w2, w3;
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                       : "r"(addr));
          st_shared_v4(addr, bf16x2_to_f16x2(w0), bf16x2_to_f16x2(w1), bf16x2_to_f16x2(w2),
                       bf16x2_to_f16x2(w3));
        }
        fence_proxy_async_smem();  // generic writes -> the tensor cores' reads
      }
      tmem_wait_st();
      float s0, s1;
      f2_split(acc2, s0, s1);
      l = l * alpha + (s0 + s1);
      if (__any_sync(0xffffffffu, rescale) && kc >= 1) {
        if (!mbar_wait_warp(smem_u32(&sh.pv_done[(kc - 1) & 1]), ((kc - 1) >> 1) & 1, abort,
                            a.err, kErrTimeout)) {
          ok = false;
          break;
        }
        fence_after_sync();
#pragma unroll 1
        for (int cc = 0; cc < DVH / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(lane_base + TMEM_O + cc * 32, o);
          tmem_wait_ld_regs(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(lane_base + TMEM_O + cc * 32, o);
        }
        tmem_wait_st();
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.p_full[kc & 1]));
      ++kc;
    }

    // ---- epilogue ------------------------------------------------------------
    if (tid == 0 && half == 0) {
      if (!a.stats_only)
        for (int w = ((nb - 1) >> 5) + 1; w < a.words; ++w) bits[w] = 0u;
      if (a.margin)
        for (int j = nb; j < a.bps; ++j) a.margin[(size_t)us * a.bps + j] = NAN;
    }
    // (Statistics mode: every block was treated as skipped, kc == 0, no output.)
    if (ok && kc > 0)
      ok = mbar_wait_warp(smem_u32(&sh.pv_done[(kc - 1) & 1]), ((kc - 1) >> 1) & 1, abort,
                          a.err, kErrTimeout);
    if (ok && !a.stats_only) {
      fence_after_sync();
      const float inv = 1.f / l;
      const size_t row = (size_t)(b * a.Hq + r) * a.n_splits + sp;
      float *orow = a.o_part + row * DV + half * DVH;
#pragma unroll 1
      for (int cc = 0; cc < DVH / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(lane_base + TMEM_O + cc * 32, o);
        tmem_wait_ld_regs(o);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 v;
          v.x = __uint_as_float(o[4 * q]) * inv;
          v.y = __uint_as_float(o[4 * q + 1]) * inv;
          v.z = __uint_as_float(o[4 * q + 2]) * inv;
          v.w = __uint_as_float(o[4 * q + 3]) * inv;
          *reinterpret_cast<float4 *>(orow + cc * 32 + 4 * q) = v;
        }
      }
      if (half == 0) a.lse_part[row] = mref * kLn2 + logf(l);
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

}  // namespace

cudaError_t launch_mla_decode(const DecodeArgs &a, cudaStream_t s) {
  // The three-CTA cluster kernel (mla_cluster.cu) computes Q.K^T once per key;
  // this two-CTA kernel serves the statistics mode and splits longer than the
  // cluster kernel's decision array.
  if (!a.stats_only && a.bps <= mla_cluster_max_bps()) return launch_mla_cluster(a, s);
  CUtensorMap mq, mkv;
  // [B, rows, 576] bf16, boxes of 64 columns x (H or BN) rows, 128-byte swizzle.
  if (!make_map_bf16_3d(&mq, a.q, DK, DK, H, a.B, H) ||
      !make_map_bf16_3d(&mkv, a.k, DK, DK, a.L, a.B, BN))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  const long ctas = 2L * a.B * a.n_splits;
  mla_decode_kernel<<<(unsigned)ctas, NTHREADS, SMEM_ALLOC, s>>>(mq, mkv, a);
  return cudaGetLastError();
}

}  // namespace attn_skip
