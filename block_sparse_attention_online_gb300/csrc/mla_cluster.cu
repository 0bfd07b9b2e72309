// Absorbed-MLA split-KV decode with softmax-threshold block skipping, as a
// cluster of three CTAs per (sequence, split): one scorer and two value CTAs.
//
// Method: the BLASST page, sections "BLASST 的判定准则" (Eq. 5) and "Decode 内核：
// 砍带宽" (MLA decode is compute-heavy, so a skipped block saves its
// exponentials and its P.V product).  128 query heads share one latent row of
// 576 bf16 (512 latent + 64 rope); the values are its first 512 columns.
//
// O (128 heads x 512 fp32) alone fills a CTA's TMEM, so the work is split by
// what each product needs:
//  * the scorer (cluster rank 0) holds Q in TMEM (latent dims 0-511, 256
//    columns) and shared memory (rope dims), streams the latent rows in
//    64-column chunks of 128 keys, and computes S = Q K^T once per 128 keys
//    (N = 128 products: the instruction count per key halves against N = 64);
//    its four softmax warps take the row maxima, the votes and the decision
//    of every 64-key block, and for a kept block write P (fp16) straight into
//    the two value CTAs' shared memory (distributed shared memory), with each
//    head's rescale factor;
//  * value CTA h (rank 1 + h) holds O[:, 256h:256h+256) in TMEM, loads only the
//    value columns [256h, 256h+256) of kept blocks (an L2 hit: the scorer has
//    just read the same rows), widens them to fp16 in place, and runs
//    O_h += P V_h (M = 128 heads, N = 256) from shared memory.
// The scorer's latent chunks are released as soon as its product has read
// them, so no value product holds the key stream.
//
// Hand-offs: a decision is one word per block in each value CTA (0 = not yet,
// 1 = skipped, 2 = kept), written with a relaxed remote store and polled (no
// ring: the array holds every block of a split); a kept block's P and the
// heads' rescale factors are staged in the scorer's shared memory and sent by
// one bulk copy per value CTA that completes on that CTA's p_full barrier
// (the scorer arms it remotely with the byte count); p_free (value CTA ->
// scorer, one arrival per value CTA after the product that read the slot
// completed) gives the slot back; the final row sums arrive by remote stores
// and fin_full.  P.V runs in fp16 (the latent values are the cache rows; P
// rounded to fp16, values <= 2^8 with the lazy rescale).
//
// Warps (384 threads in every CTA of the cluster):
//   scorer: 0-3 softmax (thread = head = TMEM lane), 4 TMA producer, 5 Q.K^T
//           issuer (allocates 512 TMEM columns);
//   value:  0-3 scale / epilogue (thread = head), 4 TMA producer of values,
//           5 P.V issuer (allocates 256 TMEM columns), 6 slot forwarder,
//           8-11 fp16 wideners.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"
#include "tc_common.cuh"

namespace attn_skip {
namespace {

using namespace tc;

constexpr int DK = 576, DV = 512, DVH = 256;
constexpr int H = 128;          // query heads (M)
constexpr int BN = 64;          // keys per block (the decision unit)
constexpr int DBN = 128;        // keys per S product (two blocks)
constexpr int GCH = 3;          // scorer: chunks per ring group (one barrier, 12 products)
constexpr int NG = 4;           // scorer: ring groups
constexpr int NC = NG * GCH;    // scorer: latent chunk ring (16 KB each)
constexpr int NST = 1;          // scorer: P staging buffers
constexpr int NV = 4;           // value CTA: value tiles (32 KB each)
constexpr int NPS = 4;          // value CTA: P slots (16 KB each)
constexpr int MAX_BPS = 2048;   // blocks per split the decision array holds
constexpr int NTHREADS = 384;
constexpr int WARP_TMA = 4, WARP_MMA = 5, WARP_FWD = 6, WARP_CV = 8;
constexpr uint32_t CH_BYTES = DBN * 64 * 2;   // 16 KB: 128 keys x 64 columns
constexpr uint32_t VCH_BYTES = BN * 64 * 2;   // 8 KB: 64 keys x 64 columns
constexpr uint32_t VT_BYTES = 4 * VCH_BYTES;  // 32 KB: a block's value half
constexpr uint32_t P_BYTES = H * BN * 2;      // 16 KB: 128 heads x 64 keys fp16
constexpr uint32_t PCOPY = P_BYTES + H * 4;    // a slot's contents: P, then the heads' rescale factors
constexpr uint32_t PX_BYTES = 17 * 1024;        // slot stride (1024-byte aligned for the swizzle)
// scorer layout
constexpr uint32_t SMEM_RING = 0;
constexpr uint32_t SMEM_ROPE = SMEM_RING + NC * CH_BYTES;  // 160 KB
constexpr uint32_t SMEM_STAGE = SMEM_ROPE + CH_BYTES;       // 176 KB
constexpr uint32_t SMEM_FIN = SMEM_STAGE + NST * PX_BYTES;  // 128 row sums (fp32)
constexpr uint32_t SCORER_TILES = SMEM_FIN + H * 4;
// value CTA layout
constexpr uint32_t SMEM_V = 0;
constexpr uint32_t SMEM_P = SMEM_V + NV * VT_BYTES;         // 128 KB: slots of PX_BYTES
constexpr uint32_t SMEM_DEC = SMEM_P + NPS * PX_BYTES;      // decision words
constexpr uint32_t VALUE_TILES = SMEM_DEC + MAX_BPS * 4;
constexpr uint32_t SMEM_TILES = SCORER_TILES > VALUE_TILES ? SCORER_TILES : VALUE_TILES;
constexpr uint32_t TMEM_Q = 0, TMEM_S = 256;   // scorer: Q [0,256), two S buffers [256,512)
constexpr uint32_t TMEM_O = 0;                 // value CTA: O half [0,256)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t IDESC_QK128 = idesc_bf16_f32(H, DBN, 0);
constexpr uint32_t IDESC_QK64 = idesc_bf16_f32(H, BN, 0);
constexpr uint32_t IDESC_PV = idesc_f16_f32(H, DVH, 1);  // fp16 P x fp16 V (MN-major)
constexpr uint32_t NEG_INF_BITS = 0xff800000u;
constexpr int kVoteBarrier = 1, kStageBarrier = 2, kFailBarrier = 3;
static_assert(SMEM_STAGE % 1024 == 0 && SMEM_P % 1024 == 0 && PX_BYTES % 1024 == 0 &&
                  PCOPY <= PX_BYTES && PCOPY % 16 == 0,
              "P slots on 1024-byte boundaries; bulk copies of whole 16-byte units");

struct Shared {
  // scorer
  uint64_t g_full[NG], g_empty[NG];
  uint64_t q_ready, rope_full;
  uint64_t s_full[2], s_free[2];
  uint64_t p_free[NPS];
  // value CTA
  uint64_t v_full[NV], v_empty[NV], v_conv[NV];
  uint64_t p_full[NPS], p_ok[NPS], pv_done[NPS];
  uint64_t fin_full;
  __align__(16) float fin_l[H];  // a bulk copy's destination
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t SMEM_ALLOC = SMEM_TILES + ((sizeof(Shared) + 127) / 128) * 128;
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");

// ------------------------------------------------------------- cluster --
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of this CTA's shared-memory location `a` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t remote(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// A decision word: one relaxed store, read by polling (no ordering with
// anything else is needed, and a release would wait for every earlier
// store of the thread).
__device__ __forceinline__ void st_remote_relaxed_u32(uint32_t a, uint32_t x) {
  asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(x) : "memory");
}
__device__ __forceinline__ unsigned ld_relaxed_u32(uint32_t a) {
  unsigned v;
  asm volatile("ld.relaxed.cluster.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
// Bulk copy of `bytes` (a multiple of 16, both ends 16-byte aligned) from this
// CTA's shared memory into another CTA's, completing on that CTA's barrier.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_cluster, uint32_t src,
                                                     uint32_t bytes, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst_cluster),
      "r"(src), "r"(bytes), "r"(bar_cluster)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed bulk groups of this thread still read their source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void arrive_remote(uint32_t bar_cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   bar_cluster_addr)
               : "memory");
}
// mbarrier wait whose phase is completed by arrivals from other CTAs of the
// cluster: the acquire is at cluster scope.  Bounded like mbar_wait.
__device__ __forceinline__ bool try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool wait_cluster(uint32_t bar, uint32_t parity, volatile int *abort,
                                             unsigned *err) {
  if (try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (try_wait_cluster(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *abort = 1;
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_cluster_warp(uint32_t bar, uint32_t parity,
                                                  volatile int *abort, unsigned *err) {
  return __all_sync(0xffffffffu, wait_cluster(bar, parity, abort, err));
}
// The decision of block j once the scorer has published it (bounded): 1 =
// skipped, 2 = kept, 0 = gave up.
__device__ __forceinline__ unsigned wait_decision(uint32_t dec_words, int j, volatile int *abort,
                                                  unsigned *err) {
  const uint32_t a = dec_words + 4u * (uint32_t)j;
  unsigned v = ld_relaxed_u32(a);
  if (v) return v;
  const uint64_t t0 = globaltimer();
  while (true) {
    v = ld_relaxed_u32(a);
    if (v) return v;
    if (*abort) return 0u;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *abort = 1;
      atomicOr(err, kErrTimeout);
      return 0u;
    }
  }
}

__global__ void __launch_bounds__(NTHREADS, 1)
    mla_cluster_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_kv128,
                       const __grid_constant__ CUtensorMap tm_kv64, const DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Shared &sh = *reinterpret_cast<Shared *>(smem_raw + SMEM_TILES);
  const uint32_t base = smem_u32(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const bool scorer = rank == 0;
  const int half = (int)rank - 1;
  const int us = (int)(blockIdx.x / 3);  // b * n_splits + split
  const int sp = us % a.n_splits, b = us / a.n_splits;
  const int j0 = (int)((long)sp * a.n_b / a.n_splits);
  const int j1 = (int)((long)(sp + 1) * a.n_b / a.n_splits);
  const int nb = j1 - j0;
  const int ndb = (nb + 1) / 2;
  volatile int *abort = &sh.abort;
  const bool aligned = (base & 1023u) == 0;  // the same in every CTA of the launch

  if (tid == 0 && aligned) {
    for (int i = 0; i < NG; ++i) {
      mbar_init(smem_u32(&sh.g_full[i]), 1);
      mbar_init(smem_u32(&sh.g_empty[i]), 1);
    }
    mbar_init(smem_u32(&sh.q_ready), 4);
    mbar_init(smem_u32(&sh.rope_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh.s_full[i]), 1);
      mbar_init(smem_u32(&sh.s_free[i]), 4);
    }
    for (int i = 0; i < NPS; ++i) {
      mbar_init(smem_u32(&sh.p_free[i]), 2);  // both value CTAs
      mbar_init(smem_u32(&sh.p_full[i]), 1);  // armed here (expect_tx), completed by the bulk copy
      mbar_init(smem_u32(&sh.p_ok[i]), 4);    // the four scale warps
      mbar_init(smem_u32(&sh.pv_done[i]), 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(smem_u32(&sh.v_full[i]), 1);
      mbar_init(smem_u32(&sh.v_empty[i]), 1);
      mbar_init(smem_u32(&sh.v_conv[i]), 4);
    }
    mbar_init(smem_u32(&sh.fin_full), 1);  // armed here (expect_tx), completed by the bulk copy
    if (rank != 0) {
      // A value CTA arms its P slots' first phases and the final row sums
      // here; the scorer's bulk copies complete them (a copy may land before
      // the arming: the transaction count may run ahead of the expectation).
      for (int i = 0; i < NPS; ++i) mbar_expect_tx(smem_u32(&sh.p_full[i]), PCOPY);
      mbar_expect_tx(smem_u32(&sh.fin_full), H * 4);
    }
    sh.abort = 0;
    fence_mbar_init();
  }
  // Decision words of a value CTA: 0 = not yet published, 1 = skipped, 2 = kept.
  if (rank != 0 && aligned)
    for (int j = tid; j < MAX_BPS; j += NTHREADS)
      asm volatile("st.shared.u32 [%0], 0;" ::"r"(base + SMEM_DEC + 4u * (uint32_t)j) : "memory");
  // Every CTA's barriers and decision words exist before any remote arrival or store.
  cluster_sync();
  if (!aligned) {  // the swizzled layouts need a 1024-byte aligned base
    if (tid == 0) atomicOr(a.err, kErrLayout);
    cluster_sync();
    return;
  }

  // Bitmap rows: one per (sequence, split), or per (sequence, head, split)
  // with per-head decisions.
  const bool ph = a.per_head != 0;
  uint32_t *bits = a.bits + (size_t)us * a.words;
  if (nb == 0) {  // empty split: no key, zero weight in the merge; no hand-off
    if (scorer) {
      if (tid < H) a.lse_part[(size_t)(b * a.Hq + tid) * a.n_splits + sp] = -INFINITY;
      if (ph) {
        for (int w = tid; w < H * a.words; w += NTHREADS)
          a.bits[((size_t)(b * a.Hq + w / a.words) * a.n_splits + sp) * a.words + w % a.words] = 0u;
      } else {
        for (int w = tid; w < a.words; w += NTHREADS) bits[w] = 0u;
      }
    } else {
      for (int idx = tid; idx < H * DVH; idx += NTHREADS) {
        const size_t row = (size_t)(b * a.Hq + idx / DVH) * a.n_splits + sp;
        a.o_part[row * DV + half * DVH + idx % DVH] = 0.f;
      }
    }
    cluster_sync();
    return;
  }

  if ((scorer && warp == WARP_MMA) || (!scorer && warp == WARP_MMA))
    tmem_alloc(smem_u32(&sh.tmem_base), scorer ? 512u : 256u);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  if (scorer) {
    if (warp == WARP_TMA) {
      // ---------------------------------------------------- latent stream --
      if (lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_kv128);
        const uint64_t pol_q = policy_evict_first(), pol_kv = policy_evict_last();
        // Q: latent chunks 0-7 staged in ring groups 0-2 (chunk c in slot c;
        // copied into TMEM by the softmax warps), the rope chunk to its home.
        for (int gq = 0; gq < 3; ++gq) {
          const int n = gq < 2 ? GCH : 8 - 2 * GCH;
          mbar_expect_tx(smem_u32(&sh.g_full[gq]), n * CH_BYTES);
          for (int c = gq * GCH; c < gq * GCH + n; ++c)
            tma_load_3d(base + SMEM_RING + c * CH_BYTES, &tm_q, smem_u32(&sh.g_full[gq]), c * 64, 0,
                        b, pol_q);
        }
        mbar_expect_tx(smem_u32(&sh.rope_full), CH_BYTES);
        tma_load_3d(base + SMEM_ROPE, &tm_q, smem_u32(&sh.rope_full), 8 * 64, 0, b, pol_q);
        // Latent: double block dj is groups 3 + 3 dj .. + 2, each three 64-column
        // chunks of 128 keys; group G uses ring group G % NG.
        int G = 3;
        for (int dj = 0; dj < ndb && !*abort; ++dj) {
          for (int gi = 0; gi < 3; ++gi, ++G) {
            const int s = G % NG;
            if (G >= NG && !mbar_wait(smem_u32(&sh.g_empty[s]), ((G / NG) - 1) & 1, abort, a.err,
                                      kErrTimeout))
              break;
            mbar_expect_tx(smem_u32(&sh.g_full[s]), GCH * CH_BYTES);
            for (int cc = 0; cc < GCH; ++cc)
              tma_load_3d(base + SMEM_RING + (s * GCH + cc) * CH_BYTES, &tm_kv128,
                          smem_u32(&sh.g_full[s]), (gi * GCH + cc) * 64, (j0 + 2 * dj) * BN, b,
                          pol_kv);
          }
        }
        // Drain: the last load issued into each ring group has landed.
        mbar_wait_drain(smem_u32(&sh.rope_full), 0);
        for (int s = 0; s < NG && s < G; ++s) {
          const int last = s + ((G - 1 - s) / NG) * NG;
          mbar_wait_drain(smem_u32(&sh.g_full[s]), (last / NG) & 1);
        }
      }
    } else if (warp == WARP_MMA) {
      // ------------------------------------------------------ Q.K^T issuer --
      if (lane == 0) {
        bool ok = mbar_wait(smem_u32(&sh.q_ready), 0, abort, a.err, kErrTimeout) &&
                  mbar_wait(smem_u32(&sh.rope_full), 0, abort, a.err, kErrTimeout);
        fence_after_sync();
        const uint64_t rope = smem_desc_sw128(base + SMEM_ROPE, 16, 1024);
        int G = 3;
        for (int dj = 0; ok && dj < ndb; ++dj) {
          const int buf = dj & 1;
          if (dj >= 2 && !mbar_wait(smem_u32(&sh.s_free[buf]), ((dj >> 1) - 1) & 1, abort, a.err,
                                    kErrTimeout))
            break;
          const uint32_t idesc = 2 * dj + 1 < nb ? IDESC_QK128 : IDESC_QK64;
          const uint32_t d = tmem + TMEM_S + buf * DBN;
          // One barrier wait per group, then its 12 products in one burst (a
          // wait or a fence between products costs about as much as a product).
          for (int gi = 0; gi < 3; ++gi, ++G) {
            const int s = G % NG;
            if (!mbar_wait(smem_u32(&sh.g_full[s]), (G / NG) & 1, abort, a.err, kErrTimeout)) {
              ok = false;
              break;
            }
            fence_after_sync();
            const uint64_t bd = smem_desc_sw128(base + SMEM_RING + s * GCH * CH_BYTES, 16, 1024);
#pragma unroll
            for (int cc = 0; cc < GCH; ++cc) {
              const int c = gi * GCH + cc;  // latent chunk
              const uint64_t bc = bd + (uint64_t)((cc * CH_BYTES) >> 4);
              if (c < 8) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_bf16_ts(d, tmem + TMEM_Q + c * 32 + kk * 8, bc + (uint64_t)(kk * 2), idesc,
                              (c > 0 || kk > 0) ? 1u : 0u);
              } else {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_bf16_ss(d, rope + (uint64_t)(kk * 2), bc + (uint64_t)(kk * 2), idesc, 1u);
              }
            }
            mma_commit(smem_u32(&sh.g_empty[s]));
          }
          if (!ok) break;
          mma_commit(smem_u32(&sh.s_full[buf]));
        }
      }
    } else if (warp < 4) {
      // ----------------------------------------------------------- softmax --
      const int r = tid;  // head == TMEM lane
      const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
      const float sl2 = a.scale * kLog2e;
      const float c2 = a.ln_lambda * kLog2e;
      bool ok = true;
      // Q latent dims [0,512) of head r: ring slots 0-7 -> TMEM columns [0,256).
#pragma unroll 1
      for (int c = 0; c < 8 && ok; ++c) {
        if (c % GCH == 0) ok = mbar_wait_warp(smem_u32(&sh.g_full[c / GCH]), 0, abort, a.err,
                                              kErrTimeout);
        if (!ok) break;
        const uint32_t rowp = base + SMEM_RING + c * CH_BYTES + (uint32_t)r * 128u;
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
        tmem_st32(lane_base + TMEM_Q + c * 32, w);
      }
      tmem_wait_st();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.q_ready));
      if (tid == 0 && ok && mbar_wait(smem_u32(&sh.q_ready), 0, abort, a.err, kErrTimeout))
        for (int gq = 0; gq < 3; ++gq) mbar_arrive(smem_u32(&sh.g_empty[gq]));  // Q groups free

      const uint32_t rk[2] = {1u, 2u};
      float m2 = -INFINITY, mref = -INFINITY, l = 0.f;
      int kc = 0;
      uint32_t word = 0;
      // Per-head decisions: this head's own bitmap row and word.
      uint32_t *hbits = a.bits + ((size_t)(b * a.Hq + r) * a.n_splits + sp) * a.words;
      uint32_t hword = 0;
      // Once a wait has failed (the abort flag is up and every later wait
      // fails at once) the loops still run to their end, so that the four
      // warps meet the vote barrier equally often.
      for (int dj = 0; dj < ndb; ++dj) {
        const int buf = dj & 1;
        if (ok) ok = mbar_wait_warp(smem_u32(&sh.s_full[buf]), (dj >> 1) & 1, abort, a.err,
                                    kErrTimeout);
        if (ok) fence_after_sync();
        for (int i = 0; i < 2; ++i) {
          const int j = 2 * dj + i;
          if (j >= nb) break;
          uint32_t x[32], y[32];
          float mt = -INFINITY;
          if (ok) {
            const uint32_t sa = lane_base + TMEM_S + buf * DBN + i * BN;
            tmem_ld32(sa, x);
            tmem_ld32(sa + 32, y);
            tmem_wait_ld_regs(x);
            tmem_wait_ld_regs(y);
            if (i == 1 || j == nb - 1) {  // the S buffer is read: the next product may use it
              fence_before_sync();
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&sh.s_free[buf]));
            }
            const int keys = min(BN, a.L - (j0 + j) * BN);
            if (keys < BN) {
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                if (e >= keys) x[e] = NEG_INF_BITS;
                if (e + 32 >= keys) y[e] = NEG_INF_BITS;
              }
            }
#pragma unroll
            for (int e = 0; e < 32; e += 2)
              mt = fmax3(mt, fmaxf(__uint_as_float(x[e]), __uint_as_float(x[e + 1])),
                         fmaxf(__uint_as_float(y[e]), __uint_as_float(y[e + 1])));
          }
          const float mt2 = mt * sl2;
          const float mnew = fmaxf(m2, mt2);
          const float diff = (mt == -INFINITY) ? -INFINITY : mt2 - m2;  // Eq. 5 (reading 2)
          // The block is kept if any head votes keep (one reduction of the four
          // warps); with per-head decisions a head that votes skip takes no
          // part in the block (P row 0, no row sum, no rescale), and the block
          // is still skipped as a whole (no value load, no P.V) only if every
          // head votes skip.
          const bool vote = ok && !(diff < c2);
          const bool keep = bar_red_or(kVoteBarrier, H, vote);
          // One outcome for the four warps: the kept path below has a barrier
          // of its own that all of them must reach.
          if (bar_red_or(kFailBarrier, H, !ok)) ok = false;
          if (!ok) continue;
          m2 = mnew;
          if (tid == 0) {
            // Publish the decision to both value CTAs (one word each).
            for (int t = 0; t < 2; ++t)
              st_remote_relaxed_u32(remote(base + SMEM_DEC + 4u * (uint32_t)j, rk[t]), keep ? 2u : 1u);
            if (!ph) {
              if (!keep) word |= 1u << (j & 31);
              if ((j & 31) == 31 || j == nb - 1) {
                bits[j >> 5] = word;
                word = 0;
              }
            }
          }
          if (ph) {
            if (!vote) hword |= 1u << (j & 31);
            if ((j & 31) == 31 || j == nb - 1) {
              hbits[j >> 5] = hword;
              hword = 0;
            }
          }
          if (!keep) continue;
          const bool mine = !ph || vote;  // this head takes part in the block
          float alpha = 1.f;
          if (mine) {
            if (mref == -INFINITY) {
              mref = mnew;
            } else if (mnew > mref + kRescaleLog2) {
              alpha = ex2(mref - mnew);
              mref = mnew;
            }
          }
          const uint64_t sl2x2 = f2(sl2, sl2), negref2 = f2(-mref, -mref);
          uint64_t acc2 = f2(0.f, 0.f);
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float e0, e1;
            f2_split(f2_fma(f2(__uint_as_float(x[2 * e]), __uint_as_float(x[2 * e + 1])), sl2x2,
                            negref2),
                     e0, e1);
            const float p0 = ex2(e0), p1 = ex2(e1);
            acc2 = f2_add(acc2, f2(p0, p1));
            pk[e] = pack_f16x2(p0, p1);
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float e0, e1;
            f2_split(f2_fma(f2(__uint_as_float(y[2 * e]), __uint_as_float(y[2 * e + 1])), sl2x2,
                            negref2),
                     e0, e1);
            const float p0 = ex2(e0), p1 = ex2(e1);
            acc2 = f2_add(acc2, f2(p0, p1));
            pk[16 + e] = pack_f16x2(p0, p1);
          }
          float s0, s1;
          f2_split(acc2, s0, s1);
          if (mine) {
            l = l * alpha + (s0 + s1);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) pk[e] = 0u;
          }
          const int ps = kc % NPS;
          const uint32_t stage = base + SMEM_STAGE;
          // The staging buffer last fed the copies of kept block kc - 1: their
          // reads of it are complete before anyone overwrites it.
          if (tid == 0) bulk_wait_read<0>();
          named_bar_sync(kStageBarrier, H);
          // Row r (K-major, 128-byte swizzle: 16-byte chunk q of the row at chunk
          // position q ^ (r % 8)), then this head's rescale factor.
          const uint32_t row = stage + (uint32_t)r * 128u;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_shared_v4(row + ((uint32_t)(q ^ (r & 7)) << 4), pk[4 * q], pk[4 * q + 1],
                         pk[4 * q + 2], pk[4 * q + 3]);
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(stage + P_BYTES + (uint32_t)r * 4u),
                       "f"(alpha)
                       : "memory");
          fence_proxy_async_smem();  // generic writes -> the bulk copy's reads
          named_bar_sync(kStageBarrier, H);
          if (tid == 0) {
            // P slot ps of the value CTAs last held kept block kc - NPS: both
            // products that read it have completed.
            if (kc < NPS ||
                wait_cluster(smem_u32(&sh.p_free[ps]), ((kc / NPS) - 1) & 1, abort, a.err)) {
              for (int t = 0; t < 2; ++t)
                bulk_copy_to_cluster(remote(base + SMEM_P + ps * PX_BYTES, rk[t]), stage, PCOPY,
                                     remote(smem_u32(&sh.p_full[ps]), rk[t]));
              bulk_commit();
            }
          }
          ++kc;
        }
      }
      // ---- epilogue: LSE here, the final row sums to the value CTAs ------
      if (ph) {
        for (int w = ((nb - 1) >> 5) + 1; w < a.words; ++w) hbits[w] = 0u;
      } else if (tid == 0) {
        for (int w = ((nb - 1) >> 5) + 1; w < a.words; ++w) bits[w] = 0u;
      }
      if (ok) {
        a.lse_part[(size_t)(b * a.Hq + r) * a.n_splits + sp] = mref * kLn2 + logf(l);
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(base + SMEM_FIN + (uint32_t)r * 4u), "f"(l)
                     : "memory");
        fence_proxy_async_smem();  // generic writes -> the bulk copy's reads
      }
      // The four warps' row sums are staged (all four reach this barrier:
      // the loops above ran to their ends).
      const bool all_ok = !bar_red_or(kFailBarrier, H, !ok);
      if (tid == 0) {
        if (all_ok)
          for (int t = 0; t < 2; ++t)
            bulk_copy_to_cluster(remote(smem_u32(&sh.fin_l[0]), rk[t]), base + SMEM_FIN, H * 4,
                                 remote(smem_u32(&sh.fin_full), rk[t]));
        bulk_commit();
        bulk_wait_read<0>();  // no copy still reads the staging buffers
      }
    }
  } else {
    // ======================================================== value CTA ==
    if (warp == WARP_TMA) {
      // ------------------------------------------------- value tile loads --
      if (lane == 0) {
        prefetch_tmap(&tm_kv64);
        const uint64_t pol = policy_evict_first();  // the last reader of these rows
        int kc = 0;
        for (int j = 0; j < nb; ++j) {
          const unsigned d = wait_decision(base + SMEM_DEC, j, abort, a.err);
          if (!d) break;
          if (d == 1u) continue;
          const int s = kc % NV;
          if (kc >= NV &&
              !mbar_wait(smem_u32(&sh.v_empty[s]), ((kc / NV) - 1) & 1, abort, a.err, kErrTimeout))
            break;
          mbar_expect_tx(smem_u32(&sh.v_full[s]), VT_BYTES);
          for (int c = 0; c < 4; ++c)
            tma_load_3d(base + SMEM_V + s * VT_BYTES + c * VCH_BYTES, &tm_kv64,
                        smem_u32(&sh.v_full[s]), (4 * half + c) * 64, (j0 + j) * BN, b, pol);
          ++kc;
        }
        for (int s = 0; s < NV && s < kc; ++s) {
          const int last = s + ((kc - 1 - s) / NV) * NV;
          mbar_wait_drain(smem_u32(&sh.v_full[s]), (last / NV) & 1);
        }
      }
    } else if (warp >= WARP_CV && warp < WARP_CV + 4) {
      // ------------------------------------------ bf16 -> fp16, in place --
      const int t0 = (warp - WARP_CV) * 32 + lane;
      int kc = 0;
      for (int j = 0; j < nb; ++j) {
        const unsigned d = wait_decision(base + SMEM_DEC, j, abort, a.err);
        if (!__all_sync(0xffffffffu, d != 0u)) break;
        if (d == 1u) continue;
        const int s = kc % NV;
        if (!mbar_wait_warp(smem_u32(&sh.v_full[s]), (kc / NV) & 1, abort, a.err, kErrTimeout))
          break;
        const uint32_t vt = base + SMEM_V + s * VT_BYTES;
#pragma unroll 4
        for (int i = 0; i < (int)(VT_BYTES / 16) / 128; ++i) {
          const uint32_t addr = vt + (uint32_t)(t0 + 128 * i) * 16u;
          uint32_t w0, w1, w2, w3;
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                       : "r"(addr));
          st_shared_v4(addr, bf16x2_to_f16x2(w0), bf16x2_to_f16x2(w1), bf16x2_to_f16x2(w2),
                       bf16x2_to_f16x2(w3));
        }
        fence_proxy_async_smem();  // generic writes -> the tensor core's reads
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.v_conv[s]));
        ++kc;
      }
    } else if (warp == WARP_MMA) {
      // -------------------------------------------------------- P.V issuer --
      if (lane == 0) {
        int kc = 0;
        for (int j = 0; j < nb; ++j) {
          const unsigned d = wait_decision(base + SMEM_DEC, j, abort, a.err);
          if (!d) break;
          if (d == 1u) continue;
          const int ps = kc % NPS, s = kc % NV;
          if (!mbar_wait(smem_u32(&sh.p_ok[ps]), (kc / NPS) & 1, abort, a.err, kErrTimeout) ||
              !mbar_wait(smem_u32(&sh.v_conv[s]), (kc / NV) & 1, abort, a.err, kErrTimeout))
            break;
          fence_after_sync();
          const uint64_t pd = smem_desc_sw128(base + SMEM_P + ps * PX_BYTES, 16, 1024);
          const uint32_t vt = base + SMEM_V + s * VT_BYTES;
          // O_h += P (128 heads x 64 keys, K-major) x V_h (64 keys x 256 columns,
          // MN-major: keys are the 128-byte rows of four 64-column chunks 8 KB apart).
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_bf16_ss(tmem + TMEM_O, pd + (uint64_t)(kk * 2),
                        smem_desc_sw128(vt + kk * 2048, VCH_BYTES, 1024), IDESC_PV,
                        (kc > 0 || kk > 0) ? 1u : 0u);
          mma_commit(smem_u32(&sh.v_empty[s]));
          mma_commit(smem_u32(&sh.pv_done[ps]));
          ++kc;
        }
      }
    } else if (warp == WARP_FWD) {
      // ------------------------------------- P slot release to the scorer --
      if (lane == 0) {
        int kc = 0;
        for (int j = 0; j < nb; ++j) {
          const unsigned d = wait_decision(base + SMEM_DEC, j, abort, a.err);
          if (!d) break;
          if (d == 1u) continue;
          const int ps = kc % NPS;
          if (!mbar_wait(smem_u32(&sh.pv_done[ps]), (kc / NPS) & 1, abort, a.err, kErrTimeout))
            break;
          // The slot's P was read: arm its next phase, then hand it back.
          mbar_expect_tx(smem_u32(&sh.p_full[ps]), PCOPY);
          arrive_remote(remote(smem_u32(&sh.p_free[ps]), 0u));
          ++kc;
        }
      }
    } else if (warp < 4) {
      // ---------------------------------------------- rescale, epilogue --
      const int r = tid;  // head == TMEM lane of the O half
      const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
      bool ok = true;
      int kc = 0;
      for (int j = 0; j < nb; ++j) {
        const unsigned d = wait_decision(base + SMEM_DEC, j, abort, a.err);
        if (!__all_sync(0xffffffffu, d != 0u)) {
          ok = false;
          break;
        }
        if (d == 1u) continue;
        const int ps = kc % NPS;
        if (!wait_cluster_warp(smem_u32(&sh.p_full[ps]), (kc / NPS) & 1, abort, a.err)) {
          ok = false;
          break;
        }
        const float alpha =
            reinterpret_cast<const float *>(smem_raw + SMEM_P + ps * PX_BYTES + P_BYTES)[r];
        if (__any_sync(0xffffffffu, alpha != 1.f) && kc >= 1) {
          if (!mbar_wait_warp(smem_u32(&sh.pv_done[(kc - 1) % NPS]), ((kc - 1) / NPS) & 1,
                              abort, a.err, kErrTimeout)) {
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
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(lane_base + TMEM_O + cc * 32, o);
          }
          tmem_wait_st();
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.p_ok[ps]));
        ++kc;
      }
      // Every split keeps its first block, so kc >= 1 here.
      if (ok) ok = wait_cluster_warp(smem_u32(&sh.fin_full), 0, abort, a.err);
      if (ok && kc > 0)
        ok = mbar_wait_warp(smem_u32(&sh.pv_done[(kc - 1) % NPS]), ((kc - 1) / NPS) & 1, abort,
                            a.err, kErrTimeout);
      if (ok) {
        fence_after_sync();
        const float inv = 1.f / sh.fin_l[r];
        // O_h / l, 32 columns at a time: each thread's row goes through a 4 KB
        // staging area of its warp (in the value tiles, idle now that every
        // product has completed; 16-byte chunk q of row i at chunk position
        // q ^ (i % 8)), then each row's 128 bytes leave as one coalesced
        // segment (8 lanes per row, 4 rows per store).
        const uint32_t stg = base + SMEM_V + (uint32_t)warp * 4096u;
        const int rr = lane >> 3, qq = lane & 7;  // read side: row of 4, chunk
#pragma unroll 1
        for (int cc = 0; cc < DVH / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(lane_base + TMEM_O + cc * 32, o);
          tmem_wait_ld_regs(o);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_shared_v4(stg + (uint32_t)lane * 128u + (uint32_t)((q ^ (lane & 7)) << 4),
                         __float_as_uint(__uint_as_float(o[4 * q]) * inv),
                         __float_as_uint(__uint_as_float(o[4 * q + 1]) * inv),
                         __float_as_uint(__uint_as_float(o[4 * q + 2]) * inv),
                         __float_as_uint(__uint_as_float(o[4 * q + 3]) * inv));
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int ro = 4 * i + rr;  // row within the warp
            float4 v;
            asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                         : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                         : "r"(stg + (uint32_t)ro * 128u + (uint32_t)((qq ^ (ro & 7)) << 4)));
            const size_t row = (size_t)(b * a.Hq + warp * 32 + ro) * a.n_splits + sp;
            *reinterpret_cast<float4 *>(a.o_part + row * DV + half * DVH + cc * 32 + 4 * qq) = v;
          }
          __syncwarp();
        }
      }
    }
  }

  __syncwarp();
  fence_before_sync();
  __syncthreads();
  if (warp == WARP_MMA) {
    fence_after_sync();
    tmem_dealloc(tmem, scorer ? 512u : 256u);
  }
  // No CTA leaves while another may still write into its shared memory.
  cluster_sync();
}

}  // namespace

// Blocks per split the cluster kernel's decision array holds; longer splits
// (and the statistics mode) use the two-CTA kernel.
int mla_cluster_max_bps() { return MAX_BPS; }

cudaError_t launch_mla_cluster(const DecodeArgs &a, cudaStream_t s) {
  CUtensorMap mq, mk128, mk64;
  // [B, rows, 576] bf16, boxes of 64 columns x (128 heads / 128 keys / 64 keys).
  if (!make_map_bf16_3d(&mq, a.q, DK, DK, H, a.B, H) ||
      !make_map_bf16_3d(&mk128, a.k, DK, DK, a.L, a.B, DBN) ||
      !make_map_bf16_3d(&mk64, a.k, DK, DK, a.L, a.B, BN))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(mla_cluster_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(3L * a.B * a.n_splits));
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = SMEM_ALLOC;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 3;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mla_cluster_kernel, mq, mk128, mk64, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace attn_skip

