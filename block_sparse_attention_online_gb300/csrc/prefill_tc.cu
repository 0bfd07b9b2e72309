// bf16 tensor-core prefill with softmax-threshold block skipping (d = 128,
// Br = Bc = 128), tcgen05 MMAs accumulating in TMEM, operands staged by TMA.
//
// Method: the BLASST page, sections "铺垫：FlashAttention 的在线 softmax"
// (Eqs. 2-4), "BLASST 的判定准则" (Eq. 5), "判定本身：几乎零成本的秘密" (a per-row
// predicate, a warp vote and a tile-wide AND) and "Prefill 内核：砍计算" (a
// skipped block costs no exponentials, no row sum and no P.V product).  Unlike
// the page's prefill kernel, the value tile of a block is loaded only once the
// block is known to be kept; decisions are taken by their own warps ahead of
// the exponentials, so that load has time to land.  P_j (bf16) is
// written back into the TMEM columns of S_j and read from there by the P.V
// MMA, so it never touches shared memory.
//
// One CTA per (batch, query head, query tile), longest causal tiles first.
// Warp roles (416 threads):
//   warps 0-3  deciders: warp w owns query rows 32w..32w+31 (TMEM lane
//              quarter w) over all 128 key columns.  Per block: the row max
//              of S_j, the row vote against the running max before the
//              block, one barrier round of the four deciders to AND the
//              votes; thread 0 publishes the decision and the bitmap.  The
//              deciders run ahead of the exponentials as far as the three S
//              buffers allow, so in a run of skipped blocks nothing else
//              waits for them;
//   warps 4-7  exponentials: warp 4+w owns the same rows; for each kept block
//              P_j = exp2(S_j - ref) (bf16 pairs into TMEM columns [0,64) of
//              the block's S buffer), the row sum, and an O rescale in TMEM
//              when the exp reference moves by > 2^8;
//   warp 8     TMA producer of Q (once) and K_j (every block);
//   warps 9, 12 Q.K^T issuers (even / odd traversed blocks): S_j = Q K_j^T
//              up to three blocks ahead (warp 9 also allocates TMEM);
//   warp 10    TMA producer of V_j, for kept blocks only, as soon as the
//              block's decision is known;
//   warp 11    P.V issuer: O += P_j V_j (P from TMEM) for kept blocks; the
//              commit of that product frees the S buffer of a kept block
//              (the decision frees that of a skipped block).
// Separate issuing threads keep one product chain from waiting on another's
// barriers: a tcgen05.mma issue is accepted at about the rate the tensor core
// retires it, so a single issuer serialises every wait with every product.
// TMEM columns: three S buffers [0,384), O [384,512).
//
// Votes: with c = ln(lambda) < 0, "rowmax(S_ij) - m_new < c" holds iff
// "rowmax(S_ij) - m_old < c" (if the block raises the max both sides are
// false).
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"
#include "tc_common.cuh"

namespace attn_skip {
namespace {

using namespace tc;

constexpr int D = 128;        // head size of keys and values
constexpr int BM = 128;       // query rows per tile
constexpr int BN = 128;       // keys per block
constexpr int NK = 4;         // K stages
constexpr int NV = 2;         // V stages
constexpr int NS = 3;         // TMEM S buffers
constexpr int NDEC = 4;       // decision ring
// Block c may be issued once one barrier, slot c % NK of the "ready" ring,
// has completed: its key tile has landed (the producer's arrival with the
// byte count) and its S buffer is free (the decision of block c - NS if that
// block was skipped, its P.V commit if kept; the first NS blocks' buffers are
// free from the start).  One wait per block: a wait or a memory operation of
// the issuing thread between two product batches stalls the tensor pipe for
// about 100-250 cycles.  The two Q.K^T issuers take alternate blocks, so with
// an even ring every slot belongs to one issuer and its phases come in that
// issuer's order; a slot's next "free" arrival (block c + NK's, made at block
// c + NK - NS's decision) cannot come before block c was issued, as NK > NS.
static_assert(NK % 2 == 0 && NK > NS, "ready ring: even, and longer than the S buffer ring");
constexpr int NQ = 4;     // decider warps (0-3) and exponential warps (4-7): one per TMEM lane quarter
constexpr int NSOFT = 2 * NQ;
constexpr int kDeciderBarrier = 1;  // named barrier of the four decider warps
constexpr int kSetupBarrier = 2;    // varlen set-up: the key producer and the tile-locating warp
// Two Q.K^T issuers (even and odd blocks): a thread that issues tcgen05.mma
// is held until the tensor pipe takes each instruction, so one issuer's
// barrier waits between blocks leave the pipe idle; with two, one waits while
// the other issues.
constexpr int NTHREADS = (NSOFT + 5) * 32;
constexpr int WARP_K = NSOFT, WARP_MMA = NSOFT + 1, WARP_V = NSOFT + 2, WARP_PV = NSOFT + 3,
              WARP_MMA2 = NSOFT + 4;
constexpr uint32_t TILE_BYTES = BM * D * 2;      // 32 KB: one 128 x 128 bf16 tile
constexpr uint32_t HALF_BYTES = TILE_BYTES / 2;  // one 64-column swizzled box
constexpr uint32_t SMEM_Q = 0;
constexpr uint32_t SMEM_K = SMEM_Q + TILE_BYTES;
constexpr uint32_t SMEM_V = SMEM_K + NK * TILE_BYTES;
constexpr uint32_t SMEM_TILES = SMEM_V + NV * TILE_BYTES;  // 224 KB
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_O = NS * BN;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // exp reference may lag the max by 2^8
constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, 0);  // K: K-major
constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, 1);   // V: MN-major
constexpr uint32_t NEG_INF_BITS = 0xff800000u;

// A tile of a variable-length batch: sequence s (-1: no tile for this CTA),
// tile index t, the sequence's first token and length, ln(lambda_s).
struct VarTile {
  int s, t, c0, len;
  float ln_lam;
};

struct Shared {
  uint64_t q_full;
  uint64_t ready[NK];    // slot c % NK: block c's key tile landed and its S buffer free
  uint64_t qk_done[NK];  // slot c % NK: block c's Q.K^T complete (scores in, key stage free)
  uint64_t v_full[NV], v_empty[NV];
  // P of kept block kc ready, slot kc % NS.  Kept blocks whose P exists but
  // whose P.V has not completed each hold an S buffer, so at most NS are
  // outstanding and a slot is never re-armed before its phase was consumed
  // (with fewer slots than S buffers the exponential warps could complete a
  // slot's next phase first when a value load is slow).
  uint64_t p_full[NS];
  // P.V of kept block kc complete, slot kc % NS.  Up to NS kept blocks can
  // have a P.V in flight (each holds its S buffer), so with NS slots each slot
  // has at most one phase pending and a wait on it has one meaning; a commit
  // also covers every earlier product of the issuing thread.  (With two slots
  // the end-of-tile wait could see an older pending phase of the other
  // parity, pass early, and let the epilogue read O before the last products
  // landed.)
  uint64_t pv_done[NS];
  uint64_t dec_full[NDEC];
  uint64_t dec_read[NDEC];  // the V producer, the P.V issuer and the exponential warps read slot j % NDEC
  uint64_t l_full;
  int dec[NDEC];
  float wstat[2][NQ];  // statistics mode: per decider warp, max over its rows of rowmax - m_new
  // [S buffer][row] running max after the buffer's block (log2 units), from
  // the deciders to the exponential warps.
  float mdec[NS][128];
  float lfin[128], mfin[128];  // row sum and exp reference for the epilogue
  VarTile vt;                  // varlen: this CTA's tile
  uint32_t tmem_base;
  int abort;
};
// Dynamic shared memory: the tiles at a 1024-byte aligned base (the 128-byte
// swizzle repeats every 1024 bytes), then the control block.
constexpr uint32_t SMEM_ALLOC = SMEM_TILES + ((sizeof(Shared) + 127) / 128) * 128;
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");

// Descriptors are built once per tile and advanced per k-step by adding the
// byte offset >> 4 to the start-address field (shared addresses stay below
// 2^18, so the 14-bit field never carries).
//
// K-major 128 x 128 bf16 tile held as two 128-byte-swizzled boxes of 64
// columns: k-step kk (16 columns) is box kk/4 at 32-byte step kk%4; 8-row
// groups are 1024 bytes apart.
__device__ __forceinline__ uint64_t kmajor_base(uint32_t tile) {
  return smem_desc_sw128(tile, 16u, 1024u);
}
__device__ __forceinline__ constexpr uint64_t kmajor_step(int kk) {
  return (uint64_t)(((uint32_t)(kk >> 2) * HALF_BYTES + (uint32_t)(kk & 3) * 32u) >> 4);
}

// MN-major value tile: rows are keys (128 bytes = 64 values per swizzled row),
// 8-key groups 1024 bytes apart (SBO), the second 64-value half 16 KB further
// (LBO); k-step kk (16 keys) starts 2048 bytes further.
__device__ __forceinline__ uint64_t vmajor_base(uint32_t tile) {
  return smem_desc_sw128(tile, HALF_BYTES, 1024u);
}
__device__ __forceinline__ constexpr uint64_t vmajor_step(int kk) {
  return (uint64_t)(((uint32_t)kk * 2048u) >> 4);
}

// Write -inf over the invisible scores of block j in this warp's TMEM lanes
// (causal: key > row; otherwise key >= T), 32 keys at a time: chunks with no
// visible key get a constant store, a partial chunk is loaded, masked and
// stored back.  Only a tile's last blocks need it; the code is kept short
// because it runs from a cold instruction cache.  Every later reader of the
// buffer (this warp after tcgen05.wait::st, the exponential warps after the
// decision is published) sees the masked scores through the normal path.
__device__ __noinline__ void mask_block_tmem(uint32_t sa, int kbase, int row, int causal, int T) {
  uint32_t ninf[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) ninf[i] = NEG_INF_BITS;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    const int lim = causal ? row - (kbase + 32 * c) + 1 : T - (kbase + 32 * c);
    if (__all_sync(0xffffffffu, lim >= 32)) continue;
    if (__all_sync(0xffffffffu, lim <= 0)) {
      tmem_st32(sa + 32 * c, ninf);
      continue;
    }
    uint32_t x[32];
    tmem_ld32(sa + 32 * c, x);
    tmem_wait_ld_regs(x);
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = i < lim ? x[i] : NEG_INF_BITS;
    tmem_st32(sa + 32 * c, x);
  }
  tmem_wait_st();
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

// P = exp2(s * sl2 - ref) for one 32-key chunk, as 16 packed bf16 pairs, with
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

// ---------------------------------------------------------- varlen schedule --
// The tiles of a variable-length batch run in decreasing tile index t (the
// longest causal tiles first, as in the fixed-length grid), then increasing
// sequence index; CTA i * Hq + h runs the i-th tile of that order for query
// head h.  The grid holds Hq * (ceil(total / Br) + n_seq) CTAs, at least one
// per tile; a CTA past the last tile clears the bitmap rows of empty
// sequences.  One warp locates its CTA's tile: with nt(s) the tile count of
// sequence s, C(t) = sum_s max(0, nt(s) - t - 1) tiles lie at levels above t,
// so the tile's level is the smallest t with C(t) <= i (bisection) and its
// sequence the (i - C(t))-th one, in index order, with nt(s) > t.
constexpr int kVarCache = 4;  // sequences 0..127 are served from registers

// Length of sequence s, or -1 when its bounds are out of range.
__device__ __forceinline__ int var_len(const PrefillArgs &a, int s) {
  const int c0 = __ldg(a.cu_seqlens + s), c1 = __ldg(a.cu_seqlens + s + 1);
  return (c0 < 0 || c1 < c0 || c1 - c0 > a.T || c1 > a.total) ? -1 : c1 - c0;
}

__device__ __forceinline__ int tiles_of(int len) { return len > 0 ? (len + BM - 1) / BM : 0; }

// Batches of up to 32 sequences (one per lane): a short, branch-light path,
// since this code runs once per CTA from a cold instruction cache.
__device__ __forceinline__ bool varlen_locate_small(const PrefillArgs &a, int i, int h, int lane,
                                                    VarTile *out) {
  int c0 = 0, c1 = 0;
  float lam = 0.f;
  if (lane < a.B) {
    c0 = __ldg(a.cu_seqlens + lane);
    c1 = __ldg(a.cu_seqlens + lane + 1);
    lam = __ldg(a.lambda_seq + lane);
  }
  const bool bad = c0 < 0 || c1 < c0 || c1 - c0 > a.T || c1 > a.total;
  const int len = bad ? -1 : c1 - c0;
  const int nt = tiles_of(len);
  if (i >= (int)__reduce_add_sync(0xffffffffu, (unsigned)nt)) return false;
  int lo = 0, hi = a.n_t - 1;  // smallest t with C(t) <= i
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((int)__reduce_add_sync(0xffffffffu, (unsigned)max(0, nt - mid - 1)) <= i) hi = mid;
    else lo = mid + 1;
  }
  const int r = i - (int)__reduce_add_sync(0xffffffffu, (unsigned)max(0, nt - lo - 1));
  const unsigned m = __ballot_sync(0xffffffffu, nt > lo);
  const bool mine = nt > lo && __popc(m & ((2u << lane) - 1u)) == r + 1;
  const int s = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
  const int sc0 = __shfl_sync(0xffffffffu, c0, s), slen = __shfl_sync(0xffffffffu, len, s);
  const float slam = __shfl_sync(0xffffffffu, lam, s);
  if (lane == 0)
    *out = VarTile{s, lo, sc0, slen, (slam > 0.f && slam < 1.f) ? logf(slam) : -INFINITY};
  if (lo == tiles_of(slen) - 1) {  // the sequence's last tile clears the rows past it
    uint32_t *bw = a.bits + ((size_t)(s * a.Hq + h) * a.n_t + lo + 1) * a.words;
    for (int w = lane; w < (a.n_t - lo - 1) * a.words; w += 32) bw[w] = 0u;
  }
  if (i == 0 && h == 0 &&
      __any_sync(0xffffffffu, lane < a.B && (len < 0 || !(lam >= 0.f && lam < 1.f))) &&
      lane == 0)
    atomicOr(a.err, kErrBadArg);
  return true;
}

// Everything the CTA needs is read in one round of loads at the start (the
// first sequences' bounds and thresholds, kept in registers); the tile's own
// values then come from the lane that holds them.
__device__ __noinline__ void varlen_locate(const PrefillArgs &a, int i, int grid_tiles, int h,
                                           int lane, VarTile *out) {
  const int nch = (a.B + 31) / 32;
  int c0c[kVarCache], lenc[kVarCache];
  float lamc[kVarCache];
#pragma unroll
  for (int c = 0; c < kVarCache; ++c) {
    const int s = c * 32 + lane;
    int c0 = 0, c1 = 0;
    float lam = 0.f;
    if (s < a.B) {
      c0 = __ldg(a.cu_seqlens + s);
      c1 = __ldg(a.cu_seqlens + s + 1);
      lam = __ldg(a.lambda_seq + s);
    }
    const bool bad = c0 < 0 || c1 < c0 || c1 - c0 > a.T || c1 > a.total;
    c0c[c] = c0;
    lenc[c] = bad ? -1 : c1 - c0;
    lamc[c] = lam;
  }
  auto nt_chunk = [&](int c) {  // tile count of sequence 32 c + lane (0 past the batch)
    if (c >= kVarCache) {
      const int s = c * 32 + lane;
      return s < a.B ? tiles_of(var_len(a, s)) : 0;
    }
    int v = 0;
#pragma unroll
    for (int k = 0; k < kVarCache; ++k) v = k == c ? lenc[k] : v;
    return tiles_of(v);
  };
  auto above = [&](int t) {  // C(t)
    int sum = 0;
    for (int c = 0; c < nch; ++c)
      sum += (int)__reduce_add_sync(0xffffffffu, (unsigned)max(0, nt_chunk(c) - t - 1));
    return sum;
  };
  const int n_tiles = above(-1);
  if (i >= n_tiles) {
    // No tile: clear the rows of the empty sequences e, e + n_extra, ...
    const int e = i - n_tiles, n_extra = grid_tiles - n_tiles;
    for (int s = e; s < a.B; s += n_extra) {
      if (var_len(a, s) > 0) continue;
      uint32_t *bw = a.bits + (size_t)(s * a.Hq + h) * a.n_t * a.words;
      for (int w = lane; w < a.n_t * a.words; w += 32) bw[w] = 0u;
    }
    if (lane == 0) *out = VarTile{-1, 0, 0, 0, -INFINITY};
    return;
  }
  int lo = 0, hi = a.n_t - 1;  // smallest t with C(t) <= i
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (above(mid) <= i) hi = mid;
    else lo = mid + 1;
  }
  const int t = lo;
  int r = i - above(t), s = -1;
  for (int c = 0; c < nch && s < 0; ++c) {
    const unsigned m = __ballot_sync(0xffffffffu, nt_chunk(c) > t);
    const int n = __popc(m);
    if (r < n) {
      const unsigned upto = (2u << lane) - 1u;  // bits 0..lane
      const bool mine = ((m >> lane) & 1u) && __popc(m & upto) == r + 1;
      s = c * 32 + __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
    } else {
      r -= n;
    }
  }
  int c0 = 0, len = 0;
  float lam = 0.f;
  if ((s >> 5) < kVarCache) {
    int v0 = 0, v1 = 0;
    float v2 = 0.f;
#pragma unroll
    for (int k = 0; k < kVarCache; ++k) {
      v0 = k == (s >> 5) ? c0c[k] : v0;
      v1 = k == (s >> 5) ? lenc[k] : v1;
      v2 = k == (s >> 5) ? lamc[k] : v2;
    }
    c0 = __shfl_sync(0xffffffffu, v0, s & 31);
    len = __shfl_sync(0xffffffffu, v1, s & 31);
    lam = __shfl_sync(0xffffffffu, v2, s & 31);
  } else {
    c0 = __ldg(a.cu_seqlens + s);
    len = var_len(a, s);
    lam = __ldg(a.lambda_seq + s);
  }
  if (lane == 0)
    *out = VarTile{s, t, c0, len, (lam > 0.f && lam < 1.f) ? logf(lam) : -INFINITY};
  if (t == tiles_of(len) - 1) {  // the sequence's last tile clears the rows past it
    uint32_t *bw = a.bits + ((size_t)(s * a.Hq + h) * a.n_t + t + 1) * a.words;
    for (int w = lane; w < (a.n_t - t - 1) * a.words; w += 32) bw[w] = 0u;
  }
  if (i == 0 && h == 0) {  // one CTA reports out-of-range lengths or thresholds
    bool bad = false;
    for (int q = lane; q < a.B; q += 32) {
      const float lq = __ldg(a.lambda_seq + q);
      bad |= var_len(a, q) < 0 || !(lq >= 0.f && lq < 1.f);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.err, kErrBadArg);
  }
}

// The tile of CTA u: (sequence b, query head h, tile index t) and what
// follows from it.  Fixed length: longest causal tiles first, CTAs ordered by
// decreasing tile index; varlen: the located tile vt.
struct Tile {
  int t, h, b, T, off, row0, nblk;
  float ln_lam;
};

template <bool VARLEN>
__device__ __forceinline__ Tile tile_of(const PrefillArgs &a, const VarTile &vt, int u) {
  const int BH = a.B * a.Hq;
  Tile x;
  x.t = VARLEN ? vt.t : a.n_t - 1 - u / BH;
  x.h = VARLEN ? u % a.Hq : (u % BH) % a.Hq;
  x.b = VARLEN ? vt.s : (u % BH) / a.Hq;
  x.T = VARLEN ? vt.len : a.T;
  x.off = VARLEN ? vt.c0 : 0;
  x.ln_lam = VARLEN ? vt.ln_lam : a.ln_lambda;
  x.row0 = x.t * BM;
  const int last_row = min(x.T, x.row0 + BM) - 1;
  x.nblk = a.causal ? last_row / BN + 1 : (VARLEN ? (x.T + BN - 1) / BN : a.n_b);
  return x;
}

// STATS: the statistics mode; SET: an explicit block set per tile (blocks
// outside it are not traversed); VARLEN: a batch of sequences of different
// lengths packed token-major, each with its own threshold.  Each is compiled
// separately so that the ordinary kernel's loops carry none of their code.
// Ring positions count the traversed blocks (c); addresses and bitmap
// positions use the block index (j).
template <bool STATS, bool SET, bool VARLEN>
__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Shared &sh = *reinterpret_cast<Shared *>(smem_raw + SMEM_TILES);
  const uint32_t base = smem_u32(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (base & 1023u) {  // the swizzled layouts need a 1024-byte aligned base
    if (tid == 0) atomicOr(a.err, kErrLayout);
    return;
  }

  // Set-up.  The key producer's lane initialises the barriers and then issues
  // Q and the first NK traversed key tiles at once, so that they are in
  // flight during the rest of the set-up (the tensor-map descriptors are
  // prefetched first thing); it resumes after the CTA barrier at block p_j,
  // load p_c.  A fixed-length tile follows from the block index; a varlen
  // CTA's tile is located by the V-producer warp meanwhile, and the two warps
  // meet on a named barrier before the loads (once each, unconditionally).
  const uint64_t keep_l2 = policy_evict_last();    // K and V are re-read by other tiles/heads
  const uint64_t stream_l2 = policy_evict_first();  // Q is read once
  int p_j = 0, p_c = 0;
  if (warp == WARP_V && lane == 0) prefetch_tmap(&tm_v);
  if (warp == WARP_K && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    mbar_init(smem_u32(&sh.q_full), 1);
    for (int i = 0; i < NK; ++i) {
      mbar_init(smem_u32(&sh.ready[i]), 2);  // the key tile (arrival + bytes), the S buffer
      mbar_init(smem_u32(&sh.qk_done[i]), 1);
    }
    for (int i = 0; i < NS; ++i) mbar_arrive(smem_u32(&sh.ready[i]));  // buffers free at first
    for (int i = 0; i < NV; ++i) {
      mbar_init(smem_u32(&sh.v_full[i]), 1);
      mbar_init(smem_u32(&sh.v_empty[i]), 1);
    }
    for (int i = 0; i < NS; ++i) mbar_init(smem_u32(&sh.p_full[i]), NQ);
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&sh.pv_done[i]), 1);
    }
    mbar_init(smem_u32(&sh.l_full), NQ);
    for (int i = 0; i < NDEC; ++i) {
      mbar_init(smem_u32(&sh.dec_full[i]), 1);
      mbar_init(smem_u32(&sh.dec_read[i]), 2 + NQ);
    }
    sh.abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();  // the initialised barriers, seen by this thread's TMA loads
  }
  if (warp == WARP_MMA) tmem_alloc(smem_u32(&sh.tmem_base), TMEM_COLS);
  if constexpr (VARLEN) {
    if (warp == WARP_V) {
      const int i = (int)(blockIdx.x / a.Hq), h = (int)(blockIdx.x % a.Hq);
      if (a.B > 32 || !varlen_locate_small(a, i, h, lane, &sh.vt))
        varlen_locate(a, i, (int)(gridDim.x / a.Hq), h, lane, &sh.vt);
    }
    if (warp == WARP_V || warp == WARP_K) named_bar_sync(kSetupBarrier, 64);
  }
  if (warp == WARP_K && lane == 0 && (!VARLEN || sh.vt.s >= 0)) {
    VarTile v0{};
    if constexpr (VARLEN) v0 = sh.vt;
    const Tile x = tile_of<VARLEN>(a, v0, (int)blockIdx.x);
    const int hk0 = x.h / (a.Hq / a.Hkv);
    const int zq = x.b * a.Hq + x.h, zkv = x.b * a.Hkv + hk0;
    const int qy = VARLEN ? x.h : x.row0, qz = VARLEN ? x.off + x.row0 : zq;
    const uint32_t *sw = SET ? a.block_set + ((size_t)zq * a.n_t + x.t) * a.words : nullptr;
    mbar_expect_tx(smem_u32(&sh.q_full), TILE_BYTES);
    tma_load_3d(base + SMEM_Q, &tm_q, smem_u32(&sh.q_full), 0, qy, qz, stream_l2);
    tma_load_3d(base + SMEM_Q + HALF_BYTES, &tm_q, smem_u32(&sh.q_full), 64, qy, qz, stream_l2);
    for (; p_j < x.nblk && p_c < NK; ++p_j) {
      if constexpr (SET) {
        if (((__ldg(sw + (p_j >> 5)) >> (p_j & 31)) & 1u) == 0u) continue;
      }
      const int ky = VARLEN ? hk0 : p_j * BN, kz = VARLEN ? x.off + p_j * BN : zkv;
      const uint32_t dst = base + SMEM_K + p_c * TILE_BYTES;
      mbar_expect_tx(smem_u32(&sh.ready[p_c]), TILE_BYTES);
      tma_load_3d(dst, &tm_k, smem_u32(&sh.ready[p_c]), 0, ky, kz, keep_l2);
      tma_load_3d(dst + HALF_BYTES, &tm_k, smem_u32(&sh.ready[p_c]), 64, ky, kz, keep_l2);
      ++p_c;
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  // Varlen: sequence b holds tokens [off, off + T) of the packed tensors.  A
  // length or a threshold outside its range raises the bad-argument bit; the
  // sequence is then treated as empty, the threshold as 0.
  VarTile vt{};
  if constexpr (VARLEN) vt = sh.vt;
  const bool has_tile = !VARLEN || vt.s >= 0;  // varlen: a CTA past the last tile has none
  const Tile tile = tile_of<VARLEN>(a, vt, (int)blockIdx.x);
  const int t = tile.t, h = tile.h, b = tile.b;
  const int bh = b * a.Hq + h;
  const int hk = h / (a.Hq / a.Hkv);
  const int T = tile.T, off = tile.off;
  const float ln_lam = tile.ln_lam;
  const int row0 = tile.row0, nblk = tile.nblk;
  volatile int *abort = &sh.abort;
  const int zkv = b * a.Hkv + hk;
  // TMA coordinates (column, y, z) of key block j: [heads, T, 128] maps take
  // (row, head); the token-major varlen maps [total, heads, 128] take (head,
  // token).  (Q's, the same, are taken in the set-up.)
  auto kv_y = [&](int j) { return VARLEN ? hk : j * BN; };
  auto kv_z = [&](int j) { return VARLEN ? off + j * BN : zkv; };
  const uint32_t *set_words = SET ? a.block_set + ((size_t)bh * a.n_t + t) * a.words : nullptr;
  auto in_set = [&](int j) { return ((__ldg(set_words + (j >> 5)) >> (j & 31)) & 1u) != 0u; };


  if (!has_tile) {
    // varlen: no tile for this CTA (its bitmap clearing is done)
  } else if (warp == WARP_K) {
    // -------------------------------------------------------- Q/K producer --
    if (lane == 0) {
      int ki = p_c, cc = p_c;
      for (int j = p_j; j < nblk && !*abort; ++j) {
        if constexpr (SET) {
          if (!in_set(j)) continue;
        }
        const int c = SET ? cc++ : j;
        const int s = c % NK;
        // Stage s last held block c - NK, whose Q.K^T has completed.
        if (c >= NK &&
            !mbar_wait(smem_u32(&sh.qk_done[s]), ((c / NK) - 1) & 1, abort, a.err, kErrTimeout))
          break;
        const uint32_t dst = base + SMEM_K + s * TILE_BYTES;
        mbar_expect_tx(smem_u32(&sh.ready[s]), TILE_BYTES);
        tma_load_3d(dst, &tm_k, smem_u32(&sh.ready[s]), 0, kv_y(j), kv_z(j), keep_l2);
        tma_load_3d(dst + HALF_BYTES, &tm_k, smem_u32(&sh.ready[s]), 64, kv_y(j), kv_z(j),
                    keep_l2);
        ++ki;
      }
      // Drain: the last load issued into each slot has landed before exit
      // (earlier loads of a slot were consumed before the slot was reused;
      // the slot's phase also waits for its S buffer, freed by every decided
      // block, so this wait is only long after a failed wait elsewhere).
      mbar_wait_drain(smem_u32(&sh.q_full), 0);
      for (int s = 0; s < NK && s < ki; ++s) {
        const int last = s + ((ki - 1 - s) / NK) * NK;
        mbar_wait_drain(smem_u32(&sh.ready[s]), (last / NK) & 1);
      }
    }
  } else if (warp == WARP_V) {
    // ---------------------------------------------------------- V producer --
    if (lane == 0) {
      int vi = 0, cc = 0;
      for (int j = 0; j < nblk && !*abort; ++j) {
        if constexpr (SET) {
          if (!in_set(j)) continue;
        }
        const int c = SET ? cc++ : j;
        if (!mbar_wait(smem_u32(&sh.dec_full[c % NDEC]), (c / NDEC) & 1, abort, a.err,
                       kErrTimeout))
          break;
        const int keep = sh.dec[c % NDEC];
        mbar_arrive(smem_u32(&sh.dec_read[c % NDEC]));
        if (!keep) continue;
        const int s = vi % NV;
        if (vi >= NV &&
            !mbar_wait(smem_u32(&sh.v_empty[s]), ((vi / NV) - 1) & 1, abort, a.err, kErrTimeout))
          break;
        const uint32_t dst = base + SMEM_V + s * TILE_BYTES;
        mbar_expect_tx(smem_u32(&sh.v_full[s]), TILE_BYTES);
        tma_load_3d(dst, &tm_v, smem_u32(&sh.v_full[s]), 0, kv_y(j), kv_z(j), keep_l2);
        tma_load_3d(dst + HALF_BYTES, &tm_v, smem_u32(&sh.v_full[s]), 64, kv_y(j), kv_z(j),
                    keep_l2);
        ++vi;
      }
      for (int s = 0; s < NV && s < vi; ++s) {
        const int last = s + ((vi - 1 - s) / NV) * NV;
        mbar_wait_drain(smem_u32(&sh.v_full[s]), (last / NV) & 1);
      }
    }
  } else if (warp == WARP_MMA || warp == WARP_MMA2) {
    // ------------------------------------------- Q.K^T issuers (c even / odd) --
    // The whole warp waits (a warp-wide poll resolves faster than one lane's);
    // lane 0 issues.
    {
      const int mine = warp == WARP_MMA ? 0 : 1;
      bool ok = mbar_wait_warp(smem_u32(&sh.q_full), 0, abort, a.err, kErrTimeout);
      fence_after_sync();
      const uint64_t qdesc = kmajor_base(base + SMEM_Q);
      int cc = 0;
      for (int j = 0; ok && j < nblk; ++j) {
        if constexpr (SET) {
          if (!in_set(j)) continue;
        }
        const int c = SET ? cc++ : j;
        if ((c & 1) != mine) continue;
        const int s = c % NK, sb = c % NS;
        // Key tile landed and S buffer sb (last: block c - NS) free.
        if (!mbar_wait_warp(smem_u32(&sh.ready[s]), (c / NK) & 1, abort, a.err, kErrTimeout)) break;
        fence_after_sync();
        if (lane == 0) {
          const uint64_t kd = kmajor_base(base + SMEM_K + s * TILE_BYTES);
          const uint32_t d_s = tmem + sb * BN;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_ss(d_s, qdesc + kmajor_step(kk), kd + kmajor_step(kk), IDESC_QK, kk > 0);
          mma_commit(smem_u32(&sh.qk_done[s]));
        }
        __syncwarp();
      }
    }
  } else if (warp == WARP_PV) {
    // ---------------------------------------------------------- P.V issuer --
    if (lane == 0) {
      int kc = 0, vi = 0, cc = 0;
      for (int j = 0; j < nblk && !*abort; ++j) {
        if constexpr (SET) {
          if (!in_set(j)) continue;
        }
        const int i = SET ? cc++ : j;  // traversed-block position
        if (!mbar_wait(smem_u32(&sh.dec_full[i % NDEC]), (i / NDEC) & 1, abort, a.err,
                       kErrTimeout))
          break;
        const int keep = sh.dec[i % NDEC];
        mbar_arrive(smem_u32(&sh.dec_read[i % NDEC]));
        if (!keep) continue;
        const int pb = kc % NS, vs = vi % NV;
        if (!mbar_wait(smem_u32(&sh.p_full[kc % NS]), (kc / NS) & 1, abort, a.err, kErrTimeout))
          break;
        if (!mbar_wait(smem_u32(&sh.v_full[vs]), (vi / NV) & 1, abort, a.err, kErrTimeout))
          break;
        fence_after_sync();
        // P_i (bf16 pairs): keys [0,128) in columns [0,64) of S buffer i % NS.
        const uint32_t pt = tmem + (i % NS) * BN;
        const uint64_t vd = vmajor_base(base + SMEM_V + vs * TILE_BYTES);
        const uint32_t d_o = tmem + TMEM_O;
        const uint32_t acc0 = kc > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_bf16_ts(d_o, pt + kk * 8, vd + vmajor_step(kk), IDESC_PV, kk > 0 ? 1u : acc0);
        mma_commit(smem_u32(&sh.v_empty[vs]));
        mma_commit(smem_u32(&sh.ready[(i + NS) % NK]));  // S buffer free for block i + NS
        mma_commit(smem_u32(&sh.pv_done[pb]));
        ++kc;
        ++vi;
      }
    }
  } else {
    // ------------------------------------------------- deciders / exponentials --
    const bool decider = warp < NQ;
    const int quarter = warp & 3;                 // TMEM lane quarter
    const int r = quarter * 32 + lane;            // row within the tile == TMEM lane
    const int row = row0 + r;
    const bool valid = row < T;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = a.scale * kLog2e;           // raw score -> log2 units
    float mref = -INFINITY;                       // exp reference (log2 units)
    float l = 0.f;                                // row sum relative to mref
    int kc = 0;                                   // kept blocks exponentiated
    bool ok = true;
    auto needs_mask = [&](int j) {
      const int key0 = j * BN;
      return a.causal ? (key0 + BN - 1 > row0) : (key0 + BN > T);
    };

    if (decider) {
      // Per block: the full row max of S_j, the row vote against the running
      // max before the block, then one barrier round of the four deciders to
      // AND the votes.  Thread 0 publishes the decision and the bitmap.
      const float c2 = ln_lam * kLog2e;           // ln(lambda) in log2 units
      float m2 = -INFINITY;                       // running max (log2 units)
      uint32_t word = 0;
      uint32_t *bits = a.bits ? a.bits + ((size_t)bh * a.n_t + t) * a.words : nullptr;
      int sb = 0, cc = 0;
      int wcur = 0;  // block-set mode: next bitmap word to write
      for (int j = 0; j < nblk; ++j) {
        if constexpr (SET) {
          if (!in_set(j)) continue;
        }
        const int c = SET ? cc++ : j;
        // Once a wait has failed (the abort flag is up and every later wait
        // fails at once) the loop still runs to its end, so that the four
        // warps meet the vote barrier equally often.
        if (ok) ok = mbar_wait_warp(smem_u32(&sh.qk_done[c % NK]), (c / NK) & 1, abort, a.err, kErrTimeout);
        bool keep_vote = false;  // warp-uniform: some row of this warp keeps the block
        float mnew = m2;
        if (ok) {
          fence_after_sync();
          const uint32_t sa = lane_base + sb * BN;
          if (needs_mask(j)) mask_block_tmem(sa, j * BN, row, a.causal, T);
          uint32_t x0[32], x1[32], x2[32], x3[32];
          tmem_ld32(sa, x0);
          tmem_ld32(sa + 32, x1);
          tmem_ld32(sa + 64, x2);
          tmem_ld32(sa + 96, x3);
          tmem_wait_ld_regs(x0);
          tmem_wait_ld_regs(x1);
          tmem_wait_ld_regs(x2);
          tmem_wait_ld_regs(x3);
          const float mt =
              fmaxf(fmaxf(chunk_max(x0), chunk_max(x1)), fmaxf(chunk_max(x2), chunk_max(x3)));
          const float pm2 = mt * sl2;
          // With c < 0, "rowmax - m_new < c" is "rowmax - m_old < c" (a block
          // that raises the max fails both).
          const float diff = (mt == -INFINITY) ? -INFINITY : pm2 - m2;
          keep_vote = !__all_sync(0xffffffffu, !valid || (diff < c2));
          mnew = fmaxf(m2, pm2);
          sh.mdec[sb][r] = mnew;
          if constexpr (STATS) {
            // rowmax - m_new = min(rowmax - m_old, 0) (log2 units) over valid rows.
            float st = (valid && mt != -INFINITY) ? fminf(diff, 0.f) : -INFINITY;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) st = fmaxf(st, __shfl_xor_sync(0xffffffffu, st, o));
            if (lane == 0) sh.wstat[c & 1][warp] = st;
          }
          fence_before_sync();  // this warp's reads of S_j are complete
        }
        // The block is kept if any of the four warps votes keep: one
        // reduction on the deciders' named barrier.
        const bool any_keep = bar_red_or(kDeciderBarrier, NQ * 32, keep_vote);
        if (!ok) continue;
        const bool skip = STATS || !any_keep;
        m2 = mnew;
        if (STATS && tid == 0) {
          const float st = fmaxf(fmaxf(sh.wstat[c & 1][0], sh.wstat[c & 1][1]),
                                 fmaxf(sh.wstat[c & 1][2], sh.wstat[c & 1][3]));
          a.margin[((size_t)bh * a.n_t + t) * a.n_b + j] = st * kLn2;
        }
        if (lane == 0 && warp == (c & (NQ - 1))) {
          // Lane 0 of decider warp c % 4 publishes (the next vote barrier
          // keeps the publications in block order).  The slot's previous
          // decision (block c - NDEC) must have been read by all its readers;
          // on a timeout the abort flag is raised and every later wait fails.
          // A skipped block's S buffer is free: every decider has read it
          // (the vote barrier above) and nothing else will.  Released first:
          // the next Q.K^T into this buffer waits for it.
          if (skip) mbar_arrive(smem_u32(&sh.ready[(c + NS) % NK]));
          if (c < NDEC || mbar_wait(smem_u32(&sh.dec_read[c % NDEC]), ((c / NDEC) - 1) & 1,
                                    abort, a.err, kErrTimeout)) {
            sh.dec[c % NDEC] = skip ? 0 : 1;
            mbar_arrive(smem_u32(&sh.dec_full[c % NDEC]));
          }
        }
        if (tid == 0) {
          if constexpr (SET) {
            // Words before this block's are complete (untraversed blocks read 0).
            for (; wcur < (j >> 5); ++wcur) {
              if (!STATS) bits[wcur] = word;
              word = 0;
            }
          }
          if (skip) word |= 1u << (j & 31);
          if (!SET && !STATS && ((j & 31) == 31 || j == nblk - 1)) {
            bits[j >> 5] = word;
            word = 0;
          }
        }
        sb = sb == NS - 1 ? 0 : sb + 1;
      }
      if (tid == 0) {
        if constexpr (SET) {
          for (; wcur < a.words; ++wcur) {
            if (!STATS) bits[wcur] = word;
            word = 0;
          }
        } else if (!STATS) {
          for (int w = ((nblk - 1) >> 5) + 1; w < a.words; ++w) bits[w] = 0u;
        }
        if (STATS)
          for (int j = nblk; j < a.n_b; ++j) a.margin[((size_t)bh * a.n_t + t) * a.n_b + j] = NAN;
      }
    } else {
      // Per kept block: P_j = exp2(S_j - ref) as bf16 pairs into columns
      // [0,64) of the block's S buffer, the row sum, and an O rescale when
      // the exp reference moves by more than 2^8.
      int sb = 0, cc = 0;  // sb = c % NS
      for (int j = 0; ok && j < nblk; ++j) {
        if constexpr (SET) {
          if (!in_set(j)) continue;
        }
        const int c = SET ? cc++ : j;
        if (c > 0) sb = sb == NS - 1 ? 0 : sb + 1;
        if (!mbar_wait_warp(smem_u32(&sh.dec_full[c % NDEC]), (c / NDEC) & 1, abort, a.err,
                            kErrTimeout)) {
          ok = false;
          break;
        }
        const int keep = sh.dec[c % NDEC];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.dec_read[c % NDEC]));
        if (!keep) continue;
        const float mnew = sh.mdec[sb][r];
        bool rescale = false;
        float alpha = 1.f;
        if (mref == -INFINITY) {
          mref = mnew;
        } else if (mnew > mref + kRescaleLog2) {
          alpha = ex2(mref - mnew);
          mref = mnew;
          rescale = true;
        }
        fence_after_sync();
        const uint32_t sa = lane_base + sb * BN;  // scores already masked by the deciders
        const uint64_t sl2x2 = f2(sl2, sl2), negref2 = f2(-mref, -mref);
        uint64_t acc2[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          // Keys [64hh, 64hh+64): their P pairs land in columns [32hh, 32hh+32),
          // whose scores were loaded by this or the previous half.
          uint32_t x[32], y[32];
          tmem_ld32(sa + 64 * hh, x);
          tmem_ld32(sa + 64 * hh + 32, y);
          tmem_wait_ld_regs(x);
          tmem_wait_ld_regs(y);
          uint32_t pk[32];
          chunk_exp(x, sl2x2, negref2, acc2, pk);
          chunk_exp(y, sl2x2, negref2, acc2, pk + 16);
          tmem_st32(sa + 32 * hh, pk);
        }
        tmem_wait_st();
        float acc[4];
        f2_split(acc2[0], acc[0], acc[1]);
        f2_split(acc2[1], acc[2], acc[3]);
        l = l * alpha + ((acc[0] + acc[1]) + (acc[2] + acc[3]));
        // O rescale of this warp's rows (warp-wide if any row needs it), after
        // the previous P.V landed.
        if (__any_sync(0xffffffffu, rescale) && kc >= 1) {
          if (!mbar_wait_warp(smem_u32(&sh.pv_done[(kc - 1) % NS]), ((kc - 1) / NS) & 1, abort,
                              a.err, kErrTimeout)) {
            ok = false;
            break;
          }
          fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            const uint32_t oa = lane_base + TMEM_O + c * 32;
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
        if (lane == 0) mbar_arrive(smem_u32(&sh.p_full[kc % NS]));
        ++kc;
      }
      if (ok && kc > 0) {
        ok = mbar_wait_warp(smem_u32(&sh.pv_done[(kc - 1) % NS]), ((kc - 1) / NS) & 1, abort,
                            a.err, kErrTimeout);
      }
      sh.lfin[r] = l;
      sh.mfin[r] = mref;
      fence_before_sync();  // the final P.V is complete (observed above)
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.l_full));
    }

    // ---- epilogue: deciders take O columns [0,64), exponential warps [64,128)
    if (ok) ok = mbar_wait_warp(smem_u32(&sh.l_full), 0, abort, a.err, kErrTimeout);
    if (ok && !STATS) {
      fence_after_sync();
      const float lrow = sh.lfin[r];
      // Block-set mode: a tile that selected no block has no mass (O = 0,
      // LSE = -inf); its O accumulator was never written.
      const bool empty = SET && !(lrow > 0.f);
      const float inv = empty ? 0.f : 1.f / lrow;
      const int col0 = decider ? 0 : 64;
      // Output rows: [heads, T, 128], or token-major [total, Hq, 128] (varlen).
      const size_t orow_idx =
          VARLEN ? (size_t)(off + row) * a.Hq + h : (size_t)bh * a.T + row;
      __nv_bfloat16 *orow = (__nv_bfloat16 *)a.o + orow_idx * D + col0;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_base + TMEM_O + col0 + c * 32, o);
        tmem_wait_ld_regs(o);
        if (empty) {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        if (valid) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * q4 + 0]) * inv, __uint_as_float(o[8 * q4 + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[8 * q4 + 2]) * inv, __uint_as_float(o[8 * q4 + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[8 * q4 + 4]) * inv, __uint_as_float(o[8 * q4 + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[8 * q4 + 6]) * inv, __uint_as_float(o[8 * q4 + 7]) * inv);
            *reinterpret_cast<uint4 *>(orow + c * 32 + q4 * 8) = v;
          }
        }
      }
      if (valid && !decider)
        a.lse[VARLEN ? (size_t)h * a.total + off + row : (size_t)bh * a.T + row] =
            empty ? -INFINITY : sh.mfin[r] * kLn2 + logf(lrow);
    }
  }

  fence_before_sync();
  __syncthreads();
  if (warp == WARP_MMA) {
    fence_after_sync();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  if (a.cu_seqlens) {
    // Token-major [total, heads, 128] bf16, boxes of 64 columns x 1 head x
    // 128 tokens (the same shared-memory image as below); tokens past the
    // end read as zero.
    const int tot = a.total > 0 ? a.total : 1;
    if (!make_map_bf16_thd(&mq, a.q, a.Hq, tot, BM) || !make_map_bf16_thd(&mk, a.k, a.Hkv, tot, BN) ||
        !make_map_bf16_thd(&mv, a.v, a.Hkv, tot, BN))
      return cudaErrorInvalidValue;
  } else {
    // [heads, T, 128] bf16, boxes of 64 columns x 128 rows; rows past T read as zero.
    if (!make_map_bf16_3d(&mq, a.q, D, D, a.T, a.B * a.Hq, BM) ||
        !make_map_bf16_3d(&mk, a.k, D, D, a.T, a.B * a.Hkv, BN) ||
        !make_map_bf16_3d(&mv, a.v, D, D, a.T, a.B * a.Hkv, BN))
      return cudaErrorInvalidValue;
  }
  auto kernel = a.cu_seqlens  ? prefill_tc_kernel<false, false, true>
                : a.stats_only ? prefill_tc_kernel<true, false, false>
                : a.block_set  ? prefill_tc_kernel<false, true, false>
                               : prefill_tc_kernel<false, false, false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  // Varlen: at least one CTA per tile (a sequence of L tokens has ceil(L/Br)
  // tiles, so there are at most ceil(total/Br) + n_seq of them).
  const long units = a.cu_seqlens ? (long)a.Hq * ((a.total + BM - 1) / BM + a.B)
                                  : (long)a.B * a.Hq * a.n_t;
  kernel<<<(unsigned)units, NTHREADS, SMEM_ALLOC, s>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

}  // namespace attn_skip
