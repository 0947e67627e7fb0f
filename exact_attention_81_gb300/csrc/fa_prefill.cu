// fa_prefill.cu -- fused exact-attention forward ("prefill") kernel for sm_103a.
//
// One persistent CTA per SM walks a list of work tiles.  A work tile is one (batch, query
// head, 256-row query block; 128 rows at d > 128): two 128-row query sub-tiles that share
// one K/V stream, the
// larger-tile / two-tile ping-pong of "FlashAttention 1-4 详解", FlashAttention 4 section
// (tile (Br, Bc) -> (Br', Bc') with Br' ~ 2 Br).  For every 128-key K/V tile j the CTA
// computes, for each sub-tile t,
//     S_t = Q_t K_j^T                       (tcgen05.mma, fp32 accumulator in TMEM)
//     m_new = max(m, rowmax S_t * c),  P = 2^(S_t c - m_new),  l = 2^(m - m_new) l + rowsum P
//     O_t = 2^(m - m_new) O_t + P V_j       (P stored to TMEM as bf16, tcgen05.mma again)
// with c = scale * log2(e) folded into one FMA before the exp2 ("flash-attention",
// section 4, scale_apply_exp2), the O rescale done only for warps whose row maxima grew
// ("FlashAttention 1-4 详解", FlashAttention 4, conditional rescale when m_new > m) and,
// for 16-bit inputs, only when a row max grew past the reference max m by more than 8 (log2
// units; m stays put otherwise, so P <= 2^8 -- O / l and m + log2 l do not depend on which
// reference max P and l share), and
// the division by l deferred to the epilogue ("FlashAttention 1-4 详解", FlashAttention 2,
// normalise once after the inner loop).  The epilogue writes O (bf16) and the natural-log
// LSE = ln2 * (m + log2 l); O goes through a per-warp shared-memory box and TMA stores where
// shared memory allows (width <= 128, no ALiBi, single CTAs).  S and P never leave the SM.
//
// Warp roles (384 threads, three warpgroups):
//   warps 0-3  softmax + correction + epilogue for sub-tile 0 (thread = query row)
//   warps 4-7  the same for sub-tile 1
//   warp  8    tile scheduler and TMA producer: Q tiles and the K/V ring (one lane)
//   warp  9    TMEM allocator and MMA issuer (the whole warp runs the issuing loop, one
//              elected lane executes each MMA)
//   warps 10-11 idle
// The third warpgroup gives registers back (setmaxnreg) so that the two softmax
// warpgroups can hold a full 128-score row per thread without spilling.
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+d), O_1 [384,384+d).
// P_t overwrites the first 64 columns of S_t as packed bf16 pairs and is the A operand of
// the PV MMA straight from TMEM.
//
// Causal masking ("FlashAttention 1-4 详解", FlashAttention 2 engineering notes: skip the
// tiles above the diagonal, ~N^2/2 work) limits each sub-tile to the K/V tiles that hold a
// visible key and masks only the tiles that straddle the diagonal or the sequence end.
// The score modifiers of the capabilities table of "flash-attention" (sliding window,
// softcap, ALiBi) run in the mask modes MASK_WINDOW (a window alone) and MASK_MOD (a
// softcap or ALiBi, with or without a window): a 256-row block streams only the K/V
// tiles between its first row's window start and its last row's window end, each
// sub-tile joins the stream steps its rows can see, and the scores are softcapped and
// biased in the log2 domain before the row max.
// Tiles are handed out dynamically: the producer lane of each CTA takes the next ticket
// from a per-launch atomic counter and passes the tile to the other roles through a small
// shared-memory ring.  Causal (and right-bounded window) tiles go out longest first within
// groups of a few (batch, head) pairs, one query-block level at a time over the group, so
// that CTAs running at the same time share a few heads' K/V in L2, long tiles start early,
// and the launch ends on short tiles instead of one head's longest ones.  On taking a
// ticket the producer prefetches the tile's Q and first K/V boxes into L2, about two steps
// before the Q buffer is free for them.
#include <atomic>
#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int BR = 128;             // query rows per sub-tile (MMA M)
constexpr int BC = 128;             // keys per K/V tile
constexpr int NTHREADS = 384;
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int SCHED_DEPTH = 4;      // tiles in flight between the scheduler and the roles
constexpr int SOFTMAX_REGS = 200;   // 2 x 128 threads x 200
constexpr int OTHER_REGS = 104;     //   + 128 threads x 104 = 384 threads x 168 at launch
constexpr int IDLE_REGS = 24;       // wide kernel: the unused second softmax warpgroup
constexpr int NUM_SCHED_SLOTS = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr int BOX_BYTES = 128 * 128;  // one TMA box: 128 rows x 64 bf16 (128 B, swizzled)
constexpr float LN2 = 0.6931471805599453f;

__host__ __device__ constexpr uint32_t s_col(int t) { return static_cast<uint32_t>(t * 128); }
__host__ __device__ constexpr uint32_t o_col(int t) {
  return static_cast<uint32_t>(256 + t * 128);
}

// D <= 128: two query sub-tiles per work tile, ring slots of one [128 x D] K or V tile.
// D = 256 ("wide"): one sub-tile with S double-buffered in TMEM (S_0, S_1, O = 512
// columns), ring slots of half a tile (the d halves), PV as two N = 128 products.
// F8 (E4M3 inputs, D = 128): one 128-byte box per row; V arrives transposed ([d, keys],
// K-major like K), P goes through shared memory as E4M3 (both PV operands K-major).
// PAIR (D = 128, 16-bit): a CTA pair computes each sub-tile as one M = 256 product
// (cta_group::2): each CTA holds 128 of its query rows; a ring slot holds this CTA's half of
// a K tile (64 keys x D) or of a V tile (128 keys x D / 2 columns), so the pair reads each
// K/V tile once and each CTA half of it.
template <int D, bool F16 = false, bool F8 = false, bool PAIR = false>
struct Cfg {
  static constexpr bool WIDE = D > 128;
  static constexpr int NSUB = WIDE ? 1 : 2;              // query sub-tiles per work tile
  static constexpr int SUB_ROWS = PAIR ? 256 : BR;       // query rows of a sub-tile (MMA M)
  static constexpr int EB = F8 ? 1 : 2;                  // bytes per element
  static constexpr int KCH = D * EB / 128;               // 128-byte boxes per row
  static constexpr int BOX_ELEMS = 128 / EB;             // elements of a row per box
  static constexpr int TILE_BYTES = KCH * BOX_BYTES;     // one [128 x D] tile
  static constexpr int SLOT_BYTES = (WIDE || PAIR) ? TILE_BYTES / 2 : TILE_BYTES;
  static constexpr int NSLOTS =
      PAIR ? 10 : (WIDE ? 5 : (F8 ? 8 : (D == 128 ? 4 : 8)));  // K/V ring depth
  static constexpr int Q_OFF = 0;
  static constexpr int RING_OFF = NSUB * TILE_BYTES;
  static constexpr int P_OFF = RING_OFF + NSLOTS * SLOT_BYTES;  // F8: E4M3 P per sub-tile
  static constexpr int P_BYTES = F8 ? NSUB * BR * BC : 0;
  static constexpr int BAR_OFF = P_OFF + P_BYTES;
  static constexpr int SMEM_BYTES = BAR_OFF + 512 + 1024;  // barriers + alignment slack
  static constexpr uint32_t IDESC_S =
      F8 ? idesc_e4m3_f32(128, BC) : idesc_bf16_f32(SUB_ROWS, BC, false, false, F16);
  static constexpr uint32_t IDESC_PV =
      F8 ? idesc_e4m3_f32(128, D) : idesc_bf16_f32(SUB_ROWS, WIDE ? 128 : D, false, true, F16);
  static_assert(!PAIR || (D == 128 && !F8), "CTA pairs: 16-bit inputs at width 128");
};
static_assert(Cfg<128, false, true>::SMEM_BYTES <= 227 * 1024, "fp8 prefill exceeds smem");
static_assert(Cfg<256>::SMEM_BYTES <= 227 * 1024, "wide prefill exceeds shared memory");
static_assert(Cfg<128, false, false, true>::SMEM_BYTES <= 227 * 1024, "pair prefill exceeds smem");

// ALiBi column bias built by the tensor core (ALiBi without a softcap; 16-bit inputs, width
// <= 128, one CTA).  On a tile whose keys all lie at or before the position of every row of
// the sub-tile, the bias -slope |pos - key| is slope (key - kbase) plus a per-row constant;
// its per-column part, divided by the score scale, enters S through one more 128 x 128 x 16
// MMA ahead of Q K^T: A is a ones matrix (1 in k = 0..2), B holds in row i a three-term bf16
// split of i slope / scale (k = 0..2).  Both are K-major and 128B-swizzled (only the first
// 32 bytes of each 128-byte row are read; the second 16 bytes stay zero), 16 KB each,
// right after the barriers.
template <int D, int MASK, bool F8, bool PAIR>
__host__ __device__ constexpr bool abias() {
  return MASK == MASK_ALIBI && !F8 && !PAIR && D <= 128;
}
constexpr int ABIAS_BYTES = 2 * BR * 128;
// Staged O stores (PrefillArgs::o_tma): one 32-row x 64-column box (4 KB, 128-byte swizzled)
// per softmax warp at STG_OFF, the place of the ALiBi operands, which leave no room for it.
template <int D, int MASK, bool F8, bool PAIR>
__host__ __device__ constexpr bool stg_ok() {
  return !PAIR && D <= 128 && MASK != MASK_ALIBI;
}
constexpr int STG_WARP_BYTES = 32 * 128;
constexpr int STG_BYTES = 8 * STG_WARP_BYTES;
template <int D, int MASK, bool F16, bool F8, bool PAIR>
__host__ __device__ constexpr int prefill_smem() {
  using C = Cfg<D, F16, F8, PAIR>;
  return abias<D, MASK, F8, PAIR>()    ? C::BAR_OFF + 1024 + ABIAS_BYTES + 1024
         : stg_ok<D, MASK, F8, PAIR>() ? C::BAR_OFF + 1024 + STG_BYTES + 1024
                                       : C::SMEM_BYTES;
}
static_assert(prefill_smem<128, MASK_CAUSAL, false, false, false>() <= 227 * 1024,
              "prefill with O staging exceeds shared memory");
static_assert(prefill_smem<128, MASK_CAUSAL, false, true, false>() <= 227 * 1024,
              "fp8 prefill with O staging exceeds shared memory");
static_assert(prefill_smem<128, MASK_ALIBI, false, false, false>() <= 227 * 1024,
              "ALiBi prefill exceeds shared memory");

// Per-launch tile-ticket counters: [slot][0] = next ticket, [slot][1] = CTAs finished.
// The host gives each launch its own slot (round robin); the last CTA of a launch to
// finish resets the slot to zero for its next user.
__device__ unsigned int g_sched[NUM_SCHED_SLOTS][2];

struct Bars {
  uint64_t sched_full[SCHED_DEPTH], sched_empty[SCHED_DEPTH];
  int sched_tile[SCHED_DEPTH];
  uint64_t q_full, q_empty;
  uint64_t kv_full[10], kv_empty[10];
  uint64_t s_full[2], p_ready[2], o_full[2], o_empty[2];  // per sub-tile (wide: per S buffer)
  uint64_t pv_done;  // wide: PV(j) complete, before the softmax of j + 1 rescales O
  uint64_t mma_done;
  uint64_t exit_bar;  // CTA pairs: both CTAs are done with each other's shared memory
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 512, "prefill barriers exceed their shared-memory region");

struct TileInfo {
  bool half;        // a half tile: sub-tile 0 only (rows shifted by 128 for the second half)
  int b, h, hk;
  int q_row0;       // first query row of the block (NSUB x 128 rows), within its sequence
  int q_tok, k_tok; // packed-token offset of the sequence (varlen), else 0
  int tma_b;        // batch coordinate of the TMA maps (0 for varlen)
  int nq, nk;       // sequence lengths
  int nrows[2];     // valid query rows per sub-tile
  // The block streams K/V tiles kv0, kv0+1, ...; sub-tile t takes part in stream steps
  // [js[t], je[t]) and so visits nkv[t] = je[t] - js[t] tiles (0: its rows see no key).
  int kv0;
  int js[2], je[2], nkv[2];
  // Key tile of stream step j: kt_first + kdir * j (kdir = -1: the tiles run last-first).
  int kt_first, kdir;
};

// SUB: query rows of a sub-tile (128; 256 for a CTA pair, whose CTAs hold 128 rows each).
// `ticket` is a tile number, or at or past a.half_from a half-tile ticket: ticket
// half_from + 2 i + s stands for half s of tile half_from + i.
template <int MASK, int NSUB, int SUB = BR>
__device__ __forceinline__ TileInfo tile_info(const PrefillArgs &a, int ticket) {
  TileInfo ti;
  int tile = ticket, half = -1;
  if (NSUB == 2 && ticket >= a.half_from) {
    const int hh = ticket - a.half_from;
    half = hh & 1;
    tile = a.half_from + (hh >> 1);
  }
  ti.half = half >= 0;
  const bool desc = MASK == MASK_CAUSAL || (mask_has_window(MASK) && a.desc);
  int bh, r;
  if (desc && a.head_group > 1) {
    // Longest first across groups of head_group (batch, head) pairs: a group's tiles go
    // out one query-block level at a time over all its pairs, so that the last tickets of
    // the launch are short blocks of many heads (head by head, the last head's longest
    // blocks started when little other work was left), while the CTAs running together
    // still share a few heads' K/V in L2.
    const int per = a.head_group * a.mblocks;
    const int g = tile / per;
    const int r2 = tile - g * per;
    const int gs = min(a.head_group, a.num_tiles / a.mblocks - g * a.head_group);
    r = r2 / gs;
    bh = g * a.head_group + (r2 - r * gs);
  } else {
    bh = tile / a.mblocks;
    r = tile - bh * a.mblocks;
  }
  const int mb = desc ? (a.mblocks - 1 - r) : r;
  ti.b = bh / a.Hq;
  ti.h = bh - ti.b * a.Hq;
  ti.hk = ti.h / a.group;
  ti.q_row0 = mb * NSUB * SUB + (half > 0 ? BR : 0);
  if (a.varlen) {
    const int q0 = a.cu_q[ti.b], q1 = a.cu_q[ti.b + 1];
    const int k0 = a.cu_k[ti.b], k1 = a.cu_k[ti.b + 1];
    const bool bad = q0 < 0 || q1 < q0 || q1 > a.total_q || k0 < 0 || k1 < k0 ||
                     k1 > a.total_k || (q1 - q0) > a.Nq;
    ti.q_tok = bad ? 0 : q0;
    ti.k_tok = bad ? 0 : k0;
    ti.nq = bad ? 0 : q1 - q0;
    ti.nk = bad ? 0 : k1 - k0;
    ti.tma_b = 0;
  } else {
    ti.q_tok = 0;
    ti.k_tok = 0;
    ti.nq = a.Nq;
    ti.nk = a.Nk;
    ti.tma_b = ti.b;
  }
  const int nkv_all = (ti.nk + BC - 1) / BC;
  int lo[2], hi[2];  // K/V tile range [lo, hi) of each sub-tile
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int first = ti.q_row0 + t * SUB;
    const int nr = t < (ti.half ? 1 : NSUB) ? min(max(ti.nq - first, 0), SUB) : 0;
    ti.nrows[t] = nr;
    lo[t] = 0;
    hi[t] = 0;
    if (nr == 0) {
    } else if (MASK == MASK_NONE) {
      hi[t] = nkv_all;
    } else if (MASK == MASK_CAUSAL) {
      const long long last_key = static_cast<long long>(first) + nr - 1 + ti.nk - ti.nq;
      hi[t] = last_key < 0 ? 0 : min(static_cast<int>(last_key / BC) + 1, nkv_all);
    } else {
      // Keys some row of the sub-tile may see: from the first row's window start to the
      // last row's window end, clipped to the sequence.
      const long long off = static_cast<long long>(ti.nk) - ti.nq;
      const long long klo = a.wl >= 0 ? max(first + off - a.wl, 0ll) : 0ll;
      const long long khi = a.wr >= 0 ? min(first + nr - 1 + off + a.wr, ti.nk - 1ll)
                                      : ti.nk - 1ll;
      if (klo <= khi) {
        lo[t] = static_cast<int>(klo / BC);
        hi[t] = static_cast<int>(khi / BC) + 1;
      }
    }
  }
  const bool act0 = hi[0] > lo[0], act1 = hi[1] > lo[1];
  ti.kv0 = act0 ? (act1 ? min(lo[0], lo[1]) : lo[0]) : (act1 ? lo[1] : 0);
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const bool act = hi[t] > lo[t];
    ti.js[t] = act ? lo[t] - ti.kv0 : 0;
    ti.je[t] = act ? hi[t] - ti.kv0 : 0;
    ti.nkv[t] = ti.je[t] - ti.js[t];
  }
  ti.kt_first = ti.kv0;
  ti.kdir = 1;
  if ((MASK == MASK_ALIBI || MASK == MASK_MOD) && a.kv_rev) {
    // Last-first: step j streams tile kv0 + n - 1 - j, so sub-tile t's tiles
    // [kv0 + js, kv0 + je) are the steps [n - je, n - js).
    const int n = max(ti.je[0], ti.je[1]);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (ti.nkv[t] > 0) {
        const int js = ti.js[t];
        ti.js[t] = n - ti.je[t];
        ti.je[t] = n - js;
      }
    }
    ti.kt_first = ti.kv0 + n - 1;
    ti.kdir = -1;
  }
  return ti;
}

// Whether every key of the tile at kbase lies at or before the position of every row of
// sub-tile t (the first row has the smallest position, so it decides for all).
__device__ __forceinline__ bool alibi_lin(const TileInfo &ti, int t, int kbase) {
  return ti.q_row0 + t * BR + (ti.nk - ti.nq) - kbase >= BC - 1;
}

__device__ __forceinline__ bool varlen_bad(const PrefillArgs &a, int b) {
  const int q0 = a.cu_q[b], q1 = a.cu_q[b + 1];
  const int k0 = a.cu_k[b], k1 = a.cu_k[b + 1];
  return q0 < 0 || q1 < q0 || q1 > a.total_q || k0 < 0 || k1 < k0 || k1 > a.total_k ||
         (q1 - q0) > a.Nq;
}

// Both issue helpers are warp-collective (the whole MMA warp runs them, one lane issues).
// S_t = Q_t K^T: D/16 MMAs of 128 x 128 x 16.  Both operands K-major, 128B-swizzled:
// k-step kk lives in box kk/4 at byte offset 32*(kk%4) inside each 128-byte row.
template <int D, bool F16, bool F8 = false>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  if constexpr (F8) {
    // E4M3: K = 32 per MMA, so D / 32 MMAs, 32 bytes of each 128-byte row apiece.
#pragma unroll
    for (int kk = 0; kk < D / 32; ++kk) {
      const uint32_t off = static_cast<uint32_t>((kk >> 2) * BOX_BYTES + (kk & 3) * 32);
      mma_f8_ss_w(d_tmem, sw128_desc(q_smem + off, 16, 1024),
                  sw128_desc(k_smem + off, 16, 1024), Cfg<D, F16, true>::IDESC_S,
                  kk > 0 ? 1u : 0u);
    }
    return;
  }
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = static_cast<uint32_t>((kk >> 2) * BOX_BYTES + (kk & 3) * 32);
    mma_bf16_ss_w(d_tmem, sw128_desc(q_smem + off, 16, 1024),
                  sw128_desc(k_smem + off, 16, 1024), Cfg<D, F16>::IDESC_S, kk > 0 ? 1u : 0u);
  }
}

// S_t = A B^T + Q_t K^T: the ALiBi column bias (bf16 MMA over the two bias operands at
// bias_smem) and then the D/16 MMAs of issue_s, accumulating onto it.
template <int D, bool F16>
__device__ __forceinline__ void issue_s_alibi(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem,
                                              uint32_t bias_smem) {
  mma_bf16_ss_w(d_tmem, sw128_desc(bias_smem, 16, 1024),
                sw128_desc(bias_smem + static_cast<uint32_t>(BR * 128), 16, 1024),
                idesc_bf16_f32(BR, BC, false, false, false), 0u);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = static_cast<uint32_t>((kk >> 2) * BOX_BYTES + (kk & 3) * 32);
    mma_bf16_ss_w(d_tmem, sw128_desc(q_smem + off, 16, 1024),
                  sw128_desc(k_smem + off, 16, 1024), Cfg<D, F16>::IDESC_S, 1u);
  }
}

// O_t (+)= P_t V: BC/16 MMAs of 128 x D x 16.  P from TMEM (8 columns of bf16 pairs per
// k-step); V MN-major, 128B-swizzled: 16 keys = 2048 bytes per k-step, d halves one box apart.
template <int D, bool F16>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_smem,
                                         bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < BC / 16; ++kk) {
    mma_bf16_ts_w(o_tmem, p_tmem + static_cast<uint32_t>(kk * 8),
                  sw128_desc(v_smem + static_cast<uint32_t>(kk * 16 * 128), BOX_BYTES, 1024),
                  Cfg<D, F16>::IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// CTA pairs (issued by the even CTA; both CTAs' operands at the same addresses).
// S_t = Q_t K^T as M = 256: each CTA's Q sub-tile holds its 128 rows (128-row boxes), its
// K half holds 64 keys (64-row boxes, 8 KB apart); D/16 MMAs of 256 x 128 x 16.
template <int D, bool F16>
__device__ __forceinline__ void issue_s_pair(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t in_row = static_cast<uint32_t>((kk & 3) * 32);
    mma_bf16_ss_pair_w(d_tmem,
                       sw128_desc(q_smem + static_cast<uint32_t>((kk >> 2) * BOX_BYTES) + in_row,
                                  16, 1024),
                       sw128_desc(k_smem + static_cast<uint32_t>((kk >> 2) * (BOX_BYTES / 2)) +
                                      in_row, 16, 1024),
                       Cfg<D, F16, false, true>::IDESC_S, kk > 0 ? 1u : 0u);
  }
}

// O_t (+)= P_t V as M = 256, N = D: P from each CTA's TMEM, each CTA's V half one MN-major box
// of D / 2 = 64 columns for the 128 keys (16 keys = 2048 bytes per k-step).
template <int D, bool F16>
__device__ __forceinline__ void issue_pv_pair(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_smem,
                                              bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < BC / 16; ++kk) {
    mma_bf16_ts_pair_w(o_tmem, p_tmem + static_cast<uint32_t>(kk * 8),
                       sw128_desc(v_smem + static_cast<uint32_t>(kk * 16 * 128), BOX_BYTES, 1024),
                       Cfg<D, F16, false, true>::IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// FP8: O_t (+)= P_t V with P_t [128 queries x 128 keys] E4M3 in shared memory and V^T
// [D x 128 keys] E4M3 from the ring, both K-major; 4 MMAs of 128 x D x 32.
template <int D>
__device__ __forceinline__ void issue_pv_f8(uint32_t o_tmem, uint32_t p_smem, uint32_t vt_smem,
                                            bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < BC / 32; ++kk) {
    const uint32_t off = static_cast<uint32_t>(kk * 32);
    mma_f8_ss_w(o_tmem, sw128_desc(p_smem + off, 16, 1024), sw128_desc(vt_smem + off, 16, 1024),
                Cfg<D, false, true>::IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// ------------------------------------------------------------------------------------
// Scheduler + producer (one lane).  Takes tickets from the launch's counter, publishes each
// tile to the scheduler ring, then issues its Q tile and its K/V ring loads (ring order
// K_0, V_0, K_1, V_1, ...).  A ticket past the last tile is published as -1 (end).

template <int D, int MASK, bool F8 = false>
__device__ void producer_role(const PrefillArgs &a, const CUtensorMap *tmq,
                              const CUtensorMap *tmk, const CUtensorMap *tmv, uint8_t *smem,
                              Bars *bars, const WaitCtl &wc) {
  using C = Cfg<D, false, F8>;
  uint32_t kv_iter = 0, q_iter = 0;
  unsigned int *ctr = g_sched[a.sched_slot];
  // One ring slot: `boxes` 64-column boxes of rows [row0, row0 + 128) from map m, the first
  // at column c0.  False if the wait gave up.
  auto load_slot = [&](const CUtensorMap *m, int c0, int boxes, int hk, int row0, int b) {
    const int slot = static_cast<int>(kv_iter % C::NSLOTS);
    const uint32_t use = kv_iter / C::NSLOTS;
    if (!mbar_wait(&bars->kv_empty[slot], (use & 1u) ^ 1u, wc)) return false;
    mbar_arrive_expect_tx(&bars->kv_full[slot], C::SLOT_BYTES);
    for (int c = 0; c < boxes; ++c)
      tma_load_4d(smem + C::RING_OFF + slot * C::SLOT_BYTES + c * BOX_BYTES, m,
                  &bars->kv_full[slot], (c0 + c) * C::BOX_ELEMS, hk, row0, b);
    ++kv_iter;
    return true;
  };
  // FP8: one [D rows x 128 keys] tile of V^T, map dims {keys, d, kv head, batch}.
  auto load_vt = [&](int hk, int key0, int b) {
    const int slot = static_cast<int>(kv_iter % C::NSLOTS);
    const uint32_t use = kv_iter / C::NSLOTS;
    if (!mbar_wait(&bars->kv_empty[slot], (use & 1u) ^ 1u, wc)) return false;
    mbar_arrive_expect_tx(&bars->kv_full[slot], C::SLOT_BYTES);
    tma_load_4d(smem + C::RING_OFF + slot * C::SLOT_BYTES, tmv, &bars->kv_full[slot], key0, 0,
                hk, b);
    ++kv_iter;
    return true;
  };
  for (uint32_t k = 0;; ++k) {
    // Failure injection: publish nothing and load nothing; every other role's first wait
    // runs into the wait limit.
    if (a.inject) break;
    const int ticket = static_cast<int>(atomicAdd(&ctr[0], 1u));
    const int tile = ticket < a.num_tickets ? ticket : -1;
    const int rs = static_cast<int>(k % SCHED_DEPTH);
    if (!mbar_wait(&bars->sched_empty[rs], ((k / SCHED_DEPTH) & 1u) ^ 1u, wc)) goto out;
    bars->sched_tile[rs] = tile;
    mbar_arrive(&bars->sched_full[rs]);
    if (tile < 0) break;
    const TileInfo ti = tile_info<MASK, C::NSUB>(a, tile);
    if (a.varlen && (ti.q_row0 == 0) && varlen_bad(a, ti.b)) atomicOr(a.err, DEVERR_BAD_CU_SEQLENS);
    const int n = max(ti.je[0], ti.je[1]);
    if (n == 0) continue;
    const int krow = ti.k_tok + ti.kt_first * BC;  // K/V row of stream step j: krow + j kst
    const int kst = ti.kdir * BC;
    if (q_iter > 0) {
      // The ticket is taken while the previous tile still has about two steps to run, and
      // the Q buffer is free only after its last S: pull this tile's Q and first K / V
      // tiles into L2 now, so that the loads below hit L2 instead of waiting on HBM (where
      // CTAs with equal-length tiles all fetch their next Q at the same time).
      for (int t = 0; t < (ti.half ? 1 : C::NSUB); ++t)
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_prefetch_4d(tmq, c * C::BOX_ELEMS, ti.h, ti.q_tok + ti.q_row0 + t * BR, ti.tma_b);
#pragma unroll
      for (int c = 0; c < C::KCH; ++c) {
        tma_prefetch_4d(tmk, c * C::BOX_ELEMS, ti.hk, krow, ti.tma_b);
        if (!F8) tma_prefetch_4d(tmv, c * C::BOX_ELEMS, ti.hk, krow, ti.tma_b);
      }
      if (!mbar_wait(&bars->q_empty, (q_iter - 1) & 1u, wc)) goto out;
    }
    {
      const int nsub = ti.half ? 1 : C::NSUB;
      mbar_arrive_expect_tx(&bars->q_full, nsub * C::TILE_BYTES);
      for (int t = 0; t < nsub; ++t)
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d(smem + C::Q_OFF + t * C::TILE_BYTES + c * BOX_BYTES, tmq, &bars->q_full,
                      c * C::BOX_ELEMS, ti.h, ti.q_tok + ti.q_row0 + t * BR, ti.tma_b);
    }
    ++q_iter;
    if (!C::WIDE && !F8 && ti.half) {
      // half tile: S is double-buffered, so K(j + 1) is needed before V(j): ring order
      // K_0, K_1, V_0, K_2, V_1, ..., V_{n-1}
      bool ok = load_slot(tmk, 0, C::KCH, ti.hk, krow, ti.tma_b) &&
                (n < 2 || load_slot(tmk, 0, C::KCH, ti.hk, krow + kst, ti.tma_b));
      for (int j = 0; ok && j < n; ++j)
        ok = load_slot(tmv, 0, C::KCH, ti.hk, krow + j * kst, ti.tma_b) &&
             (j + 2 >= n || load_slot(tmk, 0, C::KCH, ti.hk, krow + (j + 2) * kst, ti.tma_b));
      if (!ok) goto out;
    } else if constexpr (C::WIDE) {
      // Ring order K_0, K_1, V_0, K_2, V_1, ..., V_{n-1} (the MMA issues S one step ahead),
      // each tile as two slots: d columns [0, 128) then [128, 256).
      bool ok = load_slot(tmk, 0, 2, ti.hk, krow, ti.tma_b) &&
                load_slot(tmk, 2, 2, ti.hk, krow, ti.tma_b);
      for (int j = 1; ok && j < n; ++j)
        ok = load_slot(tmk, 0, 2, ti.hk, krow + j * kst, ti.tma_b) &&
             load_slot(tmk, 2, 2, ti.hk, krow + j * kst, ti.tma_b) &&
             load_slot(tmv, 0, 2, ti.hk, krow + (j - 1) * kst, ti.tma_b) &&
             load_slot(tmv, 2, 2, ti.hk, krow + (j - 1) * kst, ti.tma_b);
      ok = ok && load_slot(tmv, 0, 2, ti.hk, krow + (n - 1) * kst, ti.tma_b) &&
           load_slot(tmv, 2, 2, ti.hk, krow + (n - 1) * kst, ti.tma_b);
      if (!ok) goto out;
    } else if constexpr (F8) {
      // V^T columns of the sequence's keys: from column 0 per batch entry (dense), or, packed
      // sequences, from the 16-aligned column roundup16(first token) + 16 b that the varlen
      // transpose gives sequence b (a TMA box must start on a 16-byte boundary).
      const int vrow = (a.varlen ? ((ti.k_tok + 15) & ~15) + 16 * ti.b : 0) + ti.kt_first * BC;
      for (int j = 0; j < n; ++j)
        if (!load_slot(tmk, 0, C::KCH, ti.hk, krow + j * kst, ti.tma_b) ||
            !load_vt(ti.hk, vrow + j * kst, ti.tma_b))
          goto out;
    } else {
      for (int j = 0; j < n; ++j)
        if (!load_slot(tmk, 0, C::KCH, ti.hk, krow + j * kst, ti.tma_b) ||
            !load_slot(tmv, 0, C::KCH, ti.hk, krow + j * kst, ti.tma_b))
          goto out;
    }
  }
out:
  // This CTA takes no more tickets (it reached the end, or gave up): count it as finished.
  // Every CTA takes exactly one ticket past the last tile, so the launch took num_tiles +
  // gridDim.x tickets in all; another count means that another launch ran on the same slot
  // at the same time (or a CTA gave up, which sets its own error bit).  The last CTA of the
  // launch to finish resets the counters for the slot's next launch.
  __threadfence();
  if (atomicAdd(&ctr[1], 1u) == gridDim.x - 1) {
    const unsigned int taken = atomicAdd(&ctr[0], 0u);
    if (!a.inject && taken != static_cast<unsigned int>(a.num_tickets) + gridDim.x)
      atomicOr(a.err, DEVERR_SCHED_OVERLAP);
    atomicExch(&ctr[0], 0u);
    atomicExch(&ctr[1], 0u);
  }
  // Teardown: let every bulk copy this thread issued land before the CTA may exit.
  for (int s = 0; s < C::NSLOTS; ++s) {
    if (kv_iter > static_cast<uint32_t>(s)) {
      const uint32_t uses = (kv_iter - 1 - s) / C::NSLOTS + 1;
      mbar_wait_teardown(&bars->kv_full[s], (uses - 1) & 1u, 1000000000ull);
    }
  }
  if (q_iter > 0) mbar_wait_teardown(&bars->q_full, (q_iter - 1) & 1u, 1000000000ull);
}

// Scheduler + producer of a CTA pair (one lane in each CTA).  The even CTA takes the tickets
// and publishes each tile to both CTAs' scheduler rings (its own, and the odd CTA's through a
// shared::cluster store and a remote arrival); every consumer of both CTAs frees the entry on
// the even CTA's ring.  Each CTA loads its own 128 rows of both query sub-tiles, and its half
// of every K tile (keys [64 rank, 64 rank + 64)) and V tile (columns [64 rank, 64 rank + 64)),
// counted on the even CTA's barriers, where the even CTA posts the bytes of both halves.  The
// ring order and slot sequence are the same in both CTAs.
template <int D, int MASK>
__device__ void producer_role_pair(const PrefillArgs &a, const CUtensorMap *tmq,
                                   const CUtensorMap *tmk, const CUtensorMap *tmv, uint8_t *smem,
                                   Bars *bars, const WaitCtl &wc, uint32_t rank) {
  using C = Cfg<D, false, false, true>;
  uint32_t kv_iter = 0, q_iter = 0;
  unsigned int *ctr = g_sched[a.sched_slot];
  const uint32_t peer = rank ^ 1u;
  auto load_half = [&](bool is_v, int hk, int row0, int b) {
    const int slot = static_cast<int>(kv_iter % C::NSLOTS);
    const uint32_t use = kv_iter / C::NSLOTS;
    if (!mbar_wait(&bars->kv_empty[slot], (use & 1u) ^ 1u, wc)) return false;
    if (*wc.abort) return false;
    if (rank == 0) mbar_arrive_expect_tx(&bars->kv_full[slot], 2 * C::SLOT_BYTES);
    const uint32_t fb = mapa_shared(&bars->kv_full[slot], 0);
    uint8_t *dst = smem + C::RING_OFF + slot * C::SLOT_BYTES;
    if (is_v) {
      tma_load_4d_pair(dst, tmv, fb, static_cast<int>(rank) * 64, hk, row0, b);
    } else {
#pragma unroll
      for (int c = 0; c < C::KCH; ++c)
        tma_load_4d_pair(dst + c * (BOX_BYTES / 2), tmk, fb, c * 64, hk,
                         row0 + static_cast<int>(rank) * 64, b);
    }
    ++kv_iter;
    return true;
  };
  for (uint32_t k = 0;; ++k) {
    if (a.inject) break;  // failure injection: no ticket, no load
    const int rs = static_cast<int>(k % SCHED_DEPTH);
    int tile;
    if (rank == 0) {
      const int ticket = static_cast<int>(atomicAdd(&ctr[0], 1u));
      tile = ticket < a.num_tickets ? ticket : -1;
      if (!mbar_wait_cluster(&bars->sched_empty[rs], ((k / SCHED_DEPTH) & 1u) ^ 1u, wc)) goto out;
      bars->sched_tile[rs] = tile;
      st_cluster_u32(mapa_shared(&bars->sched_tile[rs], peer), static_cast<uint32_t>(tile));
      mbar_arrive(&bars->sched_full[rs]);
      mbar_arrive_cluster(mapa_shared(&bars->sched_full[rs], peer));
    } else {
      if (!mbar_wait_cluster(&bars->sched_full[rs], (k / SCHED_DEPTH) & 1u, wc)) goto out;
      tile = bars->sched_tile[rs];
      mbar_arrive_cluster(mapa_shared(&bars->sched_empty[rs], 0));
    }
    if (tile < 0) break;
    const TileInfo ti = tile_info<MASK, 2, C::SUB_ROWS>(a, tile);
    if (rank == 0 && a.varlen && ti.q_row0 == 0 && varlen_bad(a, ti.b))
      atomicOr(a.err, DEVERR_BAD_CU_SEQLENS);
    const int n = max(ti.je[0], ti.je[1]);
    if (n == 0) continue;
    if (q_iter > 0 && !mbar_wait(&bars->q_empty, (q_iter - 1) & 1u, wc)) goto out;
    if (*wc.abort) goto out;
    if (rank == 0) mbar_arrive_expect_tx(&bars->q_full, 2 * C::NSUB * C::TILE_BYTES);
    {
      const uint32_t qb = mapa_shared(&bars->q_full, 0);
#pragma unroll
      for (int t = 0; t < C::NSUB; ++t)
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d_pair(smem + C::Q_OFF + t * C::TILE_BYTES + c * BOX_BYTES, tmq, qb, c * 64,
                           ti.h, ti.q_tok + ti.q_row0 + t * C::SUB_ROWS + static_cast<int>(rank) * BR,
                           ti.tma_b);
    }
    ++q_iter;
    const int krow = ti.k_tok + ti.kt_first * BC;
    const int kst = ti.kdir * BC;
    for (int j = 0; j < n; ++j)
      if (!load_half(false, ti.hk, krow + j * kst, ti.tma_b) ||
          !load_half(true, ti.hk, krow + j * kst, ti.tma_b))
        goto out;
  }
out:
  if (rank == 0) {
    // As in the single-CTA producer; only even CTAs take tickets.
    const unsigned int pairs = gridDim.x / 2;
    __threadfence();
    if (atomicAdd(&ctr[1], 1u) == pairs - 1) {
      const unsigned int taken = atomicAdd(&ctr[0], 0u);
      if (!a.inject && taken != static_cast<unsigned int>(a.num_tickets) + pairs)
        atomicOr(a.err, DEVERR_SCHED_OVERLAP);
      atomicExch(&ctr[0], 0u);
      atomicExch(&ctr[1], 0u);
    }
    // Teardown: both CTAs' loads are counted here; let every armed phase complete.
    for (int s2 = 0; s2 < C::NSLOTS; ++s2) {
      if (kv_iter > static_cast<uint32_t>(s2)) {
        const uint32_t uses = (kv_iter - 1 - s2) / C::NSLOTS + 1;
        mbar_wait_teardown(&bars->kv_full[s2], (uses - 1) & 1u, 1000000000ull);
      }
    }
    if (q_iter > 0) mbar_wait_teardown(&bars->q_full, (q_iter - 1) & 1u, 1000000000ull);
  }
}

// Bounded wait by a whole warp; every lane gets the same answer.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const WaitCtl &wc) {
  const bool ok = mbar_wait(bar, parity, wc);
  return __all_sync(0xffffffffu, ok);
}

// Scheduler-ring consumer for the MMA warp: all lanes read the tile, one lane arrives (the
// ring counts one arrival for the MMA warp).
__device__ __forceinline__ bool next_tile_mma(Bars *bars, uint32_t k, int &tile, int lane,
                                              const WaitCtl &wc) {
  const int rs = static_cast<int>(k % SCHED_DEPTH);
  if (!warp_wait(&bars->sched_full[rs], (k / SCHED_DEPTH) & 1u, wc)) return false;
  tile = bars->sched_tile[rs];
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars->sched_empty[rs]);
  return true;
}

// Consumer side of the scheduler ring: the k-th tile of this CTA (-1 = no more), or false
// if the wait gave up.  WARP consumers are whole warps (all lanes call it).
template <bool WARP>
__device__ __forceinline__ bool next_tile(Bars *bars, uint32_t k, int &tile, const WaitCtl &wc) {
  const int rs = static_cast<int>(k % SCHED_DEPTH);
  bool ok = mbar_wait(&bars->sched_full[rs], (k / SCHED_DEPTH) & 1u, wc);
  if (WARP) ok = __all_sync(0xffffffffu, ok);
  if (!ok) return false;
  tile = bars->sched_tile[rs];
  mbar_arrive(&bars->sched_empty[rs]);
  return true;
}

// ------------------------------------------------------------------------------------
// MMA issuer.  Order per K/V step j (both sub-tiles):
//   PV_0(j), S_0(j+1), PV_1(j), S_1(j+1)
// so that each softmax group finds its next S ready while the tensor core works on the
// other sub-tile.  tcgen05.mma executes in issue order, so S_t(j+1) may overwrite the
// TMEM columns that PV_t(j) reads P_t(j) from.  Sub-tile t takes part only in the steps
// [js[t], je[t]) of the block's K/V stream.

template <int D, int MASK, bool F16, bool F8 = false>
__device__ void mma_role(const PrefillArgs &a, uint8_t *smem, Bars *bars, uint32_t tmem,
                         const WaitCtl &wc, int lane) {
  using C = Cfg<D, F16, F8>;
  const uint32_t p_smem[2] = {smem_u32(smem + C::P_OFF), smem_u32(smem + C::P_OFF + BR * BC)};
  uint32_t kv_iter = 0, q_iter = 0;
  uint32_t p_phase[2] = {0u, 0u}, oe_phase[2] = {0u, 0u};
  bool o_pending[2] = {false, false};
  const uint32_t q_smem[2] = {smem_u32(smem + C::Q_OFF), smem_u32(smem + C::Q_OFF + C::TILE_BYTES)};
  const uint32_t ring = smem_u32(smem + C::RING_OFF);
  constexpr bool ABIAS = abias<D, MASK, F8, false>();
  const uint32_t bias_smem = smem_u32(smem + C::BAR_OFF + 1024);
  int bias_bh = -1;  // (batch, head) whose slope the B bias operand holds
  for (uint32_t k = 0;; ++k) {
    int tile;
    if (!next_tile_mma(bars, k, tile, lane, wc)) goto out;
    if (tile < 0) break;
    const TileInfo ti = tile_info<MASK, 2>(a, tile);
    const int n = max(ti.je[0], ti.je[1]);
    if (n == 0) continue;
    if constexpr (ABIAS) {
      // The previous tile's MMAs have completed (its last P was ready, so the S before it
      // was), so B may be rewritten: row i = i slope / scale as hi + mid + lo in bf16.
      const int bh = ti.b * a.Hq + ti.h;
      if (bh != bias_bh) {
        bias_bh = bh;
        const float ratio = a.alibi[ti.b * a.alibi_sb + ti.h] * 1.4426950408889634f / a.scale_log2;
        uint8_t *bb = smem + C::BAR_OFF + 1024 + BR * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = lane * 4 + q;
          const float v = static_cast<float>(i) * ratio;
          const float vh = bf16lo_to_f32(pack_bf16x2(v, 0.f));
          const float vm = bf16lo_to_f32(pack_bf16x2(v - vh, 0.f));
          *reinterpret_cast<uint4 *>(bb + i * 128 + ((i & 7) << 4)) =
              make_uint4(pack_bf16x2(vh, vm), pack_bf16x2((v - vh) - vm, 0.f), 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
    }
    if (!warp_wait(&bars->q_full, q_iter & 1u, wc)) goto out;
    ++q_iter;
    if (!F8 && ti.half) {
      // Half tile (sub-tile 0 alone): S double-buffered in the S regions of both sub-tiles,
      // order S(0), S(1), PV(0), S(2), PV(1), ..., PV(n-1), so that the tensor core computes
      // S(j+1) while the softmax works on S(j); S(j+2) reuses the buffer of S(j) right after
      // PV(j) has read P(j) from it (issue order).  Every PV but the last is committed to
      // pv_done: the softmax of step j+1 waits for it before it rescales O.
      auto s_half = [&](int buf) -> bool {
        const int slot = static_cast<int>(kv_iter % C::NSLOTS);
        if (!warp_wait(&bars->kv_full[slot], (kv_iter / C::NSLOTS) & 1u, wc)) return false;
        ++kv_iter;
        tc_fence_after();
        issue_s<D, F16>(tmem + s_col(buf), q_smem[0], ring + slot * C::TILE_BYTES);
        mma_commit_w(&bars->s_full[buf]);
        mma_commit_w(&bars->kv_empty[slot]);
        return true;
      };
      if (!s_half(0)) goto out;
      if (n > 1 && !s_half(1)) goto out;
      if (n <= 2) mma_commit_w(&bars->q_empty);  // Q released after the last S, as below
      // p_ready phases as bits (indexed by the runtime buffer number without local memory).
      uint32_t pb = p_phase[0] | (p_phase[1] << 1);
      for (int j = 0; j < n; ++j) {
        const int buf = j & 1;
        if (j == 0 && o_pending[0]) {
          if (!warp_wait(&bars->o_empty[0], oe_phase[0], wc)) goto out;
          oe_phase[0] ^= 1u;
          o_pending[0] = false;
        }
        if (!warp_wait(&bars->p_ready[buf], (pb >> buf) & 1u, wc)) goto out;
        pb ^= 1u << buf;
        tc_fence_after();
        const int slot = static_cast<int>(kv_iter % C::NSLOTS);
        if (!warp_wait(&bars->kv_full[slot], (kv_iter / C::NSLOTS) & 1u, wc)) goto out;
        ++kv_iter;
        tc_fence_after();
        issue_pv<D, F16>(tmem + o_col(0), tmem + s_col(buf), ring + slot * C::TILE_BYTES, j > 0);
        mma_commit_w(&bars->kv_empty[slot]);
        if (j == n - 1) {
          mma_commit_w(&bars->o_full[0]);
          o_pending[0] = true;
        } else {
          mma_commit_w(&bars->pv_done);
        }
        if (j + 2 < n && !s_half(buf)) goto out;
        if (j + 3 == n) mma_commit_w(&bars->q_empty);
      }
      p_phase[0] = pb & 1u;
      p_phase[1] = (pb >> 1) & 1u;
      continue;
    }
    {
      int slot_k = static_cast<int>(kv_iter % C::NSLOTS);
      if (!warp_wait(&bars->kv_full[slot_k], (kv_iter / C::NSLOTS) & 1u, wc)) goto out;
      ++kv_iter;
      tc_fence_after();
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (ti.js[t] == 0 && ti.je[t] > 0) {
          if (ABIAS && alibi_lin(ti, t, ti.kt_first * BC))
            issue_s_alibi<D, F16>(tmem + s_col(t), q_smem[t], ring + slot_k * C::TILE_BYTES,
                                  bias_smem);
          else
            issue_s<D, F16, F8>(tmem + s_col(t), q_smem[t], ring + slot_k * C::TILE_BYTES);
          mma_commit_w(&bars->s_full[t]);
        }
      }
      mma_commit_w(&bars->kv_empty[slot_k]);
      // Q is read by the S products alone: it is released once the tile's last S is issued
      // (the commit fires when that S completes), so that the next tile's Q loads while
      // this tile's last step runs.
      if (n == 1) mma_commit_w(&bars->q_empty);
      for (int j = 0; j < n; ++j) {
        const int slot_v = static_cast<int>(kv_iter % C::NSLOTS);
        if (!warp_wait(&bars->kv_full[slot_v], (kv_iter / C::NSLOTS) & 1u, wc)) goto out;
        ++kv_iter;
        slot_k = -1;
        if (j + 1 < n) {
          slot_k = static_cast<int>(kv_iter % C::NSLOTS);
          if (!warp_wait(&bars->kv_full[slot_k], (kv_iter / C::NSLOTS) & 1u, wc)) goto out;
          ++kv_iter;
        }
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (j >= ti.js[t] && j < ti.je[t]) {
            if (j == ti.js[t] && o_pending[t]) {
              // O_t still holds the previous tile's result until its epilogue has read it.
              if (!warp_wait(&bars->o_empty[t], oe_phase[t], wc)) goto out;
              oe_phase[t] ^= 1u;
              o_pending[t] = false;
            }
            if (!warp_wait(&bars->p_ready[t], p_phase[t], wc)) goto out;
            p_phase[t] ^= 1u;
            tc_fence_after();
            if constexpr (F8)
              issue_pv_f8<D>(tmem + o_col(t), p_smem[t], ring + slot_v * C::TILE_BYTES,
                             j > ti.js[t]);
            else
              issue_pv<D, F16>(tmem + o_col(t), tmem + s_col(t), ring + slot_v * C::TILE_BYTES,
                               j > ti.js[t]);
            if (j == ti.je[t] - 1) {
              mma_commit_w(&bars->o_full[t]);
              o_pending[t] = true;
            }
          }
          if (t == 1) mma_commit_w(&bars->kv_empty[slot_v]);
          if (j + 1 >= ti.js[t] && j + 1 < ti.je[t]) {
            if (ABIAS && alibi_lin(ti, t, (ti.kt_first + ti.kdir * (j + 1)) * BC))
              issue_s_alibi<D, F16>(tmem + s_col(t), q_smem[t], ring + slot_k * C::TILE_BYTES,
                                    bias_smem);
            else
              issue_s<D, F16, F8>(tmem + s_col(t), q_smem[t], ring + slot_k * C::TILE_BYTES);
            mma_commit_w(&bars->s_full[t]);
          }
        }
        if (slot_k >= 0) mma_commit_w(&bars->kv_empty[slot_k]);
        if (j == n - 2) mma_commit_w(&bars->q_empty);  // the last S was issued in this step
      }
    }
  }
out:
  // Teardown: every MMA issued so far must finish before TMEM is released.
  mma_commit_w(&bars->mma_done);
  mbar_wait_teardown(&bars->mma_done, 0u, 1000000000ull);
}

// MMA issuer of a CTA pair (the even CTA's MMA warp): the order of mma_role, every product
// an M = 256 cta_group::2 MMA over both CTAs' rows, every commit multicast to the barrier at
// the same offset in both CTAs.  p_ready and o_empty count the softmax warps of both CTAs.
template <int D, int MASK, bool F16>
__device__ void mma_role_pair(const PrefillArgs &a, uint8_t *smem, Bars *bars, uint32_t tmem,
                              const WaitCtl &wc, int lane) {
  using C = Cfg<D, F16, false, true>;
  uint32_t kv_iter = 0, q_iter = 0;
  uint32_t p_phase[2] = {0u, 0u}, oe_phase[2] = {0u, 0u};
  bool o_pending[2] = {false, false};
  const uint32_t q_smem[2] = {smem_u32(smem + C::Q_OFF), smem_u32(smem + C::Q_OFF + C::TILE_BYTES)};
  const uint32_t ring = smem_u32(smem + C::RING_OFF);
  auto wait_c = [&](uint64_t *bar, uint32_t parity) {
    const bool ok = mbar_wait_cluster(bar, parity, wc);
    return __all_sync(0xffffffffu, ok);
  };
  for (uint32_t k = 0;; ++k) {
    int tile;
    {
      const int rs = static_cast<int>(k % SCHED_DEPTH);
      if (!wait_c(&bars->sched_full[rs], (k / SCHED_DEPTH) & 1u)) goto out;
      tile = bars->sched_tile[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->sched_empty[rs]);
    }
    if (tile < 0) break;
    {
      const TileInfo ti = tile_info<MASK, 2, C::SUB_ROWS>(a, tile);
      const int n = max(ti.je[0], ti.je[1]);
      if (n == 0) continue;
      if (!wait_c(&bars->q_full, q_iter & 1u)) goto out;
      ++q_iter;
      int slot_k = static_cast<int>(kv_iter % C::NSLOTS);
      if (!wait_c(&bars->kv_full[slot_k], (kv_iter / C::NSLOTS) & 1u)) goto out;
      ++kv_iter;
      tc_fence_after();
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (ti.js[t] == 0 && ti.je[t] > 0) {
          issue_s_pair<D, F16>(tmem + s_col(t), q_smem[t], ring + slot_k * C::SLOT_BYTES);
          mma_commit_pair_w(&bars->s_full[t]);
        }
      }
      mma_commit_pair_w(&bars->kv_empty[slot_k]);
      for (int j = 0; j < n; ++j) {
        const int slot_v = static_cast<int>(kv_iter % C::NSLOTS);
        if (!wait_c(&bars->kv_full[slot_v], (kv_iter / C::NSLOTS) & 1u)) goto out;
        ++kv_iter;
        slot_k = -1;
        if (j + 1 < n) {
          slot_k = static_cast<int>(kv_iter % C::NSLOTS);
          if (!wait_c(&bars->kv_full[slot_k], (kv_iter / C::NSLOTS) & 1u)) goto out;
          ++kv_iter;
        }
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (j >= ti.js[t] && j < ti.je[t]) {
            if (j == ti.js[t] && o_pending[t]) {
              if (!warp_wait(&bars->o_empty[t], oe_phase[t], wc)) goto out;
              oe_phase[t] ^= 1u;
              o_pending[t] = false;
            }
            if (!warp_wait(&bars->p_ready[t], p_phase[t], wc)) goto out;
            p_phase[t] ^= 1u;
            tc_fence_after();
            issue_pv_pair<D, F16>(tmem + o_col(t), tmem + s_col(t),
                                  ring + slot_v * C::SLOT_BYTES, j > ti.js[t]);
            if (j == ti.je[t] - 1) {
              mma_commit_pair_w(&bars->o_full[t]);
              o_pending[t] = true;
            }
          }
          if (t == 1) mma_commit_pair_w(&bars->kv_empty[slot_v]);
          if (j + 1 >= ti.js[t] && j + 1 < ti.je[t]) {
            issue_s_pair<D, F16>(tmem + s_col(t), q_smem[t], ring + slot_k * C::SLOT_BYTES);
            mma_commit_pair_w(&bars->s_full[t]);
          }
        }
        if (slot_k >= 0) mma_commit_pair_w(&bars->kv_empty[slot_k]);
      }
      mma_commit_pair_w(&bars->q_empty);
    }
  }
out:
  // Teardown: every MMA issued so far (into both CTAs) must finish before TMEM is released;
  // the commit reaches the odd CTA's mma_done too.
  mma_commit_pair_w(&bars->mma_done);
  mbar_wait_teardown(&bars->mma_done, 0u, 1000000000ull);
}

// MMA issuer of the wide kernel (one sub-tile, S double-buffered in TMEM columns
// [0,128) and [128,256), O in [256,512)).  Order per tile of n K/V steps:
//   S(0), S(1), PV(0), S(2), PV(1), S(3), ..., PV(n-1)
// so the tensor core computes S(j+1) while the softmax works on S(j).  S(j+2) reuses the
// buffer of S(j) right after PV(j), which reads P(j) from it (issue order).  Every PV but
// the tile's last is committed to pv_done: the softmax of step j+1 waits for it before it
// rescales O.
template <int D, int MASK, bool F16>
__device__ void mma_role_wide(const PrefillArgs &a, uint8_t *smem, Bars *bars, uint32_t tmem,
                              const WaitCtl &wc, int lane) {
  using C = Cfg<D, F16>;
  uint32_t kv_iter = 0, q_iter = 0;
  uint32_t p_phase = 0u, oe_phase = 0u;  // p_phase: bit b for S buffer b
  bool o_pending = false;
  const uint32_t q_smem = smem_u32(smem + C::Q_OFF);
  const uint32_t ring = smem_u32(smem + C::RING_OFF);
  // Next ring slot (its load has landed): its shared address, or 0 if the wait gave up.
  auto take = [&](int &slot) -> uint32_t {
    slot = static_cast<int>(kv_iter % C::NSLOTS);
    if (!warp_wait(&bars->kv_full[slot], (kv_iter / C::NSLOTS) & 1u, wc)) return 0u;
    ++kv_iter;
    tc_fence_after();
    return ring + static_cast<uint32_t>(slot * C::SLOT_BYTES);
  };
  // S(buf) = Q K^T over d in two halves (one slot each): 8 K-steps of 16 per half.
  auto issue_s_wide = [&](int buf) -> bool {
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      int slot;
      const uint32_t k_smem = take(slot);
      if (k_smem == 0u) return false;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = static_cast<uint32_t>((kk >> 2) * BOX_BYTES + (kk & 3) * 32);
        mma_bf16_ss_w(tmem + s_col(buf),
                    sw128_desc(q_smem + static_cast<uint32_t>(2 * h * BOX_BYTES) + off, 16, 1024),
                    sw128_desc(k_smem + off, 16, 1024), C::IDESC_S, (h | kk) ? 1u : 0u);
      }
      mma_commit_w(&bars->kv_empty[slot]);
    }
    mma_commit_w(&bars->s_full[buf]);
    return true;
  };
  for (uint32_t k = 0;; ++k) {
    int tile;
    if (!next_tile_mma(bars, k, tile, lane, wc)) goto out;
    if (tile < 0) break;
    {
      const TileInfo ti = tile_info<MASK, 1>(a, tile);
      const int n = ti.je[0];
      if (n == 0) continue;
      if (!warp_wait(&bars->q_full, q_iter & 1u, wc)) goto out;
      ++q_iter;
      tc_fence_after();
      if (!issue_s_wide(0)) goto out;
      if (n > 1 && !issue_s_wide(1)) goto out;
      for (int j = 0; j < n; ++j) {
        const int buf = j & 1;
        if (j == 0 && o_pending) {
          // O still holds the previous tile's result until its epilogue has read it.
          if (!warp_wait(&bars->o_empty[0], oe_phase, wc)) goto out;
          oe_phase ^= 1u;
          o_pending = false;
        }
        if (!warp_wait(&bars->p_ready[buf], (p_phase >> buf) & 1u, wc)) goto out;
        p_phase ^= 1u << buf;
        tc_fence_after();
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          int slot;
          const uint32_t v_smem = take(slot);
          if (v_smem == 0u) goto out;
          issue_pv<D, F16>(tmem + o_col(0) + static_cast<uint32_t>(h * 128), tmem + s_col(buf),
                           v_smem, j > 0);
          mma_commit_w(&bars->kv_empty[slot]);
        }
        if (j == n - 1) {
          mma_commit_w(&bars->o_full[0]);
          o_pending = true;
        } else {
          mma_commit_w(&bars->pv_done);
        }
        if (j + 2 < n && !issue_s_wide(buf)) goto out;
      }
      mma_commit_w(&bars->q_empty);
    }
  }
out:
  mma_commit_w(&bars->mma_done);
  mbar_wait_teardown(&bars->mma_done, 0u, 1000000000ull);
}

// ------------------------------------------------------------------------------------
// Softmax / correction / epilogue: one thread per query row of its sub-tile.

// PAIR: the sub-tile is 256 rows over both CTAs of a pair; this CTA holds rows
// [128 rank, 128 rank + 128) of it, and takes part in every step of the sub-tile (the MMA
// covers both CTAs) whether or not its own rows are valid.  p_ready, o_empty and the
// scheduler ring are the even CTA's: one arrival per warp, with cluster-scope release.
template <int D, int MASK, bool F16, bool F8 = false, bool PAIR = false>
__device__ void softmax_role(const PrefillArgs &a, uint8_t *smem, Bars *bars, uint32_t tmem,
                             const WaitCtl &wc, int warp, int lane, const CUtensorMap *tmo) {
  using C = Cfg<D, F16, F8, PAIR>;
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  // Arrival on a barrier of the even CTA (after this thread's tcgen05 fences): one per warp
  // for a pair, one per thread otherwise.  TMEM: the handoffs of P (p_ready) and of the read
  // O (o_empty), whose TMEM stores / loads every lane has completed (tcgen05.wait) before the
  // warp arrives; the scheduler ring's entry is shared memory and takes cluster scope.
  auto arrive_leader = [&](uint64_t *bar, bool tmem_data) {
    if constexpr (PAIR) {
      __syncwarp();
      if (lane == 0) {
        if (tmem_data)
          mbar_arrive_remote(mapa_shared(bar, 0));
        else
          mbar_arrive_cluster(mapa_shared(bar, 0));
      }
    } else {
      mbar_arrive(bar);
    }
  };
  // FP8: P is rounded to E4M3 as 2^8 P (values up to 256 of the format's 448, so that small
  // probabilities keep their significant bits); O = sum(P' V) / sum(P') is unchanged and
  // the LSE takes the 8 back out.
  constexpr float POFF = F8 ? 8.f : 0.f;
  // Rescale threshold in log2 units: 16-bit P takes values up to 2^8 without loss; FP8 P has
  // no room above its 2^8 offset, so its reference max follows every increase.
  constexpr float RTH = F8 ? 0.f : 8.f;
  constexpr bool CAUSAL = MASK == MASK_CAUSAL;
  constexpr bool MOD = mask_has_window(MASK);   // window masking
  constexpr bool SCORE_MOD = MASK == MASK_MOD;    // softcap (+ ALiBi) code
  constexpr bool ALIBI = MASK == MASK_ALIBI;      // ALiBi without a softcap
  const int t = warp >> 2;
  const int wq = warp & 3;
  const int rit = wq * 32 + lane;  // row inside the sub-tile = TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tO = tmem + lane_off + o_col(t);
  // With a softcap or ALiBi the scores are moved to the log2 domain before the max, and
  // the exp2 argument needs no further scaling.
  const bool softcap = SCORE_MOD && a.sc_out != 0.f;
  const bool alibi = SCORE_MOD && a.alibi != nullptr;
  const float c = (softcap || alibi || ALIBI) ? 1.f : a.scale_log2;
  // S buffer phases, bit b for buffer b (one buffer per sub-tile; the wide kernel's single
  // sub-tile alternates between two).
  uint32_t s_phase = 0, o_phase = 0, pv_phase = 0;
  uint16_t *obase = reinterpret_cast<uint16_t *>(a.o);  // bf16 or fp16 elements

  for (uint32_t k = 0;; ++k) {
    int tile;
    if constexpr (PAIR) {
      const int rs = static_cast<int>(k % SCHED_DEPTH);
      const bool ok = __all_sync(0xffffffffu, mbar_wait_cluster(&bars->sched_full[rs],
                                                                (k / SCHED_DEPTH) & 1u, wc));
      if (!ok) return;
      tile = bars->sched_tile[rs];
      arrive_leader(&bars->sched_empty[rs], false);
    } else {
      if (!next_tile<true>(bars, k, tile, wc)) return;
    }
    if (tile < 0) break;
    const TileInfo ti = tile_info<MASK, C::NSUB, C::SUB_ROWS>(a, tile);
    if constexpr (!C::WIDE && !PAIR) {
      // Phase bits of S buffer 1, which both groups use: a full tile completes it once per
      // step of sub-tile 1 (group 1's steps), a half tile once per odd step of its single
      // sub-tile (group 0's); each group follows the completions it does not wait for.
      if (t == 0 && !ti.half) s_phase ^= static_cast<uint32_t>(ti.nkv[1] & 1) << 1;
      if (t == 1 && ti.half) s_phase ^= static_cast<uint32_t>((ti.nkv[0] / 2) & 1) << 1;
    }
    const int sub_rows = t == 0 ? ti.nrows[0] : ti.nrows[1];  // rows of the whole sub-tile
    if (sub_rows == 0) continue;
    // S alternates between two buffers (and P(j+1) is computed while PV(j) runs) in the wide
    // kernel and in half tiles
    const bool dbuf = C::WIDE || ti.half;
    const int nkv = t == 0 ? ti.nkv[0] : ti.nkv[1];
    const int jst = t == 0 ? ti.js[0] : ti.js[1];  // this sub-tile's first stream step
    const int first_row = ti.q_row0 + t * C::SUB_ROWS + rank * BR;  // this CTA's first row
    const int nrows = min(max(sub_rows - rank * BR, 0), BR);       // this CTA's rows
    const int row = first_row + rit;
    const bool row_ok = rit < nrows;
    const int off = ti.nk - ti.nq;  // bottom-right alignment: row i sits at key position i + off
    // Keys [lo, limit] this row may see; tiles inside [all_lo, min_limit] need no mask.
    int lo = 0, all_lo = 0, limit, min_limit;
    if constexpr (MOD) {
      lo = a.wl >= 0 ? max(row + off - a.wl, 0) : 0;
      all_lo = a.wl >= 0 ? max(first_row + BR - 1 + off - a.wl, 0) : 0;
      limit = a.wr >= 0 ? min(row + off + a.wr, ti.nk - 1) : ti.nk - 1;
      min_limit = a.wr >= 0 ? min(first_row + off + a.wr, ti.nk - 1) : ti.nk - 1;
    } else {
      limit = CAUSAL ? min(row + off, ti.nk - 1) : ti.nk - 1;
      min_limit = CAUSAL ? min(first_row + off, ti.nk - 1) : ti.nk - 1;
    }
    float slope2 = 0.f;  // ALiBi slope in log2 units
    if (alibi || ALIBI) slope2 = a.alibi[ti.b * a.alibi_sb + ti.h] * 1.4426950408889634f;
    // FP8: the Q and K descale factors of (batch, kv head) multiply every score.
    float qks = 1.f, vds = 1.f;
    if constexpr (F8) {
      const int64_t di = static_cast<int64_t>(ti.b) * a.Hkv + ti.hk;
      if (a.q_descale != nullptr) qks *= a.q_descale[di];
      if (a.k_descale != nullptr) qks *= a.k_descale[di];
      if (a.v_descale != nullptr) vds = a.v_descale[di];
    }
    const float ct = F8 && !(softcap || alibi || ALIBI) ? c * qks : c;

    // l: the row sum of P (for the LSE); lq: the rounding error of the tiles' largest P
    // (l + lq divides O).
    float m = -INFINITY, l = 0.f, lq = 0.f;
    const uint64_t c2t = f2_pack(ct, ct);
    for (int j = 0; j < nkv; ++j) {
      const int sb = dbuf ? (j & 1) : t;  // S buffer, and its s_full / p_ready barriers
      const uint32_t tS = tmem + lane_off + s_col(sb);
      if (!warp_wait(&bars->s_full[sb], (s_phase >> sb) & 1u, wc)) return;
      s_phase ^= 1u << sb;
      tc_fence_after();
      float s[BC];
      {
        uint32_t r0[64], r1[64];
        tmem_ld_2x64(tS, tS + 64, r0, r1);
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          s[i] = __uint_as_float(r0[i]);
          s[64 + i] = __uint_as_float(r1[i]);
        }
      }
      const int kbase = (ti.kt_first + ti.kdir * (jst + j)) * BC;
      // ALiBi without a softcap: the stored scores are y = s scale log2e - slope2 |pos - key|
      // - toff, in log2 units, and toff (a per-row constant of the tile) goes into the max
      // and the exp2 offset.  When every key of the tile lies at or before pos (all of a
      // causal row's tiles but the diagonal one) the bias is linear in the column:
      // -slope2 (dist0 - i) = slope2 i + toff with toff = -slope2 dist0, and y = s c +
      // slope2 i is one packed FMA per pair, the slope2 i pairs stepping by 8 slope2 along
      // four independent chains that start from exact products.
      float toff = 0.f;
      float ctj = ct;  // the factor that takes this tile's scores to log2 units
      if constexpr (ALIBI) {
        const float cs = F8 ? a.scale_log2 * qks : a.scale_log2;
        const int dist0 = row + off - kbase;  // pos - the tile's first key
        if (abias<D, MASK, F8, PAIR>() && alibi_lin(ti, t, kbase)) {
          // The tensor core added slope2 i / cs to the scores: only toff is left.
          toff = -slope2 * static_cast<float>(dist0);
          ctj = cs;
        } else if (dist0 >= BC - 1) {
          toff = -slope2 * static_cast<float>(dist0);
          const uint64_t cs2 = f2_pack(cs, cs);
          const uint64_t step = f2_pack(8.f * slope2, 8.f * slope2);
          uint64_t w[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            w[q4] = f2_pack(slope2 * static_cast<float>(2 * q4),
                            slope2 * static_cast<float>(2 * q4 + 1));
#pragma unroll
          for (int i = 0; i < BC; i += 8) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int e = i + 2 * q4;
              f2_unpack(f2_fma(f2_pack(s[e], s[e + 1]), cs2, w[q4]), s[e], s[e + 1]);
              w[q4] = f2_add(w[q4], step);
            }
          }
        } else {
          const float fd = static_cast<float>(dist0);
#pragma unroll
          for (int i = 0; i < BC; ++i)
            s[i] = fmaf(s[i], cs, -slope2 * fabsf(fd - static_cast<float>(i)));
        }
        if (kbase < all_lo || kbase + BC - 1 > min_limit) {
          const int l0 = lo - kbase, lim = limit - kbase;
#pragma unroll
          for (int i = 0; i < BC; ++i)
            if (i < l0 || i > lim) s[i] = -INFINITY;
        }
      } else if constexpr (MOD) {
        if (softcap) {
          // softcap * tanh(scale * q.k / softcap), in log2 units
          const float sci = F8 ? a.sc_in * qks : a.sc_in;
#pragma unroll
          for (int i = 0; i < BC; ++i) s[i] = tanh_ex2(s[i] * sci) * a.sc_out;
        }
        if (alibi) {
          // - slope * |pos - key|, pos = row + off; the key of column i is kbase + i
          const float cs = softcap ? 1.f : (F8 ? a.scale_log2 * qks : a.scale_log2);
          const float dist0 = static_cast<float>(row + off - kbase);
#pragma unroll
          for (int i = 0; i < BC; ++i)
            s[i] = fmaf(s[i], cs, -slope2 * fabsf(dist0 - static_cast<float>(i)));
        }
        if (kbase < all_lo || kbase + BC - 1 > min_limit) {
          const int l0 = lo - kbase, lim = limit - kbase;
#pragma unroll
          for (int i = 0; i < BC; ++i)
            if (i < l0 || i > lim) s[i] = -INFINITY;
        }
      } else if (kbase + BC - 1 > min_limit) {
        const int lim = limit - kbase;
#pragma unroll
        for (int i = 0; i < BC; ++i)
          if (i > lim) s[i] = -INFINITY;
      }
      float mx0 = fmax3(s[0], s[1], s[2]), mx1 = fmax3(s[3], s[4], s[5]);
      float mx2 = fmax3(s[6], s[7], s[8]), mx3 = fmax3(s[9], s[10], s[11]);
#pragma unroll
      for (int i = 12; i < BC - 4; i += 8) {
        mx0 = fmax3(mx0, s[i], s[i + 1]);
        mx1 = fmax3(mx1, s[i + 2], s[i + 3]);
        mx2 = fmax3(mx2, s[i + 4], s[i + 5]);
        mx3 = fmax3(mx3, s[i + 6], s[i + 7]);
      }
      const float mx = fmaxf(fmax3(mx0, mx1, s[BC - 4]),
                             fmax3(mx2, mx3, fmax3(s[BC - 3], s[BC - 2], s[BC - 1])));
      // The reference max m moves only when the tile's row max exceeds it by more than RTH:
      // O and l are rescaled on those steps alone, and P = 2^(S c - m) stays below 2^RTH.
      const float mx_s = mx * ctj + toff;
      const float m_new = mx_s > m + RTH ? mx_s : m;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const bool grow = j > 0 && m_new > m;
      const float alpha = grow ? ex2_approx(m - m_use) : 1.f;
      // P = 2^(S c + toff - m_new) with the FMA and the row sum on packed fp32 pairs.
      const float negs = POFF + toff - m_use;
      const uint64_t neg2 = f2_pack(negs, negs);
      const uint64_t c2 = abias<D, MASK, F8, PAIR>() ? f2_pack(ctj, ctj) : c2t;
      uint64_t l2a = f2_pack(0.f, 0.f), l2b = l2a;
      uint32_t p[64];
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        float x0, x1, x2, x3;
        f2_unpack(f2_fma(f2_pack(s[2 * i], s[2 * i + 1]), c2, neg2), x0, x1);
        f2_unpack(f2_fma(f2_pack(s[2 * i + 2], s[2 * i + 3]), c2, neg2), x2, x3);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
        l2a = f2_add(l2a, f2_pack(p0, p1));
        l2b = f2_add(l2b, f2_pack(p2, p3));
        if constexpr (F8) {
          p[i >> 1] = pack_e4m3x4(p0, p1, p2, p3);
        } else {
          p[i] = pack2<F16>(p0, p1);
          p[i + 1] = pack2<F16>(p2, p3);
        }
      }
      // l sums P before its rounding to 16 bits, O the rounded P.  The tile's largest P (up
      // to 2^RTH, not a power of two) may carry most of the row's weight: its rounding error
      // goes into the divisor of O as well, so that a row dominated by one key still gets
      // that key's V.
      float lcorr = 0.f;
      if constexpr (!F8) {
        const float pmx = ex2_approx(fmaf(mx, ctj, negs));  // the loop's FMA and exp2
        lcorr = lo_to_f32<F16>(pack2<F16>(pmx, 0.f)) - pmx;
      }
      {
        float la, lb, lc, ld;
        f2_unpack(l2a, la, lb);
        f2_unpack(l2b, lc, ld);
        l = l * alpha + ((la + lb) + (lc + ld));
        lq = lq * alpha + lcorr;
      }
      if constexpr (F8) {
        // E4M3 row of 128 keys = 128 bytes, stored in the 128-byte-swizzled K-major layout
        // of the PV A operand: 16-byte chunk q of row r at chunk q ^ (r mod 8).
        uint8_t *prow = smem + C::P_OFF + t * (BR * BC) + rit * BC;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4 *>(prow + ((q ^ (rit & 7)) << 4)) = make_uint4(p[4 * q],
              p[4 * q + 1], p[4 * q + 2], p[4 * q + 3]);
        fence_proxy_async_smem();
      } else {
        uint32_t (&p0)[32] = *reinterpret_cast<uint32_t (*)[32]>(&p[0]);
        uint32_t (&p1)[32] = *reinterpret_cast<uint32_t (*)[32]>(&p[32]);
        tmem_st_x32(tS, p0);
        tmem_st_x32(tS + 32, p1);
      }
      if (dbuf && j > 0) {
        // S(j) was issued before PV(j-1): wait for PV(j-1) before touching O.
        if (!warp_wait(&bars->pv_done, pv_phase, wc)) return;
        pv_phase ^= 1u;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, grow)) {
        // Conditional rescale of the O accumulator held in TMEM, done after P so that the
        // whole O row fits in the registers the scores used (one TMEM round trip).
        // Two sub-tiles: PV_t(j-1) has completed, its commit precedes the one that
        // signalled S_t(j).
        if constexpr (D >= 128) {
#pragma unroll 1
          for (int h = 0; h < D / 128; ++h) {
            const uint32_t tOh = tO + static_cast<uint32_t>(h * 128);
            uint32_t o0[64], o1[64];
            tmem_ld_2x64(tOh, tOh + 64, o0, o1);
#pragma unroll
            for (int i = 0; i < 64; ++i) {
              o0[i] = __float_as_uint(__uint_as_float(o0[i]) * alpha);
              o1[i] = __float_as_uint(__uint_as_float(o1[i]) * alpha);
            }
            tmem_st_x32(tOh, *reinterpret_cast<uint32_t (*)[32]>(&o0[0]));
            tmem_st_x32(tOh + 32, *reinterpret_cast<uint32_t (*)[32]>(&o0[32]));
            tmem_st_x32(tOh + 64, *reinterpret_cast<uint32_t (*)[32]>(&o1[0]));
            tmem_st_x32(tOh + 96, *reinterpret_cast<uint32_t (*)[32]>(&o1[32]));
          }
        } else {
          uint32_t o0[64];
          tmem_ld_x64(tO, o0);
#pragma unroll
          for (int i = 0; i < 64; ++i) o0[i] = __float_as_uint(__uint_as_float(o0[i]) * alpha);
          tmem_st_x32(tO, *reinterpret_cast<uint32_t (*)[32]>(&o0[0]));
          tmem_st_x32(tO + 32, *reinterpret_cast<uint32_t (*)[32]>(&o0[32]));
        }
      }
      tmem_wait_st();
      tc_fence_before();
      arrive_leader(&bars->p_ready[sb], true);
      m = m_new;
    }

    // Epilogue: O / l -> bf16, LSE = ln2 * (m + log2 l).
    const int64_t tok = static_cast<int64_t>(ti.q_tok) + row;
    uint16_t *orow = obase + static_cast<int64_t>(ti.b) * a.o_sb + tok * a.o_sn +
                          static_cast<int64_t>(ti.h) * a.o_sh;
    if (nkv > 0) {
      if (!warp_wait(&bars->o_full[t], o_phase, wc)) return;
      o_phase ^= 1u;
      tc_fence_after();
      const float inv_l = l > 0.f ? vds / (l + lq) : 0.f;  // vds: FP8 V descale, else 1
      if (stg_ok<D, MASK, F8, PAIR>() && a.o_tma && (wq + 1) * 32 <= nrows) {
        // The warp's 32 rows go through its staging box, 64 columns at a time, each half
        // written by one TMA store: rows of 16-byte pieces per thread would cost the
        // load/store unit 8 x the wavefronts of whole 128-byte lines.  Chunk q (8 columns)
        // of row r sits at 16-byte position q ^ (r mod 8) (the map's 128-byte swizzle).
        uint8_t *stg = smem + C::BAR_OFF + 1024 + warp * STG_WARP_BYTES;
        uint8_t *srow = stg + lane * 128;
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          uint32_t r0[32], r1[32];
          tmem_ld_x32(tO + h * 64, r0);
          tmem_ld_x32(tO + h * 64 + 32, r1);
          // The previous store from this box (the last half, or the previous tile's) has
          // read it.
          if (lane == 0) bulk_wait_read();
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t *rv = q < 4 ? &r0[8 * q] : &r1[8 * (q - 4)];
            uint4 w;
            w.x = pack2<F16>(__uint_as_float(rv[0]) * inv_l, __uint_as_float(rv[1]) * inv_l);
            w.y = pack2<F16>(__uint_as_float(rv[2]) * inv_l, __uint_as_float(rv[3]) * inv_l);
            w.z = pack2<F16>(__uint_as_float(rv[4]) * inv_l, __uint_as_float(rv[5]) * inv_l);
            w.w = pack2<F16>(__uint_as_float(rv[6]) * inv_l, __uint_as_float(rv[7]) * inv_l);
            *reinterpret_cast<uint4 *>(srow + ((q ^ (lane & 7)) << 4)) = w;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_4d(tmo, stg, h * 64, ti.h, static_cast<int>(ti.q_tok) + first_row + wq * 32,
                         ti.tma_b);
            bulk_commit_group();
          }
        }
      } else {
#pragma unroll
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t r[32];
        tmem_ld_x32(tO + cc, r);
        if (row_ok) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + cc);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            if (cc + 8 * v >= a.d) break;  // columns past d are padding
            uint4 w;
            w.x = pack2<F16>(__uint_as_float(r[8 * v + 0]) * inv_l, __uint_as_float(r[8 * v + 1]) * inv_l);
            w.y = pack2<F16>(__uint_as_float(r[8 * v + 2]) * inv_l, __uint_as_float(r[8 * v + 3]) * inv_l);
            w.z = pack2<F16>(__uint_as_float(r[8 * v + 4]) * inv_l, __uint_as_float(r[8 * v + 5]) * inv_l);
            w.w = pack2<F16>(__uint_as_float(r[8 * v + 6]) * inv_l, __uint_as_float(r[8 * v + 7]) * inv_l);
            dst[v] = w;
          }
        }
      }
      }
      tc_fence_before();
      arrive_leader(&bars->o_empty[t], true);
    } else if (row_ok) {
      uint4 *dst = reinterpret_cast<uint4 *>(orow);
#pragma unroll
      for (int v = 0; v < D / 8; ++v)
        if (8 * v < a.d) dst[v] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (row_ok) {
      const float lse = l > 0.f ? (m + log2f(l) - POFF) * LN2 : -INFINITY;
      a.lse[static_cast<int64_t>(ti.b) * a.lse_sb + static_cast<int64_t>(ti.h) * a.lse_sh + tok] = lse;
    }
  }
}

template <int D, int MASK, bool F16, bool F8 = false, bool PAIR = false>
__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                   const PrefillArgs a) {
  using C = Cfg<D, F16, F8, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars *bars = reinterpret_cast<Bars *>(smem + C::BAR_OFF);
  const int warp = static_cast<int>(threadIdx.x) >> 5;
  const int lane = static_cast<int>(threadIdx.x) & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SCHED_DEPTH; ++i) {
      mbar_init(&bars->sched_full[i], 1);
      // MMA warp + every softmax thread; a pair: the even CTA's MMA warp, one arrival per
      // softmax warp of both CTAs and the odd CTA's producer
      mbar_init(&bars->sched_empty[i], PAIR ? 1 + 2 * 4 * C::NSUB + 1 : 1 + 128 * C::NSUB);
    }
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < C::NSLOTS; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_ready[t], PAIR ? 8 : 128);  // pair: 4 warps of each CTA
      mbar_init(&bars->o_full[t], 1);
      mbar_init(&bars->o_empty[t], PAIR ? 8 : 128);
    }
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->mma_done, 1);
    mbar_init(&bars->exit_bar, 2);
    bars->abort = 0;
    fence_barrier_init();
  }
  if constexpr (abias<D, MASK, F8, PAIR>()) {
    // Ones matrix A (row r: 1 in k = 0..2) and the zero second 16 bytes of every B row.
    if (threadIdx.x < BR) {
      const int r = static_cast<int>(threadIdx.x);
      uint8_t *ab = smem + C::BAR_OFF + 1024;
      const uint32_t one2 = pack_bf16x2(1.f, 1.f), one1 = pack_bf16x2(1.f, 0.f);
      *reinterpret_cast<uint4 *>(ab + r * 128 + ((r & 7) << 4)) = make_uint4(one2, one1, 0u, 0u);
      *reinterpret_cast<uint4 *>(ab + r * 128 + (((r & 7) ^ 1) << 4)) = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4 *>(ab + BR * 128 + r * 128 + (((r & 7) ^ 1) << 4)) =
          make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async_smem();
    }
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tmq);
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  if (warp == MMA_WARP) {
    if constexpr (PAIR) {
      tmem_alloc_pair(&bars->tmem_base, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&bars->tmem_base, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR) {
    // Both CTAs' barriers are initialised before either CTA signals the other's.  (The two
    // CTAs of a cluster run together, so this wait always ends.)
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort, a.err, a.timeout_ns, DEVERR_PREFILL_TIMEOUT,
                   PAIR ? mapa_shared(&bars->abort, rank ^ 1u) : 0u};

  // Each register-split branch ends the kernel on its own; the two meet at a named barrier
  // before TMEM is released.
  // Wide kernel: the second softmax warpgroup has no sub-tile and only gives its registers
  // back; the producer / MMA warpgroup then keeps its launch registers.
  // Registers: 128 x (200 + 24 + 168) = 50176 <= 384 x 168 = 64512.
  if (warp < PRODUCER_WARP) {
    if (C::WIDE && warp >= 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(IDLE_REGS));
    } else {
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(SOFTMAX_REGS));
      softmax_role<D, MASK, F16, F8, PAIR>(a, smem, bars, tmem, wc, warp, lane, &tmo);
      // The staged O stores of this warp have read shared memory and written O.
      if (stg_ok<D, MASK, F8, PAIR>() && lane == 0) bulk_wait_all();
    }
    __syncwarp();
    tc_fence_before();
    named_barrier(1, NTHREADS);
  } else {
    if constexpr (!C::WIDE) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(OTHER_REGS));
    if (warp == PRODUCER_WARP) {
      if constexpr (PAIR) {
        if (lane == 0) producer_role_pair<D, MASK>(a, &tmq, &tmk, &tmv, smem, bars, wc, rank);
      } else {
        if (lane == 0) producer_role<D, MASK, F8>(a, &tmq, &tmk, &tmv, smem, bars, wc);
      }
    } else if (warp == MMA_WARP) {
      if constexpr (PAIR) {
        if (rank == 0) {
          mma_role_pair<D, MASK, F16>(a, smem, bars, tmem, wc, lane);
        } else {
          // The even CTA's last commit (its teardown) reaches this CTA's mma_done too.
          mbar_wait_teardown(&bars->mma_done, 0u, 2 * a.timeout_ns + 1000000000ull);
        }
      } else if constexpr (C::WIDE) {
        mma_role_wide<D, MASK, F16>(a, smem, bars, tmem, wc, lane);
      } else {
        mma_role<D, MASK, F16, F8>(a, smem, bars, tmem, wc, lane);
      }
    }
    __syncwarp();
    tc_fence_before();
    named_barrier(1, NTHREADS);
    if (warp == MMA_WARP) {
      if constexpr (PAIR) {
        // Neither CTA leaves (and frees its shared memory) while the other may still signal
        // it: each arrives on both exit barriers once all its roles are done, then waits for
        // the other's arrival (bounded).
        if (lane == 0) {
          mbar_arrive_cluster(mapa_shared(&bars->exit_bar, rank ^ 1u));
          mbar_arrive(&bars->exit_bar);
        }
        __syncwarp();
        mbar_wait_teardown(&bars->exit_bar, 0u, 2 * a.timeout_ns + 1000000000ull);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, TMEM_COLS);
      } else {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
      }
    }
  }
}

template <int D, int MASK, bool F16, bool F8 = false>
cudaError_t launch_impl(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const CUtensorMap &tmo, const PrefillArgs &a, int grid,
                        cudaStream_t stream) {
  constexpr int smem = prefill_smem<D, MASK, F16, F8, false>();
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, MASK, F16, F8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  prefill_kernel<D, MASK, F16, F8><<<grid, NTHREADS, smem, stream>>>(tq, tk, tv, tmo, a);
  return cudaGetLastError();
}

// CTA pairs: clusters of two; `clusters` pairs (at most the number that fit on the GPU at
// once, from the occupancy query, so that every pair of the persistent grid runs together).
template <int MASK, bool F16>
cudaError_t launch_pair_impl(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                             const PrefillArgs &a, int tiles, cudaStream_t stream) {
  constexpr int smem = Cfg<128, F16, false, true>::SMEM_BYTES;
  auto kern = prefill_kernel<128, MASK, F16, false, true>;
  static int max_clusters[64] = {};  // per device, found on the first launch there
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters[dev] == 0) {
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    cfg.gridDim = dim3(static_cast<unsigned>(sms / 2 * 2), 1, 1);
    int n = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg)) != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    max_clusters[dev] = n;
  }
  const int clusters = tiles < max_clusters[dev] ? tiles : max_clusters[dev];
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  const CUtensorMap no_map{};  // pairs store O rows directly
  e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, no_map, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// O = 0 and LSE = -inf for B x N x H rows.
__global__ void fill_empty_kernel(uint16_t *o, float *lse, int B, int N, int H, int d,
                                  int64_t o_sb, int64_t o_sn, int64_t o_sh, int64_t lse_sb,
                                  int64_t lse_sh) {
  const int64_t rows = static_cast<int64_t>(B) * N * H;
  for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < rows;
       r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int h = static_cast<int>(r % H);
    const int64_t bn = r / H;
    const int n = static_cast<int>(bn % N);
    const int b = static_cast<int>(bn / N);
    uint16_t *orow = o + b * o_sb + n * o_sn + h * o_sh;
    for (int c = 0; c < d; ++c) orow[c] = 0;  // +0 in both bf16 and fp16
    lse[b * lse_sb + h * lse_sh + n] = -INFINITY;
  }
}

}  // namespace

int next_prefill_sched_slot() {
  static std::atomic<unsigned int> seq{0};
  return static_cast<int>(seq.fetch_add(1u) % NUM_SCHED_SLOTS);
}

int prefill_smem_bytes(int d) {
  return d == 64 ? Cfg<64>::SMEM_BYTES : (d == 128 ? Cfg<128>::SMEM_BYTES : Cfg<256>::SMEM_BYTES);
}

template <int D, bool F16, bool F8 = false>
cudaError_t launch_mask(int mask, const CUtensorMap &tq, const CUtensorMap &tk,
                        const CUtensorMap &tv, const CUtensorMap *tmo_in, PrefillArgs a,
                        int grid, cudaStream_t stream) {
  const CUtensorMap no_map{};
  if (tmo_in == nullptr) a.o_tma = 0;
  const CUtensorMap &tmo = tmo_in != nullptr ? *tmo_in : no_map;
  switch (mask) {
    case MASK_NONE: return launch_impl<D, MASK_NONE, F16, F8>(tq, tk, tv, tmo, a, grid, stream);
    case MASK_CAUSAL:
      return launch_impl<D, MASK_CAUSAL, F16, F8>(tq, tk, tv, tmo, a, grid, stream);
    case MASK_WINDOW:
      return launch_impl<D, MASK_WINDOW, F16, F8>(tq, tk, tv, tmo, a, grid, stream);
    case MASK_ALIBI: return launch_impl<D, MASK_ALIBI, F16, F8>(tq, tk, tv, tmo, a, grid, stream);
    default: return launch_impl<D, MASK_MOD, F16, F8>(tq, tk, tv, tmo, a, grid, stream);
  }
}

cudaError_t launch_prefill_fp8(int mask, const CUtensorMap &tq, const CUtensorMap &tk,
                               const CUtensorMap &tvt, const CUtensorMap *tmo,
                               const PrefillArgs &a, int grid, cudaStream_t stream) {
  return launch_mask<128, false, true>(mask, tq, tk, tvt, tmo, a, grid, stream);
}

// V [B, Nk, Hkv, d] E4M3 -> V^T [B, Hkv, d, nk_pad] (keys contiguous, zero past Nk), the
// K-major layout the FP8 PV product takes.  One block per (64-key tile, kv head, batch).
__global__ void transpose_v_kernel(const uint8_t *v, int64_t v_sb, int64_t v_sn, int64_t v_sh,
                                   uint8_t *vt, int Nk, int Hkv, int d, int nk_pad) {
  __shared__ uint8_t tile[64][128 + 4];
  const int k0 = blockIdx.x * 64, hk = blockIdx.y, b = blockIdx.z;
  const int chunks = d / 16;  // 16-byte chunks per key row
  for (int i = threadIdx.x; i < 64 * chunks; i += blockDim.x) {
    const int key = i / chunks, c = i - key * chunks;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (k0 + key < Nk)
      w = *reinterpret_cast<const uint4 *>(v + b * v_sb + static_cast<int64_t>(k0 + key) * v_sn +
                                           hk * v_sh + c * 16);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) tile[key][c * 16 + q * 4 + e] = static_cast<uint8_t>(ws[q] >> (8 * e));
  }
  __syncthreads();
  uint8_t *out = vt + (static_cast<int64_t>(b) * Hkv + hk) * d * nk_pad;
  const int kcols = min(64, nk_pad - k0);  // multiple of 16
  for (int i = threadIdx.x; i < d * (kcols / 16); i += blockDim.x) {
    const int row = i / (kcols / 16), c = i - row * (kcols / 16);
    uint32_t ws[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      ws[q] = static_cast<uint32_t>(tile[c * 16 + q * 4][row]) |
              (static_cast<uint32_t>(tile[c * 16 + q * 4 + 1][row]) << 8) |
              (static_cast<uint32_t>(tile[c * 16 + q * 4 + 2][row]) << 16) |
              (static_cast<uint32_t>(tile[c * 16 + q * 4 + 3][row]) << 24);
    *reinterpret_cast<uint4 *>(out + static_cast<int64_t>(row) * nk_pad + k0 + c * 16) =
        make_uint4(ws[0], ws[1], ws[2], ws[3]);
  }
}

cudaError_t launch_transpose_v(const void *v, int64_t v_sb, int64_t v_sn, int64_t v_sh, void *vt,
                               int B, int Nk, int Hkv, int d, int nk_pad, cudaStream_t stream) {
  if (B == 0 || nk_pad == 0) return cudaSuccess;
  const dim3 grid((nk_pad + 63) / 64, Hkv, B);
  transpose_v_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint8_t *>(v), v_sb, v_sn, v_sh,
                                              static_cast<uint8_t *>(vt), Nk, Hkv, d, nk_pad);
  return cudaGetLastError();
}

// Packed sequences: V [total_k, Hkv, d] E4M3 (contiguous) -> V^T [Hkv, d, nt], sequence b's
// keys at columns vt0(b) = roundup16(cu_k[b]) + 16 b onwards (16-aligned for the TMA), up to
// roundup16 of its length; the caller zeroes the buffer first, so the columns between
// sequences read as 0.  One block per (64-key tile of a sequence, kv head, sequence);
// sequences with inconsistent prefix sums are skipped (the prefill kernel reports them).
__global__ void transpose_v_varlen_kernel(const uint8_t *v, uint8_t *vt, const int *cu_k,
                                          int total_k, int Hkv, int d, int nt) {
  __shared__ uint8_t tile[64][128 + 4];
  const int k0 = blockIdx.x * 64, hk = blockIdx.y, b = blockIdx.z;
  const int s0 = cu_k[b], s1 = cu_k[b + 1];
  if (s0 < 0 || s1 < s0 || s1 > total_k) return;
  const int len = s1 - s0;
  if (k0 >= len) return;
  const int chunks = d / 16;  // 16-byte chunks per key row
  const int64_t v_sn = static_cast<int64_t>(Hkv) * d;
  for (int i = threadIdx.x; i < 64 * chunks; i += blockDim.x) {
    const int key = i / chunks, c = i - key * chunks;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (k0 + key < len)
      w = *reinterpret_cast<const uint4 *>(v + static_cast<int64_t>(s0 + k0 + key) * v_sn +
                                           hk * d + c * 16);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) tile[key][c * 16 + q * 4 + e] = static_cast<uint8_t>(ws[q] >> (8 * e));
  }
  __syncthreads();
  const int vt0 = ((s0 + 15) & ~15) + 16 * b;
  uint8_t *out = vt + static_cast<int64_t>(hk) * d * nt + vt0;
  const int kcols = min(64, ((len + 15) & ~15) - k0);  // multiple of 16
  for (int i = threadIdx.x; i < d * (kcols / 16); i += blockDim.x) {
    const int row = i / (kcols / 16), c = i - row * (kcols / 16);
    uint32_t ws[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      ws[q] = static_cast<uint32_t>(tile[c * 16 + q * 4][row]) |
              (static_cast<uint32_t>(tile[c * 16 + q * 4 + 1][row]) << 8) |
              (static_cast<uint32_t>(tile[c * 16 + q * 4 + 2][row]) << 16) |
              (static_cast<uint32_t>(tile[c * 16 + q * 4 + 3][row]) << 24);
    *reinterpret_cast<uint4 *>(out + static_cast<int64_t>(row) * nt + k0 + c * 16) =
        make_uint4(ws[0], ws[1], ws[2], ws[3]);
  }
}

cudaError_t launch_transpose_v_varlen(const void *v, void *vt, const int *cu_k, int B,
                                      int max_seqlen_k, int total_k, int Hkv, int d, int nt,
                                      cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(vt, 0, static_cast<size_t>(Hkv) * d * nt, stream);
  if (e != cudaSuccess || B == 0 || max_seqlen_k == 0) return e;
  const dim3 grid((max_seqlen_k + 63) / 64, Hkv, B);
  transpose_v_varlen_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint8_t *>(v),
                                                      static_cast<uint8_t *>(vt), cu_k, total_k,
                                                      Hkv, d, nt);
  return cudaGetLastError();
}

template <bool F16>
cudaError_t launch_pair_mask(int mask, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const PrefillArgs &a, int tiles,
                             cudaStream_t stream) {
  switch (mask) {
    case MASK_NONE: return launch_pair_impl<MASK_NONE, F16>(tq, tk, tv, a, tiles, stream);
    case MASK_CAUSAL: return launch_pair_impl<MASK_CAUSAL, F16>(tq, tk, tv, a, tiles, stream);
    case MASK_WINDOW: return launch_pair_impl<MASK_WINDOW, F16>(tq, tk, tv, a, tiles, stream);
    case MASK_ALIBI: return launch_pair_impl<MASK_ALIBI, F16>(tq, tk, tv, a, tiles, stream);
    default: return launch_pair_impl<MASK_MOD, F16>(tq, tk, tv, a, tiles, stream);
  }
}

cudaError_t launch_prefill_pair(int mask, bool f16, const CUtensorMap &tq, const CUtensorMap &tk,
                                const CUtensorMap &tv, const PrefillArgs &a, int tiles,
                                cudaStream_t stream) {
  return f16 ? launch_pair_mask<true>(mask, tq, tk, tv, a, tiles, stream)
             : launch_pair_mask<false>(mask, tq, tk, tv, a, tiles, stream);
}

cudaError_t launch_prefill(int d, int mask, bool f16, const CUtensorMap &tq,
                           const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap *tmo,
                           const PrefillArgs &a, int grid, cudaStream_t stream) {
  if (d == 64)
    return f16 ? launch_mask<64, true>(mask, tq, tk, tv, tmo, a, grid, stream)
               : launch_mask<64, false>(mask, tq, tk, tv, tmo, a, grid, stream);
  if (d == 256)
    return f16 ? launch_mask<256, true>(mask, tq, tk, tv, tmo, a, grid, stream)
               : launch_mask<256, false>(mask, tq, tk, tv, tmo, a, grid, stream);
  return f16 ? launch_mask<128, true>(mask, tq, tk, tv, tmo, a, grid, stream)
             : launch_mask<128, false>(mask, tq, tk, tv, tmo, a, grid, stream);
}

cudaError_t launch_fill_empty(void *o, float *lse, int B, int N, int H, int d, int64_t o_sb,
                              int64_t o_sn, int64_t o_sh, int64_t lse_sb, int64_t lse_sh,
                              cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(B) * N * H;
  if (rows == 0) return cudaSuccess;
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<int64_t>((rows + threads - 1) / threads, 4096));
  fill_empty_kernel<<<blocks, threads, 0, stream>>>(reinterpret_cast<uint16_t *>(o), lse, B,
                                                    N, H, d, o_sb, o_sn, o_sh, lse_sb, lse_sh);
  return cudaGetLastError();
}

}  // namespace fa
