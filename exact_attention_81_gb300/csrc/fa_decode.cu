// fa_decode.cu -- single-query decode against a padded KV cache, split over the key axis.
//
// "flash-attention" (ai-reference-codex.pages.dev): a short query against a long cache
// takes the split-KV branch (section 2.3); each split writes a partial output and its
// log-sum-exp and combine_attn_seqk_parallel merges them (code map); with GQA the query
// heads of one group are folded into one work item so that they share one K/V stream
// (section 4, seqlenq_ngroups_swapped).
//
// Decode reads every visible cache row exactly once and does ~4 flops per byte, so it is
// bound by HBM bandwidth.  The kernel is built for that bound:
//   * work unit = (batch b, kv head g, chunk c of `chunk` keys); persistent CTAs (one per
//     SM) walk the units in chunk-major order;
//   * a producer warp streams 128-key K and V blocks of the unit with TMA (128B-swizzled
//     boxes, 2 KB row stride of the cache handled by the tensor map) into a deep ring of
//     shared-memory slots, so many blocks per SM are in flight at all times;
//   * 8 compute warps evaluate the G = Hq/Hkv query heads of the group together; warp w
//     owns keys [16w, 16w+16) of every block and keeps its own online-softmax state
//     (running max m, sum l, fp32 P V accumulators), so a block needs no CTA-wide
//     synchronisation:
//       scores   lanes = (key, 1/TPK of d), q of the lane's slice in registers as packed
//                fp32 pairs (fma.rn.f32x2 over pairs of d), TPK-lane reduce;
//       softmax  warp-wide max per head, alpha = 2^(m_old - m_new), p = 2^(s - m_new);
//       P V      lane = 4 consecutive d, packed-pair FMAs, accumulators rescaled by alpha;
//     at the end of a unit the 8 warps' (m, l, O) are merged (the same LSE-weighted merge
//     as the split combine);
//   * each unit writes O_s / l_s (fp32) and LSE_s = ln2 (m + log2 l) to the workspace.
// Only rows below cache_seqlens[b] are used: a block's tail rows are masked to -inf in the
// scores and skipped in P V, so values past the visible prefix never enter the result.
//
// The combine kernel merges the partials of each (b, query head):
//   LSE = log sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s.
#include <atomic>
#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int KB = 128;           // keys per block (one TMA tile per d-box)
constexpr int NCOMPUTE = 256;     // compute threads (warps 0-7)
constexpr int NTHREADS = 384;     // + warpgroup 2: the TMA producer (warp 8) and 3 idle warps
constexpr int PRODUCER_WARP = 8;
// Registers: the producer's warpgroup gives most of its share to the compute warpgroups
// (2 x 128 x COMPUTE_REGS + 128 x PRODUCER_REGS = 384 threads x 168 at launch).
constexpr int COMPUTE_REGS = 232;
constexpr int PRODUCER_REGS = 40;
constexpr int BOX_BYTES = KB * 128;
constexpr float LN2 = 0.6931471805599453f;

__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }
__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

// F8: K and V are E4M3 (one byte per element, 128 elements per 128-byte box row).
template <int D, int G, bool F8 = false>
struct DCfg {
  static constexpr int EB = F8 ? 1 : 2;                        // bytes per K/V element
  static constexpr int BOX_ELEMS = 128 / EB;                   // elements of a row per box
  static constexpr int KCH = D * EB / 128;                     // boxes per row
  static constexpr int BLOCK_BYTES = KCH * BOX_BYTES;         // one K or V block
  static constexpr int NWARP = NCOMPUTE / 32;                  // compute warps
  static constexpr int KPW = KB / NWARP;                       // keys of a block per warp
  static constexpr int TPK = cmax(4, G * D / 128);             // lanes per key (scores)
  static constexpr int DP = D / TPK;                           // d elements per lane
  static constexpr int KPASS = 32 / TPK;                       // keys per pass of a warp
  static constexpr int NPASS = KPW / KPASS;                    // passes per block
  static constexpr int HPL = (G + TPK - 1) / TPK;              // heads whose p a lane makes
  static constexpr int CPL = DP * EB / 16;                     // 16-byte chunks per lane
  static constexpr int PPC = 8 / EB;                           // element pairs per chunk
  static constexpr int DQ = D / 4;                             // d quads (P V lanes)
  static constexpr int QPL = DQ > 32 ? DQ / 32 : 1;            // quads per lane (d = 256: 2)
  static constexpr int KSPLIT = DQ >= 32 ? 1 : 32 / DQ;        // key interleave in P V
  static constexpr int PW_BYTES = NWARP * KPW * G * 4;         // per-warp probabilities
  static constexpr int DS = D / QPL;                           // d columns merged per round
  static constexpr int RED_BYTES = NWARP * G * DS * 4;         // per-warp outputs at unit end
  static constexpr int MISC_BYTES = 1024;                      // (m, l) per warp, barriers
  static constexpr int BUDGET = 227 * 1024 - 1024;             // minus alignment slack
  static constexpr int NSLOTS =
      cmin(12, (BUDGET - PW_BYTES - RED_BYTES - MISC_BYTES) / BLOCK_BYTES);
  static constexpr int RING_OFF = 0;
  static constexpr int PW_OFF = NSLOTS * BLOCK_BYTES;
  static constexpr int RED_OFF = PW_OFF + PW_BYTES;
  static constexpr int MISC_OFF = RED_OFF + RED_BYTES;
  static constexpr int SMEM_BYTES = MISC_OFF + MISC_BYTES + 1024;
  static_assert(NSLOTS >= 2, "ring too small");
  static_assert(KPW % KPASS == 0, "passes must cover a warp's keys");
  static_assert(TPK <= 32 && (32 % TPK) == 0, "lanes per key must tile a warp");
  static_assert((DP * EB) % 16 == 0 && KCH >= 1, "each lane reads whole 16-byte chunks");
  static_assert((DQ <= 32 && (32 % DQ) == 0) || DQ % 32 == 0, "d quads must tile a warp");
};

constexpr int SCHED_DEPTH = 4;     // units in flight between the scheduler and the compute warps
constexpr int NUM_SCHED_SLOTS = 256;

// Per-launch unit-ticket counters: [slot][0] = next ticket, [slot][1] = CTAs finished.  The
// host gives each launch its own slot (round robin); the last CTA of a launch to finish
// checks that the launch took exactly its own tickets and resets the slot for its next user.
__device__ unsigned int g_dsched[NUM_SCHED_SLOTS][2];

struct DBars {
  uint64_t full[12], empty[12];
  uint64_t sched_full[SCHED_DEPTH], sched_empty[SCHED_DEPTH];
  int sched_unit[SCHED_DEPTH];
  uint64_t sync;  // group barrier of the 256 compute threads (bounded wait)
  float m[8][8], l[8][8];  // [warp][head] running max / sum at the end of a unit
  int abort;
};

static_assert(sizeof(DBars) <= 1024, "decode barriers exceed their shared-memory region");

struct Unit {
  int b, g, c, len, key0, nkeys;
};

// Element pair e (elements 2e, 2e + 1) of a 16-byte chunk of a K row as packed fp32: bf16
// or fp16 halves, or E4M3 bytes.
template <bool F16, bool F8>
__device__ __forceinline__ uint64_t kv_pair(const uint32_t (&xs)[4], int e) {
  if constexpr (F8) {
    const uint32_t w = xs[e >> 1];
    return (e & 1) ? e4m3x2_to_f32x2(w >> 16) : e4m3x2_to_f32x2(w & 0xFFFFu);
  } else {
    return f2_pack(lo_to_f32<F16>(xs[e]), hi_to_f32<F16>(xs[e]));
  }
}

// First key visible to the decode query of a sequence of len keys (position len - 1).
__device__ __forceinline__ int first_visible(int len, int wl) {
  return wl >= 0 ? max(len - 1 - wl, 0) : 0;
}

// Unit u = (chunk c, batch b, work item g); work item g serves query heads
// [g G, g G + G) of kv head g / nsplit.  Chunks tile the keys [first, len) from the
// first visible key on (rounded down to a page-safe multiple of 128 for paged caches), so
// a window only moves the start.  len counts an appended row.
__device__ __forceinline__ Unit unit_of(const DecodeArgs &a, int u) {
  Unit w;
  const int bg = a.B * a.Hkv;
  w.c = u / bg;
  const int r = u - w.c * bg;
  w.b = r / a.Hkv;
  w.g = r - w.b * a.Hkv;
  const int len_raw = a.cache_len[w.b] + a.len_add;
  w.len = min(max(len_raw, 0), a.Lmax);
  w.key0 = decode_first_key(w.len, a.wl, a.kalign) + w.c * a.chunk;
  w.nkeys = min(a.chunk, w.len - w.key0);  // <= 0: nothing to do
  return w;
}

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const WaitCtl &wc) {
  const bool ok = mbar_wait(bar, parity, wc);
  return __all_sync(0xffffffffu, ok);
}

// Scheduler and TMA producer: the whole warp runs the loop and its waits, lane 0 takes the
// tickets and issues the loads (a loop confined to one lane issues late next to the compute
// warps: 1.7 % of bandwidth).  Units are claimed from the launch's ticket counter, so a CTA
// that drew short units takes more of them; units without keys are skipped here and never
// reach the compute warps.  Each claimed unit goes to the compute warps through the
// scheduler ring (-1 = no more), then its K and V blocks through the load ring.
template <int D, int G, bool F8, bool MOD>
__device__ void producer(const DecodeArgs &a, const CUtensorMap *tmk, const CUtensorMap *tmv,
                         uint8_t *smem, DBars *bars, const WaitCtl &wc, int lane) {
  using C = DCfg<D, G, F8>;
  uint32_t it = 0;
  unsigned int *ctr = g_dsched[a.sched_slot];
  const uint64_t policy = policy_evict_first();  // every cache byte is read once
  if (a.inject) goto out;  // failure injection: load nothing, the consumers' waits run out
  for (uint32_t k = 0;; ++k) {
    int unit = -1;
    while (true) {
      unsigned int t = 0;
      if (lane == 0) t = atomicAdd(&ctr[0], 1u);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t >= static_cast<unsigned int>(a.num_units)) break;
      const Unit w = unit_of(a, static_cast<int>(t));
      if (w.c == 0 && w.g == 0) {
        const int len_raw = a.cache_len[w.b] + a.len_add;
        if (lane == 0 && (len_raw < 0 || len_raw > a.Lmax)) atomicOr(a.err, DEVERR_BAD_CACHE_LEN);
      }
      if (w.nkeys > 0) {
        unit = static_cast<int>(t);
        break;
      }
    }
    const int rs = static_cast<int>(k % SCHED_DEPTH);
    if (!warp_wait(&bars->sched_empty[rs], ((k / SCHED_DEPTH) & 1u) ^ 1u, wc)) goto out;
    if (lane == 0) {
      bars->sched_unit[rs] = unit;
      mbar_arrive(&bars->sched_full[rs]);
    }
    __syncwarp();
    if (unit < 0) break;
    const Unit w = unit_of(a, unit);
    const int nblk = (w.nkeys + KB - 1) / KB;
    for (int blk = 0; blk < nblk; ++blk) {
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const int slot = static_cast<int>(it % C::NSLOTS);
        const uint32_t use = it / C::NSLOTS;
        if (!warp_wait(&bars->empty[slot], (use & 1u) ^ 1u, wc)) goto out;
        // (row, batch) of the block, or (row in page, page) for a paged cache: a block
        // never crosses a page (unit starts and page sizes are multiples of 128).
        int row = w.key0 + blk * KB, outer = w.b;
        if (a.block_table != nullptr) {
          outer = a.block_table[static_cast<int64_t>(w.b) * a.bt_stride + row / a.page_size];
          if (lane == 0 && which == 0 && (outer < 0 || outer >= a.num_pages))  // zeros
            atomicOr(a.err, DEVERR_BAD_BLOCK_TABLE);
          row %= a.page_size;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->full[slot], C::BLOCK_BYTES);
#pragma unroll
          for (int cc = 0; cc < C::KCH; ++cc)
            tma_load_4d_hint(smem + C::RING_OFF + slot * C::BLOCK_BYTES + cc * BOX_BYTES,
                             which ? tmv : tmk, &bars->full[slot], cc * C::BOX_ELEMS,
                             w.g / a.nsplit, row, outer, policy);
        }
        __syncwarp();
        ++it;
      }
    }
  }
out:
  // This CTA takes no more tickets (it reached the end, or gave up): count it as finished.
  // Every CTA takes exactly one ticket past the last unit, so the launch took num_units +
  // gridDim.x tickets in all; another count means that another launch ran on the same slot
  // at the same time (or a CTA gave up, which sets its own error bit).  The last CTA to
  // finish resets the slot for its next launch.
  if (lane == 0) {
    __threadfence();
    if (atomicAdd(&ctr[1], 1u) == gridDim.x - 1) {
      const unsigned int taken = atomicAdd(&ctr[0], 0u);
      if (!a.inject && taken != static_cast<unsigned int>(a.num_units) + gridDim.x)
        atomicOr(a.err, DEVERR_SCHED_OVERLAP);
      atomicExch(&ctr[0], 0u);
      atomicExch(&ctr[1], 0u);
    }
  }
  for (int s = 0; s < C::NSLOTS; ++s) {
    if (it > static_cast<uint32_t>(s)) {
      const uint32_t uses = (it - 1 - s) / C::NSLOTS + 1;
      mbar_wait_teardown(&bars->full[s], (uses - 1) & 1u, 1000000000ull);
    }
  }
}


// Barrier among the 256 compute threads.  Built on an mbarrier rather than bar.sync so
// that the wait is bounded: a warp that has given up never leaves the others blocked.
__device__ __forceinline__ bool group_sync(uint64_t *bar, uint32_t &phase, const WaitCtl &wc) {
  mbar_arrive(bar);
  const bool ok = warp_wait(bar, phase, wc);
  phase ^= 1u;
  return ok;
}

// Releases a ring slot: one arrival per compute warp (count 8).  The slot was read with
// generic loads and its next contents arrive through TMA (the async proxy), so each lane
// orders its reads before the arrival with a proxy fence: without it a TMA write into the
// released slot could overtake reads still in flight (seen at d = 256 with one query head
// per group, where the last reads come right before the release).
__device__ __forceinline__ void release(uint64_t *bar, int lane) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// MOD: the launch has a softcap, ALiBi slopes, or a window over a paged cache (whose unit
// starts are page-aligned, so keys before the window are masked); uniform runtime branches
// inside, and the plain instances carry none of that state.
template <int D, int G, bool F16, bool F8, bool MOD>
__device__ void compute(const DecodeArgs &a, uint8_t *smem, DBars *bars, const WaitCtl &wc,
                        int tid) {
  using C = DCfg<D, G, F8>;
  const int warp = tid >> 5, lane = tid & 31;
  // scores mapping: lane = (key kl of the pass, slice `part` of d)
  const int kl = lane / C::TPK, part = lane % C::TPK;
  const int d0 = part * C::DP;
  const int sbox = d0 * C::EB / 128;
  const int schunk0 = (d0 * C::EB % 128) / 16;
  // P V mapping: lane = (d quads dq + 32 i for i < QPL, key interleave kpar)
  const int dq = lane % C::DQ, kpar = lane / C::DQ;

  float *pw = reinterpret_cast<float *>(smem + C::PW_OFF) + warp * (C::KPW * G);
  float *red = reinterpret_cast<float *>(smem + C::RED_OFF);
  const uint16_t *qg = reinterpret_cast<const uint16_t *>(a.q);  // bf16 or fp16 elements
  const bool softcap = MOD && a.sc_out != 0.f;
  const bool alibi = MOD && a.alibi != nullptr;
  uint32_t it = 0, sync_phase = 0;

  for (uint32_t k = 0;; ++k) {
    // Next unit from the scheduler ring (one arrival per warp frees the entry).
    const int rs = static_cast<int>(k % SCHED_DEPTH);
    if (!warp_wait(&bars->sched_full[rs], (k / SCHED_DEPTH) & 1u, wc)) return;
    const int u = bars->sched_unit[rs];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->sched_empty[rs]);
    if (u < 0) break;
    const Unit w = unit_of(a, u);
    const int nblk = (w.nkeys + KB - 1) / KB;

    // E4M3 caches: descale factors of (b, kv head); K's goes into q, V's into the partial
    // output.
    float qscale = a.scale_log2, vds = 1.f;
    if constexpr (F8) {
      const int64_t kh = static_cast<int64_t>(w.b) * (a.Hkv / a.nsplit) + w.g / a.nsplit;
      qscale *= a.k_descale ? a.k_descale[kh] : 1.f;
      vds = a.v_descale ? a.v_descale[kh] : 1.f;
    }
    // q slice of the G heads of group g in the log2 domain, as pairs (q[d], q[d+1]).
    uint64_t q2[G][C::DP / 2];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          qg + (static_cast<int64_t>(w.b) * a.Hq + w.g * G + gg) * a.d + d0);
#pragma unroll
      for (int v = 0; v < C::DP / 8; ++v) {
        const uint4 x = d0 + 8 * v < a.d ? src[v] : make_uint4(0u, 0u, 0u, 0u);  // padding
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          q2[gg][4 * v + e] = f2_pack(lo_to_f32<F16>(xs[e]) * qscale,
                                      hi_to_f32<F16>(xs[e]) * qscale);
      }
    }
    uint64_t acc[G][2 * C::QPL];
    float m[G], l[G];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
#pragma unroll
      for (int i = 0; i < 2 * C::QPL; ++i) acc[gg][i] = f2_pack(0.f, 0.f);
      m[gg] = -INFINITY;
      l[gg] = 0.f;
    }
    // ALiBi slopes of the group's query heads (read where used: G more live registers
    // would spill at G = 8).
    const float *slopes = alibi ? a.alibi + w.b * a.alibi_sb + w.g * G : nullptr;
    // Keys below `first` are streamed only to keep blocks page-aligned: masked.
    const int first = MOD ? first_visible(w.len, a.wl) : 0;

    for (int blk = 0; blk < nblk; ++blk) {
      const int nvalid = min(KB, w.nkeys - blk * KB);
      const int kw0 = warp * C::KPW;  // first key of this warp in the block
      // ---- scores of this warp's keys from the K block
      float sc[C::NPASS][G];
      {
        const int slot = static_cast<int>(it % C::NSLOTS);
        if (!warp_wait(&bars->full[slot], (it / C::NSLOTS) & 1u, wc)) return;
        ++it;
        const uint8_t *kblk = smem + C::RING_OFF + slot * C::BLOCK_BYTES + sbox * BOX_BYTES;
#pragma unroll
        for (int pass = 0; pass < C::NPASS; ++pass) {
          const int key = kw0 + pass * C::KPASS + kl;
          const uint8_t *krow = kblk + key * 128;
          uint64_t s2[G];
#pragma unroll
          for (int gg = 0; gg < G; ++gg) s2[gg] = f2_pack(0.f, 0.f);
#pragma unroll
          for (int v = 0; v < C::CPL; ++v) {
            const int phys = (schunk0 + v) ^ (key & 7);
            const uint4 x = *reinterpret_cast<const uint4 *>(krow + phys * 16);
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < C::PPC; ++e) {
              const uint64_t k2 = kv_pair<F16, F8>(xs, e);
#pragma unroll
              for (int gg = 0; gg < G; ++gg)
                s2[gg] = f2_fma(q2[gg][C::PPC * v + e], k2, s2[gg]);
            }
          }
#pragma unroll
          for (int gg = 0; gg < G; ++gg) {
            float lo, hi;
            f2_unpack(s2[gg], lo, hi);
            float sv = lo + hi;
#pragma unroll
            for (int off = C::TPK / 2; off > 0; off >>= 1)
              sv += __shfl_xor_sync(0xffffffffu, sv, off);
            if (softcap) sv = tanh_ex2(sv * a.sc_in) * a.sc_out;
            if (alibi)  // - slope * distance from the query at position len - 1, log2 units
              sv = fmaf(slopes[gg] * -1.4426950408889634f,
                        static_cast<float>(w.len - 1 - (w.key0 + blk * KB + key)), sv);
            const bool seen = key < nvalid && (!MOD || w.key0 + blk * KB + key >= first);
            sc[pass][gg] = seen ? sv : -INFINITY;
          }
        }
        release(&bars->empty[slot], lane);
      }
      // ---- warp-level online softmax over the warp's keys
      float alpha[G];
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        float bm = sc[0][gg];
#pragma unroll
        for (int pass = 1; pass < C::NPASS; ++pass) bm = fmaxf(bm, sc[pass][gg]);
#pragma unroll
        for (int off = C::TPK; off < 32; off <<= 1)
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
        const float m_new = fmaxf(m[gg], bm);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        alpha[gg] = m_new > m[gg] ? ex2_approx(m[gg] - m_use) : 1.f;
        m[gg] = m_new;
      }
      __syncwarp();  // the previous block's P V reads of pw are done
      float psum[C::HPL];
#pragma unroll
      for (int i = 0; i < C::HPL; ++i) {
        psum[i] = 0.f;
        const int gg = part + i * C::TPK;
        if (gg < G) {
          const float m_use = m[gg] == -INFINITY ? 0.f : m[gg];
#pragma unroll
          for (int pass = 0; pass < C::NPASS; ++pass) {
            const float p = ex2_approx(sc[pass][gg] - m_use);
            pw[(pass * C::KPASS + kl) * G + gg] = p;
            psum[i] += p;
          }
        }
#pragma unroll
        for (int off = C::TPK; off < 32; off <<= 1)
          psum[i] += __shfl_xor_sync(0xffffffffu, psum[i], off);
      }
#pragma unroll
      for (int gg = 0; gg < G; ++gg)
        l[gg] = l[gg] * alpha[gg] +
                __shfl_sync(0xffffffffu, psum[gg / C::TPK], gg % C::TPK);
      __syncwarp();  // pw visible to the whole warp
      // ---- P V of this warp's keys from the V block
      {
        const int slot = static_cast<int>(it % C::NSLOTS);
        if (!warp_wait(&bars->full[slot], (it / C::NSLOTS) & 1u, wc)) return;
        ++it;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          const uint64_t al2 = f2_pack(alpha[gg], alpha[gg]);
#pragma unroll
          for (int i = 0; i < 2 * C::QPL; ++i) acc[gg][i] = f2_mul(acc[gg][i], al2);
        }
        const uint8_t *vblk0 = smem + C::RING_OFF + slot * C::BLOCK_BYTES;
        const int kend = min(C::KPW, nvalid - kw0);
#pragma unroll 4
        for (int kk = kpar; kk < kend; kk += C::KSPLIT) {
          const int key = kw0 + kk;
          uint64_t v01[C::QPL], v23[C::QPL];
#pragma unroll
          for (int i = 0; i < C::QPL; ++i) {
            // quad dq + 32 i: its box, then its bytes inside a swizzled 16-byte chunk
            const int q4 = 4 * (dq + 32 * i);
            const int vbyte = (q4 % C::BOX_ELEMS) * C::EB;
            const int phys = (vbyte / 16) ^ (key & 7);
            const uint8_t *src =
                vblk0 + (q4 / C::BOX_ELEMS) * BOX_BYTES + key * 128 + phys * 16 + vbyte % 16;
            if constexpr (F8) {
              const uint32_t x = *reinterpret_cast<const uint32_t *>(src);
              v01[i] = e4m3x2_to_f32x2(x & 0xFFFFu);
              v23[i] = e4m3x2_to_f32x2(x >> 16);
            } else {
              const uint2 x = *reinterpret_cast<const uint2 *>(src);
              v01[i] = f2_pack(lo_to_f32<F16>(x.x), hi_to_f32<F16>(x.x));
              v23[i] = f2_pack(lo_to_f32<F16>(x.y), hi_to_f32<F16>(x.y));
            }
          }
          float p[G];
          if constexpr (G % 4 == 0) {
#pragma unroll
            for (int g4 = 0; g4 < G; g4 += 4) {
              const float4 pp = *reinterpret_cast<const float4 *>(pw + kk * G + g4);
              p[g4] = pp.x;
              p[g4 + 1] = pp.y;
              p[g4 + 2] = pp.z;
              p[g4 + 3] = pp.w;
            }
          } else {
#pragma unroll
            for (int gg = 0; gg < G; ++gg) p[gg] = pw[kk * G + gg];
          }
#pragma unroll
          for (int gg = 0; gg < G; ++gg) {
            const uint64_t p2 = f2_pack(p[gg], p[gg]);
#pragma unroll
            for (int i = 0; i < C::QPL; ++i) {
              acc[gg][2 * i] = f2_fma(v01[i], p2, acc[gg][2 * i]);
              acc[gg][2 * i + 1] = f2_fma(v23[i], p2, acc[gg][2 * i + 1]);
            }
          }
        }
        release(&bars->empty[slot], lane);
      }
    }

    // ---- unit end: merge the warps' (m, l, O) and write the normalised partial.
    float o4[G][4 * C::QPL];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
#pragma unroll
      for (int i = 0; i < C::QPL; ++i) {
        f2_unpack(acc[gg][2 * i], o4[gg][4 * i], o4[gg][4 * i + 1]);
        f2_unpack(acc[gg][2 * i + 1], o4[gg][4 * i + 2], o4[gg][4 * i + 3]);
      }
      if constexpr (C::KSPLIT > 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int off = C::DQ; off < 32; off <<= 1)
            o4[gg][i] += __shfl_xor_sync(0xffffffffu, o4[gg][i], off);
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        bars->m[warp][gg] = m[gg];
        bars->l[warp][gg] = l[gg];
      }
    }
    const int64_t row0 = (static_cast<int64_t>(w.b) * a.Hq + w.g * G) * a.maxch + w.c;
    // One round per slice of DS columns (d = 256: two rounds, so the staging buffer holds
    // half of d and the ring keeps a third slot).
#pragma unroll
    for (int i = 0; i < C::QPL; ++i) {
      if (kpar == 0) {
#pragma unroll
        for (int gg = 0; gg < G; ++gg)
          *reinterpret_cast<float4 *>(red + (warp * G + gg) * C::DS + 4 * dq) =
              make_float4(o4[gg][4 * i], o4[gg][4 * i + 1], o4[gg][4 * i + 2],
                          o4[gg][4 * i + 3]);
      }
      if (!group_sync(&bars->sync, sync_phase, wc)) return;
      for (int idx = tid; idx < G * C::DS; idx += NCOMPUTE) {
        const int gg = idx / C::DS, dd = idx - gg * C::DS;
        float M = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < C::NWARP; ++ww) M = fmaxf(M, bars->m[ww][gg]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int ww = 0; ww < C::NWARP; ++ww) {
          const float mw = bars->m[ww][gg];
          const float wgt = mw == -INFINITY ? 0.f : ex2_approx(mw - M);
          L = fmaf(bars->l[ww][gg], wgt, L);
          O = fmaf(red[(ww * G + gg) * C::DS + dd], wgt, O);
        }
        const int64_t row = row0 + static_cast<int64_t>(gg) * a.maxch;
        const int col = i * C::DS + dd;  // rows of the partials are ostride (<= D) wide
        if (col < a.ostride) a.o_part[row * a.ostride + col] = O / L * vds;
        if (i == 0 && dd == 0) a.lse_part[row] = (M + log2f(L)) * LN2;
      }
      if (!group_sync(&bars->sync, sync_phase, wc)) return;
    }
  }
}

// The decode contractions on the tensor cores: mma.sync m16n8k16 with fp32 accumulation, bf16
// or fp16 operands for 16-bit caches, f16 operands for E4M3 caches (their values convert to
// f16 exactly, in registers).  Widths 64 and 128 (E4M3: 128).  Warp w owns keys
// [16 w, 16 w + 16) of every 128-key block and its own online-softmax state, as in compute();
// lane = 4 g + t.
//   S = Q K^T: M = the work item's heads (row g < G; rows g + 8 and g >= G are zero), N = the
//   warp's 16 keys as two n-tiles (column g of n-tile n = key 8 n + g), K = d in D / 16 steps.
//   The contraction index is permuted on both operands so that lane t reads the D / 4
//   contiguous elements [t D / 4, (t + 1) D / 4) of a key row: at step ks, columns 2t + {0,1}
//   stand for d = t D / 4 + 4 ks + {0,1} and 2t + 8 + {0,1} for d = t D / 4 + 4 ks + {2,3}, so
//   the operand registers are the row's own element pairs (E4M3: each 4-byte word converts to
//   the two f16 pairs of one step).  The query enters exactly: as stored for 16-bit caches;
//   for E4M3 caches as f16 after a power-of-two scaling that puts its largest magnitude below
//   2^15 (values below 2^-38 of the largest are the only ones f16 does not hold).
//   S arrives as lane (g, t): head g at keys 2t, 2t + 1 and 8 + 2t, 9 + 2t, which is the A
//   layout of P in the second product: P goes from the softmax to the MMA in registers.
//   O += P V: M = heads, N = d in D / 8 n-tiles (column g of n-tile nd = d g D / 8 + nd),
//   K = the 16 keys: lane (g, t) reads D / 8 elements of key rows 2t, 2t + 1, 2t + 8, 2t + 9
//   and pairs the elements of two rows with byte permutes; its accumulators hold
//   O[head g][t D / 4 + nd] and O[head g][t D / 4 + D / 8 + nd], D / 4 contiguous columns.
//   P enters the product rounded to f16 (values <= 1: relative rounding 2^-11), or for bf16
//   operands as bf16(p) plus a second product with the remainder bf16(p - bf16(p)) (about 16
//   significant bits: a bf16 P alone raised the largest error of short decode rows from
//   7.7e-3 to 9.8e-3); the row sums stay fp32.  Rows of keys that take no part (past the length, before the window start) are
//   zeroed in the V operand, so 0 x NaN cannot reach O.
template <int D, int G, bool F16, bool F8, bool MOD>
__device__ void compute_mma(const DecodeArgs &a, uint8_t *smem, DBars *bars, const WaitCtl &wc,
                            int tid) {
  using C = DCfg<D, G, F8>;
  constexpr int EB = C::EB;                  // bytes per cache element
  constexpr int KSTEPS = D / 16;             // k-steps of S
  constexpr int NT = D / 8;                  // n-tiles of P V
  constexpr int KWORDS = D / 4 * EB / 4;     // 32-bit words of a key-row slice (lane t)
  constexpr int VWORDS = D / 8 * EB / 4;     // 32-bit words of a V-row slice (lane g)
  constexpr bool HALF = F8 || F16;           // f16 MMA (else bf16)
  static_assert(C::KPW == 16, "16 keys per warp and block");
  static_assert(!F8 || D == 128, "E4M3 rows are one 128-byte box");
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  float *red = reinterpret_cast<float *>(smem + C::RED_OFF);
  const uint16_t *qg = reinterpret_cast<const uint16_t *>(a.q);
  const bool softcap = MOD && a.sc_out != 0.f;
  const bool alibi = MOD && a.alibi != nullptr;
  // Element e of a ring row: box e / BOX_ELEMS, 16-byte chunk ((e % BOX_ELEMS) EB) / 16.
  const int ke0 = t * (D / 4);      // first element of this lane's key-row slice
  const int ve0 = g * (D / 8);      // first element of this lane's V-row slice
  const int kbox = ke0 / C::BOX_ELEMS, kchunk = (ke0 % C::BOX_ELEMS) * EB / 16;
  const int vbox = ve0 / C::BOX_ELEMS, vchunk = (ve0 % C::BOX_ELEMS) * EB / 16;
  uint32_t it = 0, sync_phase = 0;
  auto mma = [](float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    if constexpr (HALF)
      mma_f16_m16n8k16(d, a0, 0u, a2, 0u, b0, b1);
    else
      mma_bf16_m16n8k16(d, a0, 0u, a2, 0u, b0, b1);
  };

  for (uint32_t k = 0;; ++k) {
    const int rs = static_cast<int>(k % SCHED_DEPTH);
    if (!warp_wait(&bars->sched_full[rs], (k / SCHED_DEPTH) & 1u, wc)) return;
    const int u = bars->sched_unit[rs];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->sched_empty[rs]);
    if (u < 0) break;
    const Unit w = unit_of(a, u);
    const int nblk = (w.nkeys + KB - 1) / KB;
    float sc = a.scale_log2, vds = 1.f;
    if constexpr (F8) {
      const int64_t kh = static_cast<int64_t>(w.b) * (a.Hkv / a.nsplit) + w.g / a.nsplit;
      sc *= a.k_descale ? a.k_descale[kh] : 1.f;
      vds = a.v_descale ? a.v_descale[kh] : 1.f;
    }

    // Query of head g, elements [ke0, ke0 + D / 4): the A operand pairs of every k-step.
    uint32_t qa[KSTEPS][2];
    {
      uint32_t qw[D / 8];  // the slice as element pairs
#pragma unroll
      for (int i = 0; i < D / 8; ++i) qw[i] = 0u;
      if (g < G) {
        const uint4 *src = reinterpret_cast<const uint4 *>(
            qg + (static_cast<int64_t>(w.b) * a.Hq + w.g * G + g) * a.d + ke0);
#pragma unroll
        for (int v = 0; v < D / 32; ++v) {
          if (ke0 + 8 * v < a.d) {  // columns past d are padding
            const uint4 x = src[v];
            qw[4 * v] = x.x;
            qw[4 * v + 1] = x.y;
            qw[4 * v + 2] = x.z;
            qw[4 * v + 3] = x.w;
          }
        }
      }
      if constexpr (F8) {
        // bf16 query -> f16, scaled by sq = 2^e so that the largest magnitude is below 2^15
        float qmax = 0.f;
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
          qmax = fmaxf(qmax, fmaxf(fabsf(bf16lo_to_f32(qw[i])), fabsf(bf16hi_to_f32(qw[i]))));
#pragma unroll
        for (int off = 1; off < 32; off <<= 1)
          qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
        const int ex = static_cast<int>((__float_as_uint(qmax) >> 23) & 0xFFu) - 127;
        const float sq =
            qmax > 0.f ? __uint_as_float(static_cast<uint32_t>(min(max(141 - ex, 1), 254)) << 23)
                       : 1.f;
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
          qw[i] = pack_f16x2(bf16lo_to_f32(qw[i]) * sq, bf16hi_to_f32(qw[i]) * sq);
        sc /= sq;
      }
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        qa[ks][0] = qw[2 * ks];
        qa[ks][1] = qw[2 * ks + 1];
      }
    }
    const float slope2 = (alibi && g < G)
                             ? a.alibi[w.b * a.alibi_sb + w.g * G + g] * -1.4426950408889634f
                             : 0.f;
    const int first = MOD ? first_visible(w.len, a.wl) : 0;
    float o[NT][4];
#pragma unroll
    for (int nd = 0; nd < NT; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float m = -INFINITY, l = 0.f;

    for (int blk = 0; blk < nblk; ++blk) {
      const int nvalid = min(KB, w.nkeys - blk * KB);
      const int kw0 = warp * C::KPW;
      const int kglob = w.key0 + blk * KB + kw0;  // cache row of the warp's first key
      // keys of this lane's scores and V rows: kw0 + 2t + {0, 1, 8, 9}
      const int kl[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
      bool valid[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        valid[i] = kw0 + kl[i] < nvalid && (!MOD || kglob + kl[i] >= first);
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int slot = static_cast<int>(it % C::NSLOTS);
        if (!warp_wait(&bars->full[slot], (it / C::NSLOTS) & 1u, wc)) return;
        ++it;
        const uint8_t *kblk = smem + C::RING_OFF + slot * C::BLOCK_BYTES + kbox * BOX_BYTES;
        // one 16-byte chunk of each key row at a time, then the k-steps it holds (2 for 16-bit
        // elements, 4 for E4M3), so that the slice never sits in registers as a whole
        constexpr int KS_PER_CHUNK = 16 / (4 * EB);
#pragma unroll
        for (int c = 0; c < KWORDS / 4; ++c) {
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            const int key = kw0 + 8 * n + g;
            const uint4 x = *reinterpret_cast<const uint4 *>(
                kblk + key * 128 + (((kchunk + c) ^ (key & 7)) << 4));
            const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int j = 0; j < KS_PER_CHUNK; ++j) {
              const int ks = c * KS_PER_CHUNK + j;
              uint32_t b0, b1;
              if constexpr (F8) {
                e4m3x4_to_f16x2x2(xw[j], b0, b1);
              } else {
                b0 = xw[2 * j];
                b1 = xw[2 * j + 1];
              }
              mma(sacc[n], qa[ks][0], qa[ks][1], b0, b1);
            }
          }
        }
        release(&bars->empty[slot], lane);
      }
      // ---- online softmax of head g over the warp's 16 keys (4 per lane, 4 lanes per head)
      float sv[4] = {sacc[0][0] * sc, sacc[0][1] * sc, sacc[1][0] * sc, sacc[1][1] * sc};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (softcap) sv[i] = tanh_ex2(sv[i] * a.sc_in) * a.sc_out;
        if (alibi)  // - slope * distance from the query at position len - 1, log2 units
          sv[i] = fmaf(slope2, static_cast<float>(w.len - 1 - (kglob + kl[i])), sv[i]);
        if (!valid[i]) sv[i] = -INFINITY;
      }
      float bm = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      const float m_new = fmaxf(m, bm);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = m_new > m ? ex2_approx(m - m_use) : 1.f;
      m = m_new;
      float p[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) p[i] = ex2_approx(sv[i] - m_use);
      float ps = (p[0] + p[1]) + (p[2] + p[3]);
      ps += __shfl_xor_sync(0xffffffffu, ps, 1);
      ps += __shfl_xor_sync(0xffffffffu, ps, 2);
      l = l * alpha + ps;
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int nd = 0; nd < NT; ++nd) {
          o[nd][0] *= alpha;
          o[nd][1] *= alpha;
        }
      }
      const uint32_t pa0 = HALF ? pack_f16x2(p[0], p[1]) : pack_bf16x2(p[0], p[1]);
      const uint32_t pa2 = HALF ? pack_f16x2(p[2], p[3]) : pack_bf16x2(p[2], p[3]);
      // bf16 operands: P also enters as its rounding remainder p - bf16(p) (a second product
      // on the same V fragments), so P carries about 16 significant bits instead of 8
      uint32_t pl0 = 0u, pl2 = 0u;
      if constexpr (!HALF) {
        pl0 = pack_bf16x2(p[0] - bf16lo_to_f32(pa0), p[1] - bf16hi_to_f32(pa0));
        pl2 = pack_bf16x2(p[2] - bf16lo_to_f32(pa2), p[3] - bf16hi_to_f32(pa2));
      }
      // ---- O += P V
      {
        const int slot = static_cast<int>(it % C::NSLOTS);
        if (!warp_wait(&bars->full[slot], (it / C::NSLOTS) & 1u, wc)) return;
        ++it;
        const uint8_t *vblk = smem + C::RING_OFF + slot * C::BLOCK_BYTES + vbox * BOX_BYTES;
        uint32_t vr[4][VWORDS];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = kw0 + kl[i];
#pragma unroll
          for (int c = 0; c < (VWORDS + 3) / 4; ++c) {
            const uint4 x = *reinterpret_cast<const uint4 *>(
                vblk + row * 128 + (((vchunk + c) ^ (row & 7)) << 4));
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (4 * c + e < VWORDS) vr[i][4 * c + e] = valid[i] ? xs[e] : 0u;
          }
        }
        release(&bars->empty[slot], lane);
        if constexpr (F8) {
#pragma unroll
          for (int w4 = 0; w4 < VWORDS; ++w4) {
            uint32_t b0a, b0b, b0c, b0d, b1a, b1b, b1c, b1d;
            // (row 2t, row 2t+1) and (row 2t+8, row 2t+9) byte pairs at d = 16 g + 4 w4 + j
            e4m3x4_to_f16x2x2(byte_perm(vr[0][w4], vr[1][w4], 0x5140u), b0a, b0b);
            e4m3x4_to_f16x2x2(byte_perm(vr[0][w4], vr[1][w4], 0x7362u), b0c, b0d);
            e4m3x4_to_f16x2x2(byte_perm(vr[2][w4], vr[3][w4], 0x5140u), b1a, b1b);
            e4m3x4_to_f16x2x2(byte_perm(vr[2][w4], vr[3][w4], 0x7362u), b1c, b1d);
            mma(o[4 * w4 + 0], pa0, pa2, b0a, b1a);
            mma(o[4 * w4 + 1], pa0, pa2, b0b, b1b);
            mma(o[4 * w4 + 2], pa0, pa2, b0c, b1c);
            mma(o[4 * w4 + 3], pa0, pa2, b0d, b1d);
          }
        } else {
#pragma unroll
          for (int nd = 0; nd < NT; ++nd) {
            // element nd of the slice (word nd / 2, half nd % 2) of rows (2t, 2t+1), (2t+8, 2t+9)
            const uint32_t sel = (nd & 1) ? 0x7632u : 0x5410u;
            const uint32_t b0 = byte_perm(vr[0][nd / 2], vr[1][nd / 2], sel);
            const uint32_t b1 = byte_perm(vr[2][nd / 2], vr[3][nd / 2], sel);
            mma(o[nd], pa0, pa2, b0, b1);
            if constexpr (!HALF) mma(o[nd], pl0, pl2, b0, b1);
          }
        }
      }
    }

    // ---- unit end: merge the warps' (m, l, O) and write the normalised partial.  The staging
    // buffer holds DS columns per (warp, head) (DS = D up to width 128, half of it at 256), so
    // the merge runs in D / DS rounds; in round r the lanes whose slice [ke0, ke0 + D / 4) lies
    // in columns [r DS, (r + 1) DS) stage it.
    constexpr int DS = C::DS;
    static_assert(DS % (D / 4) == 0, "a lane's slice lies in one round");
    if (t == 0 && g < G) {
      bars->m[warp][g] = m;
      bars->l[warp][g] = l;
    }
    const int64_t row0 = (static_cast<int64_t>(w.b) * a.Hq + w.g * G) * a.maxch + w.c;
#pragma unroll 1
    for (int r = 0; r < D / DS; ++r) {
      if (g < G && ke0 / DS == r) {
        float *dst = red + (warp * G + g) * DS + (ke0 - r * DS);
#pragma unroll
        for (int nd = 0; nd < NT; ++nd) {
          dst[nd] = o[nd][0];
          dst[NT + nd] = o[nd][1];
        }
      }
      if (!group_sync(&bars->sync, sync_phase, wc)) return;
      for (int idx = tid; idx < G * DS; idx += NCOMPUTE) {
        const int gg = idx / DS, dd = idx - gg * DS;
        float M = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < C::NWARP; ++ww) M = fmaxf(M, bars->m[ww][gg]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int ww = 0; ww < C::NWARP; ++ww) {
          const float mw = bars->m[ww][gg];
          const float wgt = mw == -INFINITY ? 0.f : ex2_approx(mw - M);
          L = fmaf(bars->l[ww][gg], wgt, L);
          O = fmaf(red[(ww * G + gg) * DS + dd], wgt, O);
        }
        const int64_t row = row0 + static_cast<int64_t>(gg) * a.maxch;
        const int col = r * DS + dd;  // rows of the partials are ostride (<= D) wide
        if (col < a.ostride) a.o_part[row * a.ostride + col] = O / L * vds;
        if (r == 0 && dd == 0) a.lse_part[row] = (M + log2f(L)) * LN2;
      }
      if (!group_sync(&bars->sync, sync_phase, wc)) return;
    }
  }
}

template <int D, int G, bool F16, bool F8, bool MOD>
__global__ void __launch_bounds__(NTHREADS, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeArgs a) {
  using C = DCfg<D, G, F8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  DBars *bars = reinterpret_cast<DBars *>(smem + C::MISC_OFF);
  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < C::NSLOTS; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], NCOMPUTE / 32);
    }
    for (int i = 0; i < SCHED_DEPTH; ++i) {
      mbar_init(&bars->sched_full[i], 1);
      mbar_init(&bars->sched_empty[i], NCOMPUTE / 32);  // one arrival per compute warp
    }
    mbar_init(&bars->sync, NCOMPUTE);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  __syncthreads();
  const WaitCtl wc{&bars->abort, a.err, a.timeout_ns, DEVERR_DECODE_TIMEOUT};
  // Each register-split branch ends on its own named barrier.
  if (warp < PRODUCER_WARP) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(COMPUTE_REGS));
    if constexpr (D <= 256 && !(F8 && D == 256))
      compute_mma<D, G, F16, F8, MOD>(a, smem, bars, wc, tid);
    else
      compute<D, G, F16, F8, MOD>(a, smem, bars, wc, tid);
    __syncwarp();
    named_barrier(1, NTHREADS);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(PRODUCER_REGS));
    if (warp == PRODUCER_WARP) producer<D, G, F8, MOD>(a, &tmk, &tmv, smem, bars, wc, lane);
    __syncwarp();
    named_barrier(1, NTHREADS);
  }
}

template <int D, int G, bool F16, bool F8 = false>
cudaError_t launch_decode_impl(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeArgs &a,
                               int grid, cudaStream_t stream) {
  constexpr int smem = DCfg<D, G, F8>::SMEM_BYTES;
  const bool mod = a.sc_out != 0.f || a.alibi != nullptr || (a.wl >= 0 && a.kalign > 1);
  auto kern = mod ? decode_kernel<D, G, F16, F8, true> : decode_kernel<D, G, F16, F8, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, NTHREADS, smem, stream>>>(tk, tv, a);
  return cudaGetLastError();
}

// One block per (batch, query head); thread = output column.
template <int D, bool F16>
__global__ void __launch_bounds__(D)
    combine_kernel(const float *o_part, const float *lse_part, const int *cache_len,
                   int len_add, int Hq, int Lmax, int chunk, int maxch, int wl, int kalign,
                   int d_out, uint16_t *o, float *lse) {
  const int bh = blockIdx.x;
  const int b = bh / Hq;
  const int d = threadIdx.x;
  const int len = min(max(cache_len[b] + len_add, 0), Lmax);
  const int nch = (len - decode_first_key(len, wl, kalign) + chunk - 1) / chunk;
  const float *lp = lse_part + static_cast<int64_t>(bh) * maxch;
  const float *op = o_part + static_cast<int64_t>(bh) * maxch * D;
  if (nch == 0) {
    if (d < d_out) o[static_cast<int64_t>(bh) * d_out + d] = 0;  // +0 in bf16 and fp16
    if (d == 0) lse[bh] = -INFINITY;
    return;
  }
  float m = -INFINITY;
  for (int c = 0; c < nch; ++c) m = fmaxf(m, lp[c]);
  float wsum = 0.f, acc = 0.f;
  for (int c = 0; c < nch; ++c) {
    const float wgt = expf(lp[c] - m);
    wsum += wgt;
    acc = fmaf(wgt, op[static_cast<int64_t>(c) * D + d], acc);
  }
  if (d < d_out)
    o[static_cast<int64_t>(bh) * d_out + d] =
        static_cast<uint16_t>(pack2<F16>(acc / wsum, 0.f) & 0xFFFFu);  // round to nearest even
  if (d == 0) lse[bh] = m + logf(wsum);
}

// ------------------------------------------------------------------------------------
// In-place append ("flash-attention", section 1: the decode call writes the new key and
// value into the cache and applies rotary in the same step).  One block per sequence;
// thread = (head, dimension).  The new rows go to logical row cache_len[b]; with rotary
// tables the new key and the query are turned by the angle of that position.

// Element c of x after the rotary turn (c >= rot_dim: copied), rounded to the element type.
// The grouping is fixed (one fused multiply-add per output, the product inside it rounded
// first) so that the rounding decision is reproducible.
template <bool F16>
__device__ __forceinline__ uint16_t rotary_elem(const uint16_t *x, int c, int rot_dim,
                                                bool interleaved, const float *cs,
                                                const float *sn) {
  if (c >= rot_dim) return x[c];
  const int half = rot_dim / 2;
  const bool first = interleaved ? (c & 1) == 0 : c < half;
  const int i = interleaved ? c >> 1 : (first ? c : c - half);
  const int ia = interleaved ? 2 * i : i;
  const int ib = interleaved ? 2 * i + 1 : i + half;
  const float xa = lo_to_f32<F16>(x[ia]), xb = lo_to_f32<F16>(x[ib]);
  const float co = cs[i], si = sn[i];
  const float y = first ? __fmaf_rn(xa, co, -__fmul_rn(xb, si))
                        : __fmaf_rn(xa, si, __fmul_rn(xb, co));
  return static_cast<uint16_t>(pack2<F16>(y, 0.f) & 0xFFFFu);
}

template <bool F16>
__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a) {
  const int b = blockIdx.x;
  const int len = a.cache_len[b];
  const bool rot = a.cos != nullptr;
  bool ok = len >= 0 && len < a.Lmax && (!rot || len < a.rot_positions);
  int64_t row = 0;  // element offset of the cache row
  if (ok) {
    if (a.block_table != nullptr) {
      const int page = a.block_table[static_cast<int64_t>(b) * a.bt_stride + len / a.page_size];
      ok = page >= 0 && page < a.num_pages;
      row = static_cast<int64_t>(page) * a.c_s0 + static_cast<int64_t>(len % a.page_size) * a.c_s1;
    } else {
      row = static_cast<int64_t>(b) * a.c_s0 + static_cast<int64_t>(len) * a.c_s1;
    }
  }
  if (!ok && threadIdx.x == 0) atomicOr(a.err, DEVERR_BAD_APPEND);
  const int half = a.rot_dim / 2;
  const float *cs = rot && ok ? a.cos + static_cast<int64_t>(len) * half : nullptr;
  const float *sn = rot && ok ? a.sin + static_cast<int64_t>(len) * half : nullptr;
  if (ok) {
    const uint16_t *kn = reinterpret_cast<const uint16_t *>(a.k_new) + b * a.n_sb;
    const uint16_t *vn = reinterpret_cast<const uint16_t *>(a.v_new) + b * a.n_sb;
    uint16_t *kc = reinterpret_cast<uint16_t *>(a.k_cache) + row;
    uint16_t *vc = reinterpret_cast<uint16_t *>(a.v_cache) + row;
    for (int idx = threadIdx.x; idx < a.Hkv * a.d; idx += blockDim.x) {
      const int h = idx / a.d, c = idx - h * a.d;
      const uint16_t *kr = kn + h * a.n_sh;
      kc[h * a.c_s2 + c] = rot ? rotary_elem<F16>(kr, c, a.rot_dim, a.rot_interleaved, cs, sn)
                               : kr[c];
      vc[h * a.c_s2 + c] = vn[h * a.n_sh + c];
    }
  }
  if (rot) {  // the query at the same position (copied unturned if the append was refused)
    const uint16_t *q = reinterpret_cast<const uint16_t *>(a.q) + static_cast<int64_t>(b) * a.Hq * a.d;
    uint16_t *qr = reinterpret_cast<uint16_t *>(a.q_rot) + static_cast<int64_t>(b) * a.Hq * a.d;
    for (int idx = threadIdx.x; idx < a.Hq * a.d; idx += blockDim.x) {
      const int h = idx / a.d, c = idx - h * a.d;
      qr[idx] = ok ? rotary_elem<F16>(q + h * a.d, c, a.rot_dim, a.rot_interleaved, cs, sn)
                   : q[idx];
    }
  }
}

}  // namespace

int next_decode_sched_slot() {
  static std::atomic<unsigned int> seq{0};
  return static_cast<int>(seq.fetch_add(1u) % NUM_SCHED_SLOTS);
}

cudaError_t launch_append(bool f16, const AppendArgs &a, cudaStream_t stream) {
  if (a.B == 0) return cudaSuccess;
  if (f16)
    append_kernel<true><<<a.B, 256, 0, stream>>>(a);
  else
    append_kernel<false><<<a.B, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

template <bool F16>
cudaError_t launch_decode_typed(int d, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                                const DecodeArgs &a, int grid, cudaStream_t stream) {
  // group: the heads of one work item (DecodeArgs::nsplit items per kv head); at d = 256
  // at most 4 (more heads' staging would leave the ring two slots).
  if (d == 256) {
    switch (group) {
      case 1: return launch_decode_impl<256, 1, F16>(tk, tv, a, grid, stream);
      case 2: return launch_decode_impl<256, 2, F16>(tk, tv, a, grid, stream);
      default: return launch_decode_impl<256, 4, F16>(tk, tv, a, grid, stream);
    }
  }
  if (d == 64) {
    switch (group) {
      case 1: return launch_decode_impl<64, 1, F16>(tk, tv, a, grid, stream);
      case 2: return launch_decode_impl<64, 2, F16>(tk, tv, a, grid, stream);
      case 4: return launch_decode_impl<64, 4, F16>(tk, tv, a, grid, stream);
      default: return launch_decode_impl<64, 8, F16>(tk, tv, a, grid, stream);
    }
  }
  switch (group) {
    case 1: return launch_decode_impl<128, 1, F16>(tk, tv, a, grid, stream);
    case 2: return launch_decode_impl<128, 2, F16>(tk, tv, a, grid, stream);
    case 4: return launch_decode_impl<128, 4, F16>(tk, tv, a, grid, stream);
    default: return launch_decode_impl<128, 8, F16>(tk, tv, a, grid, stream);
  }
}

// E4M3 caches with a bf16 query: widths 128 and 256 (a 128-byte box row holds 128 elements).
cudaError_t launch_decode_e4m3(int d, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                               const DecodeArgs &a, int grid, cudaStream_t stream) {
  if (d == 256) {  // at most 4 heads per work item (DecodeArgs::nsplit)
    switch (group) {
      case 1: return launch_decode_impl<256, 1, false, true>(tk, tv, a, grid, stream);
      case 2: return launch_decode_impl<256, 2, false, true>(tk, tv, a, grid, stream);
      default: return launch_decode_impl<256, 4, false, true>(tk, tv, a, grid, stream);
    }
  }
  switch (group) {
    case 1: return launch_decode_impl<128, 1, false, true>(tk, tv, a, grid, stream);
    case 2: return launch_decode_impl<128, 2, false, true>(tk, tv, a, grid, stream);
    case 4: return launch_decode_impl<128, 4, false, true>(tk, tv, a, grid, stream);
    default: return launch_decode_impl<128, 8, false, true>(tk, tv, a, grid, stream);
  }
}

cudaError_t launch_decode(int d, int group, bool f16, bool kv_e4m3, const CUtensorMap &tk,
                          const CUtensorMap &tv, const DecodeArgs &a, int grid,
                          cudaStream_t stream) {
  if (kv_e4m3) return launch_decode_e4m3(d, group, tk, tv, a, grid, stream);
  return f16 ? launch_decode_typed<true>(d, group, tk, tv, a, grid, stream)
             : launch_decode_typed<false>(d, group, tk, tv, a, grid, stream);
}

cudaError_t launch_combine(int d, int d_out, bool f16, const float *o_part, const float *lse_part,
                           const int *cache_len, int len_add, int B, int Hq, int Lmax, int chunk,
                           int maxch, int wl, int kalign, void *o, float *lse,
                           unsigned int * /*err*/, cudaStream_t stream) {
  const int blocks = B * Hq;
  if (blocks == 0) return cudaSuccess;
  uint16_t *ob = reinterpret_cast<uint16_t *>(o);
  auto kern = d == 64    ? (f16 ? combine_kernel<64, true> : combine_kernel<64, false>)
              : d == 256 ? (f16 ? combine_kernel<256, true> : combine_kernel<256, false>)
                         : (f16 ? combine_kernel<128, true> : combine_kernel<128, false>);
  kern<<<blocks, d, 0, stream>>>(o_part, lse_part, cache_len, len_add, Hq, Lmax, chunk, maxch,
                                 wl, kalign, d_out, ob, lse);
  return cudaGetLastError();
}

}  // namespace fa
