// fa_backward.cu -- backward pass of exact attention for sm_103a.
//
// "flash-attention" (ai-reference-codex.pages.dev), sections 2.3 and 4: the backward pass
// keeps only q, k, v, out and softmax_lse, recomputes P = exp(S * scale - LSE) tile by tile
// instead of storing it, and is parallel over K/V column blocks: each block keeps its dK and
// dV on chip for the whole pass while dQ, which every key block contributes to, is
// accumulated in global memory ("FlashAttention 1-4 详解", FlashAttention 2 backward).
// With D_i = rowsum(dO_i * O_i) (computed by a preprocessing kernel):
//     S^T  = K Q^T,  P^T = 2^(S^T scale log2e - LSE_i log2e)        (masked pairs: 0)
//     dP^T = V dO^T, dS^T = P^T * (dP^T - D_i)
//     dV  += P^T dO,  dK += dS^T Q,  dQ += dS K
// and finally dK *= scale, dQ *= scale (a postprocessing kernel converts dQ).
//
// Work unit = (batch b, kv head g, 128-key block j), persistent CTAs taking units in order:
// groups of BwdArgs::head_group (b, g) pairs one after the other (8; 16 for the
// deterministic dQ order, whose CTAs wait on one another per pair; 4 at d > 128),
// key-block-major inside a group (with causal masking the first key blocks see the most
// queries, so the longest units of a group come first, and the group's dQ accumulators
// stay in L2; all heads key-block-major: 706 TFLOPS, head-major: 663, groups of 8: 737,
// measured on an earlier version of the kernel).  A unit visits every
// 128-query block i of every query head of group g whose rows can see a key of block j.
// Keys are the MMA rows (TMEM lanes) of S^T, dP^T, dV and dK, so the dK and dV
// accumulators stay in TMEM across the unit.
//
// Head dimensions up to 128 (bwd_kernel): 640 threads, no register split.
//   warps 0-15 compute: warp w takes TMEM lanes 32 (w % 4) .. +31 and, for P^T and dS^T
//              (thread = key row), queries 32 (w / 4) .. +31 of a step; for the dQ epilogue
//              (thread = query row) and the dK / dV epilogue at the end of a unit (thread =
//              key row), d columns (w / 4) D/4 .. +D/4
//   warp 16    producer: K, V (once per unit), Q, dO (per step) by TMA; LSE and D vectors
//   warp 17    TMEM allocator and MMA issuer (the whole warp, one elected lane issues)
//   warp 18    dQ issuer: TMA reduce-adds of the staged dQ tiles (and the deterministic
//              order), off the compute warps' critical path
//   warp 19    idle
// TMEM: S^T [0,128) (then P^T), dP^T [128,256) (then dS^T, then dQ), dV [256,256+d),
// dK [384,384+d).  P^T and dS^T are written back as packed 16-bit pairs, each 32-query
// quarter over the first 16 of its own 32 fp32 source columns, and feed the dV and dK MMAs
// from TMEM; dS is also written to shared memory (queries contiguous, the MN-major A
// operand of the dQ MMA).  Each step's dQ tile goes through shared memory to TMA bulk
// reduce-adds into an fp32 accumulator; the deterministic order (counters per query block)
// is a separate kernel instance.
// Per step the compute warps compute P^T as soon as S^T lands and dS^T once dP^T lands; the
// MMA issuer runs S^T (as soon as Q has landed), dP^T (once dO has landed and the previous
// dQ has been read), then dK, dV and dQ: dK and dV release Q and dO so that the next step's
// loads overlap the dQ product and its epilogue.
// Head dimensions 136..256: bwd_wide_kernel, described before its code below.
#include <climits>
#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int BKEY = 128;         // keys per unit
constexpr int BQ = 128;           // queries per step
// The d 136..256 kernel (bwd_wide_kernel): 384 threads, two compute warpgroups with a
// register split, warp 8 the producer, 9 the MMA issuer, 10 the dQ issuer, 11 idle.
constexpr int NTHREADS = 384;
constexpr int NCOMPUTE = 256;
constexpr int COMPUTE_REGS = 200;  // 2 x 128 threads x 200
constexpr int OTHER_REGS = 96;     //   + 128 threads x 96 <= 384 threads x 168 at launch
constexpr int PRODUCER_WARP = 8;
constexpr int DQ_WARP = 10;       // issues the dQ reduce-adds
constexpr int MMA_WARP = 9;
// The d <= 128 kernel (bwd_kernel): 16 compute warps, four per TMEM lane quarter (warp w:
// lanes 32 (w % 4) .. +31, queries 32 (w / 4) .. +31 of a step), 640 threads, no register
// split; warp 16 is the producer, 17 the MMA issuer, 18 the dQ issuer, 19 idle.
constexpr int NB_THREADS = 640;
constexpr int NB_COMPUTE = 512;
constexpr int NB_PRODUCER = 16, NB_MMA = 17, NB_DQ = 18;
constexpr int BOX = 128 * 128;    // one 128-byte-swizzled box: 128 rows x 128 bytes
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t T_ST = 0, T_DP = 128, T_DV = 256, T_DK = 384;
constexpr float LOG2E = 1.4426950408889634f;

template <int D, bool F16>
struct BCfg {
  static constexpr int KCH = D / 64;
  static constexpr int TILE = KCH * BOX;            // [128 x D] 16-bit tile
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TILE;
  static constexpr int Q_OFF = 2 * TILE;
  static constexpr int DO_OFF = 3 * TILE;
  static constexpr int DS_OFF = 4 * TILE;           // dS: 2 boxes (query halves) x 128 keys
  static constexpr int DQ_OFF = DS_OFF + 2 * BOX;   // fp32 dQ staging: D/32 boxes
  static constexpr int VEC_OFF = DQ_OFF + (D / 32) * BOX;  // lse2[128], dvec[128]
  static constexpr int BAR_OFF = VEC_OFF + 2 * BQ * 4;
  static constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, false, false, F16);
  static constexpr uint32_t IDESC_ACC = idesc_bf16_f32(128, D, false, true, F16);
  static constexpr uint32_t IDESC_DQ = idesc_bf16_f32(128, D, true, true, F16);
};

struct BBars {
  uint64_t kv_full, kv_empty, q_full, q_empty, do_full, do_empty, vec_full, vec_empty;
  uint64_t st_full, dp_full, p_ready, dq_full, dq_empty, acc_full, acc_empty, mma_done;
  uint64_t dq_staged, dq_free;  // dQ staging tile written (compute) / read by the TMA (issuer)
  uint64_t dq_free_r1;          // wide kernel: dq_free for the second staging round of a step
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(BBars) <= 256, "backward barriers exceed their shared-memory region");

struct BUnit {
  int b, g, j;
  int nq, nk;          // lengths of the sequence
  int q_tok, k_tok;    // packed-token offsets of the sequence (varlen), else 0
  int tma_b;           // batch coordinate of the tensor maps (0 for varlen)
  bool skip;           // key block j lies past the sequence's keys: nothing to do
  bool bad;            // varlen prefix sums out of range: the sequence is skipped
  int nqb;             // query blocks of the sequence
  int ilo, ihi;        // query blocks [ilo, ihi) of each head of the group reach key block j
  int nit;             // steps: group * (ihi - ilo)
};

template <int MASK, int QB = BQ>
__device__ __forceinline__ BUnit bunit_of(const BwdArgs &a, int u) {
  BUnit w;
  // Units run in groups of a.head_group (batch, kv head) pairs, key-block-major inside a
  // group: the CTAs running together then add dQ into a few heads' accumulators (4 MB
  // each at N = 8192, d = 128), which stay in L2, and causal work still mixes short and
  // long key blocks.
  const int bg = a.B * a.Hkv;
  const int S = a.head_group < bg ? a.head_group : bg;
  const int per = a.kblocks * S;
  const int grp = u / per;
  const int rem = u - grp * per;
  const int gs = min(S, bg - grp * S);  // the last group may be smaller
  w.j = rem / gs;
  const int r = grp * S + (rem - w.j * gs);
  w.b = r / a.Hkv;
  w.g = r - w.b * a.Hkv;
  if (a.varlen) {
    const int q0 = a.cu_q[w.b], q1 = a.cu_q[w.b + 1];
    const int k0 = a.cu_k[w.b], k1 = a.cu_k[w.b + 1];
    const bool bad = q0 < 0 || q1 < q0 || q1 > a.total_q || k0 < 0 || k1 < k0 ||
                     k1 > a.total_k || (q1 - q0) > a.Nq || (k1 - k0) > a.Nk;
    w.nq = bad ? 0 : q1 - q0;
    w.nk = bad ? 0 : k1 - k0;
    w.q_tok = bad ? 0 : q0;
    w.k_tok = bad ? 0 : k0;
    w.tma_b = 0;
    w.bad = bad;
  } else {
    w.bad = false;
    w.nq = a.Nq;
    w.nk = a.Nk;
    w.q_tok = 0;
    w.k_tok = 0;
    w.tma_b = w.b;
  }
  w.skip = w.j * BKEY >= w.nk;
  w.nqb = (w.nq + QB - 1) / QB;
  w.ilo = 0;
  w.ihi = w.nqb;
  const long long off = static_cast<long long>(w.nk) - w.nq;
  constexpr bool WIN = mask_has_window(MASK);
  const int wr = MASK == MASK_CAUSAL ? 0 : (WIN ? a.wr : -1);
  const int wl = WIN ? a.wl : -1;
  if (wr >= 0) {
    // first query block holding a row that sees a key of the block:
    // i*QB + QB-1 + off + wr >= j*128
    const long long t = static_cast<long long>(w.j) * BKEY - off - wr - (QB - 1);
    w.ilo = t <= 0 ? 0 : static_cast<int>(min((t + QB - 1) / QB, static_cast<long long>(w.nqb)));
  }
  if (wl >= 0) {
    // last query block holding a row that sees a key of the block: i*QB + off - wl <= kmax
    const long long kmax = min(static_cast<long long>(w.j) * BKEY + BKEY - 1, w.nk - 1ll);
    const long long t = kmax - off + wl;
    w.ihi = t < 0 ? 0 : static_cast<int>(min(t / QB + 1, static_cast<long long>(w.nqb)));
  }
  if (w.ihi < w.ilo) w.ihi = w.ilo;
  w.nit = w.skip ? 0 : a.group * (w.ihi - w.ilo);
  return w;
}

// Step t of a unit: query head and query block.
__device__ __forceinline__ void bstep(const BwdArgs &a, const BUnit &w, int t, int &h, int &i) {
  const int per = w.ihi - w.ilo;
  h = w.g * a.group + t / per;
  i = w.ilo + t % per;
}

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const WaitCtl &wc) {
  const bool ok = mbar_wait(bar, parity, wc);
  return __all_sync(0xffffffffu, ok);
}

// Waits (bounded) until *ctr == target, then orders later TMA global accesses after it.
__device__ __forceinline__ bool wait_counter(int *ctr, int target, const WaitCtl &c) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) break;
    if (*c.abort) return false;
    if (globaltimer_ns() - t0 > c.timeout_ns) {
      *c.abort = 1;
      atomicOr(c.err, c.code);
      return false;
    }
  }
  fence_proxy_async_global();
  return true;
}


// The issue helpers are warp-collective (the whole MMA warp runs them, one lane issues).
// M=128 x N=128 x K=D product of two K-major 128-byte-swizzled tiles (S^T and dP^T).
template <int D, bool F16>
__device__ __forceinline__ void issue_kmajor(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = static_cast<uint32_t>((kk >> 2) * BOX + (kk & 3) * 32);
    mma_bf16_ss_w(d_tmem, sw128_desc(a_smem + off, 16, 1024), sw128_desc(b_smem + off, 16, 1024),
                BCfg<D, F16>::IDESC_S, kk > 0 ? 1u : 0u);
  }
}

// TMEM column of the packed pair holding queries (2c, 2c+1): each 32-query quarter of a step
// sits at the start of its own 32 fp32 source columns.
__host__ __device__ constexpr uint32_t packed_col(int query) {
  return static_cast<uint32_t>(32 * (query >> 5) + (query & 31) / 2);
}

// Stores 8 consecutive 32-bit TMEM columns of the thread's lane (no wait).
__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n"
      :
      : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

// D[128 keys x D] (+)= A[128 keys x 128 queries] (TMEM, packed pairs) * B[128 queries x D]
// (MN-major tile: rows = queries, D contiguous).  dV and dK.
template <int D, bool F16>
__device__ __forceinline__ void issue_acc(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem,
                                          bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < BQ / 16; ++kk)
    mma_bf16_ts_w(d_tmem, a_tmem + packed_col(kk * 16),
                sw128_desc(b_smem + static_cast<uint32_t>(kk * 16 * 128), BOX, 1024),
                BCfg<D, F16>::IDESC_ACC, (accumulate || kk > 0) ? 1u : 0u);
}

// dQ[128 queries x D] = dS[128 queries x 128 keys] (shared memory, MN-major: rows = keys,
// queries contiguous) * K[128 keys x D] (MN-major: rows = keys, D contiguous).
template <int D, bool F16>
__device__ __forceinline__ void issue_dq(uint32_t d_tmem, uint32_t ds_smem, uint32_t k_smem) {
#pragma unroll
  for (int kk = 0; kk < BKEY / 16; ++kk) {
    const uint32_t off = static_cast<uint32_t>(kk * 16 * 128);
    mma_bf16_ss_w(d_tmem, sw128_desc(ds_smem + off, BOX, 1024), sw128_desc(k_smem + off, BOX, 1024),
                BCfg<D, F16>::IDESC_DQ, kk > 0 ? 1u : 0u);
  }
}

// ------------------------------------------------------------------------------------
// Producer warp.

template <int D, int MASK, bool F16>
__device__ void bwd_producer(const BwdArgs &a, const CUtensorMap *tq, const CUtensorMap *tk,
                             const CUtensorMap *tv, const CUtensorMap *tdo, uint8_t *smem,
                             BBars *bars, const WaitCtl &wc, int lane) {
  using C = BCfg<D, F16>;
  float *lse2 = reinterpret_cast<float *>(smem + C::VEC_OFF);
  float *dvec = lse2 + BQ;
  uint32_t kv_n = 0, q_n = 0;
  if (a.inject) goto out;  // failure injection: load nothing, the consumers' waits run out
  for (int u = blockIdx.x; u < a.num_units; u += gridDim.x) {
    const BUnit w = bunit_of<MASK>(a, u);
    if (w.bad && w.j == 0 && w.g == 0 && lane == 0) atomicOr(a.err, DEVERR_BAD_CU_SEQLENS);
    if (w.nit == 0) continue;
    if (kv_n > 0 && !warp_wait(&bars->kv_empty, (kv_n - 1) & 1u, wc)) goto out;
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars->kv_full, 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < C::KCH; ++c) {
        tma_load_4d(smem + C::K_OFF + c * BOX, tk, &bars->kv_full, c * 64, w.g,
                    w.k_tok + w.j * BKEY, w.tma_b);
        tma_load_4d(smem + C::V_OFF + c * BOX, tv, &bars->kv_full, c * 64, w.g,
                    w.k_tok + w.j * BKEY, w.tma_b);
      }
    }
    ++kv_n;
    for (int t = 0; t < w.nit; ++t) {
      int h, i;
      bstep(a, w, t, h, i);
      // LSE and D of the step's rows, loaded before the waits below so that their latency
      // overlaps them (rows past the sequence, the next one's for varlen, are not read).
      const int64_t base = w.b * a.lse_sb + h * a.lse_sh + w.q_tok;
      float lv[4], dv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int q = i * BQ + lane * 4 + e;
        lv[e] = q < w.nq ? a.lse[base + q] : -INFINITY;
        dv[e] = q < w.nq ? a.dvec[base + q] : 0.f;
      }
      if (q_n > 0 && !warp_wait(&bars->q_empty, (q_n - 1) & 1u, wc)) goto out;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->q_full, C::TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d(smem + C::Q_OFF + c * BOX, tq, &bars->q_full, c * 64, h,
                      w.q_tok + i * BQ, w.tma_b);
      }
      if (q_n > 0 && !warp_wait(&bars->do_empty, (q_n - 1) & 1u, wc)) goto out;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->do_full, C::TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d(smem + C::DO_OFF + c * BOX, tdo, &bars->do_full, c * 64, h,
                      w.q_tok + i * BQ, w.tma_b);
      }
      // LSE in the log2 domain (rows past the sequence or with no visible key: +inf, so
      // that P = 0) and D.
      if (q_n > 0 && !warp_wait(&bars->vec_empty, (q_n - 1) & 1u, wc)) goto out;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        lse2[lane * 4 + e] = lv[e] == -INFINITY ? INFINITY : lv[e] * LOG2E;
        dvec[lane * 4 + e] = dv[e];
      }
      __syncwarp();
      mbar_arrive(&bars->vec_full);
      ++q_n;
    }
  }
out:
  // Teardown: the last bulk copies issued must land before the CTA may exit.
  if (lane == 0) {
    if (kv_n > 0) mbar_wait_teardown(&bars->kv_full, (kv_n - 1) & 1u, 1000000000ull);
    if (q_n > 0) mbar_wait_teardown(&bars->q_full, (q_n - 1) & 1u, 1000000000ull);
    if (q_n > 0) mbar_wait_teardown(&bars->do_full, (q_n - 1) & 1u, 1000000000ull);
  }
}

// ------------------------------------------------------------------------------------
// dQ issuer: once the compute warps have staged a step's dQ tile, adds it into the fp32
// accumulator with TMA reduce-adds (one box of 32 columns x 128 rows per 32 columns), then
// frees the staging tile as soon as the TMA has read it.  The whole warp runs the loop, lane 0 issues.  Deterministic
// order: before adding, lane 0 waits until the (batch, head, query block) counter shows
// that the key blocks before this one have added, and after its own addition has landed
// it increments the counter.

template <int D, int MASK, bool F16>
__device__ void bwd_dq_issuer(const BwdArgs &a, const CUtensorMap *tdq, uint8_t *smem,
                              BBars *bars, const WaitCtl &wc, int lane) {
  using C = BCfg<D, F16>;
  uint8_t *dq_s = smem + C::DQ_OFF;
  uint32_t it = 0;
  for (int u = blockIdx.x; u < a.num_units; u += gridDim.x) {
    const BUnit w = bunit_of<MASK>(a, u);
    if (w.skip || w.nit == 0) continue;
    const int off = w.nk - w.nq;
    for (int t = 0; t < w.nit; ++t) {
      int h, i;
      bstep(a, w, t, h, i);
      const int q0 = i * BQ;
      if (!warp_wait(&bars->dq_staged, it & 1u, wc)) return;
      bool ok = true;
      if (lane == 0) {
        int *sem = a.sem ? a.sem + (static_cast<int64_t>(w.b) * a.Hq + h) * a.qblocks + i : nullptr;
        // Deterministic order: the key blocks that reach query block i are an interval
        // jmin .. jmax (jmin = 0 unless a left window bound cuts the first keys); block j
        // adds after jmin .. j-1.
        int jmin = 0;
        if (mask_has_window(MASK) && a.wl >= 0)
          jmin = max(q0 + off - a.wl, 0) / BKEY;
        ok = sem == nullptr || wait_counter(sem, w.j - jmin, wc);
        if (ok) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc)
            tma_reduce_add_4d(tdq, dq_s + cc * BOX, cc * 32, h, w.q_tok + q0, w.tma_b);
          bulk_commit_group();
          bulk_wait_read();              // the staging tile may be written again
          mbar_arrive(&bars->dq_free);
          if (sem != nullptr) {
            bulk_wait_all();             // the additions have been performed
            fence_proxy_async_global();
            __threadfence();
            atomicAdd(sem, 1);
          }
        }
      }
      if (!__all_sync(0xffffffffu, ok)) return;
      ++it;
    }
  }
}

// ------------------------------------------------------------------------------------
// MMA issuer: the whole warp runs the loop, one elected lane issues (an issuing loop
// confined to one lane is starved by the compute warps of its sub-partition).

template <int D, int MASK, bool F16>
__device__ void bwd_mma(const BwdArgs &a, uint8_t *smem, BBars *bars, uint32_t tmem,
                        const WaitCtl &wc) {
  using C = BCfg<D, F16>;
  const uint32_t sK = smem_u32(smem + C::K_OFF), sV = smem_u32(smem + C::V_OFF);
  const uint32_t sQ = smem_u32(smem + C::Q_OFF), sDO = smem_u32(smem + C::DO_OFF);
  const uint32_t sDS = smem_u32(smem + C::DS_OFF);
  uint32_t kv_n = 0, it = 0, acc_n = 0;
  for (int u = blockIdx.x; u < a.num_units; u += gridDim.x) {
    const BUnit w = bunit_of<MASK>(a, u);
    if (w.nit == 0) continue;
    if (!warp_wait(&bars->kv_full, kv_n & 1u, wc)) goto out;
    ++kv_n;
    if (acc_n > 0 && !warp_wait(&bars->acc_empty, (acc_n - 1) & 1u, wc)) goto out;
    for (int t = 0; t < w.nit; ++t) {
      if (!warp_wait(&bars->q_full, it & 1u, wc)) goto out;
      tc_fence_after();
      issue_kmajor<D, F16>(tmem + T_ST, sK, sQ);                  // S^T = K Q^T
      mma_commit_w(&bars->st_full);
      if (!warp_wait(&bars->do_full, it & 1u, wc)) goto out;
      // dP^T overwrites the previous step's dQ: wait until the epilogue has read it.
      if (it > 0 && !warp_wait(&bars->dq_empty, (it - 1) & 1u, wc)) goto out;
      tc_fence_after();
      issue_kmajor<D, F16>(tmem + T_DP, sV, sDO);                 // dP^T = V dO^T
      mma_commit_w(&bars->dp_full);
      if (!warp_wait(&bars->p_ready, it & 1u, wc)) goto out;
      tc_fence_after();
      issue_acc<D, F16>(tmem + T_DK, tmem + T_DP, sQ, t > 0);     // dK += dS^T Q
      mma_commit_w(&bars->q_empty);
      issue_acc<D, F16>(tmem + T_DV, tmem + T_ST, sDO, t > 0);    // dV += P^T dO
      mma_commit_w(&bars->do_empty);
      issue_dq<D, F16>(tmem + T_DP, sDS, sK);                     // dQ = dS K
      mma_commit_w(&bars->dq_full);
      ++it;
    }
    mma_commit_w(&bars->kv_empty);
    mma_commit_w(&bars->acc_full);
    ++acc_n;
  }
out:
  mma_commit_w(&bars->mma_done);
  mbar_wait_teardown(&bars->mma_done, 0u, 1000000000ull);
}

// ------------------------------------------------------------------------------------
// Compute warps: warp w handles TMEM lanes 32 (w % 4) .. +31, queries 32 (w / 4) .. +31 of a
// step for P^T / dS^T, and d columns (w / 4) D/4 .. +D/4 in the dQ, dK and dV epilogues.

template <int D, int MASK, bool F16, bool DET>
__device__ void bwd_compute(const BwdArgs &a, const CUtensorMap *tdq, uint8_t *smem, BBars *bars,
                            uint32_t tmem, const WaitCtl &wc, int tid) {
  using C = BCfg<D, F16>;
  const int warp = tid >> 5;
  const int qd = warp >> 2;                   // query quarter (P, dS) / d quarter (dQ, dK, dV)
  const int r = (warp & 3) * 32 + (tid & 31); // TMEM lane: key row, or query row for dQ
  constexpr int DW = D / 4;                   // d columns of a warp in the dQ, dK, dV epilogues
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const float *lse2 = reinterpret_cast<const float *>(smem + C::VEC_OFF);
  const float *dvec = lse2 + BQ;
  uint8_t *ds_s = smem + C::DS_OFF;
  uint8_t *dq_s = smem + C::DQ_OFF;
  uint32_t it = 0, acc_n = 0;
  bool vec_ready = false;  // the current step's LSE / D already waited for
  for (int u = blockIdx.x; u < a.num_units; u += gridDim.x) {
    const BUnit w = bunit_of<MASK>(a, u);
    if (w.skip) continue;
    const int off = w.nk - w.nq;  // bottom-right alignment: query q sits at key position q + off
    const int key = w.j * BKEY + r;
    uint16_t *dkrow = reinterpret_cast<uint16_t *>(a.dk) + w.b * a.dk_sb +
                      (w.k_tok + key) * a.dk_sn + w.g * a.dk_sh;
    uint16_t *dvrow = reinterpret_cast<uint16_t *>(a.dv) + w.b * a.dv_sb +
                      (w.k_tok + key) * a.dv_sn + w.g * a.dv_sh;
    if (w.nit == 0) {  // no query sees these keys: zero gradients
      if (key < w.nk) {
#pragma unroll
        for (int v = qd * (DW / 8); v < (qd + 1) * (DW / 8); ++v) {
          if (8 * v >= a.d) break;
          reinterpret_cast<uint4 *>(dkrow)[v] = make_uint4(0u, 0u, 0u, 0u);
          reinterpret_cast<uint4 *>(dvrow)[v] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      continue;
    }
    for (int t = 0; t < w.nit; ++t) {
      int h, i;
      bstep(a, w, t, h, i);
      const int q0 = i * BQ;
      const int kb = w.j * BKEY;
      bool full;  // no pair of the 128 x 128 block masked
      if constexpr (MASK == MASK_NONE) {
        full = kb + BKEY <= w.nk;
      } else if constexpr (MASK == MASK_CAUSAL) {
        full = kb + BKEY <= w.nk && kb + BKEY - 1 <= q0 + off;
      } else {
        full = kb + BKEY <= w.nk && (a.wr < 0 || kb + BKEY - 1 <= q0 + off + a.wr) &&
               (a.wl < 0 || kb >= q0 + BQ - 1 + off - a.wl);
      }
      // this key row's visible query positions (modifiers): key - wr - off <= q <= key + wl - off
      constexpr bool WIN = mask_has_window(MASK);
      constexpr bool SCORE_MOD = MASK == MASK_MOD || MASK == MASK_ALIBI;
      const int qv_lo = WIN && a.wr >= 0 ? key - a.wr - off : INT_MIN;
      const int qv_hi = WIN && a.wl >= 0 ? key + a.wl - off : INT_MAX;
      const bool softcap = MASK == MASK_MOD && a.sc_out != 0.f;
      const bool alibi = SCORE_MOD && a.alibi != nullptr;
      // ALiBi without a softcap on a block with no masked pair whose queries all sit at or
      // after its keys: the bias -slope2 (q + off - key) is linear in the query.
      const bool alibi_lin = MASK == MASK_ALIBI && full && kb + BKEY - 1 <= q0 + off;
      const float slope2 = alibi ? a.alibi[w.b * a.alibi_sb + h] * LOG2E : 0.f;
      // Phase 1, as soon as S^T has landed (the MMA of dP^T may still run): P^T of this key
      // row for the 32 queries of this quarter, to TMEM as packed 16-bit pairs over the
      // quarter's first 16 source columns (dV).  P, times dz/ds under a softcap, stays in
      // registers for phase 2.
      if (!vec_ready && !warp_wait(&bars->vec_full, it & 1u, wc)) return;
      vec_ready = false;
      if (!warp_wait(&bars->st_full, it & 1u, wc)) return;
      tc_fence_after();
      const int qq = qd * 32;  // first query of the quarter
      float pd[32];
      {
        uint32_t sr[32], pp[16];
        tmem_ld_x32(tmem + lane_off + T_ST + qq, sr);
        if (MASK == MASK_ALIBI && alibi_lin) {
          // P = 2^(S c - slope2 (q + off - key) - LSE2): the bias pairs of queries (e, e+1)
          // and (e+2, e+3) step by -4 slope2 along two chains that start from exact
          // products, on packed fp32 pairs.
          const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
          const float base = -slope2 * static_cast<float>(q0 + qq + off - key);
          uint64_t w01 = f2_pack(base, base - slope2);
          uint64_t w23 = f2_pack(base - 2.f * slope2, base - 3.f * slope2);
          const uint64_t step = f2_pack(-4.f * slope2, -4.f * slope2);
#pragma unroll
          for (int e4 = 0; e4 < 32; e4 += 4) {
            const float4 l4 = *reinterpret_cast<const float4 *>(lse2 + qq + e4);
            float z0, z1, z2, z3;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e4]), __uint_as_float(sr[e4 + 1])), sc2,
                             f2_add(w01, f2_pack(-l4.x, -l4.y))), z0, z1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e4 + 2]), __uint_as_float(sr[e4 + 3])),
                             sc2, f2_add(w23, f2_pack(-l4.z, -l4.w))), z2, z3);
            w01 = f2_add(w01, step);
            w23 = f2_add(w23, step);
            pd[e4] = ex2_approx(z0);
            pd[e4 + 1] = ex2_approx(z1);
            pd[e4 + 2] = ex2_approx(z2);
            pd[e4 + 3] = ex2_approx(z3);
            pp[e4 / 2] = pack2<F16>(pd[e4], pd[e4 + 1]);
            pp[e4 / 2 + 1] = pack2<F16>(pd[e4 + 2], pd[e4 + 3]);
          }
        } else if (!SCORE_MOD && full) {
          // No masked pair and no modifier: P = 2^(S c - LSE2) on packed fp32 pairs.
          const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
#pragma unroll
          for (int e4 = 0; e4 < 32; e4 += 4) {
            const float4 l4 = *reinterpret_cast<const float4 *>(lse2 + qq + e4);
            float z0, z1, z2, z3;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e4]), __uint_as_float(sr[e4 + 1])), sc2,
                             f2_pack(-l4.x, -l4.y)), z0, z1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e4 + 2]), __uint_as_float(sr[e4 + 3])),
                             sc2, f2_pack(-l4.z, -l4.w)), z2, z3);
            pd[e4] = ex2_approx(z0);
            pd[e4 + 1] = ex2_approx(z1);
            pd[e4 + 2] = ex2_approx(z2);
            pd[e4 + 3] = ex2_approx(z3);
            pp[e4 / 2] = pack2<F16>(pd[e4], pd[e4 + 1]);
            pp[e4 / 2 + 1] = pack2<F16>(pd[e4 + 2], pd[e4 + 3]);
          }
        } else {
#pragma unroll
          for (int e2 = 0; e2 < 32; e2 += 2) {
            float p[2];
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              const int qi = qq + e2 + x;
              const float sv = __uint_as_float(sr[e2 + x]);
              float z2, dz = 1.f;  // score in log2 units and dz/ds
              if constexpr (SCORE_MOD) {
                if (softcap) {
                  const float t = tanh_ex2(sv * a.sc_in);
                  z2 = t * a.sc_out;
                  dz = 1.f - t * t;
                } else {
                  z2 = sv * a.scale_log2;
                }
                if (alibi) z2 = fmaf(-slope2, fabsf(static_cast<float>(q0 + qi + off - key)), z2);
              } else {
                z2 = sv * a.scale_log2;
              }
              bool vis;
              if constexpr (WIN)
                vis = full || (key < w.nk && q0 + qi >= qv_lo && q0 + qi <= qv_hi);
              else
                vis = full || (key < w.nk && (MASK == MASK_NONE || key <= q0 + qi + off));
              const float pv = ex2_approx(z2 - lse2[qi]);
              p[x] = vis ? pv : 0.f;
              pd[e2 + x] = p[x] * dz;
            }
            pp[e2 / 2] = pack2<F16>(p[0], p[1]);
          }
        }
        tmem_st_x16(tmem + lane_off + T_ST + packed_col(qq), pp);
      }
      // Phase 2, once dP^T has landed: dS^T = P^T (dP^T - D) of the same 32 queries, 16 at a
      // time, to TMEM as packed pairs (dK) and to shared memory with queries contiguous (dQ).
      if (!warp_wait(&bars->dp_full, it & 1u, wc)) return;
      tc_fence_after();
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int qc = qq + c2 * 16;  // first query of the chunk
        uint32_t dr[16], dd[8];
        tmem_ld_x16(tmem + lane_off + T_DP + qc, dr);
#pragma unroll
        for (int e4 = 0; e4 < 16; e4 += 4) {
          const float4 d4 = *reinterpret_cast<const float4 *>(dvec + qc + e4);
          const float *pe = pd + c2 * 16 + e4;
          float e0, e1, e2, e3;
          f2_unpack(f2_mul(f2_pack(pe[0], pe[1]),
                           f2_add(f2_pack(__uint_as_float(dr[e4]), __uint_as_float(dr[e4 + 1])),
                                  f2_pack(-d4.x, -d4.y))), e0, e1);
          f2_unpack(f2_mul(f2_pack(pe[2], pe[3]),
                           f2_add(f2_pack(__uint_as_float(dr[e4 + 2]), __uint_as_float(dr[e4 + 3])),
                                  f2_pack(-d4.z, -d4.w))), e2, e3);
          dd[e4 / 2] = pack2<F16>(e0, e1);
          dd[e4 / 2 + 1] = pack2<F16>(e2, e3);
        }
        tmem_st_x8(tmem + lane_off + T_DP + packed_col(qc), dd);
        uint8_t *box = ds_s + (qc >> 6) * BOX + r * 128;  // box = query half
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
          const int gran = ((qc & 63) >> 3) + gi;
          *reinterpret_cast<uint4 *>(box + ((gran ^ (r & 7)) << 4)) =
              make_uint4(dd[4 * gi], dd[4 * gi + 1], dd[4 * gi + 2], dd[4 * gi + 3]);
        }
      }
      mbar_arrive(&bars->vec_empty);
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_ready);
      // dQ epilogue: TMEM -> shared memory (fp32, 128-byte swizzle); the reduce-add into
      // the accumulator is issued by the dQ issuer warp, off this critical path.
      // Barriers that complete early are polled before the staging stores below, which
      // queue ahead of any later poll in the shared-memory pipe: the issuer's previous
      // reduction has read the staging tile (unordered dQ only: in deterministic order that
      // reduction waits for other CTAs, and the TMEM handoff must not wait behind it), and
      // (within a unit) the next step's LSE / D.
      if (!DET && it > 0 && !warp_wait(&bars->dq_free, (it - 1) & 1u, wc)) return;
      if (t + 1 < w.nit) {
        if (!warp_wait(&bars->vec_full, (it + 1) & 1u, wc)) return;
        vec_ready = true;
      }
      if (!warp_wait(&bars->dq_full, it & 1u, wc)) return;
      tc_fence_after();
      {
        // this warp's DW columns of dQ: one 32-column box (D = 128) or half of one (D = 64)
        uint32_t qr[DW];
        if constexpr (DW == 32)
          tmem_ld_x32(tmem + lane_off + T_DP + qd * DW, qr);
        else
          tmem_ld_x16(tmem + lane_off + T_DP + qd * DW, qr);
        // The columns are in registers: the MMA of the next dP^T may overwrite them.
        tc_fence_before();
        mbar_arrive(&bars->dq_empty);
        if (DET && it > 0 && !warp_wait(&bars->dq_free, (it - 1) & 1u, wc)) return;
        const int c0 = qd * DW;  // first dQ column
        uint8_t *box = dq_s + (c0 >> 5) * BOX + r * 128;
#pragma unroll
        for (int gi = 0; gi < DW / 4; ++gi) {
          const int gran = ((c0 & 31) >> 2) + gi;
          *reinterpret_cast<uint4 *>(box + ((gran ^ (r & 7)) << 4)) =
              make_uint4(qr[4 * gi], qr[4 * gi + 1], qr[4 * gi + 2], qr[4 * gi + 3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->dq_staged);
      ++it;
    }
    // Unit end: dV and scale * dK of this key row (this warp's DW columns of d) -> global.
    if (!warp_wait(&bars->acc_full, acc_n & 1u, wc)) return;
    tc_fence_after();
    {
      const int cc = qd * DW;  // first d column
      uint32_t vr[DW], kr[DW];
      if constexpr (DW == 32) {
        tmem_ld_x32(tmem + lane_off + T_DV + cc, vr);
        tmem_ld_x32(tmem + lane_off + T_DK + cc, kr);
      } else {
        tmem_ld_x16(tmem + lane_off + T_DV + cc, vr);
        tmem_ld_x16(tmem + lane_off + T_DK + cc, kr);
      }
      if (key < w.nk) {
#pragma unroll
        for (int v = 0; v < DW / 8; ++v) {
          if (cc + 8 * v >= a.d) break;  // columns past d are padding
          uint4 wv, wk;
          wv.x = pack2<F16>(__uint_as_float(vr[8 * v + 0]), __uint_as_float(vr[8 * v + 1]));
          wv.y = pack2<F16>(__uint_as_float(vr[8 * v + 2]), __uint_as_float(vr[8 * v + 3]));
          wv.z = pack2<F16>(__uint_as_float(vr[8 * v + 4]), __uint_as_float(vr[8 * v + 5]));
          wv.w = pack2<F16>(__uint_as_float(vr[8 * v + 6]), __uint_as_float(vr[8 * v + 7]));
          wk.x = pack2<F16>(__uint_as_float(kr[8 * v + 0]) * a.scale, __uint_as_float(kr[8 * v + 1]) * a.scale);
          wk.y = pack2<F16>(__uint_as_float(kr[8 * v + 2]) * a.scale, __uint_as_float(kr[8 * v + 3]) * a.scale);
          wk.z = pack2<F16>(__uint_as_float(kr[8 * v + 4]) * a.scale, __uint_as_float(kr[8 * v + 5]) * a.scale);
          wk.w = pack2<F16>(__uint_as_float(kr[8 * v + 6]) * a.scale, __uint_as_float(kr[8 * v + 7]) * a.scale);
          reinterpret_cast<uint4 *>(dvrow + cc)[v] = wv;
          reinterpret_cast<uint4 *>(dkrow + cc)[v] = wk;
        }
      }
    }
    tc_fence_before();
    mbar_arrive(&bars->acc_empty);
    ++acc_n;
  }
}

// DET: deterministic dQ order (a.sem != nullptr), a separate instance so that each order's
// compute loop is scheduled on its own.
template <int D, int MASK, bool F16, bool DET>
__global__ void __launch_bounds__(NB_THREADS, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
               const __grid_constant__ CUtensorMap tdq, const BwdArgs a) {
  using C = BCfg<D, F16>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  BBars *bars = reinterpret_cast<BBars *>(smem + C::BAR_OFF);
  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    mbar_init(&bars->do_full, 1);
    mbar_init(&bars->do_empty, 1);
    mbar_init(&bars->vec_full, 32);
    mbar_init(&bars->vec_empty, NB_COMPUTE);
    mbar_init(&bars->st_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_ready, NB_COMPUTE);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_empty, NB_COMPUTE);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, NB_COMPUTE);
    mbar_init(&bars->mma_done, 1);
    mbar_init(&bars->dq_staged, NB_COMPUTE);
    mbar_init(&bars->dq_free, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == NB_PRODUCER && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&tdo);
    tma_prefetch_desc(&tdq);
  }
  if (warp == NB_MMA) {
    tmem_alloc(&bars->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort, a.err, a.timeout_ns, DEVERR_BWD_TIMEOUT};
  // Every role ends on its own; all meet at a named barrier before TMEM is released.
  if (warp < NB_PRODUCER) {
    bwd_compute<D, MASK, F16, DET>(a, &tdq, smem, bars, tmem, wc, tid);
  } else if (warp == NB_PRODUCER) {
    bwd_producer<D, MASK, F16>(a, &tq, &tk, &tv, &tdo, smem, bars, wc, lane);
  } else if (warp == NB_MMA) {
    bwd_mma<D, MASK, F16>(a, smem, bars, tmem, wc);
  } else if (warp == NB_DQ) {
    bwd_dq_issuer<D, MASK, F16>(a, &tdq, smem, bars, wc, lane);
    if (lane == 0) bulk_wait_all();  // every dQ reduction has landed
  }
  __syncwarp();
  tc_fence_before();
  named_barrier(1, NB_THREADS);
  if (warp == NB_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------------
// Head dimensions 136..256: bwd_wide_kernel<MASK, F16> (kernel width 256).
//
// dK and dV of 128 keys at d = 256 alone would fill TMEM, and 128-query Q / dO tiles would
// not fit shared memory next to K and V, so a unit of this kernel is (batch, kv head,
// 128-key block, d half h) and a step is 64 queries.  Each unit recomputes S^T and dP^T over
// the full d and accumulates only its half of dK and dV, and adds its half of the d columns
// of dQ (the two halves of a key block run as adjacent units, so the second reads K, V, Q
// and dO mostly from L2).  Per step:
//     S^T  = K Q^T,  dP^T = V dO^T          [128 keys x 64 queries], K-dim 256
//     dK_h += dS^T Q_h,  dV_h += P^T dO_h    [128 keys x 128], K-dim 64 queries, A from TMEM
//     dQ^T_h = K_h^T dS^T                    [128 d rows x 64 queries], K-dim 128 keys
// TMEM: S^T [0,64), dP^T [64,128) (then dS^T, then dQ^T_h), dV_h [128,256), dK_h [256,384).
// Warpgroup x takes queries [32x, 32x+32) of a step for P^T / dS^T (thread = key row, the
// packed 16-bit results over the first 16 of the chunk's 32 source columns), and the same
// 32 query columns of dQ^T_h (thread = d row), which go through one 16 KB staging box
// (warpgroup 0's round, then warpgroup 1's) to a TMA reduce-add into the transposed fp32
// accumulator [B, Hq, d, Nq rounded up to 4] at d rows [128h, 128h + 128).
// Shared memory: K, V 64 KB each (four 128 x 64 boxes), Q, dO 32 KB each (four 64 x 64
// boxes), dS 16 KB, dQ^T staging 16 KB, vectors and barriers: 226 KB.

constexpr int WQ = 64;                // queries per step of the wide kernel
constexpr int QBOX = WQ * 128;        // one 64-row box of Q or dO
constexpr uint32_t W_ST = 0, W_DP = 64, W_DV = 128, W_DK = 256;

struct WCfg {
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = 4 * BOX;
  static constexpr int Q_OFF = 8 * BOX;
  static constexpr int DO_OFF = Q_OFF + 4 * QBOX;
  static constexpr int DS_OFF = DO_OFF + 4 * QBOX;  // dS [128 keys x 64 queries]: one box
  static constexpr int DQ_OFF = DS_OFF + BOX;       // dQ^T staging: 128 d rows x 32 queries
  static constexpr int VEC_OFF = DQ_OFF + BOX;      // LSE (log2) [64], D [64]
  static constexpr int BAR_OFF = VEC_OFF + 2 * WQ * 4;
  static constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;
};
static_assert(WCfg::SMEM_BYTES <= 232448, "wide backward kernel shared memory");

template <bool F16>
struct WDesc {
  static constexpr uint32_t S = idesc_bf16_f32(128, WQ, false, false, F16);
  static constexpr uint32_t ACC = idesc_bf16_f32(128, 128, false, true, F16);
  static constexpr uint32_t DQT = idesc_bf16_f32(128, WQ, true, true, F16);
};

// S^T or dP^T [128 keys x 64 queries] = A [128 x 256] B [64 x 256]^T, both K-major: 16 MMAs
// of 128 x 64 x 16; A's boxes are 16 KB apart, B's 8 KB.
template <bool F16>
__device__ __forceinline__ void wide_issue_s(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem) {
#pragma unroll
  for (int kk = 0; kk < 16; ++kk) {
    const uint32_t in_row = static_cast<uint32_t>((kk & 3) * 32);
    mma_bf16_ss_w(d_tmem, sw128_desc(a_smem + static_cast<uint32_t>((kk >> 2) * BOX) + in_row, 16, 1024),
                  sw128_desc(b_smem + static_cast<uint32_t>((kk >> 2) * QBOX) + in_row, 16, 1024),
                  WDesc<F16>::S, kk > 0 ? 1u : 0u);
  }
}

// dK_h or dV_h [128 keys x 128] (+)= A [128 keys x 64 queries] (TMEM, packed pairs: queries
// 0-31 at +0, 32-63 at +32) * B [64 queries x 128] (the d half of Q or dO, MN-major: two
// 64-column boxes 8 KB apart); 4 MMAs of 128 x 128 x 16.
template <bool F16>
__device__ __forceinline__ void wide_issue_acc(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem,
                                               bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_bf16_ts_w(d_tmem, a_tmem + static_cast<uint32_t>(kk < 2 ? 8 * kk : 32 + 8 * (kk - 2)),
                  sw128_desc(b_smem + static_cast<uint32_t>(kk * 16 * 128), QBOX, 1024),
                  WDesc<F16>::ACC, (accumulate || kk > 0) ? 1u : 0u);
}

// dQ^T_h [128 d rows x 64 queries] = K_h^T [128 x 128 keys] dS^T: A = the d half of K as an
// MN-major operand (two 64-d boxes 16 KB apart), B = dS (rows = keys, queries contiguous);
// 8 MMAs of 128 x 64 x 16.
template <bool F16>
__device__ __forceinline__ void wide_issue_dqt(uint32_t d_tmem, uint32_t k_smem, uint32_t ds_smem) {
#pragma unroll
  for (int kk = 0; kk < BKEY / 16; ++kk) {
    const uint32_t off = static_cast<uint32_t>(kk * 16 * 128);
    mma_bf16_ss_w(d_tmem, sw128_desc(k_smem + off, BOX, 1024), sw128_desc(ds_smem + off, BOX, 1024),
                  WDesc<F16>::DQT, kk > 0 ? 1u : 0u);
  }
}

// One 32-query round of dQ^T (fp32 bits) into row r of the staging box, 128-byte swizzled.
__device__ __forceinline__ void wide_stage_dqt(uint8_t *box, int r, const uint32_t (&v)[32]) {
  uint8_t *row = box + r * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4 *>(row + ((c ^ (r & 7)) << 4)) =
        make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

template <int MASK, bool F16>
__device__ void wide_producer(const BwdArgs &a, const CUtensorMap *tq, const CUtensorMap *tk,
                              const CUtensorMap *tv, const CUtensorMap *tdo, uint8_t *smem,
                              BBars *bars, const WaitCtl &wc, int lane) {
  using C = WCfg;
  float *lse2 = reinterpret_cast<float *>(smem + C::VEC_OFF);
  float *dvec = lse2 + WQ;
  uint32_t kv_n = 0, q_n = 0, do_n = 0, vec_n = 0;
  if (a.inject) goto out;  // failure injection: load nothing, the consumers' waits run out
  for (int u = blockIdx.x; u < a.num_units; u += gridDim.x) {
    const BUnit w = bunit_of<MASK, WQ>(a, u >> 1);
    if (w.bad && w.j == 0 && w.g == 0 && (u & 1) == 0 && lane == 0)
      atomicOr(a.err, DEVERR_BAD_CU_SEQLENS);
    if (w.nit == 0) continue;
    if (kv_n > 0 && !warp_wait(&bars->kv_empty, (kv_n - 1) & 1u, wc)) goto out;
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars->kv_full, 8 * BOX);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tma_load_4d(smem + C::K_OFF + c * BOX, tk, &bars->kv_full, c * 64, w.g,
                    w.k_tok + w.j * BKEY, w.tma_b);
        tma_load_4d(smem + C::V_OFF + c * BOX, tv, &bars->kv_full, c * 64, w.g,
                    w.k_tok + w.j * BKEY, w.tma_b);
      }
    }
    ++kv_n;
    for (int t = 0; t < w.nit; ++t) {
      int h, i;
      bstep(a, w, t, h, i);
      if (q_n > 0 && !warp_wait(&bars->q_empty, (q_n - 1) & 1u, wc)) goto out;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->q_full, 4 * QBOX);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tma_load_4d(smem + C::Q_OFF + c * QBOX, tq, &bars->q_full, c * 64, h,
                      w.q_tok + i * WQ, w.tma_b);
      }
      ++q_n;
      if (do_n > 0 && !warp_wait(&bars->do_empty, (do_n - 1) & 1u, wc)) goto out;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->do_full, 4 * QBOX);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tma_load_4d(smem + C::DO_OFF + c * QBOX, tdo, &bars->do_full, c * 64, h,
                      w.q_tok + i * WQ, w.tma_b);
      }
      ++do_n;
      // LSE (log2 domain; rows past the sequence or with no visible key give P = 0) and D.
      if (vec_n > 0 && !warp_wait(&bars->vec_empty, (vec_n - 1) & 1u, wc)) goto out;
      const int64_t base = w.b * a.lse_sb + h * a.lse_sh + w.q_tok;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int qi = lane * 2 + e, q = i * WQ + qi;
        float l2 = INFINITY, dd = 0.f;
        if (q < w.nq) {
          const float l = a.lse[base + q];
          l2 = l == -INFINITY ? INFINITY : l * LOG2E;
          dd = a.dvec[base + q];
        }
        lse2[qi] = l2;
        dvec[qi] = dd;
      }
      __syncwarp();
      mbar_arrive(&bars->vec_full);
      ++vec_n;
    }
  }
out:
  // Teardown: the last bulk copies issued must land before the CTA may exit.
  if (lane == 0) {
    if (kv_n > 0) mbar_wait_teardown(&bars->kv_full, (kv_n - 1) & 1u, 1000000000ull);
    if (q_n > 0) mbar_wait_teardown(&bars->q_full, (q_n - 1) & 1u, 1000000000ull);
    if (do_n > 0) mbar_wait_teardown(&bars->do_full, (do_n - 1) & 1u, 1000000000ull);
  }
}

// dQ issuer of the wide kernel: per step two rounds (warpgroup 0's 32 queries, then
// warpgroup 1's), each one TMA reduce-add of the staging box (32 queries x 128 d rows).
// Deterministic order: counters per (batch, head, 64-query block, d half).
template <int MASK, bool F16>
__device__ void wide_dq_issuer(const BwdArgs &a, const CUtensorMap *tdq, uint8_t *smem,
                               BBars *bars, const WaitCtl &wc, int lane) {
  using C = WCfg;
  for (int u = blockIdx.x; u < a.num_units; u += gridDim.x) {
    const BUnit w = bunit_of<MASK, WQ>(a, u >> 1);
    const int dh = u & 1;
    if (w.skip || w.nit == 0) continue;
    const int off = w.nk - w.nq;
    for (int t = 0; t < w.nit; ++t) {
      int h, i;
      bstep(a, w, t, h, i);
      const int q0 = i * WQ;
      int *sem = a.sem ? a.sem + ((static_cast<int64_t>(w.b) * a.Hq + h) * a.qblocks + i) * 2 + dh
                       : nullptr;
      for (int x = 0; x < 2; ++x) {
        if (!warp_wait(&bars->dq_staged, static_cast<uint32_t>(x), wc)) return;
        bool ok = true;
        if (lane == 0) {
          if (sem != nullptr && x == 0) {
            int jmin = 0;
            if (mask_has_window(MASK) && a.wl >= 0) jmin = max(q0 + off - a.wl, 0) / BKEY;
            ok = wait_counter(sem, w.j - jmin, wc);
          }
          if (ok) {
            // a round wholly past the sequence's queries adds zeros: skipped
            if (q0 + 32 * x < w.nq) {
              tma_reduce_add_4d(tdq, smem + C::DQ_OFF, q0 + 32 * x, 128 * dh, h, w.b);
              bulk_commit_group();
            }
            bulk_wait_read();              // the staging box may be written again
            mbar_arrive(x == 0 ? &bars->dq_free : &bars->dq_free_r1);
            if (sem != nullptr && x == 1) {
              bulk_wait_all();             // the step's additions have been performed
              fence_proxy_async_global();
              __threadfence();
              atomicAdd(sem, 1);
            }
          }
        }
        if (!__all_sync(0xffffffffu, ok)) return;
      }
    }
  }
}

template <int MASK, bool F16>
__device__ void wide_mma(const BwdArgs &a, uint8_t *smem, BBars *bars, uint32_t tmem,
                         const WaitCtl &wc) {
  using C = WCfg;
  const uint32_t sK = smem_u32(smem + C::K_OFF), sV = smem_u32(smem + C::V_OFF);
  const uint32_t sQ = smem_u32(smem + C::Q_OFF), sDO = smem_u32(smem + C::DO_OFF);
  const uint32_t sDS = smem_u32(smem + C::DS_OFF);
  uint32_t kv_n = 0, it = 0, acc_n = 0;
  for (int u = blockIdx.x; u < a.num_units; u += gridDim.x) {
    const BUnit w = bunit_of<MASK, WQ>(a, u >> 1);
    const uint32_t dh = static_cast<uint32_t>(u & 1);
    if (w.nit == 0) continue;
    if (!warp_wait(&bars->kv_full, kv_n & 1u, wc)) goto out;
    ++kv_n;
    if (acc_n > 0 && !warp_wait(&bars->acc_empty, (acc_n - 1) & 1u, wc)) goto out;
    for (int t = 0; t < w.nit; ++t) {
      if (!warp_wait(&bars->q_full, it & 1u, wc)) goto out;
      tc_fence_after();
      wide_issue_s<F16>(tmem + W_ST, sK, sQ);                       // S^T = K Q^T
      mma_commit_w(&bars->st_full);
      if (!warp_wait(&bars->do_full, it & 1u, wc)) goto out;
      // dP^T overwrites the previous step's dQ^T: wait until the epilogue has read it.
      if (it > 0 && !warp_wait(&bars->dq_empty, (it - 1) & 1u, wc)) goto out;
      tc_fence_after();
      wide_issue_s<F16>(tmem + W_DP, sV, sDO);                      // dP^T = V dO^T
      mma_commit_w(&bars->dp_full);
      if (!warp_wait(&bars->p_ready, it & 1u, wc)) goto out;
      tc_fence_after();
      wide_issue_acc<F16>(tmem + W_DK, tmem + W_DP, sQ + 2 * dh * QBOX, t > 0);   // dK_h
      mma_commit_w(&bars->q_empty);
      wide_issue_acc<F16>(tmem + W_DV, tmem + W_ST, sDO + 2 * dh * QBOX, t > 0);  // dV_h
      mma_commit_w(&bars->do_empty);
      wide_issue_dqt<F16>(tmem + W_DP, sK + 2 * dh * BOX, sDS);                   // dQ^T_h
      mma_commit_w(&bars->dq_full);
      ++it;
    }
    mma_commit_w(&bars->kv_empty);
    mma_commit_w(&bars->acc_full);
    ++acc_n;
  }
out:
  mma_commit_w(&bars->mma_done);
  mbar_wait_teardown(&bars->mma_done, 0u, 1000000000ull);
}

// Compute warps of the wide kernel: warpgroup x = warp / 4 takes queries [32x, 32x+32) of
// every step (P^T, dS^T, and those columns of dQ^T_h) and d columns [64x, 64x+64) of the
// unit's half of dK / dV; warp w handles TMEM lanes 32 (w % 4) .. +31.
template <int MASK, bool F16>
__device__ void wide_compute(const BwdArgs &a, uint8_t *smem, BBars *bars, uint32_t tmem,
                             const WaitCtl &wc, int tid) {
  using C = WCfg;
  const int warp = tid >> 5;
  const int half = warp >> 2;
  const int r = (warp & 3) * 32 + (tid & 31);  // TMEM lane: key row, or d row of dQ^T_h
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const float *lse2 = reinterpret_cast<const float *>(smem + C::VEC_OFF);
  const float *dvec = lse2 + WQ;
  uint8_t *ds_s = smem + C::DS_OFF;
  uint8_t *stage = smem + C::DQ_OFF;
  uint32_t it = 0, acc_n = 0;
  for (int u = blockIdx.x; u < a.num_units; u += gridDim.x) {
    const BUnit w = bunit_of<MASK, WQ>(a, u >> 1);
    const int dh = u & 1;
    if (w.skip) continue;
    const int off = w.nk - w.nq;  // bottom-right alignment: query q sits at key position q + off
    const int key = w.j * BKEY + r;
    const int col0 = 128 * dh + 64 * half;  // this warp's first d column of dK / dV
    uint16_t *dkrow = reinterpret_cast<uint16_t *>(a.dk) + w.b * a.dk_sb +
                      (w.k_tok + key) * a.dk_sn + w.g * a.dk_sh + col0;
    uint16_t *dvrow = reinterpret_cast<uint16_t *>(a.dv) + w.b * a.dv_sb +
                      (w.k_tok + key) * a.dv_sn + w.g * a.dv_sh + col0;
    if (w.nit == 0) {  // no query sees these keys: zero gradients
      if (key < w.nk) {
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          if (col0 + 8 * v >= a.d) break;
          reinterpret_cast<uint4 *>(dkrow)[v] = make_uint4(0u, 0u, 0u, 0u);
          reinterpret_cast<uint4 *>(dvrow)[v] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      continue;
    }
    for (int t = 0; t < w.nit; ++t) {
      int h, i;
      bstep(a, w, t, h, i);
      const int q0 = i * WQ;
      const int qh0 = q0 + 32 * half;  // first query of this warpgroup's chunk
      const int kb = w.j * BKEY;
      bool full;  // no pair of the 128 keys x 32 queries masked
      if constexpr (MASK == MASK_NONE) {
        full = kb + BKEY <= w.nk;
      } else if constexpr (MASK == MASK_CAUSAL) {
        full = kb + BKEY <= w.nk && kb + BKEY - 1 <= qh0 + off;
      } else {
        full = kb + BKEY <= w.nk && (a.wr < 0 || kb + BKEY - 1 <= qh0 + off + a.wr) &&
               (a.wl < 0 || kb >= qh0 + 31 + off - a.wl);
      }
      // this key row's visible query positions (modifiers): key - wr - off <= q <= key + wl - off
      constexpr bool WIN = mask_has_window(MASK);
      constexpr bool SCORE_MOD = MASK == MASK_MOD || MASK == MASK_ALIBI;
      const int qv_lo = WIN && a.wr >= 0 ? key - a.wr - off : INT_MIN;
      const int qv_hi = WIN && a.wl >= 0 ? key + a.wl - off : INT_MAX;
      const bool softcap = MASK == MASK_MOD && a.sc_out != 0.f;
      const bool alibi = SCORE_MOD && a.alibi != nullptr;
      // ALiBi without a softcap on a chunk with no masked pair whose queries all sit at or
      // after its keys: the bias -slope2 (q + off - key) is linear in the query.
      const bool alibi_lin = MASK == MASK_ALIBI && full && kb + BKEY - 1 <= qh0 + off;
      const float slope2 = alibi ? a.alibi[w.b * a.alibi_sb + h] * LOG2E : 0.f;
      if (!warp_wait(&bars->vec_full, it & 1u, wc)) return;
      if (!warp_wait(&bars->st_full, it & 1u, wc)) return;
      tc_fence_after();
      {
        const int c2 = half;      // the warpgroup's 32-query chunk of the step
        const int qc = 32 * half;  // its first query
        // Phase 1, as soon as S^T has landed (dP^T may still be in the tensor core): P^T of
        // the chunk -> TMEM, packed over the first 16 of its own 32 fp32 columns (dV); P,
        // times dz/ds under a softcap, stays in registers for phase 2.
        float pd[32];
        {
          uint32_t sr[32], pp[16];
          tmem_ld_x32(tmem + lane_off + W_ST + qc, sr);
          if (MASK == MASK_ALIBI && alibi_lin) {
            // P = 2^(S c - slope2 (q + off - key) - LSE2): the bias pairs of queries (e, e+1)
            // and (e+2, e+3) step by -4 slope2 along two chains that start from exact
            // products, on packed fp32 pairs.
            const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
            const float base = -slope2 * static_cast<float>(q0 + qc + off - key);
            uint64_t w01 = f2_pack(base, base - slope2);
            uint64_t w23 = f2_pack(base - 2.f * slope2, base - 3.f * slope2);
            const uint64_t step = f2_pack(-4.f * slope2, -4.f * slope2);
#pragma unroll
            for (int e4 = 0; e4 < 32; e4 += 4) {
              const float4 l4 = *reinterpret_cast<const float4 *>(lse2 + qc + e4);
              float z0, z1, z2, z3;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e4]), __uint_as_float(sr[e4 + 1])),
                               sc2, f2_add(w01, f2_pack(-l4.x, -l4.y))), z0, z1);
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e4 + 2]), __uint_as_float(sr[e4 + 3])),
                               sc2, f2_add(w23, f2_pack(-l4.z, -l4.w))), z2, z3);
              w01 = f2_add(w01, step);
              w23 = f2_add(w23, step);
              pd[e4] = ex2_approx(z0);
              pd[e4 + 1] = ex2_approx(z1);
              pd[e4 + 2] = ex2_approx(z2);
              pd[e4 + 3] = ex2_approx(z3);
              pp[e4 / 2] = pack2<F16>(pd[e4], pd[e4 + 1]);
              pp[e4 / 2 + 1] = pack2<F16>(pd[e4 + 2], pd[e4 + 3]);
            }
          } else if (!SCORE_MOD && full) {
            // No masked pair and no modifier: P = 2^(S c - LSE2) on packed fp32 pairs.
            const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
#pragma unroll
            for (int e4 = 0; e4 < 32; e4 += 4) {
              const float4 l4 = *reinterpret_cast<const float4 *>(lse2 + qc + e4);
              float z0, z1, z2, z3;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e4]), __uint_as_float(sr[e4 + 1])),
                               sc2, f2_pack(-l4.x, -l4.y)), z0, z1);
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e4 + 2]), __uint_as_float(sr[e4 + 3])),
                               sc2, f2_pack(-l4.z, -l4.w)), z2, z3);
              pd[e4] = ex2_approx(z0);
              pd[e4 + 1] = ex2_approx(z1);
              pd[e4 + 2] = ex2_approx(z2);
              pd[e4 + 3] = ex2_approx(z3);
              pp[e4 / 2] = pack2<F16>(pd[e4], pd[e4 + 1]);
              pp[e4 / 2 + 1] = pack2<F16>(pd[e4 + 2], pd[e4 + 3]);
            }
          } else {
#pragma unroll
            for (int e2 = 0; e2 < 32; e2 += 2) {
              float p[2];
#pragma unroll
              for (int x = 0; x < 2; ++x) {
                const int qi = qc + e2 + x;
                const float sv = __uint_as_float(sr[e2 + x]);
                float z2, dz = 1.f;  // score in log2 units and dz/ds
                if constexpr (SCORE_MOD) {
                  if (softcap) {
                    const float t = tanh_ex2(sv * a.sc_in);
                    z2 = t * a.sc_out;
                    dz = 1.f - t * t;
                  } else {
                    z2 = sv * a.scale_log2;
                  }
                  if (alibi) z2 = fmaf(-slope2, fabsf(static_cast<float>(q0 + qi + off - key)), z2);
                } else {
                  z2 = sv * a.scale_log2;
                }
                bool vis;
                if constexpr (WIN)
                  vis = full || (key < w.nk && q0 + qi >= qv_lo && q0 + qi <= qv_hi);
                else
                  vis = full || (key < w.nk && (MASK == MASK_NONE || key <= q0 + qi + off));
                const float pv = ex2_approx(z2 - lse2[qi]);
                p[x] = vis ? pv : 0.f;
                pd[e2 + x] = p[x] * dz;
              }
              pp[e2 / 2] = pack2<F16>(p[0], p[1]);
            }
          }
          tmem_st_x16(tmem + lane_off + W_ST + qc, pp);
        }
        // Phase 2, once dP^T has landed: dS^T = P^T (dP^T - D) -> TMEM, packed over the first
        // 16 of the chunk's dP^T columns (dK), and dS -> shared memory, queries contiguous.
        if (!warp_wait(&bars->dp_full, it & 1u, wc)) return;
        tc_fence_after();
        uint32_t dr[32], dd[16];
        tmem_ld_x32(tmem + lane_off + W_DP + qc, dr);
#pragma unroll
        for (int e4 = 0; e4 < 32; e4 += 4) {
          const float4 d4 = *reinterpret_cast<const float4 *>(dvec + qc + e4);
          float e0, e1, e2, e3;
          f2_unpack(f2_mul(f2_pack(pd[e4], pd[e4 + 1]),
                           f2_add(f2_pack(__uint_as_float(dr[e4]), __uint_as_float(dr[e4 + 1])),
                                  f2_pack(-d4.x, -d4.y))), e0, e1);
          f2_unpack(f2_mul(f2_pack(pd[e4 + 2], pd[e4 + 3]),
                           f2_add(f2_pack(__uint_as_float(dr[e4 + 2]), __uint_as_float(dr[e4 + 3])),
                                  f2_pack(-d4.z, -d4.w))), e2, e3);
          dd[e4 / 2] = pack2<F16>(e0, e1);
          dd[e4 / 2 + 1] = pack2<F16>(e2, e3);
        }
        tmem_st_x16(tmem + lane_off + W_DP + qc, dd);
        uint8_t *box = ds_s + r * 128;  // [128 keys x 64 queries]: this chunk's 64 bytes
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
          const int gran = c2 * 4 + gi;
          *reinterpret_cast<uint4 *>(box + ((gran ^ (r & 7)) << 4)) =
              make_uint4(dd[4 * gi], dd[4 * gi + 1], dd[4 * gi + 2], dd[4 * gi + 3]);
        }
      }
      mbar_arrive(&bars->vec_empty);
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_ready);
      // dQ^T_h epilogue: this warpgroup's 32 query columns (thread = d row) through the
      // staging box, warpgroup 0 first; the reduce-add is the dQ issuer's.  Unordered dQ:
      // warpgroup 0's wait for the previous round's read (complete by now) is polled here,
      // ahead of the staging stores that would queue before it in the shared-memory pipe.
      const bool early = half == 0 && a.sem == nullptr && it > 0;
      if (early && !warp_wait(&bars->dq_free_r1, (it - 1) & 1u, wc)) return;
      if (!warp_wait(&bars->dq_full, it & 1u, wc)) return;
      tc_fence_after();
      uint32_t qv[32];
      tmem_ld_x32(tmem + lane_off + W_DP + 32 * half, qv);
      tc_fence_before();
      mbar_arrive(&bars->dq_empty);
      // The box is free once the issuer has read the round before this one: warpgroup 0's
      // round follows the previous step's second round (dq_free_r1, one completion per
      // step), warpgroup 1's this step's first (dq_free, one per step).  One barrier per
      // round keeps every wait within one phase of its barrier: warpgroup 1 can reach its
      // next round before the issuer has read its last one.
      if (half == 0 ? !early && it > 0 && !warp_wait(&bars->dq_free_r1, (it - 1) & 1u, wc)
                    : !warp_wait(&bars->dq_free, it & 1u, wc))
        return;
      wide_stage_dqt(stage, r, qv);
      fence_proxy_async_smem();
      mbar_arrive(&bars->dq_staged);
      ++it;
    }
    // Unit end: dV_h and scale * dK_h of this key row (this warp's 64 d columns) -> global.
    if (!warp_wait(&bars->acc_full, acc_n & 1u, wc)) return;
    tc_fence_after();
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
      const uint32_t cc = static_cast<uint32_t>(64 * half + 32 * c2);
      uint32_t vr[32], kr[32];
      tmem_ld_x32(tmem + lane_off + W_DV + cc, vr);
      tmem_ld_x32(tmem + lane_off + W_DK + cc, kr);
      if (key < w.nk) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          if (col0 + 32 * c2 + 8 * v >= a.d) break;  // columns past d are padding
          uint4 wv, wk;
          wv.x = pack2<F16>(__uint_as_float(vr[8 * v + 0]), __uint_as_float(vr[8 * v + 1]));
          wv.y = pack2<F16>(__uint_as_float(vr[8 * v + 2]), __uint_as_float(vr[8 * v + 3]));
          wv.z = pack2<F16>(__uint_as_float(vr[8 * v + 4]), __uint_as_float(vr[8 * v + 5]));
          wv.w = pack2<F16>(__uint_as_float(vr[8 * v + 6]), __uint_as_float(vr[8 * v + 7]));
          wk.x = pack2<F16>(__uint_as_float(kr[8 * v + 0]) * a.scale, __uint_as_float(kr[8 * v + 1]) * a.scale);
          wk.y = pack2<F16>(__uint_as_float(kr[8 * v + 2]) * a.scale, __uint_as_float(kr[8 * v + 3]) * a.scale);
          wk.z = pack2<F16>(__uint_as_float(kr[8 * v + 4]) * a.scale, __uint_as_float(kr[8 * v + 5]) * a.scale);
          wk.w = pack2<F16>(__uint_as_float(kr[8 * v + 6]) * a.scale, __uint_as_float(kr[8 * v + 7]) * a.scale);
          reinterpret_cast<uint4 *>(dvrow + 32 * c2)[v] = wv;
          reinterpret_cast<uint4 *>(dkrow + 32 * c2)[v] = wk;
        }
      }
    }
    tc_fence_before();
    mbar_arrive(&bars->acc_empty);
    ++acc_n;
  }
}

template <int MASK, bool F16>
__global__ void __launch_bounds__(NTHREADS, 1)
    bwd_wide_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const __grid_constant__ CUtensorMap tdq, const BwdArgs a) {
  using C = WCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  BBars *bars = reinterpret_cast<BBars *>(smem + C::BAR_OFF);
  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    mbar_init(&bars->do_full, 1);
    mbar_init(&bars->do_empty, 1);
    mbar_init(&bars->vec_full, 32);
    mbar_init(&bars->vec_empty, NCOMPUTE);
    mbar_init(&bars->st_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_ready, NCOMPUTE);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_empty, NCOMPUTE);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, NCOMPUTE);
    mbar_init(&bars->mma_done, 1);
    mbar_init(&bars->dq_staged, NCOMPUTE / 2);
    mbar_init(&bars->dq_free, 1);
    mbar_init(&bars->dq_free_r1, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&tdo);
    tma_prefetch_desc(&tdq);
  }
  if (warp == MMA_WARP) {
    tmem_alloc(&bars->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort, a.err, a.timeout_ns, DEVERR_BWD_TIMEOUT};
  if (warp < PRODUCER_WARP) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(COMPUTE_REGS));
    wide_compute<MASK, F16>(a, smem, bars, tmem, wc, tid);
    __syncwarp();
    tc_fence_before();
    named_barrier(1, NTHREADS);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(OTHER_REGS));
    if (warp == PRODUCER_WARP) {
      wide_producer<MASK, F16>(a, &tq, &tk, &tv, &tdo, smem, bars, wc, lane);
    } else if (warp == MMA_WARP) {
      wide_mma<MASK, F16>(a, smem, bars, tmem, wc);
    } else if (warp == DQ_WARP) {
      wide_dq_issuer<MASK, F16>(a, &tdq, smem, bars, wc, lane);
      if (lane == 0) bulk_wait_all();  // every dQ reduction has landed
    }
    __syncwarp();
    tc_fence_before();
    named_barrier(1, NTHREADS);
    if (warp == MMA_WARP) {
      tc_fence_after();
      tmem_dealloc(tmem, TMEM_COLS);
    }
  }
}

// ------------------------------------------------------------------------------------
// Preprocessing: D = rowsum(dO * O) (one warp per row), a zeroed dQ accumulator (acc_n
// floats, a multiple of 4) and zeroed counters.

template <bool F16>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint16_t *o, const uint16_t *dout,
                                                      int B, int Nq, int Hq, int d, int64_t os0,
                                                      int64_t os1, int64_t os2, int64_t ds0,
                                                      int64_t ds1, int64_t ds2, float *dvec,
                                                      float *dq_acc, int64_t acc_n, int *sem,
                                                      int nsem) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < nsem; t += gridDim.x * blockDim.x)
    sem[t] = 0;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < acc_n / 4;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x)
    reinterpret_cast<float4 *>(dq_acc)[t] = make_float4(0.f, 0.f, 0.f, 0.f);
  const int lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(B) * Nq * Hq;
  for (int64_t rw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32; rw < rows;
       rw += static_cast<int64_t>(gridDim.x) * blockDim.x / 32) {
    const int h = static_cast<int>(rw % Hq);
    const int64_t bn = rw / Hq;
    const int n = static_cast<int>(bn % Nq);
    const int b = static_cast<int>(bn / Nq);
    const uint16_t *orow = o + b * os0 + n * os1 + h * os2;
    const uint16_t *drow = dout + b * ds0 + n * ds1 + h * ds2;
    float acc = 0.f;
    for (int c = lane * 2; c < d; c += 64) {
      const uint32_t ov = *reinterpret_cast<const uint32_t *>(orow + c);
      const uint32_t dv = *reinterpret_cast<const uint32_t *>(drow + c);
      acc = fmaf(lo_to_f32<F16>(ov), lo_to_f32<F16>(dv), acc);
      acc = fmaf(hi_to_f32<F16>(ov), hi_to_f32<F16>(dv), acc);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) dvec[(static_cast<int64_t>(b) * Hq + h) * Nq + n] = acc;
  }
}

// The same with 16-byte loads (O and dO rows 16-byte aligned): 2^lpr_log2 lanes per row,
// 8 elements per lane and load, 32 >> lpr_log2 rows per warp at a time, the row's partial
// sums reduced within its lane group.  Four bytes per lane and load left too few loads in
// flight to stream O and dO at the copy rate.
template <bool F16>
__global__ void __launch_bounds__(256) bwd_pre_vec_kernel(const uint16_t *o, const uint16_t *dout,
                                                          int B, int Nq, int Hq, int d,
                                                          int64_t os0, int64_t os1, int64_t os2,
                                                          int64_t ds0, int64_t ds1, int64_t ds2,
                                                          float *dvec, float *dq_acc,
                                                          int64_t acc_n, int *sem, int nsem,
                                                          int lpr_log2) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < nsem; t += gridDim.x * blockDim.x)
    sem[t] = 0;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < acc_n / 4;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x)
    reinterpret_cast<float4 *>(dq_acc)[t] = make_float4(0.f, 0.f, 0.f, 0.f);
  const int lane = threadIdx.x & 31;
  const int lpr = 1 << lpr_log2;
  const int sub = lane & (lpr - 1);
  const int rpw = 32 >> lpr_log2;
  const int64_t rows = static_cast<int64_t>(B) * Nq * Hq;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * blockDim.x / 32;
  for (int64_t base = warp0 * rpw; base < rows; base += nwarps * rpw) {
    const int64_t rw = base + (lane >> lpr_log2);
    float acc = 0.f;
    int b = 0, n = 0, h = 0;
    if (rw < rows) {
      h = static_cast<int>(rw % Hq);
      const int64_t bn = rw / Hq;
      n = static_cast<int>(bn % Nq);
      b = static_cast<int>(bn / Nq);
      const uint16_t *orow = o + b * os0 + n * os1 + h * os2;
      const uint16_t *drow = dout + b * ds0 + n * ds1 + h * ds2;
      for (int c = sub * 8; c < d; c += lpr * 8) {
        const uint4 ov = *reinterpret_cast<const uint4 *>(orow + c);
        const uint4 dv = *reinterpret_cast<const uint4 *>(drow + c);
        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc = fmaf(lo_to_f32<F16>(ow[i]), lo_to_f32<F16>(dw[i]), acc);
          acc = fmaf(hi_to_f32<F16>(ow[i]), hi_to_f32<F16>(dw[i]), acc);
        }
      }
    }
    for (int s2 = lpr >> 1; s2 > 0; s2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s2);
    if (rw < rows && sub == 0) dvec[(static_cast<int64_t>(b) * Hq + h) * Nq + n] = acc;
  }
}

// dQ = scale * accumulator, 8 elements per thread.
template <bool F16>
__global__ void __launch_bounds__(256) bwd_post_kernel(const float *acc, float scale, uint16_t *dq,
                                                       int B, int Nq, int Hq, int d, int64_t s0,
                                                       int64_t s1, int64_t s2) {
  const int64_t total = static_cast<int64_t>(B) * Nq * Hq * (d / 8);
  for (int64_t x = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; x < total;
       x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c8 = static_cast<int>(x % (d / 8));
    const int64_t row = x / (d / 8);  // (b, n, h)
    const int h = static_cast<int>(row % Hq);
    const int64_t bn = row / Hq;
    const int n = static_cast<int>(bn % Nq);
    const int b = static_cast<int>(bn / Nq);
    const float4 v0 = reinterpret_cast<const float4 *>(acc + row * d)[2 * c8];
    const float4 v1 = reinterpret_cast<const float4 *>(acc + row * d)[2 * c8 + 1];
    uint4 w;
    w.x = pack2<F16>(v0.x * scale, v0.y * scale);
    w.y = pack2<F16>(v0.z * scale, v0.w * scale);
    w.z = pack2<F16>(v1.x * scale, v1.y * scale);
    w.w = pack2<F16>(v1.z * scale, v1.w * scale);
    *reinterpret_cast<uint4 *>(dq + b * s0 + n * s1 + h * s2 + c8 * 8) = w;
  }
}

// Wide kernel: dQ = scale * the transposed accumulator [B, Hq, d, nq_pad], 8 d columns of
// one query row per thread (queries fastest across threads: coalesced reads).  Varlen
// (cu_q non-null): B sequences of at most Nq queries, row n of sequence b is token
// cu_q[b] + n of the packed dq.
template <bool F16>
__global__ void __launch_bounds__(256) bwd_post_t_kernel(const float *acc, float scale,
                                                         uint16_t *dq, int B, int Nq, int nq_pad,
                                                         int Hq, int d, int64_t s0, int64_t s1,
                                                         int64_t s2, const int *cu_q,
                                                         int total_q) {
  const int64_t total = static_cast<int64_t>(B) * Hq * (d / 8) * Nq;
  for (int64_t x = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; x < total;
       x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(x % Nq);
    int64_t rest = x / Nq;
    const int c8 = static_cast<int>(rest % (d / 8));
    rest /= d / 8;
    const int h = static_cast<int>(rest % Hq);
    const int b = static_cast<int>(rest / Hq);
    int64_t row = n, bo = b;
    if (cu_q != nullptr) {
      const int q0 = cu_q[b], q1 = cu_q[b + 1];
      if (q0 < 0 || q1 < q0 || q1 > total_q || n >= q1 - q0) continue;
      row = q0 + n;
      bo = 0;
    }
    const float *src = acc + ((static_cast<int64_t>(b) * Hq + h) * d + 8 * c8) * nq_pad + n;
    uint4 w;
    w.x = pack2<F16>(src[0] * scale, src[nq_pad] * scale);
    w.y = pack2<F16>(src[2 * nq_pad] * scale, src[3 * nq_pad] * scale);
    w.z = pack2<F16>(src[4 * nq_pad] * scale, src[5 * nq_pad] * scale);
    w.w = pack2<F16>(src[6 * nq_pad] * scale, src[7 * nq_pad] * scale);
    *reinterpret_cast<uint4 *>(dq + bo * s0 + row * s1 + h * s2 + c8 * 8) = w;
  }
}

__global__ void zero16_kernel(uint16_t *x, int B, int N, int H, int d, int64_t s0, int64_t s1,
                              int64_t s2) {
  const int64_t total = static_cast<int64_t>(B) * N * H * (d / 8);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c8 = static_cast<int>(t % (d / 8));
    const int64_t row = t / (d / 8);
    const int h = static_cast<int>(row % H);
    const int64_t bn = row / H;
    const int n = static_cast<int>(bn % N);
    const int b = static_cast<int>(bn / N);
    *reinterpret_cast<uint4 *>(x + b * s0 + n * s1 + h * s2 + c8 * 8) = make_uint4(0u, 0u, 0u, 0u);
  }
}

int grid_for(int64_t items, int threads) {
  const int64_t g = (items + threads - 1) / threads;
  return static_cast<int>(g < 1 ? 1 : (g > 8192 ? 8192 : g));
}

template <int D, int MASK, bool F16>
cudaError_t launch_bwd_impl(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const CUtensorMap &tdo, const CUtensorMap &tdq, const BwdArgs &a,
                            int grid, cudaStream_t stream) {
  constexpr int smem = BCfg<D, F16>::SMEM_BYTES;
  static_assert(smem <= 232448, "backward kernel shared memory");
  if (a.sem != nullptr) {
    cudaError_t e = cudaFuncSetAttribute(bwd_kernel<D, MASK, F16, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    bwd_kernel<D, MASK, F16, true><<<grid, NB_THREADS, smem, stream>>>(tq, tk, tv, tdo, tdq, a);
  } else {
    cudaError_t e = cudaFuncSetAttribute(bwd_kernel<D, MASK, F16, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    bwd_kernel<D, MASK, F16, false><<<grid, NB_THREADS, smem, stream>>>(tq, tk, tv, tdo, tdq, a);
  }
  return cudaGetLastError();
}

template <int MASK, bool F16>
cudaError_t launch_wide_impl(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                             const CUtensorMap &tdo, const CUtensorMap &tdq, const BwdArgs &a,
                             int grid, cudaStream_t stream) {
  constexpr int smem = WCfg::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(bwd_wide_kernel<MASK, F16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  bwd_wide_kernel<MASK, F16><<<grid, NTHREADS, smem, stream>>>(tq, tk, tv, tdo, tdq, a);
  return cudaGetLastError();
}

template <bool F16>
cudaError_t launch_wide(int mask, const CUtensorMap &tq, const CUtensorMap &tk,
                        const CUtensorMap &tv, const CUtensorMap &tdo, const CUtensorMap &tdq,
                        const BwdArgs &a, int grid, cudaStream_t stream) {
  switch (mask) {
    case MASK_NONE: return launch_wide_impl<MASK_NONE, F16>(tq, tk, tv, tdo, tdq, a, grid, stream);
    case MASK_CAUSAL:
      return launch_wide_impl<MASK_CAUSAL, F16>(tq, tk, tv, tdo, tdq, a, grid, stream);
    case MASK_WINDOW:
      return launch_wide_impl<MASK_WINDOW, F16>(tq, tk, tv, tdo, tdq, a, grid, stream);
    case MASK_ALIBI:
      return launch_wide_impl<MASK_ALIBI, F16>(tq, tk, tv, tdo, tdq, a, grid, stream);
    default: return launch_wide_impl<MASK_MOD, F16>(tq, tk, tv, tdo, tdq, a, grid, stream);
  }
}

template <int D, bool F16>
cudaError_t launch_bwd_d(int mask, const CUtensorMap &tq, const CUtensorMap &tk,
                         const CUtensorMap &tv, const CUtensorMap &tdo, const CUtensorMap &tdq,
                         const BwdArgs &a, int grid, cudaStream_t stream) {
  switch (mask) {
    case MASK_NONE: return launch_bwd_impl<D, MASK_NONE, F16>(tq, tk, tv, tdo, tdq, a, grid, stream);
    case MASK_CAUSAL:
      return launch_bwd_impl<D, MASK_CAUSAL, F16>(tq, tk, tv, tdo, tdq, a, grid, stream);
    case MASK_WINDOW:
      return launch_bwd_impl<D, MASK_WINDOW, F16>(tq, tk, tv, tdo, tdq, a, grid, stream);
    case MASK_ALIBI:
      return launch_bwd_impl<D, MASK_ALIBI, F16>(tq, tk, tv, tdo, tdq, a, grid, stream);
    default: return launch_bwd_impl<D, MASK_MOD, F16>(tq, tk, tv, tdo, tdq, a, grid, stream);
  }
}

}  // namespace

cudaError_t launch_bwd(int d, int mask, bool f16, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &tdo, const CUtensorMap &tdq,
                       const BwdArgs &a, int grid, cudaStream_t stream) {
  if (d == 256)
    return f16 ? launch_wide<true>(mask, tq, tk, tv, tdo, tdq, a, grid, stream)
               : launch_wide<false>(mask, tq, tk, tv, tdo, tdq, a, grid, stream);
  if (d == 64)
    return f16 ? launch_bwd_d<64, true>(mask, tq, tk, tv, tdo, tdq, a, grid, stream)
               : launch_bwd_d<64, false>(mask, tq, tk, tv, tdo, tdq, a, grid, stream);
  return f16 ? launch_bwd_d<128, true>(mask, tq, tk, tv, tdo, tdq, a, grid, stream)
             : launch_bwd_d<128, false>(mask, tq, tk, tv, tdo, tdq, a, grid, stream);
}

cudaError_t launch_bwd_pre(int d, bool f16, const void *o, const void *dout, int B, int Nq,
                           int Hq, const int64_t o_st[3], const int64_t do_st[3], float *dvec,
                           float *dq_acc, int64_t acc_n, int *sem, int nsem, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(B) * Nq * Hq;
  if (rows == 0 && acc_n == 0) return cudaSuccess;
  const int64_t items = rows * 32 > acc_n / 4 ? rows * 32 : acc_n / 4;
  const int grid = grid_for(items > nsem ? items : nsem, 256);
  const uint16_t *op = reinterpret_cast<const uint16_t *>(o);
  const uint16_t *dp = reinterpret_cast<const uint16_t *>(dout);
  const bool vec = reinterpret_cast<uintptr_t>(o) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(dout) % 16 == 0 && d % 8 == 0 && d <= 256 &&
                   o_st[0] % 8 == 0 && o_st[1] % 8 == 0 && o_st[2] % 8 == 0 &&
                   do_st[0] % 8 == 0 && do_st[1] % 8 == 0 && do_st[2] % 8 == 0;
  if (vec) {
    int lpr_log2 = 0;
    while ((8 << lpr_log2) < d) ++lpr_log2;  // lanes per row: d / 8 rounded up to a power of 2
    auto vk = f16 ? bwd_pre_vec_kernel<true> : bwd_pre_vec_kernel<false>;
    vk<<<grid, 256, 0, stream>>>(op, dp, B, Nq, Hq, d, o_st[0], o_st[1], o_st[2], do_st[0],
                                 do_st[1], do_st[2], dvec, dq_acc, acc_n, sem, nsem, lpr_log2);
    return cudaGetLastError();
  }
  auto kern = f16 ? bwd_pre_kernel<true> : bwd_pre_kernel<false>;
  kern<<<grid, 256, 0, stream>>>(op, dp, B, Nq, Hq, d, o_st[0], o_st[1], o_st[2], do_st[0],
                                 do_st[1], do_st[2], dvec, dq_acc, acc_n, sem, nsem);
  return cudaGetLastError();
}

cudaError_t launch_bwd_post(int d, bool f16, const float *dq_acc, float scale, void *dq, int B,
                            int Nq, int Hq, const int64_t dq_st[3], cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(B) * Nq * Hq * (d / 8);
  if (items == 0) return cudaSuccess;
  uint16_t *out = reinterpret_cast<uint16_t *>(dq);
  if (f16)
    bwd_post_kernel<true><<<grid_for(items, 256), 256, 0, stream>>>(dq_acc, scale, out, B, Nq,
                                                                    Hq, d, dq_st[0], dq_st[1],
                                                                    dq_st[2]);
  else
    bwd_post_kernel<false><<<grid_for(items, 256), 256, 0, stream>>>(dq_acc, scale, out, B, Nq,
                                                                     Hq, d, dq_st[0], dq_st[1],
                                                                     dq_st[2]);
  return cudaGetLastError();
}

cudaError_t launch_bwd_post_t(int d, bool f16, const float *dq_acc, float scale, void *dq, int B,
                              int Nq, int nq_pad, int Hq, const int64_t dq_st[3],
                              const int *cu_q, int total_q, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(B) * Nq * Hq * (d / 8);
  if (items == 0) return cudaSuccess;
  uint16_t *out = reinterpret_cast<uint16_t *>(dq);
  if (f16)
    bwd_post_t_kernel<true><<<grid_for(items, 256), 256, 0, stream>>>(
        dq_acc, scale, out, B, Nq, nq_pad, Hq, d, dq_st[0], dq_st[1], dq_st[2], cu_q, total_q);
  else
    bwd_post_t_kernel<false><<<grid_for(items, 256), 256, 0, stream>>>(
        dq_acc, scale, out, B, Nq, nq_pad, Hq, d, dq_st[0], dq_st[1], dq_st[2], cu_q, total_q);
  return cudaGetLastError();
}

cudaError_t launch_zero16(void *x, int B, int N, int H, int d, const int64_t st[3],
                          cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(B) * N * H * (d / 8);
  if (items == 0) return cudaSuccess;
  zero16_kernel<<<grid_for(items, 256), 256, 0, stream>>>(reinterpret_cast<uint16_t *>(x), B, N,
                                                          H, d, st[0], st[1], st[2]);
  return cudaGetLastError();
}

}  // namespace fa
