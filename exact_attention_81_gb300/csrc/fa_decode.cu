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
//   * 8 compute warps evaluate the G = Hq/Hkv query heads of the group together:
//       scores   thread = (key, 1/TPK of d), q of its slice in registers, TPK-lane reduce;
//       softmax  warp g < G owns head g: block max, running (m, l), p = 2^(s - m);
//       P V      thread = (4 consecutive d, one of NSL key slices), fp32 accumulators
//                rescaled by 2^(m_old - m_new) per block (online softmax within a unit);
//   * each unit writes O_s / l_s (fp32) and LSE_s = ln2 (m + log2 l) to the workspace.
// Only rows below cache_seqlens[b] are used: a block's tail rows are masked to -inf in the
// scores and skipped in P V, so values past the visible prefix never enter the result.
//
// The combine kernel merges the partials of each (b, query head):
//   LSE = log sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s.
#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int KB = 128;           // keys per block (one TMA tile per d-box)
constexpr int NCOMPUTE = 256;     // compute threads (warps 0-7)
constexpr int NTHREADS = NCOMPUTE + 32;
constexpr int PRODUCER_WARP = 8;
constexpr int BOX_BYTES = KB * 128;
constexpr float LN2 = 0.6931471805599453f;

__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }
__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

template <int D, int G>
struct DCfg {
  static constexpr int KCH = D / 64;
  static constexpr int BLOCK_BYTES = KCH * BOX_BYTES;         // one K or V block
  static constexpr int TPK = cmax(4, G * D / 128);             // threads per key (scores)
  static constexpr int DP = D / TPK;                           // d elements per thread
  static constexpr int KPP = NCOMPUTE / TPK;                   // keys per pass
  static constexpr int NPASS = KB / KPP;
  static constexpr int DQ = D / 4;                             // d quads
  static constexpr int NSL = NCOMPUTE / DQ;                    // key slices in P V
  static constexpr int SBUF_BYTES = 2 * KB * G * 4;            // double-buffered scores
  static constexpr int RED_BYTES = NSL * G * D * 4;            // cross-slice reduction
  static constexpr int MISC_BYTES = 1024;                      // alpha, (m,l), barriers
  static constexpr int BUDGET = 227 * 1024 - 1024;             // minus alignment slack
  static constexpr int NSLOTS =
      cmin(12, (BUDGET - SBUF_BYTES - RED_BYTES - MISC_BYTES) / BLOCK_BYTES);
  static constexpr int RING_OFF = 0;
  static constexpr int SBUF_OFF = NSLOTS * BLOCK_BYTES;
  static constexpr int RED_OFF = SBUF_OFF + SBUF_BYTES;
  static constexpr int MISC_OFF = RED_OFF + RED_BYTES;
  static constexpr int SMEM_BYTES = MISC_OFF + MISC_BYTES + 1024;
  static_assert(NSLOTS >= 2, "ring too small");
  static_assert(KB % KPP == 0, "keys per pass must divide the block");
  static_assert(TPK <= 32 && (32 % TPK) == 0, "threads per key must tile a warp");
  static_assert(DP % 8 == 0, "each thread reads whole 16-byte chunks");
};

struct DBars {
  uint64_t full[12], empty[12];
  uint64_t sync;  // group barrier of the 256 compute threads (bounded wait)
  float alpha[2][8];
  float m[8], l[8];
  int abort;
};

struct Unit {
  int b, g, c, len, key0, nkeys;
};

__device__ __forceinline__ Unit unit_of(const DecodeArgs &a, int u) {
  Unit w;
  const int bg = a.B * a.Hkv;
  w.c = u / bg;
  const int r = u - w.c * bg;
  w.b = r / a.Hkv;
  w.g = r - w.b * a.Hkv;
  const int len_raw = a.cache_len[w.b];
  w.len = min(max(len_raw, 0), a.Lmax);
  w.key0 = w.c * a.chunk;
  w.nkeys = min(a.chunk, w.len - w.key0);  // <= 0: nothing to do
  return w;
}

template <int D, int G>
__device__ void producer(const DecodeArgs &a, const CUtensorMap *tmk, const CUtensorMap *tmv,
                         uint8_t *smem, DBars *bars, const WaitCtl &wc) {
  using C = DCfg<D, G>;
  uint32_t it = 0;
  const uint64_t policy = policy_evict_first();  // every cache byte is read once
  for (int u = blockIdx.x; u < a.num_units; u += gridDim.x) {
    const Unit w = unit_of(a, u);
    if (w.c == 0 && w.g == 0) {
      const int len_raw = a.cache_len[w.b];
      if (len_raw < 0 || len_raw > a.Lmax) atomicOr(a.err, DEVERR_BAD_CACHE_LEN);
    }
    if (w.nkeys <= 0) continue;
    const int nblk = (w.nkeys + KB - 1) / KB;
    for (int blk = 0; blk < nblk; ++blk) {
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const int slot = static_cast<int>(it % C::NSLOTS);
        const uint32_t use = it / C::NSLOTS;
        if (!mbar_wait(&bars->empty[slot], (use & 1u) ^ 1u, wc)) goto out;
        mbar_arrive_expect_tx(&bars->full[slot], C::BLOCK_BYTES);
#pragma unroll
        for (int cc = 0; cc < C::KCH; ++cc)
          tma_load_4d_hint(smem + C::RING_OFF + slot * C::BLOCK_BYTES + cc * BOX_BYTES,
                           which ? tmv : tmk, &bars->full[slot], cc * 64, w.g, w.key0 + blk * KB,
                           w.b, policy);
        ++it;
      }
    }
  }
out:
  for (int s = 0; s < C::NSLOTS; ++s) {
    if (it > static_cast<uint32_t>(s)) {
      const uint32_t uses = (it - 1 - s) / C::NSLOTS + 1;
      mbar_wait_teardown(&bars->full[s], (uses - 1) & 1u, 1000000000ull);
    }
  }
}

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const WaitCtl &wc) {
  const bool ok = mbar_wait(bar, parity, wc);
  return __all_sync(0xffffffffu, ok);
}

// Barrier among the 256 compute threads.  Built on an mbarrier rather than bar.sync so
// that the wait is bounded: a warp that has given up never leaves the others blocked.
__device__ __forceinline__ bool group_sync(uint64_t *bar, uint32_t &phase, const WaitCtl &wc) {
  mbar_arrive(bar);
  const bool ok = warp_wait(bar, phase, wc);
  phase ^= 1u;
  return ok;
}

// Releases a ring slot: one arrival per compute warp (count 8).
__device__ __forceinline__ void release(uint64_t *bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

template <int D, int G>
__device__ void compute(const DecodeArgs &a, uint8_t *smem, DBars *bars, const WaitCtl &wc,
                        int tid) {
  using C = DCfg<D, G>;
  const int warp = tid >> 5, lane = tid & 31;
  // scores mapping
  const int kl = tid / C::TPK, part = tid % C::TPK;
  const int d0 = part * C::DP;                 // first d of this thread's slice
  const int sbox = d0 / 64;                    // box holding the slice
  const int schunk0 = (d0 % 64) / 8;           // first 16-byte chunk in the 128-byte row
  // P V mapping
  const int dq = tid % C::DQ, ks = tid / C::DQ;
  const int vbox = (4 * dq) / 64;
  const int vbyte = ((4 * dq) % 64) * 2;
  const int vchunk = vbyte / 16, vhalf = (vbyte % 16) / 8;

  float *sbuf = reinterpret_cast<float *>(smem + C::SBUF_OFF);
  float *red = reinterpret_cast<float *>(smem + C::RED_OFF);
  const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(a.q);
  uint32_t it = 0, nblk_done = 0, sync_phase = 0;

  for (int u = blockIdx.x; u < a.num_units; u += gridDim.x) {
    const Unit w = unit_of(a, u);
    if (w.nkeys <= 0) continue;
    const int nblk = (w.nkeys + KB - 1) / KB;

    // q slice of the G heads of group g, pre-scaled into the log2 domain.
    float qr[G][C::DP];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          qg + (static_cast<int64_t>(w.b) * a.Hq + w.g * G + gg) * D + d0);
#pragma unroll
      for (int v = 0; v < C::DP / 8; ++v) {
        const uint4 x = src[v];
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          qr[gg][8 * v + 2 * e] = bf16lo_to_f32(xs[e]) * a.scale_log2;
          qr[gg][8 * v + 2 * e + 1] = bf16hi_to_f32(xs[e]) * a.scale_log2;
        }
      }
    }
    float acc[G][4];
#pragma unroll
    for (int gg = 0; gg < G; ++gg)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[gg][i] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;  // meaningful in warp `warp` < G (head = warp)

    for (int blk = 0; blk < nblk; ++blk) {
      const int nvalid = min(KB, w.nkeys - blk * KB);
      float *sb = sbuf + (nblk_done & 1u) * (KB * G);
      // ---- scores from the K block
      {
        const int slot = static_cast<int>(it % C::NSLOTS);
        if (!warp_wait(&bars->full[slot], (it / C::NSLOTS) & 1u, wc)) return;
        ++it;
        const uint8_t *kblk = smem + C::RING_OFF + slot * C::BLOCK_BYTES + sbox * BOX_BYTES;
#pragma unroll
        for (int pass = 0; pass < C::NPASS; ++pass) {
          const int key = pass * C::KPP + kl;
          const uint8_t *krow = kblk + key * 128;
          float part_s[G];
#pragma unroll
          for (int gg = 0; gg < G; ++gg) part_s[gg] = 0.f;
#pragma unroll
          for (int v = 0; v < C::DP / 8; ++v) {
            const int phys = (schunk0 + v) ^ (key & 7);
            const uint4 x = *reinterpret_cast<const uint4 *>(krow + phys * 16);
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float k0 = bf16lo_to_f32(xs[e]);
              const float k1 = bf16hi_to_f32(xs[e]);
#pragma unroll
              for (int gg = 0; gg < G; ++gg) {
                part_s[gg] = fmaf(qr[gg][8 * v + 2 * e], k0, part_s[gg]);
                part_s[gg] = fmaf(qr[gg][8 * v + 2 * e + 1], k1, part_s[gg]);
              }
            }
          }
#pragma unroll
          for (int off = C::TPK / 2; off > 0; off >>= 1)
#pragma unroll
            for (int gg = 0; gg < G; ++gg)
              part_s[gg] += __shfl_xor_sync(0xffffffffu, part_s[gg], off);
          if (part == 0) {
#pragma unroll
            for (int gg = 0; gg < G; ++gg) sb[key * G + gg] = key < nvalid ? part_s[gg] : -INFINITY;
          }
        }
        release(&bars->empty[slot], lane);
      }
      if (!group_sync(&bars->sync, sync_phase, wc)) return;
      // ---- online softmax per head (warp g owns head g)
      if (warp < G) {
        float v[KB / 32];
        float bmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < KB / 32; ++i) {
          v[i] = sb[(lane + 32 * i) * G + warp];
          bmax = fmaxf(bmax, v[i]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
          bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, off));
        const float m_new = fmaxf(m_run, bmax);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = m_new > m_run ? ex2_approx(m_run - m_use) : 1.f;
        float psum = 0.f;
#pragma unroll
        for (int i = 0; i < KB / 32; ++i) {
          const float p = ex2_approx(v[i] - m_use);
          sb[(lane + 32 * i) * G + warp] = p;
          psum += p;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
        l_run = l_run * alpha + psum;
        m_run = m_new;
        if (lane == 0) bars->alpha[nblk_done & 1u][warp] = alpha;
      }
      if (!group_sync(&bars->sync, sync_phase, wc)) return;
      // ---- P V from the V block
      {
        const int slot = static_cast<int>(it % C::NSLOTS);
        if (!warp_wait(&bars->full[slot], (it / C::NSLOTS) & 1u, wc)) return;
        ++it;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          const float al = bars->alpha[nblk_done & 1u][gg];
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[gg][i] *= al;
        }
        const uint8_t *vblk = smem + C::RING_OFF + slot * C::BLOCK_BYTES + vbox * BOX_BYTES;
        for (int key = ks; key < nvalid; key += C::NSL) {
          const int phys = vchunk ^ (key & 7);
          const uint2 x = *reinterpret_cast<const uint2 *>(vblk + key * 128 + phys * 16 + vhalf * 8);
          const float v0 = bf16lo_to_f32(x.x), v1 = bf16hi_to_f32(x.x);
          const float v2 = bf16lo_to_f32(x.y), v3 = bf16hi_to_f32(x.y);
          float p[G];
          if constexpr (G % 4 == 0) {
#pragma unroll
            for (int g4 = 0; g4 < G; g4 += 4) {
              const float4 pp = *reinterpret_cast<const float4 *>(sb + key * G + g4);
              p[g4] = pp.x;
              p[g4 + 1] = pp.y;
              p[g4 + 2] = pp.z;
              p[g4 + 3] = pp.w;
            }
          } else {
#pragma unroll
            for (int gg = 0; gg < G; ++gg) p[gg] = sb[key * G + gg];
          }
#pragma unroll
          for (int gg = 0; gg < G; ++gg) {
            acc[gg][0] = fmaf(p[gg], v0, acc[gg][0]);
            acc[gg][1] = fmaf(p[gg], v1, acc[gg][1]);
            acc[gg][2] = fmaf(p[gg], v2, acc[gg][2]);
            acc[gg][3] = fmaf(p[gg], v3, acc[gg][3]);
          }
        }
        release(&bars->empty[slot], lane);
      }
      ++nblk_done;
    }

    // ---- unit end: reduce the NSL key slices, normalise, write the partial.
#pragma unroll
    for (int gg = 0; gg < G; ++gg)
      *reinterpret_cast<float4 *>(red + (ks * G + gg) * D + 4 * dq) =
          make_float4(acc[gg][0], acc[gg][1], acc[gg][2], acc[gg][3]);
    if (warp < G && lane == 0) {
      bars->m[warp] = m_run;
      bars->l[warp] = l_run;
    }
    if (!group_sync(&bars->sync, sync_phase, wc)) return;
    const int64_t row0 = (static_cast<int64_t>(w.b) * a.Hq + w.g * G) * a.maxch + w.c;
    for (int idx = tid; idx < G * D; idx += NCOMPUTE) {
      const int gg = idx / D, dd = idx - gg * D;
      float sum = 0.f;
#pragma unroll
      for (int s = 0; s < C::NSL; ++s) sum += red[(s * G + gg) * D + dd];
      const float l = bars->l[gg];
      const int64_t row = row0 + static_cast<int64_t>(gg) * a.maxch;
      a.o_part[row * D + dd] = sum / l;
      if (dd == 0) a.lse_part[row] = (bars->m[gg] + log2f(l)) * LN2;
    }
    if (!group_sync(&bars->sync, sync_phase, wc)) return;
  }
}

template <int D, int G>
__global__ void __launch_bounds__(NTHREADS, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeArgs a) {
  using C = DCfg<D, G>;
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
  if (warp < PRODUCER_WARP) {
    compute<D, G>(a, smem, bars, wc, tid);
  } else if (lane == 0) {
    producer<D, G>(a, &tmk, &tmv, smem, bars, wc);
  }
  __syncwarp();
  __syncthreads();
}

template <int D, int G>
cudaError_t launch_decode_impl(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeArgs &a,
                               int grid, cudaStream_t stream) {
  constexpr int smem = DCfg<D, G>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  decode_kernel<D, G><<<grid, NTHREADS, smem, stream>>>(tk, tv, a);
  return cudaGetLastError();
}

// One block per (batch, query head); thread = output column.
template <int D>
__global__ void __launch_bounds__(D)
    combine_kernel(const float *o_part, const float *lse_part, const int *cache_len, int Hq,
                   int Lmax, int chunk, int maxch, __nv_bfloat16 *o, float *lse) {
  const int bh = blockIdx.x;
  const int b = bh / Hq;
  const int d = threadIdx.x;
  const int len = min(max(cache_len[b], 0), Lmax);
  const int nch = (len + chunk - 1) / chunk;
  const float *lp = lse_part + static_cast<int64_t>(bh) * maxch;
  const float *op = o_part + static_cast<int64_t>(bh) * maxch * D;
  if (nch == 0) {
    o[static_cast<int64_t>(bh) * D + d] = __float2bfloat16(0.f);
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
  o[static_cast<int64_t>(bh) * D + d] = __float2bfloat16_rn(acc / wsum);
  if (d == 0) lse[bh] = m + logf(wsum);
}

}  // namespace

int decode_smem_bytes(int d, int group) {
  if (d == 64) {
    switch (group) {
      case 1: return DCfg<64, 1>::SMEM_BYTES;
      case 2: return DCfg<64, 2>::SMEM_BYTES;
      case 4: return DCfg<64, 4>::SMEM_BYTES;
      default: return DCfg<64, 8>::SMEM_BYTES;
    }
  }
  switch (group) {
    case 1: return DCfg<128, 1>::SMEM_BYTES;
    case 2: return DCfg<128, 2>::SMEM_BYTES;
    case 4: return DCfg<128, 4>::SMEM_BYTES;
    default: return DCfg<128, 8>::SMEM_BYTES;
  }
}

cudaError_t launch_decode(int d, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                          const DecodeArgs &a, int grid, cudaStream_t stream) {
  if (d == 64) {
    switch (group) {
      case 1: return launch_decode_impl<64, 1>(tk, tv, a, grid, stream);
      case 2: return launch_decode_impl<64, 2>(tk, tv, a, grid, stream);
      case 4: return launch_decode_impl<64, 4>(tk, tv, a, grid, stream);
      default: return launch_decode_impl<64, 8>(tk, tv, a, grid, stream);
    }
  }
  switch (group) {
    case 1: return launch_decode_impl<128, 1>(tk, tv, a, grid, stream);
    case 2: return launch_decode_impl<128, 2>(tk, tv, a, grid, stream);
    case 4: return launch_decode_impl<128, 4>(tk, tv, a, grid, stream);
    default: return launch_decode_impl<128, 8>(tk, tv, a, grid, stream);
  }
}

cudaError_t launch_combine(int d, const float *o_part, const float *lse_part,
                           const int *cache_len, int B, int Hq, int Lmax, int chunk, int maxch,
                           void *o, float *lse, unsigned int * /*err*/, cudaStream_t stream) {
  const int blocks = B * Hq;
  if (blocks == 0) return cudaSuccess;
  __nv_bfloat16 *ob = reinterpret_cast<__nv_bfloat16 *>(o);
  if (d == 64)
    combine_kernel<64><<<blocks, 64, 0, stream>>>(o_part, lse_part, cache_len, Hq, Lmax, chunk,
                                                  maxch, ob, lse);
  else
    combine_kernel<128><<<blocks, 128, 0, stream>>>(o_part, lse_part, cache_len, Hq, Lmax,
                                                    chunk, maxch, ob, lse);
  return cudaGetLastError();
}

}  // namespace fa
