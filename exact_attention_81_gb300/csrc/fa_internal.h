// fa_internal.h -- declarations shared by the host API (fa_api.cu) and the kernel
// translation units.  Not part of the public C ABI (include/fa.h).
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Bits of the per-device error word that kernels set.
enum : unsigned int {
  DEVERR_PREFILL_TIMEOUT = 1u,  // a bounded wait in the prefill kernel gave up
  DEVERR_DECODE_TIMEOUT = 2u,   // a bounded wait in the decode kernel gave up
  DEVERR_BAD_CU_SEQLENS = 4u,   // varlen prefix sums out of range (sequence skipped)
  DEVERR_BAD_CACHE_LEN = 8u,    // cache_seqlens outside [0, Lmax] (clamped)
  DEVERR_BAD_APPEND = 16u,      // no room for an appended row / position past the tables
  DEVERR_BAD_BLOCK_TABLE = 32u, // a block-table entry outside [0, num_pages)
  DEVERR_BWD_TIMEOUT = 64u,     // a bounded wait in the backward kernel gave up
  DEVERR_SCHED_OVERLAP = 128u,  // a launch's ticket counter was shared with another launch
                                // running at the same time (tickets taken != expected)
};

// Arguments of the fused prefill kernel (dense and varlen share it).
struct PrefillArgs {
  void *o;              // bf16 output
  float *lse;           // fp32 output
  int64_t o_sb, o_sn, o_sh;   // output element strides (batch, token, head)
  int64_t lse_sb, lse_sh;     // lse offset = b*lse_sb + h*lse_sh + token
  int B, Hq, Hkv, group;      // group = Hq / Hkv
  int Nq, Nk;                 // dense: lengths; varlen: max_seqlen_q / max_seqlen_k
  int varlen;
  const int *cu_q, *cu_k;     // varlen prefix sums (device)
  int total_q, total_k;
  int mblocks;                // query blocks (prefill_tile_rows rows) per (batch, head)
  int num_tiles;              // B * Hq * mblocks
  int half_from;              // tiles [half_from, num_tiles) are handed out as two half tiles
                              // (one 128-row sub-tile each); = num_tiles for none
  int num_tickets;            // half_from + 2 * (num_tiles - half_from)
  float scale_log2;           // scale * log2(e)
  int sched_slot;             // this launch's tile-ticket counter slot
  int d;                      // head dimension of the tensors (the kernel's D may be larger:
                              // the columns past d arrive as zeros and are not stored)
  unsigned int *err;          // device error word
  unsigned long long timeout_ns;
  int inject;                 // failure injection: the producer issues no load at all
  // Score modifiers (read by the MASK_MOD / MASK_ALIBI / MASK_WINDOW kernels only).
  int wl, wr;                 // window bounds in keys, -1 = unbounded (causal folded: wr = 0)
  float sc_in, sc_out;        // softcap: s -> tanh(s * sc_in) * sc_out (log2 units); 0 = off
  const float *alibi;         // slopes of (b, h) at alibi[b * alibi_sb + h], or null
  int64_t alibi_sb;
  int desc;                   // hand out query blocks last-first (right-bounded windows)
  int head_group;             // last-first order: (batch, head) pairs per group (<= 1: one)
  int kv_rev;                 // stream each block's K/V tiles last-first (ALiBi, right-bounded)
  // FP8 launches: descale factors per (batch, kv head) at [b * Hkv + hk], or null (= 1).
  const float *q_descale, *k_descale, *v_descale;
  // The launch's O map (32-row boxes) is valid: a softmax warp whose 32 rows all lie in the
  // sub-tile stages its O rows in shared memory and writes them with TMA stores (kernels of
  // width <= 128 without ALiBi, single CTAs); other warps store rows directly.
  int o_tma;
};

// Masking mode of a prefill launch.
enum PrefillMask : int {
  MASK_NONE = 0,    // every key visible (tail of the key range masked)
  MASK_CAUSAL = 1,  // bottom-right causal
  MASK_MOD = 2,     // softcap, with or without ALiBi (and any window)
  MASK_WINDOW = 3,  // sliding window only: the MASK_MOD masking without the softcap / ALiBi
                    // code, which made every window call 27 % slower
  MASK_ALIBI = 4,   // ALiBi without a softcap (and any window): no tanh code
};

// Mask modes whose kernels apply a general window (left and right bounds).
__host__ __device__ constexpr bool mask_has_window(int m) {
  return m == MASK_MOD || m == MASK_WINDOW || m == MASK_ALIBI;
}

// Tile-ticket counter slot for the next prefill launch (round robin over the slots).
int next_prefill_sched_slot();

// Unit-ticket counter slot for the next decode launch (round robin over the slots).
int next_decode_sched_slot();

// f16: inputs and output are fp16 instead of bf16.  tmo: map over O with 32-row boxes
// (make_map), read when a.o_tma is set; null otherwise.
cudaError_t launch_prefill(int d, int mask, bool f16, const CUtensorMap &tq,
                           const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap *tmo,
                           const PrefillArgs &a, int grid, cudaStream_t stream);

// The width-128 16-bit prefill on CTA pairs (clusters of two computing each 256-row sub-tile
// as one cta_group::2 product; work tiles of 512 query rows): tk is a K map with 64-row boxes,
// tq and tv maps with 128-row boxes.  The grid is sized inside from `tiles`.
cudaError_t launch_prefill_pair(int mask, bool f16, const CUtensorMap &tq, const CUtensorMap &tk,
                                const CUtensorMap &tv, const PrefillArgs &a, int tiles,
                                cudaStream_t stream);

// FP8 (E4M3) prefill, d <= 128 at kernel width 128: tq, tk over E4M3 Q and K, tvt over the
// transposed V written by launch_transpose_v (dims {keys, d, kv head, batch}) or, packed
// sequences (a.varlen), by launch_transpose_v_varlen (dims {nt, d, kv head, 1}).
cudaError_t launch_prefill_fp8(int mask, const CUtensorMap &tq, const CUtensorMap &tk,
                               const CUtensorMap &tvt, const CUtensorMap *tmo,
                               const PrefillArgs &a, int grid, cudaStream_t stream);

// V [B, Nk, Hkv, d] E4M3 (byte strides v_sb, v_sn, v_sh) -> V^T [B, Hkv, d, nk_pad], keys
// contiguous, zeros in the columns [Nk, nk_pad).
cudaError_t launch_transpose_v(const void *v, int64_t v_sb, int64_t v_sn, int64_t v_sh, void *vt,
                               int B, int Nk, int Hkv, int d, int nk_pad, cudaStream_t stream);

// Packed sequences: V [total_k, Hkv, d] E4M3 (contiguous) -> V^T [Hkv, d, nt] after zeroing
// it, sequence b's keys at columns roundup16(cu_k[b]) + 16 b onwards; nt >= roundup16(total_k)
// + 16 (B + 1), a multiple of 16.
cudaError_t launch_transpose_v_varlen(const void *v, void *vt, const int *cu_k, int B,
                                      int max_seqlen_k, int total_k, int Hkv, int d, int nt,
                                      cudaStream_t stream);

// O = 0 and LSE = -inf for every row (no visible keys anywhere).
cudaError_t launch_fill_empty(void *o, float *lse, int B, int N, int H, int d, int64_t o_sb,
                              int64_t o_sn, int64_t o_sh, int64_t lse_sb, int64_t lse_sh,
                              cudaStream_t stream);

// Arguments of the split-KV decode kernel.
struct DecodeArgs {
  const void *q;              // [B, 1, Hq, d] bf16 contiguous
  const int *cache_len;       // [B] device
  float *o_part;              // [B*Hq, maxch, d] fp32 partial outputs (normalised per chunk)
  float *lse_part;            // [B*Hq, maxch] fp32 partial LSE (natural log)
  int B, Hq, Lmax;
  int Hkv;                    // work items per batch entry: kv heads * nsplit
  int nsplit;                 // each kv head's query group runs as nsplit work items of the
                              // kernel's G heads (group = nsplit * G; G <= 8, and <= 4 at
                              // d = 256, whose q, scores and accumulators must fit in
                              // registers); the items of one kv head stream the same K/V rows
  int chunk;                  // keys per split (multiple of 128)
  int maxch;                  // chunks of the longest visible range: ceil(Leff / chunk)
  int d;                      // head dimension of q and the caches (<= the kernel's D)
  int num_units;              // maxch * B * Hkv (work items)
  int sched_slot;             // this launch's unit-ticket counter slot
  float scale_log2;
  unsigned int *err;
  unsigned long long timeout_ns;
  int inject;                 // failure injection: the producer issues no load at all
  // Score modifiers (uniform runtime branches).
  int wl;                     // left window bound in keys, -1 = unbounded
  float sc_in, sc_out;        // softcap on the log2-domain score: tanh(s * sc_in) * sc_out
  const float *alibi;         // slopes of (b, h) at alibi[b * alibi_sb + h], or null
  int64_t alibi_sb;
  // KV-cache extras.
  int len_add;                // 1 after an in-place append (length = cache_len + 1)
  const int *block_table;     // paged cache: page of logical block j of b at [b*bt_stride + j]
  int bt_stride, page_size, num_pages;
  int kalign;                 // unit starts rounded down to a multiple of this (128 if paged)
  // E4M3 caches: descale factors per (batch, kv head) [B, kv heads], null = 1.
  const float *k_descale, *v_descale;
  int ostride;                // width of a partial-output row (<= the kernel's D)
};

// First key a decode unit streams: the first visible key, rounded down to `align` so that a
// 128-key block never crosses a page.  Keys before the first visible one are masked.
__host__ __device__ inline int decode_first_key(int len, int wl, int align) {
  const int first = (wl >= 0 && len - 1 - wl > 0) ? len - 1 - wl : 0;
  return first - first % align;
}

// In-place append of one new key/value row per sequence, with optional rotary embedding
// of the new key and of the query (the rotated query goes to q_rot).
struct AppendArgs {
  const void *k_new, *v_new;
  int64_t n_sb, n_sh;         // element strides (batch, head) of k_new / v_new
  void *k_cache, *v_cache;
  int64_t c_s0, c_s1, c_s2;   // cache strides: (batch or page, row, head)
  const int *cache_len;
  int B, Hq, Hkv, d, Lmax;
  const int *block_table;
  int bt_stride, page_size, num_pages;
  const float *cos, *sin;     // rotary tables [rot_positions, rot_dim / 2], or null
  int rot_dim, rot_positions, rot_interleaved;
  const void *q;              // [B, 1, Hq, d] contiguous
  void *q_rot;                // rotated query [B, 1, Hq, d] (when rotary)
  unsigned int *err;
};

cudaError_t launch_append(bool f16, const AppendArgs &a, cudaStream_t stream);

// d: the kernel width (64, 128 or 256; 128 or 256 when kv_e4m3, with a bf16 query).
cudaError_t launch_decode(int d, int group, bool f16, bool kv_e4m3, const CUtensorMap &tk,
                          const CUtensorMap &tv, const DecodeArgs &a, int grid,
                          cudaStream_t stream);

// wl, kalign, len_add: as in DecodeArgs; chunks tile the keys [decode_first_key, len) of
// each sequence, len = cache_len + len_add.
// d: the width of the partial rows (64, 128 or 256); d_out: the head dimension of o.
cudaError_t launch_combine(int d, int d_out, bool f16, const float *o_part, const float *lse_part,
                           const int *cache_len, int len_add, int B, int Hq, int Lmax, int chunk,
                           int maxch, int wl, int kalign, void *o, float *lse, unsigned int *err,
                           cudaStream_t stream);

// Width of the kernel instance that serves head dimension d (8 <= d <= 256, d % 8 == 0;
// the backward serves widths up to 128).
inline int kernel_d(int d) { return d <= 64 ? 64 : (d <= 128 ? 128 : 256); }

// Width of the decode instance over E4M3 caches (a 128-byte box row is 128 elements).
inline int kernel_d_e4m3(int d) { return d <= 128 ? 128 : 256; }

// Query rows of one prefill work tile for kernel width kd: two 128-row sub-tiles, one
// when the head dimension is above 128 (TMEM holds a single D-wide accumulator then).
inline int prefill_tile_rows(int kd) { return kd > 128 ? 128 : 256; }

// Backward pass: main kernel arguments (one work unit = batch, kv head, 128-key block).
struct BwdArgs {
  const float *lse;           // natural-log LSE of the forward pass, [B, Hq, Nq] or [Hq, total_q]
  const float *dvec;          // D = rowsum(dO * O), same layout as lse
  int64_t lse_sb, lse_sh;     // lse / dvec offset = b*lse_sb + h*lse_sh + token
  int varlen;                 // packed sequences delimited by cu_q / cu_k (device)
  const int *cu_q, *cu_k;
  int total_q, total_k;
  int qblocks;                // ceil(Nq / 128): query blocks of the longest sequence
  void *dk, *dv;              // outputs [B, Nk, Hkv, d], element strides below
  int64_t dk_sb, dk_sn, dk_sh, dv_sb, dv_sn, dv_sh;
  int B, Nq, Nk, Hq, Hkv, group;
  int kblocks;                // ceil(Nk / 128)
  int d;                      // head dimension of the tensors (<= the kernel's D)
  int *sem;                   // deterministic dQ: additions done per (b, h, query block), or null
  // Score modifiers (read by the windowed / modifier kernels only), as in PrefillArgs.
  int wl, wr;
  float sc_in, sc_out;        // softcap: z2 = tanh(s * sc_in) * sc_out, dz/ds = 1 - tanh^2
  const float *alibi;
  int64_t alibi_sb;
  int num_units;              // kblocks * B * Hkv
  int head_group;             // (batch, kv head) pairs per unit group, >= 1
  float scale, scale_log2;
  unsigned int *err;
  unsigned long long timeout_ns;
  int inject;                 // failure injection: the producer issues no load at all
};

// D = rowsum(dO * O) per query row, a zeroed fp32 dQ accumulator of acc_n floats (a
// multiple of 4) and nsem zeroed counters.
cudaError_t launch_bwd_pre(int d, bool f16, const void *o, const void *dout, int B, int Nq,
                           int Hq, const int64_t o_st[3], const int64_t do_st[3], float *dvec,
                           float *dq_acc, int64_t acc_n, int *sem, int nsem, cudaStream_t stream);

// tq, tk, tv, tdo: 16-bit maps like the forward's; tdq: fp32 map of the dQ accumulator
// (box 32 x 128 rows, 128-byte swizzle).  Kernel width d = 256 (head dimensions 136..256):
// the wide kernel, whose units are (batch, kv head, key block, d half) and steps 64 queries
// (num_units = 2 x kblocks x B x Hkv, qblocks = ceil(Nq / 64), counters per (b, h, 64-query
// block, d half)); tq and tdo with 64-row boxes, tdq the transposed accumulator
// [B, Hq, d, nq_pad] (box 32 queries x 128 d rows).
cudaError_t launch_bwd(int d, int mask, bool f16, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &tdo, const CUtensorMap &tdq,
                       const BwdArgs &a, int grid, cudaStream_t stream);

// dQ = scale * accumulator, rounded to the element type, into a strided [B, Nq, Hq, d].
cudaError_t launch_bwd_post(int d, bool f16, const float *dq_acc, float scale, void *dq, int B,
                            int Nq, int Hq, const int64_t dq_st[3], cudaStream_t stream);

// The wide kernel's dQ: scale * the transposed accumulator [B, Hq, d, nq_pad] into a strided
// [B, Nq, Hq, d]; varlen (cu_q non-null): B sequences of at most Nq queries into the packed
// [total_q, Hq, d] (strides dq_st[1], dq_st[2]).
cudaError_t launch_bwd_post_t(int d, bool f16, const float *dq_acc, float scale, void *dq, int B,
                              int Nq, int nq_pad, int Hq, const int64_t dq_st[3],
                              const int *cu_q, int total_q, cudaStream_t stream);

// Query extent of the wide kernel's transposed dQ accumulator: Nq rounded up to 4 (16-byte
// rows).
inline int dq_acc_nq(int nq) { return (nq + 3) / 4 * 4; }

// Zeroes a strided 16-bit [B, N, H, d] tensor.
cudaError_t launch_zero16(void *x, int B, int N, int H, int d, const int64_t st[3],
                          cudaStream_t stream);

// Shared-memory bytes the prefill kernel requests (for host-side checks).
int prefill_smem_bytes(int d);

}  // namespace fa
