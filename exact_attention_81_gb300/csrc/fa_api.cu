// fa_api.cu -- the C ABI of libfa.so (declared in include/fa.h): argument validation,
// TMA tensor-map construction, work decomposition and kernel launches.  No allocation,
// no synchronisation (except in fa_get_last_device_error), everything on the caller's
// stream.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

// Per-device word the kernels OR their fault bits into.
__device__ unsigned int g_device_error;

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 10ull * 1000 * 1000 * 1000;

constexpr int kMaxHostRanges = 128;  // (batch, query range) pieces of one fa_fwd_host call

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int sm_count = 0;
  unsigned int *err = nullptr;  // device address of g_device_error on this device
  // fa_fwd_host: two copy streams and the events that order them against the caller's
  // stream, created on first use; host_mutex serialises the calls that reuse them.
  bool host_ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev_start = nullptr, ev_end = nullptr;
  cudaEvent_t ev_in[kMaxHostRanges] = {}, ev_out[kMaxHostRanges] = {};
  std::mutex host_mutex;
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
unsigned long long g_timeout_ns = kDefaultTimeoutNs;
int g_inject = 0;  // fa_set_fault_injection
int g_cta_pairs = 0;  // fa_set_cta_pairs

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

thread_local char g_cuda_msg[512] = "";

fa_status cuda_fail(const char *what, cudaError_t e) {
  snprintf(g_cuda_msg, sizeof g_cuda_msg, "%s: %s (%s)", what, cudaGetErrorName(e),
           cudaGetErrorString(e));
  return FA_ERR_CUDA;
}

// Looks up the current device; fills its capabilities and the error-word address once.
fa_status current_device(DeviceInfo **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo &d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail("cudaDeviceGetAttribute", e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail("cudaDeviceGetAttribute", e);
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail("cudaDeviceGetAttribute", e);
    d.supported = (major == 10 && minor == 3);
    d.sm_count = sms;
    if (d.supported) {
      void *p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_device_error)) != cudaSuccess)
        return cuda_fail("cudaGetSymbolAddress", e);
      d.err = static_cast<unsigned int *>(p);
      if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
          return cuda_fail("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)",
                           e != cudaSuccess ? e : cudaErrorSymbolNotFound);
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
      }
    }
    d.ready = true;
  }
  if (!d.supported) return FA_ERR_UNSUPPORTED;
  *out = &d;
  return FA_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 4-D 16-bit tensor map over a (batch, seq, head, d) tensor, dimensions ordered
// {d, head, seq, batch}, box {64, 1, box_rows, 1} (64 columns x 128 rows of one head, or 64
// rows for the K halves of a CTA pair), 128-byte swizzle, zero fill past the tensor edges.
// sn/sh/sb are element strides.
fa_status make_map(CUtensorMap *map, const void *base, int d, int64_t n, int64_t h, int64_t b,
                   int64_t sn, int64_t sh, int64_t sb, int dtype, int box_rows = 128) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(h),
                        static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(b)};
  // The stride of a dimension of extent 1 is never used; give it a legal value.
  const int64_t es = dtype == FA_E4M3 ? 1 : 2;  // bytes per element
  const int64_t bh = h > 1 ? sh * es : static_cast<int64_t>(d) * es;
  const int64_t bn = n > 1 ? sn * es : bh * h;
  const int64_t bb = b > 1 ? sb * es : bn * n;
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(bh), static_cast<cuuint64_t>(bn),
                           static_cast<cuuint64_t>(bb)};
  for (int i = 0; i < 3; ++i)
    if (strides[i] == 0 || (strides[i] % 16) != 0 || strides[i] >= (cuuint64_t(1) << 40))
      return FA_ERR_INVALID_ARG;
  // 128-byte box rows: 64 16-bit or 128 8-bit elements
  cuuint32_t box[4] = {dtype == FA_E4M3 ? 128u : 64u, 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty =
      dtype == FA_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
      : (dtype == FA_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  CUresult r = g_encode(map, ty, 4, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_cuda_msg, sizeof g_cuda_msg, "cuTensorMapEncodeTiled failed (CUresult %d)",
             static_cast<int>(r));
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

// 4-D fp32 tensor map over a contiguous (batch, seq, head, d) accumulator, box
// {32, 1, 128, 1} (32 floats = 128 bytes x 128 rows), 128-byte swizzle: the target of the
// backward pass's dQ reductions.
// 4-D 8-bit map over the transposed V [B, Hkv, d, nk_pad] written by launch_transpose_v:
// dims {keys, d, kv head, batch}, box {128 keys, 128 rows of d} (rows past d read as 0).
fa_status make_map_vt(CUtensorMap *map, void *base, int nk_pad, int d, int Hkv, int B) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(nk_pad), static_cast<cuuint64_t>(d),
                        static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(nk_pad),
                           static_cast<cuuint64_t>(nk_pad) * d,
                           static_cast<cuuint64_t>(nk_pad) * d * Hkv};
  cuuint32_t box[4] = {128, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_cuda_msg, sizeof g_cuda_msg, "cuTensorMapEncodeTiled failed (CUresult %d)",
             static_cast<int>(r));
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

fa_status make_map_f32(CUtensorMap *map, void *base, int d, int64_t n, int64_t h, int64_t b) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(h),
                        static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(b)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(h * d) * 4,
                           static_cast<cuuint64_t>(n * h * d) * 4};
  cuuint32_t box[4] = {32, 1, 128, 1};  // 32 columns x the 128 rows of a backward step
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_cuda_msg, sizeof g_cuda_msg, "cuTensorMapEncodeTiled (fp32) failed (CUresult %d)",
             static_cast<int>(r));
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

// The transposed fp32 dQ accumulator [b, h, d, nq_pad] of the wide backward kernel: box =
// 32 queries (128 bytes) x 128 d rows, 128-byte swizzle (the staging layout).
fa_status make_map_dqt(CUtensorMap *map, void *base, int d, int64_t nq_pad, int64_t h,
                       int64_t b) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(nq_pad), static_cast<cuuint64_t>(d),
                        static_cast<cuuint64_t>(h), static_cast<cuuint64_t>(b)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(nq_pad) * 4,
                           static_cast<cuuint64_t>(d * nq_pad) * 4,
                           static_cast<cuuint64_t>(h * d * nq_pad) * 4};
  cuuint32_t box[4] = {32, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_cuda_msg, sizeof g_cuda_msg, "cuTensorMapEncodeTiled (fp32) failed (CUresult %d)",
             static_cast<int>(r));
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

// Backward workspace parts: the fp32 dQ accumulator ([B, Nq, Hq, d]; kernel width 256: the
// transposed [B, Hq, d, Nq rounded up to 4]) and the deterministic-order counters (per
// (b, h, 128-query block); width 256: per (b, h, 64-query block, d half)), in elements.
int64_t bwd_acc_elems(int B, int Nq, int Hq, int d) {
  return fa::kernel_d(d) == 256 ? static_cast<int64_t>(B) * Hq * d * fa::dq_acc_nq(Nq)
                                : static_cast<int64_t>(B) * Nq * Hq * d;
}
int64_t bwd_sem_elems(int B, int Nq, int Hq, int d) {
  return fa::kernel_d(d) == 256 ? static_cast<int64_t>(B) * Hq * ((Nq + 63) / 64) * 2
                                : static_cast<int64_t>(B) * Hq * ((Nq + 127) / 128);
}

bool stride_ok(int64_t s, int64_t extent) {
  if (extent <= 1) return s >= 0;
  return s > 0 && (s % 8) == 0 && s < (int64_t(1) << 38);
}

float scale_log2(float scale) {
  return static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
}

bool scale_ok(float s) { return std::isfinite(s) && s > 0.f; }

bool dtype_ok(int t) { return t == FA_BF16 || t == FA_FP16; }

// Head dimensions served: multiples of 8 up to max_d (the kernels run at width 64, 128 or
// 256; the tensor maps give the columns past d as zeros).  The forward and decode calls
// take up to 256, the backward up to 128.
bool head_dim_ok(int d, int max_d = 128) { return d >= 8 && d <= max_d && d % 8 == 0; }
constexpr int kMaxPrefillD = 256;
constexpr int kMaxDecodeD = 256;

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// The 16-bit forward at width 128 runs on CTA pairs (cta_group::2) after fa_set_cta_pairs(1).
bool use_pairs(int d) { return g_cta_pairs != 0 && fa::kernel_d(d) == 128; }

// Query rows of a prefill work tile: 512 for CTA pairs (two 256-row sub-tiles).
int tile_rows(int d, bool pairs) { return pairs ? 512 : fa::prefill_tile_rows(fa::kernel_d(d)); }

// Keys per split for the decode path (a multiple of the 128-key block).
int decode_chunk(int Lmax, int num_splits) {
  int64_t c;
  if (num_splits > 0) {
    c = (static_cast<int64_t>(Lmax) + num_splits - 1) / num_splits;
  } else {
    c = (static_cast<int64_t>(Lmax) + 15) / 16;  // about 16 splits of a full-length cache
    if (c < 256) c = 256;
  }
  c = ((c + 127) / 128) * 128;
  if (c < 128) c = 128;
  return static_cast<int>(c);
}

// Score modifiers as the kernels take them.
struct ModPlan {
  int mask = fa::MASK_NONE;  // prefill kernel mode
  int wl = -1, wr = -1;      // window bounds in keys (-1 = unbounded); causal folded into wr
  float softcap = 0.f;
  const float *alibi = nullptr;
  int64_t alibi_sb = 0;
};

constexpr int kMaxWindow = 1 << 30;  // longer windows are unbounded for every valid length

// Validates `m` (may be null) and folds `causal` into the window.
fa_status plan_mod(const fa_score_mod *m, int causal, ModPlan *out) {
  ModPlan p;
  if (m != nullptr) {
    if (!std::isfinite(m->softcap) || m->softcap < 0.f) return FA_ERR_INVALID_ARG;
    if (m->alibi_slopes != nullptr && (!aligned(m->alibi_slopes, 4) || m->alibi_batch_stride < 0))
      return FA_ERR_INVALID_ARG;
    if (m->use_window) {
      p.wl = m->window_left < 0 ? -1 : std::min(m->window_left, kMaxWindow);
      p.wr = m->window_right < 0 ? -1 : std::min(m->window_right, kMaxWindow);
    }
    p.softcap = m->softcap;
    p.alibi = m->alibi_slopes;
    p.alibi_sb = m->alibi_batch_stride;
  }
  if (causal) p.wr = 0;
  if (p.softcap != 0.f)
    p.mask = fa::MASK_MOD;
  else if (p.alibi != nullptr)
    p.mask = fa::MASK_ALIBI;
  else if (p.wl >= 0 || p.wr > 0)
    p.mask = fa::MASK_WINDOW;
  else
    p.mask = p.wr < 0 ? fa::MASK_NONE : fa::MASK_CAUSAL;
  *out = p;
  return FA_OK;
}

// The modifier fields shared by the forward and backward argument blocks.
template <class Args>
void set_mod_fields(const ModPlan &m, float scale, Args *a) {
  a->wl = m.wl;
  a->wr = m.wr;
  // raw score s: softcap * tanh(scale * s / softcap), then * log2(e)
  a->sc_in = m.softcap > 0.f ? scale / m.softcap : 0.f;
  a->sc_out = m.softcap > 0.f ? static_cast<float>(m.softcap * 1.4426950408889634) : 0.f;
  a->alibi = m.alibi;
  a->alibi_sb = m.alibi_sb;
}

// (batch, head) pairs per group of the longest-first tile order (causal and right-bounded
// windows).
static int prefill_head_group() { return 8; }

void apply_mod(const ModPlan &m, float scale, fa::PrefillArgs *pa) {
  set_mod_fields(m, scale, pa);
  pa->desc = m.wr >= 0;
  pa->head_group = prefill_head_group();
  // ALiBi with a right-bounded window: the bias grows toward the last visible key, so the
  // K/V tiles run last-first and the row max is met on the first tile instead of moving
  // (and rescaling O) on every one.  Not with a softcap: there the reversed order measured
  // slower (1.5 % on causal 8k), the softcap's tanh and not the rescale bounding the step.
  pa->kv_rev = m.alibi != nullptr && m.wr >= 0 && m.softcap == 0.f;
}

// Keys per split when the caller leaves it to the library.  Long chunks amortise the
// per-unit work (the group's query slice, the merge of the 8 warps, the partial write):
// 2048 keys (16 blocks) measured best over 16-bit caches, 8192 over E4M3 caches (half the
// bytes per key: on the decode workload 0.418 ms against 0.466 ms at 2048); they are
// halved, down to 256, only while the units ((batch, kv head) pairs x chunks) would not
// fill 4 waves of the SMs.  The result never needs more than ws_chunks chunks, the count
// the workspace was sized for.
int auto_chunk(int Leff, int64_t pairs, int sm_count, int ws_chunks, bool e4m3) {
  int c = e4m3 ? 8192 : 2048;
  while (c > 256 && pairs * ceil_div(Leff, c) < 4ll * sm_count) c /= 2;
  const int fit = (ceil_div(Leff, ws_chunks) + 127) / 128 * 128;
  return std::max(c, fit);
}

}  // namespace

extern "C" {

const char *fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported configuration or device";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA call failed";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace missing or too small";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a device-side wait gave up";
    case FA_ERR_CONCURRENT:
      return "FA_ERR_CONCURRENT: a launch shared its tile-ticket counter with another launch "
             "running at the same time";
  }
  return "unknown fa_status";
}

const char *fa_last_cuda_error(void) { return g_cuda_msg; }

size_t fa_fwd_params_size(void) { return sizeof(fa_fwd_params); }

void fa_set_wait_timeout_ns(unsigned long long ns) {
  g_timeout_ns = ns == 0 ? kDefaultTimeoutNs : ns;
}

void fa_set_fault_injection(int withhold_loads) { g_inject = withhold_loads != 0; }

void fa_set_cta_pairs(int enable) { g_cta_pairs = enable != 0; }

// Keys padded to a multiple of 16 (the byte stride of a transposed V row).
int64_t nk_pad16(int64_t nk) { return (nk + 15) / 16 * 16; }

// Byte strides of 8-bit tensors: multiples of 16 (tensor-map rule).
bool stride_ok_16b(int64_t s, int64_t extent) {
  if (extent <= 1) return s >= 0;
  return s > 0 && (s % 16) == 0 && s < (int64_t(1) << 38);
}

fa_status launch_dense(const fa_fwd_params &a, DeviceInfo *dev, const ModPlan &mod,
                       int64_t lse_sb, int64_t lse_sh, cudaStream_t stream);

// Prefill arguments of packed sequences (o [total_q, Hq, d], lse [Hq, total_q]).
fa::PrefillArgs varlen_args(void *o, float *lse, const int *cu_q, const int *cu_k, int B,
                            int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int Hq,
                            int Hkv, int d, float scale, int mblocks, int64_t tiles,
                            DeviceInfo *dev, const ModPlan &mod) {
  fa::PrefillArgs pa{};
  pa.o = o;
  pa.lse = lse;
  pa.o_sb = 0;
  pa.o_sn = static_cast<int64_t>(Hq) * d;
  pa.o_sh = d;
  pa.lse_sb = 0;
  pa.lse_sh = total_q;
  pa.B = B;
  pa.Hq = Hq;
  pa.Hkv = Hkv;
  pa.group = Hq / Hkv;
  pa.Nq = max_seqlen_q;
  pa.Nk = max_seqlen_k;
  pa.varlen = 1;
  pa.cu_q = cu_q;
  pa.cu_k = cu_k;
  pa.total_q = total_q;
  pa.total_k = total_k;
  pa.mblocks = mblocks;
  pa.num_tiles = static_cast<int>(tiles);
  pa.half_from = pa.num_tiles;
  pa.num_tickets = pa.num_tiles;
  pa.scale_log2 = scale_log2(scale);
  pa.err = dev->err;
  pa.timeout_ns = g_timeout_ns;
  pa.inject = g_inject;
  pa.sched_slot = fa::next_prefill_sched_slot();
  pa.d = d;
  apply_mod(mod, scale, &pa);
  return pa;
}

// Prefill arguments of a dense call (fa_fwd, fa_fwd_fp8).
fa::PrefillArgs dense_args(const fa_fwd_params &a, int mblocks, int64_t tiles,
                           const DeviceInfo *dev, const ModPlan &mod, int64_t lse_sb,
                           int64_t lse_sh) {
  fa::PrefillArgs pa{};
  pa.o = a.o;
  pa.lse = a.lse;
  pa.o_sb = a.o_strides[0];
  pa.o_sn = a.o_strides[1];
  pa.o_sh = a.o_strides[2];
  pa.lse_sb = lse_sb;
  pa.lse_sh = lse_sh;
  pa.B = a.B;
  pa.Hq = a.Hq;
  pa.Hkv = a.Hkv;
  pa.group = a.Hq / a.Hkv;
  pa.Nq = a.Nq;
  pa.Nk = a.Nk;
  pa.varlen = 0;
  pa.mblocks = mblocks;
  pa.num_tiles = static_cast<int>(tiles);
  pa.half_from = pa.num_tiles;
  pa.num_tickets = pa.num_tiles;
  pa.scale_log2 = scale_log2(a.scale);
  pa.err = dev->err;
  pa.timeout_ns = g_timeout_ns;
  pa.inject = g_inject;
  pa.sched_slot = fa::next_prefill_sched_slot();
  pa.d = a.d;
  apply_mod(mod, a.scale, &pa);
  return pa;
}

fa_status fa_fwd(const fa_fwd_params *p, cudaStream_t stream) {
  if (p == nullptr) return FA_ERR_INVALID_ARG;
  const fa_fwd_params &a = *p;
  if (a.B < 0 || a.Nq < 0 || a.Nk < 0 || a.Hq <= 0 || a.Hkv <= 0 || a.Hq % a.Hkv != 0)
    return FA_ERR_INVALID_ARG;
  if (!head_dim_ok(a.d, kMaxPrefillD)) return FA_ERR_UNSUPPORTED;
  if (!dtype_ok(a.dtype)) return FA_ERR_UNSUPPORTED;
  if (!scale_ok(a.scale)) return FA_ERR_INVALID_ARG;
  if (a.Nq > (1 << 30) || a.Nk > (1 << 30)) return FA_ERR_INVALID_ARG;
  if (a.B == 0 || a.Nq == 0) return FA_OK;
  if (a.q == nullptr || a.o == nullptr || a.lse == nullptr) return FA_ERR_INVALID_ARG;
  if (!aligned(a.q, 16) || !aligned(a.o, 16) || !aligned(a.lse, 4)) return FA_ERR_INVALID_ARG;
  if (!stride_ok(a.q_strides[0], a.B) || !stride_ok(a.q_strides[1], a.Nq) ||
      !stride_ok(a.q_strides[2], a.Hq) || !stride_ok(a.o_strides[0], a.B) ||
      !stride_ok(a.o_strides[1], a.Nq) || !stride_ok(a.o_strides[2], a.Hq))
    return FA_ERR_INVALID_ARG;
  if (a.Nk > 0) {
    if (a.k == nullptr || a.v == nullptr) return FA_ERR_INVALID_ARG;
    if (!aligned(a.k, 16) || !aligned(a.v, 16)) return FA_ERR_INVALID_ARG;
    if (!stride_ok(a.k_strides[0], a.B) || !stride_ok(a.k_strides[1], a.Nk) ||
        !stride_ok(a.k_strides[2], a.Hkv) || !stride_ok(a.v_strides[0], a.B) ||
        !stride_ok(a.v_strides[1], a.Nk) || !stride_ok(a.v_strides[2], a.Hkv))
      return FA_ERR_INVALID_ARG;
  }
  const int mblocks = ceil_div(a.Nq, tile_rows(a.d, false));
  const int64_t tiles = static_cast<int64_t>(a.B) * a.Hq * mblocks;
  if (tiles > INT32_MAX) return FA_ERR_INVALID_ARG;
  ModPlan mod;
  fa_status st = plan_mod(&a.mod, a.causal, &mod);
  if (st != FA_OK) return st;

  DeviceInfo *dev = nullptr;
  st = current_device(&dev);
  if (st != FA_OK) return st;
  return launch_dense(a, dev, mod, static_cast<int64_t>(a.Hq) * a.Nq, a.Nq, stream);
}

// The launch part of fa_fwd for validated arguments; lse_sb / lse_sh: LSE strides (the host
// path computes row ranges of a larger LSE array).
fa_status launch_dense(const fa_fwd_params &a, DeviceInfo *dev, const ModPlan &mod,
                       int64_t lse_sb, int64_t lse_sh, cudaStream_t stream) {
  fa_status st;
  const bool pairs = use_pairs(a.d);
  const int mblocks = ceil_div(a.Nq, tile_rows(a.d, pairs));
  const int64_t tiles = static_cast<int64_t>(a.B) * a.Hq * mblocks;
  if (a.Nk == 0) {
    cudaError_t e = fa::launch_fill_empty(a.o, a.lse, a.B, a.Nq, a.Hq, a.d, a.o_strides[0],
                                          a.o_strides[1], a.o_strides[2], lse_sb, lse_sh, stream);
    return e == cudaSuccess ? FA_OK : cuda_fail("fill kernel launch", e);
  }
  CUtensorMap tq, tk, tv;
  if ((st = make_map(&tq, a.q, a.d, a.Nq, a.Hq, a.B, a.q_strides[1], a.q_strides[2],
                     a.q_strides[0], a.dtype)) != FA_OK)
    return st;
  if ((st = make_map(&tk, a.k, a.d, a.Nk, a.Hkv, a.B, a.k_strides[1], a.k_strides[2],
                     a.k_strides[0], a.dtype, pairs ? 64 : 128)) != FA_OK)
    return st;
  if ((st = make_map(&tv, a.v, a.d, a.Nk, a.Hkv, a.B, a.v_strides[1], a.v_strides[2],
                     a.v_strides[0], a.dtype)) != FA_OK)
    return st;
  fa::PrefillArgs pa = dense_args(a, mblocks, tiles, dev, mod, lse_sb, lse_sh);
  cudaError_t e;
  if (pairs) {
    e = fa::launch_prefill_pair(mod.mask, a.dtype == FA_FP16, tq, tk, tv, pa,
                                static_cast<int>(tiles), stream);
  } else {
    const int grid = static_cast<int>(tiles < dev->sm_count ? tiles : dev->sm_count);
    // Without a mask every tile costs the same, and tiles % grid of them would run as a last,
    // partial wave; they are handed out as two half tiles each instead (S double-buffered:
    // a half tile takes about half a tile's time).
    if (mod.mask == fa::MASK_NONE && fa::kernel_d(a.d) <= 128 && tiles > grid &&
        tiles % grid != 0) {
      pa.half_from = static_cast<int>(tiles - tiles % grid);
      pa.num_tickets = pa.half_from + 2 * static_cast<int>(tiles % grid);
    }
    CUtensorMap to;
    pa.o_tma = make_map(&to, a.o, a.d, a.Nq, a.Hq, a.B, a.o_strides[1], a.o_strides[2],
                        a.o_strides[0], a.dtype, 32) == FA_OK;
    e = fa::launch_prefill(fa::kernel_d(a.d), mod.mask, a.dtype == FA_FP16, tq, tk, tv,
                           pa.o_tma ? &to : nullptr, pa, grid, stream);
  }
  return e == cudaSuccess ? FA_OK : cuda_fail("prefill kernel launch", e);
}

size_t fa_fwd_fp8_workspace_size(int B, int Nk, int Hkv, int d) {
  if (B <= 0 || Nk <= 0 || Hkv <= 0 || d <= 0) return 0;
  const int64_t bytes = static_cast<int64_t>(B) * Hkv * d * nk_pad16(Nk);
  return static_cast<size_t>((bytes + 255) / 256 * 256);
}

fa_status fa_fwd_fp8(const fa_fwd_params *p, const float *q_descale, const float *k_descale,
                     const float *v_descale, void *workspace, size_t workspace_bytes,
                     cudaStream_t stream) {
  if (p == nullptr) return FA_ERR_INVALID_ARG;
  const fa_fwd_params &a = *p;
  if (a.B < 0 || a.Nq < 0 || a.Nk < 0 || a.Hq <= 0 || a.Hkv <= 0 || a.Hq % a.Hkv != 0)
    return FA_ERR_INVALID_ARG;
  if (a.dtype != FA_E4M3) return FA_ERR_UNSUPPORTED;
  if (a.d < 16 || a.d > 128 || a.d % 16 != 0) return FA_ERR_UNSUPPORTED;
  if (!scale_ok(a.scale)) return FA_ERR_INVALID_ARG;
  if (a.Nq > (1 << 30) || a.Nk > (1 << 30)) return FA_ERR_INVALID_ARG;
  if (a.B == 0 || a.Nq == 0) return FA_OK;
  if (a.q == nullptr || a.o == nullptr || a.lse == nullptr) return FA_ERR_INVALID_ARG;
  if (!aligned(a.q, 16) || !aligned(a.o, 16) || !aligned(a.lse, 4)) return FA_ERR_INVALID_ARG;
  for (const float *ds : {q_descale, k_descale, v_descale})
    if (ds != nullptr && !aligned(ds, 4)) return FA_ERR_INVALID_ARG;
  if (!stride_ok_16b(a.q_strides[0], a.B) || !stride_ok_16b(a.q_strides[1], a.Nq) ||
      !stride_ok_16b(a.q_strides[2], a.Hq) || !stride_ok(a.o_strides[0], a.B) ||
      !stride_ok(a.o_strides[1], a.Nq) || !stride_ok(a.o_strides[2], a.Hq))
    return FA_ERR_INVALID_ARG;
  if (a.Nk > 0) {
    if (a.k == nullptr || a.v == nullptr) return FA_ERR_INVALID_ARG;
    if (!aligned(a.k, 16) || !aligned(a.v, 16)) return FA_ERR_INVALID_ARG;
    if (!stride_ok_16b(a.k_strides[0], a.B) || !stride_ok_16b(a.k_strides[1], a.Nk) ||
        !stride_ok_16b(a.k_strides[2], a.Hkv) || !stride_ok_16b(a.v_strides[0], a.B) ||
        !stride_ok_16b(a.v_strides[1], a.Nk) || !stride_ok_16b(a.v_strides[2], a.Hkv))
      return FA_ERR_INVALID_ARG;
    const size_t need = fa_fwd_fp8_workspace_size(a.B, a.Nk, a.Hkv, a.d);
    if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256))
      return FA_ERR_WORKSPACE;
  }
  const int mblocks = ceil_div(a.Nq, fa::prefill_tile_rows(128));
  const int64_t tiles = static_cast<int64_t>(a.B) * a.Hq * mblocks;
  if (tiles > INT32_MAX) return FA_ERR_INVALID_ARG;
  ModPlan mod;
  fa_status st = plan_mod(&a.mod, a.causal, &mod);
  if (st != FA_OK) return st;

  DeviceInfo *dev = nullptr;
  st = current_device(&dev);
  if (st != FA_OK) return st;
  if (a.Nk == 0) {
    cudaError_t e = fa::launch_fill_empty(a.o, a.lse, a.B, a.Nq, a.Hq, a.d, a.o_strides[0],
                                          a.o_strides[1], a.o_strides[2],
                                          static_cast<int64_t>(a.Hq) * a.Nq, a.Nq, stream);
    return e == cudaSuccess ? FA_OK : cuda_fail("fill kernel launch", e);
  }
  const int nk_pad = static_cast<int>(nk_pad16(a.Nk));
  CUtensorMap tq, tk, tvt;
  if ((st = make_map(&tq, a.q, a.d, a.Nq, a.Hq, a.B, a.q_strides[1], a.q_strides[2],
                     a.q_strides[0], FA_E4M3)) != FA_OK)
    return st;
  if ((st = make_map(&tk, a.k, a.d, a.Nk, a.Hkv, a.B, a.k_strides[1], a.k_strides[2],
                     a.k_strides[0], FA_E4M3)) != FA_OK)
    return st;
  if ((st = make_map_vt(&tvt, workspace, nk_pad, a.d, a.Hkv, a.B)) != FA_OK) return st;
  cudaError_t e = fa::launch_transpose_v(a.v, a.v_strides[0], a.v_strides[1], a.v_strides[2],
                                         workspace, a.B, a.Nk, a.Hkv, a.d, nk_pad, stream);
  if (e != cudaSuccess) return cuda_fail("V transpose launch", e);
  fa::PrefillArgs pa = dense_args(a, mblocks, tiles, dev, mod, static_cast<int64_t>(a.Hq) * a.Nq,
                                  a.Nq);
  pa.q_descale = q_descale;
  pa.k_descale = k_descale;
  pa.v_descale = v_descale;
  const int grid = static_cast<int>(tiles < dev->sm_count ? tiles : dev->sm_count);
  CUtensorMap to;
  pa.o_tma = make_map(&to, a.o, a.d, a.Nq, a.Hq, a.B, a.o_strides[1], a.o_strides[2],
                      a.o_strides[0], FA_BF16, 32) == FA_OK;
  e = fa::launch_prefill_fp8(mod.mask, tq, tk, tvt, pa.o_tma ? &to : nullptr, pa, grid, stream);
  return e == cudaSuccess ? FA_OK : cuda_fail("prefill kernel launch", e);
}

// Columns of the varlen transposed V: sequence b's keys start at roundup16(cu_k[b]) + 16 b.
int64_t vt_cols_varlen(int B, int64_t total_k) { return nk_pad16(total_k) + 16 * (B + 1ll); }

size_t fa_fwd_varlen_fp8_workspace_size(int B, int total_k, int Hkv, int d) {
  if (B <= 0 || total_k <= 0 || Hkv <= 0 || d <= 0) return 0;
  const int64_t bytes = static_cast<int64_t>(Hkv) * d * vt_cols_varlen(B, total_k);
  return static_cast<size_t>((bytes + 255) / 256 * 256);
}

fa_status fa_fwd_varlen_fp8(const void *q, const void *k, const void *v, void *o, float *lse,
                            const int *cu_seqlens_q, const int *cu_seqlens_k, int B,
                            int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int Hq,
                            int Hkv, int d, float scale, int causal, const fa_score_mod *mod_in,
                            const float *q_descale, const float *k_descale,
                            const float *v_descale, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  if (B < 0 || B > 65535 || max_seqlen_q < 0 || max_seqlen_k < 0 || total_q < 0 ||
      total_k < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
    return FA_ERR_INVALID_ARG;
  if (d < 16 || d > 128 || d % 16 != 0) return FA_ERR_UNSUPPORTED;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  if (max_seqlen_q > (1 << 30) || total_q > (1 << 30) || total_k > (1 << 30))
    return FA_ERR_INVALID_ARG;
  if (B == 0 || total_q == 0 || max_seqlen_q == 0) return FA_OK;
  if (q == nullptr || o == nullptr || lse == nullptr || cu_seqlens_q == nullptr ||
      cu_seqlens_k == nullptr)
    return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(lse, 4) || !aligned(cu_seqlens_q, 4) ||
      !aligned(cu_seqlens_k, 4))
    return FA_ERR_INVALID_ARG;
  for (const float *ds : {q_descale, k_descale, v_descale})
    if (ds != nullptr && !aligned(ds, 4)) return FA_ERR_INVALID_ARG;
  if (total_k > 0) {
    if (k == nullptr || v == nullptr || !aligned(k, 16) || !aligned(v, 16))
      return FA_ERR_INVALID_ARG;
    const size_t need = fa_fwd_varlen_fp8_workspace_size(B, total_k, Hkv, d);
    if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256))
      return FA_ERR_WORKSPACE;
  }
  const int mblocks = ceil_div(max_seqlen_q, fa::prefill_tile_rows(128));
  const int64_t tiles = static_cast<int64_t>(B) * Hq * mblocks;
  if (tiles > INT32_MAX) return FA_ERR_INVALID_ARG;
  ModPlan mod;
  fa_status st = plan_mod(mod_in, causal, &mod);
  if (st != FA_OK) return st;

  DeviceInfo *dev = nullptr;
  st = current_device(&dev);
  if (st != FA_OK) return st;
  if (total_k == 0) {
    cudaError_t e = fa::launch_fill_empty(o, lse, 1, total_q, Hq, d, 0,
                                          static_cast<int64_t>(Hq) * d, d, 0, total_q, stream);
    return e == cudaSuccess ? FA_OK : cuda_fail("fill kernel launch", e);
  }
  const int64_t nt = vt_cols_varlen(B, total_k);
  if (nt > INT32_MAX) return FA_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tvt;
  if ((st = make_map(&tq, q, d, total_q, Hq, 1, static_cast<int64_t>(Hq) * d, d, 0,
                     FA_E4M3)) != FA_OK ||
      (st = make_map(&tk, k, d, total_k, Hkv, 1, static_cast<int64_t>(Hkv) * d, d, 0,
                     FA_E4M3)) != FA_OK ||
      (st = make_map_vt(&tvt, workspace, static_cast<int>(nt), d, Hkv, 1)) != FA_OK)
    return st;
  cudaError_t e = fa::launch_transpose_v_varlen(v, workspace, cu_seqlens_k, B, max_seqlen_k,
                                                total_k, Hkv, d, static_cast<int>(nt), stream);
  if (e != cudaSuccess) return cuda_fail("V transpose launch", e);
  fa::PrefillArgs pa = varlen_args(o, lse, cu_seqlens_q, cu_seqlens_k, B, max_seqlen_q,
                                   max_seqlen_k, total_q, total_k, Hq, Hkv, d, scale, mblocks,
                                   tiles, dev, mod);
  pa.q_descale = q_descale;
  pa.k_descale = k_descale;
  pa.v_descale = v_descale;
  const int grid = static_cast<int>(tiles < dev->sm_count ? tiles : dev->sm_count);
  CUtensorMap to;
  pa.o_tma = make_map(&to, o, d, total_q, Hq, 1, static_cast<int64_t>(Hq) * d, d, 0, FA_BF16,
                      32) == FA_OK;
  e = fa::launch_prefill_fp8(mod.mask, tq, tk, tvt, pa.o_tma ? &to : nullptr, pa, grid, stream);
  return e == cudaSuccess ? FA_OK : cuda_fail("prefill kernel launch", e);
}

// Copy streams and events of fa_fwd_host on this device (created once).
fa_status host_resources(DeviceInfo *dev) {
  if (dev->host_ready) return FA_OK;
  cudaError_t e;
  if ((e = cudaStreamCreateWithFlags(&dev->h2d, cudaStreamNonBlocking)) != cudaSuccess ||
      (e = cudaStreamCreateWithFlags(&dev->d2h, cudaStreamNonBlocking)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&dev->ev_start, cudaEventDisableTiming)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&dev->ev_end, cudaEventDisableTiming)) != cudaSuccess)
    return cuda_fail("fa_fwd_host stream / event creation", e);
  for (int i = 0; i < kMaxHostRanges; ++i)
    if ((e = cudaEventCreateWithFlags(&dev->ev_in[i], cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&dev->ev_out[i], cudaEventDisableTiming)) != cudaSuccess)
      return cuda_fail("fa_fwd_host event creation", e);
  dev->host_ready = true;
  return FA_OK;
}

bool contiguous4(const int64_t s[3], int64_t n, int64_t h, int64_t d) {
  return s[2] == d && s[1] == h * d && s[0] == n * h * d;
}

fa_status fa_fwd_host(const fa_fwd_params *p, void *dev_q, void *dev_k, void *dev_v,
                      void *dev_o, float *dev_lse, int chunks, cudaStream_t stream) {
  if (p == nullptr) return FA_ERR_INVALID_ARG;
  const fa_fwd_params &a = *p;
  if (a.B < 0 || a.Nq < 0 || a.Nk < 0 || a.Hq <= 0 || a.Hkv <= 0 || a.Hq % a.Hkv != 0)
    return FA_ERR_INVALID_ARG;
  if (!head_dim_ok(a.d, kMaxPrefillD)) return FA_ERR_UNSUPPORTED;
  if (!dtype_ok(a.dtype)) return FA_ERR_UNSUPPORTED;
  if (!scale_ok(a.scale)) return FA_ERR_INVALID_ARG;
  if (a.Nq > (1 << 30) || a.Nk > (1 << 30)) return FA_ERR_INVALID_ARG;
  if (chunks < 1 || chunks > 64) return FA_ERR_INVALID_ARG;
  if (a.B == 0 || a.Nq == 0) return FA_OK;
  if (a.q == nullptr || a.o == nullptr || a.lse == nullptr || dev_q == nullptr ||
      dev_o == nullptr || dev_lse == nullptr)
    return FA_ERR_INVALID_ARG;
  if (a.Nk > 0 && (a.k == nullptr || a.v == nullptr || dev_k == nullptr || dev_v == nullptr))
    return FA_ERR_INVALID_ARG;
  if (!aligned(dev_q, 16) || !aligned(dev_o, 16) || !aligned(dev_lse, 4) ||
      (a.Nk > 0 && (!aligned(dev_k, 16) || !aligned(dev_v, 16))))
    return FA_ERR_INVALID_ARG;
  // Host and device tensors share the contiguous layout, so that a (batch, row range)
  // piece is one contiguous byte range.
  if (!contiguous4(a.q_strides, a.Nq, a.Hq, a.d) || !contiguous4(a.o_strides, a.Nq, a.Hq, a.d) ||
      !contiguous4(a.k_strides, a.Nk, a.Hkv, a.d) || !contiguous4(a.v_strides, a.Nk, a.Hkv, a.d))
    return FA_ERR_INVALID_ARG;
  ModPlan mod;
  fa_status st = plan_mod(&a.mod, a.causal, &mod);
  if (st != FA_OK) return st;
  // Row ranges need a key prefix that ends at their last row's position: only when no row
  // sees keys past its own position (causal, or a right window bound of 0).  Otherwise the
  // pieces are whole batch entries.
  const bool prefix = mod.wr == 0;
  const int per_b = prefix ? std::min<int64_t>(chunks, ceil_div(a.Nq, 128)) : 1;
  if (static_cast<int64_t>(a.B) * per_b > kMaxHostRanges) return FA_ERR_INVALID_ARG;

  DeviceInfo *dev = nullptr;
  st = current_device(&dev);
  if (st != FA_OK) return st;
  std::lock_guard<std::mutex> lock(dev->host_mutex);
  if ((st = host_resources(dev)) != FA_OK) return st;
  const int64_t es = 2;
  const int64_t qrow = static_cast<int64_t>(a.Hq) * a.d * es;   // bytes per token row
  const int64_t krow = static_cast<int64_t>(a.Hkv) * a.d * es;
  cudaError_t e;
  // The copies start after earlier work on the caller's stream (it may still use the
  // device buffers).
  if ((e = cudaEventRecord(dev->ev_start, stream)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(dev->h2d, dev->ev_start, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(dev->d2h, dev->ev_start, 0)) != cudaSuccess)
    return cuda_fail("fa_fwd_host ordering", e);
  int piece = 0;
  for (int b = 0; b < a.B; ++b) {
    int64_t k_done = 0;  // keys of batch entry b already copied
    for (int c = 0; c < per_b; ++c, ++piece) {
      // rows [r0, r1): query blocks split evenly (128-row granularity)
      const int64_t nblk = ceil_div(a.Nq, 128);
      const int64_t r0 = std::min<int64_t>(a.Nq, (nblk * c / per_b) * 128);
      const int64_t r1 = std::min<int64_t>(a.Nq, (nblk * (c + 1) / per_b) * 128);
      if (r1 <= r0) {
        // empty range: keep the piece's events in order
        if ((e = cudaEventRecord(dev->ev_in[piece], dev->h2d)) != cudaSuccess ||
            (e = cudaEventRecord(dev->ev_out[piece], stream)) != cudaSuccess)
          return cuda_fail("fa_fwd_host events", e);
        continue;
      }
      // key prefix of the range: positions up to the last row's (bottom-right alignment)
      const int64_t k_end = prefix ? std::max<int64_t>(0, std::min<int64_t>(a.Nk, r1 + a.Nk - a.Nq))
                                   : a.Nk;
      const int64_t qoff = (static_cast<int64_t>(b) * a.Nq + r0) * qrow;
      const int64_t koff = (static_cast<int64_t>(b) * a.Nk + k_done) * krow;
      if ((e = cudaMemcpyAsync(static_cast<char *>(dev_q) + qoff,
                               static_cast<const char *>(a.q) + qoff, (r1 - r0) * qrow,
                               cudaMemcpyHostToDevice, dev->h2d)) != cudaSuccess)
        return cuda_fail("fa_fwd_host Q copy", e);
      if (k_end > k_done) {
        if ((e = cudaMemcpyAsync(static_cast<char *>(dev_k) + koff,
                                 static_cast<const char *>(a.k) + koff, (k_end - k_done) * krow,
                                 cudaMemcpyHostToDevice, dev->h2d)) != cudaSuccess ||
            (e = cudaMemcpyAsync(static_cast<char *>(dev_v) + koff,
                                 static_cast<const char *>(a.v) + koff, (k_end - k_done) * krow,
                                 cudaMemcpyHostToDevice, dev->h2d)) != cudaSuccess)
          return cuda_fail("fa_fwd_host K/V copy", e);
        k_done = k_end;
      }
      if ((e = cudaEventRecord(dev->ev_in[piece], dev->h2d)) != cudaSuccess ||
          (e = cudaStreamWaitEvent(stream, dev->ev_in[piece], 0)) != cudaSuccess)
        return cuda_fail("fa_fwd_host ordering", e);
      // the range as its own problem: rows [r0, r1) of batch entry b over keys [0, k_end)
      fa_fwd_params r = a;
      r.B = 1;
      r.Nq = static_cast<int>(r1 - r0);
      r.Nk = static_cast<int>(k_end);
      r.q = static_cast<const char *>(dev_q) + qoff;
      r.o = static_cast<char *>(dev_o) + qoff;
      r.k = static_cast<const char *>(dev_k) + static_cast<int64_t>(b) * a.Nk * krow;
      r.v = static_cast<const char *>(dev_v) + static_cast<int64_t>(b) * a.Nk * krow;
      r.lse = dev_lse + static_cast<int64_t>(b) * a.Hq * a.Nq + r0;
      ModPlan rmod = mod;
      if (rmod.alibi != nullptr) rmod.alibi += static_cast<int64_t>(b) * rmod.alibi_sb;
      if ((st = launch_dense(r, dev, rmod, static_cast<int64_t>(a.Hq) * a.Nq, a.Nq, stream)) !=
          FA_OK)
        return st;
      if ((e = cudaEventRecord(dev->ev_out[piece], stream)) != cudaSuccess ||
          (e = cudaStreamWaitEvent(dev->d2h, dev->ev_out[piece], 0)) != cudaSuccess)
        return cuda_fail("fa_fwd_host ordering", e);
      if ((e = cudaMemcpyAsync(static_cast<char *>(a.o) + qoff,
                               static_cast<const char *>(dev_o) + qoff, (r1 - r0) * qrow,
                               cudaMemcpyDeviceToHost, dev->d2h)) != cudaSuccess)
        return cuda_fail("fa_fwd_host O copy", e);
      // LSE rows [r0, r1) of every head: Hq rows of (r1 - r0) floats, pitch Nq floats
      const size_t pitch = static_cast<size_t>(a.Nq) * sizeof(float);
      const int64_t loff = static_cast<int64_t>(b) * a.Hq * a.Nq + r0;
      if ((e = cudaMemcpy2DAsync(a.lse + loff, pitch, dev_lse + loff, pitch,
                                 static_cast<size_t>(r1 - r0) * sizeof(float), a.Hq,
                                 cudaMemcpyDeviceToHost, dev->d2h)) != cudaSuccess)
        return cuda_fail("fa_fwd_host LSE copy", e);
    }
  }
  // Later work on the caller's stream sees the outputs in host memory.
  if ((e = cudaEventRecord(dev->ev_end, dev->d2h)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(stream, dev->ev_end, 0)) != cudaSuccess)
    return cuda_fail("fa_fwd_host ordering", e);
  return FA_OK;
}

fa_status fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                        const int *cu_seqlens_q, const int *cu_seqlens_k, int B,
                        int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int Hq,
                        int Hkv, int d, float scale, int causal, int dtype,
                        const fa_score_mod *mod_in, cudaStream_t stream) {
  if (B < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || total_q < 0 || total_k < 0 || Hq <= 0 ||
      Hkv <= 0 || Hq % Hkv != 0)
    return FA_ERR_INVALID_ARG;
  if (!head_dim_ok(d, kMaxPrefillD)) return FA_ERR_UNSUPPORTED;
  if (!dtype_ok(dtype)) return FA_ERR_UNSUPPORTED;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  if (max_seqlen_q > (1 << 30) || total_q > (1 << 30) || total_k > (1 << 30))
    return FA_ERR_INVALID_ARG;
  if (B == 0 || total_q == 0 || max_seqlen_q == 0) return FA_OK;
  if (q == nullptr || o == nullptr || lse == nullptr || cu_seqlens_q == nullptr ||
      cu_seqlens_k == nullptr)
    return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(lse, 4) || !aligned(cu_seqlens_q, 4) ||
      !aligned(cu_seqlens_k, 4))
    return FA_ERR_INVALID_ARG;
  if (total_k > 0 && (k == nullptr || v == nullptr || !aligned(k, 16) || !aligned(v, 16)))
    return FA_ERR_INVALID_ARG;
  const bool pairs = use_pairs(d);
  const int mblocks = ceil_div(max_seqlen_q, tile_rows(d, pairs));
  const int64_t tiles = static_cast<int64_t>(B) * Hq * mblocks;
  if (tiles > INT32_MAX) return FA_ERR_INVALID_ARG;
  ModPlan mod;
  fa_status st = plan_mod(mod_in, causal, &mod);
  if (st != FA_OK) return st;

  DeviceInfo *dev = nullptr;
  st = current_device(&dev);
  if (st != FA_OK) return st;
  const int64_t o_sn = static_cast<int64_t>(Hq) * d, o_sh = d;
  if (total_k == 0) {
    cudaError_t e = fa::launch_fill_empty(o, lse, 1, total_q, Hq, d, 0, o_sn, o_sh, 0, total_q,
                                          stream);
    return e == cudaSuccess ? FA_OK : cuda_fail("fill kernel launch", e);
  }
  CUtensorMap tq, tk, tv;
  if ((st = make_map(&tq, q, d, total_q, Hq, 1, static_cast<int64_t>(Hq) * d, d, 0, dtype)) !=
      FA_OK)
    return st;
  if ((st = make_map(&tk, k, d, total_k, Hkv, 1, static_cast<int64_t>(Hkv) * d, d, 0, dtype,
                     pairs ? 64 : 128)) != FA_OK)
    return st;
  if ((st = make_map(&tv, v, d, total_k, Hkv, 1, static_cast<int64_t>(Hkv) * d, d, 0, dtype)) !=
      FA_OK)
    return st;
  fa::PrefillArgs pa = varlen_args(o, lse, cu_seqlens_q, cu_seqlens_k, B, max_seqlen_q,
                                   max_seqlen_k, total_q, total_k, Hq, Hkv, d, scale, mblocks,
                                   tiles, dev, mod);
  cudaError_t e;
  if (pairs) {
    e = fa::launch_prefill_pair(mod.mask, dtype == FA_FP16, tq, tk, tv, pa,
                                static_cast<int>(tiles), stream);
  } else {
    const int grid = static_cast<int>(tiles < dev->sm_count ? tiles : dev->sm_count);
    CUtensorMap to;
    pa.o_tma = make_map(&to, o, d, total_q, Hq, 1, o_sn, o_sh, 0, dtype, 32) == FA_OK;
    e = fa::launch_prefill(fa::kernel_d(d), mod.mask, dtype == FA_FP16, tq, tk, tv,
                           pa.o_tma ? &to : nullptr, pa, grid, stream);
  }
  return e == cudaSuccess ? FA_OK : cuda_fail("prefill kernel launch", e);
}

size_t fa_fwd_kvcache_workspace_size(int B, int Hq, int Lmax, int d, int num_splits) {
  if (B <= 0 || Hq <= 0 || Lmax <= 0 || d <= 0 || num_splits < 0) return 0;
  const int chunk = decode_chunk(Lmax, num_splits);
  const int64_t maxch = (static_cast<int64_t>(Lmax) + chunk - 1) / chunk;
  const int64_t bytes = static_cast<int64_t>(B) * Hq * maxch * (fa::kernel_d(d) + 1) * 4;
  return static_cast<size_t>((bytes + 255) / 256 * 256);
}

}  // extern "C"

namespace {

// Decode over 16-bit caches (kv_e4m3 false) or E4M3 caches with descale factors per
// (batch, kv head) and a bf16 query (kv_e4m3 true; no append or rotary).
fa_status kvcache_call(const void *q, const void *k_cache, const void *v_cache,
                       const int *cache_seqlens, int B, int Lmax, int Hq, int Hkv, int d,
                       const int64_t cache_strides[3], float scale, int num_splits,
                       void *workspace, size_t workspace_bytes, void *o, float *lse, int dtype,
                       const fa_score_mod *mod_in, const fa_kvcache_extras *ex, bool kv_e4m3,
                       const float *k_descale, const float *v_descale, cudaStream_t stream) {
  if (B < 0 || Lmax < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || num_splits < 0)
    return FA_ERR_INVALID_ARG;
  if (!head_dim_ok(d, kMaxDecodeD)) return FA_ERR_UNSUPPORTED;
  if (kv_e4m3 && (d < 16 || d % 16 != 0)) return FA_ERR_UNSUPPORTED;
  // The query heads of one kv head (any group size) run as nsplit work items of G heads,
  // G the largest of 8, 4, 2, 1 that divides the group (at most 4 at width 256, where more
  // heads' state would spill).  The items of one kv head stream the same K/V rows at about
  // the same time, so the repeated reads are mostly served by L2.
  const int group = Hq / Hkv;
  const int kd = kv_e4m3 ? fa::kernel_d_e4m3(d) : fa::kernel_d(d);
  int G = kd == 256 ? 4 : 8;
  while (group % G != 0) G /= 2;
  const int nsplit = group / G;
  if (!dtype_ok(dtype) || (kv_e4m3 && dtype != FA_BF16)) return FA_ERR_UNSUPPORTED;
  if (!aligned(k_descale, 4) || !aligned(v_descale, 4)) return FA_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  if (Lmax > (1 << 30)) return FA_ERR_INVALID_ARG;
  if (B == 0) return FA_OK;
  if (q == nullptr || o == nullptr || lse == nullptr || cache_seqlens == nullptr)
    return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(lse, 4) || !aligned(cache_seqlens, 4))
    return FA_ERR_INVALID_ARG;
  int chunk = 128, maxch = 0;
  float *o_part = nullptr, *lse_part = nullptr;
  ModPlan mod;
  fa_status st = plan_mod(mod_in, 0, &mod);  // the right bound never hides a cached key
  if (st != FA_OK) return st;
  const bool append = ex != nullptr && (ex->k_new != nullptr || ex->v_new != nullptr);
  const bool rotary = ex != nullptr && (ex->rotary_cos != nullptr || ex->rotary_sin != nullptr);
  const bool paged = ex != nullptr && ex->block_table != nullptr;
  if (kv_e4m3 && (append || rotary)) return FA_ERR_UNSUPPORTED;
  if (append) {
    if (ex->k_new == nullptr || ex->v_new == nullptr || Lmax == 0) return FA_ERR_INVALID_ARG;
    if (!aligned(ex->k_new, 2) || !aligned(ex->v_new, 2)) return FA_ERR_INVALID_ARG;
    if (ex->new_strides[0] < 0 || ex->new_strides[2] < 0) return FA_ERR_INVALID_ARG;
  }
  if (rotary) {
    if (!append || ex->rotary_cos == nullptr || ex->rotary_sin == nullptr)
      return FA_ERR_INVALID_ARG;
    if (ex->rotary_dim < 2 || ex->rotary_dim > d || (ex->rotary_dim & 1) ||
        ex->rotary_positions < 1 || !aligned(ex->rotary_cos, 4) || !aligned(ex->rotary_sin, 4))
      return FA_ERR_INVALID_ARG;
    if (o == q) return FA_ERR_INVALID_ARG;  // the rotated query is staged in o
  }
  int num_rows = Lmax, num_outer = B;  // extents of the cache tensors: (row, batch or page)
  if (paged) {
    if (ex->page_size <= 0 || ex->page_size % 128 != 0 || ex->num_pages < 1 ||
        !aligned(ex->block_table, 4) ||
        static_cast<int64_t>(ex->block_table_stride) * ex->page_size < Lmax)
      return FA_ERR_INVALID_ARG;
    num_rows = ex->page_size;
    num_outer = ex->num_pages;
  }
  if (Lmax > 0) {
    if (k_cache == nullptr || v_cache == nullptr || cache_strides == nullptr)
      return FA_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return FA_ERR_INVALID_ARG;
    if (!stride_ok(cache_strides[0], num_outer) || !stride_ok(cache_strides[1], num_rows) ||
        !stride_ok(cache_strides[2], Hkv))
      return FA_ERR_INVALID_ARG;
    const size_t need = fa_fwd_kvcache_workspace_size(B, Hq, Lmax, d, num_splits);
    if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256))
      return FA_ERR_WORKSPACE;
  }

  DeviceInfo *dev = nullptr;
  st = current_device(&dev);
  if (st != FA_OK) return st;
  if (Lmax > 0) {
    chunk = decode_chunk(Lmax, num_splits);
    maxch = ceil_div(Lmax, chunk);  // the workspace holds this many chunks per (b, h)
    // A window limits every sequence to its last wl + 1 keys: the chunks split that range.
    // (with page-aligned unit starts the range may begin up to 127 keys earlier)
    const int kalign = paged ? 128 : 1;
    const int Leff = mod.wl >= 0 ? std::min<int64_t>(Lmax, static_cast<int64_t>(mod.wl) + kalign)
                                 : Lmax;
    if (num_splits == 0)
      chunk = auto_chunk(Leff, static_cast<int64_t>(B) * Hkv * nsplit, dev->sm_count, maxch,
                         kv_e4m3);
    maxch = ceil_div(Leff, chunk);
    o_part = static_cast<float *>(workspace);
    lse_part = o_part + static_cast<int64_t>(B) * Hq * maxch * fa::kernel_d(d);
  }
  const int64_t units = static_cast<int64_t>(maxch) * B * Hkv * nsplit;
  if (units > INT32_MAX) return FA_ERR_INVALID_ARG;
  if (Lmax > 0) {
    CUtensorMap tk, tv;
    const int kv_type = kv_e4m3 ? FA_E4M3 : dtype;
    if ((st = make_map(&tk, k_cache, d, num_rows, Hkv, num_outer, cache_strides[1],
                       cache_strides[2], cache_strides[0], kv_type)) != FA_OK)
      return st;
    if ((st = make_map(&tv, v_cache, d, num_rows, Hkv, num_outer, cache_strides[1],
                       cache_strides[2], cache_strides[0], kv_type)) != FA_OK)
      return st;
    if (append) {
      fa::AppendArgs ap{};
      ap.k_new = ex->k_new;
      ap.v_new = ex->v_new;
      ap.n_sb = ex->new_strides[0];
      ap.n_sh = ex->new_strides[2];
      ap.k_cache = const_cast<void *>(k_cache);
      ap.v_cache = const_cast<void *>(v_cache);
      ap.c_s0 = cache_strides[0];
      ap.c_s1 = cache_strides[1];
      ap.c_s2 = cache_strides[2];
      ap.cache_len = cache_seqlens;
      ap.B = B;
      ap.Hq = Hq;
      ap.Hkv = Hkv;
      ap.d = d;
      ap.Lmax = Lmax;
      ap.block_table = paged ? ex->block_table : nullptr;
      ap.bt_stride = paged ? ex->block_table_stride : 0;
      ap.page_size = paged ? ex->page_size : 1;
      ap.num_pages = paged ? ex->num_pages : 0;
      ap.cos = rotary ? ex->rotary_cos : nullptr;
      ap.sin = rotary ? ex->rotary_sin : nullptr;
      ap.rot_dim = rotary ? ex->rotary_dim : 0;
      ap.rot_positions = rotary ? ex->rotary_positions : 0;
      ap.rot_interleaved = rotary ? ex->rotary_interleaved != 0 : 0;
      ap.q = q;
      ap.q_rot = rotary ? o : nullptr;
      ap.err = dev->err;
      cudaError_t e = fa::launch_append(dtype == FA_FP16, ap, stream);
      if (e != cudaSuccess) return cuda_fail("append kernel launch", e);
    }
    fa::DecodeArgs da{};
    da.q = rotary ? o : q;
    da.cache_len = cache_seqlens;
    da.o_part = o_part;
    da.lse_part = lse_part;
    da.B = B;
    da.Hq = Hq;
    da.Hkv = Hkv * nsplit;
    da.nsplit = nsplit;
    da.Lmax = Lmax;
    da.chunk = chunk;
    da.maxch = maxch;
    da.d = d;
    da.num_units = static_cast<int>(units);
    da.sched_slot = fa::next_decode_sched_slot();
    da.scale_log2 = scale_log2(scale);
    da.err = dev->err;
    da.timeout_ns = g_timeout_ns;
    da.inject = g_inject;
    da.wl = mod.wl;
    // the score arrives as scale * q.k * log2(e): softcap * tanh(z / softcap) * log2(e)
    da.sc_in = mod.softcap > 0.f
                   ? static_cast<float>(1.0 / (mod.softcap * 1.4426950408889634))
                   : 0.f;
    da.sc_out = mod.softcap > 0.f ? static_cast<float>(mod.softcap * 1.4426950408889634) : 0.f;
    da.alibi = mod.alibi;
    da.alibi_sb = mod.alibi_sb;
    da.len_add = append ? 1 : 0;
    da.block_table = paged ? ex->block_table : nullptr;
    da.bt_stride = paged ? ex->block_table_stride : 0;
    da.page_size = paged ? ex->page_size : 1;
    da.num_pages = paged ? ex->num_pages : 0;
    da.kalign = paged ? 128 : 1;
    da.k_descale = kv_e4m3 ? k_descale : nullptr;
    da.v_descale = kv_e4m3 ? v_descale : nullptr;
    da.ostride = fa::kernel_d(d);
    const int grid = static_cast<int>(units < dev->sm_count ? units : dev->sm_count);
    cudaError_t e = fa::launch_decode(kd, G, dtype == FA_FP16, kv_e4m3, tk, tv,
                                      da, grid, stream);
    if (e != cudaSuccess) return cuda_fail("decode kernel launch", e);
  }
  cudaError_t e = fa::launch_combine(fa::kernel_d(d), d, dtype == FA_FP16, o_part, lse_part,
                                     cache_seqlens,
                                     append ? 1 : 0, B, Hq, Lmax, chunk, maxch, mod.wl,
                                     paged ? 128 : 1, o, lse, dev->err, stream);
  return e == cudaSuccess ? FA_OK : cuda_fail("combine kernel launch", e);
}

}  // namespace

extern "C" {

fa_status fa_fwd_kvcache(const void *q, const void *k_cache, const void *v_cache,
                         const int *cache_seqlens, int B, int Lmax, int Hq, int Hkv, int d,
                         const int64_t cache_strides[3], float scale, int num_splits,
                         void *workspace, size_t workspace_bytes, void *o, float *lse,
                         int dtype, const fa_score_mod *mod_in, const fa_kvcache_extras *ex,
                         cudaStream_t stream) {
  return kvcache_call(q, k_cache, v_cache, cache_seqlens, B, Lmax, Hq, Hkv, d, cache_strides,
                      scale, num_splits, workspace, workspace_bytes, o, lse, dtype, mod_in, ex,
                      false, nullptr, nullptr, stream);
}

fa_status fa_fwd_kvcache_fp8(const void *q, const void *k_cache, const void *v_cache,
                             const int *cache_seqlens, int B, int Lmax, int Hq, int Hkv, int d,
                             const int64_t cache_strides[3], float scale, int num_splits,
                             const float *k_descale, const float *v_descale, void *workspace,
                             size_t workspace_bytes, void *o, float *lse,
                             const fa_score_mod *mod_in, const fa_kvcache_extras *ex,
                             cudaStream_t stream) {
  return kvcache_call(q, k_cache, v_cache, cache_seqlens, B, Lmax, Hq, Hkv, d, cache_strides,
                      scale, num_splits, workspace, workspace_bytes, o, lse, FA_BF16, mod_in, ex,
                      true, k_descale, v_descale, stream);
}

// (batch, kv head) pairs whose backward units run interleaved.  Few pairs keep the dQ
// accumulators that CTAs add into at the same time in L2; the deterministic order wants
// more, since CTAs on the same pair wait for one another's additions in key-block order.
// Measured on the causal N = 8192 backward (TFLOPS, groups 4 / 8 / 16): d = 128 1021 /
// 1035 / 998, deterministic 573 / 711 / 784; d = 256 592 / 573 / 567, deterministic
// 422 / 459 / 470.
static int bwd_head_group(bool deterministic, bool wide) {
  if (deterministic) return 16;
  return wide ? 4 : 8;
}

size_t fa_bwd_params_size(void) { return sizeof(fa_bwd_params); }

// Workspace of fa_bwd: the fp32 dQ accumulator, D [B, Hq, Nq], and the counters of the
// deterministic order (bwd_acc_elems, bwd_sem_elems), each part 256-byte aligned.
size_t fa_bwd_workspace_size(int B, int Nq, int Hq, int d) {
  if (B <= 0 || Nq <= 0 || Hq <= 0 || d <= 0) return 0;
  const int64_t acc = bwd_acc_elems(B, Nq, Hq, d) * 4;
  const int64_t vec = static_cast<int64_t>(B) * Hq * Nq * 4;
  const int64_t sem = bwd_sem_elems(B, Nq, Hq, d) * 4;
  return static_cast<size_t>((acc + 255) / 256 * 256 + (vec + 255) / 256 * 256 +
                             (sem + 255) / 256 * 256);
}

fa_status fa_bwd(const fa_bwd_params *p, cudaStream_t stream) {
  if (p == nullptr) return FA_ERR_INVALID_ARG;
  const fa_bwd_params &a = *p;
  if (a.B < 0 || a.Nq < 0 || a.Nk < 0 || a.Hq <= 0 || a.Hkv <= 0 || a.Hq % a.Hkv != 0)
    return FA_ERR_INVALID_ARG;
  if (!head_dim_ok(a.d, kMaxPrefillD)) return FA_ERR_UNSUPPORTED;
  if (!dtype_ok(a.dtype)) return FA_ERR_UNSUPPORTED;
  if (!scale_ok(a.scale)) return FA_ERR_INVALID_ARG;
  if (a.Nq > (1 << 30) || a.Nk > (1 << 30)) return FA_ERR_INVALID_ARG;
  if (a.B == 0 || (a.Nq == 0 && a.Nk == 0)) return FA_OK;
  const bool q_side = a.Nq > 0, k_side = a.Nk > 0;
  if (q_side) {
    if (a.q == nullptr || a.o == nullptr || a.dout == nullptr || a.dq == nullptr ||
        a.lse == nullptr)
      return FA_ERR_INVALID_ARG;
    if (!aligned(a.q, 16) || !aligned(a.o, 16) || !aligned(a.dout, 16) || !aligned(a.dq, 16) ||
        !aligned(a.lse, 4))
      return FA_ERR_INVALID_ARG;
    for (const int64_t *st : {a.q_strides, a.o_strides, a.do_strides, a.dq_strides})
      if (!stride_ok(st[0], a.B) || !stride_ok(st[1], a.Nq) || !stride_ok(st[2], a.Hq))
        return FA_ERR_INVALID_ARG;
  }
  if (k_side) {
    if (a.k == nullptr || a.v == nullptr || a.dk == nullptr || a.dv == nullptr)
      return FA_ERR_INVALID_ARG;
    if (!aligned(a.k, 16) || !aligned(a.v, 16) || !aligned(a.dk, 16) || !aligned(a.dv, 16))
      return FA_ERR_INVALID_ARG;
    for (const int64_t *st : {a.k_strides, a.v_strides, a.dk_strides, a.dv_strides})
      if (!stride_ok(st[0], a.B) || !stride_ok(st[1], a.Nk) || !stride_ok(st[2], a.Hkv))
        return FA_ERR_INVALID_ARG;
  }
  const size_t need = fa_bwd_workspace_size(a.B, a.Nq, a.Hq, a.d);
  if (q_side && k_side &&
      (a.workspace == nullptr || a.workspace_bytes < need || !aligned(a.workspace, 256)))
    return FA_ERR_WORKSPACE;
  ModPlan mod;
  fa_status mst = plan_mod(&a.mod, a.causal, &mod);
  if (mst != FA_OK) return mst;
  const bool wide = fa::kernel_d(a.d) == 256;  // units per d half, 64-query steps
  const int kblocks = ceil_div(a.Nk, 128);
  const int64_t units = static_cast<int64_t>(kblocks) * a.B * a.Hkv * (wide ? 2 : 1);
  if (units > INT32_MAX) return FA_ERR_INVALID_ARG;

  DeviceInfo *dev = nullptr;
  fa_status st = current_device(&dev);
  if (st != FA_OK) return st;
  cudaError_t e;
  if (!k_side) {  // no keys: dQ = 0
    e = fa::launch_zero16(a.dq, a.B, a.Nq, a.Hq, a.d, a.dq_strides, stream);
    return e == cudaSuccess ? FA_OK : cuda_fail("zero kernel launch", e);
  }
  if (!q_side) {  // no queries: dK = dV = 0
    e = fa::launch_zero16(a.dk, a.B, a.Nk, a.Hkv, a.d, a.dk_strides, stream);
    if (e == cudaSuccess) e = fa::launch_zero16(a.dv, a.B, a.Nk, a.Hkv, a.d, a.dv_strides, stream);
    return e == cudaSuccess ? FA_OK : cuda_fail("zero kernel launch", e);
  }
  float *dq_acc = static_cast<float *>(a.workspace);
  const int64_t acc_n = bwd_acc_elems(a.B, a.Nq, a.Hq, a.d);
  const int64_t acc_bytes = (acc_n * 4 + 255) / 256 * 256;
  float *dvec = reinterpret_cast<float *>(static_cast<char *>(a.workspace) + acc_bytes);
  const int64_t vec_bytes = (static_cast<int64_t>(a.B) * a.Hq * a.Nq * 4 + 255) / 256 * 256;
  int *sem = reinterpret_cast<int *>(static_cast<char *>(a.workspace) + acc_bytes + vec_bytes);
  const int nsem = a.deterministic ? static_cast<int>(bwd_sem_elems(a.B, a.Nq, a.Hq, a.d)) : 0;
  const int nq_pad = fa::dq_acc_nq(a.Nq);
  const int qrows = wide ? 64 : 128;  // Q / dO box rows: the kernel's query step
  CUtensorMap tq, tk, tv, tdo, tdq;
  if ((st = make_map(&tq, a.q, a.d, a.Nq, a.Hq, a.B, a.q_strides[1], a.q_strides[2],
                     a.q_strides[0], a.dtype, qrows)) != FA_OK ||
      (st = make_map(&tdo, a.dout, a.d, a.Nq, a.Hq, a.B, a.do_strides[1], a.do_strides[2],
                     a.do_strides[0], a.dtype, qrows)) != FA_OK ||
      (st = make_map(&tk, a.k, a.d, a.Nk, a.Hkv, a.B, a.k_strides[1], a.k_strides[2],
                     a.k_strides[0], a.dtype)) != FA_OK ||
      (st = make_map(&tv, a.v, a.d, a.Nk, a.Hkv, a.B, a.v_strides[1], a.v_strides[2],
                     a.v_strides[0], a.dtype)) != FA_OK ||
      (st = wide ? make_map_dqt(&tdq, dq_acc, a.d, nq_pad, a.Hq, a.B)
                 : make_map_f32(&tdq, dq_acc, a.d, a.Nq, a.Hq, a.B)) != FA_OK)
    return st;
  const bool f16 = a.dtype == FA_FP16;
  e = fa::launch_bwd_pre(a.d, f16, a.o, a.dout, a.B, a.Nq, a.Hq, a.o_strides, a.do_strides, dvec,
                         dq_acc, acc_n, sem, nsem, stream);
  if (e != cudaSuccess) return cuda_fail("backward preprocessing launch", e);
  fa::BwdArgs ba{};
  ba.lse = a.lse;
  ba.dvec = dvec;
  ba.lse_sb = static_cast<int64_t>(a.Hq) * a.Nq;
  ba.lse_sh = a.Nq;
  ba.varlen = 0;
  ba.qblocks = ceil_div(a.Nq, wide ? 64 : 128);
  ba.dk = a.dk;
  ba.dv = a.dv;
  ba.dk_sb = a.dk_strides[0];
  ba.dk_sn = a.dk_strides[1];
  ba.dk_sh = a.dk_strides[2];
  ba.dv_sb = a.dv_strides[0];
  ba.dv_sn = a.dv_strides[1];
  ba.dv_sh = a.dv_strides[2];
  ba.B = a.B;
  ba.Nq = a.Nq;
  ba.Nk = a.Nk;
  ba.Hq = a.Hq;
  ba.Hkv = a.Hkv;
  ba.group = a.Hq / a.Hkv;
  ba.kblocks = kblocks;
  ba.d = a.d;
  ba.sem = a.deterministic ? sem : nullptr;
  set_mod_fields(mod, a.scale, &ba);
  ba.num_units = static_cast<int>(units);
  ba.head_group = bwd_head_group(ba.sem != nullptr, wide);
  ba.scale = a.scale;
  ba.scale_log2 = scale_log2(a.scale);
  ba.err = dev->err;
  ba.timeout_ns = g_timeout_ns;
  ba.inject = g_inject;
  const int grid = static_cast<int>(units < dev->sm_count ? units : dev->sm_count);
  e = fa::launch_bwd(fa::kernel_d(a.d), mod.mask, f16, tq, tk, tv, tdo, tdq, ba, grid, stream);
  if (e != cudaSuccess) return cuda_fail("backward kernel launch", e);
  e = wide ? fa::launch_bwd_post_t(a.d, f16, dq_acc, a.scale, a.dq, a.B, a.Nq, nq_pad, a.Hq,
                                   a.dq_strides, nullptr, 0, stream)
           : fa::launch_bwd_post(a.d, f16, dq_acc, a.scale, a.dq, a.B, a.Nq, a.Hq, a.dq_strides,
                                 stream);
  return e == cudaSuccess ? FA_OK : cuda_fail("backward postprocessing launch", e);
}

fa_status fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                        const void *dout, const float *lse, void *dq, void *dk, void *dv,
                        const int *cu_seqlens_q, const int *cu_seqlens_k, int B,
                        int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int Hq,
                        int Hkv, int d, float scale, int causal, int dtype, void *workspace,
                        size_t workspace_bytes, int deterministic, const fa_score_mod *mod_in,
                        cudaStream_t stream) {
  if (B < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || total_q < 0 || total_k < 0 || Hq <= 0 ||
      Hkv <= 0 || Hq % Hkv != 0)
    return FA_ERR_INVALID_ARG;
  if (!head_dim_ok(d, kMaxPrefillD)) return FA_ERR_UNSUPPORTED;
  if (!dtype_ok(dtype)) return FA_ERR_UNSUPPORTED;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  if (max_seqlen_q > (1 << 30) || max_seqlen_k > (1 << 30) || total_q > (1 << 30) ||
      total_k > (1 << 30))
    return FA_ERR_INVALID_ARG;
  if (B == 0 || (total_q == 0 && total_k == 0)) return FA_OK;
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr || !aligned(cu_seqlens_q, 4) ||
      !aligned(cu_seqlens_k, 4))
    return FA_ERR_INVALID_ARG;
  const bool q_side = total_q > 0, k_side = total_k > 0;
  if (q_side && (q == nullptr || o == nullptr || dout == nullptr || dq == nullptr ||
                 lse == nullptr || !aligned(q, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
                 !aligned(dq, 16) || !aligned(lse, 4)))
    return FA_ERR_INVALID_ARG;
  if (k_side && (k == nullptr || v == nullptr || dk == nullptr || dv == nullptr ||
                 !aligned(k, 16) || !aligned(v, 16) || !aligned(dk, 16) || !aligned(dv, 16)))
    return FA_ERR_INVALID_ARG;
  // The dense size for (B, max_seqlen_q) covers every part of the packed layout.
  const size_t need = fa_bwd_workspace_size(B, max_seqlen_q, Hq, d);
  if (q_side && k_side &&
      (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)))
    return FA_ERR_WORKSPACE;
  const bool wide = fa::kernel_d(d) == 256;  // units per d half, 64-query steps
  const int kblocks = ceil_div(max_seqlen_k, 128);
  const int64_t units = static_cast<int64_t>(kblocks) * B * Hkv * (wide ? 2 : 1);
  if (units > INT32_MAX) return FA_ERR_INVALID_ARG;
  ModPlan mod;
  fa_status st = plan_mod(mod_in, causal, &mod);
  if (st != FA_OK) return st;

  DeviceInfo *dev = nullptr;
  st = current_device(&dev);
  if (st != FA_OK) return st;
  cudaError_t e;
  const int64_t qst[3] = {0, static_cast<int64_t>(Hq) * d, d};
  const int64_t kst[3] = {0, static_cast<int64_t>(Hkv) * d, d};
  if (!k_side || max_seqlen_k == 0) {  // no keys: dQ = 0
    e = fa::launch_zero16(dq, 1, total_q, Hq, d, qst, stream);
    return e == cudaSuccess ? FA_OK : cuda_fail("zero kernel launch", e);
  }
  if (!q_side || max_seqlen_q == 0) {  // no queries: dK = dV = 0
    e = fa::launch_zero16(dk, 1, total_k, Hkv, d, kst, stream);
    if (e == cudaSuccess) e = fa::launch_zero16(dv, 1, total_k, Hkv, d, kst, stream);
    return e == cudaSuccess ? FA_OK : cuda_fail("zero kernel launch", e);
  }
  // dQ accumulator: packed [total_q, Hq, d]; kernel width 256: per sequence, transposed
  // [B, Hq, d, max_seqlen_q rounded up to 4]
  float *dq_acc = static_cast<float *>(workspace);
  const int nq_pad = fa::dq_acc_nq(max_seqlen_q);
  const int64_t acc_n = wide ? static_cast<int64_t>(B) * Hq * d * nq_pad
                             : static_cast<int64_t>(total_q) * Hq * d;
  const int64_t acc_bytes = (acc_n * 4 + 255) / 256 * 256;
  float *dvec = reinterpret_cast<float *>(static_cast<char *>(workspace) + acc_bytes);
  const int64_t vec_bytes = (static_cast<int64_t>(Hq) * total_q * 4 + 255) / 256 * 256;
  int *sem = reinterpret_cast<int *>(static_cast<char *>(workspace) + acc_bytes + vec_bytes);
  const int qblocks = ceil_div(max_seqlen_q, wide ? 64 : 128);
  const int nsem = deterministic ? B * Hq * qblocks * (wide ? 2 : 1) : 0;
  const int qrows = wide ? 64 : 128;  // Q / dO box rows: the kernel's query step
  CUtensorMap tq, tk, tv, tdo, tdq;
  if ((st = make_map(&tq, q, d, total_q, Hq, 1, qst[1], d, 0, dtype, qrows)) != FA_OK ||
      (st = make_map(&tdo, dout, d, total_q, Hq, 1, qst[1], d, 0, dtype, qrows)) != FA_OK ||
      (st = make_map(&tk, k, d, total_k, Hkv, 1, kst[1], d, 0, dtype)) != FA_OK ||
      (st = make_map(&tv, v, d, total_k, Hkv, 1, kst[1], d, 0, dtype)) != FA_OK ||
      (st = wide ? make_map_dqt(&tdq, dq_acc, d, nq_pad, Hq, B)
                 : make_map_f32(&tdq, dq_acc, d, total_q, Hq, 1)) != FA_OK)
    return st;
  const bool f16 = dtype == FA_FP16;
  e = fa::launch_bwd_pre(d, f16, o, dout, 1, total_q, Hq, qst, qst, dvec, dq_acc, acc_n, sem,
                         nsem, stream);
  if (e != cudaSuccess) return cuda_fail("backward preprocessing launch", e);
  fa::BwdArgs ba{};
  ba.lse = lse;
  ba.dvec = dvec;
  ba.lse_sb = 0;
  ba.lse_sh = total_q;
  ba.varlen = 1;
  ba.cu_q = cu_seqlens_q;
  ba.cu_k = cu_seqlens_k;
  ba.total_q = total_q;
  ba.total_k = total_k;
  ba.qblocks = qblocks;
  ba.dk = dk;
  ba.dv = dv;
  ba.dk_sb = ba.dv_sb = 0;
  ba.dk_sn = ba.dv_sn = kst[1];
  ba.dk_sh = ba.dv_sh = d;
  ba.B = B;
  ba.Nq = max_seqlen_q;
  ba.Nk = max_seqlen_k;
  ba.Hq = Hq;
  ba.Hkv = Hkv;
  ba.group = Hq / Hkv;
  ba.kblocks = kblocks;
  ba.d = d;
  ba.sem = deterministic ? sem : nullptr;
  set_mod_fields(mod, scale, &ba);
  ba.num_units = static_cast<int>(units);
  ba.head_group = bwd_head_group(ba.sem != nullptr, wide);
  ba.scale = scale;
  ba.scale_log2 = scale_log2(scale);
  ba.err = dev->err;
  ba.timeout_ns = g_timeout_ns;
  ba.inject = g_inject;
  const int grid = static_cast<int>(units < dev->sm_count ? units : dev->sm_count);
  e = fa::launch_bwd(fa::kernel_d(d), mod.mask, f16, tq, tk, tv, tdo, tdq, ba, grid, stream);
  if (e != cudaSuccess) return cuda_fail("backward kernel launch", e);
  e = wide ? fa::launch_bwd_post_t(d, f16, dq_acc, scale, dq, B, max_seqlen_q, nq_pad, Hq, qst,
                                   cu_seqlens_q, total_q, stream)
           : fa::launch_bwd_post(d, f16, dq_acc, scale, dq, 1, total_q, Hq, qst, stream);
  return e == cudaSuccess ? FA_OK : cuda_fail("backward postprocessing launch", e);
}

fa_status fa_get_last_device_error(cudaStream_t stream) {
  DeviceInfo *dev = nullptr;
  fa_status st = current_device(&dev);
  if (st != FA_OK) return st;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_device_error, sizeof word);
  if (e != cudaSuccess) return cuda_fail("cudaMemcpyFromSymbol", e);
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
  if (e != cudaSuccess) return cuda_fail("cudaMemcpyToSymbol", e);
  if (word & (fa::DEVERR_PREFILL_TIMEOUT | fa::DEVERR_DECODE_TIMEOUT | fa::DEVERR_BWD_TIMEOUT))
    return FA_ERR_TIMEOUT;
  if (word & (fa::DEVERR_BAD_CU_SEQLENS | fa::DEVERR_BAD_CACHE_LEN | fa::DEVERR_BAD_APPEND |
              fa::DEVERR_BAD_BLOCK_TABLE))
    return FA_ERR_INVALID_ARG;
  if (word & fa::DEVERR_SCHED_OVERLAP) return FA_ERR_CONCURRENT;
  return FA_OK;
}

}  // extern "C"
