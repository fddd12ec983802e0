// C ABI of the library: argument checks, split choice, workspace layout,
// TMA descriptors and kernel launches.  Nothing here allocates device memory,
// synchronizes, or reads device memory on the host.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "fp8pa.h"
#include "fp8pa_testing.h"
#include "kernels.h"

namespace fp8pa {
#define FP8PA_DECLARE_VARIANT(name)                                                                          \
  cudaError_t launch_##name(int, int, const AttnParams&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, \
                            int, cudaStream_t);                                                             \
  int smem_##name(int, int);
FP8PA_DECLARE_VARIANT(attn_fp8_d256)
FP8PA_DECLARE_VARIANT(attn_fp8_d512)
FP8PA_DECLARE_VARIANT(attn_bf16_d512)
FP8PA_DECLARE_VARIANT(attn_bf16dqv_d512)
#undef FP8PA_DECLARE_VARIANT

cudaError_t launch_attn(int head_dim, int path, int rows, int ctas, const AttnParams& p, const CUtensorMap& tm_q,
                        const CUtensorMap& tm_k, const CUtensorMap& tm_v, int sms, cudaStream_t stream) {
  if (head_dim == 256 && path == kPathE4M3) return launch_attn_fp8_d256(rows, ctas, p, tm_q, tm_k, tm_v, sms, stream);
  if (head_dim == 512 && path == kPathE4M3) return launch_attn_fp8_d512(rows, ctas, p, tm_q, tm_k, tm_v, sms, stream);
  if (head_dim == 512 && path == kPathBf16) return launch_attn_bf16_d512(rows, ctas, p, tm_q, tm_k, tm_v, sms, stream);
  if (head_dim == 512 && path == kPathBf16DqV)
    return launch_attn_bf16dqv_d512(rows, ctas, p, tm_q, tm_k, tm_v, sms, stream);
  return cudaErrorInvalidValue;
}

int attn_smem_bytes(int head_dim, int path, int rows, int ctas) {
  if (head_dim == 256 && path == kPathE4M3) return smem_attn_fp8_d256(rows, ctas);
  if (head_dim == 512 && path == kPathE4M3) return smem_attn_fp8_d512(rows, ctas);
  if (head_dim == 512 && path == kPathBf16) return smem_attn_bf16_d512(rows, ctas);
  if (head_dim == 512 && path == kPathBf16DqV) return smem_attn_bf16dqv_d512(rows, ctas);
  return 0;
}
}  // namespace fp8pa

using namespace fp8pa;

namespace {

__device__ unsigned int g_status;

thread_local char g_err[512] = "";
// Test, tuning and profiling hooks (fp8pa_testing.h): each host thread has its
// own settings, so one caller's hooks never change another thread's calls.
thread_local cudaEvent_t g_ev_start = nullptr, g_ev_stop = nullptr;
thread_local int g_ctas_override = 0;
thread_local int g_dequant_v = 0;
thread_local unsigned g_wait_limit = 0;
thread_local int g_inject_stall = 0;
thread_local int g_grid_sms = 0;
thread_local int g_prefill_rows = 0;
thread_local int g_sm_split = 0;

// Kernel path for a Q dtype: E4M3 Q, or BF16 Q with V kept E4M3 (default) or
// dequantized to BF16 (fp8pa_set_bf16_dequant_v).
int kernel_path(bool fp8_q) { return fp8_q ? kPathE4M3 : (g_dequant_v ? kPathBf16DqV : kPathBf16); }

// CTAs per SM for a kernel variant: two co-resident CTAs where both fit
// (16-row tiles of the E4M3-Q path), else one.
int ctas_per_sm(int head_dim, int path, int rows) {
  const int forced = g_ctas_override;
  if (forced == 1 || forced == 2) {
    if (attn_smem_bytes(head_dim, path, rows, forced) > 0) return forced;
  }
  if (rows == 16 && attn_smem_bytes(head_dim, path, rows, 2) > 0) return 2;
  return 1;
}

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

}  // namespace

// Records `msg` as the message fp8pa_last_error() returns on this thread.
int fp8pa::set_last_error(int code, const char* msg) { return fail(code, "%s", msg); }

namespace {

int cuda_fail(cudaError_t e, const char* what) {
  return fail(FP8PA_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
constexpr int kDefaultSms = 152;  // GB300; used when no device is visible (host-only sizing)

int device_sms() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return kDefaultSms;
  }
  int v = cache[dev].load();
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
      cudaGetLastError();
      return kDefaultSms;
    }
    cache[dev].store(v);
  }
  return v;
}

// Device address of the status word in the current context.  Looked up on
// every call (a host-side table lookup, no device work), so it stays right
// after cudaDeviceReset or a new primary context moves the module.
unsigned* status_ptr() {
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_status) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<unsigned*>(addr);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Everything about a call that follows from host-known sizes.
struct CallPlan {
  int group;
  bool fp8_q;
  int num_classes;
  ClassInfo cls[2];
  int splits;
  bool prefill_kernel;  // class 1 runs the rows-on-lanes prefill kernel (128-row tiles)
  size_t items_max[2];
  size_t off_work[2], off_opart, off_lsepart, total;
};

int check_shape(int batch, int total_q, int max_seqlen_q, int hq, int hkv, int head_dim, int max_pages,
                int window_left, int num_splits) {
  if (batch < 0 || total_q < 0 || max_seqlen_q < 0)
    return fail(FP8PA_EINVAL, "batch, total_q and max_seqlen_q must be >= 0 (got %d, %d, %d)", batch, total_q,
                max_seqlen_q);
  if (total_q > 0 && max_seqlen_q < 1) return fail(FP8PA_EINVAL, "max_seqlen_q must be >= 1 when total_q > 0");
  if (max_seqlen_q > total_q && total_q > 0)
    return fail(FP8PA_EINVAL, "max_seqlen_q (%d) exceeds total_q (%d)", max_seqlen_q, total_q);
  if (hkv <= 0 || hq <= 0) return fail(FP8PA_EINVAL, "num_heads_q and num_heads_kv must be > 0");
  if (hq % hkv != 0)
    return fail(FP8PA_EUNSUPPORTED, "num_heads_q (%d) must be a multiple of num_heads_kv (%d)", hq, hkv);
  const int g = hq / hkv;
  if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16)
    return fail(FP8PA_EUNSUPPORTED, "query heads per KV head = %d; supported: 1, 2, 4, 8, 16", g);
  if (head_dim != 256 && head_dim != 512)
    return fail(FP8PA_EUNSUPPORTED, "head_dim %d is not supported (supported: 256 with E4M3 Q, 512 with BF16 or E4M3 Q)",
                head_dim);
  if (max_pages < 1) return fail(FP8PA_EINVAL, "max_pages_per_seq must be >= 1");
  if ((long long)max_pages * kPage > 0x7FFFFFFFLL) return fail(FP8PA_EINVAL, "max_pages_per_seq too large");
  if (window_left < -1) return fail(FP8PA_EINVAL, "window_left must be >= -1 (got %d)", window_left);
  if (num_splits < 0 || num_splits > 64) return fail(FP8PA_EINVAL, "num_splits must be in [0, 64] (got %d)", num_splits);
  if ((long long)total_q * hq > 0x7FFFFFFFLL) return fail(FP8PA_EINVAL, "total_q * num_heads_q too large");
  return FP8PA_OK;
}

// Split count for single-row-tile sequences.  Measured on GB300: once every
// SM has a (sequence, KV head) unit, decode tiles of up to 16 rows stream at
// the HBM roofline and splitting only adds partial writes and the combine, so
// they split only when there are fewer units than SMs, to about two items per
// SM, each split keeping at least four 128-key tiles.  Tiles of 32 rows (a few
// query tokens per sequence, as in speculative verification) do more work per
// byte, and a part-filled last wave of long units costs them more: between one
// and four waves of units they take the split count whose item waves leave the
// least idle tail, with a small cost per extra split (64 sequences x 4 KV
// heads, 28672 keys: 4 splits, kernel 1.287 -> 1.183 ms).
int auto_splits(int batch, int hkv, int max_pages, int window_left, int max_lq0, int rows, int sms) {
  const long long units = (long long)hkv * batch;
  if (units <= 0) return 1;
  long long pages = max_pages;
  if (window_left >= 0) pages = std::min<long long>(pages, (window_left + max_lq0 - 1) / kPage + 2);
  const long long tiles = (pages + 1) / 2;
  if (units >= sms) {
    if (rows <= 16 || units >= 4LL * sms) return 1;
    int best = 1;
    double best_cost = 1e30;
    for (int s = 1; s <= 8 && (s == 1 || tiles / s >= 4); ++s) {
      const long long waves = (units * s + sms - 1) / sms;
      const double cost = (double)waves / s * (1.0 + 0.02 * (s - 1));
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best = s;
      }
    }
    return best;
  }
  long long s = (2LL * sms + units - 1) / units;
  s = std::min<long long>(s, std::max<long long>(1, tiles / 4));
  s = std::max<long long>(1, std::min<long long>(s, 64));
  // two splits measured far slower than one or three on the sliding-window decode
  return (int)(s == 2 ? 3 : s);
}

// Cost model of the side-by-side split of the SMs between the decode and the
// prefill row classes (plan kernel), per kernel path, from measurements on
// GB300 at 2.07 GHz.  pf_ns_flop: a prefill-class tile's ns x SMs per visible
// flop, from the 4096-token chunk alone on 152 SMs (head dim 512 BF16 Q 2.32 ms,
// E4M3 Q 1.18 ms, head dim 256 E4M3 0.132 ms); the E4M3 head-dim-512 figure is
// raised 1.5x because beside the streaming decode rows that kernel measured that
// much slower (its K/V re-reads no longer stay in L2).  dec_gbs_sm, dec_gbs: the
// decode class's per-SM and whole-GPU stream rates (4032 decode rows of the mixed
// batch on 72..152 SMs: BF16 Q levels off at 7.0 TB/s from ~125 SMs, E4M3 Q at
// 7.2 TB/s from ~90; head dim 256 about 50 GB/s per SM).  Splits swept on the
// mixed batches: head dim 512 BF16 Q best at 36 prefill SMs (12.0 ms), E4M3 Q at
// 28..48 (10.1..10.3 ms), head dim 256 flat within 1 % from 4 to 24.
struct SplitCost {
  float pf_ns_flop, dec_gbs_sm, dec_gbs;
};
SplitCost split_cost(int head_dim, bool fp8_q) {
  if (!fp8_q) return {2.14e-4f, 60.f, 7000.f};
  return head_dim == 512 ? SplitCost{1.64e-4f, 75.f, 7200.f} : SplitCost{1.46e-4f, 50.f, 7000.f};
}

// Whether row class k is launched: it can hold a sequence (with one sequence,
// only the class of its total_q queries can).
bool class_launched(const CallPlan& pl, int k, int batch, int total_q) {
  const ClassInfo& c = pl.cls[k];
  if (c.lq_max < c.lq_min) return false;
  if (batch == 1) return total_q >= c.lq_min && total_q <= c.lq_max;
  return true;
}

int make_plan(int batch, int total_q, int max_seqlen_q, int hq, int hkv, int head_dim, int q_dtype, int max_pages,
              int window_left, int num_splits, CallPlan& pl) {
  int rc = check_shape(batch, total_q, max_seqlen_q, hq, hkv, head_dim, max_pages, window_left, num_splits);
  if (rc) return rc;
  if (q_dtype != FP8PA_BF16 && q_dtype != FP8PA_E4M3)
    return fail(FP8PA_EINVAL, "q_dtype must be FP8PA_BF16 (0) or FP8PA_E4M3 (1), got %d", q_dtype);
  if (head_dim == 256 && q_dtype != FP8PA_E4M3)
    return fail(FP8PA_EUNSUPPORTED,
                "q dtype bfloat16 with k/v dtype float8_e4m3fn at head_size 256 is not supported "
                "(head_size 256 takes E4M3 Q; quantize it with quantize_q_fp8)");
  pl.fp8_q = q_dtype == FP8PA_E4M3;
  // prefill-class tiles with E4M3 Q run the rows-on-lanes kernel with 128 rows (at head
  // dim 512 as two work items per row tile, one per 256-wide slice of the output dims)
  pl.prefill_kernel = pl.fp8_q;
  const int prefill_rows = pl.prefill_kernel ? 128 : (g_prefill_rows == 32 ? 32 : 64);
  const int g = hq / hkv;
  pl.group = g;
  const long long rmax = (long long)max_seqlen_q * g;
  int lq0_max;
  if (rmax <= 32) {
    pl.num_classes = 1;
    pl.cls[0] = ClassInfo{1, std::max(1, max_seqlen_q), rmax <= 16 ? 16 : 32, 1};
    lq0_max = std::max(1, max_seqlen_q);
  } else {
    lq0_max = 16 / g;
    if (lq0_max >= 1) {
      pl.num_classes = 2;
      pl.cls[0] = ClassInfo{1, lq0_max, 16, 1};
      pl.cls[1] = ClassInfo{lq0_max + 1, max_seqlen_q, prefill_rows, 1};
    } else {
      pl.num_classes = 2;  // class 0 empty
      pl.cls[0] = ClassInfo{1, 0, 16, 1};
      pl.cls[1] = ClassInfo{1, max_seqlen_q, prefill_rows, 1};
      lq0_max = 1;
    }
  }
  // With a prefill row class in the batch its tiles keep every SM busy: no split.
  pl.splits = num_splits > 0       ? num_splits
              : pl.num_classes > 1 ? 1
                                   : auto_splits(batch, hkv, max_pages, window_left, lq0_max, pl.cls[0].rows,
                                                 device_sms());
  pl.cls[0].max_splits = pl.splits;
  pl.cls[1].dhalves = pl.prefill_kernel && head_dim == 512 ? 2 : 1;
  // workspace layout: [counts][class-0 items][class-1 items][o_part][lse_part]
  pl.items_max[0] = (size_t)hkv * batch * pl.splits;
  pl.items_max[1] =
      pl.num_classes > 1 ? (size_t)hkv * ((size_t)((long long)total_q * g + 63) / 64 + 2 * (size_t)batch) : 0;
  size_t off = 256;
  for (int k = 0; k < 2; ++k) {
    pl.off_work[k] = off;
    off = round_up(off + pl.items_max[k] * sizeof(int4), 256);
  }
  pl.off_opart = off;
  if (pl.splits > 1) off = round_up(off + (size_t)pl.splits * total_q * hq * head_dim * sizeof(float), 256);
  pl.off_lsepart = off;
  if (pl.splits > 1) off = round_up(off + (size_t)pl.splits * hq * total_q * sizeof(float), 256);
  pl.total = off;
  return FP8PA_OK;
}

int encode_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
               const cuuint64_t* strides, const cuuint32_t* box, const char* what) {
  auto fn = encode_fn();
  if (!fn) return fail(FP8PA_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, dt, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FP8PA_ECUDA, "cuTensorMapEncodeTiled failed for %s (CUresult %d)", what, (int)r);
  return FP8PA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

const char* fp8pa_last_error(void) { return g_err; }

void fp8pa_set_wait_limit(unsigned int max_iterations) { g_wait_limit = max_iterations; }

void fp8pa_set_stall_injection(int on) { g_inject_stall = on ? 1 : 0; }

void fp8pa_set_ctas_per_sm(int ctas) { g_ctas_override = ctas; }

void fp8pa_set_bf16_dequant_v(int on) { g_dequant_v = on ? 1 : 0; }

void fp8pa_set_grid_sms(int sms) { g_grid_sms = sms > 0 ? sms : 0; }

void fp8pa_set_prefill_rows(int rows) { g_prefill_rows = rows; }

void fp8pa_set_sm_split(int sms) { g_sm_split = sms > 0 ? sms : 0; }

void fp8pa_set_timing_events(void* start_event, void* stop_event) {
  g_ev_start = static_cast<cudaEvent_t>(start_event);
  g_ev_stop = static_cast<cudaEvent_t>(stop_event);
}

int fp8pa_kernel_launches(int batch, int total_q, int max_seqlen_q, int num_heads_q, int num_heads_kv, int head_dim, int q_dtype,
                          int max_pages_per_seq, int window_left, int num_splits) {
  CallPlan pl;
  if (make_plan(batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv, head_dim, q_dtype, max_pages_per_seq,
                window_left, num_splits, pl))
    return 0;
  if (batch == 0 || total_q == 0) return 0;
  int n = 1;  // plan
  for (int k = 0; k < pl.num_classes; ++k)
    if (class_launched(pl, k, batch, total_q)) ++n;
  if (pl.splits > 1) ++n;
  return n;
}

int quantize_q_fp8(const void* q_bf16, void* q_e4m3, const float* q_descale, long long n_elems,
                   fp8pa_stream_t stream) {
  if (n_elems < 0) return fail(FP8PA_EINVAL, "n_elems must be >= 0 (got %lld)", n_elems);
  if (n_elems == 0) return FP8PA_OK;
  if (!q_bf16 || !q_e4m3 || !q_descale) return fail(FP8PA_EINVAL, "quantize_q_fp8: null pointer");
  cudaError_t e = launch_quantize_q(q_bf16, q_e4m3, q_descale, n_elems, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "quantize_q_fp8 launch");
  return FP8PA_OK;
}

int fp8pa_lse_combine(const void* o_parts, const float* lse_parts, int num_parts, long long total_q,
                      int num_heads_q, int head_dim, void* out, float* lse_out, fp8pa_stream_t stream) {
  if (total_q < 0) return fail(FP8PA_EINVAL, "lse_combine: total_q must be >= 0 (got %lld)", total_q);
  if (num_parts < 1 || num_heads_q < 1 || head_dim < 8 || head_dim % 8)
    return fail(FP8PA_EINVAL, "lse_combine: need num_parts >= 1, num_heads_q >= 1, head_dim a multiple of 8");
  if (total_q == 0) return FP8PA_OK;
  if (!o_parts || !lse_parts || !out) return fail(FP8PA_EINVAL, "lse_combine: null pointer");
  if (reinterpret_cast<uintptr_t>(o_parts) % 16 || reinterpret_cast<uintptr_t>(out) % 16 ||
      reinterpret_cast<uintptr_t>(lse_parts) % 4 || reinterpret_cast<uintptr_t>(lse_out) % 4)
    return fail(FP8PA_EINVAL, "lse_combine: o_parts and out need 16-byte, lse buffers 4-byte alignment");
  cudaError_t e = launch_lse_combine(o_parts, lse_parts, num_parts, total_q, num_heads_q, head_dim, out, lse_out,
                                     device_sms(), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "lse_combine launch");
  return FP8PA_OK;
}

int fp8pa_kv_cache_write(const void* key, const void* value, long long key_token_stride,
                         long long value_token_stride, uint8_t* k_cache, uint8_t* v_cache, int num_pages,
                         const int64_t* slot_mapping, long long num_tokens, int num_heads_kv, int head_dim,
                         const float* k_descale, const float* v_descale, fp8pa_stream_t stream) {
  if (num_tokens < 0) return fail(FP8PA_EINVAL, "kv_cache_write: num_tokens must be >= 0 (got %lld)", num_tokens);
  if (num_tokens == 0) return FP8PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping || !k_descale || !v_descale)
    return fail(FP8PA_EINVAL, "kv_cache_write: null pointer");
  if (num_heads_kv < 1 || head_dim < 1 || num_pages < 0)
    return fail(FP8PA_EINVAL, "kv_cache_write: num_heads_kv, head_dim must be >= 1 and num_pages >= 0");
  const long long row = (long long)num_heads_kv * head_dim;
  if (row % 8 != 0 || row > (1LL << 30))
    return fail(FP8PA_EINVAL, "kv_cache_write: num_heads_kv * head_dim = %lld is not a multiple of 8", row);
  if (key_token_stride < row || value_token_stride < row || key_token_stride % 8 || value_token_stride % 8)
    return fail(FP8PA_EINVAL, "kv_cache_write: token strides must be >= num_heads_kv * head_dim and multiples of 8");
  if (reinterpret_cast<uintptr_t>(key) % 16 || reinterpret_cast<uintptr_t>(value) % 16 ||
      reinterpret_cast<uintptr_t>(k_cache) % 8 || reinterpret_cast<uintptr_t>(v_cache) % 8)
    return fail(FP8PA_EINVAL, "kv_cache_write: key/value need 16-byte and the caches 8-byte alignment");
  unsigned* status = status_ptr();
  if (!status) return fail(FP8PA_ECUDA, "kv_cache_write: device status word unavailable");
  cudaError_t e = launch_kv_cache_write(key, value, key_token_stride, value_token_stride, k_cache, v_cache,
                                        reinterpret_cast<const long long*>(slot_mapping), num_tokens, (int)row,
                                        (long long)num_pages * FP8PA_PAGE_SIZE, k_descale, v_descale, status,
                                        device_sms(), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kv_cache_write launch");
  return FP8PA_OK;
}

size_t fp8pa_workspace_size(int batch, int total_q, int max_seqlen_q, int num_heads_q, int num_heads_kv,
                            int head_dim, int q_dtype, int max_pages_per_seq, int window_left, int num_splits) {
  CallPlan pl;
  if (make_plan(batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv, head_dim, q_dtype, max_pages_per_seq,
                window_left, num_splits, pl))
    return 0;
  return pl.total;
}

int fp8pa_num_splits(int batch, int total_q, int max_seqlen_q, int num_heads_q, int num_heads_kv, int head_dim, int q_dtype,
                     int max_pages_per_seq, int window_left, int num_splits) {
  CallPlan pl;
  if (make_plan(batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv, head_dim, q_dtype, max_pages_per_seq,
                window_left, num_splits, pl))
    return 0;
  return pl.splits;
}

namespace {

int fwd_impl(const void* q, int q_dtype, const uint8_t* k_cache, const uint8_t* v_cache, int num_pages,
             const int32_t* block_table, int max_pages_per_seq, const int32_t* cu_seqlens_q, const int32_t* seqused_k,
             int batch, int total_q, int max_seqlen_q, int num_heads_q, int num_heads_kv, int head_dim,
             const float* q_descale, const float* k_descale, const float* v_descale, int descale_batch_stride,
             int descale_head_stride, float softmax_scale, int window_left, int causal, int num_splits,
             void* workspace, size_t workspace_bytes, void* out, float* lse, const float* sinks,
             fp8pa_stream_t stream) {
  const bool fp8_q = q_dtype == FP8PA_E4M3;
  CallPlan pl;
  int rc = make_plan(batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv, head_dim, q_dtype, max_pages_per_seq,
                     window_left, num_splits, pl);
  if (rc) return rc;
  if (causal != 0 && causal != 1) return fail(FP8PA_EINVAL, "causal must be 0 or 1 (got %d)", causal);
  if (!std::isfinite(softmax_scale)) return fail(FP8PA_EINVAL, "softmax_scale must be finite");
  if (descale_batch_stride < 0 || descale_head_stride < 0) return fail(FP8PA_EINVAL, "descale strides must be >= 0");
  if (batch == 0 || total_q == 0) return FP8PA_OK;
  if (num_pages < 1) return fail(FP8PA_EINVAL, "num_pages must be >= 1 (got %d)", num_pages);
  // null descales are the unit scale (no descale read)
  if (!q || !k_cache || !v_cache || !block_table || !cu_seqlens_q || !seqused_k || !out)
    return fail(FP8PA_EINVAL, "null pointer argument");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return fail(FP8PA_EINVAL, "q, k_cache, v_cache and out must be 16-byte aligned");
  if (workspace_bytes < pl.total)
    return fail(FP8PA_EINVAL, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, pl.total);
  if (!workspace || !aligned(workspace, 256)) return fail(FP8PA_EINVAL, "workspace must be non-null and 256-byte aligned");

  cudaStream_t st = (cudaStream_t)stream;
  unsigned* status = status_ptr();
  if (!status) return fail(FP8PA_ECUDA, "cannot resolve the device status word");
  const int sms = g_grid_sms > 0 ? std::min(g_grid_sms, device_sms()) : device_sms();
  const int g = pl.group;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* counts = reinterpret_cast<int*>(ws);

  // TMA descriptors: K/V page tiles (128 bytes of head dim x 64 slots of one KV head of one page)
  CUtensorMap tm_k, tm_v, tm_q[2];
  {
    const cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)num_heads_kv, (cuuint64_t)kPage,
                                (cuuint64_t)num_pages};
    const cuuint64_t strides[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_heads_kv * head_dim,
                                   (cuuint64_t)kPage * num_heads_kv * head_dim};
    const cuuint32_t box[4] = {128, 1, (cuuint32_t)kPage, 1};
    if ((rc = encode_map(&tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, k_cache, dims, strides, box, "k_cache"))) return rc;
    if ((rc = encode_map(&tm_v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, v_cache, dims, strides, box, "v_cache"))) return rc;
  }
  const int esz = fp8_q ? 1 : 2;
  for (int k = 0; k < pl.num_classes; ++k) {
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_heads_q, (cuuint64_t)total_q};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * esz, (cuuint64_t)num_heads_q * head_dim * esz};
    const cuuint32_t box[3] = {(cuuint32_t)(128 / esz), (cuuint32_t)g, (cuuint32_t)(pl.cls[k].rows / g)};
    if ((rc = encode_map(&tm_q[k], fp8_q ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q,
                         dims, strides, box, "q")))
      return rc;
  }

  PlanParams pp{};
  pp.cu_seqlens_q = cu_seqlens_q;
  pp.seqused_k = seqused_k;
  pp.batch = batch;
  pp.total_q = total_q;
  pp.group = g;
  pp.hkv = num_heads_kv;
  pp.max_pages = max_pages_per_seq;
  pp.window_left = window_left;
  pp.causal = causal;
  pp.num_classes = pl.num_classes;
  for (int k = 0; k < 2; ++k) {
    pp.cls[k] = pl.cls[k];
    pp.work[k] = reinterpret_cast<int4*>(ws + pl.off_work[k]);
  }
  pp.counts = counts;
  pp.status = status;
  const SplitCost sc = split_cost(head_dim, fp8_q);
  pp.hq = num_heads_q;
  pp.head_dim = head_dim;
  pp.sms = sms;
  pp.pf_ns_flop = sc.pf_ns_flop;
  pp.dec_gbs_sm = sc.dec_gbs_sm;
  pp.dec_gbs = sc.dec_gbs;
  pp.forced_split = g_sm_split;
  cudaError_t e = launch_plan(pp, st);
  if (e != cudaSuccess) return cuda_fail(e, "plan launch");

  AttnParams p{};
  p.block_table = block_table;
  p.cu_seqlens_q = cu_seqlens_q;
  p.seqused_k = seqused_k;
  p.q_descale = q_descale;
  p.k_descale = k_descale;
  p.v_descale = v_descale;
  p.descale_b = descale_batch_stride;
  p.descale_h = descale_head_stride;
  p.batch = batch;
  p.total_q = total_q;
  p.hq = num_heads_q;
  p.hkv = num_heads_kv;
  p.group = g;
  p.head_dim = head_dim;
  p.max_pages = max_pages_per_seq;
  p.num_pages = num_pages;
  p.softmax_scale_log2 = softmax_scale * 1.4426950408889634f;
  p.window_left = window_left;
  p.causal = causal;
  p.out = out;
  p.lse = lse;
  p.o_part = reinterpret_cast<float*>(ws + pl.off_opart);
  p.lse_part = reinterpret_cast<float*>(ws + pl.off_lsepart);
  p.sinks = sinks;
  p.status = status;
  const unsigned wl = g_wait_limit;
  p.wait_limit = wl ? wl : kDefaultWaitLimit;
  p.inject_stall = g_inject_stall;
  const bool timed = g_ev_start && g_ev_stop;
  if (timed && (e = cudaEventRecord(g_ev_start, st)) != cudaSuccess) return cuda_fail(e, "timing event");
  // With both row classes launched they run side by side: the prefill class
  // first, on the SMs the plan kernel gave it, then the decode class on the rest.
  const bool both = pl.num_classes > 1 && class_launched(pl, 0, batch, total_q) &&
                    class_launched(pl, 1, batch, total_q);
  p.sm_split = counts + 4;
  p.grid_sms = sms;
  for (int kk = 0; kk < pl.num_classes; ++kk) {
    const int k = both ? 1 - kk : kk;
    if (!class_launched(pl, k, batch, total_q)) continue;
    p.conc_role = both ? (k == 1 ? 1 : 2) : 0;
    p.cls = pl.cls[k];
    p.work = reinterpret_cast<const int4*>(ws + pl.off_work[k]);
    p.work_count = counts + k;
    p.work_next = counts + 2 + k;
    const int path = kernel_path(fp8_q);
    if (k == 1 && pl.prefill_kernel)
      e = head_dim == 256 ? launch_attn_prefill_d256(p, tm_q[k], tm_k, tm_v, sms, st)
                          : launch_attn_prefill_d512(p, tm_q[k], tm_k, tm_v, sms, st);
    else
      e = launch_attn(head_dim, path, pl.cls[k].rows, ctas_per_sm(head_dim, path, pl.cls[k].rows), p, tm_q[k], tm_k,
                      tm_v, sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  }
  if (timed && (e = cudaEventRecord(g_ev_stop, st)) != cudaSuccess) return cuda_fail(e, "timing event");
  if (pl.splits > 1) {
    CombineParams cp{};
    cp.cu_seqlens_q = cu_seqlens_q;
    cp.seqused_k = seqused_k;
    cp.batch = batch;
    cp.total_q = total_q;
    cp.hq = num_heads_q;
    cp.group = g;
    cp.head_dim = head_dim;
    cp.max_pages = max_pages_per_seq;
    cp.window_left = window_left;
    cp.causal = causal;
    cp.cls = pl.cls[0];
    cp.o_part = p.o_part;
    cp.lse_part = p.lse_part;
    cp.out = out;
    cp.lse = lse;
    cp.sinks = sinks;
    e = launch_combine(cp, st);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  }
  return FP8PA_OK;
}

}  // namespace

int fp8_paged_attn_fwd(const void* q, int q_dtype, const uint8_t* k_cache, const uint8_t* v_cache, int num_pages,
                       const int32_t* block_table, int max_pages_per_seq, const int32_t* cu_seqlens_q,
                       const int32_t* seqused_k, int batch, int total_q, int max_seqlen_q, int num_heads_q,
                       int num_heads_kv, int head_dim, const float* q_descale, const float* k_descale,
                       const float* v_descale, int descale_batch_stride, int descale_head_stride,
                       float softmax_scale, int window_left, int causal, int num_splits, void* workspace,
                       size_t workspace_bytes, void* out, float* lse, fp8pa_stream_t stream) {
  return fwd_impl(q, q_dtype, k_cache, v_cache, num_pages, block_table, max_pages_per_seq, cu_seqlens_q, seqused_k,
                  batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv, head_dim, q_descale, k_descale, v_descale,
                  descale_batch_stride, descale_head_stride, softmax_scale, window_left, causal, num_splits, workspace,
                  workspace_bytes, out, lse, nullptr, stream);
}

int fp8_paged_attn_fwd_sinks(const void* q, int q_dtype, const uint8_t* k_cache, const uint8_t* v_cache,
                             int num_pages, const int32_t* block_table, int max_pages_per_seq,
                             const int32_t* cu_seqlens_q, const int32_t* seqused_k, int batch, int total_q,
                             int max_seqlen_q, int num_heads_q, int num_heads_kv, int head_dim, const float* q_descale,
                             const float* k_descale, const float* v_descale, int descale_batch_stride,
                             int descale_head_stride, float softmax_scale, int window_left, int causal,
                             int num_splits, void* workspace, size_t workspace_bytes, void* out, float* lse,
                             const float* sinks, fp8pa_stream_t stream) {
  if (!sinks && batch > 0 && total_q > 0) return fail(FP8PA_EINVAL, "fp8_paged_attn_fwd_sinks: null sinks");
  if (sinks && !aligned(sinks, 4)) return fail(FP8PA_EINVAL, "sinks must be 4-byte aligned");
  return fwd_impl(q, q_dtype, k_cache, v_cache, num_pages, block_table, max_pages_per_seq, cu_seqlens_q, seqused_k,
                  batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv, head_dim, q_descale, k_descale, v_descale,
                  descale_batch_stride, descale_head_stride, softmax_scale, window_left, causal, num_splits, workspace,
                  workspace_bytes, out, lse, sinks, stream);
}

int fp8pa_get_device_status(unsigned int* host_status, fp8pa_stream_t stream) {
  if (!host_status) return fail(FP8PA_EINVAL, "null host_status");
  cudaError_t e = cudaMemcpyFromSymbolAsync(host_status, g_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost,
                                            (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "status copy");
  return FP8PA_OK;
}

int fp8pa_reset_device_status(fp8pa_stream_t stream) {
  unsigned* p = status_ptr();
  if (!p) return fail(FP8PA_ECUDA, "cannot resolve the device status word");
  cudaError_t e = cudaMemsetAsync(p, 0, sizeof(unsigned), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "status reset");
  return FP8PA_OK;
}

}  // extern "C"
