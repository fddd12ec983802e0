// fp8_paged_attn_fwd_noalloc: the attention forward with its scratch memory
// (work list, split-KV partial outputs and log-sum-exps) in a fixed device
// array owned by this library instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory at call time: an inference engine
// that hands almost all HBM to its KV-cache pool at start-up (a later
// cudaMalloc fails, or would have to evict cache pages), a plugin host that
// gives kernel libraries no allocator of their own, or a latency-critical
// path that cannot afford cudaMalloc's implicit device synchronization.  For
// them this entry point needs nothing beyond the inputs and outputs.
#include <cstdio>

#include "fp8pa.h"
#include "kernels.h"

namespace {

// Every device that loads the library holds this array until the process exits.
__device__ __align__(256) unsigned char g_noalloc_scratch[FP8PA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array in the current context.  The array's
// name in host code is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress with the device current.  It is looked up on every call
// (a host-side table lookup, no device work): a cached address would go stale
// after cudaDeviceReset or a new primary context reloads the module.
int scratch_address(void** out, char* msg, size_t msg_len) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0) {
    snprintf(msg, msg_len, "no usable current device (%s)", cudaGetErrorString(e));
    return FP8PA_ECUDA;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p) {
    cudaGetLastError();
    snprintf(msg, msg_len, "cudaGetSymbolAddress of the scratch array failed: %s", cudaGetErrorString(e));
    return FP8PA_ECUDA;
  }
  *out = p;
  return FP8PA_OK;
}

thread_local char g_noalloc_err[256];

}  // namespace

extern "C" int fp8_paged_attn_fwd_noalloc(const void* q, int q_dtype, const uint8_t* k_cache,
                                          const uint8_t* v_cache, int num_pages, const int32_t* block_table,
                                          int max_pages_per_seq, const int32_t* cu_seqlens_q,
                                          const int32_t* seqused_k, int batch, int total_q, int max_seqlen_q,
                                          int num_heads_q, int num_heads_kv, int head_dim, const float* q_descale,
                                          const float* k_descale, const float* v_descale,
                                          int descale_batch_stride, int descale_head_stride, float softmax_scale,
                                          int window_left, int causal, int num_splits, void* out, float* lse,
                                          fp8pa_stream_t stream) {
  // Size check first: the same sizing as the workspace entry point.
  size_t need = fp8pa_workspace_size(batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv, head_dim, q_dtype,
                                     max_pages_per_seq, window_left, num_splits);
  if (num_splits == 0 && need > (size_t)FP8PA_NOALLOC_SCRATCH_BYTES) {
    // Automatic splits whose partials do not fit: the largest smaller split
    // count that does (a function of the call's sizes, like the automatic one).
    const int s_auto = fp8pa_num_splits(batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv, head_dim, q_dtype,
                                        max_pages_per_seq, window_left, 0);
    for (int s = s_auto - 1; s >= 1; --s) {
      const size_t n = fp8pa_workspace_size(batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv, head_dim,
                                            q_dtype, max_pages_per_seq, window_left, s);
      if (n != 0 && n <= (size_t)FP8PA_NOALLOC_SCRATCH_BYTES) {
        num_splits = s;
        need = n;
        break;
      }
    }
  }
  if (need == 0) {
    // rejected shape: let the regular entry point produce its message
    return fp8_paged_attn_fwd(q, q_dtype, k_cache, v_cache, num_pages, block_table, max_pages_per_seq,
                              cu_seqlens_q, seqused_k, batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv,
                              head_dim, q_descale, k_descale, v_descale, descale_batch_stride, descale_head_stride,
                              softmax_scale, window_left, causal, num_splits, nullptr, 0, out, lse, stream);
  }
  if (need > (size_t)FP8PA_NOALLOC_SCRATCH_BYTES) {
    snprintf(g_noalloc_err, sizeof g_noalloc_err,
             "fp8_paged_attn_fwd_noalloc: this call needs %zu bytes of scratch, more than the %zu bytes the "
             "library holds; use fp8_paged_attn_fwd with a workspace, or fewer splits",
             need, (size_t)FP8PA_NOALLOC_SCRATCH_BYTES);
    return fp8pa::set_last_error(FP8PA_EINVAL, g_noalloc_err);
  }
  void* scratch = nullptr;
  int rc = scratch_address(&scratch, g_noalloc_err, sizeof g_noalloc_err);
  if (rc != FP8PA_OK) return fp8pa::set_last_error(rc, g_noalloc_err);
  // Nothing in the scratch has to start at zero: the plan kernel rewrites the
  // work counters and list on every call, and every split partial is written
  // before the combine reads it.
  return fp8_paged_attn_fwd(q, q_dtype, k_cache, v_cache, num_pages, block_table, max_pages_per_seq, cu_seqlens_q,
                            seqused_k, batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv, head_dim, q_descale,
                            k_descale, v_descale, descale_batch_stride, descale_head_stride, softmax_scale,
                            window_left, causal, num_splits, scratch, (size_t)FP8PA_NOALLOC_SCRATCH_BYTES, out, lse,
                            stream);
}
