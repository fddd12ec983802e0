// Internal launcher interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace fp8pa {

struct PlanParams {
  const int32_t* cu_seqlens_q;
  const int32_t* seqused_k;
  int batch, total_q, group, hkv, max_pages, window_left, causal;
  int num_classes;
  ClassInfo cls[2];
  int4* work[2];
  int* counts;  // [5]: item counts of the two classes, their dynamic counters, SMs of the prefill class
  unsigned* status;
  // Side-by-side split of the SMs between the two classes (counts[4]), from the
  // classes' work: prefill-class time = visible flops * pf_ns_flop / SMs, decode-
  // class time = visible K/V bytes / min(SMs * dec_gbs_sm, dec_gbs).
  int hq, head_dim, sms;
  float pf_ns_flop;  // ns x SMs per visible flop of a prefill-class tile
  float dec_gbs_sm;  // decode-class bytes per ns one SM streams
  float dec_gbs;     // decode-class bytes per ns the whole GPU streams
  int forced_split;  // > 0: SMs of the prefill class (tuning hook), instead of the estimate
};

struct CombineParams {
  const int32_t* cu_seqlens_q;
  const int32_t* seqused_k;
  int batch, total_q, hq, group, head_dim, max_pages, window_left, causal;
  ClassInfo cls;
  const float* o_part;
  const float* lse_part;
  void* out;
  float* lse;
  const float* sinks;  // [hq] sink logits (natural log), or null
};

cudaError_t launch_plan(const PlanParams& pp, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& cp, cudaStream_t stream);
cudaError_t launch_quantize_q(const void* q_bf16, void* q_e4m3, const float* q_descale, long long n,
                              cudaStream_t stream);
cudaError_t launch_lse_combine(const void* o_parts, const float* lse_parts, int parts, long long total_q, int hq,
                               int head_dim, void* out, float* lse_out, int sms, cudaStream_t stream);
cudaError_t launch_kv_cache_write(const void* key, const void* value, long long key_stride, long long value_stride,
                                  uint8_t* k_cache, uint8_t* v_cache, const long long* slot_mapping,
                                  long long num_tokens, int row_elems, long long num_slots, const float* k_descale,
                                  const float* v_descale, unsigned* status, int sms, cudaStream_t stream);

// Attention kernel launchers, one per (head dim, Q type, rows per tile, CTAs per SM);
// every CTA is persistent over the class's work list.
// `ctas` CTAs per SM, `sms` SMs: grid = sms * ctas persistent CTAs.
// path: kPathE4M3, kPathBf16 or kPathBf16DqV (common.cuh).
cudaError_t launch_attn(int head_dim, int path, int rows, int ctas, const AttnParams& p, const CUtensorMap& tm_q,
                        const CUtensorMap& tm_k, const CUtensorMap& tm_v, int sms, cudaStream_t stream);

// Launches `kernel` with programmatic stream serialization: it may start while
// the previous kernel in the stream is still running, so it must call
// griddep_wait() before it touches memory that kernel may write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Prefill row tiles (128 packed rows, rows on the TMEM lanes), E4M3 Q at head dim 256
// or 512 (the latter with two output-dim slices per row tile): one persistent CTA per SM.
cudaError_t launch_attn_prefill_d256(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                     const CUtensorMap& tm_v, int sms, cudaStream_t stream);
cudaError_t launch_attn_prefill_d512(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                     const CUtensorMap& tm_v, int sms, cudaStream_t stream);

// Records a message for fp8pa_last_error() on this thread; returns `code`.
int set_last_error(int code, const char* msg);

// Shared-memory bytes of a kernel variant (0 if the variant does not exist).
int attn_smem_bytes(int head_dim, int path, int rows, int ctas);

}  // namespace fp8pa
