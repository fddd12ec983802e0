/*
 * fp8pa — attention forward over a paged FP8 E4M3 KV cache, for GB300 (sm_103a).
 *
 * C ABI.  Every pointer argument is a DEVICE pointer owned by the caller unless
 * stated otherwise; no call allocates device memory, synchronizes the stream or
 * reads device memory from the host, so every call can be captured in a CUDA
 * graph.  All work is enqueued on the caller's stream.  Functions return an
 * fp8pa_status; on a non-zero status nothing was launched and
 * fp8pa_last_error() gives a message naming the offending argument (dtype,
 * head size, ...).
 *
 * Sources.  The operation is the one the Gemma-4 FP8-KV attention paths in
 * vLLM compute:
 *  - "[Kernel] Integrate FA4 SM90 FP8 MMA for Gemma-4 full attention" (vLLM PR
 *    60372), Overview: head-dim-512 full attention with FP8 KV storage and
 *    native BF16 Q, FP8 MMA in-kernel; review thread: 64-token pages
 *    (page_size == tile_n == 64), splits chosen automatically with no
 *    CUDA-graph cap, unsupported combinations rejected before launch.
 *  - vLLM PR 63139, Overview: sliding-window layers at head dim 256 quantize Q
 *    to FP8 and run a native FP8 (E4M3 Q/K/V) forward.
 *  - vLLM PR 48666 summary (prhub), flash_attn_varlen_func snippet: paged FP8
 *    E4M3 K/V dequantized in-kernel with the K/V descales folded in, BF16 Q,
 *    output written in the native dtype, (batch, num_kv_heads) f32 descales,
 *    softmax_lse returned.
 */
#ifndef FP8PA_H_
#define FP8PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (0 = legacy default stream). */
typedef struct CUstream_st* fp8pa_stream_t;

typedef enum {
  FP8PA_OK = 0,
  FP8PA_EINVAL = 1,        /* bad argument: null pointer, size, alignment, workspace too small */
  FP8PA_EUNSUPPORTED = 2,  /* valid but unsupported combination (head dim, Q dtype, ...) */
  FP8PA_ECUDA = 3,         /* a CUDA runtime call failed (message has the CUDA error) */
  FP8PA_EDEVICE = 4        /* returned by fp8pa_get_device_status when device flags are set */
} fp8pa_status;

typedef enum { FP8PA_BF16 = 0, FP8PA_E4M3 = 1 } fp8pa_dtype;

/* Bits of the device status word (see fp8pa_get_device_status). */
enum {
  FP8PA_DEV_BAD_PAGE = 1,   /* a block-table entry outside [0, num_pages): that page read as zeros */
  FP8PA_DEV_TIMEOUT = 2,    /* a bounded pipeline wait ran out; the kernel stopped early */
  FP8PA_DEV_BAD_LENGTH = 4, /* seqused_k[b] > 64 * max_pages_per_seq or < 0: clamped */
  FP8PA_DEV_BAD_SLOT = 8    /* fp8pa_kv_cache_write: a slot >= 64 * num_pages; that token was skipped */
};

/* Tokens per KV-cache page.  Fixed: the cache is laid out in 64-token pages
 * (PR 60372 review thread: page_size == tile_n == 64). */
#define FP8PA_PAGE_SIZE 64

/*
 * quantize_q_fp8 — Q to E4M3 (PR 63139, Overview: sliding-window layers
 * quantize Q to FP8).
 *   q_e4m3[i] = RNE_saturate_e4m3( fl32( float(q_bf16[i]) / *q_descale ) )
 * i.e. an IEEE fp32 division, then round-to-nearest-even onto E4M3 with
 * saturation to +-448 (also for +-inf); NaN gives 0x7F with the input's sign
 * bit.  q_bf16: n_elems bf16 values; q_e4m3: n_elems bytes; q_descale: one
 * f32 on the device (per tensor).  Any layout (the op is elementwise).
 * Errors: EINVAL for null pointers or n_elems < 0.  n_elems == 0 is a no-op.
 */
int quantize_q_fp8(const void* q_bf16, void* q_e4m3, const float* q_descale, long long n_elems,
                   fp8pa_stream_t stream);

/*
 * fp8pa_kv_cache_write — quantize newly generated keys and values to E4M3 and
 * write them into the paged cache ("Why FP8 is slower than BF16": the
 * KV-cache writes row of the profiling table, the kernels that reshape and
 * write new keys and values into the paged cache, FP8 conversion included).
 *
 *   for every token t with s = slot_mapping[t] >= 0:
 *     k_cache[s / 64][s % 64][h][d] = RNE_saturate_e4m3( fl32( key[t][h][d] / *k_descale ) )
 *     v_cache[s / 64][s % 64][h][d] = RNE_saturate_e4m3( fl32( value[t][h][d] / *v_descale ) )
 *
 * with the rounding of quantize_q_fp8 (IEEE fp32 division, round to nearest
 * even, saturation to +-448, NaN to 0x7F with the input's sign bit).
 *
 * key, value: bf16, token t's num_heads_kv * head_dim elements contiguous at
 *   element offset t * key_token_stride (value_token_stride); 16-byte aligned,
 *   strides multiples of 8 elements (a slice of a fused QKV buffer qualifies).
 * k_cache, v_cache: uint8 [num_pages][64][num_heads_kv][head_dim], 8-byte
 *   aligned, the layout fp8_paged_attn_fwd reads.
 * slot_mapping: int64 [num_tokens] on the device; a negative slot is a padding
 *   token and writes nothing; a slot >= 64 * num_pages is skipped and sets
 *   FP8PA_DEV_BAD_SLOT in the device status word.
 * k_descale, v_descale: one f32 each on the device (per tensor).
 * Caller owns every buffer; nothing is allocated; graph-capturable (one
 * launch, no host synchronisation).  Two tokens mapped to one slot race: the
 * caller gives distinct slots.
 * Errors: EINVAL for null pointers, num_tokens < 0, num_heads_kv or head_dim
 * < 1, num_heads_kv * head_dim not a multiple of 8, misaligned pointers or
 * strides; ECUDA when the launch fails.  num_tokens == 0 is a no-op.
 */
int fp8pa_kv_cache_write(const void* key, const void* value, long long key_token_stride,
                         long long value_token_stride, uint8_t* k_cache, uint8_t* v_cache, int num_pages,
                         const int64_t* slot_mapping, long long num_tokens, int num_heads_kv, int head_dim,
                         const float* k_descale, const float* v_descale, fp8pa_stream_t stream);

/*
 * fp8_paged_attn_fwd_sinks — fp8_paged_attn_fwd with attention sinks (a
 * feature of the d512 kernel in the review of "[Kernel] Integrate FA4 SM90 FP8
 * MMA for Gemma-4 full attention": "including sinks").  Every argument is that
 * of fp8_paged_attn_fwd; sinks: f32 [num_heads_q] on the device, natural-log
 * units, not null.  Query head h's sink is one more logit in its softmax
 * denominator that attends to no value:
 *   out = sum_j e^{s_j} v_j / (sum_j e^{s_j} + e^{sinks[h]}),
 *   lse = ln(sum_j e^{s_j} + e^{sinks[h]});
 * a row with no visible key gets out = 0 and lse = sinks[h].  A sink of -inf
 * gives the results of fp8_paged_attn_fwd.  Errors: those of
 * fp8_paged_attn_fwd, and EINVAL for null or misaligned sinks.
 */
int fp8_paged_attn_fwd_sinks(const void* q, int q_dtype, const uint8_t* k_cache, const uint8_t* v_cache,
                             int num_pages, const int32_t* block_table, int max_pages_per_seq,
                             const int32_t* cu_seqlens_q, const int32_t* seqused_k, int batch, int total_q,
                             int max_seqlen_q, int num_heads_q, int num_heads_kv, int head_dim, const float* q_descale,
                             const float* k_descale, const float* v_descale, int descale_batch_stride,
                             int descale_head_stride, float softmax_scale, int window_left, int causal,
                             int num_splits, void* workspace, size_t workspace_bytes, void* out, float* lse,
                             const float* sinks, fp8pa_stream_t stream);

/*
 * fp8pa_lse_combine — merge attention partials computed over disjoint key
 * shards, as the context call of decode-context parallelism returns them (the
 * pages' review thread on DCP: each rank runs the non-causal context call over
 * its shard of the keys as local attention with a window covering every key,
 * and returns O and LSE).  Per (token, head) row:
 *
 *   L = ln sum_s exp(lse_parts[s]),   out = sum_s exp(lse_parts[s] - L) * o_parts[s]
 *
 * Parts with LSE = -inf add nothing; a row with no part gives out = 0 and
 * L = -inf.  Arithmetic in f32; out rounded to bf16.
 *
 * o_parts: bf16 [num_parts][total_q][num_heads_q][head_dim] (the out of each
 *   part's fp8_paged_attn_fwd call), 16-byte aligned.
 * lse_parts: f32 [num_parts][num_heads_q][total_q] (each call's lse), natural log.
 * out: bf16 [total_q][num_heads_q][head_dim], 16-byte aligned; lse_out: f32
 *   [num_heads_q][total_q] or NULL.  out must not overlap o_parts.
 * Caller owns every buffer; nothing is allocated; graph-capturable.
 * Errors: EINVAL for null pointers, num_parts < 1, total_q < 0, num_heads_q
 * < 1, head_dim not a positive multiple of 8, misaligned pointers; ECUDA when
 * the launch fails.  total_q == 0 is a no-op.
 */
int fp8pa_lse_combine(const void* o_parts, const float* lse_parts, int num_parts, long long total_q,
                      int num_heads_q, int head_dim, void* out, float* lse_out, fp8pa_stream_t stream);

/*
 * fp8_paged_attn_fwd_noalloc — the same forward as fp8_paged_attn_fwd (same
 * arguments, layouts and results) for callers that cannot allocate device
 * memory at call time: for instance an inference engine that reserves nearly
 * all HBM for its KV-cache pool at start-up, or a plugin host that gives the
 * library no allocator.  It allocates nothing: its scratch is a device array
 * of FP8PA_NOALLOC_SCRATCH_BYTES inside the library, which every device that
 * loads the library holds until the process exits.  The caller passes only
 * inputs and outputs.
 *
 * Limits and rules:
 *  - With num_splits = 0 (automatic) and an automatic split count whose
 *    partials do not fit FP8PA_NOALLOC_SCRATCH_BYTES, the call runs the
 *    largest smaller split count that fits (a function of the sizes alone);
 *    its results are those of fp8_paged_attn_fwd with that num_splits.
 *  - Any other call whose scratch need (fp8pa_workspace_size for the same
 *    arguments) exceeds FP8PA_NOALLOC_SCRATCH_BYTES is rejected with
 *    FP8PA_EINVAL and a message; nothing is launched.  Splits above 1 need the
 *    most scratch.
 *  - All calls share the one array on a device: calls whose kernels may
 *    overlap on the GPU (e.g. on different streams without ordering) race and
 *    give undefined results.  Calls ordered on one stream are fine; each call
 *    rewrites all the scratch it reads, so nothing must be cleared between calls.
 *  - Every call looks up the array's device address in the current context
 *    (cudaGetSymbolAddress, a host-side lookup), so the address stays right
 *    after cudaDeviceReset.  The first call on a device may load the library's
 *    device code into that device's context: make that first call before any
 *    stream capture on that device.
 *  - At the speculative-verify size (a few query tokens per sequence, 32 query
 *    heads at head dim 512, 64 sequences) two splits' partials already exceed
 *    the array, so automatic splits step down to one split and the call runs
 *    at the unsplit kernel's speed.
 * This entry point has no counterpart on the source pages: it is a deployment
 * convenience of this library.
 */
#define FP8PA_NOALLOC_SCRATCH_BYTES (32u << 20)
int fp8_paged_attn_fwd_noalloc(const void* q, int q_dtype, const uint8_t* k_cache, const uint8_t* v_cache,
                               int num_pages, const int32_t* block_table, int max_pages_per_seq,
                               const int32_t* cu_seqlens_q, const int32_t* seqused_k, int batch, int total_q,
                               int max_seqlen_q, int num_heads_q, int num_heads_kv, int head_dim,
                               const float* q_descale, const float* k_descale, const float* v_descale,
                               int descale_batch_stride, int descale_head_stride, float softmax_scale,
                               int window_left, int causal, int num_splits, void* out, float* lse,
                               fp8pa_stream_t stream);

/*
 * fp8pa_workspace_size — bytes of device workspace fp8_paged_attn_fwd needs for
 * these host-known sizes and Q dtype (same values as passed to fp8_paged_attn_fwd).  The
 * workspace holds the device-built work list and, when the split count is
 * above 1, the per-split partial outputs and log-sum-exps.  Returns 0 for
 * arguments fp8_paged_attn_fwd would reject.
 */
size_t fp8pa_workspace_size(int batch, int total_q, int max_seqlen_q, int num_heads_q, int num_heads_kv,
                            int head_dim, int q_dtype, int max_pages_per_seq, int window_left, int num_splits);

/*
 * fp8pa_num_splits — the split-KV count fp8_paged_attn_fwd uses for these
 * host-known sizes (num_splits = 0 asks for the automatic choice, which is a
 * pure function of its arguments, the SM count and the kernel variant's CTAs
 * per SM, so it is CUDA-graph safe).
 * Returns 0 for arguments fp8_paged_attn_fwd would reject.
 */
int fp8pa_num_splits(int batch, int total_q, int max_seqlen_q, int num_heads_q, int num_heads_kv, int head_dim, int q_dtype,
                     int max_pages_per_seq, int window_left, int num_splits);

/*
 * fp8_paged_attn_fwd — varlen attention forward over a paged E4M3 KV cache.
 *
 * Layouts (row-major, innermost last):
 *   q            [total_q][num_heads_q][head_dim]   bf16 (q_dtype = FP8PA_BF16) or
 *                                                    E4M3 bytes (FP8PA_E4M3, e.g. from quantize_q_fp8)
 *   k_cache,
 *   v_cache      [num_pages][64][num_heads_kv][head_dim] E4M3 bytes
 *   block_table  [batch][max_pages_per_seq] int32: physical page of logical page j of sequence b
 *   cu_seqlens_q [batch + 1] int32, nondecreasing, cu_seqlens_q[0] = 0, cu_seqlens_q[batch] = total_q
 *   seqused_k    [batch] int32: keys of sequence b, including its new tokens (already written)
 *   out          [total_q][num_heads_q][head_dim] bf16
 *   lse          [num_heads_q][total_q] f32, natural log; may be NULL
 *
 * Semantics, per sequence b with Lq = cu_seqlens_q[b+1] - cu_seqlens_q[b] and
 * Lk = seqused_k[b], query i (0 <= i < Lq) at position p = Lk - Lq + i and
 * query head h on KV head hk = h / (num_heads_q / num_heads_kv):
 *   visible keys J = [lo, hi], lo = max(0, p - window_left) if window_left >= 0 else 0,
 *                               hi = min(p, Lk - 1) if causal else Lk - 1
 *   s_j = softmax_scale * (q . k_j),  with q = code * q_descale (E4M3 Q) or the bf16 value,
 *         k_j = code * k_descale[b, hk]
 *   out = sum_j softmax(s)_j * v_j,   v_j = code * v_descale[b, hk];  lse = ln sum_j exp(s_j)
 *   An empty J gives out = 0 and lse = -inf.
 * q_descale: one f32 (per tensor; read only on the E4M3-Q path).  k_descale,
 * v_descale: f32 read at b * descale_batch_stride + hk * descale_head_stride
 * (0, 0 = per tensor).  A NULL descale pointer is the unit scale 1.0 and is
 * never read (the no-descale fast path for caches stored without scaling).
 *
 * Support: head_dim 256 with E4M3 Q; head_dim 512 with BF16 Q or E4M3 Q.  With
 * BF16 Q each row of Q is split in-kernel into an exact pair of E4M3 terms under
 * a power-of-two row scale (every value down to 2^-9 of the row's largest is
 * carried exactly) and QK^T runs as FP8 MMAs on the E4M3 K; the result is that
 * of a 16-bit MMA on the dequantized K.  V head dim = head_dim.  num_heads_q
 * a multiple of num_heads_kv with a group size in {1, 2, 4, 8, 16}.
 * window_left >= -1.  num_splits: 0 = automatic, else (1..64) the maximum number
 * of key splits per (sequence, KV head); splits are combined by log-sum-exp.
 * Pointers q, k_cache, v_cache, out must be 16-byte aligned.
 *
 * workspace: device buffer of at least fp8pa_workspace_size(...) bytes, 256-byte
 * aligned; contents need not be initialized and are scratch after the call.
 *
 * Device-side faults are reported, not trapped: a block-table entry outside
 * [0, num_pages) reads that page as zeros and sets FP8PA_DEV_BAD_PAGE; see
 * fp8pa_get_device_status.
 */
int fp8_paged_attn_fwd(const void* q, int q_dtype, const uint8_t* k_cache, const uint8_t* v_cache, int num_pages,
                       const int32_t* block_table, int max_pages_per_seq, const int32_t* cu_seqlens_q,
                       const int32_t* seqused_k, int batch, int total_q, int max_seqlen_q, int num_heads_q,
                       int num_heads_kv, int head_dim, const float* q_descale, const float* k_descale,
                       const float* v_descale, int descale_batch_stride, int descale_head_stride,
                       float softmax_scale, int window_left, int causal, int num_splits, void* workspace,
                       size_t workspace_bytes, void* out, float* lse, fp8pa_stream_t stream);

/*
 * fp8pa_kernel_launches — number of kernels fp8_paged_attn_fwd launches for
 * these host-known sizes (plan, one attention kernel per row class, and the
 * LSE combine when the split count is above 1).  0 for rejected arguments.
 */
int fp8pa_kernel_launches(int batch, int total_q, int max_seqlen_q, int num_heads_q, int num_heads_kv,
                          int head_dim, int q_dtype, int max_pages_per_seq, int window_left, int num_splits);

/*
 * fp8pa_get_device_status — enqueue on `stream` a copy of the current device's
 * status word (FP8PA_DEV_* bits accumulated by earlier launches) into
 * *host_status, which must be pinned host memory; the value is valid once the
 * stream has reached this point.  Returns OK or ECUDA.
 */
int fp8pa_get_device_status(unsigned int* host_status, fp8pa_stream_t stream);

/* fp8pa_reset_device_status — enqueue a clear of the current device's status word. */
int fp8pa_reset_device_status(fp8pa_stream_t stream);

/* fp8pa_last_error — message for the last non-OK status returned on this host thread. */
const char* fp8pa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8PA_H_ */
