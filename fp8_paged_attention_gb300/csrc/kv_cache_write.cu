// Paged KV-cache write: newly generated keys and values are quantized to E4M3
// and scattered into their 64-token pages ("Why FP8 is slower than BF16": the
// KV-cache writes row of the profiling table, the kernels that reshape and write
// new keys and values into the paged cache, FP8 conversion included).
//
// Token t goes to slot s = slot_mapping[t], i.e. row s % 64 of page s / 64 of
// the [pages][64][Hkv][D] cache; a negative slot is a padding token.  Each
// element is quantized like Q: E4M3_RNE_sat(fl32(x / descale)), an IEEE fp32
// division then the hardware round-to-nearest-even saturating conversion, a NaN
// quotient mapped to 0x7F with the input's sign.
//
// The op is HBM-bound (2 bytes read, 1 written per element).  One unit is one
// (token, tensor) row: Hkv * D contiguous bf16 elements in, the same number of
// contiguous bytes out.  A warp runs one unit at a time, four 16-byte vectors
// per lane in flight per pass, and fetches the slot of its next unit while it
// converts the current one; units go to warps with the stride of the grid.
//
// Each pair of elements is settled by the quantizer's fast form or queued: the
// pairs a pass leaves unsettled (quotients within a few ulps of an E4M3
// rounding boundary, NaNs) go to a per-warp queue in shared memory, the warp's
// lanes take its entries in turn through the exact form, and each lane patches
// its own codes from the results.  A warp then runs about one exact pair per
// lane per pass even when a short-mantissa descale puts many quotients on
// rounding boundaries, instead of one lane's eight while the others wait.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "fp8pa.h"
#include "kernels.h"
#include "ptx.cuh"
#include "quant_e4m3.cuh"

namespace fp8pa {

namespace {

constexpr int kWarps = 8;    // warps per block
constexpr int kPerLane = 4;  // vectors per lane per pass
constexpr int kPairs = 4 * kPerLane;  // element pairs per lane per pass

__global__ void __launch_bounds__(32 * kWarps, 4) kv_cache_write_kernel(
    const uint16_t* __restrict__ key, const uint16_t* __restrict__ value, long long key_stride,
    long long value_stride, uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
    const long long* __restrict__ slot_mapping, long long num_tokens, int row_vecs, long long num_slots,
    const float* __restrict__ k_descale, const float* __restrict__ v_descale, unsigned* status) {
  // per warp: every lane's input words and codes of a pass (staged only when some
  // pair is unsettled), and the queue of unsettled (lane, pair) positions
  __shared__ __align__(16) uint32_t s_word[kWarps][32 * kPairs];
  __shared__ __align__(16) uint32_t s_code[kWarps][32 * kPairs / 2];
  __shared__ uint16_t s_queue[kWarps][32 * kPairs];
  ptx::griddep_wait();
  const float dk = *k_descale, dv = *v_descale;
  const float rk = __frcp_rn(dk), rv = __frcp_rn(dv);
  const bool fast = quant::fast_ok(dk) && quant::fast_ok(dv);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t* sw = s_word[wid];
  uint16_t* sc = reinterpret_cast<uint16_t*>(s_code[wid]);
  uint16_t* sq = s_queue[wid];
  const long long units = 2 * num_tokens;
  const long long stride = (long long)gridDim.x * kWarps;
  auto token_of = [&](long long u) { return u >= num_tokens ? u - num_tokens : u; };
  long long u = (long long)blockIdx.x * kWarps + wid;
  long long sl = u < units ? slot_mapping[token_of(u)] : -1;
  for (; u < units; u += stride) {
    const long long un = u + stride;
    const long long sl_next = un < units ? slot_mapping[token_of(un)] : -1;  // in flight during this unit
    const bool is_v = u >= num_tokens;
    const long long t = token_of(u);
    if (sl >= num_slots) {
      if (lane == 0 && !is_v) atomicOr(status, (unsigned)FP8PA_DEV_BAD_SLOT);
    } else if (sl >= 0) {
      const uint4* src = reinterpret_cast<const uint4*>(is_v ? value + t * value_stride : key + t * key_stride);
      uint2* dst = reinterpret_cast<uint2*>((is_v ? v_cache : k_cache) + sl * (long long)row_vecs * 8);
      const float d = is_v ? dv : dk, r = is_v ? rv : rk;
      // warp-uniform passes: lane l takes vectors c0 + l + 32 k
      for (int c0 = 0; c0 < row_vecs; c0 += 32 * kPerLane) {
        uint4 a[kPerLane];
        uint2 c[kPerLane];
#pragma unroll
        for (int k = 0; k < kPerLane; ++k)
          if (c0 + lane + 32 * k < row_vecs) a[k] = __ldcs(src + c0 + lane + 32 * k);
        uint32_t m = 0;  // unsettled pairs of this lane: bit 4 k + j is word j of vector k
        if (fast) {
#pragma unroll
          for (int k = 0; k < kPerLane; ++k)
            if (c0 + lane + 32 * k < row_vecs) m |= quant::fast8_masked(a[k], r, c[k]) << (4 * k);
        } else {
#pragma unroll
          for (int k = 0; k < kPerLane; ++k)
            if (c0 + lane + 32 * k < row_vecs)
              c[k] = make_uint2(quant::exact_pair(a[k].x, d) | (quant::exact_pair(a[k].y, d) << 16),
                                quant::exact_pair(a[k].z, d) | (quant::exact_pair(a[k].w, d) << 16));
        }
        if (__any_sync(0xFFFFFFFFu, m != 0)) {
          // stage the pass in shared memory: lane l's words and codes at l * kPairs + pair
          uint4* w4 = reinterpret_cast<uint4*>(sw + lane * kPairs);
          uint2* c2 = reinterpret_cast<uint2*>(sc + lane * kPairs);
#pragma unroll
          for (int k = 0; k < kPerLane; ++k) {
            w4[k] = a[k];
            c2[k] = c[k];
          }
          // queue this warp's unsettled pairs, lanes in order
          const int cnt = __popc(m);
          int incl = cnt;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += y;
          }
          const int total = __shfl_sync(0xFFFFFFFFu, incl, 31);
          int e = incl - cnt;
          for (uint32_t mm = m; mm; mm &= mm - 1) sq[e++] = (uint16_t)(lane * kPairs + __ffs(mm) - 1);
          __syncwarp();
          // the warp's lanes take the queue's entries in turn through the exact form
          for (int i = lane; i < total; i += 32) {
            const int pos = sq[i];
            sc[pos] = (uint16_t)quant::exact_pair(sw[pos], d);
          }
          __syncwarp();
#pragma unroll
          for (int k = 0; k < kPerLane; ++k) c[k] = c2[k];
          __syncwarp();  // the staging buffers are free for the next pass
        }
#pragma unroll
        for (int k = 0; k < kPerLane; ++k)
          if (c0 + lane + 32 * k < row_vecs) dst[c0 + lane + 32 * k] = c[k];
      }
    }
    sl = sl_next;
  }
  ptx::griddep_launch_dependents();
}

}  // namespace

cudaError_t launch_kv_cache_write(const void* key, const void* value, long long key_stride, long long value_stride,
                                  uint8_t* k_cache, uint8_t* v_cache, const long long* slot_mapping,
                                  long long num_tokens, int row_elems, long long num_slots, const float* k_descale,
                                  const float* v_descale, unsigned* status, int sms, cudaStream_t stream) {
  if (num_tokens <= 0) return cudaSuccess;
  const long long units = 2 * num_tokens;
  const long long cap = 4LL * sms;  // resident blocks (64 registers a thread: four per SM)
  const long long want = (units + kWarps - 1) / kWarps;
  const unsigned blocks = (unsigned)(want < cap ? want : cap);
  return launch_pdl(kv_cache_write_kernel, dim3(blocks), dim3(32 * kWarps), 0, stream,
                    reinterpret_cast<const uint16_t*>(key), reinterpret_cast<const uint16_t*>(value), key_stride,
                    value_stride, k_cache, v_cache, slot_mapping, num_tokens, row_elems / 8, num_slots, k_descale,
                    v_descale, status);
}

}  // namespace fp8pa
