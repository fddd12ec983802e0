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
// contiguous bytes out.  A work item is one warp pass over a row: 128 16-byte
// vectors, four per lane.  Items go to warps with the stride of the grid (a
// row's items to neighbouring warps); items of one pass rather than whole rows
// keep the last round of the grid short when rows are few.
//
// Each warp streams its items through a three-stage ring in shared memory:
// every lane copies its own four vectors of an item with cp.async two items
// ahead of the one it converts, so two items' reads stay in flight while the
// lanes convert (a lane reads back only what it copied itself, so no barrier is
// needed between lanes).  The slot of the next item is fetched while the
// current one converts.
//
// The quantizer's fast form settles every element but those of NaN or infinite
// inputs and overflowing quotients; a lane redoes a vector holding such a code
// through the exact form.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "fp8pa.h"
#include "kernels.h"
#include "ptx.cuh"
#include "quant_e4m3.cuh"

namespace fp8pa {

namespace {

constexpr int kWarps = 8;                 // warps per block
constexpr int kPerLane = 4;               // vectors per lane per item
constexpr int kItemVecs = 32 * kPerLane;  // 16-byte vectors per work item
constexpr int kStages = 3;                // ring stages per warp
constexpr int kSmemBytes = kWarps * kStages * kItemVecs * 16;

__device__ __forceinline__ void cp_async16(uint4* dst, const uint4* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ptx::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__global__ void __launch_bounds__(32 * kWarps, 4) kv_cache_write_kernel(
    const uint16_t* __restrict__ key, const uint16_t* __restrict__ value, long long key_stride,
    long long value_stride, uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
    const long long* __restrict__ slot_mapping, long long num_tokens, int row_vecs, long long num_slots,
    const float* __restrict__ k_descale, const float* __restrict__ v_descale, unsigned* status) {
  extern __shared__ uint4 s_ring[];  // [kWarps][kStages][kItemVecs]
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint4* ring = s_ring + wid * (kStages * kItemVecs);
  const int ipu = (row_vecs + kItemVecs - 1) / kItemVecs;  // items per unit
  const long long units = 2 * num_tokens;
  // item i is pass i % ipu of unit i / ipu; a warp walks items with the grid's
  // stride, carried as (units, passes) so that no division runs per item
  const long long stride = (long long)gridDim.x * kWarps;
  const long long su = stride / ipu;
  const int sp = (int)(stride - su * ipu);
  auto advance = [&](long long& ui, int& pi) {
    pi += sp;
    ui += su;
    if (pi >= ipu) {
      pi -= ipu;
      ++ui;
    }
  };
  auto token_of = [&](long long x) { return x >= num_tokens ? x - num_tokens : x; };
  auto row_of = [&](long long ui) {
    const long long ti = token_of(ui);
    return reinterpret_cast<const uint4*>(ui >= num_tokens ? value + ti * value_stride : key + ti * key_stride);
  };
  // copies item (ui, pi) into ring stage `st` (this lane's vectors only); one
  // commit group per call, empty past the last unit
  auto issue = [&](long long ui, int pi, int st) {
    if (ui < units) {
      const uint4* src = row_of(ui) + pi * kItemVecs;
      const int nvec = row_vecs - pi * kItemVecs;
#pragma unroll
      for (int k = 0; k < kPerLane; ++k)
        if (lane + 32 * k < nvec) cp_async16(ring + st * kItemVecs + lane + 32 * k, src + lane + 32 * k);
    }
    cp_async_commit();
  };
  const long long first = (long long)blockIdx.x * kWarps + wid;
  long long u = first / ipu;
  int p = (int)(first - u * ipu);
  ptx::griddep_wait();
  long long ua = u;
  int pa = p;
#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) {
    issue(ua, pa, st);
    advance(ua, pa);
  }
  const float dk = *k_descale, dv = *v_descale;
  const float yk = __frcp_rn(dk), yv = __frcp_rn(dv);
  const bool fast = quant::fast_ok(dk) && quant::fast_ok(dv);
  long long sl = u < units ? slot_mapping[token_of(u)] : -1;
  int st = 0;
  while (u < units) {
    issue(ua, pa, st == 0 ? kStages - 1 : st - 1);  // the stage converted last round
    advance(ua, pa);
    long long un = u;
    int pn = p;
    advance(un, pn);
    const long long sl_next = un < units ? slot_mapping[token_of(un)] : -1;  // in flight during this item
    cp_async_wait<kStages - 1>();  // this lane's copies of the current item have landed
    const bool is_v = u >= num_tokens;
    if (sl >= num_slots) {
      if (lane == 0 && !is_v && p == 0) atomicOr(status, (unsigned)FP8PA_DEV_BAD_SLOT);
    } else if (sl >= 0) {
      uint2* dst = reinterpret_cast<uint2*>((is_v ? v_cache : k_cache) + sl * (long long)row_vecs * 8);
      const float d = is_v ? dv : dk;
      const int c0 = p * kItemVecs;
      const uint4* in = ring + st * kItemVecs;
#pragma unroll
      for (int k = 0; k < kPerLane; ++k) {
        if (c0 + lane + 32 * k < row_vecs) {
          const uint4 a = in[lane + 32 * k];
          uint2 c, f = make_uint2(1, 0);
          if (fast) c = quant::fast8(a, is_v ? yv : yk, -d, f);
          // a flagged code (NaN or infinite input, overflowing quotient): exact form for the vector
          if (f.x | f.y)
            c = make_uint2(quant::exact_pair(a.x, d) | (quant::exact_pair(a.y, d) << 16),
                           quant::exact_pair(a.z, d) | (quant::exact_pair(a.w, d) << 16));
          dst[c0 + lane + 32 * k] = c;
        }
      }
    }
    sl = sl_next;
    u = un;
    p = pn;
    st = st == kStages - 1 ? 0 : st + 1;
  }
  cp_async_wait<0>();
  ptx::griddep_launch_dependents();
}

}  // namespace

cudaError_t launch_kv_cache_write(const void* key, const void* value, long long key_stride, long long value_stride,
                                  uint8_t* k_cache, uint8_t* v_cache, const long long* slot_mapping,
                                  long long num_tokens, int row_elems, long long num_slots, const float* k_descale,
                                  const float* v_descale, unsigned* status, int sms, cudaStream_t stream) {
  if (num_tokens <= 0) return cudaSuccess;
  const long long items = 2 * num_tokens * ((row_elems / 8 + kItemVecs - 1) / kItemVecs);
  const long long cap = 4LL * sms;  // resident blocks (64 registers a thread, 48 KB of ring: four per SM)
  const long long want = (items + kWarps - 1) / kWarps;
  const unsigned blocks = (unsigned)(want < cap ? want : cap);
  // the attribute is per device; setting it again is cheap and capture-safe
  cudaError_t e = cudaFuncSetAttribute(kv_cache_write_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return launch_pdl(kv_cache_write_kernel, dim3(blocks), dim3(32 * kWarps), (size_t)kSmemBytes, stream,
                    reinterpret_cast<const uint16_t*>(key), reinterpret_cast<const uint16_t*>(value), key_stride,
                    value_stride, k_cache, v_cache, slot_mapping, num_tokens, row_elems / 8, num_slots, k_descale,
                    v_descale, status);
}

}  // namespace fp8pa
