// Q -> E4M3 quantization (the sliding-window layers quantize Q to FP8, vLLM
// PR 63139, Overview).  q8 = RNE_saturate_e4m3(fl32(q / q_descale)), computed
// bit-identically without a division (Markstein's correction, quant_e4m3.cuh)
// but for vectors holding NaN or infinite inputs or overflowing quotients; a NaN
// quotient gives 0x7F with the input's sign bit.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"
#include "quant_e4m3.cuh"

namespace fp8pa {

namespace {

// 8 elements per vector when both pointers allow 16-byte / 8-byte accesses; up
// to kV grid-strided vectors per thread and pass, loaded before any converts
// (kV = 1 for inputs that one pass of the grid covers: a short kernel's code
// stays small).
template <int kV>
__global__ void quantize_q_vec8(const uint4* __restrict__ q, uint2* __restrict__ out, const float* __restrict__ qd,
                                long long n8) {
  ptx::griddep_wait();
  const float d = *qd, y = __frcp_rn(d);
  const bool fast = quant::fast_ok(d);
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i0 = blockIdx.x * (long long)blockDim.x + threadIdx.x; i0 < n8; i0 += kV * stride) {
    uint4 v[kV];
#pragma unroll
    for (int k = 0; k < kV; ++k)
      if (i0 + k * stride < n8) v[k] = q[i0 + k * stride];
#pragma unroll
    for (int k = 0; k < kV; ++k) {
      if (i0 + k * stride >= n8) break;
      uint2 c, f = make_uint2(1, 0);
      if (fast) c = quant::fast8(v[k], y, -d, f);
      // a vector with a flagged code (NaN / infinite inputs, overflow) takes the exact form
      if (f.x | f.y)
        c = make_uint2(quant::exact_pair(v[k].x, d) | (quant::exact_pair(v[k].y, d) << 16),
                       quant::exact_pair(v[k].z, d) | (quant::exact_pair(v[k].w, d) << 16));
      out[i0 + k * stride] = c;
    }
  }
  // Let the next kernel (the forward's plan) launch only as this grid drains:
  // launched earlier, the attention grid behind it would take SM room from the
  // blocks still quantizing.
  ptx::griddep_launch_dependents();
}

__global__ void quantize_q_scalar(const uint16_t* __restrict__ q, uint8_t* __restrict__ out,
                                  const float* __restrict__ qd, long long begin, long long n) {
  ptx::griddep_wait();
  const float d = *qd;
  for (long long i = begin + blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    out[i] = (uint8_t)quant::exact_one(q[i], d);
  ptx::griddep_launch_dependents();
}

}  // namespace

cudaError_t launch_quantize_q(const void* q_bf16, void* q_e4m3, const float* q_descale, long long n,
                              cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const bool vec = (reinterpret_cast<uintptr_t>(q_bf16) % 16 == 0) && (reinterpret_cast<uintptr_t>(q_e4m3) % 8 == 0);
  long long done = 0;
  if (vec) {
    const long long n8 = n / 8;
    if (n8 > 0) {
      const long long blocks = (n8 + 255) / 256;
      const dim3 grid((unsigned)(blocks < 4096 ? blocks : 4096));
      const uint4* src = reinterpret_cast<const uint4*>(q_bf16);
      uint2* dst = reinterpret_cast<uint2*>(q_e4m3);
      cudaError_t e = blocks <= 4096 ? launch_pdl(quantize_q_vec8<1>, grid, dim3(256), 0, stream, src, dst, q_descale, n8)
                                     : launch_pdl(quantize_q_vec8<4>, grid, dim3(256), 0, stream, src, dst, q_descale, n8);
      if (e != cudaSuccess) return e;
    }
    done = n8 * 8;
  }
  if (done < n) {
    const long long rest = n - done;
    const long long blocks = (rest + 255) / 256;
    return launch_pdl(quantize_q_scalar, dim3((unsigned)(blocks < 4096 ? blocks : 4096)), dim3(256), 0, stream,
                      reinterpret_cast<const uint16_t*>(q_bf16), reinterpret_cast<uint8_t*>(q_e4m3), q_descale, done,
                      n);
  }
  return cudaSuccess;
}

}  // namespace fp8pa
