// Q -> E4M3 quantization (the sliding-window layers quantize Q to FP8, vLLM
// PR 63139, Overview).  q8 = RNE_saturate_e4m3(fl32(q / q_descale)): an IEEE
// fp32 division, then the hardware round-to-nearest-even, saturating E4M3
// conversion; a NaN quotient is mapped explicitly to 0x7F with the input's sign bit.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace fp8pa {

namespace {

// A NaN quotient (NaN input, 0/0, inf/inf) gives 0x7F carrying the sign bit of
// the bf16 input; the division itself may return a NaN of either sign.
__device__ __forceinline__ uint8_t quant_one(uint16_t bits, float d) {
  const float x = __uint_as_float((uint32_t)bits << 16);
  const float v = __fdiv_rn(x, d);
  if (v != v) return (uint8_t)(0x7F | ((bits >> 8) & 0x80));
  return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// 8 elements per thread when both pointers allow 16-byte / 8-byte accesses.
__global__ void quantize_q_vec8(const uint4* __restrict__ q, uint2* __restrict__ out, const float* __restrict__ qd,
                                long long n8) {
  ptx::griddep_wait();
  const float d = *qd;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
    const uint4 v = q[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[2] = {0, 0};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint16_t bits = (uint16_t)(w[k >> 1] >> (16 * (k & 1)));
      o[k >> 2] |= (uint32_t)quant_one(bits, d) << (8 * (k & 3));
    }
    out[i] = make_uint2(o[0], o[1]);
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
    out[i] = quant_one(q[i], d);
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
      cudaError_t e = launch_pdl(quantize_q_vec8, dim3((unsigned)(blocks < 4096 ? blocks : 4096)), dim3(256), 0, stream,
                                 reinterpret_cast<const uint4*>(q_bf16), reinterpret_cast<uint2*>(q_e4m3), q_descale,
                                 n8);
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
