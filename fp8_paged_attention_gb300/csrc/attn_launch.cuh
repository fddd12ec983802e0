// Launch helper for one attention kernel variant.
#pragma once
#include "attn_kernel.cuh"
#include "kernels.h"

namespace fp8pa {

template <int D, int kPath, int N, int kCtas>
cudaError_t launch_attn_variant(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, int sms, cudaStream_t stream) {
  using C = AttnCfg<D, kPath, N, kCtas>;
  const int grid = sms * kCtas;
  // the attribute is per device; setting it again is cheap and capture-safe
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, kPath, N, kCtas>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // programmatic launch: the prologue (barriers, tensor memory, tensor maps)
  // overlaps the plan kernel; the kernel waits for it before reading the work list
  return launch_pdl(attn_fwd_kernel<D, kPath, N, kCtas>, dim3(grid), dim3(C::kThreads), (size_t)C::kSmemBytes,
                    stream, p, tm_q, tm_k, tm_v);
}

}  // namespace fp8pa
