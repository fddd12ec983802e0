// Prefill-tile attention kernel, E4M3 Q at head dim 512 (128 packed rows per
// tile, output dims in two 256-wide work items).
#include "attn_prefill.cuh"

namespace fp8pa {

cudaError_t launch_attn_prefill_d512(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                     const CUtensorMap& tm_v, int sms, cudaStream_t stream) {
  return launch_attn_prefill<512>(p, tm_q, tm_k, tm_v, sms, stream);
}

}  // namespace fp8pa
