// Attention kernel instances: head dim 512, BF16 Q, K and V dequantized to BF16.
#include "attn_launch.cuh"

namespace fp8pa {

// rows: 16, 32 or 64 query rows per tile; ctas: CTAs per SM (1 or 2).
cudaError_t launch_attn_bf16dqv_d512(int rows, int ctas, const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                        const CUtensorMap& tm_v, int sms, cudaStream_t stream) {
  switch (rows * 2 + ctas) {
    case 16 * 2 + 1: return launch_attn_variant<512, kPathBf16DqV, 16, 1>(p, tm_q, tm_k, tm_v, sms, stream);
    case 32 * 2 + 1: return launch_attn_variant<512, kPathBf16DqV, 32, 1>(p, tm_q, tm_k, tm_v, sms, stream);
    case 64 * 2 + 1: return launch_attn_variant<512, kPathBf16DqV, 64, 1>(p, tm_q, tm_k, tm_v, sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

int smem_attn_bf16dqv_d512(int rows, int ctas) {
  switch (rows * 2 + ctas) {
    case 16 * 2 + 1: return AttnCfg<512, kPathBf16DqV, 16, 1>::kSmemBytes;
    case 32 * 2 + 1: return AttnCfg<512, kPathBf16DqV, 32, 1>::kSmemBytes;
    case 64 * 2 + 1: return AttnCfg<512, kPathBf16DqV, 64, 1>::kSmemBytes;
    default: return 0;
  }
}

}  // namespace fp8pa
