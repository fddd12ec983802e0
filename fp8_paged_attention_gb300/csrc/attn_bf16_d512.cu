// Attention kernel instances: head dim 512, BF16 Q (K/V dequantized to BF16, BF16 MMA).
#include "attn_launch.cuh"

namespace fp8pa {

cudaError_t launch_attn_bf16_d512(int rows, const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, int grid, cudaStream_t stream) {
  switch (rows) {
    case 16: return launch_attn_variant<512, false, 16>(p, tm_q, tm_k, tm_v, grid, stream);
    case 32: return launch_attn_variant<512, false, 32>(p, tm_q, tm_k, tm_v, grid, stream);
    case 64: return launch_attn_variant<512, false, 64>(p, tm_q, tm_k, tm_v, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

int smem_attn_bf16_d512(int rows) {
  switch (rows) {
    case 16: return AttnCfg<512, false, 16>::kSmemBytes;
    case 32: return AttnCfg<512, false, 32>::kSmemBytes;
    case 64: return AttnCfg<512, false, 64>::kSmemBytes;
    default: return 0;
  }
}

}  // namespace fp8pa
