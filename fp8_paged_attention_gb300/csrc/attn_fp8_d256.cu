// Attention kernel instances: head dim 256, E4M3 Q (FP8 MMA).
#include "attn_launch.cuh"

namespace fp8pa {

cudaError_t launch_attn_fp8_d256(int rows, const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, int grid, cudaStream_t stream) {
  switch (rows) {
    case 16: return launch_attn_variant<256, true, 16>(p, tm_q, tm_k, tm_v, grid, stream);
    case 32: return launch_attn_variant<256, true, 32>(p, tm_q, tm_k, tm_v, grid, stream);
    case 64: return launch_attn_variant<256, true, 64>(p, tm_q, tm_k, tm_v, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

int smem_attn_fp8_d256(int rows) {
  switch (rows) {
    case 16: return AttnCfg<256, true, 16>::kSmemBytes;
    case 32: return AttnCfg<256, true, 32>::kSmemBytes;
    case 64: return AttnCfg<256, true, 64>::kSmemBytes;
    default: return 0;
  }
}

}  // namespace fp8pa
