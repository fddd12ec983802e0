// Attention kernel instances: head dim 512, E4M3 Q (E4M3 MMAs).
#include "attn_launch.cuh"

namespace fp8pa {

// rows: 16, 32 or 64 query rows per tile; ctas: CTAs per SM (1 or 2).
cudaError_t launch_attn_fp8_d512(int rows, int ctas, const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                        const CUtensorMap& tm_v, int sms, cudaStream_t stream) {
  switch (rows * 2 + ctas) {
    case 16 * 2 + 1: return launch_attn_variant<512, kPathE4M3, 16, 1>(p, tm_q, tm_k, tm_v, sms, stream);
    case 32 * 2 + 1: return launch_attn_variant<512, kPathE4M3, 32, 1>(p, tm_q, tm_k, tm_v, sms, stream);
    case 64 * 2 + 1: return launch_attn_variant<512, kPathE4M3, 64, 1>(p, tm_q, tm_k, tm_v, sms, stream);
    case 16 * 2 + 2: return launch_attn_variant<512, kPathE4M3, 16, 2>(p, tm_q, tm_k, tm_v, sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

int smem_attn_fp8_d512(int rows, int ctas) {
  switch (rows * 2 + ctas) {
    case 16 * 2 + 1: return AttnCfg<512, kPathE4M3, 16, 1>::kSmemBytes;
    case 32 * 2 + 1: return AttnCfg<512, kPathE4M3, 32, 1>::kSmemBytes;
    case 64 * 2 + 1: return AttnCfg<512, kPathE4M3, 64, 1>::kSmemBytes;
    case 16 * 2 + 2: return AttnCfg<512, kPathE4M3, 16, 2>::kSmemBytes;
    default: return 0;
  }
}

}  // namespace fp8pa
