// Combine of attention partials computed over disjoint key shards, by their
// LSE: the context call of decode-context parallelism returns O and LSE for
// each rank's shard of the keys (the pages' review thread on DCP: the
// non-causal context call run as local attention with a window covering every
// key).  Per (token, head) row:
//
//   L = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - L) O_s
//
// with parts at LSE = -inf adding nothing and a row with no part giving O = 0,
// L = -inf.  One warp per row: every lane reads the P LSEs (one broadcast load
// each), then sums its 8-element slices of the P bf16 partial rows in f32; for
// up to four parts all of a lane's loads of a pass are issued before any is used.
#include <cuda_bf16.h>

#include "fp8pa.h"
#include "kernels.h"
#include "ptx.cuh"

namespace fp8pa {

namespace {

// kP > 0: exactly kP parts, every load of a lane's two vectors of all parts in
// flight before any is used; kP == 0: any number of parts, one part at a time.
template <int kP>
__global__ void __launch_bounds__(256) lse_combine_kernel(const uint4* __restrict__ o_parts,
                                                          const float* __restrict__ lse_parts, int parts,
                                                          long long total_q, int hq, int vecs, uint4* __restrict__ out,
                                                          float* __restrict__ lse_out) {
  ptx::griddep_wait();
  const int lane = threadIdx.x & 31;
  const long long rows = total_q * hq;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  const float NEG_INF = __int_as_float(0xFF800000);
  const int np = kP > 0 ? kP : parts;
  for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows; row += warps) {
    const long long t = row / hq;
    const int h = (int)(row - t * hq);
    const long long li = (long long)h * total_q + t;
    float m = NEG_INF;
    for (int s = 0; s < np; ++s) m = fmaxf(m, lse_parts[s * rows + li]);
    float L = NEG_INF;
    if (m != NEG_INF) {
      float sum = 0.f;
      for (int s = 0; s < np; ++s) {
        const float ls = lse_parts[s * rows + li];
        if (ls != NEG_INF) sum += expf(ls - m);
      }
      L = m + logf(sum);
    }
    auto accumulate = [&](float (&acc)[8], const uint4& x, float w) {
      const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[2 * k] = fmaf(w, __uint_as_float(u[k] << 16), acc[2 * k]);
        acc[2 * k + 1] = fmaf(w, __uint_as_float(u[k] & 0xFFFF0000u), acc[2 * k + 1]);
      }
    };
    auto store = [&](const float (&acc)[8], int v) {
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * k], acc[2 * k + 1]);
        o[k] = *reinterpret_cast<uint32_t*>(&b);
      }
      out[row * vecs + v] = make_uint4(o[0], o[1], o[2], o[3]);
    };
    if constexpr (kP > 0) {
      float w[kP];
#pragma unroll
      for (int s = 0; s < kP; ++s) {
        const float ls = lse_parts[s * rows + li];
        w[s] = (L == NEG_INF || ls == NEG_INF) ? 0.f : expf(ls - L);
      }
      for (int v = lane; v < vecs; v += 64) {
        const bool two = v + 32 < vecs;
        uint4 x[kP][2];
#pragma unroll
        for (int s = 0; s < kP; ++s) {
          x[s][0] = __ldcs(o_parts + (s * rows + row) * vecs + v);
          if (two) x[s][1] = __ldcs(o_parts + (s * rows + row) * vecs + v + 32);
        }
        float a0[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, a1[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < kP; ++s) {
          // a part with LSE -inf has weight 0 (its row may be 0 or anything finite)
          if (w[s] != 0.f) {
            accumulate(a0, x[s][0], w[s]);
            if (two) accumulate(a1, x[s][1], w[s]);
          }
        }
        store(a0, v);
        if (two) store(a1, v + 32);
      }
    } else {
      for (int v = lane; v < vecs; v += 32) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (L != NEG_INF) {
          for (int s = 0; s < np; ++s) {
            const float ls = lse_parts[s * rows + li];
            if (ls == NEG_INF) continue;
            accumulate(acc, __ldcs(o_parts + (s * rows + row) * vecs + v), expf(ls - L));
          }
        }
        store(acc, v);
      }
    }
    if (lse_out && lane == 0) lse_out[li] = L;
  }
  ptx::griddep_launch_dependents();
}

}  // namespace

cudaError_t launch_lse_combine(const void* o_parts, const float* lse_parts, int parts, long long total_q, int hq,
                               int head_dim, void* out, float* lse_out, int sms, cudaStream_t stream) {
  const long long rows = total_q * hq;
  if (rows <= 0) return cudaSuccess;
  const long long want = (rows + 7) / 8;  // eight warps per block, a row each
  const long long cap = 8LL * sms;
  const dim3 grid((unsigned)(want < cap ? want : cap)), block(256);
  const uint4* op = reinterpret_cast<const uint4*>(o_parts);
  uint4* o = reinterpret_cast<uint4*>(out);
  const int vecs = head_dim / 8;
  switch (parts) {
    case 1: return launch_pdl(lse_combine_kernel<1>, grid, block, 0, stream, op, lse_parts, parts, total_q, hq, vecs, o, lse_out);
    case 2: return launch_pdl(lse_combine_kernel<2>, grid, block, 0, stream, op, lse_parts, parts, total_q, hq, vecs, o, lse_out);
    case 3: return launch_pdl(lse_combine_kernel<3>, grid, block, 0, stream, op, lse_parts, parts, total_q, hq, vecs, o, lse_out);
    case 4: return launch_pdl(lse_combine_kernel<4>, grid, block, 0, stream, op, lse_parts, parts, total_q, hq, vecs, o, lse_out);
    default: return launch_pdl(lse_combine_kernel<0>, grid, block, 0, stream, op, lse_parts, parts, total_q, hq, vecs, o, lse_out);
  }
}

}  // namespace fp8pa
