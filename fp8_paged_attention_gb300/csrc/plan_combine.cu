// Device-side work planning and split-KV combine.
//
// plan_kernel turns (cu_seqlens_q, seqused_k) into the work lists of up to two
// sequence classes (decode-like sequences with few query rows, prefill-like
// sequences with many) without any host read of device memory, so a forward
// call stays capturable in a CUDA graph.  Items are ordered KV-head-major, then
// by sequence, row tile and split: CTAs that run side by side then touch the
// same KV head, which keeps shared-prefix pages hot in L2.
//
// combine_kernel merges the per-split partial outputs with their log-sum-exps:
//   L = log sum_s exp(lse_s),  out = sum_s exp(lse_s - L) * O_s
// Splits that saw no key carry lse = -inf and weigh nothing.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace fp8pa {

namespace {

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ int clamp_lk(int lk, int max_pages) {
  const int cap = max_pages * kPage;
  return lk < 0 ? 0 : (lk > cap ? cap : lk);
}

__device__ __forceinline__ bool in_class(int Lq, const ClassInfo& c) { return Lq >= c.lq_min && Lq <= c.lq_max; }

// Query count of sequence b, or 0 (and a status flag) when cu_seqlens_q is not a
// nondecreasing run inside [0, total_q]: such a sequence gets no work.
__device__ __forceinline__ int seq_lq(const PlanParams& pp, int b) {
  const int a = pp.cu_seqlens_q[b], e = pp.cu_seqlens_q[b + 1];
  if (a < 0 || e < a || e > pp.total_q) {
    atomicOr(pp.status, kDevBadLength);
    return 0;
  }
  return e - a;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanParams pp) {
  __shared__ int sums[2][kPlanThreads];
  const int tid = threadIdx.x;
  const int per = (pp.batch + kPlanThreads - 1) / kPlanThreads;
  const int b0 = min(pp.batch, tid * per), b1 = min(pp.batch, b0 + per);
  int cnt[2] = {0, 0};
  for (int b = b0; b < b1; ++b) {
    const int Lq = seq_lq(pp, b);
    const int Lk = clamp_lk(pp.seqused_k[b], pp.max_pages);
    for (int k = 0; k < pp.num_classes; ++k) {
      const ClassInfo& c = pp.cls[k];
      if (Lq > 0 && in_class(Lq, c))
        cnt[k] += seq_row_tiles(Lq, pp.group, c.rows) * seq_splits(Lq, Lk, pp.group, pp.window_left, pp.causal, c);
    }
  }
  sums[0][tid] = cnt[0];
  sums[1][tid] = cnt[1];
  __syncthreads();
  for (int off = 1; off < kPlanThreads; off <<= 1) {
    const int v0 = tid >= off ? sums[0][tid - off] : 0;
    const int v1 = tid >= off ? sums[1][tid - off] : 0;
    __syncthreads();
    sums[0][tid] += v0;
    sums[1][tid] += v1;
    __syncthreads();
  }
  int excl[2] = {sums[0][tid] - cnt[0], sums[1][tid] - cnt[1]};
  const int total[2] = {sums[0][kPlanThreads - 1], sums[1][kPlanThreads - 1]};
  if (tid == 0)
    for (int k = 0; k < 2; ++k) pp.counts[k] = k < pp.num_classes ? total[k] * pp.hkv : 0;
  for (int b = b0; b < b1; ++b) {
    const int Lq = seq_lq(pp, b);
    const int Lk = clamp_lk(pp.seqused_k[b], pp.max_pages);
    for (int k = 0; k < pp.num_classes; ++k) {
      const ClassInfo& c = pp.cls[k];
      if (!(Lq > 0 && in_class(Lq, c))) continue;
      const int rts = seq_row_tiles(Lq, pp.group, c.rows);
      const int ns = seq_splits(Lq, Lk, pp.group, pp.window_left, pp.causal, c);
      for (int hk = 0; hk < pp.hkv; ++hk) {
        int4* dst = pp.work[k] + (size_t)hk * total[k] + excl[k];
        for (int rt = 0; rt < rts; ++rt)
          for (int s = 0; s < ns; ++s) dst[rt * ns + s] = make_int4(b, rt, hk | (s << 16), ns);
      }
      excl[k] += rts * ns;
    }
  }
}

__global__ void __launch_bounds__(128) combine_kernel(CombineParams cp) {
  const int t = blockIdx.x;
  // sequence of token t: largest b with cu_seqlens_q[b] <= t
  int lo = 0, hi = cp.batch - 1, b = 0;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    if (cp.cu_seqlens_q[mid] <= t) {
      b = mid;
      lo = mid + 1;
    } else {
      hi = mid - 1;
    }
  }
  const int qa = cp.cu_seqlens_q[b], qe = cp.cu_seqlens_q[b + 1];
  if (qa < 0 || qe < qa || qe > cp.total_q || t >= qe) return;
  const int Lq = qe - qa;
  if (!(Lq > 0 && in_class(Lq, cp.cls))) return;
  const int Lk = clamp_lk(cp.seqused_k[b], cp.max_pages);
  const int ns = seq_splits(Lq, Lk, cp.group, cp.window_left, cp.causal, cp.cls);
  if (ns <= 1) return;
  const float NEG_INF = __int_as_float(0xFF800000);
  const size_t plane = (size_t)cp.total_q * cp.hq;
  for (int h = 0; h < cp.hq; ++h) {
    float mx = NEG_INF;
    for (int s = 0; s < ns; ++s) mx = fmaxf(mx, cp.lse_part[(size_t)s * plane + (size_t)h * cp.total_q + t]);
    float sum = 0.f;
    if (mx != NEG_INF)
      for (int s = 0; s < ns; ++s) sum += expf(cp.lse_part[(size_t)s * plane + (size_t)h * cp.total_q + t] - mx);
    const float L = (mx == NEG_INF) ? NEG_INF : mx + logf(sum);
    const size_t row = (size_t)t * cp.hq + h;
    for (int d = threadIdx.x; d < cp.head_dim; d += blockDim.x) {
      float o = 0.f;
      if (L != NEG_INF)
        for (int s = 0; s < ns; ++s) {
          const float w = expf(cp.lse_part[(size_t)s * plane + (size_t)h * cp.total_q + t] - L);
          o += w * cp.o_part[((size_t)s * plane + row) * cp.head_dim + d];
        }
      reinterpret_cast<__nv_bfloat16*>(cp.out)[row * cp.head_dim + d] = __float2bfloat16_rn(o);
    }
    if (threadIdx.x == 0 && cp.lse) cp.lse[(size_t)h * cp.total_q + t] = L;
  }
}

}  // namespace

cudaError_t launch_plan(const PlanParams& pp, cudaStream_t stream) {
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(pp);
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineParams& cp, cudaStream_t stream) {
  if (cp.total_q <= 0) return cudaSuccess;
  combine_kernel<<<cp.total_q, 128, 0, stream>>>(cp);
  return cudaGetLastError();
}

}  // namespace fp8pa
