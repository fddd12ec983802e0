// Device-side work planning and split-KV combine.
//
// plan_kernel turns (cu_seqlens_q, seqused_k) into the work lists of up to two
// sequence classes (decode-like sequences with few query rows, prefill-like
// sequences with many) without any host read of device memory, so a forward
// call stays capturable in a CUDA graph.  Items are ordered by sequence, then
// KV head, row tile and split: CTAs that run side by side read every KV head
// of the same pages (the heads of one slot are adjacent in memory), and with a
// shared prefix the same pages again a few sequences later, while still in L2.
// A prefill-like sequence with many items lists its row tiles last to first,
// so that a causal chunk's longest units start first and the grid ends on
// short ones: across all KV heads when its class runs alone, one KV head at a
// time when it runs beside the other class.
//
// combine_kernel merges the per-split partial outputs with their log-sum-exps:
//   L = log (sum_s exp(lse_s) + exp(sink)),  out = sum_s exp(lse_s - L) * O_s
// Splits that saw no key carry lse = -inf and weigh nothing; without a sink its
// term is absent.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace fp8pa {

namespace {

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ int clamp_lk(int lk, int max_pages) {
  const int cap = max_pages * kPage;
  return lk < 0 ? 0 : (lk > cap ? cap : lk);
}

__device__ __forceinline__ bool in_class(int Lq, const ClassInfo& c) { return Lq >= c.lq_min && Lq <= c.lq_max; }

// Number of visible (query, key) pairs of a sequence, the sum over its queries
// of |[lo, hi]| (visible_range), in closed form over the query positions
// p = Lk - Lq + i: a sum of arithmetic series.
__device__ long long visible_pairs(int Lq, int Lk, int wl, int causal) {
  if (Lq <= 0 || Lk <= 0) return 0;
  const long long P0 = (long long)Lk - Lq, P1 = (long long)Lk - 1;
  long long total = 0;
  if (causal) {
    // p < 0 sees nothing; p + 1 keys up to p = wl (or always without a window); wl + 1 after
    const long long a = P0 > 0 ? P0 : 0;
    if (a > P1) return 0;
    const long long m = wl < 0 ? P1 : (P1 < wl ? P1 : (long long)wl);
    if (a <= m) total += (m - a + 1) * (a + m + 2) / 2;
    if (wl >= 0) {
      const long long a2 = a > (long long)wl + 1 ? a : (long long)wl + 1;
      if (a2 <= P1) total += (P1 - a2 + 1) * ((long long)wl + 1);
    }
  } else {
    // every key up to p = wl (or always without a window); Lk + wl - p keys after
    const long long m = wl < 0 ? P1 : (P1 < wl ? P1 : (long long)wl);
    if (P0 <= m) total += (m - P0 + 1) * Lk;
    if (wl >= 0) {
      const long long a2 = P0 > (long long)wl + 1 ? P0 : (long long)wl + 1;
      if (a2 <= P1) total += (P1 - a2 + 1) * ((long long)Lk + wl) - (a2 + P1) * (P1 - a2 + 1) / 2;
    }
  }
  return total;
}

// Keys in the union of a sequence's visible ranges (its K/V rows read once per KV head).
__device__ __forceinline__ long long visible_span(int Lq, int Lk, int wl, int causal) {
  if (Lq <= 0 || Lk <= 0) return 0;
  int lo0, hi0, lo1, hi1;
  visible_range(Lq, Lk, 0, wl, causal, lo0, hi0);
  visible_range(Lq, Lk, Lq - 1, wl, causal, lo1, hi1);
  return hi1 >= lo0 ? (long long)hi1 - lo0 + 1 : 0;
}

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

// A sequence whose item list is long (a prefill-like sequence): its first item
// slot, row tiles and splits, in class kc.
struct LongList {
  int b, kc, start, rts, ns;
};
constexpr int kLongQueue = 64;  // long lists the whole block writes; more go to their own warps

// Item i of a long list.  Row tiles run last to first, so that a causal
// sequence's longest units go out first and the grid ends on short ones.
// Alone, the class takes them across all KV heads (row tile, then head, then
// split); beside the other class, whose K/V stream through L2 meanwhile, one
// head at a time (head, then row tile, then split), which keeps fewer of its
// pages hot in L2.
__device__ __forceinline__ void write_long_item(const PlanParams& pp, const LongList& l, int i, bool beside) {
  int hk, rt, s;
  if (beside) {
    const int per_head = l.rts * l.ns;
    hk = i / per_head;
    const int rem = i - hk * per_head;
    rt = l.rts - 1 - rem / l.ns;
    s = rem % l.ns;
  } else {
    const int per_tile = pp.hkv * l.ns;
    rt = l.rts - 1 - i / per_tile;
    const int rem = i % per_tile;
    hk = rem / l.ns;
    s = rem % l.ns;
  }
  pp.work[l.kc][(size_t)l.start * pp.hkv + i] = make_int4(l.b, rt, hk | (s << 16), l.ns);
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanParams pp) {
  static_assert(kPlanThreads == 32 * 32, "two-level warp scan");
  ptx::griddep_launch_dependents();  // the attention grid may start its prologue
  ptx::griddep_wait();               // inputs and the workspace belong to earlier kernels until they finish
  __shared__ int wsum[2][32];
  __shared__ long long wwork[2][32];
  __shared__ LongList long_q[kLongQueue];
  __shared__ int n_long;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) n_long = 0;  // published by the __syncthreads of the scans below
  const int per = (pp.batch + kPlanThreads - 1) / kPlanThreads;
  const int b0 = min(pp.batch, tid * per), b1 = min(pp.batch, b0 + per);
  int cnt[2] = {0, 0};
  long long work[2] = {0, 0};  // decode class: visible span keys; prefill class: visible pairs
  for (int b = b0; b < b1; ++b) {
    const int Lq = seq_lq(pp, b);
    const int Lk = clamp_lk(pp.seqused_k[b], pp.max_pages);
    for (int k = 0; k < pp.num_classes; ++k) {
      const ClassInfo& c = pp.cls[k];
      if (Lq > 0 && in_class(Lq, c)) {
        cnt[k] += seq_row_tiles(Lq, pp.group, c.rows) *
                  unit_items(seq_splits(Lq, Lk, pp.group, pp.window_left, pp.causal, c), c);
        work[k] += k == 0 ? visible_span(Lq, Lk, pp.window_left, pp.causal)
                          : visible_pairs(Lq, Lk, pp.window_left, pp.causal);
      }
    }
  }
  if (pp.num_classes > 1) {
    // SMs for the prefill class when both classes run side by side.  Thread k
    // (1 <= k < SMs) estimates the time with k SMs for the prefill class; the
    // block takes the smallest estimate and, where a range of splits is within
    // 1 % of it (the decode class at its stream cap, the prefill class done
    // sooner), the middle of that range, away from both of its edges.
    __shared__ float tmin[32];
    __shared__ int klo, khi;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) work[k] += __shfl_xor_sync(0xFFFFFFFFu, work[k], off);
      if (lane == 0) wwork[k][wid] = work[k];
    }
    if (tid == 0) {
      klo = 1 << 30;
      khi = -1;
    }
    __syncthreads();
    long long w0 = 0, w1 = 0;
    for (int i = 0; i < 32; ++i) {
      w0 += wwork[0][i];
      w1 += wwork[1][i];
    }
    const float bytes0 = (float)w0 * pp.hkv * pp.head_dim * 2.0f;
    const float t1 = (float)w1 * pp.hq * pp.head_dim * 4.0f * pp.pf_ns_flop;  // ns x SMs
    const int k = tid;
    float est = __int_as_float(0x7F800000);
    if (k >= 1 && k < pp.sms)
      est = fmaxf(t1 / k, bytes0 / fminf((float)(pp.sms - k) * pp.dec_gbs_sm, pp.dec_gbs));
    float m = est;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fminf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if (lane == 0) tmin[wid] = m;
    __syncthreads();
    float best_t = tmin[0];
    for (int i = 1; i < 32; ++i) best_t = fminf(best_t, tmin[i]);
    if (k >= 1 && k < pp.sms && est <= best_t * 1.01f) {
      atomicMin(&klo, k);
      atomicMax(&khi, k);
    }
    __syncthreads();
    if (tid == 0) {
      const int best = (w1 > 0 && w0 > 0) ? (klo + khi) / 2 : (w1 > 0 ? pp.sms : 0);
      pp.counts[4] = pp.forced_split > 0 ? min(pp.forced_split, pp.sms) : best;
    }
  }
  // exclusive prefix sums of the per-thread counts: within each warp, then over the warp totals
  int inc[2] = {cnt[0], cnt[1]};
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, inc[k], off);
      if (lane >= off) inc[k] += v;
    }
  }
  if (lane == 31) {
    wsum[0][wid] = inc[0];
    wsum[1][wid] = inc[1];
  }
  __syncthreads();
  if (wid == 0) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      int v = wsum[k][lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (lane >= off) v += t;
      }
      wsum[k][lane] = v;
    }
  }
  __syncthreads();
  int excl[2], total[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    excl[k] = inc[k] - cnt[k] + (wid > 0 ? wsum[k][wid - 1] : 0);
    total[k] = wsum[k][31];
  }
  if (tid == 0)
    for (int k = 0; k < 2; ++k) {
      pp.counts[k] = k < pp.num_classes ? total[k] * pp.hkv : 0;
      pp.counts[2 + k] = 0;  // the attention kernel's dynamic item counter
    }
  // Items of a sequence: (KV head, row tile, split), split fastest.  A thread
  // writes its own sequences' short lists; long lists (prefill sequences, in
  // the order of write_long_item) are queued and written by the whole block
  // once every thread has seen its sequences.
  const bool beside = total[0] > 0 && total[1] > 0;  // both classes run, side by side
  constexpr int kLongList = 64;
  for (int j = 0; j < per; ++j) {
    const int b = b0 + j;
    int kc = -1, start = 0, rts = 0, ns = 1;
    if (b < b1) {
      const int Lq = seq_lq(pp, b);
      const int Lk = clamp_lk(pp.seqused_k[b], pp.max_pages);
      for (int k = 0; k < pp.num_classes; ++k) {
        const ClassInfo& c = pp.cls[k];
        if (!(Lq > 0 && in_class(Lq, c))) continue;
        kc = k;
        rts = seq_row_tiles(Lq, pp.group, c.rows);
        ns = unit_items(seq_splits(Lq, Lk, pp.group, pp.window_left, pp.causal, c), c);
        start = excl[k];
        excl[k] += rts * ns;
        break;
      }
    }
    const int nitems = kc >= 0 ? rts * ns * pp.hkv : 0;
    if (kc >= 0 && nitems <= kLongList) {
      int4* dst = pp.work[kc] + (size_t)start * pp.hkv;
      for (int hk = 0; hk < pp.hkv; ++hk)
        for (int rt = 0; rt < rts; ++rt)
          for (int s = 0; s < ns; ++s) *dst++ = make_int4(b, rt, hk | (s << 16), ns);
    }
    // long lists: queued for the whole block, or written by the warp when the queue is full
    const bool long_list = nitems > kLongList;
    int qslot = -1;
    if (long_list) {
      qslot = atomicAdd(&n_long, 1);
      if (qslot < kLongQueue) long_q[qslot] = LongList{b, kc, start, rts, ns};
    }
    for (unsigned lm = __ballot_sync(0xFFFFFFFFu, long_list && qslot >= kLongQueue); lm; lm &= lm - 1) {
      const int src = __ffs(lm) - 1;
      const LongList l{__shfl_sync(0xFFFFFFFFu, b, src), __shfl_sync(0xFFFFFFFFu, kc, src),
                       __shfl_sync(0xFFFFFFFFu, start, src), __shfl_sync(0xFFFFFFFFu, rts, src),
                       __shfl_sync(0xFFFFFFFFu, ns, src)};
      for (int i = lane; i < l.rts * l.ns * pp.hkv; i += 32) write_long_item(pp, l, i, beside);
    }
  }
  __syncthreads();
  const int nq = min(n_long, kLongQueue);
  for (int q = 0; q < nq; ++q) {
    const LongList l = long_q[q];
    for (int i = tid; i < l.rts * l.ns * pp.hkv; i += kPlanThreads) write_long_item(pp, l, i, beside);
  }
}

constexpr int kCombineWarps = 8;

// One warp per (token, head) row: lane s holds split s's log-sum-exp, the
// weights exp(lse_s - L) are formed once, then the warp sums the partial rows
// with 16-byte loads.
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(CombineParams cp) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  if (row >= (long long)cp.total_q * cp.hq) return;
  const int t = (int)(row / cp.hq), h = (int)(row % cp.hq);
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
  float lse_s[2], w_s[2];  // ns <= 64: lane holds splits lane and lane + 32
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int s = lane + 32 * k;
    lse_s[k] = s < ns ? cp.lse_part[(size_t)s * plane + (size_t)h * cp.total_q + t] : NEG_INF;
  }
  // a sink joins the denominator as one more term that carries no value
  const float sink = cp.sinks ? cp.sinks[h] : NEG_INF;
  float mx = fmaxf(fmaxf(lse_s[0], lse_s[1]), sink);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    w_s[k] = (mx == NEG_INF || lse_s[k] == NEG_INF) ? 0.f : expf(lse_s[k] - mx);
    sum += w_s[k];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  if (sink != NEG_INF) sum += expf(sink - mx);
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  const float L = (mx == NEG_INF) ? NEG_INF : mx + logf(sum);
  const size_t rbase = (size_t)t * cp.hq + h;
  for (int d0 = lane * 4; d0 < cp.head_dim; d0 += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < ns; ++s) {
      const float ws = __shfl_sync(0xFFFFFFFFu, w_s[s >> 5], s & 31) * inv;
      if (ws != 0.f) {
        const float4 v = *reinterpret_cast<const float4*>(cp.o_part + ((size_t)s * plane + rbase) * cp.head_dim + d0);
        acc.x += ws * v.x;
        acc.y += ws * v.y;
        acc.z += ws * v.z;
        acc.w += ws * v.w;
      }
    }
    __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(cp.out) + rbase * cp.head_dim + d0);
    o2[0] = __floats2bfloat162_rn(acc.x, acc.y);
    o2[1] = __floats2bfloat162_rn(acc.z, acc.w);
  }
  if (lane == 0 && cp.lse) cp.lse[(size_t)h * cp.total_q + t] = L;
}

}  // namespace

cudaError_t launch_plan(const PlanParams& pp, cudaStream_t stream) {
  return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, pp);
}

cudaError_t launch_combine(const CombineParams& cp, cudaStream_t stream) {
  if (cp.total_q <= 0) return cudaSuccess;
  const long long rows = (long long)cp.total_q * cp.hq;
  combine_kernel<<<(unsigned)((rows + kCombineWarps - 1) / kCombineWarps), kCombineWarps * 32, 0, stream>>>(cp);
  return cudaGetLastError();
}

}  // namespace fp8pa
