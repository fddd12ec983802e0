// Definitions shared by the plan, attention and combine kernels: launch
// parameters, the work-item format and the per-item key ranges.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace fp8pa {

constexpr int kPage = 64;          // tokens per KV-cache page
constexpr int kTileKeys = 128;     // keys per MMA tile: two pages, the MMA's M dimension
constexpr int kStageBytes = 16384; // one TMA stage: 128 keys x 128 bytes of head dim
constexpr uint32_t kDefaultWaitLimit = 1u << 22;
constexpr uint32_t kDrainWaitLimit = 1u << 22;

enum : unsigned { kDevBadPage = 1, kDevTimeout = 2, kDevBadLength = 4 };

// Attention kernel paths: E4M3 Q; BF16 Q with K dequantized to BF16 and V kept
// E4M3; BF16 Q with K and V dequantized to BF16.
enum : int { kPathE4M3 = 0, kPathBf16 = 1, kPathBf16DqV = 2 };

// One sequence class of a launch: sequences whose Lq lies in [lq_min, lq_max]
// are cut into row tiles of `rows` (query token, head-in-group) rows.
struct ClassInfo {
  int lq_min, lq_max;
  int rows;        // N: rows per tile (multiple of 16)
  int max_splits;  // split-KV count cap for single-row-tile sequences
  int dhalves;     // > 1: each row tile is dhalves work items, one per slice of the output dims
};

// Work items per (sequence, KV head, row tile): output-dim slices, else key splits.
__host__ __device__ __forceinline__ int unit_items(int split_count, const ClassInfo& c) {
  return c.dhalves > 1 ? c.dhalves : split_count;
}

struct AttnParams {
  // problem
  const int32_t* block_table;
  const int32_t* cu_seqlens_q;
  const int32_t* seqused_k;
  const float* q_descale;
  const float* k_descale;
  const float* v_descale;
  int descale_b, descale_h;
  int batch, total_q, hq, hkv, group, head_dim;
  int max_pages, num_pages;
  float softmax_scale_log2;  // softmax_scale * log2(e)
  int window_left, causal;
  // outputs
  void* out;        // bf16 [total_q][hq][D]
  float* lse;       // [hq][total_q] or null
  float* o_part;    // f32 [splits][total_q][hq][D]
  float* lse_part;  // f32 [splits][hq][total_q]
  const float* sinks;  // [hq] sink logits (natural log), or null; folded in where a row is finished
  // plan
  ClassInfo cls;
  const int4* work;        // items of this class
  const int* work_count;   // number of items
  int* work_next;          // dynamic item counter (zeroed by the plan kernel)
  unsigned* status;
  uint32_t wait_limit;
  int inject_stall;  // test hook: the MMA issuer first waits on a barrier that nothing arrives on
  // Two row classes run side by side on disjoint SMs: the prefill class is
  // launched first (conc_role 1) and keeps *sm_split SMs; the decode class is
  // launched second (conc_role 2), as soon as every CTA of the first is
  // resident, and keeps the other grid_sms - *sm_split.  conc_role 0: the
  // launch has every SM.
  int conc_role;
  const int* sm_split;
  int grid_sms;
};

// CTAs of this launch that take work; the others leave at once.
__device__ __forceinline__ int active_ctas(const AttnParams& p, int ctas_per_sm) {
  if (p.conc_role == 0) return (int)gridDim.x;
  const int split = *p.sm_split;
  return (p.conc_role == 1 ? split : p.grid_sms - split) * ctas_per_sm;
}

// A finished row's normalization with an attention sink: a per-head logit in
// the softmax denominator that attends to no value.  l = sum_j 2^(s2_j - m2)
// over the row's keys (log2 units, s2 = score * log2(e)), sink2 = sink * log2(e).
// inv = vd / (l + 2^(sink2 - m2)), lse2 = log2 of the whole denominator (log2
// units); a row with no key gets inv = 0 and lse2 = sink2.  No overflow for any
// m2 and sink2; a sink at -inf leaves inv = vd / l and lse2 = m2 + log2(l).
__device__ __forceinline__ void fold_sink(float l, float m2, float sink2, float vd, float& inv, float& lse2) {
  if (!(l > 0.f)) {
    inv = 0.f;
    lse2 = sink2;
    return;
  }
  const float a = sink2 - m2;
  if (a <= 64.f) {
    const float lt = l + exp2f(a);
    inv = vd / lt;
    lse2 = m2 + __log2f(lt);
  } else {
    const float r = exp2f(-a);
    const float lt = fmaf(l, r, 1.0f);
    inv = vd * r / lt;
    lse2 = sink2 + __log2f(lt);
  }
}

// Visible key range of query i of a sequence (Lq queries, Lk keys); hi < lo when empty.
__host__ __device__ __forceinline__ void visible_range(int Lq, int Lk, int i, int window_left, int causal, int& lo,
                                                       int& hi) {
  int p = Lk - Lq + i;
  lo = window_left >= 0 ? max(0, p - window_left) : 0;
  hi = causal ? min(p, Lk - 1) : Lk - 1;
}

// Number of key splits of a sequence in a class: only single-row-tile
// sequences split, and never into more splits than 128-key tiles.
__host__ __device__ __forceinline__ int seq_splits(int Lq, int Lk, int group, int window_left, int causal,
                                                   const ClassInfo& c) {
  if (Lq * group > c.rows || c.max_splits <= 1 || Lk <= 0) return 1;
  int lo0, hi0, lo1, hi1;
  visible_range(Lq, Lk, 0, window_left, causal, lo0, hi0);
  visible_range(Lq, Lk, Lq - 1, window_left, causal, lo1, hi1);
  if (hi1 < lo0) return 1;
  int pages = hi1 / kPage - lo0 / kPage + 1;
  int tiles = (pages + 1) / 2;
  return max(1, min(c.max_splits, tiles));
}

__host__ __device__ __forceinline__ int seq_row_tiles(int Lq, int group, int rows) {
  return (Lq * group + rows - 1) / rows;
}

// Everything a CTA needs to know about one work item.
struct Item {
  int b, rt, hk, split, nsplit;
  int q0, Lq, Lk;
  int row0, nrows;       // first packed row of the tile, valid rows (<= N)
  int lo_min;            // first key visible to any row
  int t0, t1;            // 128-key tiles [t0, t1) of this split; tile t starts at key (pg_lo() + 2t) * 64
  int lo_max, hi_min;    // keys in [lo_max, hi_min] are visible to every valid row
  int hi_max;            // last key visible to any row (for tail sanitation)
  int dhalf;             // slice of the output dims this item computes (classes with dhalves > 1)
  __device__ __forceinline__ int pg_lo() const { return lo_min / kPage; }  // first logical page of the key union
};

// Work item encoding: {b, row_tile, hk | split << 16, nsplit}.
__device__ __forceinline__ Item decode_item(const AttnParams& p, int4 w) {
  Item it;
  it.b = w.x;
  it.rt = w.y;
  it.hk = w.z & 0xFFFF;
  it.split = w.z >> 16;
  it.nsplit = w.w;
  it.dhalf = 0;
  if (p.cls.dhalves > 1) {  // the item index selects an output-dim slice; every key is visible to it
    it.dhalf = it.split;
    it.split = 0;
    it.nsplit = 1;
  }
  it.q0 = p.cu_seqlens_q[it.b];
  it.Lq = p.cu_seqlens_q[it.b + 1] - it.q0;
  int lk = p.seqused_k[it.b];
  int lk_cap = p.max_pages * kPage;
  if (lk < 0 || lk > lk_cap) {
    atomicOr(p.status, kDevBadLength);
    lk = lk < 0 ? 0 : lk_cap;
  }
  it.Lk = lk;
  const int N = p.cls.rows;
  it.row0 = it.rt * N;
  it.nrows = min(N, it.Lq * p.group - it.row0);
  int i_first = it.row0 / p.group;
  int i_last = (it.row0 + it.nrows - 1) / p.group;
  int lo_f, hi_f, lo_l, hi_l;
  visible_range(it.Lq, it.Lk, i_first, p.window_left, p.causal, lo_f, hi_f);
  visible_range(it.Lq, it.Lk, i_last, p.window_left, p.causal, lo_l, hi_l);
  it.lo_max = lo_l;
  it.hi_min = hi_f;
  it.hi_max = hi_l;
  if (it.Lk <= 0 || hi_l < lo_f || hi_l < 0) {
    it.lo_min = 0;
    it.t0 = it.t1 = 0;
    return it;
  }
  it.lo_min = lo_f;
  int pages = hi_l / kPage - it.pg_lo() + 1;
  int tiles = (pages + 1) / 2;
  it.t0 = (int)((long long)it.split * tiles / it.nsplit);
  it.t1 = (int)((long long)(it.split + 1) * tiles / it.nsplit);
  return it;
}

// First slot of the page box read for logical page pg of the item's key union
// (decode-shaped tiles with E4M3 V).  The union's first page starts at its first
// visible slot, and its last page ends at its last visible slot (a negative
// start: the box rows before slot 0 lie outside the page), so neither edge page
// reads slots that no row can see, nor slots past the sequence end; box rows
// outside the page arrive as zeros.  0 for the other pages, and for every page
// when the union lies within one page.  Box row r of page pg then holds key
// pg * 64 + r + page_slot0(it, pg).
__device__ __forceinline__ int page_slot0(const Item& it, int pg) {
  const int first = it.pg_lo(), last = it.hi_max / kPage;
  if (first == last) return 0;
  if (pg == first) return it.lo_min - first * kPage;
  if (pg == last) return it.hi_max - last * kPage + 1 - kPage;
  return 0;
}
// True when page_slot0 trims the item's edge pages: then no tile holds rows
// past the sequence end.
__device__ __forceinline__ bool edges_trimmed(const Item& it) { return it.pg_lo() != it.hi_max / kPage; }

}  // namespace fp8pa
