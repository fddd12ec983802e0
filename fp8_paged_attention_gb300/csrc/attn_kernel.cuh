// Paged FP8-KV attention forward, sm_103a.
//
// One persistent CTA per SM walks a device-built list of work items (sequence,
// KV head, tile of packed query rows, key split).  Per item the CTA streams the
// item's 64-token K/V pages through shared memory and keeps the running output
// in tensor memory:
//
//   S^T[key, row] = K[key, :] . Q[row, :]        tcgen05.mma, M = 128 keys, N = rows
//   P = exp2(S * scale * log2 e - m)              online softmax, one thread per key
//   O^T[d, row] += V[key, d]^T P^T[key, row]     tcgen05.mma, M = 128 dims, K = keys
//
// Rows pack (query token, query head of the KV group) pairs token-major, so GQA
// shares every K/V page among all heads of its group and all query tokens of
// the tile.  Keys sit on the 128 TMEM lanes; each softmax thread owns one key.
//
// Warp roles: warp 0 takes work items from a global counter, publishes each
// decoded item to the other roles through a small ring in shared memory, and
// issues the TMA loads (Q tile, then K/V page tiles in the order the MMAs
// consume them); warp 1 allocates tensor memory and issues the MMAs from one
// thread; the next one or two warpgroups run the softmax, the O rescale and the
// epilogue (with two, each owns half the rows of every tile).  On the BF16-Q
// paths the last four warps convert each item's BF16 Q tile in place; on the
// literal path they also dequantize each E4M3 K stage to F16 straight into
// tensor memory (the A operand of the QK^T MMA; exact, every E4M3 value is an
// F16 value) and V into BF16 shared-memory tiles.
//
// Softmax per tile: with the running offsets of the previous tiles, P' is
// computed directly; only when some P' exceeds the lazy bound (a row maximum
// grew by more than tau), and on the first tile of an item, are the exact
// per-row tile maxima formed (one warp reduction per row, then across the
// four warps) and P' recomputed.  Row sums accumulate P' in f32.
//
// Paths (template parameter kPath):
//  kPathE4M3    E4M3 Q: QK^T and PV are kind::f8f6f4 MMAs.
//  kPathBf16    BF16 Q as an exact pair of E4M3 terms: per item the Q tile is
//               scaled per row by a power of two 2^k_r (the row's largest
//               magnitude in [2^7, 2^8)) and split into hi = e4m3(x) and
//               lo = e4m3(x - hi).  BF16's 8 significant bits fit the two
//               terms' 4 + 4, so hi + lo = x for every value down to 2^-9 of
//               the row's largest (below it within 2^-10 absolute, scaled).
//               QK^T is two kind::f8f6f4 MMAs per K step on the E4M3 K stage,
//               both into the same S; V stays E4M3 (exact) in the PV MMA.
//  kPathBf16DqV BF16 Q, the literal form: Q converted in place to F16 scaled
//               by 2^k_r (largest magnitude in [2^14, 2^15): every BF16 value
//               down to 2^-28 of it exact), K dequantized to F16 (exact), QK^T a
//               kind::f16 MMA; V dequantized to BF16, PV a kind::f16 MMA with
//               BF16 P.
// On both BF16-Q paths the softmax multiplies row r's scores by 2^-k_r, folded
// into its per-row score scale.
// Where the PV MMA is E4M3, P is requantized to E4M3 after a 2^4 pre-scale
// (P' = 2^(x - m + 4), at most 256 under the lazy rescale below, keeping small
// weights out of E4M3's subnormal range) as a pair on one scale:
// hi = e4m3(P'), lo = e4m3(P' - hi); both PV MMAs accumulate into the same
// TMEM O, so P carries about 8 significant bits (BF16 carries 8) instead of
// E4M3's 4.  The row sum accumulates the f32 P', which the pair matches to
// within 2^-8 relative.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace fp8pa {

// kCtas: CTAs resident per SM.  Two co-resident CTAs run two independent
// item pipelines per SM, hiding each other's per-item bubbles (epilogue,
// first-tile latency); each then gets half the shared memory and TMEM.
template <int D, int kPath, int N, int kCtas = 1>
struct AttnCfg {
  static_assert(D == 256 || D == 512, "head dim");
  static_assert(N == 16 || N == 32 || N == 64, "rows per tile");
  static_assert(kCtas == 1 || kCtas == 2, "CTAs per SM");
  static_assert(kPath >= 0 && kPath <= 2, "path");
  static constexpr bool kQ8 = kPath == kPathE4M3;     // Q and K enter QK^T as E4M3
  static constexpr bool kQSplit = kPath == kPathBf16;  // BF16 Q enters QK^T as an exact E4M3 pair, K as E4M3
  static constexpr bool kP8 = kPath != kPathBf16DqV;  // P (hi/lo) and V enter PV as E4M3
  static constexpr bool kDq = kPath != kPathE4M3;     // dequant warps: the BF16 Q tile, per item
  static constexpr bool kKDq = kPath == kPathBf16DqV; // ... K -> F16 in TMEM, per tile
  static constexpr bool kDqV = kPath == kPathBf16DqV; // ... and V -> BF16 in shared memory
  static constexpr int kDC = D / 128;                    // 128-byte chunks of an E4M3 row
  static constexpr int kQChunkElems = kQ8 ? 128 : 64;    // Q elements per 128-byte chunk
  static constexpr int kQChunks = D / kQChunkElems;
  static constexpr int kQBytes = kQChunks * N * 128;
  // P^T for 128 keys: E4M3 hi term then E4M3 lo term (N x 128 bytes each), or BF16
  static constexpr int kPBytes = kP8 ? 2 * N * 128 : N * 256;
  static constexpr int kBfSlotBytes = 32768;             // BF16 tile of 128 keys x 128 dims
  // One CTA per SM: separate QK^T and PV issuing threads (warps 1 and 2).
  static constexpr bool kTwoIssuers = kCtas == 1;
  // softmax warpgroups: each owns N / kNW rows of every tile (two for 64-row tiles)
  static constexpr int kNW = N == 64 ? 2 : 1;
  static constexpr int kNR = N / kNW;
  static constexpr int kSmWarp0 = kTwoIssuers ? 3 : 2;  // first softmax warp
  static constexpr int kDqWarp0 = kSmWarp0 + 4 * kNW;    // first dequant warp (BF16-Q paths)
  static constexpr int kThreads = 32 * kDqWarp0 + (kDq ? 128 : 0);
  // opt-in maximum per block; two blocks share the SM's 228 KB minus 1 KB reserved each
  static constexpr int kSmemLimit = kCtas == 1 ? 232448 : 115712;
  // barriers and the item ring (< 1 KB), then per-row state: ooff[N] (8 bytes),
  // red[2][4][N], lred[4][N] and 4 x [N] floats
  // (+ on the BF16-Q paths: per-row score scales of the two Q buffers, 8 * N bytes)
  static constexpr int kCtrlBytes = 1536 + 72 * N + 80 + (kDq ? 8 * N : 0);
  // Two CTAs per SM: one Q buffer, and the room goes to the stage ring (the next
  // item's Q loads while this item's last tiles and epilogue run).
  static constexpr int kQBufs =
      kCtas == 2 ? 1 : kQ8 ? ((2 * kQBytes <= 65536) ? 2 : 1) : ((2 * kQBytes <= 32768) ? 2 : 1);
  static constexpr int kBfSlots = kDqV ? 2 : 0;
  static constexpr int kFixed = kQBufs * kQBytes + 2 * kPBytes + kBfSlots * kBfSlotBytes + kCtrlBytes + 1024;
  static constexpr int kStages = (kSmemLimit - kFixed) / kStageBytes > 16 ? 16 : (kSmemLimit - kFixed) / kStageBytes;
  static_assert(kStages >= 2, "smem");
  // Stage ring(s).  Every ring needs one in-order consumer that waits on all of
  // its fills: an mbarrier phase wait only tells parities apart, so a consumer
  // that skipped the slot's previous fill could take that pending fill's phase
  // for its own.  When K and V have different consumers (dequant warps and MMA
  // thread on the BF16-Q path with E4M3 V) they get a ring each: K stages in
  // slots [0, kKStages), V stages in [kKStages, kStages).
  static constexpr bool kSplitRing = kPath == kPathBf16 || (kPath == kPathE4M3 && kTwoIssuers);
  static constexpr int kVStages = kSplitRing ? ((kStages + 1) / 2 > kDC ? (kStages + 1) / 2 : kDC) : kStages;
  static constexpr int kKStages = kSplitRing ? kStages - kVStages : kStages;
  static_assert(kKStages >= 1, "no room for a K ring");
  // E4M3 V: the tail tile's V chunks must fit in the ring together (the softmax zeroes them in place)
  static_assert(!kP8 || kVStages >= kDC, "ring shorter than one tile's V");
  static constexpr int kSmemBytes = kFixed + kStages * kStageBytes;
  // TMEM columns: S (2 buffers of N), O (kDC chunks of N), BF16 K (2 slots of 64 columns = 128 dims)
  static constexpr int kKCol = 2 * N + kDC * N;
  // F16 K chunks in TMEM (64 columns each): as many slots as fit, up to four, so
  // that the dequant warps can run ahead of the QK^T MMAs
  static constexpr int kKSlotsFit = (512 / kCtas - kKCol) / 64;
  static constexpr int kKSlots = kKDq ? (kKSlotsFit > 4 ? 4 : kKSlotsFit) : 0;
  static_assert(!kKDq || kKSlots >= 2, "TMEM for the F16 K slots");
  static constexpr int kTmemUsed = kKCol + 64 * kKSlots;
  static constexpr uint32_t kTmemCols = kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128
                                        : kTmemUsed <= 256 ? 256 : 512;
  static_assert(kTmemUsed <= 512 && kCtas * kTmemCols <= 512, "TMEM");
  // Lazy rescaling: the running max used for the exponent only moves when a
  // row's max grows by more than kTau (log2 units), so most tiles need no O
  // rescale.  P' = 2^(x - m_used + kPShift) <= 2^(kTau + kPShift) stays within
  // E4M3's range (<= 256 < 448) and keeps small weights out of its subnormals.
  static constexpr float kTau = kP8 ? 4.0f : 8.0f;
  static constexpr float kPShift = kP8 ? 4.0f : 0.0f;
};

namespace detail {

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Max over the warp.
__device__ __forceinline__ float redux_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Per-row sums over the warp, transposed: given v[j] in every lane (R rows), lane l
// returns the sum over all 32 lanes of v[l mod R].  A butterfly that halves the
// rows at each step: the lane with the step's bit set keeps the upper half.
template <int R>
__device__ __forceinline__ float transpose_sum(const float (&v)[R], int lane) {
  static_assert(R == 16 || R == 32, "rows per warp");
  float a[R];
#pragma unroll
  for (int j = 0; j < R; ++j) a[j] = v[j];
  if (R == 16) {
#pragma unroll
    for (int j = 0; j < R; ++j) a[j] += __shfl_xor_sync(0xFFFFFFFFu, a[j], 16);
  }
#pragma unroll
  for (int off = R / 2; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int j = 0; j < off; ++j) {
      const float send = upper ? a[j] : a[j + off];
      const float keep = upper ? a[j + off] : a[j];
      a[j] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
    }
  }
  return a[0];
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// P' pair -> E4M3 pair hi = e4m3(P'), lo = e4m3(P' - hi), each as 16 bits with
// p0 in the low byte.  P' is rounded to f16 first (11 significant bits); the
// residual of an f16 and its 4-bit rounding is exact in f16.
__device__ __forceinline__ void e4m3_hilo(float p0, float p1, uint32_t& hi, uint32_t& lo) {
  uint32_t h, hh, l;
  uint16_t h8, l8;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(p1), "f"(p0));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(h8) : "r"(h));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hh) : "h"(h8));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(l) : "r"(h), "r"(hh));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(l8) : "r"(l));
  hi = h8;
  lo = l8;
}

__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t res;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(res)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return res != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: gives up after `lim` rounds, after about two seconds of wall
// clock, or once another role has flagged an abort.
__device__ __forceinline__ bool pwait(uint64_t* bar, uint32_t parity, uint32_t lim, volatile int* abort_flag) {
  uint64_t t0 = 0;
  for (uint32_t i = 0; i < lim; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 31u) {
      if (*abort_flag) return false;
      const uint64_t t = global_ns();
      if (t0 == 0) t0 = t;
      else if (t - t0 > 2000000000ull) return false;
    }
  }
  return false;
}

__device__ __forceinline__ void flag_timeout(const AttnParams& p, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(p.status, kDevTimeout);
}

// Physical page of logical page `pg`, or an out-of-range page id (the TMA then
// fills zeros) for pages past the item's last visible key or bad table entries.
__device__ __forceinline__ int page_id(const AttnParams& p, const Item& it, int pg) {
  if (pg > it.hi_max / kPage) return p.num_pages;
  int phys = p.block_table[(size_t)it.b * p.max_pages + pg];
  if ((unsigned)phys >= (unsigned)p.num_pages) {
    atomicOr(p.status, kDevBadPage);
    return p.num_pages;
  }
  return phys;
}

// A null descale pointer is the unit scale: nothing is read.
__device__ __forceinline__ float load_descale(const float* d, const AttnParams& p, const Item& it) {
  return d ? d[(size_t)it.b * p.descale_b + (size_t)it.hk * p.descale_h] : 1.0f;
}

// Stage position of V tile u (0-based within the item) in the item's stream
// K(0), [K(1), V(0)], [K(2), V(1)], ..., [K(n-1), V(n-2)], V(n-1), in stages.
__device__ __forceinline__ uint32_t v_stage_offset(int u, int n, int dc) {
  return (u < n - 1) ? (uint32_t)(2 * (u + 1) * dc) : (uint32_t)((2 * n - 1) * dc);
}

// Two E4M3 codes (low byte first) -> F16x2, exact.
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint16_t v) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(v));
  return h;
}

// BF16x2 (low half first) times f, rounded to F16x2.  f is a power of two, so
// the product is exact in f32; the rounding to F16 is exact for every value in
// F16's normal range.
__device__ __forceinline__ uint32_t bf16x2_scaled_to_f16x2(uint32_t w, float f) {
  const float lo = __uint_as_float(w << 16) * f, hi = __uint_as_float(w & 0xFFFF0000u) * f;
  uint32_t h;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi), "f"(lo));
  return h;
}

// Two f32 values -> two E4M3 codes (lo first, in the low byte), round to nearest
// even, saturating.
__device__ __forceinline__ uint16_t e4m3x2_of(float lo, float hi) {
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(hi), "f"(lo));
  return c;
}

__device__ __forceinline__ __half2 u32_as_half2(uint32_t h) { return *reinterpret_cast<__half2*>(&h); }

__device__ __forceinline__ uint32_t cvt_e4m3x2_bf16x2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
  float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<uint32_t*>(&b);
}

}  // namespace detail

// One published work item; valid = 0 marks the end of the CTA's work.
struct ItemSlot {
  Item it;
  int valid;
};
constexpr int kItemSlots = 4;

template <int D, int kPath, int N, int kCtas>
__global__ void __launch_bounds__(AttnCfg<D, kPath, N, kCtas>::kThreads, kCtas)
    attn_fwd_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using C = AttnCfg<D, kPath, N, kCtas>;
  constexpr bool kQ8 = C::kQ8, kP8 = C::kP8, kDq = C::kDq, kDqV = C::kDqV, kQS = C::kQSplit, kKDq = C::kKDq;
  // Decode-shaped tiles with E4M3 V: the key union's edge pages are read trimmed
  // to their visible slots (page_slot0).  The literal path's V conversion keeps
  // whole pages, and so do 64-row tiles, whose unions are long enough that the
  // edge pages weigh little against the per-tile work the trim adds.
  constexpr bool kTrim = kP8 && N <= 32;
  using namespace ptx;
  using namespace detail;
  constexpr int S = C::kStages;
  constexpr bool kSplit = C::kSplitRing;
  constexpr int SK = C::kKStages, SV = C::kVStages;
  constexpr int SB = C::kBfSlots;
  constexpr int SBm = SB > 0 ? SB : 1;  // modulus for the BF16 V ring (literal path only)
  constexpr int QB = C::kQBufs;
  constexpr int DC = C::kDC;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* ring = smem;
  uint8_t* bfbuf = ring + S * kStageBytes;
  uint8_t* qbuf = bfbuf + SB * C::kBfSlotBytes;
  uint8_t* pbuf = qbuf + QB * C::kQBytes;
  uint8_t* ctrl = pbuf + 2 * C::kPBytes;
  uint64_t* ring_full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* ring_empty = ring_full + S;
  uint64_t* bf_full = ring_empty + S;
  uint64_t* bf_empty = bf_full + (SB > 0 ? SB : 1);
  uint64_t* q_full = bf_empty + (SB > 0 ? SB : 1);
  uint64_t* q_empty = q_full + QB;
  uint64_t* s_full = q_empty + QB;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* o_empty = pv_done + 2;
  uint64_t* v_ready = o_empty + 1;  // tail tile: its V stages have landed (MMA thread -> softmax)
  uint64_t* drain = v_ready + 1;  // [2]: one per MMA-issuing thread
  uint64_t* never = drain + 2;    // nothing arrives on it: the stall-injection test hook waits here
  uint64_t* item_full = never + 1;
  uint64_t* item_empty = item_full + kItemSlots;
  uint64_t* kt_full = item_empty + kItemSlots;  // F16 K slot in TMEM written (dequant -> MMA)
  uint64_t* kt_empty = kt_full + 4;             // F16 K slot consumed (MMA commit -> dequant)
  uint64_t* q_conv = kt_empty + 4;              // [QB] Q tile converted to scaled F16 (dequant -> MMA, softmax)
  uint64_t* srow_empty = q_conv + 2;            // [2] an item's row scales read (softmax -> dequant)
  ItemSlot* islot = reinterpret_cast<ItemSlot*>(srow_empty + 2);
  // [N] element offset of each row's output (in out, or in o_part for a split)
  long long* ooff_s = reinterpret_cast<long long*>((reinterpret_cast<uintptr_t>(islot + kItemSlots) + 15) & ~(uintptr_t)15);
  float* red = reinterpret_cast<float*>(ooff_s + N);  // [2][4][N] per-warp tile maxima
  float* lred = red + 2 * 4 * N;                      // [4][N] per-warp row sums
  float* m_s = lred + 4 * N;                          // [N] running max (log2 units)
  float* a_s = m_s + N;                               // [N] rescale factor of this tile
  float* nmsub_s = a_s + N;                           // [N] exponent offset: P' = 2^(x + nmsub)
  float* inv_s = nmsub_s + N;                         // [N] output scale v_descale / l
  float* srow_s = inv_s + N;                          // BF16-Q paths: [2][N] score scale of each row
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(srow_s + (kDq ? 2 * N : 0));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (p.conc_role == 2 && (int)blockIdx.x >= active_ctas(p, kCtas)) {
    // second launch of a side-by-side pair, with no share of the SMs: nothing to
    // do, but the launch must not end before the first one (CTA 0 waits for it)
    if (blockIdx.x == 0) griddep_wait();
    return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&ring_full[i], 1);
      // one MMA commit, or one arrive of each of the four dequant warps for the stages they consume
      mbar_init(&ring_empty[i], (kKDq && (!kSplit || i < SK)) ? 4 : 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(&bf_full[i], 4);
      mbar_init(&bf_empty[i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&kt_full[i], 4);
      mbar_init(&kt_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_conv[i], 4);
      mbar_init(&srow_empty[i], 4 * C::kNW);
    }
    for (int i = 0; i < QB; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 4 * C::kNW);
      mbar_init(&p_full[i], 4 * C::kNW);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(o_empty, 4 * C::kNW);
    mbar_init(v_ready, 1);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    mbar_init(never, 1);
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], (C::kTwoIssuers ? 2 : 1) + 4 * C::kNW + (kDq ? 4 : 0));  // MMA, softmax, dequant
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The work list, Q and the K/V cache are written by earlier kernels.  The
  // second launch of a side-by-side pair starts only once the first launch has
  // seen them complete, and waits for that first launch before it exits.
  if (p.conc_role != 2) griddep_wait();
  bool idle = false;
  if (p.conc_role == 1) {
    idle = (int)blockIdx.x >= active_ctas(p, kCtas);
    griddep_launch_dependents();  // this CTA is resident: the second launch may take the free SMs
  }
  const uint32_t tmem = *tmem_slot;
  const int n_items = *p.work_count;
  const uint32_t lim = p.wait_limit;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    // The whole warp runs the loop; one elected lane takes work items, publishes
    // them and issues the copies, and every wait is a vote of the warp.
    {
      const bool leader = elect_one();
      const int leader_lane = __ffs(__ballot_sync(0xFFFFFFFFu, leader)) - 1;
      auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xFFFFFFFFu, pwait(bar, parity, lim, abort_flag));
      };
      // idx: stage stream position (one ring); kq / vq: K and V ring positions (split rings)
      uint32_t idx = 0, kq = 0, vq = 0, qit = 0;
      bool ok = true;
      for (uint32_t ik = 0; ok; ++ik) {
        int w = n_items;  // an idle CTA takes no item
        if (leader && !idle) w = atomicAdd(p.work_next, 1);
        w = __shfl_sync(0xFFFFFFFFu, w, leader_lane);
        const bool valid = w < n_items;
        const uint32_t is = ik % kItemSlots;
        if (!(ok = wait_all(&item_empty[is], ((ik / kItemSlots) & 1) ^ 1))) break;
        Item it{};
        if (valid) it = decode_item(p, p.work[w]);
        if (leader) {
          islot[is].it = it;
          islot[is].valid = valid;
          mbar_arrive(&item_full[is]);  // release: the slot's contents are visible to waiters
        }
        __syncwarp();
        if (!valid) break;
        if (it.t1 <= it.t0) continue;
        const int qb = qit % QB;
        if (!(ok = wait_all(&q_empty[qb], ((qit / QB) & 1) ^ 1))) break;
        if (leader) {
          mbar_arrive_expect_tx(&q_full[qb], C::kQBytes);
          for (int c = 0; c < C::kQChunks; ++c)
            tma_load_3d(qbuf + qb * C::kQBytes + c * N * 128, &tm_q, &q_full[qb], c * C::kQChunkElems,
                        it.hk * p.group, it.q0 + it.row0 / p.group);
        }
        ++qit;
        const int n = it.t1 - it.t0;
        auto load_tile = [&](int u, bool is_v) -> bool {
          const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
          const int pg = it.pg_lo() + 2 * (it.t0 + u);
          const int pa = page_id(p, it, pg), pb = page_id(p, it, pg + 1);
          const int sa = kTrim ? page_slot0(it, pg) : 0, sb = kTrim ? page_slot0(it, pg + 1) : 0;
          for (int c = 0; c < DC; ++c) {
            uint32_t& pos = !kSplit ? idx : is_v ? vq : kq;
            const uint32_t len = !kSplit ? S : is_v ? SV : SK;
            const uint32_t slot = (kSplit && is_v ? SK : 0) + pos % len;
            if (!wait_all(&ring_empty[slot], ((pos / len) & 1) ^ 1)) return false;
            if (leader) {
              mbar_arrive_expect_tx(&ring_full[slot], kStageBytes);
              uint8_t* dst = ring + slot * kStageBytes;
              tma_load_4d(dst, tm, &ring_full[slot], c * 128, it.hk, sa, pa);
              tma_load_4d(dst + kStageBytes / 2, tm, &ring_full[slot], c * 128, it.hk, sb, pb);
            }
            ++pos;
          }
          return true;
        };
        ok = load_tile(0, false);
        for (int u = 1; u <= n && ok; ++u) {
          if (u < n) ok = load_tile(u, false);
          if (ok) ok = load_tile(u - 1, true);
        }
      }
      if (!ok && leader) flag_timeout(p, abort_flag);
      // drain: every issued copy must land before the CTA may exit
      auto drain_ring = [&](uint32_t pos, uint32_t len, uint32_t first) {
        for (uint32_t j = pos > len ? pos - len : 0; j < pos; ++j)
          mbar_wait(&ring_full[first + j % len], (j / len) & 1, kDrainWaitLimit);
      };
      if (kSplit) {
        drain_ring(kq, SK, 0);
        drain_ring(vq, SV, SK);
      } else {
        drain_ring(idx, S, 0);
      }
      for (uint32_t j = qit > (uint32_t)QB ? qit - QB : 0; j < qit; ++j)
        mbar_wait(&q_full[j % QB], (j / QB) & 1, kDrainWaitLimit);
    }
  } else if (warp == 1 || (C::kTwoIssuers && warp == 2)) {
    // ------------------------------------------------------------------ MMA issuers
    // One CTA per SM: warp 1 issues the QK^T MMAs and warp 2 the PV MMAs, so that
    // neither waits behind the other's operands.  Two CTAs per SM: warp 1 issues
    // both, in stage-stream order.  The whole warp runs the loop (so descriptors
    // and counters stay warp-uniform); one elected lane issues the MMAs, commits
    // and arrivals, and every wait is a vote of the warp.
    {
      const bool leader = elect_one();
      auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xFFFFFFFFu, pwait(bar, parity, lim, abort_flag));
      };
      const bool do_qk = !C::kTwoIssuers || warp == 1;
      const bool do_pv = !C::kTwoIssuers || warp == 2;
      constexpr uint32_t idesc_qk = make_idesc(kKDq ? kFmtF16 : kFmtE4M3, kKMajor, kKMajor, 128, N);
      constexpr uint32_t idesc_pv = make_idesc(kP8 ? kFmtE4M3 : kFmtBF16, kMNMajor, kMNMajor, 128, N);
      // E4M3 stages: idx = stage-stream position (one ring), or kq / vq = K and V
      // ring positions (split rings); kidx: BF16 K chunks in TMEM; bidx: BF16 V
      // tiles in shared memory
      uint32_t idx = 0, kq = 0, vq = 0, kidx = 0, bidx = 0, g = 0, qit = 0;
      auto kslot = [&](uint32_t pos) { return kSplit ? pos % SK : pos % S; };
      auto kpar = [&](uint32_t pos) { return kSplit ? (pos / SK) & 1 : (pos / S) & 1; };
      auto vslot = [&](uint32_t pos) { return kSplit ? SK + pos % SV : pos % S; };
      auto vpar = [&](uint32_t pos) { return kSplit ? (pos / SV) & 1 : (pos / S) & 1; };
      uint32_t& kpos = kSplit ? kq : idx;
      uint32_t& vpos = kSplit ? vq : idx;
      bool ok = true;
      for (uint32_t ik = 0; ok; ++ik) {
        const uint32_t is = ik % kItemSlots;
        if (!(ok = wait_all(&item_full[is], (ik / kItemSlots) & 1))) break;
        const Item it = islot[is].it;
        const bool valid = islot[is].valid != 0;
        __syncwarp();
        if (leader) mbar_arrive(&item_empty[is]);
        if (!valid) break;
        if (p.inject_stall && !(ok = wait_all(never, 0))) break;
        if (it.t1 <= it.t0) continue;
        const int qb = qit % QB;
        // E4M3 Q straight from the TMA; BF16 Q once the dequant warps have converted it
        if (do_qk && !(ok = wait_all(kDq ? &q_conv[qb] : &q_full[qb], (qit / QB) & 1))) break;
        tc_fence_after();
        const uint32_t qaddr = smem_u32(qbuf + qb * C::kQBytes);
        // S^T(gg) = K . Q^T into S buffer gg & 1
        auto qk = [&](uint32_t gg) -> bool {
          const uint32_t sb = gg & 1;
          if (!wait_all(&s_empty[sb], ((gg >> 1) & 1) ^ 1)) return false;
          tc_fence_after();
          const uint32_t d_tmem = tmem + sb * N;
          for (int c = 0; c < DC; ++c) {
            if (kQ8 || kQS) {
              const uint32_t slot = kslot(kpos);
              if (!wait_all(&ring_full[slot], kpar(kpos))) return false;
              tc_fence_after();
              // E4M3 Q: chunk c of the tile; split BF16 Q: the hi term of dims 128c.. in
              // chunk 2c of the converted tile, its lo term in chunk 2c + 1
              const uint32_t a0 = smem_u32(ring + slot * kStageBytes), b0 = qaddr + (kQS ? 2 * c : c) * N * 128;
              if (leader) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  mma_f8f6f4(d_tmem, make_sdesc(a0 + kk * 32, 16, 1024, kLayoutSW128),
                             make_sdesc(b0 + kk * 32, 16, 1024, kLayoutSW128), idesc_qk, (c | kk) != 0);
                  if (kQS)
                    mma_f8f6f4(d_tmem, make_sdesc(a0 + kk * 32, 16, 1024, kLayoutSW128),
                               make_sdesc(b0 + N * 128 + kk * 32, 16, 1024, kLayoutSW128), idesc_qk, 1);
                }
                mma_commit(&ring_empty[slot]);
              }
              ++kpos;
            } else {
              // F16 K chunk (128 dims = 64 columns) in TMEM slot kidx % kKSlots, written by the dequant warps
              constexpr uint32_t KS = C::kKSlots > 0 ? C::kKSlots : 1;
              const uint32_t ks = kidx % KS;
              if (!wait_all(&kt_full[ks], (kidx / KS) & 1)) return false;
              tc_fence_after();
              const uint32_t a_t = tmem + C::kKCol + ks * 64;
              if (leader) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                  mma_f16_tmem_a(d_tmem, a_t + kk * 8,
                                 make_sdesc(qaddr + (2 * c + (kk >> 2)) * N * 128 + (kk & 3) * 32, 16, 1024,
                                            kLayoutSW128),
                                 idesc_qk, (c | kk) != 0);
                mma_commit(&kt_empty[ks]);
              }
              ++kidx;
            }
          }
          if (leader) mma_commit(&s_full[sb]);
          return true;
        };
        // O^T += V^T . P^T(gg).  On a tail tile (keys past Lk) with E4M3 V the
        // softmax zeroes the V rows past Lk first; the in-order wait here tells it
        // the stages landed.
        auto pv = [&](uint32_t gg, bool first, bool tail) -> bool {
          const uint32_t pb = gg & 1;
          if (kP8 && tail) {
            for (int c = 0; c < DC; ++c)
              if (!wait_all(&ring_full[vslot(vpos + c)], vpar(vpos + c))) return false;
            if (leader) mbar_arrive(v_ready);
          }
          if (!wait_all(&p_full[pb], (gg >> 1) & 1)) return false;
          if (first && !wait_all(o_empty, ((qit - 1) & 1) ^ 1)) return false;
          tc_fence_after();
          const uint32_t paddr = smem_u32(pbuf + pb * C::kPBytes);
          for (int c = 0; c < DC; ++c) {
            const uint32_t d_tmem = tmem + 2 * N + c * N;
            if (kP8) {
              const uint32_t slot = vslot(vpos);
              if (!wait_all(&ring_full[slot], vpar(vpos))) return false;
              tc_fence_after();
              const uint32_t a0 = smem_u32(ring + slot * kStageBytes);
              if (leader) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  const uint64_t va = make_sdesc(a0 + kk * 4096, 16384, 1024, kLayoutSW128);
                  mma_f8f6f4(d_tmem, va, make_sdesc(paddr + kk * 512, 128, 2048, kLayoutNone), idesc_pv,
                             !(first && kk == 0));
                  mma_f8f6f4(d_tmem, va, make_sdesc(paddr + N * 128 + kk * 512, 128, 2048, kLayoutNone), idesc_pv,
                             1);
                }
                mma_commit(&ring_empty[slot]);
              }
              ++vpos;
            } else {
              const uint32_t slot = bidx % SBm;
              if (!wait_all(&bf_full[slot], (bidx / SBm) & 1)) return false;
              tc_fence_after();
              const uint32_t a0 = smem_u32(bfbuf + slot * C::kBfSlotBytes);
              if (leader) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                  mma_f16(d_tmem, make_sdesc(a0 + kk * 2048, 16384, 1024, kLayoutSW128),
                          make_sdesc(paddr + kk * 256, 128, 2048, kLayoutNone), idesc_pv, !(first && kk == 0));
                mma_commit(&bf_empty[slot]);
              }
              ++bidx;
            }
          }
          if (leader) mma_commit(&pv_done[pb]);
          return true;
        };
        ++qit;  // pv() reads qit - 1 as this item's ordinal
        const int n = it.t1 - it.t0;
        auto is_tail = [&](int u) {
          return (it.pg_lo() + 2 * (it.t0 + u)) * kPage + kTileKeys > it.Lk && !(kTrim && edges_trimmed(it));
        };
        if (C::kTwoIssuers) {
          if (do_qk) {
            for (int u = 0; u < n && ok; ++u) ok = qk(g + u);
            if (ok && leader) mma_commit(&q_empty[qb]);
          } else {
            for (int u = 0; u < n && ok; ++u) ok = pv(g + u, u == 0, is_tail(u));
          }
        } else {
          ok = qk(g);
          for (int u = 0; u < n && ok; ++u) {
            if (u + 1 < n) ok = qk(g + u + 1);
            if (!ok) break;
            if (u + 1 == n && leader) mma_commit(&q_empty[qb]);
            ok = pv(g + u, u == 0, is_tail(u));
          }
        }
        g += n;
      }
      if (!ok && leader) flag_timeout(p, abort_flag);
      uint64_t* my_drain = do_qk ? drain : drain + 1;
      if (leader) mma_commit(my_drain);
      __syncwarp();
      mbar_wait(my_drain, 0, kDrainWaitLimit);
    }
  } else if (warp < C::kDqWarp0) {
    // ------------------------------------------------------------------ softmax / correction / epilogue
    // kNW warpgroups; warpgroup wg owns rows [r0, r0 + NR) of every tile and
    // synchronizes on its own two named barriers.
    constexpr int NR = C::kNR;
    const int wg = C::kNW == 1 ? 0 : (warp - C::kSmWarp0) >> 2;
    const int r0 = wg * NR;
    const uint32_t bar_a = 1 + 2 * wg, bar_b = 2 + 2 * wg;
    const int wt = threadIdx.x - 32 * C::kSmWarp0 - 128 * wg;  // 0..127 within the warpgroup
    const int quarter = warp & 3;                // TMEM lane quarter this warp may access
    const int kl = quarter * 32 + lane;          // key (S) or head-dim (O) lane within the tile
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float NEG_INF = __int_as_float(0xFF800000);
    // Largest P' the lazy offsets allow: 2^(kTau + kPShift).
    constexpr float kPMax = 256.0f;
    static_assert(C::kTau + C::kPShift == 8.0f, "kPMax");
    // Offset of a row that has seen no key yet: any unmasked key overflows P' and
    // sends the tile down the exact-maximum path.
    constexpr float kNoKeyOffset = 1e30f;
    uint32_t g = 0, sbase = 0, tails = 0;  // sbase: first stage of the item (stream, or V ring)
    uint32_t qi = 0;                        // non-empty items so far (Q buffer and row-scale ring position)
    bool aborted = false;
    for (uint32_t ik = 0; !aborted; ++ik) {
      const uint32_t is = ik % kItemSlots;
      bool iok = pwait(&item_full[is], (ik / kItemSlots) & 1, lim, abort_flag);
      iok = __all_sync(0xFFFFFFFFu, iok);
      Item it{};
      bool valid = false;
      if (iok) {
        it = islot[is].it;
        valid = islot[is].valid != 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_empty[is]);
      } else {
        flag_timeout(p, abort_flag);
      }
      if (bar_red_or(bar_a, 128, !iok)) {  // the warpgroup leaves together
        aborted = true;
        break;
      }
      if (!valid) break;
      const int G = p.group;
      const bool split_out = it.nsplit > 1;
      const int nr = min(NR, it.nrows - r0);  // live rows of this warpgroup (may be <= 0)
      auto row_tok = [&](int n) { return it.q0 + (it.row0 + n) / G; };
      auto row_head = [&](int n) { return it.hk * G + (it.row0 + n) % G; };
      if (it.t1 <= it.t0) {
        // nothing visible: out = 0, lse = -inf
#pragma unroll 1
        for (int n = r0; n < r0 + nr; ++n) {
          const size_t r = (size_t)row_tok(n) * p.hq + row_head(n);
          for (int d = wt; d < D; d += 128) {
            if (split_out)
              p.o_part[((size_t)it.split * p.total_q * p.hq + r) * D + d] = 0.f;
            else
              reinterpret_cast<__nv_bfloat16*>(p.out)[r * D + d] = __float2bfloat16_rn(0.f);
          }
        }
        if (wt < nr) {
          const int n = r0 + wt;
          const size_t li = (size_t)row_head(n) * p.total_q + row_tok(n);
          if (split_out)
            p.lse_part[(size_t)it.split * p.hq * p.total_q + li] = NEG_INF;
          else if (p.lse)
            p.lse[li] = p.sinks ? p.sinks[row_head(n)] : NEG_INF;  // only the sink is left
        }
        continue;
      }
      const int n_t = it.t1 - it.t0;
      const float kd = load_descale(p.k_descale, p, it);
      const float vd = load_descale(p.v_descale, p, it);
      const float scale = p.softmax_scale_log2 * kd * (kQ8 && p.q_descale ? *p.q_descale : 1.0f);
      // BF16-Q paths: row r's scores carry the Q tile's 2^k_r; its score scale
      // srow[r] = scale * 2^-k_r comes from the dequant warps with the converted Q
      const uint32_t qb = qi % QB, sr = qi & 1;  // Q buffer, row-scale ring slot
      const float* srow = srow_s + sr * N;
      if (kDq) {
        bool qok = pwait(&q_conv[qb], (qi / QB) & 1, lim, abort_flag);
        qok = __all_sync(0xFFFFFFFFu, qok);
        if (!qok) flag_timeout(p, abort_flag);
        if (bar_red_or(bar_a, 128, !qok)) {
          aborted = true;
          break;
        }
      }
      ++qi;
      auto rscale = [&](int n) { return kDq ? srow[r0 + n] : scale; };
      if (wt < NR) {
        m_s[r0 + wt] = NEG_INF;
        a_s[r0 + wt] = 1.0f;
        nmsub_s[r0 + wt] = kNoKeyOffset;
      }
      float lt[NR];  // this thread's partial row sums (its keys only)
#pragma unroll
      for (int n = 0; n < NR; ++n) lt[n] = 0.f;

      for (int u = 0; u < n_t; ++u, ++g) {
        const int kb = (it.pg_lo() + 2 * (it.t0 + u)) * kPage;
        const bool trimmed = kTrim && edges_trimmed(it);
        int j = kb + kl;  // this lane's key; -1 for a box row outside its page (zero fill)
        if (trimmed) {
          const int r = (kl & (kPage - 1)) + page_slot0(it, kb / kPage + kl / kPage);
          j = (r >= 0 && r < kPage) ? kb + (kl & kPage) + r : -1;
        }
        const uint32_t sb = g & 1, pb = g & 1;
        const bool interior = kb >= it.lo_max && kb + kTileKeys - 1 <= it.hi_min;
        const bool tail = kP8 && kb + kTileKeys > it.Lk && !trimmed;
        bool ok = pwait(&s_full[sb], (g >> 1) & 1, lim, abort_flag);
        if (ok && g >= 2) ok = pwait(&pv_done[pb], ((g >> 1) - 1) & 1, lim, abort_flag);  // P buffer free
        ok = __all_sync(0xFFFFFFFFu, ok);
        float x[NR];
        // raw scores of this warpgroup's rows for this thread's key; masked keys at -inf
        auto load_scores = [&]() {
          tc_fence_after();
          if (NR == 32 && nr > 16) {
            tmem_load32f(tmem + lane_base + sb * N + r0, x);  // one 32-column load, one wait
          } else {
#pragma unroll
            for (int c = 0; c < NR; c += 16) {
              if (c < nr) {
                tmem_load16f(tmem + lane_base + sb * N + r0 + c, x + c);
              } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) x[c + i] = NEG_INF;
              }
            }
          }
          if (!interior) {
            // query i sits at p = Lk - Lq + i; rows n and n' share a token when n / G == n' / G
            const int lg = __ffs(G) - 1;
            const int p0 = it.Lk - it.Lq + ((it.row0 + r0) >> lg);
#pragma unroll
            for (int n = 0; n < NR; ++n) {
              const int pn = p0 + (n >> lg);
              const int lo = p.window_left >= 0 ? max(0, pn - p.window_left) : 0;
              const int hi = p.causal ? min(pn, it.Lk - 1) : it.Lk - 1;
              if (j < lo || j > hi) x[n] = NEG_INF;
            }
          }
#pragma unroll
          for (int n = 0; n < NR; ++n)
            if (n >= nr) x[n] = NEG_INF;
        };
        // Fast path: P' = 2^(S * scale - m_used + shift) with the running offsets,
        // valid unless some P' exceeds 2^(tau + shift), i.e. a row maximum grew by
        // more than tau; the first tile of an item always needs the exact maxima.
        bool slow = u == 0;
        if (ok) {
          load_scores();
          if (!slow) {
            float pm = 0.f;
#pragma unroll
            for (int n = 0; n < NR; n += 2) {
              const float2 t = __ffma2_rn(make_float2(x[n], x[n + 1]), make_float2(rscale(n), rscale(n + 1)),
                                          make_float2(nmsub_s[r0 + n], nmsub_s[r0 + n + 1]));
              x[n] = ex2(t.x);
              x[n + 1] = ex2(t.y);
              pm = fmax3(pm, x[n], x[n + 1]);
            }
            slow = pm > kPMax;
          }
        } else {
          flag_timeout(p, abort_flag);
        }
        bool rescale = false;
        if (bar_red_or(bar_a, 128, slow || !ok)) {
          if (bar_red_or(bar_a, 128, !ok)) {
            aborted = true;
            break;
          }
          // exact tile maxima: the fast-path attempt (if any) overwrote x
          if (u > 0) load_scores();
#pragma unroll
          for (int n = 0; n < NR; n += 2) {
            const float2 t = __fmul2_rn(make_float2(x[n], x[n + 1]), make_float2(rscale(n), rscale(n + 1)));
            x[n] = t.x;
            x[n + 1] = t.y;
          }
          float* rb = red + (g & 1) * 4 * N + quarter * N + r0;
          float mine0 = NEG_INF, mine1 = NEG_INF;
#pragma unroll
          for (int n = 0; n < NR; ++n) {
            if (n < nr) {
              const float mx = redux_max(x[n]);
              if (n < 32) mine0 = lane == n ? mx : mine0;
              else mine1 = lane == n - 32 ? mx : mine1;
            }
          }
          if (lane < nr) rb[lane] = mine0;
          if (NR > 32 && lane + 32 < nr) rb[lane + 32] = mine1;
          named_bar_sync(bar_a, 128);
          // row owners fold the four warp maxima into the running max
          bool resc = false;
          if (wt < nr) {
            const int n = r0 + wt;
            const float* rr = red + (g & 1) * 4 * N + n;
            const float tmax = fmaxf(fmaxf(rr[0], rr[N]), fmaxf(rr[2 * N], rr[3 * N]));
            const float mo = m_s[n];
            float mn = mo, alpha = 1.0f;
            if (tmax > mo + C::kTau) {
              mn = tmax;
              // a row that has seen no key yet has O = 0 and l = 0: nothing to rescale
              if (mo != NEG_INF) alpha = ex2(mo - mn);
            }
            m_s[n] = mn;
            a_s[n] = alpha;
            nmsub_s[n] = mn == NEG_INF ? kNoKeyOffset : C::kPShift - mn;
            resc = alpha != 1.0f;
          }
          rescale = bar_red_or(bar_b, 128, resc);
#pragma unroll
          for (int n = 0; n < NR; n += 2) {
            const float2 t = __fadd2_rn(make_float2(x[n], x[n + 1]), make_float2(nmsub_s[r0 + n], nmsub_s[r0 + n + 1]));
            x[n] = ex2(t.x);
            x[n + 1] = ex2(t.y);
          }
          if (rescale) {
#pragma unroll
            for (int n = 0; n < NR; ++n) lt[n] *= a_s[r0 + n];
          }
        }
        // P^T of this warpgroup's rows, and the row sums of P'
        uint8_t* pdst = pbuf + pb * C::kPBytes;
        if (kP8) {
#pragma unroll
          for (int blk = 0; blk < NR / 16; ++blk) {
            if (blk * 16 >= nr) break;
            uint32_t hi_w[4], lo_w[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int n0 = blk * 16 + q4 * 4;
              uint32_t h01, l01, h23, l23;
              e4m3_hilo(x[n0], x[n0 + 1], h01, l01);
              e4m3_hilo(x[n0 + 2], x[n0 + 3], h23, l23);
              hi_w[q4] = h01 | (h23 << 16);
              lo_w[q4] = l01 | (l23 << 16);
            }
            const int o = (r0 / 16 + blk) * 2048 + kl * 16;
            *reinterpret_cast<uint4*>(pdst + o) = make_uint4(hi_w[0], hi_w[1], hi_w[2], hi_w[3]);
            *reinterpret_cast<uint4*>(pdst + N * 128 + o) = make_uint4(lo_w[0], lo_w[1], lo_w[2], lo_w[3]);
          }
        } else {
#pragma unroll
          for (int blk = 0; blk < NR / 8; ++blk) {
            if (blk * 8 >= nr) break;
            uint32_t packed[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int n0 = blk * 8 + q4 * 2;
              __nv_bfloat162 b2 = __floats2bfloat162_rn(x[n0], x[n0 + 1]);
              packed[q4] = *reinterpret_cast<uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(pdst + (r0 / 8 + blk) * 2048 + kl * 16) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
          }
        }
#pragma unroll
        for (int n = 0; n < NR; n += 2) {
          const float2 s = __fadd2_rn(make_float2(lt[n], lt[n + 1]), make_float2(x[n], x[n + 1]));
          lt[n] = s.x;
          lt[n + 1] = s.y;
        }
        // rows of the last page past the sequence end may hold anything (even NaN):
        // zero those V rows so that 0 * V stays 0 in the PV MMA
        if (tail) {
          const int zr = max(0, it.Lk - kb);
          ok = pwait(v_ready, tails & 1, lim, abort_flag);
          ok = __all_sync(0xFFFFFFFFu, ok);
          ++tails;
#pragma unroll 1
          for (int c = 0; c < DC && ok; ++c) {
            const uint32_t vi = kSplit ? sbase + u * DC + c : sbase + v_stage_offset(u, n_t, DC) + c;
            uint8_t* st = ring + (kSplit ? SK + vi % SV : vi % S) * kStageBytes;
            for (int x16 = zr * 8 + wt + 128 * wg; x16 < kTileKeys * 8; x16 += 128 * C::kNW)
              *reinterpret_cast<uint4*>(st + x16 * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        // rescale the running O when a row max grew (not needed on an item's first tile)
        if (ok && rescale && u > 0) {
          ok = pwait(&pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, lim, abort_flag);
          ok = __all_sync(0xFFFFFFFFu, ok);
          if (ok) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < DC; ++c) {
#pragma unroll
              for (int cc = 0; cc < NR; cc += 16) {
                if (cc >= nr) break;
                uint32_t r[16];
                const uint32_t ta = tmem + lane_base + 2 * N + c * N + r0 + cc;
                tmem_load16(ta, r);
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * a_s[r0 + cc + i]);
                tmem_store16(ta, r);
              }
            }
          }
        }
        if (tail || rescale) {
          if (!ok) flag_timeout(p, abort_flag);
          if (bar_red_or(bar_a, 128, !ok)) {
            aborted = true;
            break;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&s_empty[sb]);
          mbar_arrive(&p_full[pb]);
        }
      }
      if (aborted) break;
      if (kDq) {  // this item's row scales are no longer read
        __syncwarp();
        if (lane == 0) mbar_arrive(&srow_empty[sr]);
      }
      sbase += (kSplit ? 1 : 2) * n_t * DC;
      // ---------------- epilogue: O / l, lse
      // The row sums, scales and lse do not depend on O: they are formed while
      // the item's last PV completes, and only the O read waits for it.
      {
        const float rs = transpose_sum(lt, lane);  // this warp's sum for row (lane mod NR)
        if (lane < NR) lred[quarter * N + r0 + lane] = rs;
      }
      named_bar_sync(bar_a, 128);
      // row owners: output scale vd / l, output offset and lse, once per row
      if (wt < nr) {
        const int n = r0 + wt;
        const float l = (lred[n] + lred[N + n]) + (lred[2 * N + n] + lred[3 * N + n]);
        const int tok = row_tok(n), head = row_head(n);
        const long long row = (long long)tok * p.hq + head;
        inv_s[n] = l > 0.f ? vd / l : 0.f;
        ooff_s[n] = (split_out ? (long long)it.split * p.total_q * p.hq + row : row) * D;
        float lse = l > 0.f ? (m_s[n] - C::kPShift + __log2f(l)) * 0.69314718055994531f : NEG_INF;
        if (p.sinks && !split_out) {
          // the sink joins the denominator here; split partials get it in the combine
          float inv, lse2;
          fold_sink(l, m_s[n] - C::kPShift, p.sinks[head] * 1.4426950408889634f, vd, inv, lse2);
          inv_s[n] = inv;
          lse = lse2 * 0.69314718055994531f;
        }
        const size_t li = (size_t)head * p.total_q + tok;
        if (split_out)
          p.lse_part[(size_t)it.split * p.hq * p.total_q + li] = lse;
        else if (p.lse)
          p.lse[li] = lse;
      }
      bool ok = pwait(&pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, lim, abort_flag);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) flag_timeout(p, abort_flag);
      if (bar_red_or(bar_b, 128, !ok)) {  // also publishes the row owners' scales and offsets
        aborted = true;
        break;
      }
      tc_fence_after();
      // O^T columns of this warpgroup's rows, 16 at a time, scaled and stored
      auto store_rows = [&](const uint32_t* r, int cc, int cnt, int d) {
        if (split_out) {
#pragma unroll
          for (int i = 0; i < cnt; ++i)
            if (cc + i < nr) p.o_part[ooff_s[r0 + cc + i] + d] = __uint_as_float(r[i]) * inv_s[r0 + cc + i];
        } else {
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll
          for (int i = 0; i < cnt; ++i)
            if (cc + i < nr)
              out[ooff_s[r0 + cc + i] + d] = __float2bfloat16_rn(__uint_as_float(r[i]) * inv_s[r0 + cc + i]);
        }
      };
      if (N != 32 && !split_out) {
        // 16- and 64-row tiles, bf16 out: each 128-dim chunk of this
        // warpgroup's rows is staged in its own rows of the P buffers (free: every
        // PV of the item has completed, and only this warpgroup writes them), then
        // leaves as 16-byte pieces of whole rows.  Staged row j: the first half of
        // the rows in the P hi term's region, the second half in the lo term's
        // (E4M3 P), or one region (BF16 P).  Measured on the 4096-token chunk at
        // head dim 512: the item epilogue ~29k -> ~14k cycles; the mixed hd512
        // batch 11.95 -> 11.75 ms.  32-row tiles (verify, mostly split) keep the
        // direct stores: with this path compiled in they measured 5 % slower.
        auto stg_row = [&](int j) -> uint8_t* {
          if (kP8) return pbuf + (j < NR / 2 ? 0 : N * 128) + r0 * 128 + (j % (NR / 2)) * 256;
          return pbuf + r0 * 256 + j * 256;
        };
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll 1
        for (int c = 0; c < DC; ++c) {
#pragma unroll
          for (int cc = 0; cc < NR; cc += 16) {
            if (cc >= nr) break;
            uint32_t r[16];
            tmem_load16(tmem + lane_base + 2 * N + c * N + r0 + cc, r);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              *reinterpret_cast<__nv_bfloat16*>(stg_row(cc + i) + kl * 2) =
                  __float2bfloat16_rn(__uint_as_float(r[i]) * inv_s[r0 + cc + i]);
          }
          named_bar_sync(bar_a, 128);
          // 16 pieces of 16 bytes per staged row; consecutive threads take consecutive pieces
#pragma unroll
          for (int k = 0; k < NR / 8; ++k) {
            const int idx = wt + 128 * k, j = idx >> 4, pc = idx & 15;
            if (j < nr)
              *reinterpret_cast<uint4*>(out + ooff_s[r0 + j] + c * 128 + pc * 8) =
                  *reinterpret_cast<const uint4*>(stg_row(j) + pc * 16);
          }
          named_bar_sync(bar_a, 128);  // the staged rows are free for the next chunk
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < DC; ++c) {
          const int d = c * 128 + kl;
#pragma unroll
          for (int cc = 0; cc < NR; cc += 16) {
            if (cc >= nr) break;
            uint32_t r[16];
            tmem_load16(tmem + lane_base + 2 * N + c * N + r0 + cc, r);
            store_rows(r, cc, 16, d);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);
    }
  } else {
    // ------------------------------------------------------------------ dequant warps (BF16-Q paths)
    // Each of the four warps works on its own quarter of the rows and keys (its
    // TMEM lane quarter) and meets the other roles only through mbarriers: per
    // item it converts its rows of the BF16 Q tile in place to F16 scaled by
    // 2^k_r and publishes their score scales; per K chunk it writes its 32 key
    // rows as F16 into a TMEM slot (the A operand of QK^T); on the literal path
    // it also writes its part of each V tile as BF16 into shared memory.
    if (kDq) {
      const int quarter = warp & 3;
      const int wq = warp - C::kDqWarp0;  // 0..3
      const int row = quarter * 32 + lane;  // this thread's key row = its TMEM lane
      const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
      constexpr uint32_t KS = C::kKSlots > 0 ? C::kKSlots : 1;
      constexpr uint32_t KR = kSplit ? SK : S;
      // Q conversion: warp wq owns rows [wq * N / 4, (wq + 1) * N / 4); QP lanes per row,
      // each taking every QP-th 128-byte chunk of its row
      constexpr int QP = 128 / N;
      constexpr int kQCh = C::kQChunks;
      static_assert(!kDq || kQCh % QP == 0, "Q chunks per lane");
      const int qrow = wq * (N / 4) + lane / QP, qpart = lane % QP;
      // idx: stage stream position (literal path, one ring) or K ring position (split rings)
      uint32_t idx = 0, kidx = 0, bidx = 0, qi = 0;
      bool ok = true;
      auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xFFFFFFFFu, pwait(bar, parity, lim, abort_flag));
      };
      for (uint32_t ik = 0; ok; ++ik) {
        const uint32_t is = ik % kItemSlots;
        if (!(ok = wait_all(&item_full[is], (ik / kItemSlots) & 1))) break;
        const Item it = islot[is].it;
        const bool valid = islot[is].valid != 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_empty[is]);
        if (!valid) break;
        if (it.t1 <= it.t0) continue;
        const int n = it.t1 - it.t0;
        // ---- this warp's rows of the Q tile: BF16 -> F16 x 2^k_r in place, score scales out
        {
          const uint32_t qb = qi % QB, sr = qi & 1;  // Q buffer, row-scale ring slot (two slots)
          ok = wait_all(&q_full[qb], (qi / QB) & 1) && wait_all(&srow_empty[sr], ((qi >> 1) & 1) ^ 1);
          if (!ok) break;
          uint8_t* qrow_base = qbuf + qb * C::kQBytes + qrow * 128;
          uint32_t mx = 0;  // largest |q| of the row's bits (positive BF16 bit patterns order like their values)
#pragma unroll 1
          for (int c = qpart; c < kQCh; c += QP) {
            const uint4* src = reinterpret_cast<const uint4*>(qrow_base + c * N * 128);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint4 v = src[j];
              mx = __vmaxu2(mx, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                         __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
            }
          }
          mx = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
          for (int o = 1; o < QP; o <<= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
          int k;
          if constexpr (kQS) {
            // 2^k_r puts the row's largest magnitude in [2^7, 2^8) (an all-zero row keeps
            // k = 0).  Dims 128j .. 128j + 127 of the row (BF16 chunks 2j and 2j + 1) become
            // hi = e4m3(x), lo = e4m3(x - hi) with x = q 2^k_r, hi in chunk 2j and lo in
            // chunk 2j + 1 as E4M3 rows (128 bytes, 16-byte pieces swizzled by row).  x has
            // BF16's 8 significant bits and hi keeps the top 4 (rounded), so x - hi is exact
            // and has at most 4 more; lo holds it exactly whenever |x| >= 2^-2, i.e. for every
            // value down to 2^-9 of the row's largest, and within 2^-10 below that.
            const int e = (int)(mx >> 7);
            k = mx == 0 ? 0 : min(120, 134 - e);
            const float f = __int_as_float((k + 127) << 23);
            const int sw = qrow & 7;
#pragma unroll 1
            for (int j = qpart; j < kQCh / 2; j += QP) {
              uint8_t* c0 = qrow_base + 2 * j * N * 128;  // the row in chunk 2j
              uint8_t* c1 = c0 + N * 128;                 // and in chunk 2j + 1
              uint4 v[16];                                // BF16 pieces in dim order (8 dims each)
#pragma unroll
              for (int t = 0; t < 8; ++t) {
                v[t] = *reinterpret_cast<const uint4*>(c0 + ((t ^ sw) << 4));
                v[8 + t] = *reinterpret_cast<const uint4*>(c1 + ((t ^ sw) << 4));
              }
#pragma unroll
              for (int t = 0; t < 8; ++t) {  // E4M3 piece t: dims 16t .. 16t + 15 of the 128
                const uint32_t w[8] = {v[2 * t].x,     v[2 * t].y,     v[2 * t].z,     v[2 * t].w,
                                       v[2 * t + 1].x, v[2 * t + 1].y, v[2 * t + 1].z, v[2 * t + 1].w};
                uint32_t h[4], l[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  uint32_t hq[2], lq[2];
#pragma unroll
                  for (int b = 0; b < 2; ++b) {
                    const uint32_t x2 = w[2 * q + b];
                    const float2 x = __fmul2_rn(make_float2(__uint_as_float(x2 << 16), __uint_as_float(x2 & 0xFFFF0000u)),
                                                make_float2(f, f));
                    const uint16_t hc = e4m3x2_of(x.x, x.y);
                    const float2 hv = __half22float2(u32_as_half2(cvt_e4m3x2_f16x2(hc)));
                    hq[b] = hc;
                    lq[b] = e4m3x2_of(x.x - hv.x, x.y - hv.y);
                  }
                  h[q] = hq[0] | (hq[1] << 16);
                  l[q] = lq[0] | (lq[1] << 16);
                }
                *reinterpret_cast<uint4*>(c0 + ((t ^ sw) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4*>(c1 + ((t ^ sw) << 4)) = make_uint4(l[0], l[1], l[2], l[3]);
              }
            }
          } else {
            // 2^k_r puts the row's largest magnitude in [2^14, 2^15); an all-zero row keeps k = 0
            const int e = (int)(mx >> 7);
            k = mx == 0 ? 0 : min(120, 141 - e);
            const float f = __int_as_float((k + 127) << 23);
#pragma unroll 1
            for (int c = qpart; c < kQCh; c += QP) {
              uint4* src = reinterpret_cast<uint4*>(qrow_base + c * N * 128);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                uint4 v = src[j];
                uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
                for (int i = 0; i < 4; ++i) w[i] = bf16x2_scaled_to_f16x2(w[i], f);
                src[j] = v;
              }
            }
          }
          if (qpart == 0) {
            const float scale = p.softmax_scale_log2 * load_descale(p.k_descale, p, it) * 1.0f;
            srow_s[sr * N + qrow] = scale * __int_as_float((127 - k) << 23);
          }
          fence_proxy_async_smem();  // the MMA reads the converted tile through the async proxy
          __syncwarp();
          if (lane == 0) mbar_arrive(&q_conv[qb]);
          ++qi;
        }
        if constexpr (kQS) continue;  // K and V reach the MMAs as E4M3: nothing to convert per tile
        // K tile u: each chunk (128 dims) -> F16 in TMEM slot kidx % KS, one key row per thread
        auto convert_k = [&](int u) -> bool {
          if (!kKDq) return true;
          for (int c = 0; c < DC; ++c) {
            const uint32_t slot = idx % KR, ks = kidx % KS;
            if (!wait_all(&ring_full[slot], (idx / KR) & 1) || !wait_all(&kt_empty[ks], ((kidx / KS) & 1) ^ 1))
              return false;
            tc_fence_after();
            const uint8_t* src = ring + slot * kStageBytes + row * 128;
            uint4 vin[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) vin[j] = *reinterpret_cast<const uint4*>(src + ((j ^ (row & 7)) << 4));
            const uint32_t ta = tmem + lane_base + C::kKCol + ks * 64;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              uint32_t o[16];
#pragma unroll
              for (int jj = 0; jj < 2; ++jj) {
                const uint4 v = vin[2 * h + jj];
                const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  o[jj * 8 + 2 * i] = cvt_e4m3x2_f16x2((uint16_t)(in[i] & 0xFFFF));
                  o[jj * 8 + 2 * i + 1] = cvt_e4m3x2_f16x2((uint16_t)(in[i] >> 16));
                }
              }
              tmem_store16_nowait(ta + h * 16, o);  // dims 32h .. 32h+31 -> columns 16h .. 16h+15
            }
            __syncwarp();  // every lane's stage bytes have been read and converted
            if (lane == 0) mbar_arrive(&ring_empty[slot]);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&kt_full[ks]);
            ++idx;
            ++kidx;
          }
          return true;
        };
        // V tile u, literal path: -> BF16 in shared memory; rows past Lk become zeros.
        // Warp wq converts the 16-byte pieces wq * 32 + lane + 128 j of each stage.
        auto convert_v = [&](int u) -> bool {
          if (!kDqV) return true;  // the PV MMA reads these stages as E4M3, from the V ring
          const int kb = (it.pg_lo() + 2 * (it.t0 + u)) * kPage;
          const int zero_from = (kb + kTileKeys > it.Lk) ? max(0, it.Lk - kb) : kTileKeys;
          const int dt = wq * 32 + lane;
          for (int c = 0; c < DC; ++c) {
            const uint32_t slot = idx % S, bslot = bidx % SBm;
            if (!wait_all(&ring_full[slot], (idx / S) & 1) || !wait_all(&bf_empty[bslot], ((bidx / SBm) & 1) ^ 1))
              return false;
            const uint8_t* src = ring + slot * kStageBytes;
            uint8_t* dst = bfbuf + bslot * C::kBfSlotBytes;
            uint4 vin[8];
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) {
              const int x16 = dt + k8 * 128, r = x16 >> 3, c16 = x16 & 7;
              vin[k8] = r < zero_from ? *reinterpret_cast<const uint4*>(src + r * 128 + ((c16 ^ (r & 7)) << 4))
                                      : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) {
              const int x16 = dt + k8 * 128;
              const int r = x16 >> 3, c16 = x16 & 7, sw = r & 7;
              const uint4 v = vin[k8];
              const uint32_t in[4] = {v.x, v.y, v.z, v.w};
              uint32_t o[8];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                o[2 * i] = cvt_e4m3x2_bf16x2((uint16_t)(in[i] & 0xFFFF));
                o[2 * i + 1] = cvt_e4m3x2_bf16x2((uint16_t)(in[i] >> 16));
              }
              const int h = c16 >> 2, k0 = (c16 & 3) * 2;
              uint8_t* drow = dst + h * 16384 + r * 128;
              *reinterpret_cast<uint4*>(drow + ((k0 ^ sw) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
              *reinterpret_cast<uint4*>(drow + (((k0 + 1) ^ sw) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(&ring_empty[slot]);
              mbar_arrive(&bf_full[bslot]);
            }
            ++idx;
            ++bidx;
          }
          return true;
        };
        ok = convert_k(0);
        for (int u = 1; u <= n && ok; ++u) {
          if (u < n) ok = convert_k(u);
          if (ok) ok = convert_v(u - 1);
        }
      }
      if (!ok) flag_timeout(p, abort_flag);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (p.conc_role == 2) griddep_wait();  // the pair ends when the first launch has ended too
}

}  // namespace fp8pa
