// Paged FP8-KV attention forward for prefill row tiles, sm_103a: E4M3 Q, K and
// V at head dim 256 or 512, 128 packed query rows per tile.
//
// The decode kernel puts keys on the TMEM lanes (swap-AB) so that a handful of
// query rows still fills an MMA.  A prefill tile has rows to spare, so here the
// rows sit on the lanes and every row reduction is thread-local:
//
//   S[row, key] = Q[row, :] . K[key, :]     tcgen05.mma  M = 128 rows, N = 128 keys
//   P'[row, key] = 2^(S * scale - m + 4)    one softmax thread per row
//   O[row, d] += P[row, key] V[key, d]       tcgen05.mma  A = P from TMEM, N = D
//
// Rows pack (query token, query head of the KV group) token-major, as in the
// decode kernel.  P' is requantized as an E4M3 pair hi = e4m3(P'),
// lo = e4m3(P' - hi) with both terms accumulated into O, and the running row
// maximum m moves only when a tile maximum exceeds it by more than 4 (log2
// units), so P' <= 256.
//
// Tensor memory (512 columns): two S buffers of 128 columns; P's hi and lo
// terms (32 columns each, four keys per column) overwrite the first 64 columns
// of their S buffer once the row's scores are in registers; O takes 256
// columns.  At head dim 512 the output dims come in two slices of 256, each a
// work item of its own: both compute the full S and P, each accumulates O for
// its slice against that slice of V.
//
// Warps: 0 TMA producer (Q and K), 1 QK^T issuer (and TMEM owner), 2 PV issuer,
// 3 V loader, then softmax / O correction / epilogue in kSW warpgroups (kSW
// warps per row quarter, each thread 1 / kSW of a row's keys and output dims).
// The loaders and the issuers run warp-uniform loops with one elected lane
// issuing; they and the softmax warps synchronize only through mbarriers.
#pragma once
#include "attn_kernel.cuh"
#include "kernels.h"

namespace fp8pa {

namespace detail {

// P' pair from its exponent pair: 2^t with t rounded to f16 first (ex2 on f16x2).
__device__ __forceinline__ uint32_t ex2_f16x2(float t0, float t1) {
  uint32_t h, e;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(t1), "f"(t0));
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(e) : "r"(h));
  return e;
}

// f16x2 P' -> E4M3 pair hi = e4m3(P'), lo = e4m3(P' - hi) (exact in f16), 16 bits each.
__device__ __forceinline__ void e4m3_hilo_f16x2(uint32_t h, uint32_t& hi, uint32_t& lo) {
  uint32_t hh, l;
  uint16_t h8, l8;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(h8) : "r"(h));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hh) : "h"(h8));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(l) : "r"(h), "r"(hh));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(l8) : "r"(l));
  hi = h8;
  lo = l8;
}

__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ float2 f16x2_to_f32(uint32_t h) {
  __half2 v = *reinterpret_cast<__half2*>(&h);
  return __half22float2(v);
}

}  // namespace detail

template <int D>
struct PrefillCfg {
  static_assert(D == 256 || D == 512, "head dim");
  static constexpr int kRows = 128;
  static constexpr int kDC = D / 128;                     // 128-byte chunks of an E4M3 row (Q, K)
  static constexpr int kDO = 256;                         // output dims per work item
  static constexpr int kSlices = D / kDO;                 // work items per row tile
  static constexpr int kVC = kDO / 128;                   // V chunks per work item and tile
  static constexpr int kQBytes = kDC * kRows * 128;       // chunk c of every row at c * 16 KB
  static constexpr int kQBufs = D == 256 ? 2 : 1;
  static constexpr int kKStageBytes = kStageBytes;        // 128 keys x one 128-byte chunk
  static constexpr int kVStageBytes = kVC * kStageBytes;  // 128 keys x kDO bytes, chunk c at c * 16 KB
  // QK^T in two N = 64 halves: keys 64..127 (S columns 64..127) as soon as the
  // softmax has read the buffer's previous scores, keys 0..63 (the columns P
  // overwrites) once the PV of that tile has released them.  At head dim 512
  // the halves read Q twice over four chunks and a one-tile K ring cannot run
  // ahead, so there S(g) stays one N = 128 MMA per step.
  static constexpr bool kSplitQK = D == 256;
  static constexpr int kKStages = (D == 256 && !kSplitQK) ? 3 : 4;
  static constexpr int kVStages = 2;
  static constexpr int kSW = 2;                          // softmax warpgroups: each takes 128 / kSW keys of a row
  static constexpr int kKT = kTileKeys / kSW;            // keys of a tile per softmax thread
  static constexpr int kHO = kDO / kSW;                  // output dims per softmax thread
  static constexpr int kOC = kSW == 2 ? 64 : 32;         // O columns per TMEM load in the correction and epilogue
  static constexpr bool kVWarp = true;                   // V loaded by a warp of its own (else by the producer)
  static constexpr int kSm0 = kVWarp ? 4 : 3;            // first softmax warp
  static constexpr int kThreads = (kSm0 + 4 * kSW) * 32; // producer(s), 2 issuers, kSW softmax warpgroups
  static constexpr int kCtrlBytes = 1024;
  static constexpr int kXchgBytes = 3 * kSW * 512;       // row-group exchange: maxima [2][kSW][128], sums [kSW][128]
  static constexpr int kSeg = kSW == 2 ? 64 : 32;        // epilogue row segment (bytes) per staging pass
  static constexpr int kOStageBytes = 4 * kSW * 32 * kSeg;  // epilogue: 32 rows x kSeg bytes per softmax warp
  static constexpr int kSmemBytes = kQBufs * kQBytes + kKStages * kKStageBytes + kVStages * kVStageBytes +
                                    kOStageBytes + kXchgBytes + kCtrlBytes + 1024;
  static_assert(kSmemBytes <= 232448, "smem");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kOCol = 256;  // O columns [256, 256 + kDO)
  static_assert(kOCol + kDO <= 512, "TMEM");
  static constexpr float kTau = 4.0f;
  static constexpr float kPShift = 4.0f;
};

template <int D>
__global__ void __launch_bounds__(PrefillCfg<D>::kThreads, 1)
    attn_prefill_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using C = PrefillCfg<D>;
  using namespace ptx;
  using namespace detail;
  constexpr int DC = C::kDC, SK = C::kKStages, SV = C::kVStages, QB = C::kQBufs, VC = C::kVC, DO = C::kDO;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  // V ring lowest: its MMA operand spans two 16 KB blocks of a stage, and every
  // byte past a stage still lies inside this CTA's allocation
  uint8_t* vring = smem;
  uint8_t* kring = vring + SV * C::kVStageBytes;
  uint8_t* qbuf = kring + SK * C::kKStageBytes;
  uint8_t* ostage = qbuf + QB * C::kQBytes;
  uint8_t* xchg = ostage + C::kOStageBytes;
  uint8_t* ctrl = xchg + C::kXchgBytes;
  uint64_t* k_full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* k_empty = k_full + SK;
  uint64_t* v_full = k_empty + SK;
  uint64_t* v_empty = v_full + SV;
  uint64_t* q_full = v_empty + SV;
  uint64_t* q_empty = q_full + QB;
  uint64_t* s_full = q_empty + QB;  // [2] QK^T done: S buffer readable
  uint64_t* s_free = s_full + 2;    // [2] PV done: S/P buffer reusable, O up to date
  uint64_t* p_full = s_free + 2;    // [2] P written (every softmax warp)
  uint64_t* o_empty = p_full + 2;   // epilogue read O (every softmax warp)
  uint64_t* v_ready = o_empty + 1;  // tail tile: its V stage landed (PV issuer -> softmax)
  uint64_t* drain = v_ready + 1;    // [2] one per issuer
  uint64_t* never = drain + 2;      // nothing arrives on it: the stall-injection hook waits here
  uint64_t* s_read = never + 1;     // [2] S buffer's scores in registers (every softmax warp)
  uint64_t* item_full = s_read + 2;
  uint64_t* item_empty = item_full + kItemSlots;
  ItemSlot* islot = reinterpret_cast<ItemSlot*>(item_empty + kItemSlots);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(islot + kItemSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < SK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < SV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < QB; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 1);
      mbar_init(&p_full[i], 4 * C::kSW);
      mbar_init(&drain[i], 1);
      mbar_init(&s_read[i], 4 * C::kSW);
    }
    mbar_init(o_empty, 4 * C::kSW);
    mbar_init(v_ready, 1);
    mbar_init(never, 1);
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], C::kSm0 - 1 + 4 * C::kSW);  // issuers, V loader, every softmax warp
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
  griddep_wait();  // the work list, Q and the K/V cache are written by earlier kernels
  bool idle = false;
  if (p.conc_role == 1) {  // first launch of a side-by-side pair (never the second)
    idle = (int)blockIdx.x >= active_ctas(p, 1);
    griddep_launch_dependents();  // this CTA is resident: the second launch may take the free SMs
  }
  const uint32_t tmem = *tmem_slot;
  const int n_items = *p.work_count;
  const uint32_t lim = p.wait_limit;

  if (warp < C::kSm0) {
    // ---------------------------------------------------------------- producer and MMA issuers
    const bool leader = elect_one();
    const int leader_lane = __ffs(__ballot_sync(0xFFFFFFFFu, leader)) - 1;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xFFFFFFFFu, pwait(bar, parity, lim, abort_flag));
    };
    uint32_t kq = 0, vq = 0, qit = 0, g = 0;  // K / V ring positions, Q tiles, S/P tiles
    bool ok = true;
    for (uint32_t ik = 0; ok; ++ik) {
      const uint32_t is = ik % kItemSlots;
      Item it{};
      bool valid;
      if (warp == 0) {
        int w = n_items;  // an idle CTA takes no item
        if (leader && !idle) w = atomicAdd(p.work_next, 1);
        w = __shfl_sync(0xFFFFFFFFu, w, leader_lane);
        valid = w < n_items;
        if (!(ok = wait_all(&item_empty[is], ((ik / kItemSlots) & 1) ^ 1))) break;
        if (valid) it = decode_item(p, p.work[w]);
        if (leader) {
          islot[is].it = it;
          islot[is].valid = valid;
          mbar_arrive(&item_full[is]);  // release: the slot's contents are visible to waiters
        }
        __syncwarp();
      } else {
        if (!(ok = wait_all(&item_full[is], (ik / kItemSlots) & 1))) break;
        it = islot[is].it;
        valid = islot[is].valid != 0;
        __syncwarp();
        if (leader) mbar_arrive(&item_empty[is]);
        if (valid && p.inject_stall && !(ok = wait_all(never, 0))) break;
      }
      if (!valid) break;
      if (it.t1 <= it.t0) continue;
      const int n = it.t1 - it.t0;
      const int qb = qit % QB;
      const uint32_t qpar = (qit / QB) & 1;
      ++qit;
      auto load_k = [&](int u) -> bool {
        const int pg = it.pg_lo() + 2 * (it.t0 + u);
        const int pa = page_id(p, it, pg), pb = page_id(p, it, pg + 1);
        for (int c = 0; c < DC; ++c) {
          const uint32_t slot = kq % SK;
          if (!wait_all(&k_empty[slot], ((kq / SK) & 1) ^ 1)) return false;
          if (leader) {
            uint8_t* dst = kring + slot * C::kKStageBytes;
            mbar_arrive_expect_tx(&k_full[slot], C::kKStageBytes);
            tma_load_4d(dst, &tm_k, &k_full[slot], c * 128, it.hk, 0, pa);
            tma_load_4d(dst + C::kKStageBytes / 2, &tm_k, &k_full[slot], c * 128, it.hk, 0, pb);
          }
          ++kq;
        }
        return true;
      };
      auto load_v = [&](int u) -> bool {
        const int pg = it.pg_lo() + 2 * (it.t0 + u);
        const int pa = page_id(p, it, pg), pb = page_id(p, it, pg + 1);
        const uint32_t slot = vq % SV;
        if (!wait_all(&v_empty[slot], ((vq / SV) & 1) ^ 1)) return false;
        if (leader) {
          uint8_t* dst = vring + slot * C::kVStageBytes;
          mbar_arrive_expect_tx(&v_full[slot], C::kVStageBytes);
          for (int c = 0; c < VC; ++c) {
            const int cv = (it.dhalf * VC + c) * 128;  // this item's slice of the head dims
            tma_load_4d(dst + c * kStageBytes, &tm_v, &v_full[slot], cv, it.hk, 0, pa);
            tma_load_4d(dst + c * kStageBytes + kStageBytes / 2, &tm_v, &v_full[slot], cv, it.hk, 0, pb);
          }
        }
        ++vq;
        return true;
      };
      if (warp == 0) {
        // Q tile, then K(0), [K(1), V(0)], [K(2), V(1)], ..., V(n-1); or Q and the K tiles
        // alone when V has a loader warp of its own
        if (!(ok = wait_all(&q_empty[qb], qpar ^ 1))) break;
        if (leader) {
          mbar_arrive_expect_tx(&q_full[qb], C::kQBytes);
          for (int c = 0; c < DC; ++c)
            tma_load_3d(qbuf + qb * C::kQBytes + c * C::kRows * 128, &tm_q, &q_full[qb], c * 128, it.hk * p.group,
                        it.q0 + it.row0 / p.group);
        }
        if constexpr (C::kVWarp) {
          for (int u = 0; u < n && ok; ++u) ok = load_k(u);
        } else {
          ok = load_k(0);
          for (int u = 1; u <= n && ok; ++u) {
            if (u < n) ok = load_k(u);
            if (ok) ok = load_v(u - 1);
          }
        }
      } else if (C::kVWarp && warp == 3) {
        for (int u = 0; u < n && ok; ++u) ok = load_v(u);
      } else if (warp == 1) {
        // S(g) = Q . K^T into S buffer g & 1, once PV(g - 2) has released it; with
        // kSplitQK, keys 64..127 already once the softmax has read S(g - 2)
        constexpr uint32_t idesc = make_idesc(kFmtE4M3, kKMajor, kKMajor, 128, C::kSplitQK ? 64 : 128);
        if (!(ok = wait_all(&q_full[qb], qpar))) break;
        tc_fence_after();
        const uint32_t qaddr = smem_u32(qbuf + qb * C::kQBytes);
        // one half of S(gg): keys [64 h, 64 h + 64) of the tile's K stages into columns [64 h, 64 h + 64)
        auto qk_half = [&](uint32_t sb, int h, bool wait_k) -> bool {
          for (int c = 0; c < DC; ++c) {
            const uint32_t pos = kq + c, slot = pos % SK;
            if (wait_k) {
              if (!wait_all(&k_full[slot], (pos / SK) & 1)) return false;
              tc_fence_after();
            }
            const uint32_t a0 = qaddr + c * C::kRows * 128;
            const uint32_t b0 = smem_u32(kring + slot * C::kKStageBytes) + h * (C::kKStageBytes / 2);
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f8f6f4(tmem + sb * 128 + 64 * h, make_sdesc(a0 + kk * 32, 16, 1024, kLayoutSW128),
                           make_sdesc(b0 + kk * 32, 16, 1024, kLayoutSW128), idesc, (c | kk) != 0);
              if (h == 0) mma_commit(&k_empty[slot]);  // the stage's last MMAs
            }
          }
          return true;
        };
        for (int u = 0; u < n && ok; ++u) {
          const uint32_t gg = g + u, sb = gg & 1;
          if constexpr (C::kSplitQK) {
            if (!(ok = wait_all(&s_read[sb], ((gg >> 1) & 1) ^ 1))) break;
            tc_fence_after();
            if (!(ok = qk_half(sb, 1, true))) break;
            if (!(ok = wait_all(&s_free[sb], ((gg >> 1) & 1) ^ 1))) break;
            tc_fence_after();
            if (!(ok = qk_half(sb, 0, false))) break;
          } else {
            if (!(ok = wait_all(&s_free[sb], ((gg >> 1) & 1) ^ 1))) break;
            tc_fence_after();
            for (int c = 0; c < DC && ok; ++c) {
              const uint32_t slot = (kq + c) % SK;
              if (!(ok = wait_all(&k_full[slot], ((kq + c) / SK) & 1))) break;
              tc_fence_after();
              const uint32_t a0 = qaddr + c * C::kRows * 128, b0 = smem_u32(kring + slot * C::kKStageBytes);
              // issued by the converged warp, predicated on the elected lane: at four
              // chunks per tile the issuing thread's cost per MMA otherwise shows
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f8f6f4_p(leader, tmem + sb * 128, make_sdesc(a0 + kk * 32, 16, 1024, kLayoutSW128),
                             make_sdesc(b0 + kk * 32, 16, 1024, kLayoutSW128), idesc, (c | kk) != 0);
              mma_commit_p(leader, &k_empty[slot]);
            }
            if (!ok) break;
          }
          kq += DC;
          mma_commit_p(leader, &s_full[sb]);
        }
        if (ok && leader) mma_commit(&q_empty[qb]);
      } else {
        // O += P(g) . V(g): A = P hi and lo terms from TMEM, B = V slice (MN-major, N = kDO)
        constexpr uint32_t idesc = make_idesc(kFmtE4M3, kKMajor, kMNMajor, 128, DO);
        for (int u = 0; u < n && ok; ++u) {
          const uint32_t gg = g + u, sb = gg & 1;
          const uint32_t slot = vq % SV, vpar = (vq / SV) & 1;
          const bool tail = (it.pg_lo() + 2 * (it.t0 + u)) * kPage + kTileKeys > it.Lk;
          if (tail) {
            // the softmax zeroes this tile's V rows past Lk once the stage has landed
            if (!(ok = wait_all(&v_full[slot], vpar))) break;
            if (leader) mbar_arrive(v_ready);
          }
          if (!(ok = wait_all(&p_full[sb], (gg >> 1) & 1))) break;
          if (u == 0 && !(ok = wait_all(o_empty, ((qit - 1) & 1) ^ 1))) break;
          if (!(ok = wait_all(&v_full[slot], vpar))) break;
          tc_fence_after();
          const uint32_t v0 = smem_u32(vring + slot * C::kVStageBytes);
          if constexpr (C::kSplitQK) {
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t vb = make_sdesc(v0 + kk * 4096, kStageBytes, 1024, kLayoutSW128);
                mma_f8f6f4_tmem_a(tmem + C::kOCol, tmem + sb * 128 + kk * 8, vb, idesc, !(u == 0 && kk == 0));
                mma_f8f6f4_tmem_a(tmem + C::kOCol, tmem + sb * 128 + 32 + kk * 8, vb, idesc, 1);
              }
              mma_commit(&v_empty[slot]);
              mma_commit(&s_free[sb]);
            }
          } else {  // head dim 512: from the converged warp, as QK^T
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t vb = make_sdesc(v0 + kk * 4096, kStageBytes, 1024, kLayoutSW128);
              mma_f8f6f4_tmem_a_p(leader, tmem + C::kOCol, tmem + sb * 128 + kk * 8, vb, idesc, !(u == 0 && kk == 0));
              mma_f8f6f4_tmem_a_p(leader, tmem + C::kOCol, tmem + sb * 128 + 32 + kk * 8, vb, idesc, 1);
            }
            mma_commit_p(leader, &v_empty[slot]);
            mma_commit_p(leader, &s_free[sb]);
          }
          ++vq;
        }
      }
      g += n;
    }
    if (!ok && leader) flag_timeout(p, abort_flag);
    if (warp == 0 || (C::kVWarp && warp == 3)) {
      // every issued copy must land before the CTA may exit (each loader drains its own)
      for (uint32_t j = kq > (uint32_t)SK ? kq - SK : 0; j < kq; ++j)
        mbar_wait(&k_full[j % SK], (j / SK) & 1, kDrainWaitLimit);
      for (uint32_t j = vq > (uint32_t)SV ? vq - SV : 0; j < vq; ++j)
        mbar_wait(&v_full[j % SV], (j / SV) & 1, kDrainWaitLimit);
      if (warp == 0)
        for (uint32_t j = qit > (uint32_t)QB ? qit - QB : 0; j < qit; ++j)
          mbar_wait(&q_full[j % QB], (j / QB) & 1, kDrainWaitLimit);
    } else {
      uint64_t* my_drain = &drain[warp - 1];
      if (leader) mma_commit(my_drain);
      __syncwarp();
      mbar_wait(my_drain, 0, kDrainWaitLimit);
    }
  } else {
    // ---------------------------------------------------------------- softmax, O correction, epilogue
    // kSW warpgroups.  The kSW warps of lane quarter q (one per group) own rows
    // 32q .. 32q + 31; warpgroup hw takes keys [KT hw, KT hw + KT) of every tile
    // and output dims [hw * HO, (hw + 1) * HO).  The warps of a row group
    // exchange their partial tile maxima (and finally their row sums) through
    // shared memory on named barrier 1 + q, and every early exit is a vote on
    // that barrier, so the warps of a group always leave together.
    constexpr int SW = C::kSW, KT = C::kKT, HO = C::kHO, OC = C::kOC;
    const int hw = (warp - C::kSm0) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // this thread's row = its TMEM lane
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t pair_bar = 1 + quarter;
    const float NEG_INF = __int_as_float(0xFF800000);
    float* xmax = reinterpret_cast<float*>(xchg);  // [2][SW][128] partial tile maxima, by tile parity
    float* lsum = xmax + 2 * SW * 128;             // [SW][128] partial row sums
    uint32_t g = 0, vq = 0, tails = 0;
    auto wait_w = [&](uint64_t* bar, uint32_t parity) {
      const bool w_ok = __all_sync(0xFFFFFFFFu, pwait(bar, parity, lim, abort_flag));
      if (!w_ok) flag_timeout(p, abort_flag);
      return w_ok;
    };
    auto pair_fail = [&](bool ok_here) { return bar_red_or(pair_bar, 32 * SW, !ok_here); };
    bool aborted = false;
    for (uint32_t ik = 0; !aborted; ++ik) {
      const uint32_t is = ik % kItemSlots;
      const bool iok = wait_w(&item_full[is], (ik / kItemSlots) & 1);
      if (pair_fail(iok)) break;
      const Item it = islot[is].it;
      const bool valid = islot[is].valid != 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[is]);
      if (!valid) break;
      const int G = p.group;
      const bool live = r < it.nrows;
      const int tok = it.q0 + (it.row0 + r) / G;
      const int head = it.hk * G + (it.row0 + r) % G;
      const size_t orow = (size_t)tok * p.hq + head;
      const size_t li = (size_t)head * p.total_q + tok;
      const int dbase = it.dhalf * DO + hw * HO;  // first output dim of this warpgroup
      if (it.t1 <= it.t0) {
        // nothing visible: out = 0, lse = -inf
        if (live) {
          uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow * D + dbase);
          for (int i = 0; i < HO / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
          if (p.lse && it.dhalf == 0 && hw == 0) p.lse[li] = p.sinks ? p.sinks[head] : NEG_INF;
        }
        continue;
      }
      const int n = it.t1 - it.t0;
      const float kd = load_descale(p.k_descale, p, it);
      const float vd = load_descale(p.v_descale, p, it);
      const float scale = p.softmax_scale_log2 * kd * (p.q_descale ? *p.q_descale : 1.0f);
      // this row's visible keys [lo_r, hi_r]; an empty range for padding rows
      const int pq = it.Lk - it.Lq + (it.row0 + r) / G;
      int lo_r = p.window_left >= 0 ? max(0, pq - p.window_left) : 0;
      int hi_r = p.causal ? min(pq, it.Lk - 1) : it.Lk - 1;
      if (!live) {
        lo_r = 1;
        hi_r = 0;
      }
      float m = NEG_INF, l0 = 0.f, l1 = 0.f;
      bool sticky = true;  // waits after a tile's vote that failed; reported at the next vote
      for (int u = 0; u < n; ++u, ++g) {
        const int kb = (it.pg_lo() + 2 * (it.t0 + u)) * kPage + KT * hw;  // first key of this part
        const uint32_t sb = g & 1;
        const bool sok = wait_w(&s_full[sb], (g >> 1) & 1);
        float x[KT];
        if (sok) {
          tc_fence_after();
          if constexpr (KT == 64)
            tmem_load64f(tmem + lane_base + sb * 128 + KT * hw, x);
          else
            tmem_load32f(tmem + lane_base + sb * 128 + KT * hw, x);
        } else {
#pragma unroll
          for (int i = 0; i < KT; ++i) x[i] = NEG_INF;
        }
        if constexpr (C::kSplitQK) {
          // the scores are in registers: keys 64..127 of S(g + 2) may go to this buffer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_read[sb]);
        }
        if (!(kb >= lo_r && kb + KT - 1 <= hi_r)) {
#pragma unroll
          for (int i = 0; i < KT; ++i)
            if (kb + i < lo_r || kb + i > hi_r) x[i] = NEG_INF;
        }
        // partial tile maximum (raw scores; scale > 0), then the row group's
        float t[KT / 4];
#pragma unroll
        for (int i = 0; i < KT / 4; ++i) t[i] = fmax3(x[4 * i], x[4 * i + 1], fmaxf(x[4 * i + 2], x[4 * i + 3]));
#pragma unroll
        for (int w = KT / 8; w >= 1; w >>= 1)
#pragma unroll
          for (int i = 0; i < w; ++i) t[i] = fmaxf(t[i], t[i + w]);
        xmax[(sb * SW + hw) * 128 + r] = t[0];
        if (pair_fail(sok && sticky)) {
          aborted = true;
          break;
        }
        float tmax = xmax[(sb * SW) * 128 + r];
#pragma unroll
        for (int j = 1; j < SW; ++j) tmax = fmaxf(tmax, xmax[(sb * SW + j) * 128 + r]);
        const float ts = tmax * scale;
        float alpha = 1.0f;
        bool resc = false;
        if (ts > m + C::kTau) {
          // a row that has seen no key yet has O = 0 and l = 0: nothing to rescale
          if (m != NEG_INF) {
            alpha = ex2(m - ts);
            resc = true;
          }
          m = ts;
        }
        const float nm = m == NEG_INF ? 0.0f : C::kPShift - m;
        if (__any_sync(0xFFFFFFFFu, resc)) {
          l0 *= alpha;
          l1 *= alpha;
          // this warpgroup's O columns *= alpha once PV(g - 1) has accumulated into O
          if (u > 0) sticky = wait_w(&s_free[(g - 1) & 1], ((g - 1) >> 1) & 1) && sticky;
          tc_fence_after();
#pragma unroll 1
          for (int q = 0; q < HO / OC; ++q) {
            float o[OC];
            const uint32_t ta = tmem + lane_base + C::kOCol + hw * HO + OC * q;
            if constexpr (OC == 64)
              tmem_load64f(ta, o);
            else
              tmem_load32f(ta, o);
#pragma unroll
            for (int i = 0; i < OC; i += 2) {
              const float2 v = __fmul2_rn(make_float2(o[i], o[i + 1]), make_float2(alpha, alpha));
              o[i] = v.x;
              o[i + 1] = v.y;
            }
            if constexpr (OC == 64)
              tmem_store64f(ta, o);
            else
              tmem_store32f(ta, o);
          }
        }
        // P' = 2^(x * scale - m + shift) as an E4M3 pair, 32 keys (8 columns) at a time;
        // this part's words are columns [KT/4 hw, KT/4 (hw + 1)) of the hi and lo terms, which
        // overwrite the first 64 columns of this S buffer (the group's scores are in registers)
#pragma unroll
        for (int q = 0; q < KT / 32; ++q) {
          uint32_t hi[8], lo[8];
          uint32_t sa = 0, sb2 = 0;  // f16x2 partial row sums of these 32 keys
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int k = 32 * q + 4 * i;
            const float2 a = __ffma2_rn(make_float2(x[k], x[k + 1]), make_float2(scale, scale), make_float2(nm, nm));
            const float2 b =
                __ffma2_rn(make_float2(x[k + 2], x[k + 3]), make_float2(scale, scale), make_float2(nm, nm));
            const uint32_t h01 = ex2_f16x2(a.x, a.y), h23 = ex2_f16x2(b.x, b.y);
            sa = hadd2(sa, h01);
            sb2 = hadd2(sb2, h23);
            uint32_t e01, f01, e23, f23;
            e4m3_hilo_f16x2(h01, e01, f01);
            e4m3_hilo_f16x2(h23, e23, f23);
            hi[i] = e01 | (e23 << 16);
            lo[i] = f01 | (f23 << 16);
          }
          const float2 fa = f16x2_to_f32(sa), fb = f16x2_to_f32(sb2);
          l0 += fa.x + fb.x;
          l1 += fa.y + fb.y;
          tmem_store8(tmem + lane_base + sb * 128 + (KT / 4) * hw + 8 * q, hi);
          tmem_store8(tmem + lane_base + sb * 128 + 32 + (KT / 4) * hw + 8 * q, lo);
        }
        tmem_wait_st();
        // rows of the last page past the sequence end may hold anything (even NaN):
        // zero those V rows so that 0 * V stays 0 in the PV MMA
        const int kt = (it.pg_lo() + 2 * (it.t0 + u)) * kPage;
        if (kt + kTileKeys > it.Lk) {
          sticky = wait_w(v_ready, tails & 1) && sticky;
          ++tails;
          const int zr = max(0, it.Lk - kt);
          uint8_t* st = vring + (vq % SV) * C::kVStageBytes;
          for (int c = 0; c < VC; ++c)
            for (int x16 = zr * 8 + hw * 128 + r; x16 < kTileKeys * 8; x16 += 128 * SW)
              *reinterpret_cast<uint4*>(st + c * kStageBytes + x16 * 16) = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
        }
        ++vq;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[sb]);
      }
      if (aborted) break;
      // ---------------- epilogue: O / l, lse
      // Row sums, scales and destinations need the last tile's P, not its PV:
      // they are formed while that PV completes, and O is read after it.
      lsum[hw * 128 + r] = l0 + l1;
      if (pair_fail(sticky)) break;
      float l = lsum[r];
#pragma unroll
      for (int j = 1; j < SW; ++j) l += lsum[j * 128 + r];
      float inv = l > 0.f ? vd / l : 0.f;
      float lse2 = l > 0.f ? m - C::kPShift + __log2f(l) : NEG_INF;
      if (p.sinks && live) fold_sink(l, m - C::kPShift, p.sinks[head] * 1.4426950408889634f, vd, inv, lse2);
      // Each kSeg-byte column segment of this warp's 32 rows goes through a
      // 32 x kSeg staging buffer (row-major, 16-byte pieces swizzled by row), then
      // out as kSeg-byte row segments: lane l stores piece l % NP of row
      // i * (32 / NP) + l / NP, with NP = kSeg / 16 pieces per segment.
      constexpr int SEG = C::kSeg, NP = SEG / 16, SC = SEG / 2;  // bytes, pieces, columns per segment
      const int sw_shift = NP == 4 ? 1 : 2;                      // piece swizzle: (row >> sw_shift) & (NP - 1)
      uint8_t* stg = ostage + (warp - C::kSm0) * 32 * SEG;
      __nv_bfloat16* dst_row[NP];
      bool dst_live[NP];
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const int rr = quarter * 32 + i * (32 / NP) + lane / NP;
        dst_live[i] = rr < it.nrows;
        const size_t row = (size_t)(it.q0 + (it.row0 + rr) / G) * p.hq + it.hk * G + (it.row0 + rr) % G;
        dst_row[i] = reinterpret_cast<__nv_bfloat16*>(p.out) + row * D + dbase + (lane % NP) * 8;
      }
      const bool eok = wait_w(&s_free[(g - 1) & 1], ((g - 1) >> 1) & 1);
      if (pair_fail(eok)) break;
      tc_fence_after();
#pragma unroll 1
      for (int q2 = 0; q2 < HO / OC; ++q2) {
        float o[OC];
        if constexpr (OC == 64)
          tmem_load64f(tmem + lane_base + C::kOCol + hw * HO + OC * q2, o);
        else
          tmem_load32f(tmem + lane_base + C::kOCol + hw * HO + OC * q2, o);
#pragma unroll
        for (int hh = 0; hh < OC / SC; ++hh) {
          const int q = (OC / SC) * q2 + hh;
#pragma unroll
          for (int c = 0; c < NP; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              __nv_bfloat162 b2 =
                  __floats2bfloat162_rn(o[SC * hh + 8 * c + 2 * i] * inv, o[SC * hh + 8 * c + 2 * i + 1] * inv);
              w[i] = *reinterpret_cast<uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(stg + lane * SEG + ((c ^ ((lane >> sw_shift) & (NP - 1))) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < NP; ++i) {
            const int rr = i * (32 / NP) + lane / NP, c = lane % NP;
            const uint4 v = *reinterpret_cast<const uint4*>(stg + rr * SEG + ((c ^ ((rr >> sw_shift) & (NP - 1))) << 4));
            if (dst_live[i]) *reinterpret_cast<uint4*>(dst_row[i] + SC * q) = v;
          }
          __syncwarp();
        }
      }
      if (live && p.lse && it.dhalf == 0 && hw == 0) p.lse[li] = lse2 * 0.69314718055994531f;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch_attn_prefill(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, int sms, cudaStream_t stream) {
  using C = PrefillCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(attn_prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_prefill_kernel<D>, dim3(sms), dim3(C::kThreads), (size_t)C::kSmemBytes, stream, p, tm_q,
                    tm_k, tm_v);
}

}  // namespace fp8pa
