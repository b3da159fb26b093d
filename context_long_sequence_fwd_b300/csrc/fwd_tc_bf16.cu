// bf16 ring-attention forward on the sm_103a tensor cores (tcgen05 + TMEM).
//
// Persistent: one CTA per SM claims the planner's items, longest first, from
// a work counter as it becomes free (one item per CTA in stepwise mode).  An
// item is two 128-row query tiles (A and B) that read the same key/value head,
// and the item's key ranges in ring order (ring
// step s visits the K/V shard of rank (r - s) mod P; axolotl "Sequence
// Parallelism" page, introduction; aicassindra "tm_sp_math", "Context
// parallelism is the axis that is independent").  No T x T score matrix is
// formed: each 128 x 128 block of scores lives in tensor memory only while
// its softmax runs (FlashAttention-style tiling, archcrux interview page).
//
// Roles (384 threads), each looping over the CTA's items:
//   warp 0      TMA producer: Q_A, Q_B once per item (as soon as the previous
//               item's last S MMAs have read the Q buffer), then K_j, V_j into
//               a ring of shared-memory slots (128 B swizzle; five 32 KB slots
//               at head dimension 128, eight 16 KB slots at 64) that runs on
//               across items.
//   warp 1      allocates TMEM; one thread issues every tcgen05.mma:
//                 S_X = Q_X K_j^T      (SS, both operands K-major)
//                 O_X += P_X V_j       (TS: P from TMEM, V MN-major)
//               ordered PV_A(j), S_A(j+1), PV_B(j), S_B(j+1) so one tile's
//               softmax overlaps the other tile's MMAs.
//   warps 4-7   softmax of tile A, warps 8-11 softmax of tile B: one query
//               row per thread, read from TMEM lane (warp % 4) * 32 + lane.
// TMEM columns: S_A 0-127, S_B 128-255, O_A from 256, O_B from 384 (D
// columns each, D = 64 or 128).  P (bf16,
// two per column) overwrites the first 64 columns of its S block; tcgen05
// MMAs of one thread execute in issue order, so S_X(j+1) cannot overwrite
// P_X(j) before PV_X(j) has read it.  At an item boundary the next item's
// S_X(0) follows the current item's last PV_X at once, while the softmax warps
// run the epilogue; the next item's first P_X, and with it the PV_X that
// overwrites O_X, comes only after the epilogue has read O_X.
//
// Online softmax, in the log2 domain (scores pre-multiplied by
// scale * log2 e): the running maximum is only raised when a tile's maximum
// exceeds it by more than 8 (a factor 256), so O in TMEM is rescaled rarely;
// the final O / l and lse = ln 2 * (m + log2 l) are exact whatever maximum
// was used.  Carrying (m, l, O) from one ring step to the next is exactly
// the log-sum-exp merge of the steps' partial results.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "device_common.cuh"
#include "launch.h"
#include "sm103_ptx.cuh"
#include "trace.h"

namespace ra {

namespace {

// Per head dimension (64 or 128): a 128 x D bf16 tile is D / 64 boxes of
// 128 rows x 64 columns, each one 128-byte swizzle span wide.
template <int kD>
struct FwdCfg {
  static constexpr int kBN = 128;                   // keys per K/V tile
  static constexpr int kStages = kD == 128 ? 5 : 8; // K/V slots
  static constexpr int kTileBytes = kBN * kD * 2;   // one 128 x D bf16 tile
  static constexpr int kOffQ = 0;                   // Q_A, Q_B
  static constexpr int kOffKV = 2 * kTileBytes;     // K/V ring
  static constexpr int kOffCtl = kOffKV + kStages * kTileBytes;
  static constexpr int kSmemBytes = kOffCtl + 512 + 1024;  // control block + alignment slack
  static constexpr uint32_t kIdescQK = make_idesc_bf16(128, 128, false, false);
  static constexpr uint32_t kIdescPV = make_idesc_bf16(128, kD, false, true);
  static_assert(kD == 64 || kD == 128, "head dimension");
  static_assert(kSmemBytes <= 232448, "dynamic shared memory of one CTA");
};

constexpr int kBN = 128;                     // keys per K/V tile
constexpr int kHalfBytes = 128 * 64 * 2;     // 128 rows x 64 columns (one swizzle span)
constexpr int kMaxStages = 8;
constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 8.0f;    // log2 units
constexpr int kSchedSlots = 4;               // item indices in flight inside a CTA

struct Ctl {
  uint64_t q_full;
  uint64_t q_empty;  // the item's last S MMAs have read Q
  uint64_t kv_full[kMaxStages];
  uint64_t kv_empty[kMaxStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full[2];
  uint64_t mma_done;
  uint64_t sched_full[kSchedSlots];   // item index published by the producer
  uint64_t sched_empty[kSchedSlots];  // read by the MMA thread and the 8 softmax warps
  int sched[kSchedSlots];             // item index, -1 = no more items
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Ctl) <= 512, "control block");

template <int kD>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
    mma_bf16_ss(d_tmem, make_sdesc_sw128(q_smem + off, 16, 1024),
                make_sdesc_sw128(k_smem + off, 16, 1024), FwdCfg<kD>::kIdescQK, kk > 0);
  }
}

template <int kD>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem,
                                         bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk) {
    mma_bf16_ts(d_tmem, p_tmem + kk * 8, make_sdesc_sw128(v_smem + kk * 2048, kHalfBytes, 1024),
                FwdCfg<kD>::kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// Number of K/V tiles an item visits (the same count in every role).
__device__ __forceinline__ int item_tiles(const PlanItem& it, const FwdParams& p) {
  int n = 0;
  for (int si = 0; si < it.seg_count; ++si) {
    const PlanSegment sg = p.segs[checked(it.seg_begin + si, p.num_segs, p.status, kSiteFwdSeg)];
    if (seg_selected(sg, p.step_filter)) n += (sg.k1 - sg.k0 + kBN - 1) / kBN;
  }
  return n;
}

template <int kD>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_bf16_kernel(const __grid_constant__ CUtensorMap map_q,
                       const __grid_constant__ CUtensorMap map_k,
                       const __grid_constant__ CUtensorMap map_v, const FwdParams p) {
  using Cfg = FwdCfg<kD>;
  constexpr int kStages = Cfg::kStages;
  constexpr int kTileBytes = Cfg::kTileBytes;
  constexpr int kOffQ = Cfg::kOffQ;
  constexpr int kOffKV = Cfg::kOffKV;
  constexpr int kOffCtl = Cfg::kOffCtl;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kOffCtl);
  const uint32_t sQ = smem_u32(smem + kOffQ);
  const uint32_t sKV = smem_u32(smem + kOffKV);
  volatile int* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&ctl->q_full, 1);
    mbar_init(&ctl->q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->kv_full[s], 1);
      mbar_init(&ctl->kv_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&ctl->s_full[x], 1);
      mbar_init(&ctl->p_full[x], 128);
      mbar_init(&ctl->o_full[x], 1);
    }
    mbar_init(&ctl->mma_done, 1);
    for (int s = 0; s < kSchedSlots; ++s) {
      mbar_init(&ctl->sched_full[s], 1);
      mbar_init(&ctl->sched_empty[s], 9);
    }
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;

  // Items: with a work counter (persistent launch) the producer claims the
  // next item of the longest-first list with an atomic add whenever it is
  // ready for one, and publishes its index to the other roles through a small
  // ring in shared memory (-1 ends the list); without one, CTA i runs item i.
  // Items with no K/V tile in the selected ring step take part in no barrier.
  auto next_item = [&](int* spos, bool* ok) -> int {  // consumers of the ring
    const int s = *spos % kSchedSlots;
    *ok = __all_sync(__activemask(), mbar_wait(&ctl->sched_full[s], (*spos / kSchedSlots) & 1,
                                               p.status, abort));
    if (!*ok) return -1;
    const int k = *reinterpret_cast<volatile int*>(&ctl->sched[s]);
    __syncwarp(__activemask());
    if (warp == 1 || lane == 0) mbar_arrive(&ctl->sched_empty[s]);
    ++*spos;
    return k;
  };
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one_sync()) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_v);
      int li = 0;      // K/V ring position, continued across items
      int items = 0;   // items with work so far (Q buffer uses)
      int spos = 0;    // item-index ring position
      bool ok = true;
      for (bool first = true; ok; first = false) {
        int k = -1;
        if (p.work_counter) {
          k = atomicAdd(p.work_counter, 1);
          if (k >= p.num_items) k = -1;
        } else if (first) {
          k = blockIdx.x;
        }
        const int s = spos % kSchedSlots;
        if (spos >= kSchedSlots &&
            !mbar_wait(&ctl->sched_empty[s], ((spos / kSchedSlots) - 1) & 1, p.status, abort)) {
          ok = false;
          break;
        }
        ctl->sched[s] = k;
        mbar_arrive(&ctl->sched_full[s]);
        ++spos;
        if (k < 0) break;
        const PlanItem it = p.items[checked(k, p.num_items, p.status, kSiteFwdItem)];
        const int n = item_tiles(it, p);
        if (n == 0) continue;
        const bool has_b = it.qlen[1] > 0;
        const int g = it.head[0] / p.group;
        // the previous item's last S MMAs have read the Q buffer
        if (items > 0 && !mbar_wait(&ctl->q_empty, (items - 1) & 1, p.status, abort)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&ctl->q_full, (has_b ? 2 : 1) * kTileBytes);
        const int qa = local_row(p.qmap, it.q0[0]), qb = local_row(p.qmap, it.q0[1]);
        index_ok(qa, p.q_rows, p.status, kSiteFwdQRow);
        index_ok(it.head[0], p.hq, p.status, kSiteHead);
        if (has_b) {
          index_ok(qb, p.q_rows, p.status, kSiteFwdQRow);
          index_ok(it.head[1], p.hq, p.status, kSiteHead);
        }
        index_ok(g, p.hkv, p.status, kSiteHead);
        for (int hf = 0; hf < kD / 64; ++hf) {
          tma_load_3d(smem + kOffQ + hf * kHalfBytes, &map_q, &ctl->q_full, hf * 64, it.head[0],
                      qa);
          if (has_b)
            tma_load_3d(smem + kOffQ + kTileBytes + hf * kHalfBytes, &map_q, &ctl->q_full,
                        hf * 64, it.head[1], qb);
        }
        ++items;
        for (int si = 0; si < it.seg_count && ok; ++si) {
          const PlanSegment sg =
              p.segs[checked(it.seg_begin + si, p.num_segs, p.status, kSiteFwdSeg)];
          if (!seg_selected(sg, p.step_filter)) continue;
          for (int kt = sg.k0; kt < sg.k1 && ok; kt += kBN) {
            for (int kv = 0; kv < 2; ++kv, ++li) {
              const int slot = li % kStages;
              if (li >= kStages &&
                  !mbar_wait(&ctl->kv_empty[slot], ((li / kStages) - 1) & 1, p.status, abort)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&ctl->kv_full[slot], kTileBytes);
              const CUtensorMap* map = kv == 0 ? &map_k : &map_v;
              index_ok(local_row(p.kmap, kt), p.k_rows, p.status, kSiteFwdKvRow);
              for (int hf = 0; hf < kD / 64; ++hf)
                tma_load_3d(smem + kOffKV + slot * kTileBytes + hf * kHalfBytes, map,
                            &ctl->kv_full[slot], hf * 64, g, local_row(p.kmap, kt));
            }
          }
        }
      }
      if (!ok) *abort = 1;
      // let every copy this thread started land before the CTA can exit
      for (int s = 0; s < kStages && s < li; ++s) {
        const int last = s + ((li - 1 - s) / kStages) * kStages;
        mbar_wait(&ctl->kv_full[s], (last / kStages) & 1, p.status, nullptr);
      }
      if (items > 0) mbar_wait(&ctl->q_full, (items - 1) & 1, p.status, nullptr);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (elect_one_sync()) {
      const uint32_t tS[2] = {tmem + 0, tmem + 128};
      const uint32_t tO[2] = {tmem + 256, tmem + 384};
      const uint32_t sQx[2] = {sQ, sQ + kTileBytes};
      auto kv_ready = [&](int li) {
        return mbar_wait(&ctl->kv_full[li % kStages], (li / kStages) & 1, p.status, abort);
      };
      auto slot_addr = [&](int li) { return sKV + (li % kStages) * kTileBytes; };
      int li = 0;            // K/V ring position
      int items = 0;         // items with work so far
      int done[2] = {0, 0};  // P tiles consumed so far, per query tile (p_full phases)
      int spos = 0;
      bool ok = true;
      for (;;) {
        const int k = next_item(&spos, &ok);
        if (k < 0) break;
        const PlanItem it = p.items[checked(k, p.num_items, p.status, kSiteFwdItem)];
        const int n = item_tiles(it, p);
        if (n == 0) continue;
        const bool has_b = it.qlen[1] > 0;
        if (!(ok = mbar_wait(&ctl->q_full, items & 1, p.status, abort) && kv_ready(li))) break;
        tc_fence_after_sync();
        issue_qk<kD>(tS[0], sQx[0], slot_addr(li));
        mma_commit(&ctl->s_full[0]);
        if (has_b) {
          issue_qk<kD>(tS[1], sQx[1], slot_addr(li));
          mma_commit(&ctl->s_full[1]);
        }
        mma_commit(&ctl->kv_empty[li % kStages]);
        if (n == 1) mma_commit(&ctl->q_empty);  // no further S of this item reads Q
        for (int j = 0; j < n && ok; ++j) {
          const int liV = li + 2 * j + 1, liK = li + 2 * j + 2;
          if (!(ok = kv_ready(liV))) break;
          if (!(ok = mbar_wait(&ctl->p_full[0], done[0] & 1, p.status, abort))) break;
          ++done[0];
          tc_fence_after_sync();
          issue_pv<kD>(tO[0], tS[0], slot_addr(liV), j > 0);
          if (j == n - 1) mma_commit(&ctl->o_full[0]);
          const bool more = j + 1 < n;
          if (more) {
            if (!(ok = kv_ready(liK))) break;
            tc_fence_after_sync();
            issue_qk<kD>(tS[0], sQx[0], slot_addr(liK));
            mma_commit(&ctl->s_full[0]);
          }
          if (has_b) {
            if (!(ok = mbar_wait(&ctl->p_full[1], done[1] & 1, p.status, abort))) break;
            ++done[1];
            tc_fence_after_sync();
            issue_pv<kD>(tO[1], tS[1], slot_addr(liV), j > 0);
            if (j == n - 1) mma_commit(&ctl->o_full[1]);
          }
          mma_commit(&ctl->kv_empty[liV % kStages]);
          if (more) {
            if (has_b) {
              issue_qk<kD>(tS[1], sQx[1], slot_addr(liK));
              mma_commit(&ctl->s_full[1]);
            }
            mma_commit(&ctl->kv_empty[liK % kStages]);
            if (j + 2 == n) mma_commit(&ctl->q_empty);  // that was the item's last S
          }
        }
        li += 2 * n;
        ++items;
      }
      if (!ok) *abort = 1;
      // every MMA this thread issued has completed before TMEM is released
      mma_commit(&ctl->mma_done);
      mbar_wait(&ctl->mma_done, 0, p.status, nullptr);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int x = (warp - 4) >> 2;  // query tile
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + x * 128;
    const uint32_t tO = tmem + lane_off + 256 + x * 128;
    const float sl2 = p.scale_log2;
    int seen = 0;   // S tiles of this query-tile slot so far (s_full phases)
    int items = 0;  // items of this slot with work so far (o_full phases)
    int spos = 0;
    bool ok = true;
    for (;;) {
      const int k = next_item(&spos, &ok);
      if (k < 0) break;
      const PlanItem it = p.items[checked(k, p.num_items, p.status, kSiteFwdItem)];
      if (x == 1 && it.qlen[1] == 0) continue;
      const int n = item_tiles(it, p);
      // x is uniform per warp: select fields instead of indexing the item
      const int row = (x ? it.q0[1] : it.q0[0]) + r;
      const bool valid = r < (x ? it.qlen[1] : it.qlen[0]);
      const int head = x ? it.head[1] : it.head[0];
      int lo = 0, hi = 0;
      if (valid) row_key_interval(p, row, &lo, &hi);
      const int mlo = x ? it.mask_lo[1] : it.mask_lo[0];
      const int mhi = x ? it.mask_hi[1] : it.mask_hi[0];
      float m2 = -INFINITY;  // running max, log2 units
      float l = 0.f;
      int j = 0;
      for (int si = 0; si < it.seg_count && ok; ++si) {
        const PlanSegment sg =
            p.segs[checked(it.seg_begin + si, p.num_segs, p.status, kSiteFwdSeg)];
        if (!seg_selected(sg, p.step_filter)) continue;
        const int a = max(lo, sg.k0), b = min(hi, sg.k1);
        const int full_lo = max(sg.k0, mlo), full_hi = min(sg.k1, mhi);
        for (int kt = sg.k0; kt < sg.k1; kt += kBN, ++j, ++seen) {
          // .sync.aligned TMEM accesses follow: keep the warp's decision uniform
          ok = __all_sync(0xffffffffu, mbar_wait(&ctl->s_full[x], seen & 1, p.status, abort));
          if (!ok) break;
          tc_fence_after_sync();
          float s[kBN];
          {
            uint32_t u[kBN];  // one load of the row's 128 scores, one wait
            tmem_load_128(tS, u);
#pragma unroll
            for (int i = 0; i < kBN; ++i) s[i] = __uint_as_float(u[i]);
          }
          // keys outside [a, b) are hidden unless the whole tile is visible
          // to every row of this query tile
          if (!(kt >= full_lo && kt + kBN <= full_hi)) {
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
              const int key = kt + c;
              if (key < a || key >= b) s[c] = -INFINITY;
            }
          }
          // row max: four interleaved chains of 3-input maxes
          float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
          for (int c = 4; c < kBN - 4; c += 8) {
            m4[0] = fmax3(m4[0], s[c], s[c + 1]);
            m4[1] = fmax3(m4[1], s[c + 2], s[c + 3]);
            m4[2] = fmax3(m4[2], s[c + 4], s[c + 5]);
            m4[3] = fmax3(m4[3], s[c + 6], s[c + 7]);
          }
          m4[0] = fmax3(m4[0], s[kBN - 4], s[kBN - 3]);
          m4[1] = fmax3(m4[1], s[kBN - 2], s[kBN - 1]);
          const float mx = fmax3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
          const float m_new = fmaxf(m2, mx * sl2);
          const bool resc = m_new > m2 + kRescaleThreshold;
          float alpha = 1.f;
          if (resc) {
            alpha = fast_exp2(m2 - m_new);
            m2 = m_new;
          }
          const float m_use = (m2 == -INFINITY) ? 0.f : m2;
          // P = 2^(S scale log2 e - m), two columns per paired FMA and add
          const uint64_t sl2x2 = f32x2(sl2, sl2), negm2 = f32x2(-m_use, -m_use);
          uint64_t acc[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
          uint32_t pk[kBN / 2];
#pragma unroll
          for (int c = 0; c < kBN / 2; ++c) {
            float x0, x1;
            f32x2_split(ffma2(f32x2(s[2 * c], s[2 * c + 1]), sl2x2, negm2), &x0, &x1);
            const float p0 = fast_exp2(x0);
            const float p1 = fast_exp2(x1);
            acc[c & 1] = fadd2(acc[c & 1], f32x2(p0, p1));
            pk[c] = pack_bf16x2(p0, p1);
          }
          float sum;
          {
            float a0, a1, b0, b1;
            f32x2_split(acc[0], &a0, &a1);
            f32x2_split(acc[1], &b0, &b1);
            sum = (a0 + b0) + (a1 + b1);
          }
          l = l * alpha + sum;
          tmem_store_64(tS, pk);
          if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
            for (int c = 0; c < kD / 32; ++c) {
              uint32_t u[32];
              tmem_load_32(tO + c * 32, u);
#pragma unroll
              for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
              tmem_store_32(tO + c * 32, u);
            }
          }
          tmem_store_wait();
          tc_fence_before_sync();
          mbar_arrive(&ctl->p_full[x]);
        }
      }
      if (ok && n > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl->o_full[x], items & 1, p.status, abort));
        ++items;
      }
      if (!ok) break;
      tc_fence_after_sync();
      // ------------------------------------------------------- epilogue
      const bool empty = !(l > 0.f);
      const float inv_l = empty ? 0.f : 1.f / l;
      const int lrow = local_row(p.qmap, row);
      const size_t ob = ((size_t)lrow * p.hq + head) * kD;
      // half of a split item: its partial (O / l, lse) goes to its fp32 slot
      const bool to_part = it.part >= 0;
      const size_t pslot = ((size_t)it.part * 2 + x) * 128 + r;
      const bool store = valid && (to_part ? index_ok(pslot, (long long)p.num_parts * 256, p.status,
                                                      kSiteFwdPart)
                                           : index_ok(lrow, p.q_rows, p.status, kSiteFwdOut) &&
                                                 index_ok(head, p.hq, p.status, kSiteHead));
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t u[32];
        if (n > 0) {
          tmem_load_32(tO + c * 32, u);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = 0u;
        }
        if (store) {
          if (to_part || p.out_fp32) {
            float* base = to_part ? p.part_o + pslot * kD : static_cast<float*>(p.out) + ob;
            float4* dst = reinterpret_cast<float4*>(base + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(u[4 * i]) * inv_l,
                                   __uint_as_float(u[4 * i + 1]) * inv_l,
                                   __uint_as_float(u[4 * i + 2]) * inv_l,
                                   __uint_as_float(u[4 * i + 3]) * inv_l);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + ob + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pack_bf16x2(__uint_as_float(u[8 * i]) * inv_l,
                                              __uint_as_float(u[8 * i + 1]) * inv_l),
                                  pack_bf16x2(__uint_as_float(u[8 * i + 2]) * inv_l,
                                              __uint_as_float(u[8 * i + 3]) * inv_l),
                                  pack_bf16x2(__uint_as_float(u[8 * i + 4]) * inv_l,
                                              __uint_as_float(u[8 * i + 5]) * inv_l),
                                  pack_bf16x2(__uint_as_float(u[8 * i + 6]) * inv_l,
                                              __uint_as_float(u[8 * i + 7]) * inv_l));
          }
        }
      }
      if (store) {
        const float L = empty ? -INFINITY : (m2 + log2f(l)) * 0.69314718055994530942f;
        if (to_part)
          p.part_lse[pslot] = L;
        else
          p.lse[(size_t)head * p.lse_stride + lrow] = L;
      }
      // the epilogue's TMEM reads precede the next item's first P (and with
      // it the PV MMA that overwrites O)
      tc_fence_before_sync();
    }
    if (!ok) *abort = 1;
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

namespace {

template <int kD>
cudaError_t launch_fwd_tc_bf16_d(const FwdParams& p, const CUtensorMap& map_q,
                                 const CUtensorMap& map_k, const CUtensorMap& map_v,
                                 cudaStream_t stream) {
  static bool configured[64] = {};
  constexpr int smem = FwdCfg<kD>::kSmemBytes;
  cudaError_t e = ensure_smem_limit(fwd_tc_bf16_kernel<kD>, smem, configured);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (shared memory and TMEM allow no more), each
  // claiming items from the work counter; without one, one item per CTA
  const int grid = p.work_counter ? p.num_ctas : p.num_items;
  if (grid == 0) return cudaSuccess;
  TraceScope trace_scope(stream, "fwd_tc_bf16_kernel");
  fwd_tc_bf16_kernel<kD><<<grid, kThreads, smem, stream>>>(map_q, map_k, map_v, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc_bf16(const FwdParams& p, const CUtensorMap& map_q,
                               const CUtensorMap& map_k, const CUtensorMap& map_v,
                               cudaStream_t stream) {
  if (p.num_items == 0) return cudaSuccess;
  if (p.D == 128) return launch_fwd_tc_bf16_d<128>(p, map_q, map_k, map_v, stream);
  if (p.D == 64) return launch_fwd_tc_bf16_d<64>(p, map_q, map_k, map_v, stream);
  return cudaErrorInvalidValue;
}

}  // namespace ra
