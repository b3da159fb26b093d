// bf16 ring-attention backward on the sm_103a tensor cores (tcgen05 + TMEM).
//
// With P_ij = exp(scale q_i.k_j - lse_i), dP_ij = dO_i . v_j and
// D_i = dO_i . O_i (preprocess kernel):
//   dS_ij = P_ij (dP_ij - D_i),
//   dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j.
// The sums over the ring are split by output, so no output is accumulated
// with atomics and the result does not depend on scheduling:
//
//   bwd_dkdv_kernel  one CTA per 128-key tile of one key/value head.  It walks
//     the query tiles that see the keys -- those of the ring steps: at step s
//     the keys of rank src sit on rank (src + s) mod P -- in the order of its
//     plan's segments (the whole-GPU plan goes from the end of the sequence
//     down, for L2 reuse across CTAs) and, for GQA, every query head of the
//     group, accumulating dK and dV in TMEM (so they come out summed over the
//     group).  Each query tile is split into two 64-row halves handled
//     by two softmax warpgroups, so one half's elementwise work overlaps the
//     other half's MMAs:
//       S^T  = K Q_h^T        (M = 128 keys, N = 64 queries, K = D)
//       dP^T = V dO_h^T
//       dV  += P^T dO_h       (TS: P^T from TMEM, dO MN-major)
//       dK  += dS^T Q_h       (TS: dS^T from TMEM, Q MN-major)
//     TMEM: S^T_a 0-63, dP^T_a 64-127, S^T_b 128-191, dP^T_b 192-255,
//     dV 256-383, dK 384-511; P^T and dS^T (bf16, two per column) overwrite
//     the first 32 columns of their S^T / dP^T block.
//     The tensor cores' fp32 accumulation loses a little toward zero at
//     every step, so a long walk moves dV and dK to fp32 memory every
//     flush_pairs (query tile, head) pairs and restarts them; the epilogue
//     adds the flushed sums.
//
//   bwd_dq_kernel  one CTA per 128-row query tile (the forward plan's tiles),
//     walking its key ranges in ring order, one 128-key tile at a time:
//       S  = Q K_j^T,  dP = dO V_j^T   (M = 128 queries, N = 128 keys)
//       dQ += dS K_j                   (TS: dS from TMEM, K MN-major; two
//                                       64-key halves, one per warpgroup)
//     TMEM: S in two buffers 0-127 and 128-255 (key tile j in j % 2), dP
//     256-383, dQ 384-511.
//
// Roles in both kernels (384 threads): warp 0 TMA producer, warp 1 TMEM
// allocation and the single MMA-issuing thread, warps 2-3 (dK/dV only) load
// the per-query-row values (lse, D, visible key range) of each stage, warps 4-7
// and 8-11 the two softmax warpgroups.  Every barrier wait is bounded.
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

constexpr int kTile = 128;
constexpr int kHalfBytes = 128 * 64 * 2;     // one box: 128 rows x 64 columns (a swizzle span)
constexpr int kRowsHalf = 64 * 128;          // byte offset of row 64 in a 64-column box
constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;

constexpr uint32_t kIdescN64 = make_idesc_bf16(128, 64, false, false);    // S-type, K-major B
constexpr uint32_t kIdescN128 = make_idesc_bf16(128, 128, false, false);  // S-type, 128 keys

// Per head dimension D (64 or 128): a 128 x D bf16 tile is D / 64 boxes.
template <int kD>
struct BwdCfg {
  static_assert(kD == 64 || kD == 128, "head dimension");
  static constexpr int kTileBytes = kTile * kD * 2;
  static constexpr uint32_t kIdescMN = make_idesc_bf16(128, kD, false, true);  // X += A_tmem * B(MN)
};

// X[128 x 64] = A[128 x D] * B[64 x D]^T, both K-major; b_smem points at the
// first of B's 64 rows inside a 128-row, 128-byte-swizzled tile.
template <int kD>
__device__ __forceinline__ void mma_rows_x_half(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem) {
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
    mma_bf16_ss(d_tmem, make_sdesc_sw128(a_smem + off, 16, 1024),
                make_sdesc_sw128(b_smem + off, 16, 1024), kIdescN64, kk > 0);
  }
}

// X[128 x D] (+)= A_tmem[128 x 64] * B[64 x D]; B is 64 rows (the K
// dimension) of a 128-row tile whose D values are contiguous (MN-major).
template <int kD>
__device__ __forceinline__ void mma_tmem_x_rows(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem,
                                                bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 64 / 16; ++kk) {
    mma_bf16_ts(d_tmem, a_tmem + kk * 8, make_sdesc_sw128(b_smem + kk * 2048, kHalfBytes, 1024),
                BwdCfg<kD>::kIdescMN, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// A 128-row tile of head `head` from row `row`: D / 64 boxes of 64 columns,
// with an L2 eviction policy (l2_evict_last_policy for tiles other CTAs read
// again, l2_evict_first_policy for tiles read once).
template <int kD>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                          int head, int row, uint64_t policy) {
#pragma unroll
  for (int hf = 0; hf < kD / 64; ++hf)
    tma_load_3d_hint(dst + hf * kHalfBytes, map, bar, hf * 64, head, row, policy);
}

// Stores 32 fp32 values (times `mul`) as fp32 at dst (16-byte aligned).
__device__ __forceinline__ void store_f32x32(float* dst, const uint32_t (&u)[32], float mul) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    d[i] = make_float4(__uint_as_float(u[4 * i]) * mul, __uint_as_float(u[4 * i + 1]) * mul,
                       __uint_as_float(u[4 * i + 2]) * mul, __uint_as_float(u[4 * i + 3]) * mul);
}

// Adds 32 fp32 values (times `mul`) into fp32 dst (16-byte aligned); each
// element has one writer per launch, so no atomics are needed.
__device__ __forceinline__ void add_f32x32(float* dst, const uint32_t (&u)[32], float mul) {
  float4* d = reinterpret_cast<float4*>(dst);
  float4 old[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) old[i] = d[i];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    d[i] = make_float4(old[i].x + __uint_as_float(u[4 * i]) * mul,
                       old[i].y + __uint_as_float(u[4 * i + 1]) * mul,
                       old[i].z + __uint_as_float(u[4 * i + 2]) * mul,
                       old[i].w + __uint_as_float(u[4 * i + 3]) * mul);
}

// Stores 32 fp32 values (times `mul`) as bf16 at dst (16-byte aligned).
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const uint32_t (&u)[32], float mul) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    d[i] = make_uint4(pack_bf16x2(__uint_as_float(u[8 * i]) * mul, __uint_as_float(u[8 * i + 1]) * mul),
                      pack_bf16x2(__uint_as_float(u[8 * i + 2]) * mul, __uint_as_float(u[8 * i + 3]) * mul),
                      pack_bf16x2(__uint_as_float(u[8 * i + 4]) * mul, __uint_as_float(u[8 * i + 5]) * mul),
                      pack_bf16x2(__uint_as_float(u[8 * i + 6]) * mul, __uint_as_float(u[8 * i + 7]) * mul));
}

// Stores acc + 32 fp32 values (times `mul`) as bf16 at dst; acc holds the
// earlier partial sums of the same 32 outputs (fp32, 16-byte aligned).
__device__ __forceinline__ void store_bf16x32_plus(__nv_bfloat16* dst, const float* acc,
                                                   const uint32_t (&u)[32], float mul) {
  const float4* a = reinterpret_cast<const float4*>(acc);
  float v[32];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 t = a[i];
    v[4 * i] = t.x + __uint_as_float(u[4 * i]) * mul;
    v[4 * i + 1] = t.y + __uint_as_float(u[4 * i + 1]) * mul;
    v[4 * i + 2] = t.z + __uint_as_float(u[4 * i + 2]) * mul;
    v[4 * i + 3] = t.w + __uint_as_float(u[4 * i + 3]) * mul;
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    d[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                      pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
}

// Elementwise core of the backward for 32 score columns of one TMEM row:
//   P = 2^(S scale log2(e) - lse log2(e)),  dS = P (dP - D),
// two columns per paired fp32 instruction, with the columns the mask hides
// forced to P = 0 by an exponent of -inf (2^-inf = +0): a select, never a
// branch around the exponential.  kMasked is false for tiles every column of
// which is visible.  The per-column statistics come from `stat` (dK/dV: one
// query per column, stored per column pair as (-lse log2 e, -lse log2 e,
// -D, -D) and read with one 16-byte load) and `range` (its visible keys), or
// are the thread's own (dQ: one query per row, stat == nullptr).
template <bool kMasked, bool kWantP>
__device__ __forceinline__ void bwd_elementwise32(const uint32_t (&us)[32], const uint32_t (&ud)[32],
                                                  const float4* stat, const int2* range,
                                                  float lse2, float Dv, int key, int key0, int a,
                                                  int b, float sl2, uint32_t (&pp)[16],
                                                  uint32_t (&pd)[16]) {
  const uint64_t sl2x2 = f32x2(sl2, sl2);
  const uint64_t own_nl2 = f32x2(-lse2, -lse2), own_nd = f32x2(-Dv, -Dv);
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    uint64_t nl2 = own_nl2, nd = own_nd;
    if (stat != nullptr) {
      const float4 st = stat[c / 2];
      nl2 = f32x2(st.x, st.y);
      nd = f32x2(st.z, st.w);
    }
    float x[2];
    f32x2_split(ffma2(f32x2(__uint_as_float(us[c]), __uint_as_float(us[c + 1])), sl2x2, nl2),
                &x[0], &x[1]);
    if (kMasked) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        bool vis;
        if (stat != nullptr) {  // fixed key row, one query per column
          const int2 rg = range[c + e];
          vis = key >= rg.x && key < rg.y;
        } else {                // fixed query row, one key per column
          vis = key0 + c + e >= a && key0 + c + e < b;
        }
        x[e] = vis ? x[e] : -INFINITY;
      }
    }
    const float p0 = fast_exp2(x[0]), p1 = fast_exp2(x[1]);
    const uint64_t pv = f32x2(p0, p1);
    const uint64_t t = fadd2(f32x2(__uint_as_float(ud[c]), __uint_as_float(ud[c + 1])), nd);
    float d0, d1;
    f32x2_split(fmul2(pv, t), &d0, &d1);
    if (kWantP) pp[c / 2] = pack_bf16x2(p0, p1);
    pd[c / 2] = pack_bf16x2(d0, d1);
  }
}

// ============================================================== dK / dV

constexpr int kMaxKvStages = 4;
// per stage: (-lse log2 e, -D) of the 128 query rows, interleaved by column
// pair | their visible key ranges | 2 flags
constexpr int kInfoBytes = 128 * sizeof(float2) + 128 * sizeof(int2) + 16;
constexpr int kInfoStride = (kInfoBytes + 127) / 128 * 128;

template <int kD>
struct KvCfg {
  static constexpr int kTileBytes = BwdCfg<kD>::kTileBytes;
  static constexpr int kKvStages = kD == 128 ? 2 : 4;         // Q/dO stages
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffStage = 2 * kTileBytes;             // per stage: Q, dO
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kOffInfo = kOffStage + kKvStages * kStageBytes;  // per stage: row values
  static constexpr int kOffCtlKV = kOffInfo + kKvStages * kInfoStride;
  static constexpr int kSmemKV = kOffCtlKV + 256 + 1024;
  static_assert(kKvStages <= kMaxKvStages, "stages");
  static_assert(kSmemKV <= 232448, "dynamic shared memory of one CTA");
};

struct CtlKV {
  uint64_t kv_full;
  uint64_t q_full[kMaxKvStages];
  uint64_t info_full[kMaxKvStages];
  uint64_t stage_empty[kMaxKvStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t acc_full;   // dV, dK complete: at each flush and at the end
  uint64_t acc_empty;  // a flush has read dV, dK out of TMEM
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(CtlKV) <= 256, "control block");

template <int kD>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                    const BwdParams p) {
  using Cfg = KvCfg<kD>;
  constexpr int kTileBytes = Cfg::kTileBytes;
  constexpr int kKvStages = Cfg::kKvStages;
  constexpr int kOffK = Cfg::kOffK, kOffV = Cfg::kOffV, kOffStage = Cfg::kOffStage;
  constexpr int kStageBytes = Cfg::kStageBytes, kOffInfo = Cfg::kOffInfo;
  constexpr int kOffCtlKV = Cfg::kOffCtlKV;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  CtlKV* ctl = reinterpret_cast<CtlKV*>(smem + kOffCtlKV);
  volatile int* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BwdItem it = p.bitems[checked(blockIdx.x, p.num_bitems, p.status, kSiteBwdItem)];
  const int g = it.kv_head;
  const int G = p.group;
  const int kend = it.k0 + it.klen;

  int n = 0;  // (query tile, head) pairs
  for (int si = 0; si < it.seg_count; ++si) {
    const BwdSegment sg = p.bsegs[checked(it.seg_begin + si, p.num_bsegs, p.status, kSiteBwdSeg)];
    n += (sg.q1 - sg.q0 + kTile - 1) / kTile * G;
  }

  if (threadIdx.x == 0) {
    mbar_init(&ctl->kv_full, 1);
    for (int s = 0; s < kKvStages; ++s) {
      mbar_init(&ctl->q_full[s], 1);
      mbar_init(&ctl->info_full[s], 64);
      mbar_init(&ctl->stage_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&ctl->s_full[x], 1);
      mbar_init(&ctl->p_full[x], 128);
    }
    mbar_init(&ctl->acc_full, 1);
    mbar_init(&ctl->acc_empty, 256);
    mbar_init(&ctl->mma_done, 1);
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

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer
    if (elect_one_sync() && n > 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_do);
      mbar_arrive_expect_tx(&ctl->kv_full, 2 * kTileBytes);
      const int k0l = local_row(p.kmap, it.k0);
      index_ok(k0l, p.k_rows, p.status, kSiteBwdKvRow);
      index_ok(g, p.hkv, p.status, kSiteHead);
      const uint64_t once = l2_evict_first_policy(), again = l2_evict_last_policy();
      load_tile<kD>(smem + kOffK, &map_k, &ctl->kv_full, g, k0l, once);
      load_tile<kD>(smem + kOffV, &map_v, &ctl->kv_full, g, k0l, once);
      int li = 0;
      bool ok = true;
      for (int si = 0; si < it.seg_count && ok; ++si) {
        const BwdSegment sg =
            p.bsegs[checked(it.seg_begin + si, p.num_bsegs, p.status, kSiteBwdSeg)];
        for (int i0 = sg.q0; i0 < sg.q1 && ok; i0 += kTile) {
          for (int h = g * G; h < (g + 1) * G; ++h, ++li) {
            const int slot = li % kKvStages;
            if (li >= kKvStages &&
                !mbar_wait(&ctl->stage_empty[slot], ((li / kKvStages) - 1) & 1, p.status, abort)) {
              ok = false;
              break;
            }
            uint8_t* st = smem + kOffStage + slot * kStageBytes;
            mbar_arrive_expect_tx(&ctl->q_full[slot], 2 * kTileBytes);
            const int i0l = local_row(p.qmap, i0);
            index_ok(i0l, p.q_rows, p.status, kSiteBwdQRow);
            index_ok(h, p.hq, p.status, kSiteHead);
            load_tile<kD>(st, &map_q, &ctl->q_full[slot], h, i0l, again);
            load_tile<kD>(st + kTileBytes, &map_do, &ctl->q_full[slot], h, i0l, again);
          }
        }
      }
      if (!ok) *abort = 1;
      for (int s = 0; s < kKvStages && s < li; ++s) {
        const int last = s + ((li - 1 - s) / kKvStages) * kKvStages;
        mbar_wait(&ctl->q_full[s], (last / kKvStages) & 1, p.status, nullptr);
      }
      mbar_wait(&ctl->kv_full, 0, p.status, nullptr);
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------ per-row values of each stage
    // warp 2 fills rows 0-63, warp 3 rows 64-127; each lane's two rows are
    // loaded together so their global-memory latencies overlap
    const int rbase = (warp - 2) * 64;
    int li = 0;
    bool ok = true;
    for (int si = 0; si < it.seg_count && ok; ++si) {
      const BwdSegment sg =
          p.bsegs[checked(it.seg_begin + si, p.num_bsegs, p.status, kSiteBwdSeg)];
      for (int i0 = sg.q0; i0 < sg.q1 && ok; i0 += kTile) {
        // the document of the stage's first row; rows past its end search again
        int ds0, de0;
        doc_bounds(p.cu, p.num_docs, i0, &ds0, &de0);
        for (int h = g * G; h < (g + 1) * G; ++h, ++li) {
          const int slot = li % kKvStages;
          if (li >= kKvStages) {
            ok = __all_sync(0xffffffffu, mbar_wait(&ctl->stage_empty[slot], ((li / kKvStages) - 1) & 1,
                                                   p.status, abort));
            if (!ok) break;
          }
          uint8_t* info = smem + kOffInfo + slot * kInfoStride;
          float* stat = reinterpret_cast<float*>(info);  // [64 pairs][nl2 a, nl2 b, nd a, nd b]
          int2* range = reinterpret_cast<int2*>(info + 128 * sizeof(float2));
          float lv[2], dv[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int i = i0 + rbase + lane + 32 * k;
            const bool valid = i < sg.q1;
            const size_t at =
                checked((long long)h * p.lse_stride + (valid ? local_row(p.qmap, i) : 0),
                        (long long)p.hq * p.lse_stride, p.status, kSiteBwdRowStat);
            lv[k] = valid ? p.lse[at] : 0.f;
            dv[k] = valid ? p.Dvec[at] : 0.f;
          }
          bool full = true;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int r = rbase + lane + 32 * k;
            const int i = i0 + r;
            float2 st = make_float2(0.f, 0.f);  // (lse log2 e, D)
            int2 rg = make_int2(0, 0);  // rows outside the segment see no key
            if (i < sg.q1) {
              int ds = ds0, de = de0;
              if (i >= de0) doc_bounds(p.cu, p.num_docs, i, &ds, &de);
              st = make_float2(lv[k] * kLog2e, dv[k]);
              rg = make_int2(ds, p.causal ? i + 1 : de);
            }
            // the tile needs no mask if every row is in the segment and sees
            // every key of the tile
            full = full && (i < sg.q1) && rg.x <= it.k0 && rg.y >= kend;
            stat[(r >> 1) * 4 + (r & 1)] = -st.x;
            stat[(r >> 1) * 4 + 2 + (r & 1)] = -st.y;
            range[r] = rg;
          }
          full = __all_sync(0xffffffffu, full);
          if (lane == 0)
            reinterpret_cast<int*>(info + 128 * (sizeof(float2) + sizeof(int2)))[warp - 2] =
                full ? 1 : 0;
          __syncwarp();
          mbar_arrive(&ctl->info_full[slot]);
        }
      }
    }
    if (!ok) *abort = 1;
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA
    if (elect_one_sync() && n > 0) {
      const uint32_t sK = smem_u32(smem + kOffK), sV = smem_u32(smem + kOffV);
      auto sQ = [&](int li) { return smem_u32(smem + kOffStage + (li % kKvStages) * kStageBytes); };
      const uint32_t tS[2] = {tmem + 0, tmem + 128};
      const uint32_t tdP[2] = {tmem + 64, tmem + 192};
      const uint32_t tdV = tmem + 256, tdK = tmem + 384;
      auto q_ready = [&](int li) {
        return mbar_wait(&ctl->q_full[li % kKvStages], (li / kKvStages) & 1, p.status, abort);
      };
      // S^T and dP^T of half x of pair li
      auto issue_s = [&](int li, int x) {
        const uint32_t q = sQ(li) + x * kRowsHalf, dO = sQ(li) + kTileBytes + x * kRowsHalf;
        mma_rows_x_half<kD>(tS[x], sK, q);
        mma_rows_x_half<kD>(tdP[x], sV, dO);
        mma_commit(&ctl->s_full[x]);
      };
      auto issue_acc = [&](int li, int x, bool accumulate) {
        const uint32_t q = sQ(li) + x * kRowsHalf, dO = sQ(li) + kTileBytes + x * kRowsHalf;
        mma_tmem_x_rows<kD>(tdV, tS[x], dO, accumulate);
        mma_tmem_x_rows<kD>(tdK, tdP[x], q, accumulate);
      };
      bool ok = mbar_wait(&ctl->kv_full, 0, p.status, abort) && q_ready(0);
      if (ok) {
        tc_fence_after_sync();
        issue_s(0, 0);
        issue_s(0, 1);
      }
      int flushes = 0;  // dV, dK handed to the flush so far
      for (int j = 0; j < n && ok; ++j) {
        const bool more = j + 1 < n;
        // the first pair after a flush starts dV, dK afresh once the flush
        // has read them
        const bool fresh = j > 0 && p.flush_pairs > 0 && j % p.flush_pairs == 0;
        if (!(ok = mbar_wait(&ctl->p_full[0], j & 1, p.status, abort))) break;
        if (fresh && !(ok = mbar_wait(&ctl->acc_empty, (flushes - 1) & 1, p.status, abort))) break;
        tc_fence_after_sync();
        issue_acc(j, 0, j > 0 && !fresh);
        if (more) {
          if (!(ok = q_ready(j + 1))) break;
          tc_fence_after_sync();
          issue_s(j + 1, 0);
        }
        if (!(ok = mbar_wait(&ctl->p_full[1], j & 1, p.status, abort))) break;
        tc_fence_after_sync();
        issue_acc(j, 1, true);
        mma_commit(&ctl->stage_empty[j % kKvStages]);
        if (more && p.flush_pairs > 0 && (j + 1) % p.flush_pairs == 0) {
          mma_commit(&ctl->acc_full);
          ++flushes;
        }
        if (more) issue_s(j + 1, 1);
      }
      if (ok) mma_commit(&ctl->acc_full);
      if (!ok) *abort = 1;
      mma_commit(&ctl->mma_done);
      mbar_wait(&ctl->mma_done, 0, p.status, nullptr);
    }
  } else if (warp >= 4) {
    // --------------------------------------------------- softmax halves
    const int x = (warp - 4) >> 2;  // query-row half of each stage
    const int quarter = warp & 3;
    const int kr = quarter * 32 + lane;  // key row of the tile (TMEM lane)
    const int j = it.k0 + kr;            // global key index
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + x * 128;
    const uint32_t tdP = tS + 64;
    const float sl2 = p.scale_log2;
    // half 0 writes dV, half 1 writes dK (times the softmax scale), at the
    // flushes and at the end
    const uint32_t tAcc = tmem + lane_off + (x == 0 ? 256 : 384);
    const int jl = local_row(p.kmap, j);
    const bool store = kr < it.klen && index_ok(jl, p.k_rows, p.status, kSiteBwdDkDv) &&
                       index_ok(g, p.hkv, p.status, kSiteHead);
    const size_t off = ((size_t)jl * p.hkv + g) * kD;
    void* dst = x == 0 ? p.dv : p.dk;
    float* const acc_base = x == 0 ? p.dv_acc : p.dk_acc;  // fp32 sums of the flushes, or null
    const float mul = x == 0 ? 1.f : p.scale;
    int flushes = 0;
    bool ok = true;
    for (int jj = 0; jj < n; ++jj) {
      const int slot = jj % kKvStages;
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->info_full[slot], (jj / kKvStages) & 1, p.status, abort));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&ctl->s_full[x], jj & 1, p.status, abort));
      if (!ok) break;
      tc_fence_after_sync();
      const uint8_t* info = smem + kOffInfo + slot * kInfoStride;
      const int* flags = reinterpret_cast<const int*>(info + 128 * (sizeof(float2) + sizeof(int2)));
      const bool full = flags[0] != 0 && flags[1] != 0;
      const float4* hstat = reinterpret_cast<const float4*>(info) + x * 32;
      const int2* hrange = reinterpret_cast<const int2*>(info + 128 * sizeof(float2)) + x * 64;
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t us[32], ud[32];
        tmem_load_2x32(tS + c2 * 32, us, tdP + c2 * 32, ud);
        uint32_t pp[16], pd[16];
        if (full)
          bwd_elementwise32<false, true>(us, ud, hstat + c2 * 16, hrange + c2 * 32, 0.f, 0.f, j,
                                         0, 0, 0, sl2, pp, pd);
        else
          bwd_elementwise32<true, true>(us, ud, hstat + c2 * 16, hrange + c2 * 32, 0.f, 0.f, j,
                                        0, 0, 0, sl2, pp, pd);
        tmem_store_16(tS + c2 * 16, pp);
        tmem_store_16(tdP + c2 * 16, pd);
      }
      tmem_store_wait();
      tc_fence_before_sync();
      mbar_arrive(&ctl->p_full[x]);
      // flush: after every flush_pairs pairs (the last pair excepted) dV and
      // dK leave TMEM for fp32 memory, and the MMAs start them afresh, so
      // that no accumulation in TMEM runs longer than flush_pairs pairs
      if (p.flush_pairs > 0 && jj + 1 < n && (jj + 1) % p.flush_pairs == 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl->acc_full, flushes & 1, p.status, abort));
        if (!ok) break;
        tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t u[32];
          tmem_load_32(tAcc + c * 32, u);
          if (store) {
            if (flushes == 0 && !p.accumulate)
              store_f32x32(acc_base + off + c * 32, u, mul);
            else
              add_f32x32(acc_base + off + c * 32, u, mul);
          }
        }
        tc_fence_before_sync();
        mbar_arrive(&ctl->acc_empty);
        ++flushes;
      }
    }
    if (!ok) *abort = 1;
    if (ok && n > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->acc_full, flushes & 1, p.status, abort));
    tc_fence_after_sync();
    // epilogue: TMEM plus the flushed partial sums
#pragma unroll
    for (int c = 0; c < kD / 32; ++c) {
      uint32_t u[32];
      if (ok && n > 0) {
        tmem_load_32(tAcc + c * 32, u);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) u[i] = 0u;
      }
      if (ok && store) {
        if (flushes > 0 && !p.accumulate && !p.grad_fp32)
          store_bf16x32_plus(static_cast<__nv_bfloat16*>(dst) + off + c * 32,
                             acc_base + off + c * 32, u, mul);
        else if (p.accumulate || flushes > 0)
          add_f32x32(static_cast<float*>(dst) + off + c * 32, u, mul);
        else if (p.grad_fp32)
          store_f32x32(static_cast<float*>(dst) + off + c * 32, u, mul);
        else
          store_bf16x32(static_cast<__nv_bfloat16*>(dst) + off + c * 32, u, mul);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================== dQ
//
// One CTA per 128-row query tile, key tiles of 128 in ring order.  Q and dO
// stay in shared memory; K and V stream through separate rings (K: 3 slots,
// since K(j) is read by S(j) and again by dQ(j); V: 2 slots).  Tensor memory:
// S in two buffers (S(j) in buffer j % 2), dP in one, dQ in one:
//   cols 0-127 S_0 | 128-255 S_1 | 256-383 dP | 384-511 dQ.
// The MMA thread issues, per key tile j,
//   dP(j+1) = dO V_{j+1}^T   once both warpgroups have read dP(j),
//   dQ += dS(j) K_j          in two 64-key halves, as each warpgroup stores
//                            its half of dS(j) (bf16, over its half of S(j)),
//   S(j+2) = Q K_{j+2}^T     into the buffer dS(j) has just been read from,
// so the elementwise work of tile j+1 is ready to start the moment tile j's
// is done.  Warpgroup w (warps 4-7: w = 0, 8-11: w = 1) handles keys
// [64 w, 64 w + 64) of every tile, one query row per thread.  Because dP(j+1)
// is released before the MMA thread waits for dS(j), a warpgroup can finish
// tile j+1 before that wait: dS(j) therefore signals on one of two barriers
// per warpgroup (by j % 2), so no barrier runs two phases ahead of its waiter.

constexpr int kMaxKSlots = 4, kMaxVSlots = 3;

template <int kD>
struct QCfg {
  static constexpr int kTileBytes = BwdCfg<kD>::kTileBytes;
  static constexpr int kKSlots = kD == 128 ? 3 : 4;
  static constexpr int kVSlots = kD == 128 ? 2 : 3;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kTileBytes;
  static constexpr int kOffKq = 2 * kTileBytes;
  static constexpr int kOffVq = kOffKq + kKSlots * kTileBytes;
  static constexpr int kOffCtlQ = kOffVq + kVSlots * kTileBytes;
  static constexpr int kSmemQ = kOffCtlQ + 256 + 1024;
  static_assert(kKSlots <= kMaxKSlots && kVSlots <= kMaxVSlots, "slots");
  static_assert(kSmemQ <= 232448, "dynamic shared memory of one CTA");
};

struct CtlQ {
  uint64_t qd_full;
  uint64_t k_full[kMaxKSlots];
  uint64_t k_empty[kMaxKSlots];
  uint64_t v_full[kMaxVSlots];
  uint64_t v_empty[kMaxVSlots];
  uint64_t s_full[2];   // S(j) in buffer j % 2
  uint64_t dp_full;     // dP(j)
  uint64_t dp_free;     // every softmax thread has read dP(j)
  uint64_t ds_full[2][2];  // [w][j % 2]: warpgroup w stored its half of dS(j)
  uint64_t acc_full;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(CtlQ) <= 256, "control block");

// X[128 x 128] = A[128 x D] * B[128 x D]^T, both K-major, 128-row tiles.
template <int kD>
__device__ __forceinline__ void mma_rows_x_rows(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem) {
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
    mma_bf16_ss(d_tmem, make_sdesc_sw128(a_smem + off, 16, 1024),
                make_sdesc_sw128(b_smem + off, 16, 1024), kIdescN128, kk > 0);
  }
}

template <int kD>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                  const BwdParams p) {
  using Cfg = QCfg<kD>;
  constexpr int kTileBytes = Cfg::kTileBytes;
  constexpr int kKSlots = Cfg::kKSlots, kVSlots = Cfg::kVSlots;
  constexpr int kOffQ = Cfg::kOffQ, kOffDO = Cfg::kOffDO, kOffKq = Cfg::kOffKq;
  constexpr int kOffVq = Cfg::kOffVq, kOffCtlQ = Cfg::kOffCtlQ;
  const PlanItem it = p.items[checked(blockIdx.x >> 1, p.num_items, p.status, kSiteBwdItem)];
  const bool second = (blockIdx.x & 1) != 0;  // which of the item's two query tiles
  const int qlen = second ? it.qlen[1] : it.qlen[0];
  if (qlen == 0) return;  // whole CTA: this item has one query tile
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  CtlQ* ctl = reinterpret_cast<CtlQ*>(smem + kOffCtlQ);
  volatile int* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = second ? it.head[1] : it.head[0];
  const int g = head / p.group;
  const int q0 = second ? it.q0[1] : it.q0[0];

  int n = 0;  // key tiles
  for (int si = 0; si < it.seg_count; ++si) {
    const PlanSegment sg = p.segs[checked(it.seg_begin + si, p.num_segs, p.status, kSiteBwdSeg)];
    n += (sg.k1 - sg.k0 + kTile - 1) / kTile;
  }

  if (threadIdx.x == 0) {
    mbar_init(&ctl->qd_full, 1);
    for (int s = 0; s < kKSlots; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 1);
    }
    for (int s = 0; s < kVSlots; ++s) {
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&ctl->s_full[x], 1);
      mbar_init(&ctl->ds_full[x][0], 128);
      mbar_init(&ctl->ds_full[x][1], 128);
    }
    mbar_init(&ctl->dp_full, 1);
    mbar_init(&ctl->dp_free, 256);
    mbar_init(&ctl->acc_full, 1);
    mbar_init(&ctl->mma_done, 1);
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

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer
    if (elect_one_sync() && n > 0) {
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_v);
      mbar_arrive_expect_tx(&ctl->qd_full, 2 * kTileBytes);
      const int q0l = local_row(p.qmap, q0);
      index_ok(q0l, p.q_rows, p.status, kSiteBwdQRow);
      index_ok(head, p.hq, p.status, kSiteHead);
      index_ok(g, p.hkv, p.status, kSiteHead);
      const uint64_t once = l2_evict_first_policy(), again = l2_evict_last_policy();
      load_tile<kD>(smem + kOffQ, &map_q, &ctl->qd_full, head, q0l, once);
      load_tile<kD>(smem + kOffDO, &map_do, &ctl->qd_full, head, q0l, once);
      int j = 0, nk = 0, nv = 0;  // tiles visited, K and V loads issued
      bool ok = true;
      for (int si = 0; si < it.seg_count && ok; ++si) {
        const PlanSegment sg =
            p.segs[checked(it.seg_begin + si, p.num_segs, p.status, kSiteBwdSeg)];
        for (int kt = sg.k0; kt < sg.k1; kt += kTile, ++j) {
          const int ks = j % kKSlots, vs = j % kVSlots;
          index_ok(local_row(p.kmap, kt), p.k_rows, p.status, kSiteBwdKvRow);
          if (j >= kKSlots &&
              !mbar_wait(&ctl->k_empty[ks], ((j / kKSlots) - 1) & 1, p.status, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&ctl->k_full[ks], kTileBytes);
          load_tile<kD>(smem + kOffKq + ks * kTileBytes, &map_k, &ctl->k_full[ks], g,
                        local_row(p.kmap, kt), again);
          ++nk;
          if (j >= kVSlots &&
              !mbar_wait(&ctl->v_empty[vs], ((j / kVSlots) - 1) & 1, p.status, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&ctl->v_full[vs], kTileBytes);
          load_tile<kD>(smem + kOffVq + vs * kTileBytes, &map_v, &ctl->v_full[vs], g,
                        local_row(p.kmap, kt), again);
          ++nv;
        }
      }
      if (!ok) *abort = 1;
      // let every copy this thread started land before the CTA can exit
      for (int s = 0; s < kKSlots && s < nk; ++s) {
        const int last = s + ((nk - 1 - s) / kKSlots) * kKSlots;
        mbar_wait(&ctl->k_full[s], (last / kKSlots) & 1, p.status, nullptr);
      }
      for (int s = 0; s < kVSlots && s < nv; ++s) {
        const int last = s + ((nv - 1 - s) / kVSlots) * kVSlots;
        mbar_wait(&ctl->v_full[s], (last / kVSlots) & 1, p.status, nullptr);
      }
      mbar_wait(&ctl->qd_full, 0, p.status, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA
    if (elect_one_sync() && n > 0) {
      const uint32_t sQ = smem_u32(smem + kOffQ), sdO = smem_u32(smem + kOffDO);
      auto sK = [&](int j) { return smem_u32(smem + kOffKq + (j % kKSlots) * kTileBytes); };
      auto sV = [&](int j) { return smem_u32(smem + kOffVq + (j % kVSlots) * kTileBytes); };
      auto tS = [&](int j) { return tmem + static_cast<uint32_t>(j & 1) * 128u; };
      const uint32_t tdP = tmem + 256, tdQ = tmem + 384;
      auto k_ready = [&](int j) {
        return mbar_wait(&ctl->k_full[j % kKSlots], (j / kKSlots) & 1, p.status, abort);
      };
      auto v_ready = [&](int j) {
        return mbar_wait(&ctl->v_full[j % kVSlots], (j / kVSlots) & 1, p.status, abort);
      };
      auto issue_s = [&](int j) {  // S(j) into buffer j % 2
        mma_rows_x_rows<kD>(tS(j), sQ, sK(j));
        mma_commit(&ctl->s_full[j & 1]);
      };
      auto issue_dp = [&](int j) {  // dP(j); V(j) is then no longer needed
        mma_rows_x_rows<kD>(tdP, sdO, sV(j));
        mma_commit(&ctl->dp_full);
        mma_commit(&ctl->v_empty[j % kVSlots]);
      };
      bool ok = mbar_wait(&ctl->qd_full, 0, p.status, abort) && k_ready(0);
      if (ok) {
        tc_fence_after_sync();
        issue_s(0);
        ok = v_ready(0);
      }
      if (ok) {
        tc_fence_after_sync();
        issue_dp(0);
        if (n > 1 && (ok = k_ready(1))) {
          tc_fence_after_sync();
          issue_s(1);
        }
      }
      for (int j = 0; j < n && ok; ++j) {
        if (j + 1 < n) {
          if (!(ok = mbar_wait(&ctl->dp_free, j & 1, p.status, abort) && v_ready(j + 1))) break;
          tc_fence_after_sync();
          issue_dp(j + 1);
        }
        for (int w = 0; w < 2; ++w) {
          if (!(ok = mbar_wait(&ctl->ds_full[w][j & 1], (j >> 1) & 1, p.status, abort))) break;
          tc_fence_after_sync();
          // dQ += dS(j)[:, 64 w : 64 w + 64] K_j[64 w : 64 w + 64, :]
          mma_tmem_x_rows<kD>(tdQ, tS(j) + 64 * w, sK(j) + w * kRowsHalf, j > 0 || w > 0);
        }
        if (!ok) break;
        mma_commit(&ctl->k_empty[j % kKSlots]);
        if (j + 2 < n) {
          if (!(ok = k_ready(j + 2))) break;
          tc_fence_after_sync();
          issue_s(j + 2);
        }
      }
      if (ok) mma_commit(&ctl->acc_full);
      if (!ok) *abort = 1;
      // every MMA this thread issued has completed before TMEM is released
      mma_commit(&ctl->mma_done);
      mbar_wait(&ctl->mma_done, 0, p.status, nullptr);
    }
  } else if (warp >= 4) {
    // -------------------------------------------- elementwise, key half w
    const int w = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int row = q0 + r;
    const bool valid = r < qlen;
    int lo = 0, hi = 0;
    float lse2 = 0.f, Dv = 0.f;
    if (valid) {
      int ds, de;
      doc_bounds(p.cu, p.num_docs, row, &ds, &de);
      lo = ds;
      hi = p.causal ? row + 1 : de;
      const size_t at = checked((long long)head * p.lse_stride + local_row(p.qmap, row),
                                (long long)p.hq * p.lse_stride, p.status, kSiteBwdRowStat);
      lse2 = p.lse[at] * kLog2e;
      Dv = p.Dvec[at];
    }
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tdP = tmem + lane_off + 256 + 64 * w;
    const int mlo = second ? it.mask_lo[1] : it.mask_lo[0];
    const int mhi = second ? it.mask_hi[1] : it.mask_hi[0];
    const float sl2 = p.scale_log2;
    bool ok = true;
    int j = 0;
    for (int si = 0; si < it.seg_count && ok; ++si) {
      const PlanSegment sg =
          p.segs[checked(it.seg_begin + si, p.num_segs, p.status, kSiteBwdSeg)];
      const int a = max(lo, sg.k0), b = min(hi, sg.k1);
      const int full_lo = max(sg.k0, mlo), full_hi = min(sg.k1, mhi);
      for (int kt = sg.k0; kt < sg.k1; kt += kTile, ++j) {
        // .sync.aligned TMEM accesses follow: keep the warp's decision uniform
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl->s_full[j & 1], (j >> 1) & 1, p.status, abort));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&ctl->dp_full, j & 1, p.status, abort));
        if (!ok) break;
        tc_fence_after_sync();
        uint32_t ud[64];  // this warpgroup's 64 dP columns, one load
        tmem_load_64(tdP, ud);
        tc_fence_before_sync();
        mbar_arrive(&ctl->dp_free);  // dP(j+1) may now overwrite dP(j)
        const uint32_t tS = tmem + lane_off + (j & 1) * 128 + 64 * w;
        const int kb = kt + 64 * w;  // first key of this half
        const bool full = kb >= full_lo && kb + 64 <= full_hi;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t us[32];
          tmem_load_32(tS + c2 * 32, us);
          uint32_t pp[16], pd[16];  // pp unused: dQ needs dS only
          const uint32_t(&udc)[32] = *reinterpret_cast<const uint32_t(*)[32]>(ud + c2 * 32);
          if (full)
            bwd_elementwise32<false, false>(us, udc, nullptr, nullptr, lse2, Dv, 0, kb + c2 * 32,
                                            a, b, sl2, pp, pd);
          else
            bwd_elementwise32<true, false>(us, udc, nullptr, nullptr, lse2, Dv, 0, kb + c2 * 32,
                                           a, b, sl2, pp, pd);
          // dS over the first half of the columns this warpgroup just read
          tmem_store_16(tS + c2 * 16, pd);
        }
        tmem_store_wait();
        tc_fence_before_sync();
        mbar_arrive(&ctl->ds_full[w][j & 1]);
      }
    }
    if (!ok) *abort = 1;
    if (ok && n > 0) ok = __all_sync(0xffffffffu, mbar_wait(&ctl->acc_full, 0, p.status, abort));
    tc_fence_after_sync();
    // epilogue: warpgroup w writes columns [w D / 2, (w + 1) D / 2) of its row of dQ
    const int lrow = valid ? local_row(p.qmap, row) : 0;
    const bool store = valid && index_ok(lrow, p.q_rows, p.status, kSiteBwdDq) &&
                       index_ok(head, p.hq, p.status, kSiteHead);
    const size_t off = ((size_t)lrow * p.hq + head) * kD + w * (kD / 2);
#pragma unroll
    for (int c = 0; c < kD / 64; ++c) {
      uint32_t u[32];
      if (ok && n > 0) {
        tmem_load_32(tmem + lane_off + 384 + w * (kD / 2) + c * 32, u);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) u[i] = 0u;
      }
      if (ok && store) {
        if (p.accumulate)
          add_f32x32(static_cast<float*>(p.dq) + off + c * 32, u, p.scale);
        else if (p.grad_fp32)
          store_f32x32(static_cast<float*>(p.dq) + off + c * 32, u, p.scale);
        else
          store_bf16x32(static_cast<__nv_bfloat16*>(p.dq) + off + c * 32, u, p.scale);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <int kD>
cudaError_t launch_bwd_tc_bf16_d(const BwdParams& p, const CUtensorMap& map_q,
                                 const CUtensorMap& map_k, const CUtensorMap& map_v,
                                 const CUtensorMap& map_do, cudaStream_t stream) {
  static bool dkdv_configured[64] = {};
  static bool dq_configured[64] = {};
  constexpr int smem_kv = KvCfg<kD>::kSmemKV, smem_q = QCfg<kD>::kSmemQ;
  cudaError_t e0 = ensure_smem_limit(bwd_dkdv_kernel<kD>, smem_kv, dkdv_configured);
  if (e0 == cudaSuccess) e0 = ensure_smem_limit(bwd_dq_kernel<kD>, smem_q, dq_configured);
  if (e0 != cudaSuccess) return e0;
  if (p.num_items > 0) {
    TraceScope trace_scope(stream, "bwd_dq_kernel");
    bwd_dq_kernel<kD><<<2 * p.num_items, kThreads, smem_q, stream>>>(map_q, map_k, map_v, map_do, p);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.num_bitems > 0) {
    TraceScope trace_scope(stream, "bwd_dkdv_kernel");
    bwd_dkdv_kernel<kD><<<p.num_bitems, kThreads, smem_kv, stream>>>(map_q, map_k, map_v, map_do, p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc_bf16(const BwdParams& p, const CUtensorMap& map_q,
                               const CUtensorMap& map_k, const CUtensorMap& map_v,
                               const CUtensorMap& map_do, cudaStream_t stream) {
  if (p.D == 128) return launch_bwd_tc_bf16_d<128>(p, map_q, map_k, map_v, map_do, stream);
  if (p.D == 64) return launch_bwd_tc_bf16_d<64>(p, map_q, map_k, map_v, map_do, stream);
  return cudaErrorInvalidValue;
}

}  // namespace ra
