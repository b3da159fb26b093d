// Chunk scan of the context-parallel Mamba2 selective scan (SSD) on the
// sm_103a tensor cores, for state size N = 128.
//
// Same contract as ssd_chunk_scan_kernel (ssd_cp.cu): CTA (h, r) scans rank
// r's chunk of head h from a zero state and writes y of the chunk, the
// chunk's final state and its carry factor; the state pass and the additive
// correction that follow are unchanged (axolotl "Sequence Parallelism" page,
// "Mamba/SSM Hybrid Models": each rank scans its chunk, passes its final
// state on, and a linear correction accounts for the state it did not start
// from).
//
// The recurrence S <- exp(dt A) S + dt x B^T, y = S C + D x is evaluated a
// block of Q = 128 tokens at a time in its chunked form.  With
// l_t = dt_t A log2(e), P_t its running sum over the block, rc_t the number
// of sample starts (position 0) at or before token t in the block, and S0 the
// state before the block:
//   same(t, j) = (j <= t and rc_j == rc_t)            no sample starts in (j, t]
//   y_t  = [rc_t == 0] 2^P_t (C_t . S0)               the block's incoming state
//        + sum_j same(t, j) 2^(P_t - P_j) dt_j (C_t . B_j) x_j + D x_t
//   S    = [rc_end == 0] 2^P_end S0 + sum_j [rc_j == rc_end] 2^(P_end - P_j) dt_j x_j B_j^T
// as products on the tensor cores, every one with M = 128:
//   [G | Yoff] = C [B | S0]^T  (tokens x (tokens + head dim), over the     TMEM cols 0-191
//                              state: one N = 192 product)
//   Ydia = M X, M = G o mask o dt  (tokens x head dim, over tokens)        TMEM cols 192-255
//   S^T += (v o B)^T X     (state x head dim, over tokens; the fp32 state   TMEM cols 256-319
//                           lives in TMEM across the blocks)
// The scan is checked to fp32-level accuracy (2e-5 relative), which one
// 16-bit product per term cannot reach, so every operand a is split into
// fp16 a_hi + a_lo (a_hi: a rounded to 11 significant bits; a_lo = a - a_hi,
// rounded once) and each product a b is formed as a_hi b_hi + a_hi b_lo +
// a_lo b_hi, accumulated in fp32: the dropped a_lo b_lo and the rounding of
// the lo parts leave about 2^-22 of each product.  fp16 keeps 11 significant
// bits where bf16 keeps 8; the operands here (inputs of order 1, decay
// factors <= 1) sit well inside its range.
//
// C and M, the A operands of the token products, live in TMEM (cols 320-447,
// two fp16 per column), written by the threads with tcgen05.st.  B, x, v o B
// and S0 are in shared memory with the 128-byte swizzle the MMA descriptors
// describe: B's 128 token rows and S0's 64 rows form one K-major operand
// (K = state); B's rows, once scaled by v_j in place, are read as the
// MN-major A operand of the state update; x is the MN-major B operand of both
// token contractions.  The inputs are fp32 in memory: TMA stages a block's
// rows (C in swizzled boxes of its own, B and x in the space of their split
// operands) and the threads split them.
// One CTA per (head, rank), 512 threads; one thread issues the MMAs.  A block
// runs: C, B and x split | [G | Yoff] issued, the next block's C staged and
// the decay scan while it runs | the masked M, the scaling of B by v, the
// state's decay | Ydia, S^T issued | the next block's B and x staged, S0 out,
// y out.  Every barrier wait is bounded.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "device_common.cuh"
#include "launch.h"
#include "sm103_ptx.cuh"
#include "ssd_tc_common.cuh"
#include "trace.h"

namespace ra {

namespace {

using namespace ssd_tc;

constexpr int kQ = 128;       // tokens per block
constexpr int kP = 64;        // head dimension
constexpr int kN = 128;       // state size
constexpr int kThreads = 512;
constexpr float kLog2e = 1.4426950408889634f;

// Each operand is stored as an fp16 hi part followed by its lo part.
constexpr int kPartCB = kQ * kN * 2;  // 128 rows x 128 fp16: two 16 KB swizzle blocks
constexpr int kPartX = kQ * kP * 2;   // 128 token rows x 64 fp16
// B's 128 token rows and S0's 64 head-dim rows share one K-major operand
// (K = state), so that G and Yoff are one product of N = 192: each 64-value
// K block holds 192 rows.
constexpr int kRowsBS = kQ + kP;
constexpr int kBlkBS = kRowsBS * 128;
constexpr int kPartBS = 2 * kBlkBS;
constexpr int kOffC = 0;  // C's fp32 rows, staged (C and M themselves live in TMEM)
constexpr int kOffBS = kOffC + 2 * kPartCB;   // B (then v o B) and S0
constexpr int kOffX = kOffBS + 2 * kPartBS;
constexpr int kOffVec = kOffX + 2 * kPartX;

struct Vec {
  // running sum of dt A log2(e) over the block through the token, as an
  // unevaluated pair hi + lo (summed in float-float arithmetic): differences
  // of two of them keep fp32 accuracy however large the sums grow
  float Ph[kQ], Pl[kQ];
  float dt[kQ];
  float v[kQ];    // [rc == rc_end] 2^(P_end - P) dt: weight of the token in the final state
  float w[kQ];    // [rc == 0] 2^P: how much of the incoming state reaches the token
  int rc[kQ];     // sample starts at or before the token, in the block
  float wsh[4], wsl[4];  // per-warp totals of the scans
  int wcnt[4];
  float Pend;     // P at the block's last token
  int rcend;
};
constexpr int kOffCtl = kOffVec + ((sizeof(Vec) + 127) / 128) * 128;

struct Ctl {
  uint64_t mma_bar;
  uint64_t done_bar;
  uint64_t tma_c_bar;   // C's rows of a block
  uint64_t tma_bx_bar;  // B's and x's rows of a block
  uint32_t tmem_base;
  int pad;
};
constexpr int kSmem = kOffCtl + 128 + 1024;  // + alignment slack
static_assert(sizeof(Ctl) <= 128, "control block");
static_assert(kSmem <= 232448, "dynamic shared memory of one CTA");

constexpr uint32_t kColG = 0, kColYoff = 128, kColYdia = 192, kColS = 256;
// C's split parts (hi 320-383, lo 384-447: the A operand of [G | Yoff]), then
// M's (the A operand of Ydia), two fp16 per column
constexpr uint32_t kColA = 320, kColAlo = 384;

constexpr uint32_t kIdescGY = make_idesc_f16(128, 192, false, false);
constexpr uint32_t kIdescYdia = make_idesc_f16(128, 64, false, true);
constexpr uint32_t kIdescS = make_idesc_f16(128, 64, true, true);

// The same for row `row` (B's token rows 0-127, S0's rows 128-191) of the
// shared B / S0 operand.
__device__ __forceinline__ uint32_t bs_chunk(int row, int kc) {
  return static_cast<uint32_t>((kc >> 3) * kBlkBS + (row >> 3) * 1024 + (row & 7) * 128 +
                               (((kc & 7) ^ (row & 7)) << 4));
}

// A block's fp32 rows are staged by TMA.  C's go to their own 64 KB, as four
// boxes of 32 state values x 128 tokens with the 128-byte swizzle (16-byte
// unit u of row t at unit u ^ (t mod 8)), so that each thread reads the 32
// values of its own token without bank conflicts.  B's go to the four 16 KB
// pieces of the B / S0 operand that B's rows take (32 rows each: K block
// k & 1 of part k >> 1), S0's rows staying untouched; x's 128 rows (256 B)
// to where x goes.  Those two are split in place.
constexpr uint32_t kStageBytesC = kQ * kN * 4;
constexpr uint32_t kStageBytesBX = kQ * kN * 4 + kQ * kP * 4;
// chunks of 8 values per thread: C and B (16 per token), x (8 per token)
constexpr int kTasksCB = kQ * 16 / kThreads;
constexpr int kTasksX = kQ * 8 / kThreads;
__device__ __forceinline__ uint32_t b_piece(int k) {
  return static_cast<uint32_t>(kOffBS + (k >> 1) * kPartBS + (k & 1) * kBlkBS);
}

__global__ void __launch_bounds__(kThreads, 1)
    ssd_chunk_scan_tc_kernel(const SsdParams p, const __grid_constant__ CUtensorMap map_c_sw,
                             const __grid_constant__ CUtensorMap map_b,
                             const __grid_constant__ CUtensorMap map_x) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  Vec& vec = *reinterpret_cast<Vec*>(smem + kOffVec);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kOffCtl);
  const int h = blockIdx.x, r = blockIdx.y;
  const int g = h / (p.H / p.G);
  const int L = p.T / p.R;
  const int c0 = r * L;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // every index below is the CTA's head, group and rank plus offsets inside
  // the tile shapes and the chunk's rows: checking those checks them all
  if (!index_ok(h, p.H, p.status, kSiteSsd) || !index_ok(g, p.G, p.status, kSiteSsd) ||
      !index_ok(r, p.R, p.status, kSiteSsd) ||
      !index_ok((long long)c0 + L - 1, p.T, p.status, kSiteSsd))
    return;
  const float A2 = p.A[h] * kLog2e;
  const float Dh = p.D ? p.D[h] : 0.f;

  const Operand opBS{sbase + kOffBS, kPartBS, kBlkBS, false};
  const Operand opVB{sbase + kOffBS, kPartBS, kBlkBS, true};  // v o B, rows = tokens
  const Operand opX{sbase + kOffX, kPartX, kPartX, true};

  if (threadIdx.x == 0) {
    mbar_init(&ctl->mma_bar, 1);
    mbar_init(&ctl->done_bar, 1);
    mbar_init(&ctl->tma_c_bar, 1);
    mbar_init(&ctl->tma_bx_bar, 1);
    fence_barrier_init();
    tma_prefetch_map(&map_c_sw);
    tma_prefetch_map(&map_b);
    tma_prefetch_map(&map_x);
  }
  if (warp == 0) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  // TMEM lanes of this warp (a warp reaches lanes 32 (warp mod 4) ...) and the
  // quarter of each accumulator's columns it takes
  const int row = (warp & 3) * 32 + lane;
  const int cg = warp >> 2;
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;

  // the state before the first block is zero (S0's rows of both K blocks,
  // hi and lo); then the first block's operands
  for (int i = threadIdx.x; i < 4 * kP * 128 / 16; i += kThreads) {
    const int part = i / (kP * 128 / 16), k = i % (kP * 128 / 16);
    reinterpret_cast<uint4*>(smem + kOffBS + (part >> 1) * kPartBS + (part & 1) * kBlkBS +
                             kQ * 128)[k] = make_uint4(0u, 0u, 0u, 0u);
  }
  // warps 4-7 scan the decays, one token each (warp 0 issues the MMAs):
  // this thread's token of the next block to scan, its dt and position (a
  // sample starts at position 0)
  const bool scanner = warp >= 4 && warp < 8;
  const int tok = static_cast<int>(threadIdx.x) - 128;
  float tok_dt = 0.f;
  int tok_pos = 1;
  auto load_token = [&](int tb, int nb) {
    const bool in = scanner && tok < nb;
    tok_dt = in ? p.dt[(size_t)(tb + tok) * p.H + h] : 0.f;
    tok_pos = (in && p.pos != nullptr) ? p.pos[tb + tok] : 1;
  };
  // thread 0 stages a block's rows (tokens tb ...; rows past the tensor's
  // end read as zeros, rows past the chunk's end are zeroed in the split)
  auto stage_c = [&](int tb) {
    mbar_arrive_expect_tx(&ctl->tma_c_bar, kStageBytesC);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      tma_load_3d(smem + kOffC + k * kQ * 128, &map_c_sw, &ctl->tma_c_bar, 32 * k, g, tb);
  };
  auto stage_bx = [&](int tb) {
    mbar_arrive_expect_tx(&ctl->tma_bx_bar, kStageBytesBX);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      tma_load_3d(smem + b_piece(k), &map_b, &ctl->tma_bx_bar, 0, g, tb + 32 * k);
    tma_load_3d(smem + kOffX, &map_x, &ctl->tma_bx_bar, 0, h, tb);
  };
  load_token(c0, min(kQ, L));
  __syncthreads();  // barriers initialised; S0's rows zeroed; TMEM allocated
  tc_fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;
  if (threadIdx.x == 0) {
    stage_c(c0);
    stage_bx(c0);
  }

  float log2carry = 0.f;  // sum of dt A log2(e) over the chunk
  bool reset = false;     // a sample starts inside the chunk
  int uses = 0;           // phases of mma_bar so far
  bool ok = true;
  const int nblocks = (L + kQ - 1) / kQ;
  for (int b = 0; b < nblocks && ok; ++b) {
    const int t0 = c0 + b * kQ;
    const int n = min(kQ, c0 + L - t0);
    // ---- the block's staged rows, split: C into TMEM (this thread's token,
    // 32 state values), B and x in place (every thread reads all its values
    // before any thread overwrites them)
    ok = __syncthreads_and(mbar_wait(&ctl->tma_c_bar, b & 1, p.status, nullptr) &&
                           mbar_wait(&ctl->tma_bx_bar, b & 1, p.status, nullptr)) != 0;
    if (!ok) break;
    tc_fence_after_sync();
    {
      const uint8_t* crow = smem + kOffC + cg * kQ * 128 + row * 128;
      float cv[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 f = *reinterpret_cast<const float4*>(crow + ((u ^ (row & 7)) << 4));
        cv[4 * u] = f.x;
        cv[4 * u + 1] = f.y;
        cv[4 * u + 2] = f.z;
        cv[4 * u + 3] = f.w;
      }
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (row < n)
          split2(cv[2 * i], cv[2 * i + 1], &hi[i], &lo[i]);
        else
          hi[i] = lo[i] = 0u;
      }
      tmem_store_16(tmem + lane_off + kColA + cg * 16, hi);
      tmem_store_16(tmem + lane_off + kColAlo + cg * 16, lo);
    }
    // B's values stay in registers until they are scaled by v
    float bv[kTasksCB][8];
    {
      float xv[kTasksX][8];
#pragma unroll
      for (int u = 0; u < kTasksCB; ++u) {
        const int q = threadIdx.x + u * kThreads;
        const int t = q >> 4, kc = q & 15;
        load_staged8(smem + b_piece(t >> 5) + (t & 31) * kN * 4, kc, bv[u]);
      }
#pragma unroll
      for (int u = 0; u < kTasksX; ++u) {
        const int q = threadIdx.x + u * kThreads;
        load_staged8(smem + kOffX + (q >> 3) * kP * 4, q & 7, xv[u]);
      }
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kTasksCB; ++u) {
        const int q = threadIdx.x + u * kThreads;
        const int t = q >> 4, kc = q & 15;
        if (t >= n) {
#pragma unroll
          for (int i = 0; i < 8; ++i) bv[u][i] = 0.f;
        }
        const uint32_t ab = bs_chunk(t, kc);
        split8(bv[u], reinterpret_cast<uint4*>(smem + kOffBS + ab),
               reinterpret_cast<uint4*>(smem + kOffBS + kPartBS + ab));
      }
#pragma unroll
      for (int u = 0; u < kTasksX; ++u) {
        const int q = threadIdx.x + u * kThreads;
        const int t = q >> 3;
        if (t >= n) {
#pragma unroll
          for (int i = 0; i < 8; ++i) xv[u][i] = 0.f;
        }
        const uint32_t at = sw_chunk(kQ, t, q & 7);
        split8(xv[u], reinterpret_cast<uint4*>(smem + kOffX + at),
               reinterpret_cast<uint4*>(smem + kOffX + kPartX + at));
      }
    }
    tmem_store_wait();
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const bool more = b + 1 < nblocks;
    const int tn = t0 + kQ;
    // ---- [G | Yoff] = C [B | S0]^T; C's staging is free again, so the next
    // block's rows of C are staged from here on
    if (threadIdx.x == 0) {
      mma_split_ta(tmem + kColG, tmem + kColA, tmem + kColAlo, opBS, kIdescGY, false);
      mma_commit(&ctl->mma_bar);
      if (more) stage_c(tn);
    }
    // ---- while it runs: per-token decays and sample starts, inclusive
    // scans over the block
    float ph = 0.f, pl = 0.f;  // this token's running sum within its warp
    int cw = 0;
    if (scanner) {
      ph = tok_dt * A2;
      cw = tok_pos == 0 ? 1 : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float uh = __shfl_up_sync(0xffffffffu, ph, o);
        const float ul = __shfl_up_sync(0xffffffffu, pl, o);
        const int cu = __shfl_up_sync(0xffffffffu, cw, o);
        if (lane >= o) {
          ff_add(ph, pl, uh, ul);
          cw += cu;
        }
      }
      if (lane == 31) {
        vec.wsh[warp - 4] = ph;
        vec.wsl[warp - 4] = pl;
        vec.wcnt[warp - 4] = cw;
      }
    }
    __syncthreads();
    if (scanner) {
      const int t = tok;
      float eh = 0.f, el = 0.f;  // P at the block's end
      int rc = cw, rcend = 0;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        if (w < warp - 4) {
          ff_add(ph, pl, vec.wsh[w], vec.wsl[w]);
          rc += vec.wcnt[w];
        }
        ff_add(eh, el, vec.wsh[w], vec.wsl[w]);
        rcend += vec.wcnt[w];
      }
      vec.Ph[t] = ph;
      vec.Pl[t] = pl;
      vec.rc[t] = rc;
      vec.dt[t] = tok_dt;
      vec.v[t] = rc == rcend ? fast_exp2((eh - ph) + (el - pl)) * tok_dt : 0.f;
      vec.w[t] = rc == 0 ? fast_exp2(ph + pl) : 0.f;
      if (t == 0) {
        vec.Pend = eh + el;
        vec.rcend = rcend;
      }
    }
    ok = cta_wait_mma(&ctl->mma_bar, uses & 1, p.status);
    ++uses;
    if (!ok) break;
    tc_fence_after_sync();
    const float Pend = vec.Pend;
    const int rcend = vec.rcend;
    // ---- M = G o mask o dt (rows = tokens t, K = tokens j), into C's TMEM
    // columns; a warp whose 32 columns all lie above its 32 rows writes zeros
    {
      uint32_t hi[16], lo[16];
      if (cg > (warp & 3)) {
#pragma unroll
        for (int i = 0; i < 16; ++i) hi[i] = lo[i] = 0u;
      } else {
        uint32_t gv[32];
        tmem_load_32(tmem + lane_off + kColG + cg * 32, gv);
        const float pht = vec.Ph[row], plt = vec.Pl[row];
        const int rct = vec.rc[row];
#pragma unroll
        for (int i4 = 0; i4 < 32; i4 += 4) {
          const int j0 = cg * 32 + i4;
          const float4 phj = *reinterpret_cast<const float4*>(&vec.Ph[j0]);
          const float4 plj = *reinterpret_cast<const float4*>(&vec.Pl[j0]);
          const float4 dj = *reinterpret_cast<const float4*>(&vec.dt[j0]);
          const int4 rj = *reinterpret_cast<const int4*>(&vec.rc[j0]);
          const float phv[4] = {phj.x, phj.y, phj.z, phj.w};
          const float plv[4] = {plj.x, plj.y, plj.z, plj.w};
          const float djv[4] = {dj.x, dj.y, dj.z, dj.w};
          const int rjv[4] = {rj.x, rj.y, rj.z, rj.w};
          float m[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = j0 + i;
            const bool vis = j <= row && rjv[i] == rct;
            const float e = fast_exp2(vis ? (pht - phv[i]) + (plt - plv[i]) : -INFINITY);
            m[i] = __uint_as_float(gv[i4 + i]) * e * djv[i];
          }
          split2(m[0], m[1], &hi[i4 / 2], &lo[i4 / 2]);
          split2(m[2], m[3], &hi[i4 / 2 + 1], &lo[i4 / 2 + 1]);
        }
      }
      tmem_store_16(tmem + lane_off + kColA + cg * 16, hi);
      tmem_store_16(tmem + lane_off + kColAlo + cg * 16, lo);
    }
    // ---- B_j scaled by v_j, over B's split in place: (v o B) read MN-major
    // is (v o B)^T
#pragma unroll
    for (int u = 0; u < kTasksCB; ++u) {
      const int q = threadIdx.x + u * kThreads;
      const int j = q >> 4;
      const uint32_t at = bs_chunk(j, q & 15);
      const float vj = vec.v[j];
#pragma unroll
      for (int i = 0; i < 8; ++i) bv[u][i] *= vj;
      split8(bv[u], reinterpret_cast<uint4*>(smem + kOffBS + at),
             reinterpret_cast<uint4*>(smem + kOffBS + kPartBS + at));
    }
    // ---- the state before the block decays through it (or dies at a sample start)
    if (b > 0) {
      const float keep = rcend == 0 ? fast_exp2(Pend) : 0.f;
      uint32_t sv[16];
      tmem_load_16(tmem + lane_off + kColS + cg * 16, sv);
#pragma unroll
      for (int i = 0; i < 16; ++i) sv[i] = __float_as_uint(__uint_as_float(sv[i]) * keep);
      tmem_store_16(tmem + lane_off + kColS + cg * 16, sv);
    }
    tmem_store_wait();
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    // ---- Ydia = M X, S^T += (v o B)^T X; meanwhile the scanning warps load
    // the next block's tokens
    if (more) load_token(tn, min(kQ, c0 + L - tn));
    if (threadIdx.x == 0) {
      tc_fence_after_sync();
      mma_split_ta(tmem + kColYdia, tmem + kColA, tmem + kColAlo, opX, kIdescYdia, false);
      mma_split(tmem + kColS, opVB, opX, kIdescS, b > 0);
      mma_commit(&ctl->mma_bar);
    }
    ok = cta_wait_mma(&ctl->mma_bar, uses & 1, p.status);
    ++uses;
    if (!ok) break;
    tc_fence_after_sync();
    // B's and x's space is free again: the next block's rows are staged
    // there while this block's state and y are written out
    if (more && threadIdx.x == 0) stage_bx(tn);
    float4 xr[4];
    const size_t orow = ((size_t)(t0 + row) * p.H + h) * kP + cg * 16;
    if (row < n) {
#pragma unroll
      for (int i = 0; i < 4; ++i) xr[i] = *reinterpret_cast<const float4*>(p.x + orow + 4 * i);
    }
    // ---- the state after the block: S0 (rows 128 + p of the B / S0
    // operand, K = state) for the next block's Yoff, and the chunk's final state
    {
      uint32_t sv[16];
      tmem_load_16(tmem + lane_off + kColS + cg * 16, sv);
      const int nn = row;  // this lane's state index
      const uint32_t in_chunk = (nn & 7) * 2;
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        uint32_t hi, lo;
        split2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1]), &hi, &lo);
        const uint32_t a0 = bs_chunk(kQ + cg * 16 + i, nn >> 3) + in_chunk;
        const uint32_t a1 = bs_chunk(kQ + cg * 16 + i + 1, nn >> 3) + in_chunk;
        *reinterpret_cast<uint16_t*>(smem + kOffBS + a0) = static_cast<uint16_t>(hi);
        *reinterpret_cast<uint16_t*>(smem + kOffBS + a1) = static_cast<uint16_t>(hi >> 16);
        *reinterpret_cast<uint16_t*>(smem + kOffBS + kPartBS + a0) = static_cast<uint16_t>(lo);
        *reinterpret_cast<uint16_t*>(smem + kOffBS + kPartBS + a1) = static_cast<uint16_t>(lo >> 16);
      }
      if (!more) {
        float* Sout = p.chunk_state + ((size_t)r * p.H + h) * kP * kN;
#pragma unroll
        for (int i = 0; i < 16; ++i) Sout[(size_t)(cg * 16 + i) * kN + nn] = __uint_as_float(sv[i]);
      }
    }
    // ---- y of the block: [rc_t == 0] 2^P_t Yoff + Ydia + D x
    {
      uint32_t yo[16], yd[16];
      tmem_load_16(tmem + lane_off + kColYoff + cg * 16, yo);
      tmem_load_16(tmem + lane_off + kColYdia + cg * 16, yd);
      if (row < n) {
        const float w = vec.w[row];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float4 yv;
          yv.x = fmaf(w, __uint_as_float(yo[4 * i]), __uint_as_float(yd[4 * i])) + Dh * xr[i].x;
          yv.y = fmaf(w, __uint_as_float(yo[4 * i + 1]), __uint_as_float(yd[4 * i + 1])) +
                 Dh * xr[i].y;
          yv.z = fmaf(w, __uint_as_float(yo[4 * i + 2]), __uint_as_float(yd[4 * i + 2])) +
                 Dh * xr[i].z;
          yv.w = fmaf(w, __uint_as_float(yo[4 * i + 3]), __uint_as_float(yd[4 * i + 3])) +
                 Dh * xr[i].w;
          *reinterpret_cast<float4*>(p.y + orow + 4 * i) = yv;
        }
      }
    }
    log2carry += Pend;
    reset = reset || rcend > 0;
  }
  if (ok && threadIdx.x == 0) p.carry[(size_t)r * p.H + h] = reset ? 0.f : exp2f(log2carry);
  // every MMA has completed before TMEM is released
  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0) {
    mma_commit(&ctl->done_bar);
    mbar_wait(&ctl->done_bar, 0, p.status, nullptr);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(ctl->tmem_base, 512);
  }
}

bool g_configured[64] = {};

}  // namespace

cudaError_t launch_ssd_chunk_scan_tc(const SsdParams& p, const SsdMaps& maps,
                                     cudaStream_t stream) {
  cudaError_t e = ensure_smem_limit(ssd_chunk_scan_tc_kernel, kSmem, g_configured);
  if (e != cudaSuccess) return e;
  TraceScope trace_scope(stream, "ssd_chunk_scan_tc_kernel");
  ssd_chunk_scan_tc_kernel<<<dim3(p.H, p.R), kThreads, kSmem, stream>>>(p, maps.c_sw, maps.b,
                                                                         maps.x);
  return cudaGetLastError();
}

}  // namespace ra
