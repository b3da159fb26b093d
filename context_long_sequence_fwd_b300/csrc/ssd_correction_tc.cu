// Additive correction of the context-parallel Mamba2 selective scan on the
// sm_103a tensor cores, for state size N = 128.
//
// Same contract as ssd_correction_kernel (ssd_cp.cu).  Rank r >= 1 scanned
// its chunk from a zero state; the state it should have started from is H_r
// (the ring of states).  The recurrence is linear in its initial state, so
// the difference is y_t += exp(A sum_{chunk start <= u <= t} dt_u) H_r C_t for
// the chunk's tokens before its first sample start (axolotl "Sequence
// Parallelism" page, "Mamba/SSM Hybrid Models": an additive correction, no
// second forward pass).
//
// CTA (h, r, segment), 256 threads, a block of 128 tokens at a time:
//   Yc = C H_r^T    (M = 128 tokens, N = 64 head dims, K = 128 state) in TMEM,
//   y_t += w_t Yc_t,  w_t = 2^(lam_t) before the first sample start, else 0,
// with lam_t the running sum of dt A log2(e) from the chunk start, kept in
// float-float arithmetic.  A chunk's blocks are cut into kSegs segments, one
// CTA each, which starts from the exponent summed over the chunk's tokens
// before it.  C and H are split into fp16 hi + lo and the
// product is formed from three fp16 products (ssd_tc_common.cuh), which
// keeps fp32-level accuracy.  C's fp32 rows are staged by TMA in the space
// of their split operand and split in place; the next block's rows are
// staged as soon as the product has read the current ones, so the copy runs
// under the y update.  The CTA stops after the block holding the chunk's
// first sample start, or after the block where the exponent has fallen below
// kDeadLog2: every later factor is exactly zero in fp32 (the exponent only
// falls), so each later token would add an exact zero.  About 100 KB of
// shared memory and 64 TMEM columns: two CTAs share an SM and overlap each
// other's phases.  Every barrier wait is bounded.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"
#include "sm103_ptx.cuh"
#include "ssd_tc_common.cuh"
#include "trace.h"

namespace ra {

namespace {

using namespace ssd_tc;

constexpr int kQ = 128;  // tokens per block
constexpr int kP = 64;   // head dimension
constexpr int kN = 128;  // state size
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
// log2 of a factor that is exactly zero in fp32 (denormals underflow below
// 2^-149), with a margin for the float-float rounding of the exponent
constexpr float kDeadLog2 = -160.f;
// A chunk's blocks are split into this many segments, one CTA each: the
// chains of weakly decaying heads without an early sample start, which walk
// the whole chunk, would otherwise set the kernel's length.
constexpr int kSegs = 4;

constexpr int kPartH = kP * kN * 2;  // H_r: 64 rows x 128 fp16, two 8 KB K blocks
constexpr int kPartC = kQ * kN * 2;  // C: 128 rows x 128 fp16, two 16 KB K blocks
constexpr int kOffH = 0;
constexpr int kOffC = kOffH + 2 * kPartH;  // staged fp32 rows, then split in place
constexpr int kOffVec = kOffC + 2 * kPartC;

struct Vec {
  float w[kQ];           // factor of each token's correction (0 after a sample start)
  float wsh[4], wsl[4];  // per-warp totals of the exponent scan
  int wcnt[4];           // per-warp sample starts
  float lam_h, lam_l;    // exponent at the end of the blocks so far
  int stop;              // the CTA ends after this block
  float red_h[8], red_l[8];  // per-warp parts of the segment's starting exponent
  int red_c[8];              // and of the sample starts before it
};
constexpr int kOffCtl = kOffVec + ((sizeof(Vec) + 127) / 128) * 128;

struct Ctl {
  uint64_t mma_bar;
  uint64_t tma_bar;
  uint64_t done_bar;
  uint32_t tmem_base;
  int pad;
};
constexpr int kSmem = kOffCtl + 128 + 1024;  // + alignment slack
static_assert(sizeof(Ctl) <= 128, "control block");
static_assert(2 * kSmem <= 232448, "two CTAs per SM");

constexpr uint32_t kIdesc = make_idesc_f16(128, 64, false, false);
constexpr uint32_t kStageBytes = kQ * kN * 4;
constexpr int kTasksC = kQ * 16 / kThreads;  // 8-value chunks of C per thread
constexpr int kTasksH = kP * 16 / kThreads;

__global__ void __launch_bounds__(kThreads, 2)
    ssd_correction_tc_kernel(const SsdParams p, const __grid_constant__ CUtensorMap map_c) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  Vec& vec = *reinterpret_cast<Vec*>(smem + kOffVec);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kOffCtl);
  const int h = blockIdx.x, r = blockIdx.y + 1;
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
  // this CTA's segment: blocks [bb, be) of the chunk
  const int nblocks = (L + kQ - 1) / kQ;
  const int bps = (nblocks + kSegs - 1) / kSegs;
  const int bb = blockIdx.z * bps, be = min(bb + bps, nblocks);
  if (bb >= be) return;
  const int s0 = c0 + bb * kQ;  // the segment's first token
  // the exponent at the segment's start (float-float sum of dt A log2(e) over
  // the chunk's tokens before it) and the sample starts there: after one,
  // or once the exponent is dead, the segment corrects nothing
  float lam0_h = 0.f, lam0_l = 0.f;
  {
    float sh = 0.f, sl = 0.f;
    int starts = 0;
    for (int t = c0 + static_cast<int>(threadIdx.x); t < s0; t += kThreads) {
      ff_add(sh, sl, p.dt[(size_t)t * p.H + h] * A2, 0.f);
      if (p.pos != nullptr && p.pos[t] == 0) ++starts;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float uh = __shfl_down_sync(0xffffffffu, sh, o);
      const float ul = __shfl_down_sync(0xffffffffu, sl, o);
      starts += __shfl_down_sync(0xffffffffu, starts, o);
      ff_add(sh, sl, uh, ul);
    }
    if (lane == 0) {
      vec.red_h[warp] = sh;
      vec.red_l[warp] = sl;
      vec.red_c[warp] = starts;
    }
    __syncthreads();
    int total = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      ff_add(lam0_h, lam0_l, vec.red_h[w], vec.red_l[w]);
      total += vec.red_c[w];
    }
    if (total > 0 || lam0_h + lam0_l < kDeadLog2) return;  // the same for every thread
  }

  const Operand opC{sbase + kOffC, kPartC, kQ * 128, false};
  const Operand opH{sbase + kOffH, kPartH, kP * 128, false};

  if (threadIdx.x == 0) {
    mbar_init(&ctl->mma_bar, 1);
    mbar_init(&ctl->tma_bar, 1);
    mbar_init(&ctl->done_bar, 1);
    fence_barrier_init();
    tma_prefetch_map(&map_c);
    vec.lam_h = lam0_h;
    vec.lam_l = lam0_l;
  }
  if (warp == 0) {
    tmem_alloc(&ctl->tmem_base, 64);
    tmem_relinquish();
  }
  // thread 0 stages the rows of C of the block at tb (rows past the tensor's
  // end read as zeros; rows past the chunk are zeroed in the split)
  auto stage_rows = [&](int tb) {
    mbar_arrive_expect_tx(&ctl->tma_bar, kStageBytes);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      tma_load_3d(smem + kOffC + k * 32 * kN * 4, &map_c, &ctl->tma_bar, 0, g, tb + 32 * k);
  };
  // H_r, split into the K-major B operand (rows = head dim, K = state)
  {
    const float* Hr = p.incoming + ((size_t)r * p.H + h) * kP * kN;
#pragma unroll
    for (int u = 0; u < kTasksH; ++u) {
      const int q = threadIdx.x + u * kThreads;
      const int pr = q >> 4, kc = q & 15;
      const float4 a = *reinterpret_cast<const float4*>(Hr + pr * kN + kc * 8);
      const float4 b = *reinterpret_cast<const float4*>(Hr + pr * kN + kc * 8 + 4);
      float v8[8];
      unpack8(a, b, v8);
      const uint32_t at = sw_chunk(kP, pr, kc);
      split8(v8, reinterpret_cast<uint4*>(smem + kOffH + at),
             reinterpret_cast<uint4*>(smem + kOffH + kPartH + at));
    }
  }
  // this thread's token (warps 0-3) of the next block: dt and position
  float tok_dt = 0.f;
  int tok_pos = 1;
  auto load_token = [&](int tb, int nb) {
    const bool in = warp < 4 && static_cast<int>(threadIdx.x) < nb;
    tok_dt = in ? p.dt[(size_t)(tb + threadIdx.x) * p.H + h] : 0.f;
    tok_pos = (in && p.pos != nullptr) ? p.pos[tb + threadIdx.x] : 1;
  };
  load_token(s0, min(kQ, c0 + L - s0));
  __syncthreads();  // barriers initialised
  if (threadIdx.x == 0) stage_rows(s0);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;
  const int row = (warp & 3) * 32 + lane;
  const int half = warp >> 2;
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;

  bool ok = true;
  for (int b = bb; b < be; ++b) {
    const int t0 = c0 + b * kQ;
    const int n = min(kQ, c0 + L - t0);
    const uint32_t phase = (b - bb) & 1;
    ok = __syncthreads_and(mbar_wait(&ctl->tma_bar, phase, p.status, nullptr)) != 0;
    if (!ok) break;
    // ---- the exponent of each token and the sample starts: inclusive scans
    // (warps 0-3, one token each), on top of the blocks before
    float ph = 0.f, pl = 0.f;
    int cw = 0;
    // the exponent at the block's start, read before thread 0 moves it on
    const float lam_h0 = vec.lam_h, lam_l0 = vec.lam_l;
    if (warp < 4) {
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
        vec.wsh[warp] = ph;
        vec.wsl[warp] = pl;
        vec.wcnt[warp] = cw;
      }
    }
    // ---- C's staged rows, read before the barrier, split in place after it
    float cv[kTasksC][8];
#pragma unroll
    for (int u = 0; u < kTasksC; ++u) {
      const int q = threadIdx.x + u * kThreads;
      load_staged8(smem + kOffC + (q >> 4) * kN * 4, q & 15, cv[u]);
    }
    __syncthreads();
    if (warp < 4) {
      float eh = lam_h0, el = lam_l0;  // exponent at the block's start
      int rc = cw, rcend = 0;
      float th = 0.f, tl = 0.f;              // the block's total
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        if (w < warp) {
          ff_add(ph, pl, vec.wsh[w], vec.wsl[w]);
          rc += vec.wcnt[w];
        }
        ff_add(th, tl, vec.wsh[w], vec.wsl[w]);
        rcend += vec.wcnt[w];
      }
      float xh = eh, xl = el;
      ff_add(xh, xl, ph, pl);
      vec.w[threadIdx.x] = (rc == 0 && static_cast<int>(threadIdx.x) < n) ? fast_exp2(xh + xl) : 0.f;
      // all lanes of warps 0-3 hold the same block total; one writes
      if (threadIdx.x == 0) {
        ff_add(eh, el, th, tl);
        vec.lam_h = eh;
        vec.lam_l = el;
        vec.stop = rcend > 0 || eh + el < kDeadLog2;
      }
    }
#pragma unroll
    for (int u = 0; u < kTasksC; ++u) {
      const int q = threadIdx.x + u * kThreads;
      const int t = q >> 4, kc = q & 15;
      if (t >= n) {
#pragma unroll
        for (int i = 0; i < 8; ++i) cv[u][i] = 0.f;
      }
      const uint32_t at = sw_chunk(kQ, t, kc);
      split8(cv[u], reinterpret_cast<uint4*>(smem + kOffC + at),
             reinterpret_cast<uint4*>(smem + kOffC + kPartC + at));
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    // ---- Yc = C H_r^T
    if (threadIdx.x == 0) {
      tc_fence_after_sync();
      mma_split(tmem, opC, opH, kIdesc, false);
      mma_commit(&ctl->mma_bar);
    }
    const bool last = vec.stop != 0 || b + 1 == be;
    if (!last) {
      const int tn = t0 + kQ;
      load_token(tn, min(kQ, c0 + L - tn));
    }
    ok = cta_wait_mma(&ctl->mma_bar, phase, p.status);
    if (!ok) break;
    tc_fence_after_sync();
    // C's space is free: the next block's rows are staged under the y update
    if (!last && threadIdx.x == 0) stage_rows(t0 + kQ);
    // ---- y_t += w_t Yc_t
    {
      uint32_t yc[32];
      tmem_load_32(tmem + lane_off + half * 32, yc);
      const float w = vec.w[row];
      if (w != 0.f) {
        float* yr = p.y + ((size_t)(t0 + row) * p.H + h) * kP + half * 32;
        float4 yv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) yv[i] = *reinterpret_cast<const float4*>(yr + 4 * i);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          yv[i].x = fmaf(w, __uint_as_float(yc[4 * i]), yv[i].x);
          yv[i].y = fmaf(w, __uint_as_float(yc[4 * i + 1]), yv[i].y);
          yv[i].z = fmaf(w, __uint_as_float(yc[4 * i + 2]), yv[i].z);
          yv[i].w = fmaf(w, __uint_as_float(yc[4 * i + 3]), yv[i].w);
          *reinterpret_cast<float4*>(yr + 4 * i) = yv[i];
        }
      }
    }
    tc_fence_before_sync();
    __syncthreads();  // TMEM and the factors are read before the next block
    if (last) break;
  }
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
    tmem_dealloc(tmem, 64);
  }
}

bool g_configured[64] = {};

}  // namespace

cudaError_t launch_ssd_correction_tc(const SsdParams& p, const SsdMaps& maps,
                                     cudaStream_t stream) {
  if (p.R < 2) return cudaSuccess;
  cudaError_t e = ensure_smem_limit(ssd_correction_tc_kernel, kSmem, g_configured);
  if (e != cudaSuccess) return e;
  TraceScope trace_scope(stream, "ssd_correction_tc_kernel");
  ssd_correction_tc_kernel<<<dim3(p.H, p.R - 1, kSegs), kThreads, kSmem, stream>>>(p, maps.c);
  return cudaGetLastError();
}

}  // namespace ra
