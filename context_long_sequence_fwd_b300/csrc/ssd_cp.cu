// Context-parallel selective scan of a Mamba2 layer (the SSD recurrence) on
// CUDA cores, fp32.
//
// The axolotl "Sequence Parallelism" page ("Mamba/SSM Hybrid Models"): SSM
// layers are recurrent, so under context parallelism each rank scans its own
// chunk, sends its final hidden state to the next rank, and applies an
// additive correction for the state it did not start from -- the SSM is
// linear in its initial state, so no second forward pass is needed.  Packed
// samples reset the state where they start (position 0 in position_ids).
// Per head h (group g), token t:
//   S <- 0 if pos[t] == 0;  S <- exp(dt A) S + dt x_t B_t^T;  y_t = S C_t + D x_t.
// All P virtual ranks run on one GPU, as three launches:
//   1. ssd_chunk_scan_kernel  (head, rank): the rank's chunk from S = 0; writes
//      y, the chunk's final state and its carry factor -- exp(A sum dt) over
//      the chunk, or 0 if a sample starts inside it (the incoming state dies
//      there).  For state size 128 the tensor-core form of this scan
//      (ssd_chunk_tc.cu) runs instead; the kernel here serves state size 64.
//   2. ssd_state_pass_kernel  (head): the ring of states, rank by rank:
//      H_0 = 0, H_r = carry_{r-1} H_{r-1} + S_{r-1} (what rank r would receive).
//   3. ssd_correction_kernel  (head, rank >= 1): y_t += exp(A sum_{chunk start
//      <= u <= t} dt_u) H_r C_t for the chunk's tokens before its first sample
//      start, up to the block where that factor has underflowed to zero.  For
//      state size 128 the tensor-core form (ssd_correction_tc.cu) runs instead.
// Threads: 256 per CTA.  A thread owns two rows of the state (2 rp, 2 rp + 1)
// and N / 8 of their columns: thread cs of a row pair holds columns
// 32 j + 4 cs + e (e < 4), so each B or C value it reads from shared memory
// feeds two rows, it reads them with 16-byte loads, and the eight threads of
// a row pair read 128 contiguous bytes (no bank conflicts).  A row's output is
// an 8-lane shuffle sum.  Inputs are staged in shared memory 32 tokens at a
// time, with each token's decay exp(dt A) computed once.
#include <cuda_runtime.h>

#include <cmath>

#include "launch.h"
#include "sm103_ptx.cuh"
#include "trace.h"

namespace ra {

namespace {

constexpr int kP = 64;       // head dimension
constexpr int kThreads = 256;
constexpr int kTok = 32;     // tokens staged per block

// The scan keeps the state of each 32-token block scaled: with rho_k the
// product of the decays exp(dt A) from the block start through token k,
// S~_k = S_k / rho_k obeys S~_k = S~_{k-1} + (dt_k / rho_k) x_k B_k^T (one
// FMA per entry instead of a multiply and an FMA), y_k = rho_k S~_k C_k, and
// S = rho S~ again at the block end.  If rho would fall below kTinyRho, the
// block rebases: S~ is first rescaled to the true state of the previous
// token (pre = that token's rho) and rho restarts from the current decay, or,
// when that decay itself is below kTinyRho, the previous state is dropped
// (pre = 0: it would contribute less than 1e-20 of itself).
constexpr float kTinyRho = 1e-20f;

// x and y rows are padded to kPX floats: the output step reads x and writes y
// of eight different tokens at once, which 64-float rows put on one bank.
constexpr int kPX = kP + 4;

template <int N>
struct Stage {
  float x[kTok][kPX];
  float B[kTok][N];
  float C[kTok][N];
  float dt[kTok];
  float rho[kTok];   // decay product since the block start (or the last rebase)
  float irho[kTok];  // 1 / rho
  float pre[kTok];   // factor applied to S~ before token k (1 = none)
  int pos[kTok];
  float y[kTok][kPX];
};

// Column of the state a thread's i-th entry (of each of its rows) holds.
__device__ __forceinline__ int ssd_col(int cs, int i) {
  return 32 * (i >> 2) + 4 * cs + (i & 3);
}

// Loads tokens [t0, t0 + n) of head h (group g) into shared memory; warp 0
// also forms the block's decay products (a multiplicative warp scan, so each
// rho carries at most a few roundings).
template <int N>
__device__ __forceinline__ void stage_tokens(Stage<N>& st, const SsdParams& p, int h, int g, int t0,
                                             int n) {
  // every 16-byte copy of the block is in flight at once
  constexpr int kX4 = kTok * kP / 4 / kThreads, kB4 = kTok * N / 4 / kThreads;
#pragma unroll
  for (int u = 0; u < kX4; ++u) {
    const int i = threadIdx.x + u * kThreads, k = i / (kP / 4), c4 = i % (kP / 4);
    cp_async16(&st.x[k][4 * c4], &p.x[((size_t)(t0 + min(k, n - 1)) * p.H + h) * kP + 4 * c4], k < n);
  }
#pragma unroll
  for (int u = 0; u < kB4; ++u) {
    const int i = threadIdx.x + u * kThreads, k = i / (N / 4), c4 = i % (N / 4);
    const size_t o = ((size_t)(t0 + min(k, n - 1)) * p.G + g) * N + 4 * c4;
    cp_async16(&st.B[k][4 * c4], &p.B[o], k < n);
    cp_async16(&st.C[k][4 * c4], &p.C[o], k < n);
  }
  if (threadIdx.x < 32) {
    const int k = threadIdx.x;
    const bool in = k < n;
    const float d = in ? p.dt[(size_t)(t0 + k) * p.H + h] : 0.f;
    const float a = in ? expf(d * p.A[h]) : 1.f;
    float rho = a;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, rho, o);
      if (k >= o) rho *= u;
    }
    if (in) {
      st.dt[k] = d;
      st.pos[k] = p.pos ? p.pos[t0 + k] : 1;
    }
    if (__ballot_sync(0xffffffffu, in && rho < kTinyRho) == 0) {
      if (in) {
        st.rho[k] = rho;
        st.irho[k] = 1.f / rho;
        st.pre[k] = 1.f;
      }
    } else {
      // rare: the block decays past kTinyRho; rebase token by token
      const float ak = a;
      float r = 1.f;
      for (int j = 0; j < n; ++j) {
        const float aj = __shfl_sync(0xffffffffu, ak, j);
        float pre = 1.f;
        const float rn = r * aj;
        if (rn >= kTinyRho) {
          r = rn;
        } else if (aj >= kTinyRho) {
          pre = r;  // S~ becomes the true state of token j - 1
          r = aj;
        } else {
          pre = 0.f;  // the previous state is dropped
          r = 1.f;
        }
        if (k == 0) {
          st.rho[j] = r;
          st.irho[j] = 1.f / r;
          st.pre[j] = pre;
        }
      }
    }
  }
  cp_async_wait_all();
}

// Sums v[t] (t < 8: eight tokens' partial row values of this thread) over the
// eight lanes of a row pair and leaves token cs's total in the result:
// three halving exchanges (xor 4, 2, 1) instead of a full reduction per token.
__device__ __forceinline__ float reduce_scatter8(const float (&v)[8], int cs) {
  float w[4];
  const bool b2 = (cs & 4) != 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float send = b2 ? v[t] : v[t + 4];
    w[t] = (b2 ? v[t + 4] : v[t]) + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  const bool b1 = (cs & 2) != 0;
  float u[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const float send = b1 ? w[t] : w[t + 2];
    u[t] = (b1 ? w[t + 2] : w[t]) + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  const bool b0 = (cs & 1) != 0;
  const float send = b0 ? u[0] : u[1];
  return (b0 ? u[1] : u[0]) + __shfl_xor_sync(0xffffffffu, send, 1);
}

template <int N>
__global__ void __launch_bounds__(kThreads, 4) ssd_chunk_scan_kernel(const SsdParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Stage<N>& st = *reinterpret_cast<Stage<N>*>(smem_raw);
  constexpr int kCols = N / 8;  // columns per thread, for each of its two rows
  const int h = blockIdx.x, r = blockIdx.y;
  const int g = h / (p.H / p.G);
  const int rp = threadIdx.x >> 3, cs = threadIdx.x & 7;
  const int L = p.T / p.R;
  const int c0 = r * L;
  // every index below is the CTA's head, group and rank plus offsets inside
  // [0, kP), [0, N) and the chunk's rows: checking those checks them all
  if (!index_ok(h, p.H, p.status, kSiteSsd) || !index_ok(g, p.G, p.status, kSiteSsd) ||
      !index_ok(r, p.R, p.status, kSiteSsd) ||
      !index_ok((long long)c0 + L - 1, p.T, p.status, kSiteSsd))
    return;
  const float A = p.A[h];
  const float Dh = p.D ? p.D[h] : 0.f;
  // rows 2 rp and 2 rp + 1 of S~, two adjacent columns per 64-bit register
  // pair: the update and the read-out run on paired fp32 instructions
  uint64_t S0[kCols / 2], S1[kCols / 2];
#pragma unroll
  for (int i = 0; i < kCols / 2; ++i) S0[i] = S1[i] = f32x2(0.f, 0.f);
  float logcarry = 0.f;  // A * sum dt over the chunk
  bool reset = false;    // a sample starts inside the chunk
  for (int t0 = c0; t0 < c0 + L; t0 += kTok) {
    const int n = min(kTok, c0 + L - t0);
    __syncthreads();  // the previous block's y has been written out
    stage_tokens<N>(st, p, h, g, t0, n);
    __syncthreads();
    for (int k8 = 0; k8 < n; k8 += 8) {
      float v0[8], v1[8];  // this thread's partial y of rows 2 rp, 2 rp + 1
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int k = k8 + kk;
        v0[kk] = v1[kk] = 0.f;
        if (k < n) {
          if (st.pos[k] == 0) {
#pragma unroll
            for (int i = 0; i < kCols / 2; ++i) S0[i] = S1[i] = f32x2(0.f, 0.f);
            reset = true;
            logcarry = 0.f;
          }
          const float pre = st.pre[k];
          if (pre != 1.f) {
            const uint64_t pp = f32x2(pre, pre);
#pragma unroll
            for (int i = 0; i < kCols / 2; ++i) {
              S0[i] = fmul2(pp, S0[i]);
              S1[i] = fmul2(pp, S1[i]);
            }
          }
          const float d = st.dt[k];
          logcarry = fmaf(d, A, logcarry);
          const float2 x2 = *reinterpret_cast<const float2*>(&st.x[k][2 * rp]);
          const float di = d * st.irho[k];
          const uint64_t dx0 = f32x2(di * x2.x, di * x2.x), dx1 = f32x2(di * x2.y, di * x2.y);
          uint64_t acc0 = f32x2(0.f, 0.f), acc1 = f32x2(0.f, 0.f);
#pragma unroll
          for (int j = 0; j < kCols / 4; ++j) {
            const float4 b4 = *reinterpret_cast<const float4*>(&st.B[k][ssd_col(cs, 4 * j)]);
            const float4 c4 = *reinterpret_cast<const float4*>(&st.C[k][ssd_col(cs, 4 * j)]);
            const uint64_t b01 = f32x2(b4.x, b4.y), b23 = f32x2(b4.z, b4.w);
            const uint64_t c01 = f32x2(c4.x, c4.y), c23 = f32x2(c4.z, c4.w);
            S0[2 * j] = ffma2(dx0, b01, S0[2 * j]);
            S0[2 * j + 1] = ffma2(dx0, b23, S0[2 * j + 1]);
            S1[2 * j] = ffma2(dx1, b01, S1[2 * j]);
            S1[2 * j + 1] = ffma2(dx1, b23, S1[2 * j + 1]);
            acc0 = ffma2(S0[2 * j], c01, acc0);
            acc0 = ffma2(S0[2 * j + 1], c23, acc0);
            acc1 = ffma2(S1[2 * j], c01, acc1);
            acc1 = ffma2(S1[2 * j + 1], c23, acc1);
          }
          float p0, p1, q0, q1;
          f32x2_split(acc0, &p0, &p1);
          f32x2_split(acc1, &q0, &q1);
          v0[kk] = p0 + p1;
          v1[kk] = q0 + q1;
        }
      }
      // lane cs of the row pair finishes token k8 + cs of both rows
      const float y0 = reduce_scatter8(v0, cs), y1 = reduce_scatter8(v1, cs);
      const int k = k8 + cs;
      if (k < n) {
        const float2 x2 = *reinterpret_cast<const float2*>(&st.x[k][2 * rp]);
        const float rk = st.rho[k];
        *reinterpret_cast<float2*>(&st.y[k][2 * rp]) =
            make_float2(fmaf(Dh, x2.x, rk * y0), fmaf(Dh, x2.y, rk * y1));
      }
    }
    // back to the true state for the next block
    const uint64_t rr = f32x2(st.rho[n - 1], st.rho[n - 1]);
#pragma unroll
    for (int i = 0; i < kCols / 2; ++i) {
      S0[i] = fmul2(rr, S0[i]);
      S1[i] = fmul2(rr, S1[i]);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n * (kP / 4); i += kThreads) {
      const int k = i / (kP / 4), c4 = i % (kP / 4);
      *reinterpret_cast<float4*>(&p.y[((size_t)(t0 + k) * p.H + h) * kP + 4 * c4]) =
          *reinterpret_cast<const float4*>(&st.y[k][4 * c4]);
    }
  }
  // the chunk's final state and the factor an incoming state survives with
  float* Sout = p.chunk_state + (((size_t)r * p.H + h) * kP + 2 * rp) * N;
#pragma unroll
  for (int i = 0; i < kCols / 2; ++i) {  // pair i holds columns ssd_col(cs, 2 i), + 1
    float lo, hi;
    f32x2_split(S0[i], &lo, &hi);
    *reinterpret_cast<float2*>(&Sout[ssd_col(cs, 2 * i)]) = make_float2(lo, hi);
    f32x2_split(S1[i], &lo, &hi);
    *reinterpret_cast<float2*>(&Sout[N + ssd_col(cs, 2 * i)]) = make_float2(lo, hi);
  }
  if (threadIdx.x == 0) p.carry[(size_t)r * p.H + h] = reset ? 0.f : expf(logcarry);
}

// H_r for every rank r >= 1 (into incoming[r]) and, if asked, the state after
// the last rank.  One CTA per head; each thread owns P N / 256 entries.
__global__ void __launch_bounds__(kThreads) ssd_state_pass_kernel(const SsdParams p) {
  const int h = blockIdx.x;
  if (!index_ok(h, p.H, p.status, kSiteSsd)) return;
  const int per = kP * p.N;
  for (int e = threadIdx.x; e < per; e += kThreads) {
    float Hs = 0.f;  // rank 0 starts from zero
    for (int r = 1; r <= p.R; ++r) {
      const float c = p.carry[(size_t)(r - 1) * p.H + h];
      const float s = p.chunk_state[((size_t)(r - 1) * p.H + h) * per + e];
      Hs = fmaf(c, Hs, s);
      if (r < p.R)
        p.incoming[((size_t)r * p.H + h) * per + e] = Hs;
      else if (p.final_state)
        p.final_state[(size_t)h * per + e] = Hs;
    }
  }
}

// Shared memory of the correction: the received state H (64 x N) and a block
// of 32 tokens' C, rows padded by 4 floats so that the float4 reads of 16
// different rows fall on distinct bank groups.
template <int N>
struct CorrStage {
  float H[kP][N + 4];
  float C[kTok][N + 4];
  float y[kTok][kP + 16];  // rows 16 banks apart: two tokens' rows per warp store
  float decay[kTok];  // exp(A sum dt) from the chunk start through the token
  int m;              // tokens of the block before the first sample start
  int dead;           // every later token's decay is exactly zero
};

// A sum dt below which expf is exactly 0 in fp32 (denormals included: it
// underflows near -103.97).  The running sum only falls: its terms are <= 0,
// a rounded sum of terms <= 0 is <= 0, and rounding is monotone, so once the
// sum at a block's end is below this, every later token adds an exact zero
// to y and the correction can stop there with the same result.
constexpr float kDeadExponent = -110.f;

// Y[t, :] += exp(A sum_{c0 <= u <= t} dt_u) H C_t for the block's tokens t
// before the first sample start: a 32 x 64 x N product per block, on CUDA
// cores in fp32.  Thread (ty, tx) computes tokens ty and ty + 16 for head-dim
// rows tx + 16 i (i < 4), accumulating even and odd n in the two halves of
// paired registers.
template <int N>
__global__ void __launch_bounds__(kThreads) ssd_correction_kernel(const SsdParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  CorrStage<N>& st = *reinterpret_cast<CorrStage<N>*>(smem_raw);
  const int h = blockIdx.x, r = blockIdx.y + 1;
  const int g = h / (p.H / p.G);
  if (!index_ok(h, p.H, p.status, kSiteSsd) || !index_ok(g, p.G, p.status, kSiteSsd) ||
      !index_ok(r, p.R, p.status, kSiteSsd) ||
      !index_ok((long long)(r + 1) * (p.T / p.R) - 1, p.T, p.status, kSiteSsd))
    return;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = p.T / p.R;
  const int c0 = r * L;
  const float A = p.A[h];
  {
    const float4* src = reinterpret_cast<const float4*>(p.incoming + ((size_t)r * p.H + h) * kP * N);
    for (int i = threadIdx.x; i < kP * N / 4; i += kThreads) {
      const int row = i / (N / 4), c4 = i % (N / 4);
      *reinterpret_cast<float4*>(&st.H[row][4 * c4]) = src[i];
    }
  }
  float lam = 0.f;  // A sum dt before the block (warp 0)
  for (int t0 = c0; t0 < c0 + L; t0 += kTok) {
    const int n = min(kTok, c0 + L - t0);
    __syncthreads();  // the previous block's C and y are consumed
    {
      constexpr int kC4 = kTok * N / 4 / kThreads;
#pragma unroll
      for (int u = 0; u < kC4; ++u) {
        const int i = threadIdx.x + u * kThreads, k = i / (N / 4), c4 = i % (N / 4);
        cp_async16(&st.C[k][4 * c4], &p.C[((size_t)(t0 + min(k, n - 1)) * p.G + g) * N + 4 * c4],
                   k < n);
      }
    }
    if (warp == 0) {
      // prefix sum of dt A over the block, and the first sample start
      const bool in = lane < n;
      float v = in ? p.dt[(size_t)(t0 + lane) * p.H + h] * A : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      const float lk = lam + v;
      st.decay[lane] = expf(lk);
      lam = __shfl_sync(0xffffffffu, lk, 31);
      const unsigned starts =
          __ballot_sync(0xffffffffu, in && p.pos != nullptr && p.pos[t0 + lane] == 0);
      if (lane == 0) {
        st.m = starts ? __ffs(starts) - 1 : n;
        st.dead = lam < kDeadExponent;
      }
    }
    cp_async_wait_all();
    __syncthreads();
    const int m = st.m;
    const bool dead = st.dead != 0;
    if (m > 0) {
      uint64_t acc[2][4];
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[a][i] = f32x2(0.f, 0.f);
#pragma unroll 4
      for (int c = 0; c < N; c += 4) {
        const float4 ca = *reinterpret_cast<const float4*>(&st.C[ty][c]);
        const float4 cb = *reinterpret_cast<const float4*>(&st.C[ty + 16][c]);
        const uint64_t ca01 = f32x2(ca.x, ca.y), ca23 = f32x2(ca.z, ca.w);
        const uint64_t cb01 = f32x2(cb.x, cb.y), cb23 = f32x2(cb.z, cb.w);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 hv = *reinterpret_cast<const float4*>(&st.H[tx + 16 * i][c]);
          const uint64_t h01 = f32x2(hv.x, hv.y), h23 = f32x2(hv.z, hv.w);
          acc[0][i] = ffma2(ca01, h01, acc[0][i]);
          acc[0][i] = ffma2(ca23, h23, acc[0][i]);
          acc[1][i] = ffma2(cb01, h01, acc[1][i]);
          acc[1][i] = ffma2(cb23, h23, acc[1][i]);
        }
      }
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const int k = ty + 16 * a;
        const float dk = st.decay[k];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float lo, hi;
          f32x2_split(acc[a][i], &lo, &hi);
          st.y[k][tx + 16 * i] = dk * (lo + hi);
        }
      }
    }
    __syncthreads();
    {
      // y += the block's correction: both 16-byte reads in flight before the adds
      constexpr int kY4 = kTok * kP / 4 / kThreads;
      float4 ry[kY4];
#pragma unroll
      for (int u = 0; u < kY4; ++u) {
        const int i = threadIdx.x + u * kThreads, k = i / (kP / 4), c4 = i % (kP / 4);
        if (k < m) ry[u] = *reinterpret_cast<const float4*>(&p.y[((size_t)(t0 + k) * p.H + h) * kP + 4 * c4]);
      }
#pragma unroll
      for (int u = 0; u < kY4; ++u) {
        const int i = threadIdx.x + u * kThreads, k = i / (kP / 4), c4 = i % (kP / 4);
        if (k < m) {
          const float4 c = *reinterpret_cast<const float4*>(&st.y[k][4 * c4]);
          *reinterpret_cast<float4*>(&p.y[((size_t)(t0 + k) * p.H + h) * kP + 4 * c4]) =
              make_float4(ry[u].x + c.x, ry[u].y + c.y, ry[u].z + c.z, ry[u].w + c.w);
        }
      }
    }
    // a sample starts here, or the received state has decayed to exact zeros
    if (m < n || dead) break;
  }
}

template <int N>
cudaError_t launch_n(const SsdParams& p, const SsdMaps* maps, cudaStream_t stream) {
  const size_t smem = sizeof(Stage<N>), smem_corr = sizeof(CorrStage<N>);
  static bool scan_configured[64] = {}, corr_configured[64] = {};
  cudaError_t e0 = ensure_smem_limit(ssd_chunk_scan_kernel<N>, (int)smem, scan_configured);
  if (e0 == cudaSuccess)
    e0 = ensure_smem_limit(ssd_correction_kernel<N>, (int)smem_corr, corr_configured);
  if (e0 != cudaSuccess) return e0;
  cudaError_t e;
  if (N == 128) {
    if (maps == nullptr) return cudaErrorInvalidValue;
    e = launch_ssd_chunk_scan_tc(p, *maps, stream);
  } else {
    TraceScope trace_scope(stream, "ssd_chunk_scan_kernel");
    ssd_chunk_scan_kernel<N><<<dim3(p.H, p.R), kThreads, smem, stream>>>(p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  {
    TraceScope trace_scope(stream, "ssd_state_pass_kernel");
    ssd_state_pass_kernel<<<p.H, kThreads, 0, stream>>>(p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess || p.R < 2) return e;
  if (N == 128) return launch_ssd_correction_tc(p, *maps, stream);
  {
    TraceScope trace_scope(stream, "ssd_correction_kernel");
    ssd_correction_kernel<N><<<dim3(p.H, p.R - 1), kThreads, smem_corr, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ssd_cp(const SsdParams& p, const SsdMaps* maps, cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  return p.N == 64 ? launch_n<64>(p, maps, stream) : launch_n<128>(p, maps, stream);
}

}  // namespace ra
