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
//      there).
//   2. ssd_state_pass_kernel  (head): the ring of states, rank by rank:
//      H_0 = 0, H_r = carry_{r-1} H_{r-1} + S_{r-1} (what rank r would receive).
//   3. ssd_correction_kernel  (head, rank >= 1): y_t += exp(A sum_{chunk start
//      <= u <= t} dt_u) H_r C_t for the chunk's tokens before its first sample
//      start.
// Threads: 256 per CTA; the P = 64 rows of the state are spread over 4
// threads each: thread `sub` of a row owns columns 16 j + 4 sub + e (j < N/16,
// e < 4), so it reads B and C with 16-byte loads and the four threads of a
// row read 64 contiguous bytes (no bank conflicts).  A row's output is a
// 4-lane shuffle sum.  Inputs are staged in shared memory 32 tokens at a
// time, with each token's decay exp(dt A) computed once.
#include <cuda_runtime.h>

#include <cmath>

#include "launch.h"
#include "trace.h"

namespace ra {

namespace {

constexpr int kP = 64;       // head dimension
constexpr int kThreads = 256;
constexpr int kTok = 32;     // tokens staged per block

template <int N>
struct Stage {
  float x[kTok][kP];
  float B[kTok][N];
  float C[kTok][N];
  float dt[kTok];
  float decay[kTok];  // exp(dt A)
  int pos[kTok];
  float y[kTok][kP];
};

// Column of the state a thread's i-th entry holds (see the layout above).
__device__ __forceinline__ int ssd_col(int sub, int i) {
  return 16 * (i >> 2) + 4 * sub + (i & 3);
}

// Loads tokens [t0, t0 + n) of head h (group g) into shared memory.
template <int N, bool kWantX, bool kWantB>
__device__ __forceinline__ void stage_tokens(Stage<N>& st, const SsdParams& p, int h, int g, int t0,
                                             int n) {
  for (int i = threadIdx.x; i < n * kP; i += kThreads) {
    const int k = i / kP, c = i % kP;
    if (kWantX) st.x[k][c] = p.x[((size_t)(t0 + k) * p.H + h) * kP + c];
  }
  for (int i = threadIdx.x; i < n * N; i += kThreads) {
    const int k = i / N, c = i % N;
    const size_t o = ((size_t)(t0 + k) * p.G + g) * N + c;
    if (kWantB) st.B[k][c] = p.B[o];
    st.C[k][c] = p.C[o];
  }
  const float A = p.A[h];
  for (int k = threadIdx.x; k < n; k += kThreads) {
    const float d = p.dt[(size_t)(t0 + k) * p.H + h];
    st.dt[k] = d;
    st.decay[k] = expf(d * A);
    st.pos[k] = p.pos ? p.pos[t0 + k] : 1;
  }
}

template <int N>
__global__ void __launch_bounds__(kThreads) ssd_chunk_scan_kernel(const SsdParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Stage<N>& st = *reinterpret_cast<Stage<N>*>(smem_raw);
  constexpr int kCols = N / 4;
  const int h = blockIdx.x, r = blockIdx.y;
  const int g = h / (p.H / p.G);
  const int row = threadIdx.x >> 2, sub = threadIdx.x & 3;
  const int L = p.T / p.R;
  const int c0 = r * L;
  const float A = p.A[h];
  const float Dh = p.D ? p.D[h] : 0.f;
  float S[kCols];
#pragma unroll
  for (int i = 0; i < kCols; ++i) S[i] = 0.f;
  float logcarry = 0.f;  // A * sum dt over the chunk
  bool reset = false;    // a sample starts inside the chunk
  for (int t0 = c0; t0 < c0 + L; t0 += kTok) {
    const int n = min(kTok, c0 + L - t0);
    __syncthreads();  // the previous block's y has been written out
    stage_tokens<N, true, true>(st, p, h, g, t0, n);
    __syncthreads();
    for (int k = 0; k < n; ++k) {
      if (st.pos[k] == 0) {
#pragma unroll
        for (int i = 0; i < kCols; ++i) S[i] = 0.f;
        reset = true;
        logcarry = 0.f;
      }
      const float d = st.dt[k];
      const float a = st.decay[k];
      logcarry += d * A;
      const float dx = d * st.x[k][row];
      float acc4[4] = {0.f, 0.f, 0.f, 0.f};  // four chains: the sum is not one long dependency
#pragma unroll
      for (int j = 0; j < kCols / 4; ++j) {
        const float4 b4 = *reinterpret_cast<const float4*>(&st.B[k][ssd_col(sub, 4 * j)]);
        const float4 c4 = *reinterpret_cast<const float4*>(&st.C[k][ssd_col(sub, 4 * j)]);
        const float bb[4] = {b4.x, b4.y, b4.z, b4.w}, cc[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float& s_ = S[4 * j + e];
          s_ = fmaf(a, s_, dx * bb[e]);
          acc4[e] = fmaf(s_, cc[e], acc4[e]);
        }
      }
      float acc = (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (sub == 0) st.y[k][row] = fmaf(Dh, st.x[k][row], acc);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n * kP; i += kThreads) {
      const int k = i / kP, c = i % kP;
      p.y[((size_t)(t0 + k) * p.H + h) * kP + c] = st.y[k][c];
    }
  }
  // the chunk's final state and the factor an incoming state survives with
  float* Sout = p.chunk_state + (((size_t)r * p.H + h) * kP + row) * N;
#pragma unroll
  for (int i = 0; i < kCols; ++i) Sout[ssd_col(sub, i)] = S[i];
  if (threadIdx.x == 0) p.carry[(size_t)r * p.H + h] = reset ? 0.f : expf(logcarry);
}

// H_r for every rank r >= 1 (into incoming[r]) and, if asked, the state after
// the last rank.  One CTA per head; each thread owns P N / 256 entries.
__global__ void __launch_bounds__(kThreads) ssd_state_pass_kernel(const SsdParams p) {
  const int h = blockIdx.x;
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

template <int N>
__global__ void __launch_bounds__(kThreads) ssd_correction_kernel(const SsdParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Stage<N>& st = *reinterpret_cast<Stage<N>*>(smem_raw);
  constexpr int kCols = N / 4;
  const int h = blockIdx.x, r = blockIdx.y + 1;
  const int g = h / (p.H / p.G);
  const int row = threadIdx.x >> 2, sub = threadIdx.x & 3;
  const int L = p.T / p.R;
  const int c0 = r * L;
  const float A = p.A[h];
  float Hin[kCols];
  const float* src = p.incoming + (((size_t)r * p.H + h) * kP + row) * N;
#pragma unroll
  for (int i = 0; i < kCols; ++i) Hin[i] = src[ssd_col(sub, i)];
  float lam = 0.f;  // A * sum dt from the chunk start
  bool done = false;
  for (int t0 = c0; t0 < c0 + L && !done; t0 += kTok) {
    const int n = min(kTok, c0 + L - t0);
    __syncthreads();
    stage_tokens<N, false, false>(st, p, h, g, t0, n);
    __syncthreads();
    int m = n;  // tokens of this block before the first sample start
    for (int k = 0; k < n; ++k) {
      if (st.pos[k] == 0) {
        m = k;
        done = true;
        break;
      }
      lam = fmaf(st.dt[k], A, lam);
      const float decay = expf(lam);
      float acc4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < kCols / 4; ++j) {
        const float4 c4 = *reinterpret_cast<const float4*>(&st.C[k][ssd_col(sub, 4 * j)]);
        acc4[0] = fmaf(Hin[4 * j], c4.x, acc4[0]);
        acc4[1] = fmaf(Hin[4 * j + 1], c4.y, acc4[1]);
        acc4[2] = fmaf(Hin[4 * j + 2], c4.z, acc4[2]);
        acc4[3] = fmaf(Hin[4 * j + 3], c4.w, acc4[3]);
      }
      float acc = (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (sub == 0) st.y[k][row] = decay * acc;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < m * kP; i += kThreads) {
      const int k = i / kP, c = i % kP;
      p.y[((size_t)(t0 + k) * p.H + h) * kP + c] += st.y[k][c];
    }
  }
}

template <int N>
cudaError_t launch_n(const SsdParams& p, cudaStream_t stream) {
  const size_t smem = sizeof(Stage<N>);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(ssd_chunk_scan_kernel<N>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(ssd_correction_kernel<N>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  {
    TraceScope trace_scope(stream, "ssd_chunk_scan_kernel");
    ssd_chunk_scan_kernel<N><<<dim3(p.H, p.R), kThreads, smem, stream>>>(p);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    TraceScope trace_scope(stream, "ssd_state_pass_kernel");
    ssd_state_pass_kernel<<<p.H, kThreads, 0, stream>>>(p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess || p.R < 2) return e;
  {
    TraceScope trace_scope(stream, "ssd_correction_kernel");
    ssd_correction_kernel<N><<<dim3(p.H, p.R - 1), kThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ssd_cp(const SsdParams& p, cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  return p.N == 64 ? launch_n<64>(p, stream) : launch_n<128>(p, stream);
}

}  // namespace ra
