// Backward preprocess: D_i = sum_d dO[i,h,d] * O[i,h,d] for every (head, row).
//
// D_i equals sum_j P_ij dP_ij (the row sums of P o dP), which the backward
// needs in dS_ij = P_ij (dP_ij - D_i); computing it from O and dO costs one
// read of each instead of a pass over the keys.  Memory-bound: a group of
// D/32 threads reads one row of O and of dO, four 16-byte (bf16) or 2 x
// 16-byte (fp32) loads of each per thread, and reduces with shuffles; (row, head) pairs are numbered in
// memory order of O, so the grid streams O and dO front to back (the 4-byte
// D stores, strided by T, are merged into full sectors in L2).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "trace.h"

namespace ra {

namespace {

template <bool kF32>
__device__ __forceinline__ float dot8(const void* a, const void* b, size_t idx) {
  float s = 0.f;
  if (kF32) {
    const float4* pa = reinterpret_cast<const float4*>(static_cast<const float*>(a) + idx);
    const float4* pb = reinterpret_cast<const float4*>(static_cast<const float*>(b) + idx);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float4 x = pa[i], y = pb[i];
      s = fmaf(x.x, y.x, s);
      s = fmaf(x.y, y.y, s);
      s = fmaf(x.z, y.z, s);
      s = fmaf(x.w, y.w, s);
    }
  } else {
    const uint4 x = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a) + idx);
    const uint4 y = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(b) + idx);
    const uint32_t wx[4] = {x.x, x.y, x.z, x.w}, wy[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s = fmaf(__uint_as_float(wx[i] << 16), __uint_as_float(wy[i] << 16), s);
      s = fmaf(__uint_as_float(wx[i] & 0xFFFF0000u), __uint_as_float(wy[i] & 0xFFFF0000u), s);
    }
  }
  return s;
}

// Four chunks of 8 values per thread, all loads issued before the sums.
constexpr int kChunks = 4;

template <bool kF32>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const void* out, const void* dout,
                                                             float* Dvec, int T, int hq, int D,
                                                             long long rows, int* status) {
  const int tpr = D / (8 * kChunks);  // threads per row; divides 32
  const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long r = gt / tpr;
  const int part = (int)(gt % tpr);
  float s = 0.f;
  int h = 0, i = 0;
  const bool in = r < rows && index_ok(r * D + (long long)(part + 1) * 8 * kChunks - 1,
                                       rows * D, status, kSitePreprocess);
  if (in) {
    i = (int)(r / hq);
    h = (int)(r % hq);
    const size_t idx = ((size_t)i * hq + h) * D + (size_t)part * 8 * kChunks;
    float t[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) t[c] = dot8<kF32>(out, dout, idx + 8 * c);
    s = (t[0] + t[1]) + (t[2] + t[3]);
  }
  for (int off = tpr / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (in && part == 0 && index_ok((long long)h * T + i, rows, status, kSitePreprocess))
    Dvec[(size_t)h * T + i] = s;
}

}  // namespace

cudaError_t launch_bwd_preprocess(const void* out, const void* dout, bool fp32, float* Dvec, int T,
                                  int hq, int D, int* status, cudaStream_t stream) {
  const long long rows = (long long)T * hq;
  if (rows == 0) return cudaSuccess;
  const long long threads = rows * (D / (8 * kChunks));
  const long long grid = (threads + 255) / 256;
  TraceScope trace_scope(stream, "bwd_preprocess_kernel");
  if (fp32)
    bwd_preprocess_kernel<true><<<(unsigned)grid, 256, 0, stream>>>(out, dout, Dvec, T, hq, D, rows, status);
  else
    bwd_preprocess_kernel<false><<<(unsigned)grid, 256, 0, stream>>>(out, dout, Dvec, T, hq, D, rows, status);
  return cudaGetLastError();
}

}  // namespace ra
