// Log-sum-exp merge of two partial attention results over disjoint key sets.
//
// This is how the pages' ring steps are aggregated (axolotl "Sequence
// Parallelism" page, introduction: each shard's partial result is combined
// through the ring).  Per (row, head):
//   lse = max(a, b) + log1p(exp(-|a - b|)),
//   o   = exp(a - lse) o_a + exp(b - lse) o_b,
// a side with lse = -inf (no visible key) contributes nothing, and two empty
// sides give o = 0, lse = -inf.
//
// Memory-bound: each (row, head) pair is D contiguous values; a group of D/8
// threads moves them with 16-byte (bf16) or 2 x 16-byte (fp32) accesses.
// Pairs are numbered head-major so that the lse reads/writes of a warp are
// contiguous.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "launch.h"
#include "trace.h"

namespace ra {

namespace {

struct Vec8 {
  float x[8];
};

__device__ __forceinline__ Vec8 load8(const void* base, bool fp32, size_t idx) {
  Vec8 r;
  if (fp32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
    const float4 a = p[0], b = p[1];
    r.x[0] = a.x; r.x[1] = a.y; r.x[2] = a.z; r.x[3] = a.w;
    r.x[4] = b.x; r.x[5] = b.y; r.x[6] = b.z; r.x[7] = b.w;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + idx);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      r.x[2 * i] = __uint_as_float(w[i] << 16);
      r.x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  return r;
}

__device__ __forceinline__ void store8(void* base, bool fp32, size_t idx, const Vec8& r) {
  if (fp32) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + idx);
    p[0] = make_float4(r.x[0], r.x[1], r.x[2], r.x[3]);
    p[1] = make_float4(r.x[4], r.x[5], r.x[6], r.x[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(r.x[2 * i], r.x[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + idx) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__global__ void __launch_bounds__(256) lse_merge_kernel(const void* o_a, bool a_fp32,
                                                        const float* lse_a, const void* o_b,
                                                        bool b_fp32, const float* lse_b,
                                                        void* o_out, bool out_fp32,
                                                        float* lse_out, int rows, int heads,
                                                        int D, long long pairs) {
  const int tpp = D / 8;  // threads per (row, head) pair; divides 32
  const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long pair = gt / tpp;
  const int part = (int)(gt % tpp);
  const bool active = pair < pairs;
  float a = -INFINITY, b = -INFINITY;
  int h = 0, row = 0;
  if (active) {
    h = (int)(pair / rows);
    row = (int)(pair % rows);
    a = lse_a[(size_t)h * rows + row];
    b = lse_b[(size_t)h * rows + row];
  }
  // every lane of the pair has read lse_a before any lane overwrites it
  __syncwarp();
  if (!active) return;
  const size_t idx = ((size_t)row * heads + h) * D + (size_t)part * 8;
  Vec8 r;
  float L;
  if (a == -INFINITY && b == -INFINITY) {
#pragma unroll
    for (int i = 0; i < 8; ++i) r.x[i] = 0.f;
    L = -INFINITY;
  } else if (b == -INFINITY) {
    r = load8(o_a, a_fp32, idx);
    L = a;
  } else if (a == -INFINITY) {
    r = load8(o_b, b_fp32, idx);
    L = b;
  } else {
    const float mx = fmaxf(a, b);
    L = mx + log1pf(expf(-fabsf(a - b)));
    const float wa = expf(a - L), wb = expf(b - L);
    const Vec8 x = load8(o_a, a_fp32, idx), y = load8(o_b, b_fp32, idx);
#pragma unroll
    for (int i = 0; i < 8; ++i) r.x[i] = fmaf(wa, x.x[i], wb * y.x[i]);
  }
  store8(o_out, out_fp32, idx, r);
  if (part == 0) lse_out[(size_t)h * rows + row] = L;
}

}  // namespace

cudaError_t launch_lse_merge(const void* o_a, bool a_fp32, const float* lse_a, const void* o_b,
                             bool b_fp32, const float* lse_b, void* o_out, bool out_fp32,
                             float* lse_out, int rows, int heads, int D, cudaStream_t stream) {
  const long long pairs = (long long)rows * heads;
  if (pairs == 0) return cudaSuccess;
  const long long threads = pairs * (D / 8);
  const int block = 256;
  const long long grid = (threads + block - 1) / block;
  TraceScope trace_scope(stream, "lse_merge_kernel");
  lse_merge_kernel<<<(unsigned)grid, block, 0, stream>>>(o_a, a_fp32, lse_a, o_b, b_fp32, lse_b,
                                                         o_out, out_fp32, lse_out, rows, heads, D,
                                                         pairs);
  return cudaGetLastError();
}

}  // namespace ra
