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
// Memory-bound: each (row, head) pair is D contiguous values, moved in chunks
// of 8 with 16-byte (bf16) or 2 x 16-byte (fp32) accesses.
// Pairs are numbered in memory order of o (row-major), so the grid streams
// o_a, o_b and the output front to back; the 4-byte lse accesses, strided by
// rows, are merged into full sectors in L2 (the lse arrays are 1/64 of the
// bytes at D = 128 in bf16).
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

// kC chunks of 8 values per thread (kC = min(4, D / 8)): every load of the
// thread (both lse values and 2 kC chunks of o) is issued before any is
// used, so each thread keeps up to 8 16-byte reads in flight.  Registers are
// capped for three blocks per SM (24 warps): at two blocks (86 registers) the
// kernel moved 4.6 TB/s, at three 5.9 TB/s.
template <int kC>
__global__ void __launch_bounds__(256, 3) lse_merge_kernel(const void* o_a, bool a_fp32,
                                                        const float* lse_a, const void* o_b,
                                                        bool b_fp32, const float* lse_b,
                                                        void* o_out, bool out_fp32,
                                                        float* lse_out, int rows, int heads,
                                                        int D, long long pairs, int* status) {
  const int tpp = D / (8 * kC);  // threads per (row, head) pair; divides 32
  const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long pair = gt / tpp;
  const int part = (int)(gt % tpp);
  const bool active = pair < pairs;
  float a = -INFINITY, b = -INFINITY;
  int h = 0, row = 0;
  Vec8 x[kC], y[kC];
  size_t idx = 0;
  const long long n_o = (long long)rows * heads * D, n_l = (long long)rows * heads;
  bool in = active;
  if (active) {
    row = (int)(pair / heads);
    h = (int)(pair % heads);
    const long long at = checked((long long)h * rows + row, n_l, status, kSiteMerge);
    a = lse_a[at];
    b = lse_b[at];
    idx = ((size_t)row * heads + h) * D + (size_t)part * 8 * kC;
    // the thread's last value lies inside o as well
    in = index_ok((long long)idx + 8 * kC - 1, n_o, status, kSiteMerge);
    // a side with lse = -inf is read too (its values are then not used)
    if (in) {
#pragma unroll
      for (int c = 0; c < kC; ++c) {
        x[c] = load8(o_a, a_fp32, idx + 8 * c);
        y[c] = load8(o_b, b_fp32, idx + 8 * c);
      }
    }
  }
  // every lane of the pair has read lse_a before any lane overwrites it
  __syncwarp();
  if (!in) return;
  const bool ea = a == -INFINITY, eb = b == -INFINITY;
  float L = -INFINITY, wa = 0.f, wb = 0.f;
  if (!ea && !eb) {
    const float mx = fmaxf(a, b);
    L = mx + log1pf(expf(-fabsf(a - b)));
    wa = expf(a - L);
    wb = expf(b - L);
  } else if (!ea) {
    L = a;
  } else if (!eb) {
    L = b;
  }
#pragma unroll
  for (int c = 0; c < kC; ++c) {
    Vec8 r;
    // an empty side contributes exactly nothing, whatever its o holds
#pragma unroll
    for (int i = 0; i < 8; ++i)
      r.x[i] = ea ? (eb ? 0.f : y[c].x[i])
                  : (eb ? x[c].x[i] : fmaf(wa, x[c].x[i], wb * y[c].x[i]));
    store8(o_out, out_fp32, idx + 8 * c, r);
  }
  if (part == 0 && index_ok((long long)h * rows + row, n_l, status, kSiteMerge))
    lse_out[(size_t)h * rows + row] = L;
}

// Both inputs fp32 (the stepwise forward's running result and a step's
// partial): one warp per (row, head) pair and 16 bytes per lane, so each load
// instruction of a warp reads one pair's D contiguous floats (512 B at
// D = 128; at D = 64 a half-warp per pair, two pairs per instruction); each
// warp keeps kPairs pairs' loads in flight before it computes.
template <int kD, int kPairs>
__global__ void __launch_bounds__(256) lse_merge_f32_kernel(const float* o_a, const float* lse_a,
                                                          const float* o_b, const float* lse_b,
                                                          void* o_out, bool out_fp32,
                                                          float* lse_out, int rows, int heads,
                                                          long long pairs, int* status) {
  constexpr int kLanes = kD / 4;        // lanes per pair
  constexpr int kPerWarp = 32 / kLanes;  // pairs per warp instruction
  const int lane = threadIdx.x & 31;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int sub = lane / kLanes, col = (lane % kLanes) * 4;
  const long long n_l = (long long)rows * heads;
  float4 x[kPairs], y[kPairs];
  float a[kPairs], b[kPairs];
  long long pr[kPairs];
#pragma unroll
  for (int i = 0; i < kPairs; ++i) {
    pr[i] = (warp * kPairs + i) * kPerWarp + sub;  // pair = row * heads + head
    a[i] = b[i] = -INFINITY;
    if (pr[i] < pairs && !index_ok(pr[i] * kD + col + 3, pairs * kD, status, kSiteMerge))
      pr[i] = pairs;  // (debug build) a failed check skips the pair
    if (pr[i] < pairs) {
      const int row = (int)(pr[i] / heads), h = (int)(pr[i] % heads);
      const long long at = checked((long long)h * rows + row, n_l, status, kSiteMerge);
      a[i] = lse_a[at];
      b[i] = lse_b[at];
      x[i] = *reinterpret_cast<const float4*>(o_a + pr[i] * kD + col);
      y[i] = *reinterpret_cast<const float4*>(o_b + pr[i] * kD + col);
    }
  }
  // every lane of a pair has read lse_a before any lane overwrites it
  __syncwarp();
#pragma unroll
  for (int i = 0; i < kPairs; ++i) {
    if (pr[i] >= pairs) continue;
    const bool ea = a[i] == -INFINITY, eb = b[i] == -INFINITY;
    float L = -INFINITY, wa = 0.f, wb = 0.f;
    if (!ea && !eb) {
      const float mx = fmaxf(a[i], b[i]);
      L = mx + log1pf(expf(-fabsf(a[i] - b[i])));
      wa = expf(a[i] - L);
      wb = expf(b[i] - L);
    } else if (!ea) {
      L = a[i];
      wa = 1.f;
    } else if (!eb) {
      L = b[i];
      wb = 1.f;
    }
    // an empty side contributes exactly nothing, whatever its o holds
    float r[4];
    const float xa[4] = {x[i].x, x[i].y, x[i].z, x[i].w}, yb[4] = {y[i].x, y[i].y, y[i].z, y[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      r[e] = ea ? (eb ? 0.f : yb[e]) : (eb ? xa[e] : fmaf(wa, xa[e], wb * yb[e]));
    const long long idx = pr[i] * kD + col;
    if (out_fp32) {
      *reinterpret_cast<float4*>(static_cast<float*>(o_out) + idx) = make_float4(r[0], r[1], r[2], r[3]);
    } else {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(r[0], r[1]), hi = __floats2bfloat162_rn(r[2], r[3]);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o_out) + idx) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
    if (col == 0) {
      const int row = (int)(pr[i] / heads), h = (int)(pr[i] % heads);
      lse_out[(size_t)h * rows + row] = L;
    }
  }
}

// The two halves of each split item of the fused forward.  One warp per row
// of a split query tile (CTA c covers rows 4 (c % 32) .. + 3 of tile
// (c / 32) % 2 of pair c / 64), so every row's loads are in flight at once;
// the lanes hold D / 32 consecutive values of the row, read and written with
// vector accesses.  Same merge rule as above, from the halves' fp32 slots
// into out (bf16 or fp32) and lse at the tile's rows.
template <int kD>
__global__ void __launch_bounds__(128) split_merge_kernel(const SplitPair* pairs,
                                                          const float* part_o,
                                                          const float* part_lse, void* out,
                                                          bool out_fp32, float* lse, int hq,
                                                          int lse_stride, int num_pairs,
                                                          int* status) {
  constexpr int kV = kD / 32;  // values per lane: 4 (D = 128) or 2 (D = 64)
  const int pair = blockIdx.x >> 6;
  const int x = (blockIdx.x >> 5) & 1;
  const int r = (blockIdx.x & 31) * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const SplitPair sp = pairs[checked(pair, num_pairs, status, kSiteSplitMerge)];
  if (r >= sp.qlen[x]) return;
  const long long n_slot = (long long)num_pairs * 2 * 256;  // rows of all partial slots
  const size_t sa = checked(((long long)sp.part[0] * 2 + x) * 128 + r, n_slot, status,
                            kSiteSplitMerge);
  const size_t sb = checked(((long long)sp.part[1] * 2 + x) * 128 + r, n_slot, status,
                            kSiteSplitMerge);
  const float a = part_lse[sa], b = part_lse[sb];
  float oa[kV], ob[kV];
  if constexpr (kV == 4) {
    const float4 va = reinterpret_cast<const float4*>(part_o + sa * kD)[lane];
    const float4 vb = reinterpret_cast<const float4*>(part_o + sb * kD)[lane];
    oa[0] = va.x; oa[1] = va.y; oa[2] = va.z; oa[3] = va.w;
    ob[0] = vb.x; ob[1] = vb.y; ob[2] = vb.z; ob[3] = vb.w;
  } else {
    const float2 va = reinterpret_cast<const float2*>(part_o + sa * kD)[lane];
    const float2 vb = reinterpret_cast<const float2*>(part_o + sb * kD)[lane];
    oa[0] = va.x; oa[1] = va.y;
    ob[0] = vb.x; ob[1] = vb.y;
  }
  const bool ea = a == -INFINITY, eb = b == -INFINITY;
  float L = -INFINITY, wa = 0.f, wb = 0.f;
  if (!ea && !eb) {
    const float mx = fmaxf(a, b);
    L = mx + log1pf(expf(-fabsf(a - b)));
    wa = expf(a - L);
    wb = expf(b - L);
  } else if (!ea) {
    L = a;
    wa = 1.f;
  } else if (!eb) {
    L = b;
    wb = 1.f;
  }
  float o[kV];
#pragma unroll
  for (int i = 0; i < kV; ++i) o[i] = (ea ? 0.f : wa * oa[i]) + (eb ? 0.f : wb * ob[i]);
  const int row = sp.q0[x] + r;
  if (!index_ok(row, lse_stride, status, kSiteSplitMerge) ||
      !index_ok(sp.head[x], hq, status, kSiteHead))
    return;
  const size_t at = ((size_t)row * hq + sp.head[x]) * kD + lane * kV;
  if (out_fp32) {
#pragma unroll
    for (int i = 0; i < kV; ++i) static_cast<float*>(out)[at + i] = o[i];
  } else if constexpr (kV == 4) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(o[0], o[1]);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(o[2], o[3]);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&lo);
    w.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + at) = w;
  } else {
    *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(out) + at) =
        __floats2bfloat162_rn(o[0], o[1]);
  }
  if (lane == 0) lse[(size_t)sp.head[x] * lse_stride + row] = L;
}

}  // namespace

cudaError_t launch_split_merge(const SplitPair* pairs, int num_pairs, const float* part_o,
                               const float* part_lse, void* out, bool out_fp32, float* lse,
                               int hq, int lse_stride, int D, int* status, cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  TraceScope trace_scope(stream, "split_merge_kernel");
  if (D == 128)
    split_merge_kernel<128><<<64 * num_pairs, 128, 0, stream>>>(
        pairs, part_o, part_lse, out, out_fp32, lse, hq, lse_stride, num_pairs, status);
  else if (D == 64)
    split_merge_kernel<64><<<64 * num_pairs, 128, 0, stream>>>(
        pairs, part_o, part_lse, out, out_fp32, lse, hq, lse_stride, num_pairs, status);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const void* o_a, bool a_fp32, const float* lse_a, const void* o_b,
                             bool b_fp32, const float* lse_b, void* o_out, bool out_fp32,
                             float* lse_out, int rows, int heads, int D, int* status,
                             cudaStream_t stream) {
  const long long pairs = (long long)rows * heads;
  if (pairs == 0) return cudaSuccess;
  if (a_fp32 && b_fp32 && (D == 128 || D == 64)) {
    constexpr int kPairs = 4;
    const long long warps = (pairs * (D / 4) / 32 + kPairs - 1) / kPairs;
    const unsigned grid = (unsigned)((warps * 32 + 255) / 256);
    TraceScope trace_scope(stream, "lse_merge_kernel");
    if (D == 128)
      lse_merge_f32_kernel<128, kPairs><<<grid, 256, 0, stream>>>(
          static_cast<const float*>(o_a), lse_a, static_cast<const float*>(o_b), lse_b, o_out,
          out_fp32, lse_out, rows, heads, pairs, status);
    else
      lse_merge_f32_kernel<64, kPairs><<<grid, 256, 0, stream>>>(
          static_cast<const float*>(o_a), lse_a, static_cast<const float*>(o_b), lse_b, o_out,
          out_fp32, lse_out, rows, heads, pairs, status);
    return cudaGetLastError();
  }
  const int chunks = D / 8 < 4 ? D / 8 : 4;
  const long long threads = pairs * (D / 8 / chunks);
  const int block = 256;
  const unsigned grid = (unsigned)((threads + block - 1) / block);
  TraceScope trace_scope(stream, "lse_merge_kernel");
  if (chunks == 4)
    lse_merge_kernel<4><<<grid, block, 0, stream>>>(o_a, a_fp32, lse_a, o_b, b_fp32, lse_b, o_out,
                                                    out_fp32, lse_out, rows, heads, D, pairs, status);
  else if (chunks == 2)
    lse_merge_kernel<2><<<grid, block, 0, stream>>>(o_a, a_fp32, lse_a, o_b, b_fp32, lse_b, o_out,
                                                    out_fp32, lse_out, rows, heads, D, pairs, status);
  else
    lse_merge_kernel<1><<<grid, block, 0, stream>>>(o_a, a_fp32, lse_a, o_b, b_fp32, lse_b, o_out,
                                                    out_fp32, lse_out, rows, heads, D, pairs, status);
  return cudaGetLastError();
}

}  // namespace ra
