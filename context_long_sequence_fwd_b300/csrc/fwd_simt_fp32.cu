// fp32 ring-attention forward on CUDA cores.
//
// Used for fp32 inputs, where the result must match exact attention to about
// 1e-5: tensor-core tf32 cannot, so this path keeps every product and sum in
// fp32.  One CTA walks one planner item: 256 threads, one query row each
// (threads 0-127 tile A, 128-255 tile B); K/V tiles of 32 keys are staged in
// shared memory and shared by both tiles (they read the same K/V head).  The
// online softmax (running max m, sum l, output o) is carried across tiles and
// ring steps, which is the log-sum-exp merge of the per-step results.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "device_common.cuh"
#include "launch.h"
#include "trace.h"

namespace ra {

namespace {

constexpr int kKeys = 32;

template <int D>
__global__ void __launch_bounds__(256) fwd_simt_fp32_kernel(FwdParams p) {
  __shared__ float Ks[kKeys][D];
  __shared__ float Vs[kKeys][D];
  const PlanItem it = p.items[checked(blockIdx.x, p.num_items, p.status, kSiteSimtFwd)];
  const int tile = threadIdx.x >> 7, r = threadIdx.x & 127;
  const int row = it.q0[tile] + r;
  const int h = it.head[tile];
  const bool valid = r < it.qlen[tile] && index_ok(row, p.q_rows, p.status, kSiteSimtFwd) &&
                     index_ok(h, p.hq, p.status, kSiteHead);
  const int g = it.head[0] / p.group;
  const float* q = static_cast<const float*>(p.q);
  const float* k = static_cast<const float*>(p.k);
  const float* v = static_cast<const float*>(p.v);

  int lo = 0, hi = 0;
  float qr[D];
  if (valid) {
    row_key_interval(p, row, &lo, &hi);
    const float* qp = q + ((size_t)row * p.hq + h) * D;
#pragma unroll
    for (int d = 0; d < D; ++d) qr[d] = qp[d];
  } else {
#pragma unroll
    for (int d = 0; d < D; ++d) qr[d] = 0.f;
  }
  float o[D];
#pragma unroll
  for (int d = 0; d < D; ++d) o[d] = 0.f;
  float m = -INFINITY, l = 0.f;

  for (int si = 0; si < it.seg_count; ++si) {
    const PlanSegment seg = p.segs[checked(it.seg_begin + si, p.num_segs, p.status, kSiteSimtFwd)];
    if (!seg_selected(seg, p.step_filter)) continue;
    const int a = max(lo, seg.k0), b = min(hi, seg.k1);
    for (int kt = seg.k0; kt < seg.k1; kt += kKeys) {
      __syncthreads();
      for (int x = threadIdx.x; x < kKeys * D; x += blockDim.x) {
        const int j = x / D, d = x % D, key = kt + j;
        float kv = 0.f, vv = 0.f;
        if (key < seg.k1 && index_ok(key, p.k_rows, p.status, kSiteSimtFwd)) {
          kv = k[((size_t)key * p.hkv + g) * D + d];
          vv = v[((size_t)key * p.hkv + g) * D + d];
        }
        Ks[j][d] = kv;
        Vs[j][d] = vv;
      }
      __syncthreads();
      float s[kKeys];
      float tmax = -INFINITY;
#pragma unroll 4
      for (int j = 0; j < kKeys; ++j) {
        const int key = kt + j;
        float acc = 0.f;
#pragma unroll
        for (int d = 0; d < D; ++d) acc = fmaf(qr[d], Ks[j][d], acc);
        s[j] = (key >= a && key < b) ? acc * p.scale : -INFINITY;
        tmax = fmaxf(tmax, s[j]);
      }
      if (tmax != -INFINITY) {
        const float m_new = fmaxf(m, tmax);
        const float alpha = expf(m - m_new);  // 0 when m = -inf
        l *= alpha;
#pragma unroll
        for (int d = 0; d < D; ++d) o[d] *= alpha;
        for (int j = 0; j < kKeys; ++j) {
          const float pj = expf(s[j] - m_new);  // 0 for masked keys
          l += pj;
#pragma unroll
          for (int d = 0; d < D; ++d) o[d] = fmaf(pj, Vs[j][d], o[d]);
        }
        m = m_new;
      }
    }
  }

  if (!valid) return;
  const size_t ob = ((size_t)row * p.hq + h) * D;
  const bool empty = !(l > 0.f);
  if (p.out_fp32) {
    float* out = static_cast<float*>(p.out);
#pragma unroll
    for (int d = 0; d < D; ++d) out[ob + d] = empty ? 0.f : o[d] / l;
  } else {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
    for (int d = 0; d < D; ++d) out[ob + d] = __float2bfloat16_rn(empty ? 0.f : o[d] / l);
  }
  if (index_ok((long long)h * p.lse_stride + row, (long long)p.hq * p.lse_stride, p.status,
               kSiteSimtFwd))
    p.lse[(size_t)h * p.lse_stride + row] = empty ? -INFINITY : m + logf(l);
}

}  // namespace

cudaError_t launch_fwd_simt_fp32(const FwdParams& p, cudaStream_t stream) {
  if (p.num_items == 0) return cudaSuccess;
  TraceScope trace_scope(stream, "fwd_simt_fp32_kernel");
  if (p.D == 64)
    fwd_simt_fp32_kernel<64><<<p.num_items, 256, 0, stream>>>(p);
  else
    fwd_simt_fp32_kernel<128><<<p.num_items, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ra
