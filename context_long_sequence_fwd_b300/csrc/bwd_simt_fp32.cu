// fp32 ring-attention backward on CUDA cores (fp32 arithmetic throughout).
//
// Same split as the tensor-core backward, so no output needs atomics:
//   bwd_dq_simt    one thread per query row (forward plan items, 2 x 128 rows
//                  per CTA), keys staged 32 at a time in shared memory:
//                  dQ_i = scale sum_j P_ij (dP_ij - D_i) k_j
//   bwd_dkdv_simt  one thread per key of a 128-key tile (backward plan items),
//                  query rows of every head of the group staged 32 at a time:
//                  dV_j = sum P_ij dO_i, dK_j = scale sum dS_ij q_i
// with P_ij = exp(scale q_i.k_j - lse_i), dP_ij = dO_i . v_j, D_i = dO_i . O_i.
#include <cuda_runtime.h>

#include <cmath>

#include "device_common.cuh"
#include "launch.h"
#include "trace.h"

namespace ra {

namespace {

constexpr int kRows = 32;

template <int D>
__global__ void __launch_bounds__(256) bwd_dq_simt_kernel(BwdParams p) {
  __shared__ float Ks[kRows][D];
  __shared__ float Vs[kRows][D];
  const PlanItem it = p.items[checked(blockIdx.x, p.num_items, p.status, kSiteSimtBwd)];
  const int tile = threadIdx.x >> 7, r = threadIdx.x & 127;
  const int row = it.q0[tile] + r;
  const int h = it.head[tile];
  const bool valid = r < it.qlen[tile] && index_ok(row, p.q_rows, p.status, kSiteSimtBwd) &&
                     index_ok(h, p.hq, p.status, kSiteHead);
  const int g = it.head[0] / p.group;
  const float* q = static_cast<const float*>(p.q);
  const float* k = static_cast<const float*>(p.k);
  const float* v = static_cast<const float*>(p.v);
  const float* dout = static_cast<const float*>(p.dout);
  float qr[D], dor[D], dq[D];
  int lo = 0, hi = 0;
  float lse = 0.f, Dv = 0.f;
  if (valid) {
    int ds, de;
    doc_bounds(p.cu, p.num_docs, row, &ds, &de);
    lo = ds;
    hi = p.causal ? row + 1 : de;
    const long long at = checked((long long)h * p.lse_stride + row,
                                 (long long)p.hq * p.lse_stride, p.status, kSiteSimtBwd);
    lse = p.lse[at];
    Dv = p.Dvec[at];
  }
#pragma unroll
  for (int d = 0; d < D; ++d) {
    const size_t o = ((size_t)row * p.hq + h) * D + d;
    qr[d] = valid ? q[o] : 0.f;
    dor[d] = valid ? dout[o] : 0.f;
    dq[d] = 0.f;
  }
  for (int si = 0; si < it.seg_count; ++si) {
    const PlanSegment sg = p.segs[checked(it.seg_begin + si, p.num_segs, p.status, kSiteSimtBwd)];
    const int a = max(lo, sg.k0), b = min(hi, sg.k1);
    for (int kt = sg.k0; kt < sg.k1; kt += kRows) {
      __syncthreads();
      for (int x = threadIdx.x; x < kRows * D; x += blockDim.x) {
        const int jj = x / D, d = x % D, key = kt + jj;
        const bool in = key < sg.k1 && index_ok(key, p.k_rows, p.status, kSiteSimtBwd);
        Ks[jj][d] = in ? k[((size_t)key * p.hkv + g) * D + d] : 0.f;
        Vs[jj][d] = in ? v[((size_t)key * p.hkv + g) * D + d] : 0.f;
      }
      __syncthreads();
      for (int jj = 0; jj < kRows; ++jj) {
        const int key = kt + jj;
        if (key < a || key >= b) continue;
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int d = 0; d < D; ++d) {
          s = fmaf(qr[d], Ks[jj][d], s);
          dp = fmaf(dor[d], Vs[jj][d], dp);
        }
        const float pij = expf(s * p.scale - lse);
        const float dsij = pij * (dp - Dv);
#pragma unroll
        for (int d = 0; d < D; ++d) dq[d] = fmaf(dsij, Ks[jj][d], dq[d]);
      }
    }
  }
  if (!valid) return;
  float* out = static_cast<float*>(p.dq) + ((size_t)row * p.hq + h) * D;
#pragma unroll
  for (int d = 0; d < D; ++d) out[d] = dq[d] * p.scale;
}

template <int D>
__global__ void __launch_bounds__(128) bwd_dkdv_simt_kernel(BwdParams p) {
  __shared__ float Qs[kRows][D];
  __shared__ float Os[kRows][D];  // dO rows
  __shared__ float Ls[kRows], Ds[kRows];
  __shared__ int Lo[kRows], Hi[kRows];
  const BwdItem it = p.bitems[checked(blockIdx.x, p.num_bitems, p.status, kSiteSimtBwd)];
  const int g = it.kv_head;
  const int kr = threadIdx.x;
  const int j = it.k0 + kr;
  const bool valid = kr < it.klen && index_ok(j, p.k_rows, p.status, kSiteSimtBwd) &&
                     index_ok(g, p.hkv, p.status, kSiteHead);
  const float* q = static_cast<const float*>(p.q);
  const float* k = static_cast<const float*>(p.k);
  const float* v = static_cast<const float*>(p.v);
  const float* dout = static_cast<const float*>(p.dout);
  float kk[D], vv[D], dk[D], dv[D];
#pragma unroll
  for (int d = 0; d < D; ++d) {
    const size_t o = ((size_t)j * p.hkv + g) * D + d;
    kk[d] = valid ? k[o] : 0.f;
    vv[d] = valid ? v[o] : 0.f;
    dk[d] = 0.f;
    dv[d] = 0.f;
  }
  for (int si = 0; si < it.seg_count; ++si) {
    const BwdSegment sg = p.bsegs[checked(it.seg_begin + si, p.num_bsegs, p.status, kSiteSimtBwd)];
    for (int i0 = sg.q0; i0 < sg.q1; i0 += kRows) {
      for (int h = g * p.group; h < (g + 1) * p.group; ++h) {
        __syncthreads();
        for (int x = threadIdx.x; x < kRows * D; x += blockDim.x) {
          const int rr = x / D, d = x % D, i = i0 + rr;
          const bool in = i < sg.q1 && index_ok(i, p.q_rows, p.status, kSiteSimtBwd);
          Qs[rr][d] = in ? q[((size_t)i * p.hq + h) * D + d] : 0.f;
          Os[rr][d] = in ? dout[((size_t)i * p.hq + h) * D + d] : 0.f;
        }
        if (threadIdx.x < kRows) {
          const int i = i0 + threadIdx.x;
          int lo = 0, hi = 0;
          float l = 0.f, dd = 0.f;
          if (i < sg.q1) {
            int ds, de;
            doc_bounds(p.cu, p.num_docs, i, &ds, &de);
            lo = ds;
            hi = p.causal ? i + 1 : de;
            const long long at = checked((long long)h * p.lse_stride + i,
                                         (long long)p.hq * p.lse_stride, p.status, kSiteSimtBwd);
            l = p.lse[at];
            dd = p.Dvec[at];
          }
          Lo[threadIdx.x] = lo;
          Hi[threadIdx.x] = hi;
          Ls[threadIdx.x] = l;
          Ds[threadIdx.x] = dd;
        }
        __syncthreads();
        for (int rr = 0; rr < kRows; ++rr) {
          if (j < Lo[rr] || j >= Hi[rr]) continue;
          float s = 0.f, dp = 0.f;
#pragma unroll
          for (int d = 0; d < D; ++d) {
            s = fmaf(Qs[rr][d], kk[d], s);
            dp = fmaf(Os[rr][d], vv[d], dp);
          }
          const float pij = expf(s * p.scale - Ls[rr]);
          const float dsij = pij * (dp - Ds[rr]);
#pragma unroll
          for (int d = 0; d < D; ++d) {
            dv[d] = fmaf(pij, Os[rr][d], dv[d]);
            dk[d] = fmaf(dsij, Qs[rr][d], dk[d]);
          }
        }
      }
    }
  }
  if (!valid) return;
  float* odk = static_cast<float*>(p.dk) + ((size_t)j * p.hkv + g) * D;
  float* odv = static_cast<float*>(p.dv) + ((size_t)j * p.hkv + g) * D;
#pragma unroll
  for (int d = 0; d < D; ++d) {
    odk[d] = dk[d] * p.scale;
    odv[d] = dv[d];
  }
}

}  // namespace

cudaError_t launch_bwd_simt_fp32(const BwdParams& p, cudaStream_t stream) {
  if (p.num_items > 0) {
    TraceScope trace_scope(stream, "bwd_dq_simt_kernel");
    if (p.D == 64)
      bwd_dq_simt_kernel<64><<<p.num_items, 256, 0, stream>>>(p);
    else
      bwd_dq_simt_kernel<128><<<p.num_items, 256, 0, stream>>>(p);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.num_bitems > 0) {
    TraceScope trace_scope(stream, "bwd_dkdv_simt_kernel");
    if (p.D == 64)
      bwd_dkdv_simt_kernel<64><<<p.num_bitems, 128, 0, stream>>>(p);
    else
      bwd_dkdv_simt_kernel<128><<<p.num_bitems, 128, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace ra
