// Internal launchers (host side).  Each returns the CUDA error of the launch.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "device_common.cuh"

namespace ra {

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device (`done` is the kernel's own per-device record).
template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel kernel, int bytes, bool (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

// fp32 forward on CUDA cores (D = 64 or 128).
cudaError_t launch_fwd_simt_fp32(const FwdParams& p, cudaStream_t stream);

// bf16 forward on tcgen05 tensor cores (D = 64 or 128).  The tensor maps describe
// q [T, Hq, D] and k, v [T, Hkv, D] with 64 x 1 x 128 boxes, 128 B swizzle.
cudaError_t launch_fwd_tc_bf16(const FwdParams& p, const CUtensorMap& map_q,
                               const CUtensorMap& map_k, const CUtensorMap& map_v,
                               cudaStream_t stream);

// Log-sum-exp merge of (o_b, lse_b) into (o_a, lse_a), written to
// (o_out, lse_out) (which may alias a).  o_* are [rows, heads, D]; each of
// them is fp32 when its *_fp32 flag is set, else bf16.  lse_* are [heads, rows].
cudaError_t launch_lse_merge(const void* o_a, bool a_fp32, const float* lse_a, const void* o_b,
                             bool b_fp32, const float* lse_b, void* o_out, bool out_fp32,
                             float* lse_out, int rows, int heads, int D, int* status,
                             cudaStream_t stream);

// Folds the two halves of each split item of the fused forward (fp32 partial
// slots) into out [T, Hq, D] (bf16, or fp32 when out_fp32) and lse [Hq, lse_stride].
cudaError_t launch_split_merge(const SplitPair* pairs, int num_pairs, const float* part_o,
                               const float* part_lse, void* out, bool out_fp32, float* lse,
                               int hq, int lse_stride, int D, int* status, cudaStream_t stream);

// D_i = dO_i . O_i into Dvec [Hq, T] (O, dO fp32 when `fp32`, else bf16).
cudaError_t launch_bwd_preprocess(const void* out, const void* dout, bool fp32, float* Dvec, int T,
                                  int hq, int D, int* status, cudaStream_t stream);

// bf16 backward on tcgen05 (D = 64 or 128): dQ (query-tile-major, over the forward
// plan) and dK, dV (key-tile-major, over the backward plan).  Tensor maps as
// for the forward, plus dout [T, Hq, D].
cudaError_t launch_bwd_tc_bf16(const BwdParams& p, const CUtensorMap& map_q,
                               const CUtensorMap& map_k, const CUtensorMap& map_v,
                               const CUtensorMap& map_do, cudaStream_t stream);

// One CTA whose single bounded wait is never satisfied: after the wait
// limit it records RA_ERR_TIMEOUT in *status and exits (failure-path test).
cudaError_t launch_wait_timeout_selftest(int* status, cudaStream_t stream);

// fp32 backward on CUDA cores (D = 64 or 128).
cudaError_t launch_bwd_simt_fp32(const BwdParams& p, cudaStream_t stream);

// Context-parallel selective scan (Mamba2 SSD): chunk scans, state passing
// and the additive correction (head_dim 64, state size 64 or 128).
// `maps` (host memory) describes C, B and x for the tensor-core chunk scan
// of state size 128 (see SsdMaps); it may be null for state size 64.
struct SsdMaps {
  CUtensorMap c;     // C [T, G, 128] fp32 as (state, group, token); box 128 x 1 x 32
  CUtensorMap c_sw;  // C as above; box 32 x 1 x 128, 128-byte swizzle
  CUtensorMap b;     // B, as c
  CUtensorMap x;     // x [T, H, 64] fp32 as (head dim, head, token); box 64 x 1 x 128
};
cudaError_t launch_ssd_cp(const SsdParams& p, const SsdMaps* maps, cudaStream_t stream);

// The chunk scan of launch_ssd_cp on the tensor cores (state size 128): y of
// every rank's chunk from a zero state, the chunks' final states and carries.
cudaError_t launch_ssd_chunk_scan_tc(const SsdParams& p, const SsdMaps& maps,
                                     cudaStream_t stream);

// The additive correction of launch_ssd_cp on the tensor cores (state size
// 128): y_t += exp(A sum dt) H_r C_t on ranks r >= 1 up to their chunk's first
// sample start.
cudaError_t launch_ssd_correction_tc(const SsdParams& p, const SsdMaps& maps,
                                     cudaStream_t stream);

}  // namespace ra
