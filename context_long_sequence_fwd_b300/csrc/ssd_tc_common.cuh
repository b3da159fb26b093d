// Helpers shared by the tensor-core kernels of the Mamba2 selective scan
// (ssd_chunk_tc.cu, ssd_correction_tc.cu): fp16 hi + lo splitting of fp32
// operands, their 128-byte-swizzled shared-memory layout and descriptors,
// the three-product MMA of a split pair, and float-float sums.
#pragma once
#include <cuda_fp16.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace ra {
namespace ssd_tc {

// Instruction descriptor of kind::f16 with fp16 A and B (format 0) and fp32
// accumulation; a_mn, b_mn: operand stored MN-major.
__host__ __device__ constexpr uint32_t make_idesc_f16(uint32_t m, uint32_t n, bool a_mn,
                                                      bool b_mn) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((n >> 3) << 17) |
         ((m >> 4) << 24);
}
// Byte offset of 16-byte chunk kc (values 8 kc .. 8 kc + 7 along the row) of
// row `row` of an operand of `rows` rows: 64-value blocks of rows x 128 B,
// 8-row atoms of 1024 B, chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t sw_chunk(int rows, int row, int kc) {
  const int blk = kc >> 3, c = kc & 7;
  return static_cast<uint32_t>(blk * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 +
                               ((c ^ (row & 7)) << 4));
}

// An operand in shared memory: hi part at `base`, lo part `lo` bytes on.
//   K-major:  rows along M (or N), 128 values of K; `blk` = bytes of one
//             64-value K block (rows x 128).
//   MN-major: rows along K (16 per MMA step), 64 values of M (or N) per 128-B
//             row; `blk` = bytes between 64-wide M (or N) blocks.
struct Operand {
  uint32_t base, lo, blk;
  bool mn;
};

__device__ __forceinline__ uint64_t op_desc(const Operand& o, bool lo_part, int kk) {
  const uint32_t a = o.base + (lo_part ? o.lo : 0u);
  return o.mn ? make_sdesc_sw128(a + kk * 2048, o.blk, 1024)
              : make_sdesc_sw128(a + (kk >> 2) * o.blk + (kk & 3) * 32, 16, 1024);
}

// D (+)= A B over K = 128 with split operands: hi hi, hi lo, lo hi.
// (mma_bf16_ss issues kind::f16; the fp16 type comes from the descriptor.)
__device__ __forceinline__ void mma_split(uint32_t d_tmem, const Operand& a, const Operand& b,
                                          uint32_t idesc, bool accumulate) {
#pragma unroll
  for (int pass = 0; pass < 3; ++pass) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16_ss(d_tmem, op_desc(a, pass == 2, kk), op_desc(b, pass == 1, kk), idesc,
                  (accumulate || pass > 0 || kk > 0) ? 1u : 0u);
  }
}

// The same with A's split parts in TMEM (hi at a_hi, lo at a_lo: 128 lanes
// x 64 columns each, two fp16 per column, K index 2c in the low half of
// column c) and B in shared memory.
__device__ __forceinline__ void mma_split_ta(uint32_t d_tmem, uint32_t a_hi, uint32_t a_lo,
                                             const Operand& b, uint32_t idesc, bool accumulate) {
#pragma unroll
  for (int pass = 0; pass < 3; ++pass) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16_ts(d_tmem, (pass == 2 ? a_lo : a_hi) + kk * 8, op_desc(b, pass == 1, kk), idesc,
                  (accumulate || pass > 0 || kk > 0) ? 1u : 0u);
  }
}

// Waits for the MMAs committed to `bar` (phase `parity`): thread 0 polls the
// mbarrier (bounded) and the rest of the CTA waits at a barrier, which does
// not compete with the tensor core for shared-memory bandwidth the way 512
// polling threads do.  Returns false for the whole CTA if the wait gave up.
// The threads read the results (TMEM) after tcgen05.fence::after_thread_sync.
__device__ __forceinline__ bool cta_wait_mma(uint64_t* bar, uint32_t parity, int* status) {
  bool ok = true;
  if (threadIdx.x == 0) ok = mbar_wait(bar, parity, status, nullptr);
  return __syncthreads_and(ok) != 0;
}

// hi + lo split of a pair of fp32 values into fp16 pairs.  hi is x rounded
// to 11 significant bits by Veltkamp's splitting (c = (2^13 + 1) x,
// hi = c - (c - x), in fp32 arithmetic, each step rounded on its own: the
// _rn intrinsics are never fused into an FMA), so it converts to fp16
// exactly wherever fp16 is normal; lo = x - hi is exact in fp32 and rounded
// once to fp16.  One packed conversion per pair and part.
__device__ __forceinline__ float veltkamp_hi(float x) {
  const float c = __fmul_rn(x, 8193.f);
  return __fsub_rn(c, __fsub_rn(c, x));
}
__device__ __forceinline__ void split2(float a, float b, uint32_t* hi, uint32_t* lo) {
  const float ha = veltkamp_hi(a), hb = veltkamp_hi(b);
  const __half2 h = __floats2half2_rn(ha, hb);
  const __half2 l = __floats2half2_rn(__fsub_rn(a, ha), __fsub_rn(b, hb));
  *hi = *reinterpret_cast<const uint32_t*>(&h);
  *lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Splits 8 fp32 values into fp16 hi and lo parts, 16 bytes each.
__device__ __forceinline__ void split8(const float (&v)[8], uint4* hi, uint4* lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) split2(v[2 * i], v[2 * i + 1], &h[i], &l[i]);
  *hi = make_uint4(h[0], h[1], h[2], h[3]);
  *lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void unpack8(const float4& a, const float4& b, float (&v)[8]) {
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// (ah, al) += (bh, bl) in float-float arithmetic: the sum's rounding error
// is carried in the lo word (two-sum, then a renormalising fast two-sum).
__device__ __forceinline__ void ff_add(float& ah, float& al, float bh, float bl) {
  const float s = ah + bh;
  const float bb = s - ah;
  float e = (ah - (s - bb)) + (bh - bb);
  e += al + bl;
  ah = s + e;
  al = e - (ah - s);
}

// Loads 8 staged fp32 values (the 16-byte units 2 c and 2 c + 1 of a row),
// the unit with the same parity as c >> 2 first: the eight lanes that load
// c = 8 i .. 8 i + 7 of one row then touch eight different bank groups.
__device__ __forceinline__ void load_staged8(const uint8_t* row, int c, float (&v)[8]) {
  const int s = (c >> 2) & 1;
  const float4 f0 = *reinterpret_cast<const float4*>(row + (2 * c + s) * 16);
  const float4 f1 = *reinterpret_cast<const float4*>(row + (2 * c + 1 - s) * 16);
  const float4 lo = s ? f1 : f0, hi = s ? f0 : f1;
  unpack8(lo, hi, v);
}

}  // namespace ssd_tc
}  // namespace ra
