// Device-side view of the planner's work list and the parameters shared by
// the forward kernels.
#pragma once
#include <cstdint>

#include "planner.h"

namespace ra {

// ------------------------------------------------------------ debug checks
// The debug build (compiled with -DRINGATTN_DEBUG into libringattn_debug.so)
// checks every computed global index before it is used.  An index outside
// its array records RA_ERR_BOUNDS (-7) in the status word and, for the first
// failure only, (site << 48 | index) in the 8 bytes after it; the access is
// then skipped (a store) or made at element 0 (a load), so nothing outside
// the buffers is touched and nothing traps.  In the normal build every check
// is the constant true and compiles to nothing.
#ifdef RINGATTN_DEBUG
constexpr bool kBoundsChecks = true;
#else
constexpr bool kBoundsChecks = false;
#endif

// Where a failed check was made (the site recorded with the index).
enum CheckSite : int {
  kSiteFwdItem = 1, kSiteFwdSeg, kSiteFwdQRow, kSiteFwdKvRow, kSiteFwdOut, kSiteFwdLse,
  kSiteFwdPart, kSiteBwdItem, kSiteBwdSeg, kSiteBwdQRow, kSiteBwdKvRow, kSiteBwdRowStat,
  kSiteBwdDq, kSiteBwdDkDv, kSiteMerge, kSiteSplitMerge, kSitePreprocess, kSiteSimtFwd,
  kSiteSimtBwd, kSiteHead, kSiteSsd
};

__device__ __forceinline__ bool index_ok(long long i, long long n, int* status, int site) {
  if constexpr (!kBoundsChecks) {
    return true;
  } else {
    if (i >= 0 && i < n) return true;
    if (status != nullptr) {
      atomicCAS(status, 0, -7 /* RA_ERR_BOUNDS */);
      unsigned long long* where = reinterpret_cast<unsigned long long*>(status + 2);
      atomicCAS(where, 0ull,
                (static_cast<unsigned long long>(site) << 48) |
                    (static_cast<unsigned long long>(i) & 0xFFFFFFFFFFFFull));
    }
    return false;
  }
}

// A load index: i itself, or 0 (after recording the failure) when outside [0, n).
__device__ __forceinline__ long long checked(long long i, long long n, int* status, int site) {
  return index_ok(i, n, status, site) ? i : 0;
}

// Where global token t lives in a buffer: chunk [a0, b0) holds rows
// [0, b0 - a0) and chunk [a1, ...) the rows after them.  Whole-sequence
// buffers use the identity (a0 = 0, b0 = INT_MAX); one rank's shard-local
// buffer of a multi-GPU ring holds its chunk(s) back to back (ZIGZAG: chunk r,
// then chunk 2P-1-r).  Masks always use global positions; loads, stores and
// lse rows use the buffer's rows.
struct RowMap {
  int a0, b0, a1;
};
__device__ __forceinline__ int local_row(const RowMap& m, int t) {
  return t < m.b0 ? t - m.a0 : t - m.a1 + (m.b0 - m.a0);
}

struct FwdParams {
  const void* q;          // [T, Hq, D]
  const void* k;          // [T, Hkv, D]
  const void* v;          // [T, Hkv, D]
  void* out;              // [T, Hq, D], bf16 or fp32 (out_fp32)
  float* lse;             // [Hq, T]
  const PlanItem* items;  // device copy of the plan
  const PlanSegment* segs;
  const int32_t* cu;      // document offsets, num_docs + 1
  int num_docs;
  int num_items;
  int T, hq, hkv, D;
  int group;              // Hq / Hkv
  int causal;
  float scale;            // 1 / sqrt(D)
  float scale_log2;       // scale * log2(e)
  int* work_counter;       // persistent launch: next unclaimed item, zeroed before the launch
                          // (nullptr: CTA i runs item i)
  int num_ctas;           // grid of the persistent launch
  int step_filter;        // -1: every ring step; s >= 0: only segments of step s
  int out_fp32;           // 1: out is fp32, 0: out is bf16
  int* status;            // device status word (first error wins)
  RowMap qmap;            // rows of q, out and lse (identity: whole sequence)
  RowMap kmap;            // rows of k and v
  int lse_stride;         // rows per head of lse: [Hq, lse_stride]
  // partial results of split items (PlanItem.part >= 0): slot s holds the two
  // query tiles' O / l, fp32 [2][128][D], at part_o + s * 2 * 128 * D, and
  // their lse at part_lse + s * 2 * 128
  float* part_o;
  float* part_lse;
  // extents for the debug build's checks
  int num_segs;           // entries of segs
  int num_parts;          // partial-result slots
  int q_rows, k_rows;     // rows of the q / out buffers and of the k, v buffers
};

struct BwdParams {
  const void* q;            // [T, Hq, D]
  const void* k;            // [T, Hkv, D]
  const void* v;            // [T, Hkv, D]
  const void* dout;         // [T, Hq, D]
  const float* lse;         // [Hq, T], natural log
  const float* Dvec;        // [Hq, T]: D_i = dO_i . O_i
  void* dq;                 // [T, Hq, D]
  void* dk;                 // [T, Hkv, D]
  void* dv;                 // [T, Hkv, D]
  const PlanItem* items;    // forward plan: query tiles and their key ranges
  const PlanSegment* segs;
  const BwdItem* bitems;    // key tiles and their query ranges
  const BwdSegment* bsegs;
  const int32_t* cu;
  int num_docs;
  int num_items, num_bitems;
  int T, hq, hkv, D;
  int group;                // Hq / Hkv
  int causal;
  float scale;              // 1 / sqrt(D)
  float scale_log2;         // scale * log2(e)
  int grad_fp32;            // 1: dq, dk, dv are fp32, else bf16
  int* status;
  RowMap qmap;              // rows of q, dout, dq, lse and Dvec (identity: whole sequence)
  RowMap kmap;              // rows of k, v, dk and dv
  int lse_stride;           // rows per head of lse and Dvec
  int accumulate;           // 1: add into fp32 dq, dk, dv instead of writing them
  // dK/dV: every flush_pairs (query tile, head) pairs of a key tile's walk
  // (0: never) the TMEM sums are added to fp32 dk_acc, dv_acc [rows, Hkv, D]
  // (dk, dv themselves when they are fp32) and restarted
  int flush_pairs;
  float* dk_acc;
  float* dv_acc;
  // extents for the debug build's checks
  int num_segs, num_bsegs;  // entries of segs and bsegs
  int q_rows, k_rows;       // rows of the q-side buffers and of the k-side buffers
};

// Context-parallel selective scan (Mamba2 SSD), fp32.
struct SsdParams {
  const float* x;        // [T, H, P]
  const float* dt;       // [T, H], > 0
  const float* A;        // [H], < 0
  const float* B;        // [T, G, N]
  const float* C;        // [T, G, N]
  const float* D;        // [H] or nullptr
  const int32_t* pos;    // [T] position ids (0 starts a packed sample) or nullptr
  float* y;              // [T, H, P]
  float* final_state;    // [H, P, N] or nullptr
  float* chunk_state;    // workspace [R, H, P, N]: each rank's final state from zero
  float* incoming;       // workspace [R, H, P, N]: the state each rank receives
  float* carry;          // workspace [R, H]: how much of an incoming state survives a chunk
  int T, H, G, N, R;     // tokens, heads, groups, state size, ranks (shards)
  int* status;           // device status word (the debug build's checks)
};

// Start and end of the document holding token t (binary search over cu).
__device__ __forceinline__ void doc_bounds(const int32_t* cu, int num_docs, int t, int* start,
                                           int* end) {
  int lo = 0, hi = num_docs;  // cu[lo] <= t < cu[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(cu + mid) <= t)
      lo = mid;
    else
      hi = mid;
  }
  *start = __ldg(cu + lo);
  *end = __ldg(cu + lo + 1);
}

// Keys query row `row` may see: [lo, hi) (same document, and <= row if causal).
__device__ __forceinline__ void row_key_interval(const FwdParams& p, int row, int* lo, int* hi) {
  int s, e;
  doc_bounds(p.cu, p.num_docs, row, &s, &e);
  *lo = s;
  *hi = p.causal ? row + 1 : e;
}

__device__ __forceinline__ bool seg_selected(const PlanSegment& s, int step_filter) {
  return step_filter < 0 || s.step == step_filter;
}

}  // namespace ra
