// C ABI of the ring-attention library: argument checks, the per-problem plan
// cache, tensor-map encoding and kernel launches.  See include/ringattn.h for
// the contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <list>
#include <mutex>
#include <string>
#include <vector>

#include "launch.h"
#include "planner.h"
#include "ringattn.h"
#include "trace.h"

namespace ra {

// Word 0: the first kernel-side error since the last ringattn_get_status
// (0 = none).  Words 2-3: the debug build's first failed bounds check,
// (site << 48 | index), 0 = none.
__device__ __align__(8) int g_status_word[4];

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kMaxCachedPlans = 128;
constexpr int kMaxHeadDim = 128;

struct DeviceState {
  bool ready = false;
  ra_status why = RA_OK;
  int* status = nullptr;  // device address of g_status_word
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

struct CachedPlan {
  int dev = -1;
  PlanInput key;
  Plan plan;
  void* buf = nullptr;  // items | segments | cu on the device
  PlanItem* items = nullptr;
  PlanSegment* segs = nullptr;
  int32_t* cu = nullptr;
  int num_ctas = 0;  // grid of the persistent forward: min(items, SMs)
  cudaEvent_t last_use = nullptr;
  // the persistent fused forward's claim order and split items, and the fp32
  // slots of the split halves' partial results
  FusedPlan fused;
  void* fused_buf = nullptr;
  PlanItem* fitems = nullptr;
  PlanSegment* fsegs = nullptr;
  SplitPair* fpairs = nullptr;
  float* part_o = nullptr;
  float* part_lse = nullptr;
  int fused_ctas = 0;
  // key-side backward schedule, built on the first backward call
  BwdPlan bwd;
  void* bwd_buf = nullptr;
  BwdItem* bitems = nullptr;
  BwdSegment* bsegs = nullptr;
  bool has_bwd = false;
};
std::list<CachedPlan> g_plans;  // most recently used first

bool same_key(const PlanInput& a, const PlanInput& b) {
  return a.T == b.T && a.hq == b.hq && a.hkv == b.hkv && a.num_shards == b.num_shards &&
         a.layout == b.layout && a.causal == b.causal && a.heads_k_stride == b.heads_k_stride &&
         a.exchange == b.exchange && a.q_rank == b.q_rank && a.k_rank == b.k_rank &&
         a.cu == b.cu;
}

// Checks the current device once: it must be an sm_103 part.
ra_status current_device(int* dev_out, DeviceState** st_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RA_ERR_CUDA;
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return RA_ERR_CUDA;
    if (!(prop.major == 10 && prop.minor == 3)) {
      st.why = RA_ERR_UNSUPPORTED;
    } else {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return RA_ERR_CUDA;
      if (cudaMemset(addr, 0, 4 * sizeof(int)) != cudaSuccess) return RA_ERR_CUDA;
      st.status = static_cast<int*>(addr);
      st.why = RA_OK;
    }
    st.ready = true;
  }
  if (st.why != RA_OK) return st.why;
  *dev_out = dev;
  *st_out = &st;
  return RA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

// [T, H, D] bf16 tensor viewed as 3-D (D, H, T); box 64 x 1 x 128, 128 B swizzle.
bool encode_thd(CUtensorMap* map, const void* ptr, int T, int H, int D) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [T, M, inner] tensor viewed as 3-D (inner, M, T); box box_inner x 1 x
// rows.  Without swizzle the rows land in shared memory as they are in
// memory; with it (box_inner = 32: 128-byte rows) the 16-byte units of row t
// of the box are permuted by XOR with t mod 8.
bool encode_f32_rows(CUtensorMap* map, const void* ptr, int T, int M, int inner, int box_inner,
                     int rows, bool swizzle) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)M, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)inner * 4, (cuuint64_t)M * inner * 4};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, 1, (cuuint32_t)rows};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PlanInput make_input(const int32_t* cu_seqlens, const ra_dims& d, int P, int layout, int causal) {
  PlanInput in;
  in.T = d.total_tokens;
  in.hq = d.hq;
  in.hkv = d.hkv;
  in.num_shards = P;
  in.layout = layout;
  in.causal = causal ? 1 : 0;
  in.heads_k_stride = d.heads_k_stride == 0 ? 1 : d.heads_k_stride;
  in.exchange = d.kv_exchange;
  if (cu_seqlens && d.num_seqs >= 1) {
    in.cu.assign(cu_seqlens, cu_seqlens + d.num_seqs + 1);
  } else {
    in.cu = {0, d.total_tokens};
  }
  return in;
}

// Common argument checks; returns RA_OK and fills `in`.
ra_status check_problem(const int32_t* cu_seqlens, const ra_dims& d, int P, int layout, int causal,
                        PlanInput* in) {
  if (d.total_tokens < 0 || d.hq < 1 || d.hkv < 1 || d.head_dim < 1) return RA_ERR_INVALID_ARG;
  if (d.heads_k_stride < 0) return RA_ERR_INVALID_ARG;
  if (cu_seqlens && d.num_seqs < 1) return RA_ERR_INVALID_ARG;
  if (P < 1 || (layout != RA_CONTIGUOUS && layout != RA_ZIGZAG)) return RA_ERR_INVALID_ARG;
  const long long parts = layout == RA_ZIGZAG ? 2LL * P : P;
  if (d.total_tokens % parts) return RA_ERR_NOT_DIVISIBLE;
  if (d.dtype != RA_BF16 && d.dtype != RA_FP32) return RA_ERR_UNSUPPORTED;
  if (d.head_dim != 64 && d.head_dim != 128) return RA_ERR_UNSUPPORTED;
  if ((long long)d.total_tokens * d.hq * d.head_dim >= (1LL << 40)) return RA_ERR_UNSUPPORTED;
  *in = make_input(cu_seqlens, d, P, layout, causal);
  if (!plan_check(*in).empty()) return RA_ERR_INVALID_ARG;
  return RA_OK;
}

// Finds or builds (and uploads) the plan; caller holds g_mu.
ra_status get_plan(int dev, const PlanInput& in, cudaStream_t stream, CachedPlan** out) {
  for (auto it = g_plans.begin(); it != g_plans.end(); ++it) {
    if (it->dev == dev && same_key(it->key, in)) {
      g_plans.splice(g_plans.begin(), g_plans, it);
      *out = &g_plans.front();
      return RA_OK;
    }
  }
  while (g_plans.size() >= kMaxCachedPlans) {
    CachedPlan& old = g_plans.back();
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(old.dev);
    if (old.last_use) {
      cudaEventSynchronize(old.last_use);
      cudaEventDestroy(old.last_use);
    }
    cudaFree(old.buf);
    if (old.bwd_buf) cudaFree(old.bwd_buf);
    if (old.fused_buf) cudaFree(old.fused_buf);
    cudaSetDevice(cur);
    g_plans.pop_back();
  }
  CachedPlan cp;
  cp.dev = dev;
  cp.key = in;
  cp.plan = build_fwd_plan(in);
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return RA_ERR_CUDA;
  const int n_items = static_cast<int>(cp.plan.items.size());
  cp.num_ctas = n_items < sms ? n_items : sms;
  const size_t nb_items = cp.plan.items.size() * sizeof(PlanItem);
  const size_t nb_segs = cp.plan.segs.size() * sizeof(PlanSegment);
  const size_t nb_cu = cp.plan.cu.size() * sizeof(int32_t);
  const size_t off_segs = (nb_items + 255) & ~size_t(255);
  const size_t off_cu = off_segs + ((nb_segs + 255) & ~size_t(255));
  const size_t total = off_cu + nb_cu;
  if (cudaMalloc(&cp.buf, total) != cudaSuccess) return RA_ERR_CUDA;
  char* b = static_cast<char*>(cp.buf);
  cp.items = reinterpret_cast<PlanItem*>(b);
  cp.segs = reinterpret_cast<PlanSegment*>(b + off_segs);
  cp.cu = reinterpret_cast<int32_t*>(b + off_cu);
  // synchronous uploads: the plan is built once per distinct problem
  if ((nb_items && cudaMemcpy(cp.items, cp.plan.items.data(), nb_items, cudaMemcpyHostToDevice)) ||
      (nb_segs && cudaMemcpy(cp.segs, cp.plan.segs.data(), nb_segs, cudaMemcpyHostToDevice)) ||
      cudaMemcpy(cp.cu, cp.plan.cu.data(), nb_cu, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(cp.buf);
    return RA_ERR_CUDA;
  }
  if (cudaEventCreateWithFlags(&cp.last_use, cudaEventDisableTiming) != cudaSuccess) {
    cudaFree(cp.buf);
    return RA_ERR_CUDA;
  }
  // the fused forward's list (a single ring step's plan runs one item per CTA
  // and never uses it)
  if (in.q_rank < 0 && in.k_rank < 0 && !cp.plan.items.empty()) {
    cp.fused = build_fused_plan(cp.plan, sms);
    cp.fused_ctas = static_cast<int>(cp.fused.items.size()) < sms
                        ? static_cast<int>(cp.fused.items.size()) : sms;
    const size_t fb_items = cp.fused.items.size() * sizeof(PlanItem);
    const size_t fb_segs = cp.fused.segs.size() * sizeof(PlanSegment);
    const size_t fb_pairs = cp.fused.pairs.size() * sizeof(SplitPair);
    const size_t nparts = 2 * cp.fused.pairs.size();  // slots of 2 query tiles x 128 rows
    const size_t fb_po = nparts * 2 * 128 * (size_t)kMaxHeadDim * sizeof(float);
    const size_t fb_pl = nparts * 2 * 128 * sizeof(float);
    size_t off = 0;
    auto take = [&](size_t n) { const size_t o = off; off += (n + 255) & ~size_t(255); return o; };
    const size_t o_items = take(fb_items), o_segs = take(fb_segs), o_pairs = take(fb_pairs);
    const size_t o_po = take(fb_po), o_pl = take(fb_pl);
    if (cudaMalloc(&cp.fused_buf, off + 256) != cudaSuccess) {
      cudaFree(cp.buf);
      cudaEventDestroy(cp.last_use);
      return RA_ERR_CUDA;
    }
    char* fb = static_cast<char*>(cp.fused_buf);
    cp.fitems = reinterpret_cast<PlanItem*>(fb + o_items);
    cp.fsegs = reinterpret_cast<PlanSegment*>(fb + o_segs);
    cp.fpairs = reinterpret_cast<SplitPair*>(fb + o_pairs);
    cp.part_o = reinterpret_cast<float*>(fb + o_po);
    cp.part_lse = reinterpret_cast<float*>(fb + o_pl);
    if ((fb_items && cudaMemcpy(cp.fitems, cp.fused.items.data(), fb_items,
                                cudaMemcpyHostToDevice) != cudaSuccess) ||
        (fb_segs && cudaMemcpy(cp.fsegs, cp.fused.segs.data(), fb_segs,
                               cudaMemcpyHostToDevice) != cudaSuccess) ||
        (fb_pairs && cudaMemcpy(cp.fpairs, cp.fused.pairs.data(), fb_pairs,
                                cudaMemcpyHostToDevice) != cudaSuccess)) {
      cudaFree(cp.buf);
      cudaFree(cp.fused_buf);
      cudaEventDestroy(cp.last_use);
      return RA_ERR_CUDA;
    }
  }
  (void)stream;
  g_plans.push_front(std::move(cp));
  *out = &g_plans.front();
  return RA_OK;
}

// Adds the key-side backward schedule to a cached plan; caller holds g_mu.
ra_status get_bwd_plan(CachedPlan* cp) {
  if (cp->has_bwd) return RA_OK;
  cp->bwd = build_bwd_plan(cp->key);
  const size_t nb_items = cp->bwd.items.size() * sizeof(BwdItem);
  const size_t nb_segs = cp->bwd.segs.size() * sizeof(BwdSegment);
  const size_t off_segs = (nb_items + 255) & ~size_t(255);
  if (cudaMalloc(&cp->bwd_buf, off_segs + nb_segs + 16) != cudaSuccess) return RA_ERR_CUDA;
  char* b = static_cast<char*>(cp->bwd_buf);
  cp->bitems = reinterpret_cast<BwdItem*>(b);
  cp->bsegs = reinterpret_cast<BwdSegment*>(b + off_segs);
  if ((nb_items && cudaMemcpy(cp->bitems, cp->bwd.items.data(), nb_items, cudaMemcpyHostToDevice)) ||
      (nb_segs && cudaMemcpy(cp->bsegs, cp->bwd.segs.data(), nb_segs, cudaMemcpyHostToDevice))) {
    cudaFree(cp->bwd_buf);
    cp->bwd_buf = nullptr;
    return RA_ERR_CUDA;
  }
  cp->has_bwd = true;
  return RA_OK;
}

FwdParams make_params(const void* q, const void* k, const void* v, void* out, float* lse,
                      const ra_dims& d, int causal, const CachedPlan& cp, int* status) {
  FwdParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.lse = lse;
  p.items = cp.items;
  p.segs = cp.segs;
  p.cu = cp.cu;
  p.num_docs = static_cast<int>(cp.plan.cu.size()) - 1;
  p.num_items = static_cast<int>(cp.plan.items.size());
  p.T = d.total_tokens;
  p.hq = d.hq;
  p.hkv = d.hkv;
  p.D = d.head_dim;
  p.group = d.hq / d.hkv;
  p.causal = causal ? 1 : 0;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d.head_dim));
  p.scale_log2 = p.scale * 1.4426950408889634f;
  p.work_counter = nullptr;  // set by launch_fwd for the persistent launch
  p.num_ctas = cp.num_ctas;
  p.step_filter = -1;
  p.out_fp32 = d.dtype == RA_FP32 ? 1 : 0;
  p.status = status;
  p.qmap = RowMap{0, INT_MAX, 0};  // whole-sequence buffers
  p.kmap = RowMap{0, INT_MAX, 0};
  p.lse_stride = d.total_tokens;
  p.num_segs = static_cast<int>(cp.plan.segs.size());
  p.num_parts = 0;
  p.q_rows = d.total_tokens;
  p.k_rows = d.total_tokens;
  return p;
}

// Rows of rank r's shard-local buffer: its chunk(s) back to back.
RowMap rank_rows(int T, int P, int layout, int r) {
  int ch[2][2], n;
  rank_chunks(T, P, layout, r, ch, &n);
  return RowMap{ch[0][0], ch[0][1], n > 1 ? ch[1][0] : ch[0][1]};
}

struct Maps {
  CUtensorMap q, k, v;
};

// Work counters of the persistent forward.  Each launch takes a slot whose
// previous launch has finished (its event has completed), zeroes it on the
// launch stream and records the slot's event after the launch, so launches
// in flight on different streams never share a counter.  Caller holds g_mu.
constexpr int kCounterSlots = 64;
__device__ int g_work_counters[kCounterSlots];
struct CounterPool {
  int* base = nullptr;
  cudaEvent_t ev[kCounterSlots] = {};
  int next = 0;
};
CounterPool g_counters[kMaxDevices];

ra_status claim_counter(int dev, cudaStream_t s, int** counter, cudaEvent_t* ev) {
  CounterPool& pool = g_counters[dev];
  if (!pool.base) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_work_counters) != cudaSuccess) return RA_ERR_CUDA;
    pool.base = static_cast<int*>(a);
  }
  int slot = -1;
  for (int t = 0; t < kCounterSlots && slot < 0; ++t) {
    const int c = (pool.next + t) % kCounterSlots;
    if (!pool.ev[c]) {
      if (cudaEventCreateWithFlags(&pool.ev[c], cudaEventDisableTiming) != cudaSuccess)
        return RA_ERR_CUDA;
      slot = c;
    } else {
      const cudaError_t q = cudaEventQuery(pool.ev[c]);
      if (q == cudaSuccess) slot = c;
      else if (q != cudaErrorNotReady) return RA_ERR_CUDA;
    }
  }
  // a busy slot is not an error: clear it from the last-error state
  const cudaError_t last = cudaGetLastError();
  if (last != cudaSuccess && last != cudaErrorNotReady) return RA_ERR_CUDA;
  if (slot < 0) {  // every slot busy: wait for the oldest
    slot = pool.next;
    if (cudaEventSynchronize(pool.ev[slot]) != cudaSuccess) return RA_ERR_CUDA;
  }
  pool.next = (slot + 1) % kCounterSlots;
  if (cudaMemsetAsync(pool.base + slot, 0, sizeof(int), s) != cudaSuccess) return RA_ERR_CUDA;
  *counter = pool.base + slot;
  *ev = pool.ev[slot];
  return RA_OK;
}

ra_status launch_fwd(const FwdParams& p, const ra_dims& d, const Maps* maps, cudaStream_t stream) {
  cudaError_t e;
  if (d.dtype == RA_FP32)
    e = launch_fwd_simt_fp32(p, stream);
  else
    e = launch_fwd_tc_bf16(p, maps->q, maps->k, maps->v, stream);
  return e == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

ra_status prepare_maps(const void* q, const void* k, const void* v, const ra_dims& d, Maps* maps) {
  if (d.dtype != RA_BF16) return RA_OK;
  if (!encode_thd(&maps->q, q, d.total_tokens, d.hq, d.head_dim) ||
      !encode_thd(&maps->k, k, d.total_tokens, d.hkv, d.head_dim) ||
      !encode_thd(&maps->v, v, d.total_tokens, d.hkv, d.head_dim))
    return RA_ERR_CUDA;
  return RA_OK;
}

// Checks shared by the rank-step calls; fills `in` (with the step's rank
// filters) and the shard's row count.
ra_status check_rank_step(const int32_t* cu_seqlens, const ra_dims& dims, int P, int layout,
                          int causal, int rank, int step, PlanInput* in, int* Tr) {
  ra_status st = check_problem(cu_seqlens, dims, P, layout, causal, in);
  if (st != RA_OK) return st;
  if (dims.dtype != RA_BF16 || dims.kv_exchange != RA_RING) return RA_ERR_UNSUPPORTED;
  if (rank < 0 || rank >= P || step < 0 || step >= P) return RA_ERR_INVALID_ARG;
  in->q_rank = rank;
  in->k_rank = ((rank - step) % P + P) % P;
  *Tr = dims.total_tokens / P;
  return RA_OK;
}

size_t fp32_o_bytes(const ra_dims& d) {
  return ((size_t)d.total_tokens * d.hq * d.head_dim * 4 + 255) & ~size_t(255);
}
size_t lse_bytes(const ra_dims& d) { return ((size_t)d.hq * d.total_tokens * 4 + 255) & ~size_t(255); }
size_t kv_f32_bytes(const ra_dims& d) {
  return ((size_t)d.total_tokens * d.hkv * d.head_dim * 4 + 255) & ~size_t(255);
}

// (query tile, head) pairs after which the dK/dV kernel moves its TMEM sums
// to fp32 memory and restarts them (0: never).  The tensor cores' fp32
// accumulation loses a little toward zero at every step, so bounding the
// run bounds that loss whatever the sequence length.
std::atomic<int> g_bwd_flush_pairs{1024};

// Whether some key tile's walk can be longer than `flush` pairs: it visits
// at most every query tile of every head of its group.
bool bwd_may_flush(const ra_dims& d, int flush) {
  if (flush <= 0 || d.hkv < 1 || d.hq % d.hkv) return false;
  return (long long)((d.total_tokens + 127) / 128) * (d.hq / d.hkv) > flush;
}

size_t bwd_workspace_bytes(const ra_dims& d, int flush) {
  size_t n = lse_bytes(d);  // D_i = dO_i . O_i, fp32 [Hq, T]
  // bf16 gradients whose dK/dV walks can outlast the flush interval: the
  // fp32 sums of dk and dv
  if (d.dtype == RA_BF16 && !d.grad_fp32 && bwd_may_flush(d, flush)) n += 2 * kv_f32_bytes(d);
  return n;
}

// Where the dK/dV flushes go: fp32 outputs themselves, else the fp32 sums
// after the D_i vector in the workspace (none: no walk outlasts `flush`).
void set_bwd_flush(BwdParams* p, const ra_dims& d, void* workspace, int flush) {
  p->flush_pairs = flush;
  if (p->grad_fp32) {
    p->dk_acc = static_cast<float*>(p->dk);
    p->dv_acc = static_cast<float*>(p->dv);
  } else if (bwd_may_flush(d, flush)) {
    char* w = static_cast<char*>(workspace) + lse_bytes(d);
    p->dk_acc = reinterpret_cast<float*>(w);
    p->dv_acc = reinterpret_cast<float*>(w + kv_f32_bytes(d));
  } else {
    p->flush_pairs = 0;
  }
}

}  // namespace
}  // namespace ra

using namespace ra;

extern "C" {

ra_status ringattn_fwd(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                       ra_dims dims, int num_shards, int shard_layout, int causal, void* out,
                       float* lse, void* stream) {
  NvtxRange nvtx("ringattn_fwd");
  PlanInput in;
  ra_status st = check_problem(cu_seqlens, dims, num_shards, shard_layout, causal, &in);
  if (st != RA_OK) return st;
  if (dims.total_tokens == 0) return RA_OK;
  if (!q || !k || !v || !out || !lse) return RA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return RA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev;
  DeviceState* ds;
  if ((st = current_device(&dev, &ds)) != RA_OK) return st;
  Maps maps;
  if ((st = prepare_maps(q, k, v, dims, &maps)) != RA_OK) return st;
  CachedPlan* cp;
  if ((st = get_plan(dev, in, static_cast<cudaStream_t>(stream), &cp)) != RA_OK) return st;
  FwdParams p = make_params(q, k, v, out, lse, dims, causal, *cp, ds->status);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool tc = dims.dtype == RA_BF16 && cp->fitems != nullptr;
  if (tc) {  // the persistent launch's claim order, with long items split
    p.items = cp->fitems;
    p.segs = cp->fsegs;
    p.num_items = static_cast<int>(cp->fused.items.size());
    p.num_ctas = cp->fused_ctas;
    p.part_o = cp->part_o;
    p.part_lse = cp->part_lse;
    p.num_segs = static_cast<int>(cp->fused.segs.size());
    p.num_parts = 2 * static_cast<int>(cp->fused.pairs.size());
  }
  const int npairs = tc ? static_cast<int>(cp->fused.pairs.size()) : 0;
  // the plan's partial slots are free once its previous launch is done
  // (launches of one problem on other streams are ordered behind it)
  if (npairs > 0 && cudaStreamWaitEvent(s, cp->last_use, 0) != cudaSuccess) return RA_ERR_CUDA;
  cudaEvent_t counter_ev = nullptr;
  if (dims.dtype == RA_BF16 && p.num_items > 0 &&
      (st = claim_counter(dev, s, &p.work_counter, &counter_ev)) != RA_OK)
    return st;
  if ((st = launch_fwd(p, dims, &maps, s)) != RA_OK) return st;
  if (npairs > 0 &&
      launch_split_merge(cp->fpairs, npairs, cp->part_o, cp->part_lse, out, false, lse, dims.hq,
                         dims.total_tokens, dims.head_dim, ds->status, s) != cudaSuccess)
    return RA_ERR_CUDA;
  if (counter_ev && cudaEventRecord(counter_ev, s) != cudaSuccess) return RA_ERR_CUDA;
  if (cudaEventRecord(cp->last_use, s) != cudaSuccess) return RA_ERR_CUDA;
  return RA_OK;
}

size_t ringattn_fwd_stepwise_workspace_size(ra_dims dims) {
  if (dims.total_tokens < 0 || dims.hq < 1 || dims.head_dim < 1) return 0;
  return 2 * (fp32_o_bytes(dims) + lse_bytes(dims));
}

ra_status ringattn_fwd_stepwise(const void* q, const void* k, const void* v,
                                const int32_t* cu_seqlens, ra_dims dims, int num_shards,
                                int shard_layout, int causal, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx("ringattn_fwd_stepwise");
  PlanInput in;
  ra_status st = check_problem(cu_seqlens, dims, num_shards, shard_layout, causal, &in);
  if (st != RA_OK) return st;
  if (dims.total_tokens == 0) return RA_OK;
  if (!q || !k || !v || !out || !lse) return RA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return RA_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < ringattn_fwd_stepwise_workspace_size(dims) ||
      !aligned16(workspace))
    return RA_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev;
  DeviceState* ds;
  if ((st = current_device(&dev, &ds)) != RA_OK) return st;
  Maps maps;
  if ((st = prepare_maps(q, k, v, dims, &maps)) != RA_OK) return st;
  CachedPlan* cp;
  if ((st = get_plan(dev, in, static_cast<cudaStream_t>(stream), &cp)) != RA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(workspace);
  float* acc_o = reinterpret_cast<float*>(w);
  float* acc_l = reinterpret_cast<float*>(w + fp32_o_bytes(dims));
  float* stp_o = reinterpret_cast<float*>(w + fp32_o_bytes(dims) + lse_bytes(dims));
  float* stp_l = reinterpret_cast<float*>(w + 2 * fp32_o_bytes(dims) + lse_bytes(dims));
  const bool out_fp32 = dims.dtype == RA_FP32;
  // ring steps; an all-gather exchange is one step
  const int num_steps = dims.kv_exchange == RA_ALLGATHER ? 1 : num_shards;
  for (int step = 0; step < num_steps; ++step) {
    const bool last = step == num_steps - 1;
    // step 0 starts the accumulator; one shard writes the result directly
    void* o_dst = step == 0 ? (last ? out : static_cast<void*>(acc_o)) : stp_o;
    float* l_dst = step == 0 ? (last ? lse : acc_l) : stp_l;
    FwdParams p = make_params(q, k, v, o_dst, l_dst, dims, causal, *cp, ds->status);
    p.step_filter = step;

    p.out_fp32 = (step == 0 && last) ? (out_fp32 ? 1 : 0) : 1;
    if ((st = launch_fwd(p, dims, &maps, s)) != RA_OK) return st;
    if (step > 0) {
      cudaError_t e = launch_lse_merge(acc_o, true, acc_l, stp_o, true, stp_l,
                                       last ? out : static_cast<void*>(acc_o),
                                       last ? out_fp32 : true, last ? lse : acc_l,
                                       dims.total_tokens, dims.hq, dims.head_dim, ds->status, s);
      if (e != cudaSuccess) return RA_ERR_CUDA;
    }
  }
  if (cudaEventRecord(cp->last_use, s) != cudaSuccess) return RA_ERR_CUDA;
  return RA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Stepwise forward with a fixed, library-owned scratch area.
//
// Some callers cannot allocate device memory at the point where they run
// attention: code inside a custom allocator or memory-pool callback, host
// runtimes that hand out only the input and output buffers, or a process whose
// allocations all go through a framework that is not reachable from this
// call.  For them this entry point keeps its fp32 partial results and its work
// list in a statically sized __device__ array instead of a caller workspace or
// the plan cache.  Every GPU that loads the library holds the array until the
// process exits.  All calls share it, so calls that overlap on the GPU (on
// different streams, or from different threads) race on it; calls on one
// stream are ordered.  Nothing in it needs to start at zero: each call writes
// every byte it later reads.
// ---------------------------------------------------------------------------
namespace ra {
namespace {

constexpr size_t kNoAllocScratchBytes = RA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
unsigned char* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).
ra_status noalloc_scratch(int dev, unsigned char** out) {
  if (!g_noalloc_ptr[dev]) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr)
      return RA_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<unsigned char*>(addr);
  }
  *out = g_noalloc_ptr[dev];
  return RA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace ra

extern "C" ra_status ringattn_fwd_stepwise_noalloc(const void* q, const void* k, const void* v,
                                                   const int32_t* cu_seqlens, ra_dims dims,
                                                   int num_shards, int shard_layout, int causal,
                                                   void* out, float* lse, void* stream) {
  NvtxRange nvtx("ringattn_fwd_stepwise_noalloc");
  PlanInput in;
  ra_status st = check_problem(cu_seqlens, dims, num_shards, shard_layout, causal, &in);
  if (st != RA_OK) return st;
  if (dims.total_tokens == 0) return RA_OK;
  if (!q || !k || !v || !out || !lse) return RA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return RA_ERR_INVALID_ARG;
  // scratch layout: acc O | acc lse | step O | step lse | items | segments | cu
  const size_t ws = ringattn_fwd_stepwise_workspace_size(dims);
  CachedPlan cp;  // host plan; its device copy lives in the scratch array
  cp.plan = build_fwd_plan(in);
  const size_t nb_items = cp.plan.items.size() * sizeof(PlanItem);
  const size_t nb_segs = cp.plan.segs.size() * sizeof(PlanSegment);
  const size_t nb_cu = cp.plan.cu.size() * sizeof(int32_t);
  const size_t need = ws + round256(nb_items) + round256(nb_segs) + round256(nb_cu);
  if (need > kNoAllocScratchBytes) return RA_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev;
  DeviceState* ds;
  if ((st = current_device(&dev, &ds)) != RA_OK) return st;
  unsigned char* base;
  if ((st = noalloc_scratch(dev, &base)) != RA_OK) return st;
  Maps maps;
  if ((st = prepare_maps(q, k, v, dims, &maps)) != RA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cp.items = reinterpret_cast<PlanItem*>(base + ws);
  cp.segs = reinterpret_cast<PlanSegment*>(base + ws + round256(nb_items));
  cp.cu = reinterpret_cast<int32_t*>(base + ws + round256(nb_items) + round256(nb_segs));
  // pageable-source copies: staged before the call returns, ordered on `s`
  if ((nb_items &&
       cudaMemcpyAsync(cp.items, cp.plan.items.data(), nb_items, cudaMemcpyHostToDevice, s)) ||
      (nb_segs &&
       cudaMemcpyAsync(cp.segs, cp.plan.segs.data(), nb_segs, cudaMemcpyHostToDevice, s)) ||
      cudaMemcpyAsync(cp.cu, cp.plan.cu.data(), nb_cu, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return RA_ERR_CUDA;
  float* acc_o = reinterpret_cast<float*>(base);
  float* acc_l = reinterpret_cast<float*>(base + fp32_o_bytes(dims));
  float* stp_o = reinterpret_cast<float*>(base + fp32_o_bytes(dims) + lse_bytes(dims));
  float* stp_l = reinterpret_cast<float*>(base + 2 * fp32_o_bytes(dims) + lse_bytes(dims));
  const bool out_fp32 = dims.dtype == RA_FP32;
  // ring steps; an all-gather exchange is one step
  const int num_steps = dims.kv_exchange == RA_ALLGATHER ? 1 : num_shards;
  for (int step = 0; step < num_steps; ++step) {
    const bool last = step == num_steps - 1;
    void* o_dst = step == 0 ? (last ? out : static_cast<void*>(acc_o)) : stp_o;
    float* l_dst = step == 0 ? (last ? lse : acc_l) : stp_l;
    FwdParams p = make_params(q, k, v, o_dst, l_dst, dims, causal, cp, ds->status);
    p.step_filter = step;

    p.out_fp32 = (step == 0 && last) ? (out_fp32 ? 1 : 0) : 1;
    if ((st = launch_fwd(p, dims, &maps, s)) != RA_OK) return st;
    if (step > 0) {
      cudaError_t e = launch_lse_merge(acc_o, true, acc_l, stp_o, true, stp_l,
                                       last ? out : static_cast<void*>(acc_o),
                                       last ? out_fp32 : true, last ? lse : acc_l,
                                       dims.total_tokens, dims.hq, dims.head_dim, ds->status, s);
      if (e != cudaSuccess) return RA_ERR_CUDA;
    }
  }
  return RA_OK;
}

extern "C" {

size_t ringattn_bwd_workspace_size(ra_dims dims) {
  if (dims.total_tokens < 0 || dims.hq < 1 || dims.head_dim < 1) return 0;
  return bwd_workspace_bytes(dims, g_bwd_flush_pairs.load());
}

ra_status ringattn_set_bwd_flush_interval(int pairs) {
  if (pairs < 0) return RA_ERR_INVALID_ARG;
  g_bwd_flush_pairs.store(pairs);
  return RA_OK;
}

ra_status ringattn_bwd(const void* q, const void* k, const void* v, const void* out,
                       const float* lse, const void* dout, const int32_t* cu_seqlens,
                       ra_dims dims, int num_shards, int shard_layout, int causal, void* dq,
                       void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx("ringattn_bwd");
  PlanInput in;
  ra_status st = check_problem(cu_seqlens, dims, num_shards, shard_layout, causal, &in);
  if (st != RA_OK) return st;
  if (dims.total_tokens == 0) return RA_OK;
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return RA_ERR_INVALID_ARG;
  for (const void* t : {q, k, v, out, dout, static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv)})
    if (!aligned16(t)) return RA_ERR_INVALID_ARG;
  const int flush = g_bwd_flush_pairs.load();  // one reading for the size check and the launch
  if (!workspace || workspace_bytes < bwd_workspace_bytes(dims, flush) || !aligned16(workspace))
    return RA_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev;
  DeviceState* ds;
  if ((st = current_device(&dev, &ds)) != RA_OK) return st;
  Maps maps;
  CUtensorMap map_do;
  if ((st = prepare_maps(q, k, v, dims, &maps)) != RA_OK) return st;
  if (dims.dtype == RA_BF16 && !encode_thd(&map_do, dout, dims.total_tokens, dims.hq, dims.head_dim))
    return RA_ERR_CUDA;
  CachedPlan* cp;
  if ((st = get_plan(dev, in, static_cast<cudaStream_t>(stream), &cp)) != RA_OK) return st;
  if ((st = get_bwd_plan(cp)) != RA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* Dvec = static_cast<float*>(workspace);
  const bool f32 = dims.dtype == RA_FP32;
  if (launch_bwd_preprocess(out, dout, f32, Dvec, dims.total_tokens, dims.hq, dims.head_dim,
                            ds->status, s) !=
      cudaSuccess)
    return RA_ERR_CUDA;
  BwdParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.dout = dout;
  p.lse = lse;
  p.Dvec = Dvec;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.items = cp->items;
  p.segs = cp->segs;
  p.bitems = cp->bitems;
  p.bsegs = cp->bsegs;
  p.cu = cp->cu;
  p.num_docs = static_cast<int>(cp->plan.cu.size()) - 1;
  p.num_items = static_cast<int>(cp->plan.items.size());
  p.num_bitems = static_cast<int>(cp->bwd.items.size());
  p.T = dims.total_tokens;
  p.hq = dims.hq;
  p.hkv = dims.hkv;
  p.D = dims.head_dim;
  p.group = dims.hq / dims.hkv;
  p.causal = causal ? 1 : 0;
  p.scale = 1.0f / std::sqrt(static_cast<float>(dims.head_dim));
  p.scale_log2 = p.scale * 1.4426950408889634f;
  p.grad_fp32 = (f32 || dims.grad_fp32) ? 1 : 0;
  p.status = ds->status;
  p.qmap = RowMap{0, INT_MAX, 0};
  p.kmap = RowMap{0, INT_MAX, 0};
  p.lse_stride = dims.total_tokens;
  p.accumulate = 0;
  p.num_segs = static_cast<int>(cp->plan.segs.size());
  p.num_bsegs = static_cast<int>(cp->bwd.segs.size());
  p.q_rows = dims.total_tokens;
  p.k_rows = dims.total_tokens;
  set_bwd_flush(&p, dims, workspace, flush);
  cudaError_t e = f32 ? launch_bwd_simt_fp32(p, s)
                      : launch_bwd_tc_bf16(p, maps.q, maps.k, maps.v, map_do, s);
  if (e != cudaSuccess) return RA_ERR_CUDA;
  if (cudaEventRecord(cp->last_use, s) != cudaSuccess) return RA_ERR_CUDA;
  return RA_OK;
}

// ---------------------------------------------------------------------------
// One ring step of one rank, on shard-local buffers (the multi-GPU ring: each
// GPU holds its own query rows and receives the K/V shard of rank
// (rank - step) mod P into its own memory before the step).
// ---------------------------------------------------------------------------

size_t ringattn_fwd_rank_workspace_size(ra_dims dims, int num_shards) {
  if (dims.total_tokens < 0 || dims.hq < 1 || dims.head_dim < 1 || num_shards < 1) return 0;
  ra_dims r = dims;
  r.total_tokens = dims.total_tokens / num_shards;
  return fp32_o_bytes(r) + lse_bytes(r);
}

ra_status ringattn_fwd_rank_step(const void* q, const void* k, const void* v,
                                 const int32_t* cu_seqlens, ra_dims dims, int num_shards,
                                 int shard_layout, int causal, int rank, int step, float* o_acc,
                                 float* lse_acc, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  NvtxRange nvtx("ringattn_fwd_rank_step");
  PlanInput in;
  int Tr = 0;
  ra_status st = check_rank_step(cu_seqlens, dims, num_shards, shard_layout, causal, rank, step,
                                 &in, &Tr);
  if (st != RA_OK) return st;
  if (dims.total_tokens == 0) return RA_OK;
  const bool first = step == 0, last = step == num_shards - 1;
  if (!q || !k || !v || !aligned16(q) || !aligned16(k) || !aligned16(v)) return RA_ERR_INVALID_ARG;
  if (!(first && last) && (!o_acc || !lse_acc || !aligned16(o_acc))) return RA_ERR_INVALID_ARG;
  if (last && (!out || !lse || !aligned16(out))) return RA_ERR_INVALID_ARG;
  if (!first && (!workspace || !aligned16(workspace) ||
                 workspace_bytes < ringattn_fwd_rank_workspace_size(dims, num_shards)))
    return RA_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev;
  DeviceState* ds;
  if ((st = current_device(&dev, &ds)) != RA_OK) return st;
  Maps maps;
  if (!encode_thd(&maps.q, q, Tr, dims.hq, dims.head_dim) ||
      !encode_thd(&maps.k, k, Tr, dims.hkv, dims.head_dim) ||
      !encode_thd(&maps.v, v, Tr, dims.hkv, dims.head_dim))
    return RA_ERR_CUDA;
  CachedPlan* cp;
  if ((st = get_plan(dev, in, static_cast<cudaStream_t>(stream), &cp)) != RA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ra_dims rd = dims;
  rd.total_tokens = Tr;
  float* stp_o = static_cast<float*>(workspace);
  float* stp_l = reinterpret_cast<float*>(static_cast<char*>(workspace) + fp32_o_bytes(rd));
  // the step's partial result: straight to the output when it is the only
  // step, to the running result when it starts it, else to the workspace
  void* o_dst = first ? (last ? out : static_cast<void*>(o_acc)) : stp_o;
  float* l_dst = first ? (last ? lse : lse_acc) : stp_l;
  FwdParams p = make_params(q, k, v, o_dst, l_dst, dims, causal, *cp, ds->status);
  p.qmap = rank_rows(dims.total_tokens, num_shards, shard_layout, rank);
  p.kmap = rank_rows(dims.total_tokens, num_shards, shard_layout, in.k_rank);
  p.lse_stride = Tr;
  p.q_rows = Tr;
  p.k_rows = Tr;
  p.out_fp32 = (first && last) ? 0 : 1;
  // every query tile of the rank is an item (one CTA each); a tile that sees
  // no key of this shard writes O = 0, lse = -inf
  if ((st = launch_fwd(p, dims, &maps, s)) != RA_OK) return st;
  if (!first) {
    if (launch_lse_merge(o_acc, true, lse_acc, stp_o, true, stp_l,
                         last ? out : static_cast<void*>(o_acc), last ? false : true,
                         last ? lse : lse_acc, Tr, dims.hq, dims.head_dim, ds->status,
                         s) != cudaSuccess)
      return RA_ERR_CUDA;
  }
  if (cudaEventRecord(cp->last_use, s) != cudaSuccess) return RA_ERR_CUDA;
  return RA_OK;
}

size_t ringattn_bwd_rank_workspace_size(ra_dims dims, int num_shards) {
  if (dims.total_tokens < 0 || dims.hq < 1 || dims.head_dim < 1 || num_shards < 1) return 0;
  ra_dims r = dims;
  r.total_tokens = dims.total_tokens / num_shards;
  return lse_bytes(r);  // D_i = dO_i . O_i of the rank's rows, fp32 [Hq, Tr]
}

ra_status ringattn_bwd_rank_step(const void* q, const void* k, const void* v, const void* out,
                                 const float* lse, const void* dout, const int32_t* cu_seqlens,
                                 ra_dims dims, int num_shards, int shard_layout, int causal,
                                 int rank, int step, float* dq, float* dk, float* dv,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx("ringattn_bwd_rank_step");
  PlanInput in;
  int Tr = 0;
  ra_status st = check_rank_step(cu_seqlens, dims, num_shards, shard_layout, causal, rank, step,
                                 &in, &Tr);
  if (st != RA_OK) return st;
  if (dims.total_tokens == 0) return RA_OK;
  for (const void* t : {q, k, v, out, dout, static_cast<const void*>(dq),
                        static_cast<const void*>(dk), static_cast<const void*>(dv)})
    if (!t || !aligned16(t)) return RA_ERR_INVALID_ARG;
  if (!lse) return RA_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < ringattn_bwd_rank_workspace_size(dims, num_shards))
    return RA_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev;
  DeviceState* ds;
  if ((st = current_device(&dev, &ds)) != RA_OK) return st;
  Maps maps;
  CUtensorMap map_do;
  if (!encode_thd(&maps.q, q, Tr, dims.hq, dims.head_dim) ||
      !encode_thd(&maps.k, k, Tr, dims.hkv, dims.head_dim) ||
      !encode_thd(&maps.v, v, Tr, dims.hkv, dims.head_dim) ||
      !encode_thd(&map_do, dout, Tr, dims.hq, dims.head_dim))
    return RA_ERR_CUDA;
  CachedPlan* cp;
  if ((st = get_plan(dev, in, static_cast<cudaStream_t>(stream), &cp)) != RA_OK) return st;
  if ((st = get_bwd_plan(cp)) != RA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* Dvec = static_cast<float*>(workspace);
  // step 0 computes the rank's D_i once; the caller keeps the workspace
  // for the later steps
  if (step == 0 &&
      launch_bwd_preprocess(out, dout, false, Dvec, Tr, dims.hq, dims.head_dim, ds->status, s) !=
          cudaSuccess)
    return RA_ERR_CUDA;
  BwdParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.dout = dout;
  p.lse = lse;
  p.Dvec = Dvec;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.items = cp->items;
  p.segs = cp->segs;
  p.bitems = cp->bitems;
  p.bsegs = cp->bsegs;
  p.cu = cp->cu;
  p.num_docs = static_cast<int>(cp->plan.cu.size()) - 1;
  p.num_items = static_cast<int>(cp->plan.items.size());
  p.num_bitems = static_cast<int>(cp->bwd.items.size());
  p.T = dims.total_tokens;
  p.hq = dims.hq;
  p.hkv = dims.hkv;
  p.D = dims.head_dim;
  p.group = dims.hq / dims.hkv;
  p.causal = causal ? 1 : 0;
  p.scale = 1.0f / std::sqrt(static_cast<float>(dims.head_dim));
  p.scale_log2 = p.scale * 1.4426950408889634f;
  p.grad_fp32 = 1;
  p.status = ds->status;
  p.qmap = rank_rows(dims.total_tokens, num_shards, shard_layout, rank);
  p.kmap = rank_rows(dims.total_tokens, num_shards, shard_layout, in.k_rank);
  p.lse_stride = Tr;
  p.num_segs = static_cast<int>(cp->plan.segs.size());
  p.num_bsegs = static_cast<int>(cp->bwd.segs.size());
  p.q_rows = Tr;
  p.k_rows = Tr;
  // step 0 starts dq (this rank's rows) and dk, dv (its own keys, which
  // then travel the ring); later steps add to them
  p.accumulate = step == 0 ? 0 : 1;
  set_bwd_flush(&p, dims, nullptr, g_bwd_flush_pairs.load());  // fp32 outputs take the flushes
  if (launch_bwd_tc_bf16(p, maps.q, maps.k, maps.v, map_do, s) != cudaSuccess) return RA_ERR_CUDA;
  if (cudaEventRecord(cp->last_use, s) != cudaSuccess) return RA_ERR_CUDA;
  return RA_OK;
}

ra_status attn_lse_merge(void* o_a, float* lse_a, const void* o_b, const float* lse_b, int rows,
                         int heads, int head_dim, int dtype, void* stream) {
  NvtxRange nvtx("attn_lse_merge");
  if (rows < 0 || heads < 1 || head_dim < 8 || head_dim % 8 || 32 % (head_dim / 8))
    return RA_ERR_INVALID_ARG;
  if (dtype != RA_BF16 && dtype != RA_FP32) return RA_ERR_UNSUPPORTED;
  if (rows == 0) return RA_OK;
  if (!o_a || !lse_a || !o_b || !lse_b) return RA_ERR_INVALID_ARG;
  if (!aligned16(o_a) || !aligned16(o_b)) return RA_ERR_INVALID_ARG;
  int dev;
  DeviceState* ds;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ra_status st = current_device(&dev, &ds);
    if (st != RA_OK) return st;
  }
  const bool f32 = dtype == RA_FP32;
  cudaError_t e = launch_lse_merge(o_a, f32, lse_a, o_b, f32, lse_b, o_a, f32, lse_a, rows, heads,
                                   head_dim, ds->status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

size_t ssd_cp_workspace_size(ssd_dims dims, int num_shards) {
  if (dims.total_tokens < 0 || dims.heads < 1 || dims.state_dim < 1 || num_shards < 1) return 0;
  const size_t states = (size_t)num_shards * dims.heads * 64 * dims.state_dim * sizeof(float);
  const size_t carry = (size_t)num_shards * dims.heads * sizeof(float);
  return 2 * ((states + 255) & ~size_t(255)) + ((carry + 255) & ~size_t(255));
}

ra_status ssd_cp_fwd(const float* x, const float* dt, const float* A, const float* B,
                     const float* C, const float* D, const int32_t* position_ids, ssd_dims dims,
                     int num_shards, float* y, float* final_state, void* workspace,
                     size_t workspace_bytes, void* stream) {
  NvtxRange nvtx("ssd_cp_fwd");
  if (dims.total_tokens < 0 || dims.heads < 1 || dims.groups < 1 || num_shards < 1)
    return RA_ERR_INVALID_ARG;
  if (dims.heads % dims.groups) return RA_ERR_INVALID_ARG;
  if (dims.head_dim != 64 || (dims.state_dim != 64 && dims.state_dim != 128))
    return RA_ERR_UNSUPPORTED;
  if (dims.total_tokens % num_shards) return RA_ERR_NOT_DIVISIBLE;
  if ((long long)dims.total_tokens * dims.heads * 64 >= (1LL << 40)) return RA_ERR_UNSUPPORTED;
  if (dims.total_tokens == 0) return RA_OK;
  if (!x || !dt || !A || !B || !C || !y) return RA_ERR_INVALID_ARG;
  // the kernels move x, B, C and y in 16-byte pieces
  for (const void* q : {static_cast<const void*>(x), static_cast<const void*>(B),
                        static_cast<const void*>(C), static_cast<const void*>(y)})
    if (reinterpret_cast<uintptr_t>(q) & 15u) return RA_ERR_INVALID_ARG;
  const size_t need = ssd_cp_workspace_size(dims, num_shards);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return RA_ERR_WORKSPACE;
  int dev;
  DeviceState* ds;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ra_status st = current_device(&dev, &ds);
    if (st != RA_OK) return st;
  }
  const size_t states = ((size_t)num_shards * dims.heads * 64 * dims.state_dim * sizeof(float) +
                         255) & ~size_t(255);
  char* w = static_cast<char*>(workspace);
  SsdParams p{};
  p.x = x;
  p.dt = dt;
  p.A = A;
  p.B = B;
  p.C = C;
  p.D = D;
  p.pos = position_ids;
  p.y = y;
  p.final_state = final_state;
  p.chunk_state = reinterpret_cast<float*>(w);
  p.incoming = reinterpret_cast<float*>(w + states);
  p.carry = reinterpret_cast<float*>(w + 2 * states);
  p.T = dims.total_tokens;
  p.H = dims.heads;
  p.G = dims.groups;
  p.N = dims.state_dim;
  p.R = num_shards;
  p.status = ds->status;
  SsdMaps maps;
  if (dims.state_dim == 128 &&
      (!encode_f32_rows(&maps.c, C, dims.total_tokens, dims.groups, 128, 128, 32, false) ||
       !encode_f32_rows(&maps.c_sw, C, dims.total_tokens, dims.groups, 128, 32, 128, true) ||
       !encode_f32_rows(&maps.b, B, dims.total_tokens, dims.groups, 128, 128, 32, false) ||
       !encode_f32_rows(&maps.x, x, dims.total_tokens, dims.heads, 64, 64, 128, false)))
    return RA_ERR_CUDA;
  return launch_ssd_cp(p, dims.state_dim == 128 ? &maps : nullptr,
                       static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RA_OK
             : RA_ERR_CUDA;
}

ra_status ringattn_get_status(void* stream) {
  int dev;
  DeviceState* ds;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ra_status st = current_device(&dev, &ds);
    if (st != RA_OK) return st;
  }
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return RA_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, ds->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return RA_ERR_CUDA;
  if (word != 0 && cudaMemset(ds->status, 0, sizeof(int)) != cudaSuccess) return RA_ERR_CUDA;
  return static_cast<ra_status>(word);
}

ra_status ringattn_selftest_wait_timeout(void* stream) {
  int dev;
  DeviceState* ds;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ra_status st = current_device(&dev, &ds);
    if (st != RA_OK) return st;
  }
  return launch_wait_timeout_selftest(ds->status, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RA_OK
             : RA_ERR_CUDA;
}

const char* ringattn_status_string(int status) {
  switch (status) {
    case RA_OK: return "ok";
    case RA_ERR_INVALID_ARG: return "invalid argument";
    case RA_ERR_NOT_DIVISIBLE: return "total_tokens not divisible by the number of shard chunks";
    case RA_ERR_UNSUPPORTED: return "unsupported dtype, head_dim or device";
    case RA_ERR_CUDA: return "CUDA runtime error";
    case RA_ERR_TIMEOUT: return "a kernel wait timed out";
    case RA_ERR_WORKSPACE: return "workspace missing or too small";
    case RA_ERR_BOUNDS: return "an index failed a bounds check of the debug build";
    default: return "unknown status";
  }
}

int ringattn_version(void) { return 100; }

int ringattn_debug_report(void* stream, long long* site, long long* index) {
  int dev;
  DeviceState* ds;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (current_device(&dev, &ds) != RA_OK) return -1;
  }
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return -1;
  unsigned long long where = 0;
  if (cudaMemcpy(&where, ds->status + 2, sizeof(where), cudaMemcpyDeviceToHost) != cudaSuccess)
    return -1;
  if (where != 0 && cudaMemset(ds->status + 2, 0, sizeof(where)) != cudaSuccess) return -1;
  if (site) *site = static_cast<long long>(where >> 48);
  if (index) *index = static_cast<long long>(where & 0xFFFFFFFFFFFFull);
#ifdef RINGATTN_DEBUG
  return 1;
#else
  return 0;
#endif
}

ra_status ringattn_plan_fwd(const int32_t* cu_seqlens, ra_dims dims, int num_shards,
                            int shard_layout, int causal, int32_t* items, int max_items,
                            int32_t* segments, int max_segments, int* num_items,
                            int* num_segments) {
  PlanInput in;
  // the plan does not depend on dtype or head_dim: check shapes only
  ra_dims d = dims;
  d.dtype = RA_FP32;
  d.head_dim = 64;
  ra_status st = check_problem(cu_seqlens, d, num_shards, shard_layout, causal, &in);
  if (st != RA_OK) return st;
  if (!num_items || !num_segments) return RA_ERR_INVALID_ARG;
  const Plan plan = build_fwd_plan(in);
  *num_items = static_cast<int>(plan.items.size());
  *num_segments = static_cast<int>(plan.segs.size());
  if (*num_items > max_items || *num_segments > max_segments) return RA_ERR_WORKSPACE;
  if (*num_items && items) std::memcpy(items, plan.items.data(), plan.items.size() * sizeof(PlanItem));
  if (*num_segments && segments)
    std::memcpy(segments, plan.segs.data(), plan.segs.size() * sizeof(PlanSegment));
  return RA_OK;
}

ra_status ringattn_plan_fwd_fused(const int32_t* cu_seqlens, ra_dims dims, int num_shards,
                                  int shard_layout, int causal, int num_sms, int32_t* items,
                                  int max_items, int32_t* segments, int max_segments,
                                  int* num_items, int* num_segments) {
  PlanInput in;
  ra_dims d = dims;
  d.dtype = RA_FP32;
  d.head_dim = 64;
  ra_status st = check_problem(cu_seqlens, d, num_shards, shard_layout, causal, &in);
  if (st != RA_OK) return st;
  if (!num_items || !num_segments || num_sms < 1) return RA_ERR_INVALID_ARG;
  const FusedPlan plan = build_fused_plan(build_fwd_plan(in), num_sms);
  *num_items = static_cast<int>(plan.items.size());
  *num_segments = static_cast<int>(plan.segs.size());
  if (*num_items > max_items || *num_segments > max_segments) return RA_ERR_WORKSPACE;
  if (*num_items && items) std::memcpy(items, plan.items.data(), plan.items.size() * sizeof(PlanItem));
  if (*num_segments && segments)
    std::memcpy(segments, plan.segs.data(), plan.segs.size() * sizeof(PlanSegment));
  return RA_OK;
}

ra_status ringattn_plan_bwd(const int32_t* cu_seqlens, ra_dims dims, int num_shards,
                            int shard_layout, int causal, int32_t* items, int max_items,
                            int32_t* segments, int max_segments, int* num_items,
                            int* num_segments) {
  PlanInput in;
  ra_dims d = dims;
  d.dtype = RA_FP32;
  d.head_dim = 64;
  ra_status st = check_problem(cu_seqlens, d, num_shards, shard_layout, causal, &in);
  if (st != RA_OK) return st;
  if (!num_items || !num_segments) return RA_ERR_INVALID_ARG;
  const BwdPlan plan = build_bwd_plan(in);
  *num_items = static_cast<int>(plan.items.size());
  *num_segments = static_cast<int>(plan.segs.size());
  if (*num_items > max_items || *num_segments > max_segments) return RA_ERR_WORKSPACE;
  if (*num_items && items) std::memcpy(items, plan.items.data(), plan.items.size() * sizeof(BwdItem));
  if (*num_segments && segments)
    std::memcpy(segments, plan.segs.data(), plan.segs.size() * sizeof(BwdSegment));
  return RA_OK;
}

}  // extern "C"
