/*
 * ringattn.h -- C ABI of the B300 (sm_103a) ring-attention library.
 *
 * Ring attention (context parallelism) splits the token sequence into P
 * shards ("virtual ranks"); each shard's queries visit every key/value shard
 * in ring order and the partial results are aggregated (axolotl "Sequence
 * Parallelism" page, introduction and "Implementation Details"; aicassindra
 * "tm_sp_math", section "Context parallelism is the axis that is
 * independent": K/V blocks rotate around a ring so no device holds the whole
 * sequence, at the price of a causal-mask load-balance problem).  Here all P
 * virtual ranks run on ONE GPU: a ring step indexes a K/V chunk that is
 * already resident in device memory, and the partial results of the steps are
 * folded with a log-sum-exp merge, so no T x T score matrix is ever formed
 * (FlashAttention-style tiling: archcrux interview page; aicassindra page,
 * "Why FlashAttention makes SP more valuable").
 *
 * Conventions shared by every call:
 *   - Tensors are dense, row-major, 16-byte aligned DEVICE memory owned by the
 *     caller.  q / out / dout / dq: [T, Hq, D]; k / v / dk / dv: [T, Hkv, D];
 *     lse: fp32 [Hq, T], natural logarithm.  T = dims.total_tokens.
 *   - Token order is the natural global order for every shard layout: the
 *     layout changes the schedule (which shard's queries visit which K/V
 *     chunk at which ring step), never the meaning of the result.
 *   - cu_seqlens, when not NULL, is a HOST array of num_seqs + 1 int32
 *     offsets (0 = cu[0] <= cu[1] <= ... <= cu[num_seqs] = T) describing
 *     packed documents; positions restart at each document (axolotl page,
 *     "Sample Packing with Sequence Parallelism"), so a query sees only keys
 *     of its own document.  NULL means one document of T tokens.  The library
 *     copies what it needs; the array may be freed after the call returns.
 *   - Shards: CONTIGUOUS gives rank r tokens [r T/P, (r+1) T/P); ZIGZAG cuts
 *     the sequence into 2P chunks and gives rank r chunks r and 2P-1-r, which
 *     balances causal work.  T must be divisible by P (CONTIGUOUS) or 2P
 *     (ZIGZAG), else RA_ERR_NOT_DIVISIBLE: the pages require the sequence to
 *     split into equal chunks (axolotl page, "Implementation Details";
 *     aicassindra page, "The knob you cannot turn on its own": s must be
 *     divisible by the degree).
 *   - GQA: query head h reads key/value head h / (Hq / Hkv).
 *   - heads_k_stride (0 means 1) is the number of key/value heads processed
 *     per pass over the ring (axolotl page, "Configuration").  It changes the
 *     order of work only; results do not depend on it.  It must divide Hkv.
 *   - Softmax scale is 1 / sqrt(D).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Argument errors are returned synchronously and launch
 *     nothing.  There is no fallback path: an unsupported shape or dtype
 *     returns RA_ERR_UNSUPPORTED (the archcrux page warns that a silent
 *     fallback of the attention kernel defeats the memory plan).
 *   - Errors raised inside kernels (a bounded wait that timed out) are
 *     recorded in a device status word that ringattn_get_status() reads.
 *   - The library allocates no device memory per call.  It caches work lists
 *     (one small device buffer per distinct problem, up to 32 problems) and
 *     keeps one status word and 64 work counters of the persistent forward
 *     per device in static device arrays.
 */
#ifndef RINGATTN_H
#define RINGATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = -1,   /* null pointer, bad size, bad cu_seqlens */
  RA_ERR_NOT_DIVISIBLE = -2, /* T not divisible by P (or 2P for ZIGZAG) */
  RA_ERR_UNSUPPORTED = -3,   /* dtype / head_dim / device not supported */
  RA_ERR_CUDA = -4,          /* a CUDA runtime call failed */
  RA_ERR_TIMEOUT = -5,       /* a kernel's bounded wait gave up */
  RA_ERR_WORKSPACE = -6,     /* workspace missing or too small */
  RA_ERR_BOUNDS = -7         /* debug build only: an index failed its bounds check */
} ra_status;

typedef enum { RA_BF16 = 0, RA_FP32 = 1 } ra_dtype;
typedef enum { RA_CONTIGUOUS = 0, RA_ZIGZAG = 1 } ra_layout;

/*
 * The two ring_attn_func choices of the axolotl page ("Configuration"):
 *   RA_RING (batch_ring): at ring step s rank r holds the K/V shard of rank
 *     (r - s) mod P, and its partial results are merged step by step;
 *   RA_ALLGATHER (varlen_llama3): every rank gathers the K/V of all shards,
 *     heads_k_stride key/value heads at a time, and attends to them in token
 *     order in one pass (the page's default with sample packing).
 * On one GPU both read K/V where it already lies; they differ in the order
 * the key tiles are visited, not in the result.  The stepwise forward runs
 * RA_ALLGATHER as a single step.
 */
typedef enum { RA_RING = 0, RA_ALLGATHER = 1 } ra_exchange;

typedef struct {
  int total_tokens;   /* T >= 0 */
  int num_seqs;       /* packed documents; ignored when cu_seqlens is NULL */
  int hq;             /* query heads */
  int hkv;            /* key/value heads, divides hq */
  int head_dim;       /* D: 64 or 128 */
  int dtype;          /* ra_dtype of q, k, v, out (and dout, dq, dk, dv) */
  int heads_k_stride; /* key/value heads per ring pass; 0 = 1 */
  int grad_fp32;      /* backward only: 1 = dq, dk, dv are fp32 whatever dtype
                         is (bf16 cannot hold gradients of magnitude >= 4 to
                         within 1/64); 0 = they are in dtype */
  int kv_exchange;    /* ra_exchange: how a rank reaches the other shards' K/V */
} ra_dims;

/*
 * Ring-attention forward (fused): every virtual rank's queries visit the K/V
 * chunks of ranks (r - s) mod P for ring steps s = 0 .. P-1 in order; K/V
 * tiles that the causal or document mask hides completely are skipped; the
 * running (max, sum, O) of the online softmax is carried across tiles and
 * steps, which is the log-sum-exp merge of the per-step partial results.
 *   out: [T, Hq, D] in dims.dtype;  lse: fp32 [Hq, T].
 * fp32 inputs run a CUDA-core path (fp32 arithmetic throughout); bf16 inputs
 * run the tensor-core path (bf16 operands, fp32 accumulation).
 */
ra_status ringattn_fwd(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                       ra_dims dims, int num_shards, int shard_layout, int causal, void* out,
                       float* lse, void* stream);

/*
 * Ring-attention forward, one launch per ring step: step s computes every
 * rank's partial result over the single K/V shard it holds at that step
 * (rows that see no key there get O = 0, lse = -inf), and attn_lse_merge
 * folds it into the running result.  Same result as ringattn_fwd up to
 * rounding; it is the literal ring algorithm, and the shape one step of a
 * multi-GPU ring would take.  Needs a caller-owned device workspace of
 * ringattn_fwd_stepwise_workspace_size(dims) bytes (fp32 partials).
 */
size_t ringattn_fwd_stepwise_workspace_size(ra_dims dims);
ra_status ringattn_fwd_stepwise(const void* q, const void* k, const void* v,
                                const int32_t* cu_seqlens, ra_dims dims, int num_shards,
                                int shard_layout, int causal, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Stepwise forward that allocates nothing.  There is no counterpart on the
 * pages: this is an interface for callers that cannot allocate device memory
 * where they call attention (inside an allocator or memory-pool callback, or
 * in a host runtime that only hands out input and output buffers).  Same
 * arguments, same work and same result as ringattn_fwd_stepwise, but the fp32
 * partial results and the work list live in one library-owned __device__
 * array of RA_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads the
 * library holds until the process exits.  No cudaMalloc, cudaFree or other
 * allocating call is made.
 *   - Problems whose partials and work list need more than the array holds
 *     (about T * Hq * (D + 1) * 8 bytes plus the work list) return
 *     RA_ERR_WORKSPACE and launch nothing.
 *   - All calls share the array: calls that overlap on the GPU (different
 *     streams or threads) race; calls on one stream are ordered.
 *   - Every call builds its work list on the host and copies it into the
 *     array with cudaMemcpyAsync on `stream` (from host memory that the call
 *     frees when it returns) before it launches the kernels.
 *   - The first call on a device looks up the array's device address; make
 *     that first call before any stream capture.
 */
#define RA_NOALLOC_SCRATCH_BYTES (32u << 20)
ra_status ringattn_fwd_stepwise_noalloc(const void* q, const void* k, const void* v,
                                        const int32_t* cu_seqlens, ra_dims dims, int num_shards,
                                        int shard_layout, int causal, void* out, float* lse,
                                        void* stream);

/*
 * Ring-attention backward.  Inputs q, k, v, out, lse from the forward and
 * dout = dL/dout; outputs dq [T, Hq, D], dk and dv [T, Hkv, D] (summed over
 * the query heads of each GQA group), in dims.dtype, or fp32 when
 * dims.grad_fp32 is set.  With
 * P_ij = exp(scale q_i.k_j - lse_i), D_i = dout_i . out_i:
 *   dv_j = sum_i P_ij dout_i,  dS_ij = P_ij (dout_i . v_j - D_i),
 *   dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i.
 * Needs a caller-owned device workspace of ringattn_bwd_workspace_size(dims)
 * bytes: the fp32 D_i vector [Hq, T], and for bf16 gradients of long
 * sequences the fp32 sums of dk and dv (2 x [T, Hkv, D], see below).  dq
 * accumulates in tensor memory over each query tile's whole ring, and dk,
 * dv over each key tile's, so no output is accumulated with atomics and the
 * result does not depend on the schedule.  bf16 runs on the tensor cores,
 * fp32 on CUDA cores.
 *
 * The tensor cores' fp32 accumulation loses a little toward zero at every
 * step (measured on B300: about 2^-26 of the sum per K = 16 step); a key
 * tile's walk is up to T G / 16 such steps for G query heads per key/value
 * head, which shrank dk and dv by about 2e-9 T at G = 4.  So the dk/dv
 * kernel moves its sums to fp32 memory and restarts them every
 * ringattn_set_bwd_flush_interval() (query tile, head) pairs (default 1024:
 * only walks of more than 1024 = (T / 128) G pairs flush, e.g. above 32K
 * tokens at G = 4): into dk, dv when they are fp32, else into the
 * workspace's fp32 sums, which the last step adds before rounding to bf16.
 */
size_t ringattn_bwd_workspace_size(ra_dims dims);

/*
 * Sets the dk/dv flush interval above, in (query tile, head) pairs; 0 turns
 * the flushes off.  Process-wide; it changes ringattn_bwd_workspace_size()'s
 * answer, so set it before sizing a workspace and not while a backward call
 * is being made on another thread.  RA_ERR_INVALID_ARG for pairs < 0.
 */
ra_status ringattn_set_bwd_flush_interval(int pairs);
ra_status ringattn_bwd(const void* q, const void* k, const void* v, const void* out,
                       const float* lse, const void* dout, const int32_t* cu_seqlens,
                       ra_dims dims, int num_shards, int shard_layout, int causal, void* dq,
                       void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream);

/*
 * One ring step of one rank of a MULTI-GPU ring, on shard-local buffers.
 * The pages' deployment of ring attention puts one rank on each GPU: the rank
 * keeps its own query rows, and the K/V blocks rotate around the ring so that
 * no device ever holds the whole sequence (aicassindra "tm_sp_math", "Context
 * parallelism is the axis that is independent"; axolotl "Sequence
 * Parallelism" page, introduction and "Implementation Details": results are
 * aggregated through a ring communication pattern).  The caller moves the
 * K/V shards between GPUs (into this GPU's own memory) and calls one step per
 * shard; these calls do the step's attention and fold it into the rank's
 * running result.  bf16 only, RA_RING exchange only (else RA_ERR_UNSUPPORTED).
 *   - dims describe the WHOLE problem (total_tokens = T, cu_seqlens of the
 *     whole sequence, host array); Tr = T / num_shards rows per rank.
 *   - rank r's buffers hold its rows back to back: CONTIGUOUS tokens
 *     [r Tr, (r+1) Tr); ZIGZAG chunk r then chunk 2P-1-r (each Tr / 2 tokens).
 *   - step s (0 .. P-1) is the step at which rank r holds the K/V shard of
 *     rank src = (r - s) mod P; k, v are that shard's rows [Tr, Hkv, D], laid
 *     out as src's own buffers.  Steps must be called in order s = 0 .. P-1
 *     on one stream.  Masks use global positions, so causal and document
 *     masks are exact; a shard the rank cannot see (causal, src > r with
 *     CONTIGUOUS) gives an all-masked partial that the merge ignores.
 *
 * Forward: q [Tr, Hq, D]; o_acc fp32 [Tr, Hq, D] and lse_acc fp32 [Hq, Tr]
 * hold the running result between steps (unused when P = 1); the last step
 * (s = P-1) writes out [Tr, Hq, D] bf16 and lse [Hq, Tr] (natural log).
 * Steps after the first need a device workspace of
 * ringattn_fwd_rank_workspace_size(dims, num_shards) bytes (one step's fp32
 * partial result).
 */
size_t ringattn_fwd_rank_workspace_size(ra_dims dims, int num_shards);
ra_status ringattn_fwd_rank_step(const void* q, const void* k, const void* v,
                                 const int32_t* cu_seqlens, ra_dims dims, int num_shards,
                                 int shard_layout, int causal, int rank, int step, float* o_acc,
                                 float* lse_acc, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * Backward of one ring step of one rank (same conventions as
 * ringattn_fwd_rank_step).  q, out, lse, dout are the rank's own rows (out
 * and lse from its forward); k, v the K/V shard it holds at step s.  The
 * gradients are fp32: dq [Tr, Hq, D] of the rank's rows; dk, dv [Tr, Hkv, D]
 * of the keys of rank src, which travel around the ring with k and v.  Step 0
 * (src = rank) writes dq and the rank's own dk, dv; every later step adds to
 * them, so after step P-1 dq is complete and the dk, dv the rank holds (those
 * of rank (rank + 1) mod P) are complete and go back to their owner.  The
 * workspace (ringattn_bwd_rank_workspace_size bytes: D_i = dout_i . out_i of
 * the rank's rows) is filled by step 0 and must be kept for the later steps.
 */
size_t ringattn_bwd_rank_workspace_size(ra_dims dims, int num_shards);
ra_status ringattn_bwd_rank_step(const void* q, const void* k, const void* v, const void* out,
                                 const float* lse, const void* dout, const int32_t* cu_seqlens,
                                 ra_dims dims, int num_shards, int shard_layout, int causal,
                                 int rank, int step, float* dq, float* dk, float* dv,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Log-sum-exp merge of two partial attention results over disjoint key sets,
 * in place into (o_a, lse_a) -- how the pages' ring steps are aggregated
 * (axolotl page, introduction).  Per row:
 *   lse = max(a, b) + log1p(exp(-|a - b|)),
 *   o   = exp(a - lse) o_a + exp(b - lse) o_b;
 * a side with lse = -inf contributes nothing; two empty sides give o = 0,
 * lse = -inf.  o_*: [rows, heads, head_dim] in dtype; lse_*: fp32
 * [heads, rows].  rows = 0 is a no-op.
 */
ra_status attn_lse_merge(void* o_a, float* lse_a, const void* o_b, const float* lse_b, int rows,
                         int heads, int head_dim, int dtype, void* stream);

/*
 * Context-parallel selective scan of a Mamba2 layer (the SSD recurrence),
 * fp32.  The axolotl "Sequence Parallelism" page ("Mamba/SSM Hybrid Models")
 * runs hybrid models' SSM layers under context parallelism: each rank scans
 * its chunk of the sequence, passes its final hidden state to the next rank,
 * and an additive correction accounts for the state it did not start from
 * (the recurrence is linear in its initial state, so no second forward pass
 * is needed); packed samples reset the state where they start, found from
 * position_ids.  Per head h of group g = h / (heads / groups) and token t:
 *   S <- 0 when position_ids[t] == 0 (a packed sample starts);
 *   S <- exp(dt[t,h] A[h]) S + dt[t,h] x[t,h,:] B[t,g,:]^T;
 *   y[t,h,:] = S C[t,g,:] + D[h] x[t,h,:],
 * starting from S = 0.  All num_shards ranks (contiguous chunks of T /
 * num_shards tokens; T must divide, else RA_ERR_NOT_DIVISIBLE) run on this
 * GPU: chunk scans from zero, the ring of states, then the correction.
 *   x, y: [T, heads, 64] fp32;  dt: [T, heads];  A, D: [heads] (D may be
 *   NULL);  B, C: [T, groups, state_dim] fp32, state_dim 64 or 128;
 *   position_ids: DEVICE int32 [T], or NULL for one sample;
 *   final_state: [heads, 64, state_dim] fp32 or NULL -- the state after the
 *   last token (what a following chunk would receive).
 * Device pointers owned by the caller; x, B, C and y 16-byte aligned (else
 * RA_ERR_INVALID_ARG); asynchronous on `stream`; needs a device workspace of
 * ssd_cp_workspace_size(dims, num_shards) bytes (256-byte aligned; each
 * rank's final state, the states passed along the ring, the carry factors).
 * State size 128 scans and corrects on the tensor cores with fp16 operands
 * split into hi + lo parts (three products per term, fp32 accumulation);
 * state size 64 on fp32 CUDA cores.  Both are accurate to about 1e-6 of the
 * output scale.
 */
typedef struct {
  int total_tokens; /* T >= 0 */
  int heads;        /* H */
  int head_dim;     /* 64 */
  int state_dim;    /* N: 64 or 128 */
  int groups;       /* G: divides heads (B and C are shared inside a group) */
} ssd_dims;
size_t ssd_cp_workspace_size(ssd_dims dims, int num_shards);
ra_status ssd_cp_fwd(const float* x, const float* dt, const float* A, const float* B,
                     const float* C, const float* D, const int32_t* position_ids, ssd_dims dims,
                     int num_shards, float* y, float* final_state, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Synchronises `stream`, returns the first kernel-side error recorded since
 * the last call (RA_OK if none) and clears it. */
ra_status ringattn_get_status(void* stream);

/*
 * Self-test of the failure path of every kernel wait.  Launches one CTA that
 * waits on a barrier nothing ever arrives at; the wait gives up after its
 * time limit (1 s), records RA_ERR_TIMEOUT in the status word and the kernel
 * exits normally, so the context stays usable.  Asynchronous on `stream`;
 * ringattn_get_status(stream) afterwards returns RA_ERR_TIMEOUT (and clears
 * it).  Returns RA_OK if the launch succeeded.  The status word is shared by
 * every stream of the device, so run the self-test while no other call of
 * this library is in flight on the device: a concurrent caller's
 * ringattn_get_status would otherwise report (and clear) this timeout.
 */
ra_status ringattn_selftest_wait_timeout(void* stream);

/*
 * Debug build.  libringattn_debug.so is this library compiled with
 * RINGATTN_DEBUG: every kernel checks each global index it computes (work-list
 * entries, tensor rows and heads, output, lse and partial-result offsets)
 * against its array's extent before using it.  A failed check records
 * RA_ERR_BOUNDS in the status word (read by ringattn_get_status) and skips the
 * access (a load reads element 0 instead), so the kernel neither touches
 * memory outside its buffers nor traps.  ringattn_debug_report synchronises
 * `stream`, stores the first failed check since its last call as a site
 * number and the index (both 0 if none), clears it, and returns 1 in the
 * debug build, 0 in the normal build (which makes no checks) and -1 on a CUDA
 * error.
 */
int ringattn_debug_report(void* stream, long long* site, long long* index);

/* Static text for a status code. */
const char* ringattn_status_string(int status);

/* Library version as MAJOR * 10000 + MINOR * 100 + PATCH. */
int ringattn_version(void);

/*
 * Host-only work-list introspection (no GPU needed), for tests and tools.
 * Fills the forward schedule: items of RA_PLAN_ITEM_FIELDS int32 each and
 * segments of RA_PLAN_SEG_FIELDS int32 each (layouts below).  Returns
 * RA_OK and the counts; if a capacity is too small nothing is written
 * beyond it and RA_ERR_WORKSPACE is returned with the counts still set.
 *   item:    q0_a, q0_b, qlen_a, qlen_b, head_a, head_b, seg_begin,
 *            seg_count, rank, cost (kv tiles), mask_lo_a, mask_lo_b,
 *            mask_hi_a, mask_hi_b, pass, part (-1 here; see below)
 *            (tile a/b: first query row, valid rows, query head; the key
 *            range a tile may skip masking in is [mask_lo, mask_hi))
 *   segment: k0, k1, step, src  (keys [k0, k1) of rank src at ring step)
 */
#define RA_PLAN_BWD_ITEM_FIELDS 8
#define RA_PLAN_ITEM_FIELDS 16
#define RA_PLAN_SEG_FIELDS 4
ra_status ringattn_plan_fwd(const int32_t* cu_seqlens, ra_dims dims, int num_shards,
                            int shard_layout, int causal, int32_t* items, int max_items,
                            int32_t* segments, int max_segments, int* num_items,
                            int* num_segments);

/*
 * Host-only: the work list the fused forward (ringattn_fwd) runs on a GPU of
 * num_sms SMs, in the order its persistent CTAs claim it (same item and
 * segment layout as ringattn_plan_fwd).  Passes over key/value heads are
 * merged into ordering groups of at least 2 num_sms items, longest first
 * inside a group; an item longer than the mean work per SM is split into two
 * items over the first and second half of its key tiles in ring order, whose
 * `part` fields are 2 i and 2 i + 1 (their partial results are merged with
 * the log-sum-exp rule after the launch).  Same return conventions.
 */
ra_status ringattn_plan_fwd_fused(const int32_t* cu_seqlens, ra_dims dims, int num_shards,
                                  int shard_layout, int causal, int num_sms, int32_t* items,
                                  int max_items, int32_t* segments, int max_segments,
                                  int* num_items, int* num_segments);

/*
 * Host-only backward work list (key side): items of RA_PLAN_BWD_ITEM_FIELDS
 * int32 (k0, klen, kv_head, src, seg_begin, seg_count, cost, pad) and
 * segments of RA_PLAN_SEG_FIELDS int32 (q0, q1, step, rank: queries
 * [q0, q1) of rank `rank` meet the tile's keys at ring step `step`).  Same
 * return conventions as ringattn_plan_fwd.
 */
ra_status ringattn_plan_bwd(const int32_t* cu_seqlens, ra_dims dims, int num_shards,
                            int shard_layout, int causal, int32_t* items, int max_items,
                            int32_t* segments, int max_segments, int* num_items,
                            int* num_segments);

/*
 * Per-kernel timing of this library's launches (profiling support; the pages
 * ask for peak memory and timed steps when diagnosing a long-context run,
 * archcrux interview page).  While tracing is on, every kernel launch is
 * bracketed by two CUDA events recorded on the stream it is launched on.
 * ringattn_trace_collect() waits for all recorded launches, fills one entry
 * per kernel name (launch count and summed device milliseconds), clears the
 * record and returns RA_OK; with too few entries it fills max_entries of
 * them, still sets *num_entries to the number needed and returns
 * RA_ERR_WORKSPACE.  Host-only bookkeeping: no device memory is allocated.
 * At most 65536 launches are recorded between two collects.
 */
typedef struct {
  char kernel[40];  /* kernel name, NUL-terminated */
  int launches;
  double total_ms;
} ra_trace_entry;
ra_status ringattn_trace_enable(int on);
ra_status ringattn_trace_collect(ra_trace_entry* entries, int max_entries, int* num_entries);

#ifdef __cplusplus
}
#endif

#endif /* RINGATTN_H */
