// Host-side shard / ring-step planner.
//
// Turns (T, heads, P, layout, causal, documents) into a flat work list the
// kernels walk: each item is one CTA's worth of queries (two 128-row query
// tiles that share a key/value head) together with the list of key ranges
// it must visit, in ring order.  Work that the causal or document mask hides
// completely is never emitted (causal skip), and items are ordered longest
// first inside each pass over the key/value heads.
#pragma once
#include <cstdint>
#include <string>
#include <vector>

namespace ra {

constexpr int kTileRows = 128;  // query rows per tile; also keys per K/V tile

// One CTA of work: query tiles A (index 0) and B (index 1).
struct PlanItem {
  int32_t q0[2];       // first query token of each tile
  int32_t qlen[2];     // valid rows of each tile (0 = tile absent)
  int32_t head[2];     // query head of each tile
  int32_t seg_begin;   // first segment of this item
  int32_t seg_count;   // segments, in ring order
  int32_t rank;        // virtual rank that owns the queries
  int32_t cost;        // K/V tiles visited (scheduling weight)
  int32_t mask_lo[2];  // per tile: largest first-visible key over its rows
  int32_t mask_hi[2];  // per tile: smallest end-of-visible-keys over its rows
  int32_t pass;        // pass over key/value heads (heads_k_stride groups)
  int32_t part;        // -1: writes the output; else the partial-result slot of a
                       // split item (fused forward only, see build_fused_plan)
};
static_assert(sizeof(PlanItem) == 16 * 4, "PlanItem is 16 int32");

// Keys [k0, k1) of rank `src`, visited at ring step `step` (all-gather
// exchange: one step 0 and src -1, the keys gathered from every rank).
struct PlanSegment {
  int32_t k0, k1, step, src;
};

struct PlanInput {
  int T = 0, hq = 0, hkv = 0;
  int num_shards = 1, layout = 0, causal = 0, heads_k_stride = 1;
  int exchange = 0;  // 0: ring order of K/V shards; 1: all-gathered, token order
  std::vector<int32_t> cu;  // num_docs + 1 offsets (always filled: one doc if none given)
  // One ring step of one rank (multi-GPU form): only the queries of rank
  // q_rank and only the keys of rank k_rank (-1: every rank).  Ring exchange only.
  int q_rank = -1, k_rank = -1;
};

struct Plan {
  std::vector<PlanItem> items;
  std::vector<PlanSegment> segs;
  std::vector<int32_t> cu;  // document offsets (copied to the device with the plan)
};

// Backward, key/value side: one CTA per 128-key tile of one key/value head.
// Its query ranges are those of the ring steps: at step s the K/V shard of
// rank `src` sits on rank (src + s) mod P, whose queries contribute to its
// dK, dV.  In the whole-GPU plan they come from the end of the sequence down
// (L2 reuse across co-resident CTAs); with a rank filter, in ring order.
struct BwdItem {
  int32_t k0;         // first key of the tile
  int32_t klen;       // keys of the tile (<= 128; the tile stays in one chunk)
  int32_t kv_head;
  int32_t src;        // rank that holds the keys
  int32_t seg_begin;  // query segments, in ring order
  int32_t seg_count;
  int32_t cost;       // (query tile, head) pairs visited
  int32_t pad;
};
static_assert(sizeof(BwdItem) == 8 * 4, "BwdItem is 8 int32");

// Queries [q0, q1) of rank `rank`, visited at ring step `step` (all-gather
// exchange: step 0 and rank -1, every rank's queries in token order).
struct BwdSegment {
  int32_t q0, q1, step, rank;
};

struct BwdPlan {
  std::vector<BwdItem> items;
  std::vector<BwdSegment> segs;
};

// Two items that split one item's key tiles: the same query tiles, each half
// writing its partial (O, lse) to a slot, merged afterwards.
struct SplitPair {
  int32_t q0[2], qlen[2], head[2];
  int32_t part[2];  // partial-result slots of the first and second half
};
static_assert(sizeof(SplitPair) == 8 * 4, "SplitPair is 8 int32");

// The persistent fused forward's work list: the plan's items in claim order,
// with long items split (see build_fused_plan).
struct FusedPlan {
  std::vector<PlanItem> items;
  std::vector<PlanSegment> segs;
  std::vector<SplitPair> pairs;
};

// Claim order and splits of the forward plan for a persistent launch of
// `num_ctas` CTAs that claim items as they become free:
//  - passes over key/value heads are merged into ordering groups of at least
//    2 num_ctas items (the last smaller rest joins the group before it), and
//    items run longest first inside a group.  A big problem keeps one pass
//    per group, so the K/V of few heads are in flight at once; a small one
//    is ordered longest first as a whole, which is what balances it.
//  - when an item is longer than the mean work per CTA, it is split into two
//    items over the first and the second half of its key tiles (in ring
//    order); each half writes a partial (O, lse) that a merge folds together.
FusedPlan build_fused_plan(const Plan& plan, int num_ctas);

// Builds the key/value-side backward schedule.  `in` must have passed plan_check.
BwdPlan build_bwd_plan(const PlanInput& in);

// Key ranges [a, b) of the chunks rank r holds (one for CONTIGUOUS, two for
// ZIGZAG, ascending).
void rank_chunks(int T, int P, int layout, int r, int out[2][2], int* n);

// Validates the input; returns "" if fine, else a reason.
std::string plan_check(const PlanInput& in);

// Builds the forward schedule.  `in` must have passed plan_check.
Plan build_fwd_plan(const PlanInput& in);

}  // namespace ra
