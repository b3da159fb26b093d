// Host-side shard / ring-step planner (see planner.h).
//
// Ring schedule: virtual rank r holds the query rows of its chunk(s); at ring
// step s = 0 .. P-1 it uses the keys/values of rank (r - s) mod P, so step 0
// is its own shard (axolotl "Sequence Parallelism" page: results aggregated
// through a ring pattern; aicassindra "tm_sp_math", "Context parallelism is
// the axis that is independent": K/V blocks rotate around the ring).
// ZIGZAG gives rank r chunks r and 2P-1-r of 2P, which evens out the causal
// work per rank (the "causal-mask load-balance problem" on the same page).
#include "planner.h"

#include <algorithm>
#include <climits>

namespace ra {

void rank_chunks(int T, int P, int layout, int r, int out[2][2], int* n) {
  if (layout == 0) {
    const int C = T / P;
    out[0][0] = r * C;
    out[0][1] = (r + 1) * C;
    *n = 1;
  } else {
    const int C = T / (2 * P);
    out[0][0] = r * C;
    out[0][1] = (r + 1) * C;
    out[1][0] = (2 * P - 1 - r) * C;
    out[1][1] = (2 * P - r) * C;
    *n = 2;
  }
}

std::string plan_check(const PlanInput& in) {
  if (in.T < 0) return "total_tokens < 0";
  if (in.hq < 1 || in.hkv < 1) return "head counts must be >= 1";
  if (in.hq % in.hkv) return "hq must be a multiple of hkv";
  if (in.num_shards < 1 || in.num_shards > 65536) return "num_shards out of range";
  if (in.layout != 0 && in.layout != 1) return "unknown shard layout";
  if (in.heads_k_stride < 1 || in.hkv % in.heads_k_stride) return "heads_k_stride must divide hkv";
  if (in.exchange != 0 && in.exchange != 1) return "unknown K/V exchange";
  if (in.q_rank < -1 || in.q_rank >= in.num_shards || in.k_rank < -1 ||
      in.k_rank >= in.num_shards)
    return "rank out of range";
  if ((in.q_rank >= 0 || in.k_rank >= 0) && in.exchange != 0)
    return "a single ring step needs the ring exchange";
  if (in.cu.size() < 2) return "cu_seqlens needs at least two entries";
  if (in.cu.front() != 0 || in.cu.back() != in.T) return "cu_seqlens must run from 0 to T";
  for (size_t i = 1; i < in.cu.size(); ++i)
    if (in.cu[i] < in.cu[i - 1]) return "cu_seqlens must not decrease";
  return "";
}

namespace {

struct Docs {
  const std::vector<int32_t>& cu;
  int doc_of(int t) const {  // last document d with cu[d] <= t
    auto it = std::upper_bound(cu.begin(), cu.end(), t);
    return static_cast<int>(it - cu.begin()) - 1;
  }
  int start(int t) const { return cu[doc_of(t)]; }
  int end(int t) const { return cu[doc_of(t) + 1]; }
};

}  // namespace

Plan build_fwd_plan(const PlanInput& in) {
  Plan plan;
  plan.cu = in.cu;
  if (in.T == 0) return plan;
  const Docs docs{plan.cu};
  const int P = in.num_shards;
  const int G = in.hq / in.hkv;
  const bool head_pairs = (G % 2) == 0;
  const int npass = in.hkv / in.heads_k_stride;

  for (int pass = 0; pass < npass; ++pass) {
    const size_t first_item = plan.items.size();
    for (int g = pass * in.heads_k_stride; g < (pass + 1) * in.heads_k_stride; ++g) {
      for (int r = 0; r < P; ++r) {
        if (in.q_rank >= 0 && r != in.q_rank) continue;
        int qch[2][2], nq;
        rank_chunks(in.T, P, in.layout, r, qch, &nq);
        for (int c = 0; c < nq; ++c) {
          const int a = qch[c][0], b = qch[c][1];
          const int row_step = head_pairs ? kTileRows : 2 * kTileRows;
          for (int t0 = a; t0 < b; t0 += row_step) {
            const int hstep = head_pairs ? 2 : 1;
            for (int h = g * G; h < (g + 1) * G; h += hstep) {
              PlanItem it{};
              it.part = -1;
              for (int x = 0; x < 2; ++x) {
                int q0 = head_pairs ? t0 : t0 + x * kTileRows;
                int len = std::max(0, std::min(kTileRows, b - q0));
                it.q0[x] = q0;
                it.qlen[x] = len;
                it.head[x] = head_pairs ? h + x : h;
                if (len > 0) {
                  const int last = q0 + len - 1;
                  it.mask_lo[x] = docs.start(last);
                  it.mask_hi[x] = in.causal ? q0 + 1 : docs.end(q0);
                } else {
                  it.mask_lo[x] = 0;
                  it.mask_hi[x] = 0;
                }
              }
              // keys any row of the item may see: from the first row's
              // document start to the last row (causal) or its document end
              const int first_row = it.q0[0];
              const int last_row =
                  it.qlen[1] > 0 ? it.q0[1] + it.qlen[1] - 1 : it.q0[0] + it.qlen[0] - 1;
              const int lo = docs.start(first_row);
              const int hi = in.causal ? last_row + 1 : docs.end(last_row);
              it.seg_begin = static_cast<int32_t>(plan.segs.size());
              it.rank = r;
              it.pass = pass;
              int cost = 0;
              if (in.exchange == 1) {
                // all-gathered K/V: the visible keys in token order, one range
                if (lo < hi) {
                  plan.segs.push_back(PlanSegment{lo, hi, 0, -1});
                  cost += (hi - lo + kTileRows - 1) / kTileRows;
                }
              } else {
                for (int s = 0; s < P; ++s) {
                  const int src = ((r - s) % P + P) % P;
                  if (in.k_rank >= 0 && src != in.k_rank) continue;
                  int kch[2][2], nk;
                  rank_chunks(in.T, P, in.layout, src, kch, &nk);
                  for (int kc = 0; kc < nk; ++kc) {
                    const int k0 = std::max(kch[kc][0], lo);
                    const int k1 = std::min(kch[kc][1], hi);
                    if (k0 >= k1) continue;  // fully masked at this step: skipped
                    plan.segs.push_back(PlanSegment{k0, k1, s, src});
                    cost += (k1 - k0 + kTileRows - 1) / kTileRows;
                  }
                }
              }
              it.seg_count = static_cast<int32_t>(plan.segs.size()) - it.seg_begin;
              it.cost = cost;
              plan.items.push_back(it);
            }
          }
        }
      }
    }
    // longest first inside the pass, so the CTAs that start last are short
    std::stable_sort(plan.items.begin() + first_item, plan.items.end(),
                     [](const PlanItem& x, const PlanItem& y) { return x.cost > y.cost; });
  }
  return plan;
}

FusedPlan build_fused_plan(const Plan& plan, int num_ctas) {
  FusedPlan f;
  if (plan.items.empty() || num_ctas < 1) return f;
  long long total = 0;
  for (const PlanItem& it : plan.items) total += it.cost;
  const double mean = static_cast<double>(total) / num_ctas;
  for (const PlanItem& it : plan.items) {
    const PlanSegment* sg = plan.segs.data() + it.seg_begin;
    if (it.cost < 2 || it.cost <= mean) {
      PlanItem c = it;
      c.seg_begin = static_cast<int32_t>(f.segs.size());
      f.segs.insert(f.segs.end(), sg, sg + it.seg_count);
      f.items.push_back(c);
      continue;
    }
    // first half: the first ceil(cost / 2) key tiles in ring order
    const int first = (it.cost + 1) / 2;
    const int pair = static_cast<int>(f.pairs.size());
    PlanItem half[2] = {it, it};
    int tiles = 0;
    int h = 0;
    half[0].seg_begin = static_cast<int32_t>(f.segs.size());
    for (int si = 0; si < it.seg_count; ++si) {
      PlanSegment cur = sg[si];
      while (cur.k0 < cur.k1) {
        const int n = (cur.k1 - cur.k0 + kTileRows - 1) / kTileRows;
        if (h == 0 && tiles + n > first) {
          // cut the segment where the first half's tiles end
          PlanSegment a = cur;
          a.k1 = cur.k0 + (first - tiles) * kTileRows;
          f.segs.push_back(a);
          tiles = first;
          cur.k0 = a.k1;
        } else {
          f.segs.push_back(cur);
          tiles += n;
          cur.k0 = cur.k1;
        }
        if (h == 0 && tiles == first) {
          half[0].seg_count = static_cast<int32_t>(f.segs.size()) - half[0].seg_begin;
          half[1].seg_begin = static_cast<int32_t>(f.segs.size());
          h = 1;
        }
      }
    }
    half[1].seg_count = static_cast<int32_t>(f.segs.size()) - half[1].seg_begin;
    half[0].cost = first;
    half[1].cost = it.cost - first;
    half[0].part = 2 * pair;
    half[1].part = 2 * pair + 1;
    f.items.push_back(half[0]);
    f.items.push_back(half[1]);
    SplitPair sp{};
    for (int x = 0; x < 2; ++x) {
      sp.q0[x] = it.q0[x];
      sp.qlen[x] = it.qlen[x];
      sp.head[x] = it.head[x];
      sp.part[x] = 2 * pair + x;
    }
    f.pairs.push_back(sp);
  }
  // ordering groups of consecutive passes, at least 2 num_ctas items each
  int max_pass = 0;
  for (const PlanItem& it : plan.items) max_pass = std::max(max_pass, static_cast<int>(it.pass));
  std::vector<long long> per_pass(max_pass + 1, 0);
  for (const PlanItem& it : plan.items) ++per_pass[it.pass];
  std::vector<int> group(max_pass + 1, 0);
  int g = 0;
  long long in_group = 0;
  for (int p = 0; p <= max_pass; ++p) {
    group[p] = g;
    in_group += per_pass[p];
    if (in_group >= 2LL * num_ctas) {
      ++g;
      in_group = 0;
    }
  }
  if (in_group > 0 && g > 0)  // a small rest joins the group before it
    for (int p = 0; p <= max_pass; ++p)
      if (group[p] == g) group[p] = g - 1;
  std::stable_sort(f.items.begin(), f.items.end(), [&](const PlanItem& x, const PlanItem& y) {
    if (group[x.pass] != group[y.pass]) return group[x.pass] < group[y.pass];
    return x.cost > y.cost;
  });
  return f;
}

BwdPlan build_bwd_plan(const PlanInput& in) {
  BwdPlan plan;
  if (in.T == 0) return plan;
  const Docs docs{in.cu};
  const int P = in.num_shards;
  const int G = in.hq / in.hkv;
  const int npass = in.hkv / in.heads_k_stride;
  for (int pass = 0; pass < npass; ++pass) {
    const size_t first_item = plan.items.size();
    for (int g = pass * in.heads_k_stride; g < (pass + 1) * in.heads_k_stride; ++g) {
      for (int src = 0; src < P; ++src) {
        if (in.k_rank >= 0 && src != in.k_rank) continue;
        int kch[2][2], nk;
        rank_chunks(in.T, P, in.layout, src, kch, &nk);
        for (int c = 0; c < nk; ++c) {
          for (int k0 = kch[c][0]; k0 < kch[c][1]; k0 += kTileRows) {
            BwdItem it{};
            it.k0 = k0;
            it.klen = std::min(kTileRows, kch[c][1] - k0);
            it.kv_head = g;
            it.src = src;
            it.seg_begin = static_cast<int32_t>(plan.segs.size());
            const int k_last = k0 + it.klen - 1;
            // queries that see some key of the tile: from the tile start
            // (causal) or its first document's start, to the end of the last
            // key's document
            const int lo = in.causal ? k0 : docs.start(k0);
            const int hi = docs.end(k_last);
            int cost = 0;
            if (in.exchange == 1) {
              // all-gathered: the queries that see the tile, in token order
              if (lo < hi) {
                plan.segs.push_back(BwdSegment{lo, hi, 0, -1});
                cost += (hi - lo + kTileRows - 1) / kTileRows * G;
              }
            } else {
              for (int s = 0; s < P; ++s) {
                const int r = (src + s) % P;
                if (in.q_rank >= 0 && r != in.q_rank) continue;
                int qch[2][2], nq;
                rank_chunks(in.T, P, in.layout, r, qch, &nq);
                for (int qc = 0; qc < nq; ++qc) {
                  const int q0 = std::max(qch[qc][0], lo);
                  const int q1 = std::min(qch[qc][1], hi);
                  if (q0 >= q1) continue;  // fully masked at this step: skipped
                  plan.segs.push_back(BwdSegment{q0, q1, s, r});
                  cost += (q1 - q0 + kTileRows - 1) / kTileRows * G;
                }
              }
            }
            it.seg_count = static_cast<int32_t>(plan.segs.size()) - it.seg_begin;
            // The whole-GPU plan walks an item's query segments from the end of
            // the sequence down instead of in ring order: the co-resident CTAs
            // of a pass then read the same query chunks at about the same
            // time, so each Q/dO tile comes from DRAM about once per pass
            // instead of once per CTA that misses it in L2.  The sum over the
            // segments is the same up to fp32 rounding order; each segment
            // keeps its ring step and rank.
            if (in.q_rank < 0 && in.k_rank < 0)
              std::sort(plan.segs.begin() + it.seg_begin, plan.segs.end(),
                        [](const BwdSegment& x, const BwdSegment& y) { return x.q0 > y.q0; });
            it.cost = cost;
            plan.items.push_back(it);
          }
        }
      }
    }
    std::stable_sort(plan.items.begin() + first_item, plan.items.end(),
                     [](const BwdItem& x, const BwdItem& y) { return x.cost > y.cost; });
  }
  return plan;
}

}  // namespace ra
