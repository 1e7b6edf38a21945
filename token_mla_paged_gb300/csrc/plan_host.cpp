// Host work/split planner.
//
// Whoever builds a decode CSR builds its split plan next to it, on the host, so
// that no forward call writes a plan and every CUDA graph reads constant memory
// ("[DSV4] Tuned ASM FP8 decode with split plans; HCA on aiter's persistent
// V4-NM kernel", Summary part 1).  In STATIC mode the plan depends only on the
// query-row counts and a KV capacity; in DYNAMIC and HOST mode on the real KV
// lengths (DYNAMIC: the same plan the device planner rebuilds at every call,
// Summary part 2; HOST: built here from the CSR and used as is).
//
// Rules (integers only, 64-bit intermediates):
//   G_b = ceil(H*T_b/128) row groups; N_b = ceil(L_b/64) tiles (DYNAMIC, HOST) or
//   ceil(cap/64) (STATIC); target = max(4, ceil(sum G_b*N_b / W));
//   S_b = clamp(ceil(N_b/target), 1, 16); one item per (b, split s, group g),
//   enumerated b-major, then s, then g; items sorted by min(cost, 65535)
//   descending with cost = tiles of the split + 1, ties in enumeration order.
#include <algorithm>
#include <cstring>
#include <vector>

#include "mla_internal.h"

namespace mla {

mla_status plan_build_host(const mla_plan_params& p, const int32_t* kv_indptr,
                           const int32_t* qo_indptr, int32_t* out) {
  if (p.batch < 0 || p.num_heads < 1 || p.max_q_len < 0 || p.num_workers < 1 ||
      (p.mode != MLA_PLAN_STATIC && p.mode != MLA_PLAN_DYNAMIC && p.mode != MLA_PLAN_HOST))
    return MLA_ERR_INVALID_ARG;
  if (p.mode == MLA_PLAN_STATIC && p.kv_len_cap < 0) return MLA_ERR_INVALID_ARG;
  if (p.batch > 0 && qo_indptr == nullptr) return MLA_ERR_INVALID_ARG;
  const bool real_lengths = p.mode != MLA_PLAN_STATIC;
  if (real_lengths && p.batch > 0 && kv_indptr == nullptr) return MLA_ERR_INVALID_ARG;

  const PlanGeom geom = plan_geom(p);
  if (geom.items_cap > kCostClamp) return MLA_ERR_UNSUPPORTED;
  const int B = p.batch;
  std::vector<int64_t> G(B), N(B), S(B);
  int64_t total = 0;
  for (int b = 0; b < B; ++b) {
    const int64_t T = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
    if (T < 0 || T > p.max_q_len) return MLA_ERR_INVALID_ARG;
    int64_t L;
    if (real_lengths) {
      L = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
      if (L < 0) return MLA_ERR_INVALID_ARG;
    } else {
      L = p.kv_len_cap;
    }
    G[b] = cdiv64((int64_t)p.num_heads * T, kRows);
    N[b] = cdiv64(L, kBlockN);
    total += G[b] * N[b];
  }
  const int64_t target = std::max<int64_t>(kMinTiles, cdiv64(total, p.num_workers));
  for (int b = 0; b < B; ++b)
    S[b] = std::min<int64_t>(kMaxSplits, std::max<int64_t>(1, cdiv64(N[b], target)));

  struct Rec { int32_t key_cost; int32_t order; int32_t b, s, g, slot; };
  std::vector<Rec> items;
  std::vector<int32_t> gbase(B + 1, 0), pbase(B, -1);
  int64_t run_partials = 0;
  for (int b = 0; b < B; ++b) {
    gbase[b + 1] = (int32_t)(gbase[b] + G[b]);
    if (S[b] > 1) {
      pbase[b] = (int32_t)run_partials;
      run_partials += S[b] * G[b];
    }
    for (int64_t s = 0; s < S[b]; ++s) {
      const int64_t t0 = s * N[b] / S[b];
      const int64_t t1 = (s + 1) * N[b] / S[b];
      const int64_t cost = std::min<int64_t>(t1 - t0 + 1, kCostClamp);
      for (int64_t g = 0; g < G[b]; ++g) {
        Rec r;
        r.key_cost = (int32_t)cost;
        r.order = (int32_t)items.size();
        r.b = b;
        r.s = (int32_t)s;
        r.g = (int32_t)g;
        r.slot = S[b] > 1 ? (int32_t)(pbase[b] + s * G[b] + g) : -1;
        items.push_back(r);
        if ((int64_t)items.size() > geom.items_cap) return MLA_ERR_UNSUPPORTED;
      }
    }
  }
  std::stable_sort(items.begin(), items.end(),
                   [](const Rec& a, const Rec& c) { return a.key_cost > c.key_cost; });

  std::memset(out, 0, sizeof(int32_t) * (size_t)geom.total_ints);
  const int64_t cap = p.mode == MLA_PLAN_STATIC ? p.kv_len_cap : 0;
  int32_t* h = out;
  h[kHMagic] = kPlanMagic;
  h[kHVersion] = kPlanVersion;
  h[kHBatch] = p.batch;
  h[kHHeads] = p.num_heads;
  h[kHMaxQ] = p.max_q_len;
  h[kHWorkers] = p.num_workers;
  h[kHMode] = p.mode;
  h[kHNItems] = (int32_t)items.size();
  h[kHNPartials] = (int32_t)run_partials;
  h[kHNGroups] = gbase[B];
  h[kHCapLo] = (int32_t)(uint32_t)(cap & 0xFFFFFFFFLL);
  h[kHCapHi] = (int32_t)(uint32_t)((cap >> 32) & 0xFFFFFFFFLL);
  h[kHRows] = kRows;
  h[kHBlockN] = kBlockN;
  h[kHItemsCap] = geom.items_cap;
  for (int b = 0; b < B; ++b) out[geom.off_S + b] = (int32_t)S[b];
  for (int b = 0; b <= B; ++b) out[geom.off_gbase + b] = gbase[b];
  for (int b = 0; b < B; ++b) out[geom.off_pbase + b] = pbase[b];
  for (size_t k = 0; k < items.size(); ++k) {
    int32_t* it = out + geom.off_items + 4 * k;
    it[0] = items[k].b;
    it[1] = items[k].s;
    it[2] = items[k].g;
    it[3] = items[k].slot;
  }
  return MLA_OK;
}

}  // namespace mla
