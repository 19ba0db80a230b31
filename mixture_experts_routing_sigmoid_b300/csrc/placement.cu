// Redundant-expert placement planner (host only; "DeepSeek-V3的Group-Limited Expert Routing与负载
// 均衡优化实践", sections 2 and 4): from each expert's measured load, give the hottest experts
// extra replicas ("分身") and place all replicas on the GPUs of an expert-parallel deployment so
// that every GPU carries about the same load.
//   global (section 4, decode): replicate over the whole deployment, then place;
//   hierarchical (section 2, prefill; when the nodes divide the expert groups): first spread the
//   expert groups evenly over the nodes, then replicate and place inside each node.
// The pages name the steps, not the rules; the rules taken here:
//   replicate: R times, add a replica to the expert whose load per replica is largest
//              (ties: lower expert), among those with fewer replicas than GPUs while any
//              such expert remains; a replica carries load / replicas;
//   place:     replicas by decreasing load (ties: lower expert, lower replica), each onto the
//              least-loaded GPU that has a free slot and no replica of that expert yet (ties:
//              lower GPU); only when every free GPU already hosts it, onto the least-loaded
//              GPU with a free slot;
//   groups:    groups by decreasing load (ties: lower group) onto the least-loaded node that
//              still has room for a group.
#include <cstring>
#include <vector>

#include "../../include/moe.h"
#include "internal.h"

namespace {

// Replicate `ids` (expert ids, loads in `load`) into `slots` replicas in total, at most `cap`
// (the GPUs in scope) per expert while some expert is below the cap.
void replicate(const std::vector<int>& ids, const int64_t* load, int slots, int cap,
               std::vector<int>& reps) {
  for (int e : ids) reps[e] = 1;
  for (int r = (int)ids.size(); r < slots; ++r) {
    bool any_below = false;
    for (int e : ids) any_below = any_below || reps[e] < cap;
    int best = -1;
    for (int e : ids) {
      if (any_below && reps[e] >= cap) continue;
      if (best < 0) { best = e; continue; }
      // load[e] / reps[e] > load[best] / reps[best], compared exactly in integers
      const __int128 lhs = (__int128)load[e] * reps[best];
      const __int128 rhs = (__int128)load[best] * reps[e];
      if (lhs > rhs) best = e;  // ids ascend, so ties keep the lower expert
    }
    reps[best] += 1;
  }
}

struct Item {
  int e, j;
  double w;
};

// Place the replicas of `ids` onto GPUs [g0, g0 + ng), `slots` slots each.
void place(const std::vector<int>& ids, const int64_t* load, const std::vector<int>& reps, int g0,
           int ng, int slots, std::vector<int>& fill, std::vector<double>& gl,
           std::vector<std::vector<int>>& hosted) {
  std::vector<Item> items;
  for (int e : ids)
    for (int j = 0; j < reps[e]; ++j) items.push_back({e, j, (double)load[e] / reps[e]});
  // stable insertion by (w desc, e asc, j asc): items are generated in (e asc, j asc) order
  std::vector<Item> sorted;
  for (const Item& it : items) {
    size_t pos = sorted.size();
    while (pos > 0 && sorted[pos - 1].w < it.w) --pos;
    sorted.insert(sorted.begin() + pos, it);
  }
  for (const Item& it : sorted) {
    int pick = -1;
    for (int pass = 0; pass < 2 && pick < 0; ++pass) {
      for (int g = g0; g < g0 + ng; ++g) {
        if (fill[g] >= slots) continue;
        if (pass == 0) {
          bool has = false;
          for (int x : hosted[g]) has = has || x == it.e;
          if (has) continue;
        }
        if (pick < 0 || gl[g] < gl[pick]) pick = g;
      }
    }
    hosted[pick].push_back(it.e);
    fill[pick] += 1;
    gl[pick] += it.w;
  }
}

}  // namespace

extern "C" moe_status moe_plan_placement(const moe_placement_config* pc, const int64_t* load,
                                         int32_t* replicas, int32_t* gpu_expert,
                                         double* gpu_load) {
  if (pc == nullptr || load == nullptr || replicas == nullptr || gpu_expert == nullptr)
    return moe::abi_fail(MOE_ERR_INVALID_ARG, "pc, load, replicas and gpu_expert must be given");
  const int N = pc->n_experts, G = pc->n_gpus, slots = pc->slots_per_gpu;
  const int nodes = pc->n_nodes > 1 ? pc->n_nodes : 1, ngroups = pc->n_groups;
  if (N <= 0 || G <= 0 || slots <= 0 || (long long)G * slots < N)
    return moe::abi_fail(MOE_ERR_INVALID_ARG, "need n_experts > 0 and n_gpus * slots >= n_experts");
  if ((long long)G * slots > (1 << 24))
    return moe::abi_fail(MOE_ERR_UNSUPPORTED, "more than 2^24 replica slots");
  for (int e = 0; e < N; ++e)
    if (load[e] < 0) return moe::abi_fail(MOE_ERR_INVALID_ARG, "negative load");
  if (nodes > 1) {
    if (G % nodes != 0) return moe::abi_fail(MOE_ERR_INVALID_ARG, "n_nodes must divide n_gpus");
    if (ngroups <= 0 || N % ngroups != 0 || ngroups % nodes != 0)
      return moe::abi_fail(MOE_ERR_INVALID_ARG,
                           "hierarchical placement needs n_groups dividing n_experts and "
                           "n_nodes dividing n_groups");
    const int gpn = G / nodes, per_group = N / ngroups;
    if ((long long)gpn * slots < (long long)(ngroups / nodes) * per_group)
      return moe::abi_fail(MOE_ERR_INVALID_ARG, "a node's slots cannot hold its groups");
  }

  std::vector<int> reps(N, 0), fill(G, 0);
  std::vector<double> gl(G, 0.0);
  std::vector<std::vector<int>> hosted(G);
  if (nodes == 1) {
    std::vector<int> ids(N);
    for (int e = 0; e < N; ++e) ids[e] = e;
    replicate(ids, load, G * slots, G, reps);
    place(ids, load, reps, 0, G, slots, fill, gl, hosted);
  } else {
    const int gpn = G / nodes, per_group = N / ngroups, gpnode = ngroups / nodes;
    std::vector<long long> gload(ngroups, 0);
    for (int g = 0; g < ngroups; ++g)
      for (int e = g * per_group; e < (g + 1) * per_group; ++e) gload[g] += load[e];
    std::vector<int> order(ngroups);
    for (int g = 0; g < ngroups; ++g) order[g] = g;
    for (int i = 1; i < ngroups; ++i)  // stable sort by load desc
      for (int k = i; k > 0 && gload[order[k - 1]] < gload[order[k]]; --k)
        std::swap(order[k - 1], order[k]);
    std::vector<long long> nload(nodes, 0);
    std::vector<int> ncount(nodes, 0);
    std::vector<std::vector<int>> node_groups(nodes);
    for (int g : order) {
      int pick = -1;
      for (int n = 0; n < nodes; ++n) {
        if (ncount[n] >= gpnode) continue;
        if (pick < 0 || nload[n] < nload[pick]) pick = n;
      }
      node_groups[pick].push_back(g);
      ncount[pick] += 1;
      nload[pick] += gload[g];
    }
    for (int n = 0; n < nodes; ++n) {
      std::vector<int> ids;
      std::vector<int> gs = node_groups[n];
      for (int i = 1; i < (int)gs.size(); ++i)  // experts in ascending id
        for (int k = i; k > 0 && gs[k - 1] > gs[k]; --k) std::swap(gs[k - 1], gs[k]);
      for (int g : gs)
        for (int e = g * per_group; e < (g + 1) * per_group; ++e) ids.push_back(e);
      replicate(ids, load, gpn * slots, gpn, reps);
      place(ids, load, reps, n * gpn, gpn, slots, fill, gl, hosted);
    }
  }
  for (int e = 0; e < N; ++e) replicas[e] = reps[e];
  for (int g = 0; g < G; ++g) {
    for (int s = 0; s < slots; ++s)
      gpu_expert[(size_t)g * slots + s] = s < (int)hosted[g].size() ? hosted[g][s] : -1;
    if (gpu_load != nullptr) gpu_load[g] = gl[g];
  }
  return MOE_OK;
}
