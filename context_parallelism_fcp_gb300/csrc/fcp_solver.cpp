// Congestion-free communication solver ("Unleashing Scalable Context Parallelism for
// Foundation Models Pre-Training via FCP", Section 4.2, Lemmas 1 and 2, Figure 8).
//
// The data flow of a plan is a bipartite multigraph: N send nodes S, N receive nodes R and
// one edge S(i) -> R(j) for every block worker j must pull from worker i. A sub-stage in
// which each worker sends at most one block and receives at most one block is a matching
// (Lemma 1), and the worker of maximum degree Delta needs at least Delta sub-stages
// (Lemma 2). A bipartite multigraph's edges always split into Delta matchings (Konig): the
// graph is padded to Delta-regular with dummy edges, and Delta perfect matchings (Hall's
// condition holds in a regular bipartite graph) are peeled off one by one with
// Hopcroft-Karp; the real edges of the k-th matching form sub-stage k.
#include <algorithm>
#include <set>
#include <queue>
#include <vector>

#include "fcp_internal.h"

namespace fcp {
namespace {

// Maximum matching of a bipartite graph with n left and n right vertices (adjacency lists
// of right vertices per left vertex) by Hopcroft-Karp: BFS layers from the free left
// vertices, then vertex-disjoint shortest augmenting paths by DFS, until none is left.
// Recursion depth is bounded by the path length (at most n).
struct HopcroftKarp {
  static constexpr int32_t kInf = 0x3fffffff;
  int32_t n;
  const std::vector<std::vector<int32_t>>& adj;
  std::vector<int32_t> match_l, match_r, dist, it;

  HopcroftKarp(int32_t n_, const std::vector<std::vector<int32_t>>& a)
      : n(n_), adj(a), match_l(n_, -1), match_r(n_, -1), dist(n_, 0), it(n_, 0) {}

  bool bfs() {
    std::queue<int32_t> q;
    bool found = false;
    for (int32_t u = 0; u < n; ++u) {
      dist[u] = match_l[u] < 0 ? 0 : kInf;
      if (match_l[u] < 0) q.push(u);
    }
    while (!q.empty()) {
      const int32_t u = q.front();
      q.pop();
      for (int32_t v : adj[u]) {
        const int32_t w = match_r[v];
        if (w < 0) {
          found = true;
        } else if (dist[w] == kInf) {
          dist[w] = dist[u] + 1;
          q.push(w);
        }
      }
    }
    return found;
  }

  bool dfs(int32_t u) {
    for (; it[u] < static_cast<int32_t>(adj[u].size()); ++it[u]) {
      const int32_t v = adj[u][it[u]];
      const int32_t w = match_r[v];
      if (w < 0 || (dist[w] == dist[u] + 1 && dfs(w))) {
        match_l[u] = v;
        match_r[v] = u;
        return true;
      }
    }
    dist[u] = kInf;
    return false;
  }

  std::vector<int32_t> run() {
    while (bfs()) {
      std::fill(it.begin(), it.end(), 0);
      for (int32_t u = 0; u < n; ++u)
        if (match_l[u] < 0) dfs(u);
    }
    return match_l;
  }
};

constexpr int32_t kMaxSubStages = 1 << 24;

// Edges of the data-flow graph: distinct (KV block, receiver) pairs whose block lives on
// another worker, in work-list order, sub-stage unset.
void build_edges(fcp_plan* p) {
  p->transfers.clear();
  std::vector<std::vector<int32_t>> pulled(static_cast<size_t>(p->n_workers));
  for (const fcp_item& it : p->work_list) {
    const int32_t src = p->blocks[it.kv_block].worker;
    const int32_t dst = it.worker;
    if (src == dst) continue;
    auto& seen = pulled[dst];
    if (std::find(seen.begin(), seen.end(), it.kv_block) != seen.end()) continue;
    seen.push_back(it.kv_block);
    p->transfers.push_back(fcp_transfer{it.kv_block, src, dst, -1, p->blocks[it.kv_block].tokens, 0});
  }
}

}  // namespace
}  // namespace fcp

using namespace fcp;

extern "C" {

fcp_status fcp_solve_stages(fcp_plan* p) {
  if (p == nullptr) return FCP_ERR_INVALID;
  if (!p->distributed) return FCP_ERR_STATE;
  const int32_t N = p->n_workers;
  build_edges(p);
  std::vector<int32_t> deg_s(static_cast<size_t>(N), 0), deg_r(static_cast<size_t>(N), 0);
  for (const fcp_transfer& t : p->transfers) {
    ++deg_s[t.src];
    ++deg_r[t.dst];
  }
  int32_t delta = 0;
  for (int32_t w = 0; w < N; ++w) delta = std::max({delta, deg_s[w], deg_r[w]});

  // parallel edges grouped per (sender, receiver) pair: a stack of transfer ids (popped
  // lowest id first) plus a count of padding edges
  std::vector<std::vector<int32_t>> pair_ids;
  std::vector<int32_t> pair_pad, pair_u, pair_v;
  std::vector<int32_t> pair_of(static_cast<size_t>(N) * static_cast<size_t>(N), -1);
  auto pair_index = [&](int32_t u, int32_t v) -> int32_t {
    int32_t& slot = pair_of[static_cast<size_t>(u) * N + v];
    if (slot < 0) {
      slot = static_cast<int32_t>(pair_ids.size());
      pair_ids.emplace_back();
      pair_pad.push_back(0);
      pair_u.push_back(u);
      pair_v.push_back(v);
    }
    return slot;
  };
  for (int32_t i = static_cast<int32_t>(p->transfers.size()) - 1; i >= 0; --i)
    pair_ids[pair_index(p->transfers[i].src, p->transfers[i].dst)].push_back(i);
  // pad to delta-regular: pair senders short of delta with receivers short of delta
  int32_t v = 0;
  for (int32_t u = 0; u < N; ++u) {
    while (deg_s[u] < delta) {
      while (deg_r[v] >= delta) ++v;
      const int32_t k = std::min(delta - deg_s[u], delta - deg_r[v]);
      pair_pad[pair_index(u, v)] += k;
      deg_s[u] += k;
      deg_r[v] += k;
    }
  }
  // peel delta perfect matchings; a matched pair gives up one real edge if it has one
  for (int32_t stage = 0; stage < delta; ++stage) {
    std::vector<std::vector<int32_t>> adj(static_cast<size_t>(N));
    for (size_t q = 0; q < pair_ids.size(); ++q)
      if (!pair_ids[q].empty() || pair_pad[q] > 0) adj[pair_u[q]].push_back(pair_v[q]);
    for (auto& list : adj) std::sort(list.begin(), list.end());
    const std::vector<int32_t> match = HopcroftKarp(N, adj).run();
    for (int32_t u = 0; u < N; ++u) {
      if (match[u] < 0) {
        p->transfers.clear();
        p->solved = false;
        set_last_error("no perfect matching in a regular bipartite graph");
        return FCP_ERR_STATE;  // impossible by Hall's theorem
      }
      const int32_t q = pair_of[static_cast<size_t>(u) * N + match[u]];
      if (!pair_ids[q].empty()) {
        p->transfers[pair_ids[q].back()].stage = stage;
        pair_ids[q].pop_back();
      } else {
        --pair_pad[q];
      }
    }
  }
  p->n_stages = delta;
  p->solved = true;
  return FCP_OK;
}

fcp_status fcp_set_stages(fcp_plan* p, const int32_t* stages, int32_t n_transfers) {
  if (p == nullptr || n_transfers < 0 || (n_transfers > 0 && stages == nullptr)) return FCP_ERR_INVALID;
  if (!p->distributed) return FCP_ERR_STATE;
  build_edges(p);
  p->solved = false;
  if (static_cast<size_t>(n_transfers) != p->transfers.size()) {
    p->transfers.clear();
    set_last_error("fcp_set_stages: the stage count does not match the plan's transfers");
    return FCP_ERR_INVALID;
  }
  int32_t n_stages = 0;
  for (int32_t i = 0; i < n_transfers; ++i) {
    if (stages[i] < 0 || stages[i] >= kMaxSubStages) {
      p->transfers.clear();
      set_last_error("fcp_set_stages: sub-stage out of range");
      return FCP_ERR_INVALID;
    }
    n_stages = std::max(n_stages, stages[i] + 1);
  }
  // every sub-stage a matching: one send and one receive per worker
  std::set<std::pair<int32_t, int32_t>> sends, recvs;
  for (int32_t i = 0; i < n_transfers; ++i) {
    const fcp_transfer& t = p->transfers[i];
    if (!sends.insert({stages[i], t.src}).second || !recvs.insert({stages[i], t.dst}).second) {
      p->transfers.clear();
      set_last_error("fcp_set_stages: a sub-stage is not a matching");
      return FCP_ERR_INVALID;
    }
  }
  for (int32_t i = 0; i < n_transfers; ++i) p->transfers[i].stage = stages[i];
  p->n_stages = n_stages;
  p->solved = true;
  return FCP_OK;
}

fcp_status fcp_plan_transfers(const fcp_plan* p, const fcp_transfer** transfers, int32_t* n_transfers,
                              int32_t* n_stages) {
  if (p == nullptr || transfers == nullptr || n_transfers == nullptr || n_stages == nullptr) return FCP_ERR_INVALID;
  if (!p->solved) return FCP_ERR_STATE;
  *transfers = p->transfers.data();
  *n_transfers = static_cast<int32_t>(p->transfers.size());
  *n_stages = p->n_stages;
  return FCP_OK;
}

}  // extern "C"
