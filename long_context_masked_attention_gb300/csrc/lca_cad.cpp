// lca_cad.cpp — host planner for core attention disaggregation ("Efficient
// Long-context Language Model Training by Core Attention Disaggregation":
// core attention is stateless and composable, so it is cut into token-level
// tasks that attention servers rebatch to balance compute).  Host only; no
// CUDA call.  Declared in include/lca_attn.h (lca_cad_plan).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <functional>
#include <numeric>
#include <queue>
#include <vector>

#include "../../include/lca_attn.h"

namespace {

struct Piece {
  int32_t doc, start, len;
};

// Causal attention cells of query rows [a, b) of a document (row i attends
// keys 0..i): sum of (i + 1) = (b(b+1) - a(a+1)) / 2.
int64_t cells(int64_t a, int64_t b) { return (b * (b + 1) - a * (a + 1)) / 2; }

int64_t cost(const Piece& p) { return cells(p.start, static_cast<int64_t>(p.start) + p.len); }

// Longest-processing-time assignment: most expensive piece first, to the
// least-loaded server (ties: lower server index; equal costs: document order).
std::vector<int32_t> assign(const std::vector<Piece>& pieces, int32_t n_servers, std::vector<int64_t>& load) {
  std::vector<int32_t> order(pieces.size());
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) { return cost(pieces[x]) > cost(pieces[y]); });
  using Slot = std::pair<int64_t, int32_t>;  // (load, server)
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int32_t s = 0; s < n_servers; ++s) heap.push({0, s});
  std::vector<int32_t> server(pieces.size());
  load.assign(n_servers, 0);
  for (int32_t i : order) {
    const Slot top = heap.top();
    heap.pop();
    server[i] = top.second;
    load[top.second] = top.first + cost(pieces[i]);
    heap.push({load[top.second], top.second});
  }
  return server;
}

// Row t in (a, b) where the cells of [a, t) are closest to half of [a, b).
int32_t cost_midpoint(int64_t a, int64_t b) {
  const double half = 0.5 * static_cast<double>(a * (a + 1) + b * (b + 1));  // t(t+1) at the midpoint
  int64_t t = static_cast<int64_t>(std::floor((-1.0 + std::sqrt(1.0 + 4.0 * half)) / 2.0));
  t = std::max(a + 1, std::min(b - 1, t));
  if (t + 1 < b && std::llabs(cells(a, t + 1) - cells(t + 1, b)) < std::llabs(cells(a, t) - cells(t, b))) ++t;
  return static_cast<int32_t>(t);
}

}  // namespace

extern "C" {

lca_status lca_cad_plan(const int32_t* doc_len, int32_t n_docs, int32_t n_servers, int32_t min_shard,
                        int32_t max_shard, double tolerance, lca_cad_shard* shards, int32_t max_shards,
                        int32_t* n_shards, int64_t* server_cells) {
  if (!doc_len || n_docs < 0 || n_servers < 1 || min_shard < 1 || max_shard < 0 || !n_shards ||
      !(tolerance >= 0.0) || max_shards < 0 || (max_shards > 0 && !shards))
    return LCA_ERR_INVALID_ARG;
  if (max_shard > 0 && max_shard < 2 * min_shard) return LCA_ERR_INVALID_ARG;
  // 1. documents cut into equal pieces no longer than max_shard
  std::vector<Piece> pieces;
  for (int32_t d = 0; d < n_docs; ++d) {
    const int32_t L = doc_len[d];
    if (L < 0) return LCA_ERR_INVALID_ARG;
    if (L == 0) continue;
    const int32_t n = (max_shard > 0) ? (L + max_shard - 1) / max_shard : 1;
    int32_t a = 0;
    for (int32_t k = 0; k < n; ++k) {
      const int32_t len = L / n + (k < L % n ? 1 : 0);
      pieces.push_back({d, a, len});
      a += len;
    }
  }
  // 2. + 3. assign, then cut the heaviest server's costliest splittable piece at its cost midpoint
  std::vector<int64_t> load;
  std::vector<int32_t> server = assign(pieces, n_servers, load);
  const int64_t total = std::accumulate(load.begin(), load.end(), int64_t{0});
  const double mean = static_cast<double>(total) / n_servers;
  for (int guard = 0; guard < 1 << 16; ++guard) {
    const int32_t hot = static_cast<int32_t>(std::max_element(load.begin(), load.end()) - load.begin());
    if (static_cast<double>(load[hot]) <= mean * (1.0 + tolerance)) break;
    int32_t pick = -1;
    for (int32_t i = 0; i < static_cast<int32_t>(pieces.size()); ++i) {
      if (server[i] != hot || pieces[i].len < 2 * min_shard) continue;
      if (pick < 0 || cost(pieces[i]) > cost(pieces[pick])) pick = i;
    }
    if (pick < 0) break;  // nothing left to cut on the hottest server
    const Piece p = pieces[pick];
    int32_t t = cost_midpoint(p.start, static_cast<int64_t>(p.start) + p.len);
    t = std::max(p.start + min_shard, std::min(p.start + p.len - min_shard, t));
    pieces[pick] = {p.doc, p.start, t - p.start};
    pieces.push_back({p.doc, t, p.start + p.len - t});
    server = assign(pieces, n_servers, load);
  }
  // output: by server, then document order
  std::vector<int32_t> order(pieces.size());
  std::iota(order.begin(), order.end(), 0);
  std::sort(order.begin(), order.end(), [&](int32_t x, int32_t y) {
    if (server[x] != server[y]) return server[x] < server[y];
    if (pieces[x].doc != pieces[y].doc) return pieces[x].doc < pieces[y].doc;
    return pieces[x].start < pieces[y].start;
  });
  *n_shards = static_cast<int32_t>(pieces.size());
  if (server_cells)
    for (int32_t s = 0; s < n_servers; ++s) server_cells[s] = load[s];
  if (static_cast<int32_t>(pieces.size()) > max_shards) return LCA_ERR_WORKSPACE;
  for (size_t k = 0; k < order.size(); ++k) {
    const Piece& p = pieces[order[k]];
    shards[k] = {p.doc, p.start, p.len, server[order[k]]};
  }
  return LCA_OK;
}

}  // extern "C"
