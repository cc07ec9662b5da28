// DDTree: the best-first draft tree, with confidence pruning, that feeds the
// heavy-light schedule.
//
// Luce DFlash README, "How it works": instead of one chain of candidates, a
// best-first tree of up to `budget` nodes spans the draft's top-K branches at
// each position; flag table: --ddtree-budget (22) and --ddtree-tau (a
// confidence margin; SpecLA sets 6).  SpecLA article, section "一键开启":
// nodes whose score falls below q* - tau are pruned; section "正确性如何保证":
// cumulative-score pruning, ancestor closure and the budget cap.
//
// A node is a sequence of ranks; its score is the cumulative log-probability
// from the root, accumulated in double.  q* is the best candidate score (the
// best depth-1 log-probability, as scores never rise along a path); a node is
// eligible when score >= q* - tau.  The optional chain seed inserts the greedy
// chain first.  Then the best eligible frontier candidate is added until the
// budget is reached, in the order (higher score, lower depth, lexicographically
// smaller rank sequence); ancestors always precede descendants in that order,
// so the tree is closed under ancestors.  Nodes are numbered in DFS preorder
// with children by rank.  Trees have at most GDN_MAX_NODES nodes, so plain
// scans of the frontier are cheaper than any heap.
#include <cmath>
#include <vector>

#include "gdn_internal.h"

using gdn::fail;

namespace {

constexpr int kMaxTopK = 1024;

struct Node {
  int parent, depth, rank;
  double score;
};

struct Cand {
  int parent, rank;
  double score;
};

// rank sequence of node a < that of node b, for two distinct nodes of equal depth
bool seq_less(const std::vector<Node>& t, int a, int b) {
  while (t[a].parent != t[b].parent) {
    a = t[a].parent;
    b = t[b].parent;
  }
  return t[a].rank < t[b].rank;
}

// candidate x goes before candidate y
bool before(const std::vector<Node>& t, const Cand& x, const Cand& y) {
  if (x.score != y.score) return x.score > y.score;
  const int dx = t[x.parent].depth, dy = t[y.parent].depth;
  if (dx != dy) return dx < dy;
  if (x.parent != y.parent) return seq_less(t, x.parent, y.parent);
  return x.rank < y.rank;
}

gdn_status build_one(const float* logp, int depth_max, int top_k, int budget, double tau, bool chain_seed,
                     int32_t* parent, int32_t* depth, int32_t* rank, double* score, int32_t* n_out) {
  for (int i = 0; i < depth_max * top_k; ++i)
    if (std::isnan(logp[i]) || logp[i] > 0.f)
      return fail(GDN_ERR_INVALID_ARG, "logp[%d] = %g is not a log-probability", i, static_cast<double>(logp[i]));

  double thr = -INFINITY;
  if (tau >= 0.0 && depth_max > 0) {
    double q_star = logp[0];
    for (int r = 1; r < top_k; ++r) q_star = logp[r] > q_star ? logp[r] : q_star;
    thr = q_star - tau;
  }

  std::vector<Node> t;
  t.reserve(budget);
  t.push_back({-1, 0, -1, 0.0});
  std::vector<char> taken(static_cast<size_t>(budget) * (top_k > 0 ? top_k : 1), 0);   // (node, rank) added

  if (chain_seed) {
    int cur = 0;
    for (int d = 1; d <= depth_max && static_cast<int>(t.size()) < budget; ++d) {
      const float* row = logp + static_cast<size_t>(d - 1) * top_k;
      int r = 0;
      for (int j = 1; j < top_k; ++j)
        if (row[j] > row[r]) r = j;
      const double s = t[cur].score + static_cast<double>(row[r]);
      if (s < thr) break;
      taken[static_cast<size_t>(cur) * top_k + r] = 1;
      t.push_back({cur, d, r, s});
      cur = static_cast<int>(t.size()) - 1;
    }
  }

  std::vector<Cand> frontier;
  auto push_children = [&](int v) {
    if (t[v].depth >= depth_max) return;
    const float* row = logp + static_cast<size_t>(t[v].depth) * top_k;
    for (int r = 0; r < top_k; ++r) {
      if (taken[static_cast<size_t>(v) * top_k + r]) continue;
      const double s = t[v].score + static_cast<double>(row[r]);
      if (s >= thr) frontier.push_back({v, r, s});
    }
  };
  for (int v = 0; v < static_cast<int>(t.size()); ++v) push_children(v);
  while (static_cast<int>(t.size()) < budget && !frontier.empty()) {
    size_t best = 0;
    for (size_t i = 1; i < frontier.size(); ++i)
      if (before(t, frontier[i], frontier[best])) best = i;
    const Cand c = frontier[best];
    frontier[best] = frontier.back();
    frontier.pop_back();
    taken[static_cast<size_t>(c.parent) * top_k + c.rank] = 1;
    t.push_back({c.parent, t[c.parent].depth + 1, c.rank, c.score});
    push_children(static_cast<int>(t.size()) - 1);
  }

  // DFS preorder, children by rank
  const int n = static_cast<int>(t.size());
  std::vector<std::vector<int>> kids(n);
  for (int v = 1; v < n; ++v) kids[t[v].parent].push_back(v);
  for (auto& k : kids)
    for (size_t i = 1; i < k.size(); ++i)   // insertion sort by rank (a few children)
      for (size_t j = i; j > 0 && t[k[j]].rank < t[k[j - 1]].rank; --j) std::swap(k[j], k[j - 1]);
  std::vector<int> id(n, -1), stack{0};
  int next = 0;
  while (!stack.empty()) {
    const int v = stack.back();
    stack.pop_back();
    id[v] = next++;
    for (auto it = kids[v].rbegin(); it != kids[v].rend(); ++it) stack.push_back(*it);
  }
  for (int v = 0; v < n; ++v) {
    const int i = id[v];
    parent[i] = v == 0 ? -1 : id[t[v].parent];
    if (depth) depth[i] = t[v].depth;
    if (rank) rank[i] = t[v].rank;
    if (score) score[i] = t[v].score;
  }
  *n_out = n;
  return GDN_OK;
}

gdn_status check_sizes(int depth_max, int top_k, int budget) {
  if (depth_max < 0) return fail(GDN_ERR_INVALID_ARG, "depth_max = %d", depth_max);
  if (depth_max > 0 && (top_k < 1 || top_k > kMaxTopK))
    return fail(GDN_ERR_UNSUPPORTED, "top_k = %d outside 1..%d", top_k, kMaxTopK);
  if (budget < 1 || budget > GDN_MAX_NODES)
    return fail(GDN_ERR_UNSUPPORTED, "budget = %d outside 1..%d", budget, GDN_MAX_NODES);
  return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_ddtree_build(const float* logp, int32_t depth_max, int32_t top_k, int32_t budget,
                                       double tau, int32_t flags, int32_t* parent, int32_t* depth, int32_t* rank,
                                       double* score, int32_t* n_out) {
  gdn::clear_error();
  if (!parent || !n_out || (depth_max > 0 && !logp)) return fail(GDN_ERR_INVALID_ARG, "NULL argument to gdn_ddtree_build");
  if (std::isnan(tau)) return fail(GDN_ERR_INVALID_ARG, "tau is NaN");
  if (flags & ~GDN_DDTREE_CHAIN_SEED) return fail(GDN_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  gdn_status st = check_sizes(depth_max, top_k, budget);
  if (st != GDN_OK) return st;
  return build_one(logp, depth_max, top_k, budget, tau, (flags & GDN_DDTREE_CHAIN_SEED) != 0, parent, depth, rank,
                   score, n_out);
}

extern "C" gdn_status gdn_ddtree_build_batch(const float* logp, int32_t B, int32_t depth_max, int32_t top_k,
                                             int32_t budget, double tau, int32_t flags, int32_t n_max,
                                             int32_t* parents, int32_t* n) {
  gdn::clear_error();
  if (!parents || !n || (depth_max > 0 && !logp)) return fail(GDN_ERR_INVALID_ARG, "NULL argument to gdn_ddtree_build_batch");
  if (B < 1) return fail(GDN_ERR_INVALID_ARG, "B = %d", B);
  if (std::isnan(tau)) return fail(GDN_ERR_INVALID_ARG, "tau is NaN");
  if (flags & ~GDN_DDTREE_CHAIN_SEED) return fail(GDN_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  gdn_status st = check_sizes(depth_max, top_k, budget);
  if (st != GDN_OK) return st;
  if (n_max < budget || n_max > GDN_MAX_NODES)
    return fail(GDN_ERR_INVALID_ARG, "n_max = %d must be in budget (%d)..%d", n_max, budget, GDN_MAX_NODES);
  const size_t table = static_cast<size_t>(depth_max) * top_k;
  for (int b = 0; b < B; ++b) {
    int32_t* row = parents + static_cast<size_t>(b) * n_max;
    for (int i = 0; i < n_max; ++i) row[i] = -1;
    st = build_one(logp + b * table, depth_max, top_k, budget, tau, (flags & GDN_DDTREE_CHAIN_SEED) != 0, row,
                   nullptr, nullptr, nullptr, n + b);
    if (st != GDN_OK) return fail(st, "request %d: %s", b, gdn_last_error());
  }
  return GDN_OK;
}
