// Heavy-light schedule of a draft tree and its packed (compact) form.
//
// SpecLA article, section "链分解与依赖波 HLD 调度": heavy child = child with the
// largest subtree; heavy edges continue a state-resident chain, light edges
// start a new one; only boundary states are materialised; chains form
// dependency waves.  Because parent[i] < i, one reverse pass gives subtree
// sizes and one forward pass gives heavy children, chain membership and waves.
#include <cstring>
#include <vector>

#include "gdn_internal.h"

using gdn::fail;

namespace {

struct Hld {
  int n = 0, n_chains = 0, n_waves = 0, n_boundary = 0;
  std::vector<int32_t> subtree, heavy, chain_of, pos, chain_head, chain_len, chain_off, chain_nodes, chain_wave,
      chain_src, wave_off, bslot, bnode;
};

gdn_status build(const int32_t* parent, int n, Hld& h) {
  if (!parent) return fail(GDN_ERR_INVALID_ARG, "parent is NULL");
  if (n < 1) return fail(GDN_ERR_INVALID_TREE, "a tree needs at least one node (n = %d)", n);
  if (parent[0] != -1) return fail(GDN_ERR_INVALID_TREE, "parent[0] = %d, the root must have parent -1", parent[0]);
  for (int i = 1; i < n; ++i)
    if (parent[i] < 0 || parent[i] >= i)
      return fail(GDN_ERR_INVALID_TREE, "parent[%d] = %d is not an earlier node", i, parent[i]);

  h.n = n;
  h.subtree.assign(n, 1);
  for (int i = n - 1; i >= 1; --i) h.subtree[parent[i]] += h.subtree[i];

  // Ascending scan of children: a later child replaces the heavy one only if strictly larger.
  h.heavy.assign(n, -1);
  for (int i = 1; i < n; ++i) {
    const int p = parent[i];
    if (h.heavy[p] < 0 || h.subtree[i] > h.subtree[h.heavy[p]]) h.heavy[p] = i;
  }

  // Chain membership and wave of every node in one forward pass.
  std::vector<int32_t> head_of(n), wave(n);
  h.pos.assign(n, 0);
  std::vector<char> is_head(n, 0), is_boundary(n, 0);
  for (int i = 0; i < n; ++i) {
    const int p = parent[i];
    if (i == 0 || h.heavy[p] != i) {
      is_head[i] = 1;
      head_of[i] = i;
      h.pos[i] = 0;
      wave[i] = (i == 0) ? 0 : wave[p] + 1;
      if (i != 0) is_boundary[p] = 1;
    } else {
      head_of[i] = head_of[p];
      h.pos[i] = h.pos[p] + 1;
      wave[i] = wave[p];
    }
  }
  int max_wave = 0;
  for (int i = 0; i < n; ++i)
    if (is_head[i] && wave[i] > max_wave) max_wave = wave[i];
  h.n_waves = max_wave + 1;

  // Chains ordered by (wave, head): bucket heads by wave in ascending index order.
  h.wave_off.assign(h.n_waves + 1, 0);
  for (int i = 0; i < n; ++i)
    if (is_head[i]) h.wave_off[wave[i] + 1]++;
  for (int w = 0; w < h.n_waves; ++w) h.wave_off[w + 1] += h.wave_off[w];
  h.n_chains = h.wave_off[h.n_waves];
  h.chain_head.assign(h.n_chains, 0);
  std::vector<int32_t> fill(h.wave_off.begin(), h.wave_off.end() - 1);
  for (int i = 0; i < n; ++i)
    if (is_head[i]) h.chain_head[fill[wave[i]]++] = i;

  // Boundary slots in ascending node order.
  h.bslot.assign(n, -1);
  h.bnode.clear();
  for (int i = 0; i < n; ++i)
    if (is_boundary[i]) {
      h.bslot[i] = static_cast<int32_t>(h.bnode.size());
      h.bnode.push_back(i);
    }
  h.n_boundary = static_cast<int>(h.bnode.size());

  std::vector<int32_t> chain_id_of_head(n, -1);
  h.chain_len.assign(h.n_chains, 0);
  h.chain_off.assign(h.n_chains + 1, 0);
  h.chain_wave.assign(h.n_chains, 0);
  h.chain_src.assign(h.n_chains, -1);
  h.chain_nodes.clear();
  for (int c = 0; c < h.n_chains; ++c) {
    const int hd = h.chain_head[c];
    chain_id_of_head[hd] = c;
    h.chain_wave[c] = wave[hd];
    h.chain_src[c] = (hd == 0) ? -1 : h.bslot[parent[hd]];
    for (int v = hd; v >= 0; v = h.heavy[v]) h.chain_nodes.push_back(v);
    h.chain_off[c + 1] = static_cast<int32_t>(h.chain_nodes.size());
    h.chain_len[c] = h.chain_off[c + 1] - h.chain_off[c];
  }
  h.chain_of.assign(n, 0);
  for (int i = 0; i < n; ++i) h.chain_of[i] = chain_id_of_head[head_of[i]];
  return GDN_OK;
}

void copy_out(const std::vector<int32_t>& v, int32_t* dst) {
  if (!v.empty()) std::memcpy(dst, v.data(), v.size() * sizeof(int32_t));
}

}  // namespace

extern "C" gdn_status gdn_hld_schedule(const int32_t* parent, int32_t n, gdn_schedule* out) {
  gdn::clear_error();
  if (!out) return fail(GDN_ERR_INVALID_ARG, "out is NULL");
  int32_t* arrays[] = {out->subtree,    out->heavy,      out->chain_of,       out->pos_in_chain, out->chain_head,
                       out->chain_len,  out->chain_off,  out->chain_nodes,    out->chain_wave,   out->chain_src_slot,
                       out->wave_off,   out->boundary_slot, out->boundary_node};
  for (int32_t* a : arrays)
    if (!a) return fail(GDN_ERR_INVALID_ARG, "an output array of gdn_schedule is NULL");
  Hld h;
  gdn_status st = build(parent, n, h);
  if (st != GDN_OK) return st;
  out->n = h.n;
  out->n_chains = h.n_chains;
  out->n_waves = h.n_waves;
  out->n_boundary = h.n_boundary;
  copy_out(h.subtree, out->subtree);
  copy_out(h.heavy, out->heavy);
  copy_out(h.chain_of, out->chain_of);
  copy_out(h.pos, out->pos_in_chain);
  copy_out(h.chain_head, out->chain_head);
  copy_out(h.chain_len, out->chain_len);
  copy_out(h.chain_off, out->chain_off);
  copy_out(h.chain_nodes, out->chain_nodes);
  copy_out(h.chain_wave, out->chain_wave);
  copy_out(h.chain_src, out->chain_src_slot);
  copy_out(h.wave_off, out->wave_off);
  copy_out(h.bslot, out->boundary_slot);
  copy_out(h.bnode, out->boundary_node);
  return GDN_OK;
}

extern "C" int32_t gdn_schedule_words(int32_t n_max) { return gdn::SchedLayout{n_max}.words(); }

// The verify's walk of one tree: a depth-first order in which every node follows its parent, and
// the stash traffic it implies.  Heavy-light (the SpecLA chains): children are visited light ones
// first (ascending index), the heavy child last, so a chain continues in registers through every
// node with one child.  A branching node's state is materialised and stashed once; its first child
// continues from the registers, each later child reloads the stash, and the stash is released when
// the last (heavy) child starts -- so at most (light edges on the root path) stashes are live, and
// the first kTmemLevels of them sit in tensor memory, deeper ones in the node's boundary slot.
// Per-node states (the comparison schedule): children by ascending index, every node with children
// stashes its state in its boundary slot and every child reloads it from there.
static void emit_ops(const int32_t* parent, int n, const int32_t* heavy, bool per_node,
                     const std::vector<int32_t>& slot, int32_t* ops, int32_t* nflags, int* levels_used) {
  std::vector<std::vector<int>> kids(n);
  for (int i = 1; i < n; ++i) kids[parent[i]].push_back(i);
  if (!per_node)
    for (int v = 0; v < n; ++v) {
      auto& k = kids[v];
      for (size_t i = 0; i + 1 < k.size(); ++i)
        if (k[i] == heavy[v]) std::swap(k[i], k[i + 1]);   // bubble the heavy child to the end
    }
  int next = 0, depth = 0, used = 0;
  struct Frame { int v; size_t child; int32_t stash; bool pushed; };
  std::vector<Frame> stack;
  auto enter = [&](int v, int32_t src) {
    int32_t op = v | src;
    const auto& ch = kids[v];
    int32_t stash = 0;
    bool pushed = false;
    if (ch.empty()) {
      op |= gdn::kOpLeaf;
    } else if (per_node || ch.size() >= 2) {
      pushed = true;
      if (per_node || depth >= gdn::kTmemLevels || slot[v] < 0) {
        op |= gdn::kOpPush | gdn::kOpPushGlobal;
        stash = gdn::kOpReload | gdn::kOpReloadGlobal;
      } else {
        op |= gdn::kOpPush | (depth << gdn::kOpPushLevelShift);
        stash = gdn::kOpReload | (depth << gdn::kOpReloadLevelShift);
        used = depth + 1 > used ? depth + 1 : used;
      }
      ++depth;
    }
    ops[next++] = op;
    nflags[v] = pushed ? gdn::kNodeMaterialised : 0;
    stack.push_back({v, 0, stash, pushed});
  };
  enter(0, 0);
  while (!stack.empty()) {
    Frame& f = stack.back();
    const auto& ch = kids[f.v];
    if (f.child == ch.size()) {
      stack.pop_back();
      continue;
    }
    const size_t i = f.child++;
    const bool last = f.child == ch.size();
    const int32_t src = (i == 0 && !per_node) ? 0 : f.stash;
    if (f.pushed && last) --depth;   // the last child takes the stash over; its level is free again
    enter(ch[i], src);               // may reallocate the stack: f is not used after this
  }
  *levels_used = used;
}

// One packed record (layout in gdn_tree.h).
static void write_record(const int32_t* parent, int n, const gdn::SchedLayout& lay, int n_chains, int n_boundary,
                         int n_waves, const std::vector<int32_t>& slot, const int32_t* heavy, bool per_node,
                         int32_t* w) {
  for (int i = 0; i < lay.words(); ++i) w[i] = -1;
  w[0] = n;
  w[1] = n_chains;
  w[2] = n_boundary;
  w[3] = n_waves;
  for (int i = 0; i < n; ++i) {
    w[lay.parent() + i] = parent[i];
    w[lay.bslot() + i] = slot[i];
  }
  int levels = 0;
  emit_ops(parent, n, heavy, per_node, slot, w + lay.ops(), w + lay.nflags(), &levels);
  w[4] = levels;
}

// Per-node-state schedule: every node with children gets a boundary slot (ascending node order).
static gdn_status pack_per_node(const int32_t* parent, int n, const gdn::SchedLayout& lay, int32_t* w,
                                int* nb_out) {
  if (n < 1 || parent[0] != -1) return fail(GDN_ERR_INVALID_TREE, "parent[0] must be -1");
  std::vector<int32_t> depth(n, 0), kids(n, 0);
  for (int i = 1; i < n; ++i) {
    if (parent[i] < 0 || parent[i] >= i) return fail(GDN_ERR_INVALID_TREE, "parent[%d] = %d", i, parent[i]);
    depth[i] = depth[parent[i]] + 1;
    kids[parent[i]]++;
  }
  int max_depth = 0;
  for (int i = 0; i < n; ++i) max_depth = depth[i] > max_depth ? depth[i] : max_depth;
  std::vector<int32_t> slot(n, -1);
  int nb = 0;
  for (int i = 0; i < n; ++i)
    if (kids[i] > 0) slot[i] = nb++;
  write_record(parent, n, lay, n, nb, max_depth + 1, slot, nullptr, true, w);
  *nb_out = nb;
  return GDN_OK;
}

// Depth of the deepest node of a valid tree (parent[i] < i).
static int tree_depth(const int32_t* parent, int n) {
  std::vector<int> depth(n, 0);
  int m = 0;
  for (int i = 1; i < n; ++i) {
    depth[i] = depth[parent[i]] + 1;
    m = depth[i] > m ? depth[i] : m;
  }
  return m;
}

extern "C" gdn_status gdn_pack_schedules_per_node(const int32_t* parents, const int32_t* n, int32_t B,
                                                  int32_t n_max, int32_t* words, int32_t* nb_max_out,
                                                  int32_t* depth_max_out) {
  gdn::clear_error();
  if (!parents || !n || !words) return fail(GDN_ERR_INVALID_ARG, "NULL argument to gdn_pack_schedules_per_node");
  if (B < 1) return fail(GDN_ERR_INVALID_ARG, "B = %d", B);
  if (n_max < 1 || n_max > GDN_MAX_NODES)
    return fail(GDN_ERR_UNSUPPORTED, "n_max = %d outside 1..%d", n_max, GDN_MAX_NODES);
  const gdn::SchedLayout lay{n_max};
  int nb_max = 0, depth_max = 0;
  for (int b = 0; b < B; ++b) {
    if (n[b] < 1 || n[b] > n_max)
      return fail(GDN_ERR_INVALID_TREE, "request %d: n = %d outside 1..n_max (%d)", b, n[b], n_max);
    int nb = 0;
    gdn_status st = pack_per_node(parents + static_cast<size_t>(b) * n_max, n[b], lay,
                                  words + static_cast<size_t>(b) * lay.words(), &nb);
    if (st != GDN_OK) return st;
    nb_max = nb > nb_max ? nb : nb_max;
    const int dp = tree_depth(parents + static_cast<size_t>(b) * n_max, n[b]);
    depth_max = dp > depth_max ? dp : depth_max;
  }
  if (nb_max_out) *nb_max_out = nb_max;
  if (depth_max_out) *depth_max_out = depth_max;
  return GDN_OK;
}

extern "C" gdn_status gdn_pack_schedules(const int32_t* parents, const int32_t* n, int32_t B, int32_t n_max,
                                         int32_t* words, int32_t* nb_max_out, int32_t* depth_max_out) {
  gdn::clear_error();
  if (!parents || !n || !words) return fail(GDN_ERR_INVALID_ARG, "NULL argument to gdn_pack_schedules");
  if (B < 1) return fail(GDN_ERR_INVALID_ARG, "B = %d", B);
  if (n_max < 1 || n_max > GDN_MAX_NODES)
    return fail(GDN_ERR_UNSUPPORTED, "n_max = %d outside 1..%d", n_max, GDN_MAX_NODES);
  const gdn::SchedLayout lay{n_max};
  int nb_max = 0, depth_max = 0;
  Hld h;
  for (int b = 0; b < B; ++b) {
    if (n[b] < 1 || n[b] > n_max)
      return fail(GDN_ERR_INVALID_TREE, "request %d: n = %d outside 1..n_max (%d)", b, n[b], n_max);
    gdn_status st = build(parents + static_cast<size_t>(b) * n_max, n[b], h);
    if (st != GDN_OK) return fail(st, "request %d: %s", b, gdn_last_error());
    write_record(parents + static_cast<size_t>(b) * n_max, h.n, lay, h.n_chains, h.n_boundary, h.n_waves, h.bslot,
                 h.heavy.data(), false, words + static_cast<size_t>(b) * lay.words());
    if (h.n_boundary > nb_max) nb_max = h.n_boundary;
    const int dp = tree_depth(parents + static_cast<size_t>(b) * n_max, h.n);
    depth_max = dp > depth_max ? dp : depth_max;
  }
  if (nb_max_out) *nb_max_out = nb_max;
  if (depth_max_out) *depth_max_out = depth_max;
  return GDN_OK;
}
