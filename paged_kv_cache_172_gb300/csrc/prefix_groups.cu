// prefix_groups.cu -- host helper: the groups pa_decode_shared_prefix takes,
// derived from the block tables themselves.
//
// Sequences that share a prompt point at the same physical blocks (study notes
// "DataWhale组队学习笔记--llm-algo-leetcode(五)", "4. PagedAttention 带来的核心红利";
// tutorial chapter "4. PagedAttention机制", block table per sequence).  Two
// sequences share logical block i exactly when both tables hold the same
// physical id at position i and at every position before it.  A prefix tree
// over the physical ids of each sequence's full blocks finds every shared
// prefix: the sequences below a node share the node's depth in blocks.
//
// Grouping, from each child of the root down:
//   * follow the chain while every sequence of the node continues into one
//     child (they keep sharing);
//   * at the node where they part (depth d blocks), if d already reaches the
//     minimum shared length and the node holds at most max_group_size
//     sequences, they form one group sharing d blocks;
//   * otherwise each child holding two or more sequences is visited in turn
//     (they share more), and, once d reaches the minimum, the sequences left
//     over (alone in their child, or ending at this node) are cut into groups
//     of at most max_group_size sharing d blocks.
// Host code only; no CUDA call.
#include <algorithm>
#include <cstdint>
#include <map>
#include <memory>
#include <vector>

#include "pagedkv.h"

namespace {

struct Node {
  std::map<int32_t, std::unique_ptr<Node>> child;  // keyed by physical block id
  std::vector<int> seqs;  // sequences whose chain of full blocks passes through here
};

struct Grouper {
  int min_blocks = 1, gmax = 2;
  std::vector<char> below;  // scratch: sequence continues into a child
  std::vector<std::vector<int>> groups;
  std::vector<int> depth;  // shared blocks of each group

  void emit(const std::vector<int>& members, int d) {
    for (size_t i = 0; i + 1 < members.size(); i += gmax) {
      const size_t e = std::min(members.size(), i + (size_t)gmax);
      groups.emplace_back(members.begin() + i, members.begin() + e);
      depth.push_back(d);
    }
  }

  // v: a node at depth d (blocks) holding two or more ungrouped sequences.
  void visit(const Node* v, int d) {
    while (v->child.size() == 1 && v->child.begin()->second->seqs.size() == v->seqs.size()) {
      v = v->child.begin()->second.get();
      ++d;
    }
    if (d >= min_blocks && (int)v->seqs.size() <= gmax) {
      emit(v->seqs, d);
      return;
    }
    // sequences ending at v (no child holds them), found before recursing
    // since the recursion reuses the scratch marks
    std::vector<int> rest;
    for (const auto& kv : v->child)
      for (int s : kv.second->seqs) below[s] = 1;
    for (int s : v->seqs) {
      if (!below[s]) rest.push_back(s);
      below[s] = 0;
    }
    for (const auto& kv : v->child) {
      const Node* c = kv.second.get();
      if (c->seqs.size() >= 2)
        visit(c, d + 1);
      else
        rest.push_back(c->seqs[0]);
    }
    if (d >= min_blocks) {
      std::sort(rest.begin(), rest.end());
      emit(rest, d);
    }
  }
};

}  // namespace

extern "C" pa_status pa_shared_prefix_groups(const int32_t* block_tables,
                                             const int32_t* context_lens, int B,
                                             int max_blocks_per_seq, int block_size,
                                             int min_shared_tokens, int max_group_size,
                                             int32_t* seq_group, int32_t* group_offsets,
                                             int32_t* group_seqs, int32_t* group_prefix_len,
                                             int* num_groups) {
  if (num_groups == nullptr) return PA_ERR_INVALID;
  *num_groups = 0;
  if (B < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || min_shared_tokens < 0 ||
      max_group_size < 2)
    return PA_ERR_INVALID;
  if (B == 0) {
    if (group_offsets) group_offsets[0] = 0;
    return PA_OK;
  }
  if (!block_tables || !context_lens || !seq_group || !group_offsets || !group_seqs ||
      !group_prefix_len)
    return PA_ERR_INVALID;

  Node root;
  const long long cap = (long long)max_blocks_per_seq * block_size;
  for (int b = 0; b < B; ++b) {
    const long long ctx = std::min<long long>(std::max(context_lens[b], 0), cap);
    const int full = (int)(ctx / block_size);
    const int32_t* row = block_tables + (size_t)b * max_blocks_per_seq;
    Node* v = &root;
    for (int i = 0; i < full && row[i] >= 0; ++i) {
      std::unique_ptr<Node>& c = v->child[row[i]];
      if (!c) c.reset(new Node());
      v = c.get();
      v->seqs.push_back(b);
    }
  }

  Grouper g;
  g.min_blocks = std::max(1, (min_shared_tokens + block_size - 1) / block_size);
  g.gmax = max_group_size;
  g.below.assign(B, 0);
  for (const auto& kv : root.child)
    if (kv.second->seqs.size() >= 2) g.visit(kv.second.get(), 1);

  // disjoint groups of >= 2 members: at most B/2 groups and B members, the
  // sizes the caller allocated
  size_t members = 0;
  for (const auto& m : g.groups) members += m.size();
  if (2 * g.groups.size() > (size_t)B || members > (size_t)B) return PA_ERR_INVALID;
  // groups in increasing order of their first (smallest) member
  std::vector<int> order(g.groups.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = (int)i;
  std::sort(order.begin(), order.end(),
            [&](int x, int y) { return g.groups[x][0] < g.groups[y][0]; });
  for (int b = 0; b < B; ++b) seq_group[b] = -1;
  int off = 0;
  group_offsets[0] = 0;
  for (size_t i = 0; i < order.size(); ++i) {
    for (int s : g.groups[order[i]]) {
      seq_group[s] = (int32_t)i;
      group_seqs[off++] = s;
    }
    group_offsets[i + 1] = off;
    group_prefix_len[i] = g.depth[order[i]] * block_size;
  }
  *num_groups = (int)g.groups.size();
  return PA_OK;
}
