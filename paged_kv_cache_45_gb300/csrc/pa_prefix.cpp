// pa_prefix.cpp -- host-side block pool with a radix prefix cache and
// copy-on-write (no device code).
//
// Sources: "Text Generation Inference: Hugging Face's production-grade LLM
// inference server", section "Under the Hood: PagedAttention" (prefix sharing:
// tables pointing at the same blocks, copy-on-write before a write into a
// shared block); pyshine "text-generation-inference", sections "The radix
// prefix cache" (block 0 reserved, free list plus a compressed prefix tree at
// block granularity, references on the match before any eviction, LRU eviction
// of unreferenced prefixes, node splits on partial overlap, double-cached
// blocks back to the free list on release) and "Inside the batching task" (a
// fully cached prompt gives one token back).
//
// Rules (the same as the plain model the tests compare against):
//   * a cached block holds one full block of tokens and is keyed by the whole
//     token prefix it ends; the tree's nodes hold runs of such blocks;
//   * every mutating call advances one tick; matching, inserting and the
//     touch on release stamp the blocks on the request's path with it;
//   * eviction frees one block at a time: among tail blocks of childless
//     nodes that no sequence references, the oldest (tick, block id);
//   * fresh blocks are taken lowest id first;
//   * a write into a block that is cached or referenced twice copies it;
//   * a call needing more fresh blocks than the free blocks plus the blocks
//     eviction could free at its start fails before changing anything.
//
// Data structures: a free-block bitmap (lowest id out first); per-block
// reference counts, use ticks and (node, index) of cached blocks; children
// keyed by their first block's tokens; a lazily validated min-heap of
// (tick, block) eviction candidates; and the number of blocks eviction could
// free, kept up to date on every reference, cache and eviction change so
// that a capacity check under pressure costs O(1), not a walk of the tree.
// Per node: its referenced blocks (nref), the highest index among them
// (last_ref) and its children whose subtrees hold a referenced block
// (pinned_children). A node's evictable blocks are then the ones after
// last_ref, unless a child is pinned (then none).

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <functional>
#include <map>
#include <memory>
#include <queue>
#include <unordered_map>
#include <utility>
#include <vector>

#include "pagedkv.h"

namespace pa {
namespace {

struct Node {
  Node* parent = nullptr;
  std::vector<int32_t> tokens;  // block_size tokens per block
  std::vector<int32_t> blocks;
  std::map<std::vector<int32_t>, std::unique_ptr<Node>> children;  // by first block's tokens
  int32_t nref = 0;             // blocks of this node a live sequence references
  int32_t last_ref = -1;        // highest index of such a block (-1: none)
  int32_t pinned_children = 0;  // children whose subtree holds a referenced block
};

struct Seq {
  std::vector<int32_t> blocks;
  int32_t ntok = 0;
};

// The free blocks as a bitmap: freeing sets a bit, taking clears the lowest
// set one. `low` is a word index below which every word is zero.
struct FreeBlocks {
  std::vector<uint64_t> words;
  int32_t count = 0;
  size_t low = 0;

  void init(int32_t num_blocks) {
    words.assign(((size_t)num_blocks + 63) / 64, 0);
    count = 0;
    low = words.size();
  }
  void insert(int32_t b) {
    uint64_t& w = words[(size_t)b >> 6];
    const uint64_t m = 1ull << (b & 63);
    if (w & m) return;
    w |= m;
    ++count;
    low = std::min(low, (size_t)b >> 6);
  }
  bool empty() const { return count == 0; }
  int32_t size() const { return count; }
  int32_t take_lowest() {  // callers check empty() first
    while (words[low] == 0) ++low;
    const int32_t b = (int32_t)(low * 64) + __builtin_ctzll(words[low]);
    words[low] &= words[low] - 1;
    --count;
    return b;
  }
};

}  // namespace
}  // namespace pa

struct pa_prefix_cache {
  int32_t nb = 0, bs = 0;
  int64_t tick = 0, next_seq = 1;
  pa::FreeBlocks free_set;
  std::vector<int32_t> ref;
  std::vector<pa::Node*> node_of;  // cached block -> its node (nullptr: not cached)
  std::vector<int32_t> idx_of;     // index of a cached block in its node
  std::vector<int64_t> last_use;   // tick of a cached block
  int32_t cached = 0, used = 0;
  int64_t evictable = 0;  // blocks repeated eviction could free
  pa::Node root;
  std::unordered_map<int64_t, pa::Seq> seqs;
  using Cand = std::pair<int64_t, int32_t>;
  std::priority_queue<Cand, std::vector<Cand>, std::greater<Cand>> heap;

  // ---------------------------------------------------------------- helpers
  std::vector<int32_t> key_at(const int32_t* t) const { return std::vector<int32_t>(t, t + bs); }

  bool evictable_now(int32_t b) const {
    const pa::Node* n = node_of[b];
    return n && ref[b] == 0 && n->children.empty() &&
           idx_of[b] == (int32_t)n->blocks.size() - 1;
  }
  void maybe_push(int32_t b) {
    if (evictable_now(b)) heap.push({last_use[b], b});
  }
  // ---- the evictable count ------------------------------------------------
  // Blocks repeated eviction could free: cached, unreferenced, with nothing
  // referenced after them in their node or below it.
  int64_t node_evictable(const pa::Node& n) const {
    if (&n == &root || n.pinned_children > 0) return 0;
    return (int64_t)n.blocks.size() - 1 - n.last_ref;
  }
  static bool active(const pa::Node& n) { return n.nref > 0 || n.pinned_children > 0; }
  // n's subtree went from holding a referenced block (`was`) to active(*n):
  // tell the ancestors, up to the first whose own state does not change.
  void propagate(pa::Node* n, bool was) {
    while (n != &root) {
      const bool now = active(*n);
      if (now == was) return;
      pa::Node* p = n->parent;
      const bool p_was = active(*p);
      const int64_t e0 = node_evictable(*p);
      p->pinned_children += now ? 1 : -1;
      evictable += node_evictable(*p) - e0;
      n = p;
      was = p_was;
    }
  }
  // Cached block b just became referenced (ref 0 -> 1) or unreferenced (1 -> 0).
  void ref_changed(int32_t b, bool referenced) {
    pa::Node* n = node_of[b];
    const bool was = active(*n);
    const int64_t e0 = node_evictable(*n);
    const int32_t i = idx_of[b];
    if (referenced) {
      ++n->nref;
      if (i > n->last_ref) n->last_ref = i;
    } else {
      --n->nref;
      if (i == n->last_ref) {
        int32_t k = i - 1;
        while (k >= 0 && ref[n->blocks[k]] == 0) --k;
        n->last_ref = k;
      }
    }
    evictable += node_evictable(*n) - e0;
    propagate(n, was);
  }
  // nref and last_ref of n from its blocks' reference counts.
  void recount(pa::Node& n) {
    n.nref = 0;
    n.last_ref = -1;
    for (int32_t i = 0; i < (int32_t)n.blocks.size(); ++i)
      if (ref[n.blocks[i]] > 0) {
        ++n.nref;
        n.last_ref = i;
      }
  }

  void add_ref(int32_t b) {
    if (ref[b]++ == 0) {
      ++used;
      if (node_of[b]) ref_changed(b, true);
    }
  }
  void drop_ref(int32_t b) {
    if (--ref[b] == 0) {
      --used;
      if (node_of[b]) {
        ref_changed(b, false);
        maybe_push(b);
      } else {
        free_set.insert(b);
      }
    }
  }
  // A reference taken back before anything else changed (no heap push: the
  // block's tick and its candidate entry are as they were).
  void undo_ref(int32_t b) {
    if (--ref[b] == 0) {
      --used;
      if (node_of[b]) ref_changed(b, false);
    }
  }

  bool reserve(int64_t needed) const {
    return needed <= (int64_t)free_set.size() + evictable;
  }

  void evict_one() {
    while (!heap.empty()) {
      const Cand c = heap.top();
      heap.pop();
      const int32_t b = c.second;
      if (!evictable_now(b) || last_use[b] != c.first) continue;  // stale entry
      pa::Node* n = node_of[b];
      node_of[b] = nullptr;
      --cached;
      --evictable;  // b was the last unreferenced block of an unpinned leaf
      free_set.insert(b);
      if (n->blocks.size() > 1) {
        n->blocks.pop_back();
        n->tokens.resize(n->blocks.size() * bs);
        maybe_push(n->blocks.back());
      } else {
        // the node empties: erase it from its parent by its key (it held no
        // referenced block, so the parent's pinned count does not change)
        pa::Node* parent = n->parent;
        parent->children.erase(key_at(n->tokens.data()));  // destroys n
        if (parent != &root && parent->children.empty()) maybe_push(parent->blocks.back());
      }
      return;
    }
  }

  // Re-seed the candidate heap from the tree (only if it ran dry while
  // eviction was still possible, which the bookkeeping should never allow).
  void rebuild_heap() {
    std::function<void(pa::Node&)> visit = [&](pa::Node& n) {
      for (auto& kv : n.children) visit(*kv.second);
      if (&n != &root && !n.blocks.empty()) maybe_push(n.blocks.back());
    };
    visit(root);
  }

  // Lowest free block, evicting first if none is free; -1 if nothing can be
  // freed (callers have checked capacity, so this does not happen).
  int32_t take() {
    if (free_set.empty()) evict_one();
    if (free_set.empty()) {
      rebuild_heap();
      evict_one();
    }
    if (free_set.empty()) return -1;
    return free_set.take_lowest();
  }

  // Longest cached block prefix of tokens[0, n): its blocks in order.
  std::vector<int32_t> match(const int32_t* tokens, int32_t n) const {
    std::vector<int32_t> out;
    const pa::Node* node = &root;
    int32_t pos = 0;
    while (pos + bs <= n) {
      auto it = node->children.find(key_at(tokens + pos));
      if (it == node->children.end()) break;
      const pa::Node* c = it->second.get();
      size_t j = 0;
      while (j < c->blocks.size() && pos + bs <= n &&
             std::equal(tokens + pos, tokens + pos + bs, c->tokens.begin() + j * bs)) {
        out.push_back(c->blocks[j]);
        ++j;
        pos += bs;
      }
      if (j < c->blocks.size()) break;
      node = c;
    }
    return out;
  }

  // Split c so that its first j blocks form a new node; returns that node.
  pa::Node* split(pa::Node* c, size_t j) {
    const int64_t e0 = node_evictable(*c);
    pa::Node* parent = c->parent;
    auto it = parent->children.find(key_at(c->tokens.data()));
    std::unique_ptr<pa::Node> own = std::move(it->second);
    auto up = std::make_unique<pa::Node>();
    up->parent = parent;
    up->blocks.assign(c->blocks.begin(), c->blocks.begin() + j);
    up->tokens.assign(c->tokens.begin(), c->tokens.begin() + j * bs);
    c->blocks.erase(c->blocks.begin(), c->blocks.begin() + j);
    c->tokens.erase(c->tokens.begin(), c->tokens.begin() + j * bs);
    for (size_t i = 0; i < up->blocks.size(); ++i) {
      node_of[up->blocks[i]] = up.get();
      idx_of[up->blocks[i]] = (int32_t)i;
    }
    for (size_t i = 0; i < c->blocks.size(); ++i) idx_of[c->blocks[i]] = (int32_t)i;
    c->parent = up.get();
    pa::Node* u = up.get();
    recount(*u);
    recount(*c);
    u->pinned_children = active(*c) ? 1 : 0;  // u is as active as c was: the parent is unchanged
    evictable += node_evictable(*u) + node_evictable(*c) - e0;
    u->children[key_at(c->tokens.data())] = std::move(own);
    it->second = std::move(up);
    return u;
  }
};

extern "C" pa_status pa_prefix_fork(pa_prefix_cache* pc, int64_t seq_id, int64_t* child_id);
extern "C" pa_status pa_prefix_release(pa_prefix_cache* pc, int64_t seq_id,
                                       const int32_t* tokens, int32_t num_tokens);

namespace {

pa_status seq_of(pa_prefix_cache* pc, int64_t id, pa::Seq** out) {
  if (!pc) return PA_ERR_INVALID_ARG;
  auto it = pc->seqs.find(id);
  if (it == pc->seqs.end()) return PA_ERR_INVALID_ARG;
  *out = &it->second;
  return PA_OK;
}

// Fresh blocks a write of positions [p0, p1) needs (growth + copies).
int64_t blocks_needed(const pa_prefix_cache* pc, const pa::Seq& s, int32_t p0, int32_t p1) {
  if (p1 <= p0) return 0;
  int64_t need = 0;
  for (int32_t i = p0 / pc->bs; i <= (p1 - 1) / pc->bs; ++i) {
    if (i >= (int32_t)s.blocks.size()) ++need;
    else if (pc->ref[s.blocks[i]] > 1 || pc->node_of[s.blocks[i]]) ++need;
  }
  return need;
}

// Existing blocks of [p0, p1) a write must copy first.
int64_t copies_needed(const pa_prefix_cache* pc, const pa::Seq& s, int32_t p0, int32_t p1) {
  if (p1 <= p0) return 0;
  int64_t n = 0;
  for (int32_t i = p0 / pc->bs; i <= (p1 - 1) / pc->bs && i < (int32_t)s.blocks.size(); ++i)
    if (pc->ref[s.blocks[i]] > 1 || pc->node_of[s.blocks[i]]) ++n;
  return n;
}

// The write itself (capacity already checked), one block at a time: a block
// past the end is taken fresh, a cached or shared one is copied first (its
// first written position decides, as the later ones then see the fresh
// block); then the block's positions get their slots. Copies are appended.
bool do_write(pa_prefix_cache* pc, pa::Seq& s, int32_t p0, int32_t p1, int64_t* slots,
              std::vector<std::pair<int32_t, int32_t>>& copies) {
  const int32_t bs = pc->bs;
  if (p1 <= p0) return true;
  for (int32_t i = p0 / bs; i <= (p1 - 1) / bs; ++i) {
    if (i == (int32_t)s.blocks.size()) {
      const int32_t b = pc->take();
      if (b < 0) return false;
      pc->add_ref(b);
      s.blocks.push_back(b);
    } else {
      const int32_t old = s.blocks[i];
      if (pc->ref[old] > 1 || pc->node_of[old]) {
        const int32_t nb = pc->take();
        if (nb < 0) return false;
        pc->add_ref(nb);
        copies.emplace_back(old, nb);
        s.blocks[i] = nb;
        pc->drop_ref(old);
      }
    }
    const int32_t q0 = std::max(p0, i * bs), q1 = std::min(p1, (i + 1) * bs);
    if (slots) {
      int64_t slot = (int64_t)s.blocks[i] * bs + (q0 - i * bs);
      for (int32_t p = q0; p < q1; ++p) slots[p - p0] = slot++;
    }
    s.ntok = std::max(s.ntok, q1);
  }
  return true;
}

}  // namespace

extern "C" pa_status pa_prefix_cache_create(int32_t num_blocks, int32_t block_size,
                                            pa_prefix_cache** out) {
  if (!out || num_blocks < 2 || block_size < 1) return PA_ERR_INVALID_ARG;
  *out = nullptr;
  auto* pc = new (std::nothrow) pa_prefix_cache;
  if (!pc) return PA_ERR_CAPACITY;
  pc->nb = num_blocks;
  pc->bs = block_size;
  pc->ref.assign(num_blocks, 0);
  pc->node_of.assign(num_blocks, nullptr);
  pc->idx_of.assign(num_blocks, 0);
  pc->last_use.assign(num_blocks, 0);
  pc->free_set.init(num_blocks);
  for (int32_t b = 1; b < num_blocks; ++b) pc->free_set.insert(b);
  *out = pc;
  return PA_OK;
}

extern "C" void pa_prefix_cache_destroy(pa_prefix_cache* pc) { delete pc; }

extern "C" pa_status pa_prefix_admit(pa_prefix_cache* pc, const int32_t* tokens,
                                     int32_t num_tokens, int64_t* seq_id,
                                     int32_t* cached_tokens) {
  if (!pc || !tokens || !seq_id || !cached_tokens || num_tokens < 1) return PA_ERR_INVALID_ARG;
  pc->tick += 1;
  const std::vector<int32_t> matched = pc->match(tokens, num_tokens);
  for (int32_t b : matched) pc->add_ref(b);  // references first: no eviction can take them
  const int64_t need = ((int64_t)num_tokens + pc->bs - 1) / pc->bs - (int64_t)matched.size();
  if (!pc->reserve(need)) {
    for (int32_t b : matched) pc->undo_ref(b);
    return PA_ERR_CAPACITY;
  }
  for (int32_t b : matched) pc->last_use[b] = pc->tick;
  pa::Seq s;
  s.blocks = matched;
  while ((int64_t)s.blocks.size() * pc->bs < num_tokens) {
    const int32_t b = pc->take();
    if (b < 0) {
      for (int32_t x : s.blocks) pc->drop_ref(x);
      return PA_ERR_CAPACITY;
    }
    pc->add_ref(b);
    s.blocks.push_back(b);
  }
  s.ntok = num_tokens;
  int32_t cached = (int32_t)matched.size() * pc->bs;
  if (cached == num_tokens) cached = num_tokens - 1;  // one position is always computed
  const int64_t id = pc->next_seq++;
  pc->seqs.emplace(id, std::move(s));
  *seq_id = id;
  *cached_tokens = cached;
  return PA_OK;
}

extern "C" pa_status pa_prefix_write_slots(pa_prefix_cache* pc, int64_t seq_id, int32_t pos_begin,
                                           int32_t pos_end, int64_t* slots, int32_t* copy_src,
                                           int32_t* copy_dst, int32_t max_copies,
                                           int32_t* num_copies) {
  pa::Seq* s = nullptr;
  pa_status st = seq_of(pc, seq_id, &s);
  if (st != PA_OK) return st;
  if (pos_begin < 0 || pos_begin > s->ntok || pos_end < pos_begin || !num_copies ||
      (pos_end > pos_begin && !slots))
    return PA_ERR_INVALID_ARG;
  const int64_t need = blocks_needed(pc, *s, pos_begin, pos_end);
  const int64_t ncopy = copies_needed(pc, *s, pos_begin, pos_end);
  if (ncopy > 0 && (max_copies < ncopy || !copy_src || !copy_dst)) return PA_ERR_INVALID_ARG;
  pc->tick += 1;
  if (!pc->reserve(need)) return PA_ERR_CAPACITY;
  std::vector<std::pair<int32_t, int32_t>> copies;
  const bool ok = do_write(pc, *s, pos_begin, pos_end, slots, copies);
  for (size_t i = 0; i < copies.size(); ++i) {
    copy_src[i] = copies[i].first;
    copy_dst[i] = copies[i].second;
  }
  *num_copies = (int32_t)copies.size();
  return ok ? PA_OK : PA_ERR_CAPACITY;
}

extern "C" pa_status pa_prefix_append_tokens(pa_prefix_cache* pc, const int64_t* seq_ids,
                                             int32_t num_seqs, int64_t* slots, int32_t* copy_src,
                                             int32_t* copy_dst, int32_t max_copies,
                                             int32_t* num_copies, int32_t* num_done) {
  if (!pc || num_seqs < 0 || !num_copies || !num_done || (num_seqs > 0 && (!seq_ids || !slots)))
    return PA_ERR_INVALID_ARG;
  if (num_seqs > 0 && (max_copies < num_seqs || !copy_src || !copy_dst)) return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < num_seqs; ++i)
    if (!pc->seqs.count(seq_ids[i])) return PA_ERR_INVALID_ARG;
  *num_copies = 0;
  *num_done = 0;
  std::vector<std::pair<int32_t, int32_t>> copies;
  pa_status result = PA_OK;
  for (int32_t i = 0; i < num_seqs; ++i) {
    pa::Seq& s = pc->seqs.find(seq_ids[i])->second;
    const int32_t p = s.ntok;
    pc->tick += 1;
    if (!pc->reserve(blocks_needed(pc, s, p, p + 1)) || !do_write(pc, s, p, p + 1, slots + i, copies)) {
      result = PA_ERR_CAPACITY;
      break;
    }
    *num_done = i + 1;
  }
  for (size_t c = 0; c < copies.size(); ++c) {
    copy_src[c] = copies[c].first;
    copy_dst[c] = copies[c].second;
  }
  *num_copies = (int32_t)copies.size();
  return result;
}

extern "C" pa_status pa_prefix_fork(pa_prefix_cache* pc, int64_t seq_id, int64_t* child_id) {
  pa::Seq* s = nullptr;
  pa_status st = seq_of(pc, seq_id, &s);
  if (st != PA_OK) return st;
  if (!child_id) return PA_ERR_INVALID_ARG;
  pc->tick += 1;
  pa::Seq c = *s;
  for (int32_t b : c.blocks) pc->add_ref(b);
  const int64_t id = pc->next_seq++;
  pc->seqs.emplace(id, std::move(c));
  *child_id = id;
  return PA_OK;
}

extern "C" pa_status pa_prefix_fork_batch(pa_prefix_cache* pc, const int64_t* seq_ids,
                                          int32_t num_seqs, int64_t* child_ids) {
  if (!pc || num_seqs < 0 || (num_seqs > 0 && (!seq_ids || !child_ids))) return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < num_seqs; ++i)
    if (!pc->seqs.count(seq_ids[i])) return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < num_seqs; ++i) {
    const pa_status st = pa_prefix_fork(pc, seq_ids[i], child_ids + i);
    if (st != PA_OK) return st;
  }
  return PA_OK;
}

extern "C" pa_status pa_prefix_discard(pa_prefix_cache* pc, const int64_t* seq_ids,
                                       int32_t num_seqs) {
  if (!pc || num_seqs < 0 || (num_seqs > 0 && !seq_ids)) return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < num_seqs; ++i)
    if (!pc->seqs.count(seq_ids[i])) return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < num_seqs; ++i) {
    const pa_status st = pa_prefix_release(pc, seq_ids[i], nullptr, 0);
    if (st != PA_OK) return st;
  }
  return PA_OK;
}

extern "C" pa_status pa_prefix_release(pa_prefix_cache* pc, int64_t seq_id,
                                       const int32_t* tokens, int32_t num_tokens) {
  pa::Seq* sp = nullptr;
  pa_status st = seq_of(pc, seq_id, &sp);
  if (st != PA_OK) return st;
  if (num_tokens < 0 || (num_tokens > 0 && !tokens)) return PA_ERR_INVALID_ARG;
  pa::Seq s = std::move(*sp);
  pc->seqs.erase(seq_id);
  pc->tick += 1;
  const int32_t bs = pc->bs;
  const int32_t nfull = std::min(num_tokens, s.ntok) / bs;
  // walk the cached path, touching it; then cache the first uncached run
  pa::Node* node = &pc->root;
  pa::Node* cut = nullptr;  // the path diverges inside this node ...
  size_t cut_at = 0;        // ... after this many of its blocks
  int32_t i = 0;
  while (i < nfull) {
    auto it = node->children.find(pc->key_at(tokens + (size_t)i * bs));
    if (it == node->children.end()) break;
    pa::Node* c = it->second.get();
    size_t j = 0;
    while (j < c->blocks.size() && i < nfull &&
           std::equal(tokens + (size_t)i * bs, tokens + (size_t)(i + 1) * bs,
                      c->tokens.begin() + j * bs)) {
      pc->last_use[c->blocks[j]] = pc->tick;
      pc->maybe_push(c->blocks[j]);
      ++j;
      ++i;
    }
    if (j < c->blocks.size()) {
      cut = c;
      cut_at = j;
      break;
    }
    node = c;
  }
  int32_t k = i;
  while (k < nfull && !pc->node_of[s.blocks[k]]) ++k;  // a block holding another prefix stops it
  if (k > i) {
    pa::Node* parent = cut ? pc->split(cut, cut_at) : node;
    auto n = std::make_unique<pa::Node>();
    n->parent = parent;
    n->tokens.assign(tokens + (size_t)i * bs, tokens + (size_t)k * bs);
    n->blocks.assign(s.blocks.begin() + i, s.blocks.begin() + k);
    for (int32_t q = i; q < k; ++q) {
      const int32_t b = s.blocks[q];
      pc->node_of[b] = n.get();
      pc->idx_of[b] = q - i;
      pc->last_use[b] = pc->tick;
      ++pc->cached;
    }
    // the releasing sequence still references every block of the new leaf:
    // nothing in it is evictable yet, and its parent's subtree is pinned
    pa::Node* leaf = n.get();
    pc->recount(*leaf);
    parent->children[pc->key_at(tokens + (size_t)i * bs)] = std::move(n);
    pc->evictable += pc->node_evictable(*leaf);
    pc->propagate(leaf, false);
  }
  for (int32_t b : s.blocks) pc->drop_ref(b);
  return PA_OK;
}

extern "C" pa_status pa_prefix_table(pa_prefix_cache* pc, int64_t seq_id, int32_t* table,
                                     int32_t max_blocks, int32_t* num_blocks,
                                     int32_t* num_tokens) {
  pa::Seq* s = nullptr;
  pa_status st = seq_of(pc, seq_id, &s);
  if (st != PA_OK) return st;
  if (!num_blocks || (int32_t)s->blocks.size() > max_blocks || (max_blocks > 0 && !table))
    return PA_ERR_INVALID_ARG;
  std::copy(s->blocks.begin(), s->blocks.end(), table);
  *num_blocks = (int32_t)s->blocks.size();
  if (num_tokens) *num_tokens = s->ntok;
  return PA_OK;
}

extern "C" pa_status pa_prefix_tables(pa_prefix_cache* pc, const int64_t* seq_ids,
                                      int32_t num_seqs, int32_t* tables, int32_t max_blocks,
                                      int32_t* context_lens) {
  if (!pc || num_seqs < 0 || (num_seqs > 0 && (!seq_ids || !tables || !context_lens)))
    return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < num_seqs; ++i) {
    auto it = pc->seqs.find(seq_ids[i]);
    if (it == pc->seqs.end() || (int32_t)it->second.blocks.size() > max_blocks)
      return PA_ERR_INVALID_ARG;
  }
  for (int32_t i = 0; i < num_seqs; ++i) {
    const pa::Seq& s = pc->seqs.find(seq_ids[i])->second;
    int32_t* row = tables + (size_t)i * max_blocks;
    std::copy(s.blocks.begin(), s.blocks.end(), row);
    std::fill(row + s.blocks.size(), row + max_blocks, 0);
    context_lens[i] = s.ntok;
  }
  return PA_OK;
}

extern "C" pa_status pa_prefix_evictable(const pa_prefix_cache* pc, int32_t* evictable_blocks) {
  if (!pc || !evictable_blocks) return PA_ERR_INVALID_ARG;
  *evictable_blocks = (int32_t)pc->evictable;
  return PA_OK;
}

extern "C" pa_status pa_prefix_stats(const pa_prefix_cache* pc, int32_t* free_blocks,
                                     int32_t* cached_blocks, int32_t* used_blocks) {
  if (!pc) return PA_ERR_INVALID_ARG;
  if (free_blocks) *free_blocks = (int32_t)pc->free_set.size();
  if (cached_blocks) *cached_blocks = pc->cached;
  if (used_blocks) *used_blocks = pc->used;
  return PA_OK;
}
