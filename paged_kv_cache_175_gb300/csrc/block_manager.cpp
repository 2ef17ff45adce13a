// Host KV block manager: cross-request reuse through a tree of full blocks, priority-LRU
// eviction with retention ranges, and a host tier for offloaded blocks.  The policy is
// stated in include/pkv_bm.h ("KV 캐시 시스템 (KV Cache System)": "요청 간 재사용",
// "보존 정책", "호스트 메모리로의 오프로딩", "제한된 어텐션 윈도우 크기").
//
// Data structures: free GPU blocks and free host slots in ordered sets (lowest id first);
// unreferenced cached GPU blocks and occupied host slots in ordered sets keyed by
// (priority, time, -depth, id), so the victim is the first element; tree nodes in a slot
// vector with generation numbers (a sequence remembers its chain's last node by slot and
// generation, so a dropped and recycled slot is never taken for its parent); a hash index
// from (parent, block tokens) to nodes, with the tokens compared on every hit.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <set>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "../../include/pkv_bm.h"

namespace {

constexpr int kRoot = -1;

struct VictimKey {
  int prio;
  int64_t time;
  int neg_depth;
  int id;
  bool operator<(const VictimKey& o) const {
    return std::tie(prio, time, neg_depth, id) < std::tie(o.prio, o.time, o.neg_depth, o.id);
  }
};

struct Node {
  bool alive = false;
  uint32_t gen = 0;
  int parent = kRoot;
  int depth = 0;
  int prio = 0;
  int64_t time = 0;
  bool on_host = false;
  int where = -1;                  // GPU block or host slot
  uint64_t hash = 0;
  std::vector<int32_t> key;        // the block's token ids
  std::vector<int> children;
};

struct ChainRef {                  // last registered node of a sequence's chain
  int slot = kRoot;                // kRoot: the chain is at the root
  uint32_t gen = 0;
  bool broken = false;
};

struct Seq {
  std::vector<int32_t> tokens;
  std::vector<int> blocks;
  std::vector<int> prios;
  std::vector<pkv_token_range> ranges;
  ChainRef chain;
  int first = 0;                   // first block still held (after window slides)
};

}  // namespace

struct pkv_block_manager {
  int N, bs, H, offload_min, default_prio;
  std::vector<int> gpu_ref, gpu_node, host_node;
  std::set<int> free_gpu, free_host;
  std::set<VictimKey> cached_gpu, cached_host;
  std::vector<Node> nodes;
  std::vector<int> free_nodes;
  std::unordered_multimap<uint64_t, int> index;
  std::unordered_map<int64_t, Seq> seqs;
  int64_t clock = 0;
  std::vector<pkv_block_copy> copies;
  int64_t reused_tokens = 0, evictions = 0, offloads = 0, onloads = 0, drops = 0;

  // ---- helpers ------------------------------------------------------------------------------
  static uint64_t mix(uint64_t h, uint64_t x) {
    h ^= x + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
    return h * 0xff51afd7ed558ccdull;
  }
  uint64_t key_hash(int parent, const int32_t* toks) const {
    uint64_t h = mix(0x84222325cbf29ce4ull, (uint64_t)(int64_t)parent);
    for (int i = 0; i < bs; ++i) h = mix(h, (uint64_t)(uint32_t)toks[i]);
    return h;
  }
  int find(int parent, const int32_t* toks, uint64_t h) const {
    auto range = index.equal_range(h);
    for (auto it = range.first; it != range.second; ++it) {
      const Node& n = nodes[it->second];
      if (n.parent == parent && std::memcmp(n.key.data(), toks, sizeof(int32_t) * bs) == 0) return it->second;
    }
    return -1;
  }
  void unindex(int id) {
    auto range = index.equal_range(nodes[id].hash);
    for (auto it = range.first; it != range.second; ++it)
      if (it->second == id) {
        index.erase(it);
        return;
      }
  }
  VictimKey vkey(int id) const {
    const Node& n = nodes[id];
    return VictimKey{n.prio, n.time, -n.depth, n.where};
  }
  bool chain_alive(const ChainRef& c) const {
    if (c.broken) return false;
    if (c.slot == kRoot) return true;
    return nodes[c.slot].alive && nodes[c.slot].gen == c.gen;
  }

  int priority(const std::vector<pkv_token_range>& ranges, int i) const {
    const int64_t lo = (int64_t)i * bs, hi = (int64_t)(i + 1) * bs;
    int best = -1;
    for (const auto& r : ranges) {
      const int64_t e = r.end < 0 ? hi : r.end;
      if (r.start < hi && e > lo) best = std::max(best, (int)r.priority);
    }
    return best < 0 ? default_prio : best;
  }

  // Remove a node and its subtree from the tree.
  void drop(int root_id) {
    std::vector<int> stack{root_id};
    const int parent = nodes[root_id].parent;
    if (parent != kRoot) {
      auto& ch = nodes[parent].children;
      ch.erase(std::remove(ch.begin(), ch.end(), root_id), ch.end());
    }
    while (!stack.empty()) {
      const int x = stack.back();
      stack.pop_back();
      Node& n = nodes[x];
      for (int c : n.children) stack.push_back(c);
      if (n.on_host) {
        cached_host.erase(vkey(x));
        host_node[n.where] = -1;
        free_host.insert(n.where);
      } else {
        const int b = n.where;
        if (gpu_ref[b] == 0) {
          cached_gpu.erase(vkey(x));
          free_gpu.insert(b);
        }
        gpu_node[b] = -1;
      }
      unindex(x);
      n.alive = false;
      ++n.gen;
      n.children.clear();
      n.key.clear();
      free_nodes.push_back(x);
      ++drops;
    }
  }

  // A free host slot, dropping a host block if needed; -1 if there is none.
  int host_slot() {
    if (!free_host.empty()) return *free_host.begin();
    if (cached_host.empty()) return -1;
    const int h = cached_host.begin()->id;
    drop(host_node[h]);
    return h;
  }

  // Evict one unreferenced cached GPU block; false if there is none.
  bool evict_one() {
    if (cached_gpu.empty()) return false;
    const VictimKey v = *cached_gpu.begin();
    const int b = v.id, nid = gpu_node[b];
    ++evictions;
    if (v.prio >= offload_min && H > 0) {
      const int h = host_slot();
      if (h >= 0 && gpu_node[b] == nid) {      // the host eviction may have dropped it
        cached_gpu.erase(v);
        copies.push_back(pkv_block_copy{PKV_COPY_OFFLOAD, b, h});
        free_host.erase(h);
        Node& n = nodes[nid];
        n.on_host = true;
        n.where = h;
        host_node[h] = nid;
        cached_host.insert(vkey(nid));
        gpu_node[b] = -1;
        free_gpu.insert(b);
        ++offloads;
        return true;
      }
    }
    if (gpu_node[b] == nid) drop(nid);
    return true;
  }

  // A free GPU block (not yet marked used); -1 if every block is referenced.
  int alloc() {
    while (free_gpu.empty())
      if (!evict_one()) return -1;
    return *free_gpu.begin();
  }
  void take_gpu(int b) { free_gpu.erase(b); }

  void register_block(Seq& s, int i, int b) {
    if (!chain_alive(s.chain)) {
      s.chain.broken = true;
      return;
    }
    const int parent = s.chain.slot;
    const int32_t* toks = s.tokens.data() + (size_t)i * bs;
    const uint64_t h = key_hash(parent, toks);
    if (find(parent, toks, h) >= 0) {          // registered by another sequence first
      s.chain.broken = true;
      return;
    }
    int id;
    if (!free_nodes.empty()) {
      id = free_nodes.back();
      free_nodes.pop_back();
    } else {
      id = (int)nodes.size();
      nodes.emplace_back();
    }
    Node& n = nodes[id];
    n.alive = true;
    n.parent = parent;
    n.depth = parent == kRoot ? 1 : nodes[parent].depth + 1;
    n.prio = s.prios[i];
    n.time = clock;
    n.on_host = false;
    n.where = b;
    n.hash = h;
    n.key.assign(toks, toks + bs);
    n.children.clear();
    if (parent != kRoot) nodes[parent].children.push_back(id);
    index.emplace(h, id);
    gpu_node[b] = id;
    s.chain.slot = id;
    s.chain.gen = n.gen;
  }

  void release_block(int b) {
    if (--gpu_ref[b] > 0) return;
    const int nid = gpu_node[b];
    if (nid >= 0) {
      nodes[nid].time = clock;
      cached_gpu.insert(vkey(nid));
    } else {
      free_gpu.insert(b);
    }
  }
  void release_seq(Seq& s) {
    for (size_t i = (size_t)s.first; i < s.blocks.size(); ++i) release_block(s.blocks[i]);
  }

  // ---- API --------------------------------------------------------------------------------------
  int add_sequence(int64_t seq_id, const int32_t* tokens, int n, const pkv_token_range* ranges, int n_ranges,
                   int32_t* table, int table_cap) {
    if (seqs.count(seq_id)) return PKV_EINVAL;
    const int nb = (n + bs - 1) / bs;
    if (table_cap < nb) return PKV_ERANGE;
    ++clock;
    Seq s;
    s.tokens.assign(tokens, tokens + n);
    s.ranges.assign(ranges, ranges + n_ranges);
    s.prios.resize(nb);
    for (int i = 0; i < nb; ++i) s.prios[i] = priority(s.ranges, i);
    // longest matching chain, one token left to compute
    std::vector<int> matched;
    int parent = kRoot;
    const int max_reuse = std::max(0, (n - 1) / bs);
    for (int i = 0; i < max_reuse; ++i) {
      const int32_t* toks = tokens + (size_t)i * bs;
      const int id = find(parent, toks, key_hash(parent, toks));
      if (id < 0) break;
      matched.push_back(id);
      parent = id;
    }
    std::vector<uint32_t> gens(matched.size());
    for (size_t i = 0; i < matched.size(); ++i) gens[i] = nodes[matched[i]].gen;
    bool failed = false;
    for (size_t i = 0; i < matched.size(); ++i) {
      const int nid = matched[i];
      if (!nodes[nid].alive || nodes[nid].gen != gens[i]) break;   // dropped making room
      int b;
      if (nodes[nid].on_host) {
        const int h = nodes[nid].where;
        b = alloc();
        if (b < 0) {
          failed = true;
          break;
        }
        if (!nodes[nid].alive || nodes[nid].gen != gens[i] || !nodes[nid].on_host || nodes[nid].where != h) break;
        take_gpu(b);
        copies.push_back(pkv_block_copy{PKV_COPY_ONLOAD, h, b});
        cached_host.erase(vkey(nid));
        host_node[h] = -1;
        free_host.insert(h);
        nodes[nid].on_host = false;
        nodes[nid].where = b;
        gpu_node[b] = nid;
        ++onloads;
      } else {
        b = nodes[nid].where;
        if (gpu_ref[b] == 0) cached_gpu.erase(vkey(nid));
      }
      ++gpu_ref[b];
      nodes[nid].prio = s.prios[i];
      nodes[nid].time = clock;
      s.blocks.push_back(b);
      s.chain.slot = nid;
      s.chain.gen = nodes[nid].gen;
    }
    const int reused = (int)s.blocks.size();
    if (!failed) {
      for (int i = reused; i < nb; ++i) {
        const int b = alloc();
        if (b < 0) {
          failed = true;
          break;
        }
        take_gpu(b);
        gpu_ref[b] = 1;
        s.blocks.push_back(b);
      }
    }
    if (failed) {
      release_seq(s);                         // nothing new was registered
      return PKV_ENOSPC;
    }
    for (int i = reused; i < nb; ++i)
      if ((int64_t)(i + 1) * bs <= n) register_block(s, i, s.blocks[i]);
    reused_tokens += (int64_t)reused * bs;
    std::copy(s.blocks.begin(), s.blocks.end(), table);
    seqs.emplace(seq_id, std::move(s));
    return reused * bs;
  }

  int append_token(Seq& s, int32_t token, int64_t* slot) {
    ++clock;
    const int t = (int)s.tokens.size();
    const int i = t / bs;
    if (t % bs == 0) {
      const int b = alloc();
      if (b < 0) return PKV_ENOSPC;
      take_gpu(b);
      gpu_ref[b] = 1;
      s.blocks.push_back(b);
      s.prios.push_back(priority(s.ranges, i));
    }
    s.tokens.push_back(token);
    const int b = s.blocks[i];
    if (t % bs == bs - 1) register_block(s, i, b);
    *slot = (int64_t)b * bs + t % bs;
    return PKV_OK;
  }
};

extern "C" {

pkv_block_manager* pkv_bm_create(int num_blocks, int block_size, int host_blocks, int offload_min_priority,
                                 int default_priority) {
  if (num_blocks < 1 || block_size < 1 || host_blocks < 0 || offload_min_priority < 0 ||
      offload_min_priority > 101 || default_priority < 0 || default_priority > 100)
    return nullptr;
  auto* bm = new (std::nothrow) pkv_block_manager();
  if (!bm) return nullptr;
  try {
    bm->N = num_blocks;
    bm->bs = block_size;
    bm->H = host_blocks;
    bm->offload_min = offload_min_priority;
    bm->default_prio = default_priority;
    bm->gpu_ref.assign(num_blocks, 0);
    bm->gpu_node.assign(num_blocks, -1);
    bm->host_node.assign(host_blocks, -1);
    for (int b = 0; b < num_blocks; ++b) bm->free_gpu.insert(bm->free_gpu.end(), b);
    for (int h = 0; h < host_blocks; ++h) bm->free_host.insert(bm->free_host.end(), h);
  } catch (...) {
    delete bm;
    return nullptr;
  }
  return bm;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

int pkv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens, int n_tokens,
                        const pkv_token_range* ranges, int n_ranges, int32_t* table, int table_cap) {
  if (!bm || !tokens || n_tokens < 1 || n_ranges < 0 || (n_ranges && !ranges) || !table) return PKV_EINVAL;
  for (int i = 0; i < n_ranges; ++i)
    if (ranges[i].priority < 0 || ranges[i].priority > 100 || ranges[i].start < 0) return PKV_EINVAL;
  try {
    return bm->add_sequence(seq_id, tokens, n_tokens, ranges, n_ranges, table, table_cap);
  } catch (...) {
    return PKV_ENOSPC;
  }
}

int pkv_bm_append_tokens(pkv_block_manager* bm, const int64_t* seq_ids, const int32_t* tokens, int n,
                         int64_t* slots, int* n_done) {
  if (n_done) *n_done = 0;
  if (!bm || n < 0 || (n && (!seq_ids || !tokens || !slots))) return PKV_EINVAL;
  for (int i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return PKV_EINVAL;
    int st;
    try {
      st = bm->append_token(it->second, tokens[i], &slots[i]);
    } catch (...) {
      st = PKV_ENOSPC;
    }
    if (st != PKV_OK) return st;
    if (n_done) *n_done = i + 1;
  }
  return PKV_OK;
}

int pkv_bm_release(pkv_block_manager* bm, int64_t seq_id) {
  if (!bm) return PKV_EINVAL;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_EINVAL;
  ++bm->clock;
  bm->release_seq(it->second);
  bm->seqs.erase(it);
  return PKV_OK;
}

int pkv_bm_slide_window(pkv_block_manager* bm, int64_t seq_id, int window) {
  if (!bm || window < 1) return PKV_EINVAL;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_EINVAL;
  ++bm->clock;
  Seq& s = it->second;
  const int n = (int)s.tokens.size();
  const int first = std::max(0, n - window) / bm->bs;
  for (int i = s.first; i < first; ++i) bm->release_block(s.blocks[i]);
  s.first = std::max(s.first, first);
  return s.first;
}

int pkv_bm_tables(pkv_block_manager* bm, const int64_t* seq_ids, int n, int32_t* tables, int max_blocks,
                  int32_t* context_lens) {
  if (!bm || n < 0 || max_blocks < 0 || (n && (!seq_ids || !tables || !context_lens))) return PKV_EINVAL;
  for (int r = 0; r < n; ++r) {
    auto it = bm->seqs.find(seq_ids[r]);
    if (it == bm->seqs.end()) return PKV_EINVAL;
    const Seq& s = it->second;
    if ((int)s.blocks.size() > max_blocks) return PKV_ERANGE;
    int32_t* row = tables + (size_t)r * max_blocks;
    for (int i = 0; i < max_blocks; ++i)
      row[i] = (i >= s.first && i < (int)s.blocks.size()) ? s.blocks[i] : -1;
    context_lens[r] = (int32_t)s.tokens.size();
  }
  return PKV_OK;
}

int pkv_bm_take_copies(pkv_block_manager* bm, pkv_block_copy* out, int cap) {
  if (!bm || cap < 0 || (cap && !out)) return PKV_EINVAL;
  const int n = (int)bm->copies.size();
  if (n > cap) return PKV_ERANGE;
  std::copy(bm->copies.begin(), bm->copies.end(), out);
  bm->copies.clear();
  return n;
}

int pkv_bm_pending_copies(const pkv_block_manager* bm) { return bm ? (int)bm->copies.size() : PKV_EINVAL; }

void pkv_bm_counts(const pkv_block_manager* bm, int64_t* out) {
  if (!bm || !out) return;
  const int64_t fr = (int64_t)bm->free_gpu.size(), ca = (int64_t)bm->cached_gpu.size();
  out[0] = fr;
  out[1] = bm->N - fr - ca;
  out[2] = ca;
  out[3] = (int64_t)bm->cached_host.size();
  out[4] = bm->reused_tokens;
  out[5] = bm->evictions;
  out[6] = bm->offloads;
  out[7] = bm->onloads;
  out[8] = bm->drops;
}

}  // extern "C"
