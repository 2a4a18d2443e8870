// pa_block_manager.cpp -- host block manager (include/pa_block_manager.h):
// refcounted physical blocks, per-sequence block tables, copy on write, fork,
// and a prefix cache of full blocks with least-recently-released eviction
// ("03 - Engines Papers", section 2 PagedAttention (vLLM) and section 4
// SGLang (RadixAttention) / automatic prefix caching; "The LLM inference
// engine playbook", Theme 3).
//
// Prefix cache.  A registered (cached) full block records its parent block
// (the cached block before it in its sequence, or none for a first block),
// its token ids and a key hashed over the parent's key and those tokens.
// The key only finds a candidate; a match is accepted when the candidate's
// parent is the block just matched and its tokens equal the prompt's.  The
// cached blocks form a forest: when a cached block is evicted, every cached
// descendant is dropped from the cache with it (none of them could be
// matched again), so a cached block's parent is always the very allocation
// it was registered under, and a full block is never written while
// allocated (appends go to a new block, copy on write only touches partly
// filled blocks): a match is exact.
//
// Steps: blocks released to refcount 0 are parked until pa_bm_end_step, and
// every block that gets a slot is stamped with the step number, so that a
// copy on write of a block written in the same step can be refused.
#include "../../include/pa_block_manager.h"

#include <stdint.h>

#include <algorithm>
#include <deque>
#include <new>
#include <unordered_map>
#include <utility>
#include <vector>

#include "../../include/pa.h"

namespace {

constexpr uint64_t kRootKey = 0x243f6a8885a308d3ull;

inline uint64_t mix64(uint64_t x) {  // splitmix64 finalizer
  x += 0x9e3779b97f4a7c15ull;
  x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
  x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
  return x ^ (x >> 31);
}

inline uint64_t chain_key(uint64_t parent_key, const int32_t* tok, int n) {
  uint64_t h = mix64(parent_key);
  for (int i = 0; i < n; ++i) h = mix64(h ^ static_cast<uint32_t>(tok[i]));
  return h;
}

// Room for `extra` more elements, growing geometrically (so that a
// reservation before a state change keeps appends amortized O(1)).
template <class V>
void make_room(V& v, size_t extra) {
  if (v.size() + extra > v.capacity()) v.reserve(std::max(v.size() + extra, 2 * v.capacity() + 16));
}

struct Seq {
  std::vector<int32_t> blocks;
  std::vector<int32_t> tokens;
};

}  // namespace

struct pa_block_manager {
  int64_t nb = 0;
  int B = 0;
  bool caching = false;
  std::vector<int32_t> ref;
  std::deque<int32_t> free_q;
  std::unordered_map<int64_t, Seq> seqs;
  std::vector<int64_t> copies;  // this step's (src, dst) pairs
  // steps
  uint64_t step = 1;
  std::vector<uint64_t> written;  // step in which the block last got a slot
  // parked blocks: parked_at[b] = tick of its latest parking (0 = not
  // parked); parked_list holds (block, tick) in parking order, and an entry
  // whose tick is not the block's latest is stale
  std::vector<uint64_t> parked_at;
  std::vector<std::pair<int32_t, uint64_t>> parked_list;
  uint64_t park_tick = 0;
  int64_t n_parked = 0;
  // prefix cache, per block
  std::vector<uint8_t> reg;     // registered
  std::vector<uint64_t> key;    // chain key
  std::vector<int32_t> parent;  // parent block (-1 = first block of its chain)
  std::vector<int32_t> child, sib_prev, sib_next;  // registered children lists
  std::vector<int32_t> tok;     // [nb * B] token ids of registered blocks
  std::unordered_map<uint64_t, int32_t> by_key;
  // evictable (registered, refcount 0) blocks, least recently released first
  std::vector<int32_t> lru_prev, lru_next;
  std::vector<uint8_t> in_lru;
  int32_t lru_head = -1, lru_tail = -1;
  int64_t n_lru = 0;

  int64_t available() const { return static_cast<int64_t>(free_q.size()) + n_lru; }

  void lru_push(int32_t b) {
    lru_prev[b] = lru_tail;
    lru_next[b] = -1;
    if (lru_tail >= 0) lru_next[lru_tail] = b; else lru_head = b;
    lru_tail = b;
    in_lru[b] = 1;
    ++n_lru;
  }
  void lru_remove(int32_t b) {
    const int32_t p = lru_prev[b], q = lru_next[b];
    if (p >= 0) lru_next[p] = q; else lru_head = q;
    if (q >= 0) lru_prev[q] = p; else lru_tail = p;
    in_lru[b] = 0;
    --n_lru;
  }
  // Drop one block from the cache (not its descendants).
  void unregister_one(int32_t b) {
    auto it = by_key.find(key[b]);
    if (it != by_key.end() && it->second == b) by_key.erase(it);
    const int32_t p = parent[b];
    if (sib_prev[b] >= 0) sib_next[sib_prev[b]] = sib_next[b]; else if (p >= 0) child[p] = sib_next[b];
    if (sib_next[b] >= 0) sib_prev[sib_next[b]] = sib_prev[b];
    sib_prev[b] = sib_next[b] = -1;
    parent[b] = -1;
    reg[b] = 0;
  }
  // Evict block b (registered, refcount 0, in the eviction order) for reuse:
  // it and all its cached descendants leave the cache; descendants that no
  // sequence holds move from the eviction order to the free queue's tail in
  // ascending block id.
  void evict(int32_t b) {
    lru_remove(b);
    std::vector<int32_t> desc, stack;
    for (int32_t c = child[b]; c >= 0; c = sib_next[c]) stack.push_back(c);
    while (!stack.empty()) {
      const int32_t c = stack.back();
      stack.pop_back();
      desc.push_back(c);
      for (int32_t d = child[c]; d >= 0; d = sib_next[d]) stack.push_back(d);
    }
    for (int32_t c : desc) {
      child[c] = -1;  // its own children are in desc too
      unregister_one(c);
    }
    child[b] = -1;
    unregister_one(b);
    std::sort(desc.begin(), desc.end());
    for (int32_t c : desc) {
      if (in_lru[c]) {
        lru_remove(c);
        free_q.push_back(c);
      }
    }
  }
  // Precondition: available() > 0.
  int32_t alloc() {
    int32_t b;
    if (!free_q.empty()) {
      b = free_q.front();
      free_q.pop_front();
    } else {
      b = lru_head;
      evict(b);
    }
    ref[b] = 1;
    return b;
  }
  void acquire(int32_t b) {
    if (ref[b] == 0) {
      if (in_lru[b]) {
        lru_remove(b);
      } else if (parked_at[b]) {
        parked_at[b] = 0;  // its entry in parked_list goes stale
        --n_parked;
      }
    }
    ++ref[b];
  }
  void release(int32_t b) {
    if (--ref[b] == 0) {
      parked_at[b] = ++park_tick;
      parked_list.emplace_back(b, park_tick);
      ++n_parked;
    }
  }
  // Register full block j of a sequence (blocks, tokens) if its parent is
  // cached and no cached block holds its key.
  void maybe_register(const std::vector<int32_t>& blocks, const std::vector<int32_t>& tokens,
                      size_t j) {
    if (!caching) return;
    const int32_t b = blocks[j];
    if (reg[b]) return;
    uint64_t pk = kRootKey;
    int32_t pb = -1;
    if (j > 0) {
      pb = blocks[j - 1];
      if (!reg[pb]) return;
      pk = key[pb];
    }
    const uint64_t k = chain_key(pk, tokens.data() + j * B, B);
    if (by_key.count(k)) return;  // the same chain (or a colliding key) is cached already
    by_key.emplace(k, b);
    reg[b] = 1;
    key[b] = k;
    parent[b] = pb;
    child[b] = -1;
    sib_prev[b] = -1;
    sib_next[b] = -1;
    if (pb >= 0) {
      sib_next[b] = child[pb];
      if (child[pb] >= 0) sib_prev[child[pb]] = b;
      child[pb] = b;
    }
    for (int i = 0; i < B; ++i) tok[static_cast<size_t>(b) * B + i] = tokens[j * B + i];
  }
  // Longest run of cached blocks matching tokens from the start, at most
  // max_blocks of them.
  void match(const int32_t* tokens, int64_t max_blocks, std::vector<int32_t>& out) const {
    uint64_t pk = kRootKey;
    int32_t pb = -1;
    for (int64_t j = 0; j < max_blocks; ++j) {
      const int32_t* t = tokens + j * B;
      auto it = by_key.find(chain_key(pk, t, B));
      if (it == by_key.end()) break;
      const int32_t b = it->second;
      if (parent[b] != pb) break;
      bool same = true;
      for (int i = 0; i < B && same; ++i) same = tok[static_cast<size_t>(b) * B + i] == t[i];
      if (!same) break;
      out.push_back(b);
      pk = key[b];
      pb = b;
    }
  }
};

extern "C" {

pa_block_manager* pa_bm_create(int64_t num_blocks, int block_size, int prefix_caching) {
  if (num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0) return nullptr;
  pa_block_manager* bm = new (std::nothrow) pa_block_manager();
  if (!bm) return nullptr;
  try {
    bm->nb = num_blocks;
    bm->B = block_size;
    bm->caching = prefix_caching != 0;
    const size_t n = static_cast<size_t>(num_blocks);
    bm->ref.assign(n, 0);
    bm->written.assign(n, 0);
    bm->parked_at.assign(n, 0);
    bm->reg.assign(n, 0);
    bm->in_lru.assign(n, 0);
    for (int64_t b = 0; b < num_blocks; ++b) bm->free_q.push_back(static_cast<int32_t>(b));
    if (bm->caching) {
      bm->key.assign(n, 0);
      bm->parent.assign(n, -1);
      bm->child.assign(n, -1);
      bm->sib_prev.assign(n, -1);
      bm->sib_next.assign(n, -1);
      bm->tok.assign(n * block_size, 0);
      bm->lru_prev.assign(n, -1);
      bm->lru_next.assign(n, -1);
    }
  } catch (...) {
    delete bm;
    return nullptr;
  }
  return bm;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

int pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens, int n,
                       int64_t* slots, int* num_cached) {
  if (!bm || !tokens || !slots || n < 1) return PA_ERR_INVALID;
  if (bm->seqs.count(seq_id)) return PA_ERR_INVALID;
  const int B = bm->B;
  const int64_t need_blocks = (static_cast<int64_t>(n) + B - 1) / B;
  try {
    std::vector<int32_t> hit;
    if (bm->caching) bm->match(tokens, (static_cast<int64_t>(n) - 1) / B, hit);
    int64_t hit_evictable = 0;
    for (int32_t b : hit) hit_evictable += bm->in_lru[b] ? 1 : 0;
    const int64_t fresh = need_blocks - static_cast<int64_t>(hit.size());
    if (bm->available() - hit_evictable < fresh) return PA_ERR_NO_BLOCKS;
    Seq& s = bm->seqs[seq_id];  // the only step that may throw after this is none
    s.tokens.assign(tokens, tokens + n);
    s.blocks.reserve(need_blocks);
    for (int32_t b : hit) {
      bm->acquire(b);
      s.blocks.push_back(b);
    }
    for (int64_t j = 0; j < fresh; ++j) {
      const int32_t b = bm->alloc();
      bm->written[b] = bm->step;
      s.blocks.push_back(b);
    }
    const int64_t cached = static_cast<int64_t>(hit.size()) * B;
    for (int64_t p = 0; p < n; ++p)
      slots[p] = p < cached ? -1 : static_cast<int64_t>(s.blocks[p / B]) * B + p % B;
    for (size_t j = hit.size(); j < static_cast<size_t>(n / B); ++j)
      bm->maybe_register(s.blocks, s.tokens, j);
    if (num_cached) *num_cached = static_cast<int>(cached);
  } catch (...) {
    return PA_ERR_INVALID;  // host memory exhausted: the manager must be destroyed
  }
  return PA_OK;
}

int pa_bm_append_token(pa_block_manager* bm, int64_t seq_id, int32_t token, int64_t* slot) {
  if (!bm || !slot) return PA_ERR_INVALID;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_INVALID;
  Seq& s = it->second;
  const int B = bm->B;
  const int64_t p = static_cast<int64_t>(s.tokens.size());
  const int64_t j = p / B;
  const bool new_block = p % B == 0;
  const bool cow = !new_block && bm->ref[s.blocks[j]] > 1;
  if (cow && bm->written[s.blocks[j]] == bm->step) return PA_ERR_BM_STEP;
  if ((new_block || cow) && bm->available() < 1) return PA_ERR_NO_BLOCKS;
  try {
    make_room(s.tokens, 1);
    if (new_block) make_room(s.blocks, 1);
    if (cow) {
      make_room(bm->copies, 2);
      make_room(bm->parked_list, 1);
    }
    if (new_block) {
      s.blocks.push_back(bm->alloc());
    } else if (cow) {
      const int32_t old = s.blocks[j];
      const int32_t fresh = bm->alloc();
      bm->copies.push_back(old);
      bm->copies.push_back(fresh);
      bm->release(old);
      s.blocks[j] = fresh;
    }
    s.tokens.push_back(token);
    bm->written[s.blocks[j]] = bm->step;
    *slot = static_cast<int64_t>(s.blocks[j]) * B + p % B;
    if ((p + 1) % B == 0) bm->maybe_register(s.blocks, s.tokens, static_cast<size_t>(j));
  } catch (...) {
    return PA_ERR_INVALID;  // host memory exhausted: the manager must be destroyed
  }
  return PA_OK;
}

int pa_bm_append_tokens(pa_block_manager* bm, const int64_t* seq_ids, const int32_t* tokens,
                        int n, int64_t* slots, int* status) {
  int st = PA_OK, done = 0;
  if (!bm || n < 0 || (n > 0 && (!seq_ids || !tokens || !slots))) {
    st = PA_ERR_INVALID;
  } else {
    for (; done < n; ++done) {
      st = pa_bm_append_token(bm, seq_ids[done], tokens[done], slots + done);
      if (st != PA_OK) break;
    }
  }
  if (status) *status = st;
  return done;
}

int pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id) {
  if (!bm) return PA_ERR_INVALID;
  auto it = bm->seqs.find(parent_id);
  if (it == bm->seqs.end() || bm->seqs.count(child_id)) return PA_ERR_INVALID;
  try {
    Seq c = it->second;
    for (int32_t b : c.blocks) bm->acquire(b);
    bm->seqs.emplace(child_id, std::move(c));
  } catch (...) {
    return PA_ERR_INVALID;  // host memory exhausted: the manager must be destroyed
  }
  return PA_OK;
}

int pa_bm_free_sequence(pa_block_manager* bm, int64_t seq_id) {
  if (!bm) return PA_ERR_INVALID;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_INVALID;
  try {
    const std::vector<int32_t>& blocks = it->second.blocks;
    make_room(bm->parked_list, blocks.size());
    for (size_t k = blocks.size(); k-- > 0;) bm->release(blocks[k]);
    bm->seqs.erase(it);
  } catch (...) {
    return PA_ERR_INVALID;  // host memory exhausted: the manager must be destroyed
  }
  return PA_OK;
}

int64_t pa_bm_num_step_copies(const pa_block_manager* bm) {
  return bm ? static_cast<int64_t>(bm->copies.size() / 2) : -1;
}

int pa_bm_end_step(pa_block_manager* bm, int64_t* pairs, int max_pairs) {
  if (!bm) return PA_ERR_INVALID;
  const int64_t n = static_cast<int64_t>(bm->copies.size() / 2);
  if (n > max_pairs || (n > 0 && !pairs)) return PA_ERR_INVALID;
  for (int64_t i = 0; i < 2 * n; ++i) pairs[i] = bm->copies[i];
  bm->copies.clear();
  for (const auto& e : bm->parked_list) {
    const int32_t b = e.first;
    if (bm->parked_at[b] != e.second) continue;  // re-acquired (and maybe re-parked) since
    bm->parked_at[b] = 0;
    if (bm->reg[b]) bm->lru_push(b); else bm->free_q.push_back(b);
  }
  bm->parked_list.clear();
  bm->n_parked = 0;
  ++bm->step;
  return static_cast<int>(n);
}

int pa_bm_build_tables(const pa_block_manager* bm, const int64_t* seq_ids, int n,
                       int32_t* tables, int max_blocks, int32_t* seq_lens) {
  if (!bm || n < 0 || max_blocks < 0) return PA_ERR_INVALID;
  if (n > 0 && (!seq_ids || !seq_lens || (max_blocks > 0 && !tables))) return PA_ERR_INVALID;
  for (int i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return PA_ERR_INVALID;
    if (it->second.blocks.size() > static_cast<size_t>(max_blocks)) return PA_ERR_INVALID;
  }
  for (int i = 0; i < n; ++i) {
    const Seq& s = bm->seqs.find(seq_ids[i])->second;
    int32_t* row = tables + static_cast<int64_t>(i) * max_blocks;
    for (int j = 0; j < max_blocks; ++j)
      row[j] = j < static_cast<int>(s.blocks.size()) ? s.blocks[j] : -1;
    seq_lens[i] = static_cast<int32_t>(s.tokens.size());
  }
  return PA_OK;
}

int64_t pa_bm_num_free_blocks(const pa_block_manager* bm) {
  return bm ? static_cast<int64_t>(bm->free_q.size()) : -1;
}

int64_t pa_bm_num_parked_blocks(const pa_block_manager* bm) { return bm ? bm->n_parked : -1; }

int64_t pa_bm_num_cached_blocks(const pa_block_manager* bm) {
  return bm ? static_cast<int64_t>(bm->by_key.size()) : -1;
}

int64_t pa_bm_num_evictable_blocks(const pa_block_manager* bm) { return bm ? bm->n_lru : -1; }

int pa_bm_refcount(const pa_block_manager* bm, int64_t block) {
  if (!bm || block < 0 || block >= bm->nb) return -1;
  return bm->ref[block];
}

int64_t pa_bm_seq_len(const pa_block_manager* bm, int64_t seq_id) {
  if (!bm) return -1;
  auto it = bm->seqs.find(seq_id);
  return it == bm->seqs.end() ? -1 : static_cast<int64_t>(it->second.tokens.size());
}

}  // extern "C"
