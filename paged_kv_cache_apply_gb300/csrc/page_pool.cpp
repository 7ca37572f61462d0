// Paged-pool bookkeeping on the host: a bitmask page allocator with per-page reference counts
// and LRU eviction, and a radix cache of complete token pages.
//
// AstrAI inference guide, "KVCache System": PagePool orchestrates KVStorage, ReqToTokenPool,
// a bitmask-based page allocator with ref-counts and LRU, and RadixCache, which indexes complete
// token pages as parent-linked edges, compares each page's exact token tuple while walking from
// the root (so a page is reused only under the same parent prefix; hashes never decide a
// match), admits only fully materialised pages, and lets a later request resume prefill right
// after its longest complete-page hit. AstrAI internals, "Cache Architecture": prefix sharing
// exists when page_size > 1; partial pages stay private to their request.
//
// Page p owns token slots [p * page_size, (p + 1) * page_size) of the flat KV buffers.
// A page is in exactly one of three states: free (its bit is set), referenced (held by at
// least one request, ref > 0), or cached with no reference (in the radix, ref = 0; evictable
// once it is a leaf). Every call takes the pool's mutex.
#include <stdint.h>

#include <mutex>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "../../include/astr.h"
#include "launch.h"

namespace {

struct Node {
  int32_t parent = -1;          // node index; -1: a child of the root
  std::vector<int32_t> toks;    // the page's exact token tuple
  int32_t page = -1;            // physical page
  uint64_t hash = 0;            // FNV-1a over (parent hash, tokens): introspection only
  uint64_t last_use = 0;        // logical clock of the last match or record through it
  int32_t n_children = 0;
  bool alive = false;
};

uint64_t fnv1a(uint64_t h, const int32_t *t, int32_t n) {
  const unsigned char *p = reinterpret_cast<const unsigned char *>(t);
  for (int64_t i = 0; i < (int64_t)n * 4; ++i) h = (h ^ p[i]) * 1099511628211ull;
  return h;
}

constexpr uint64_t kFnvBasis = 14695981039346656037ull;

}  // namespace

struct astr_page_pool {
  int32_t n_pages = 0, page_size = 0;
  std::vector<uint64_t> free_bits;  // bit p of word p / 64: page p is free
  int32_t n_free = 0;
  std::vector<int32_t> ref;         // references held on each page
  std::vector<int32_t> node_of;     // radix node holding each page, or -1
  std::vector<Node> nodes;
  std::vector<int32_t> dead_nodes;  // reusable node indices
  // (parent, tuple hash) -> nodes with that key; equality is always by the exact tuple
  std::unordered_map<uint64_t, std::vector<int32_t>> children;
  std::set<std::pair<uint64_t, int32_t>> evictable;  // (last_use, page) of unreferenced leaves
  uint64_t clock = 0;
  std::mutex mu;

  bool radix_on() const { return page_size > 1; }

  static uint64_t child_key(int32_t parent, uint64_t tuple_hash) {
    return (tuple_hash ^ ((uint64_t)(uint32_t)(parent + 1) * 0x9E3779B97F4A7C15ull));
  }

  // the child of `parent` whose tuple equals t[0..page_size), or -1
  int32_t find_child(int32_t parent, const int32_t *t) const {
    auto it = children.find(child_key(parent, fnv1a(kFnvBasis, t, page_size)));
    if (it == children.end()) return -1;
    for (int32_t c : it->second) {
      const Node &nd = nodes[c];
      bool same = nd.parent == parent;
      for (int32_t k = 0; same && k < page_size; ++k) same = nd.toks[k] == t[k];
      if (same) return c;
    }
    return -1;
  }

  bool is_free(int32_t p) const { return (free_bits[p >> 6] >> (p & 63)) & 1u; }
  void set_free(int32_t p) { free_bits[p >> 6] |= uint64_t(1) << (p & 63); ++n_free; }
  void take(int32_t p) { free_bits[p >> 6] &= ~(uint64_t(1) << (p & 63)); --n_free; }

  void mark_if_evictable(int32_t n) {
    const Node &nd = nodes[n];
    if (nd.alive && nd.n_children == 0 && ref[nd.page] == 0) evictable.insert({nd.last_use, nd.page});
  }

  void unmark(int32_t n) { evictable.erase({nodes[n].last_use, nodes[n].page}); }

  // drop the least recently used unreferenced leaf; its parent may become one
  bool evict_one() {
    if (evictable.empty()) return false;
    const int32_t page = evictable.begin()->second;
    evictable.erase(evictable.begin());
    const int32_t n = node_of[page];
    Node &nd = nodes[n];
    auto &bucket = children[child_key(nd.parent, fnv1a(kFnvBasis, nd.toks.data(), page_size))];
    for (size_t i = 0; i < bucket.size(); ++i)
      if (bucket[i] == n) {
        bucket[i] = bucket.back();
        bucket.pop_back();
        break;
      }
    if (nd.parent >= 0) {
      --nodes[nd.parent].n_children;
      mark_if_evictable(nd.parent);
    }
    nd.alive = false;
    node_of[page] = -1;
    dead_nodes.push_back(n);
    set_free(page);
    return true;
  }
};

namespace astr {
void set_last_error_message(const char *msg);
}

namespace {

astr_status pool_fail(astr_status st, const char *msg) {
  astr::set_last_error_message(msg);
  return st;
}

astr_status pool_ok() {
  astr::set_last_error_message("");
  return ASTR_OK;
}

}  // namespace

extern "C" {

astr_status astr_pool_create(int32_t n_pages, int32_t page_size, astr_page_pool **out) {
  if (!out) return pool_fail(ASTR_ERR_INVALID, "astr_pool_create: out is NULL");
  *out = nullptr;
  if (n_pages < 1 || page_size < 1 || (int64_t)n_pages * page_size > INT32_MAX)
    return pool_fail(ASTR_ERR_INVALID, "astr_pool_create: need n_pages >= 1, page_size >= 1 and "
                                       "n_pages * page_size < 2^31 slots");
  auto *p = new astr_page_pool();
  p->n_pages = n_pages;
  p->page_size = page_size;
  p->free_bits.assign((n_pages + 63) / 64, 0);
  for (int32_t i = 0; i < n_pages; ++i) p->set_free(i);
  p->ref.assign(n_pages, 0);
  p->node_of.assign(n_pages, -1);
  *out = p;
  return pool_ok();
}

astr_status astr_pool_destroy(astr_page_pool *pool) {
  delete pool;
  return pool_ok();
}

astr_status astr_pool_match(astr_page_pool *pool, const int32_t *tokens, int64_t n_tokens,
                            int32_t max_pages, int32_t *pages, int32_t *n_matched) {
  if (!pool || !n_matched || (n_tokens > 0 && !tokens) || max_pages < 0 || (max_pages > 0 && !pages) ||
      n_tokens < 0)
    return pool_fail(ASTR_ERR_INVALID, "astr_pool_match: bad argument");
  std::lock_guard<std::mutex> lock(pool->mu);
  *n_matched = 0;
  if (!pool->radix_on()) return pool_ok();
  const int64_t whole = n_tokens / pool->page_size;
  int32_t parent = -1, m = 0;
  while (m < whole && m < max_pages) {
    const int32_t c = pool->find_child(parent, tokens + (int64_t)m * pool->page_size);
    if (c < 0) break;
    Node &nd = pool->nodes[c];
    if (pool->ref[nd.page]++ == 0) pool->unmark(c);
    nd.last_use = ++pool->clock;
    pages[m++] = nd.page;
    parent = c;
  }
  *n_matched = m;
  return pool_ok();
}

astr_status astr_pool_alloc(astr_page_pool *pool, int32_t n, int32_t *pages) {
  if (!pool || n < 0 || (n > 0 && !pages)) return pool_fail(ASTR_ERR_INVALID, "astr_pool_alloc: bad argument");
  std::lock_guard<std::mutex> lock(pool->mu);
  while (pool->n_free < n && pool->evict_one()) {
  }
  if (pool->n_free < n)
    return pool_fail(ASTR_ERR_NO_SPACE, "astr_pool_alloc: not enough free or evictable pages");
  int32_t got = 0;
  for (size_t w = 0; w < pool->free_bits.size() && got < n; ++w) {
    while (pool->free_bits[w] && got < n) {
      const int32_t p = (int32_t)(w * 64 + __builtin_ctzll(pool->free_bits[w]));
      pool->take(p);
      pool->ref[p] = 1;
      pages[got++] = p;
    }
  }
  return pool_ok();
}

astr_status astr_pool_record(astr_page_pool *pool, const int32_t *tokens, int64_t n_materialized,
                             const int32_t *pages, int32_t n_pages) {
  if (!pool || n_materialized < 0 || (n_materialized > 0 && !tokens) || n_pages < 0 || (n_pages > 0 && !pages))
    return pool_fail(ASTR_ERR_INVALID, "astr_pool_record: bad argument");
  std::lock_guard<std::mutex> lock(pool->mu);
  if (!pool->radix_on()) return pool_ok();
  const int64_t whole = n_materialized / pool->page_size;
  if (whole > n_pages) return pool_fail(ASTR_ERR_INVALID, "astr_pool_record: fewer pages than complete pages");
  for (int64_t i = 0; i < whole; ++i)
    if (pages[i] < 0 || pages[i] >= pool->n_pages || pool->ref[pages[i]] < 1)
      return pool_fail(ASTR_ERR_INVALID, "astr_pool_record: a page the caller does not hold");
  // check the whole path first, so that a rejected call changes nothing
  {
    int32_t parent = -1;
    for (int64_t i = 0; i < whole; ++i) {
      const int32_t c = pool->find_child(parent, tokens + i * pool->page_size);
      if (c >= 0) {
        parent = c;
        continue;
      }
      std::set<int32_t> seen;
      for (int64_t k = i; k < whole; ++k)
        if (pool->node_of[pages[k]] >= 0 || !seen.insert(pages[k]).second)
          return pool_fail(ASTR_ERR_INVALID,
                           "astr_pool_record: a page is already cached, or given twice, on this path");
      break;
    }
  }
  int32_t parent = -1;
  for (int64_t i = 0; i < whole; ++i) {
    const int32_t *t = tokens + i * pool->page_size;
    int32_t c = pool->find_child(parent, t);
    if (c < 0) {  // a new edge; a duplicate tuple keeps the page already cached
      if (!pool->dead_nodes.empty()) {
        c = pool->dead_nodes.back();
        pool->dead_nodes.pop_back();
      } else {
        c = (int32_t)pool->nodes.size();
        pool->nodes.emplace_back();
      }
      Node &nd = pool->nodes[c];
      nd.parent = parent;
      nd.toks.assign(t, t + pool->page_size);
      nd.page = pages[i];
      nd.hash = fnv1a(parent >= 0 ? pool->nodes[parent].hash : kFnvBasis, t, pool->page_size);
      nd.n_children = 0;
      nd.alive = true;
      pool->node_of[nd.page] = c;
      pool->children[astr_page_pool::child_key(parent, fnv1a(kFnvBasis, t, pool->page_size))].push_back(c);
      if (parent >= 0) {
        pool->unmark(parent);  // no longer a leaf
        ++pool->nodes[parent].n_children;
      }
    }
    Node &nd = pool->nodes[c];
    const bool was = nd.n_children == 0 && pool->ref[nd.page] == 0;
    if (was) pool->unmark(c);
    nd.last_use = ++pool->clock;
    pool->mark_if_evictable(c);
    parent = c;
  }
  return pool_ok();
}

astr_status astr_pool_release(astr_page_pool *pool, const int32_t *pages, int32_t n) {
  if (!pool || n < 0 || (n > 0 && !pages)) return pool_fail(ASTR_ERR_INVALID, "astr_pool_release: bad argument");
  std::lock_guard<std::mutex> lock(pool->mu);
  {  // validate first (counting repeats), so that a rejected call changes nothing
    std::unordered_map<int32_t, int32_t> want;
    for (int32_t i = 0; i < n; ++i) {
      if (pages[i] < 0 || pages[i] >= pool->n_pages)
        return pool_fail(ASTR_ERR_INVALID, "astr_pool_release: page out of range");
      if (++want[pages[i]] > pool->ref[pages[i]])
        return pool_fail(ASTR_ERR_INVALID, "astr_pool_release: releases a reference not held");
    }
  }
  for (int32_t i = 0; i < n; ++i) {
    const int32_t p = pages[i];
    if (--pool->ref[p] > 0) continue;
    const int32_t c = pool->node_of[p];
    if (c >= 0) pool->mark_if_evictable(c);
    else pool->set_free(p);
  }
  return pool_ok();
}

astr_status astr_pool_stats(astr_page_pool *pool, int32_t *free_pages, int32_t *cached_pages,
                            int32_t *evictable_pages) {
  if (!pool || !free_pages || !cached_pages || !evictable_pages)
    return pool_fail(ASTR_ERR_INVALID, "astr_pool_stats: NULL argument");
  std::lock_guard<std::mutex> lock(pool->mu);
  *free_pages = pool->n_free;
  int32_t cached = 0;
  for (int32_t c : pool->node_of) cached += c >= 0;
  *cached_pages = cached;
  *evictable_pages = (int32_t)pool->evictable.size();
  return pool_ok();
}

astr_status astr_pool_page_info(astr_page_pool *pool, int32_t page, int32_t *refs, int32_t *cached,
                                uint64_t *hash) {
  if (!pool || !refs || !cached || !hash || page < 0 || page >= pool->n_pages)
    return pool_fail(ASTR_ERR_INVALID, "astr_pool_page_info: bad argument");
  std::lock_guard<std::mutex> lock(pool->mu);
  *refs = pool->ref[page];
  const int32_t c = pool->node_of[page];
  *cached = c >= 0;
  *hash = c >= 0 ? pool->nodes[c].hash : 0;
  return pool_ok();
}

astr_status astr_pool_slots(astr_page_pool *pool, const int32_t *pages, int32_t n_pages,
                            int64_t n_tokens, int32_t *slots) {
  if (!pool || n_tokens < 0 || n_pages < 0 || (n_tokens > 0 && (!pages || !slots)))
    return pool_fail(ASTR_ERR_INVALID, "astr_pool_slots: bad argument");
  const int64_t ps = pool->page_size;
  if (n_tokens > (int64_t)n_pages * ps)
    return pool_fail(ASTR_ERR_INVALID, "astr_pool_slots: the pages cannot hold n_tokens tokens");
  // the page table is not read: the pool's lock is not needed
  for (int64_t j = 0; j < n_tokens; ++j) {
    const int32_t pg = pages[j / ps];
    if (pg < 0 || pg >= pool->n_pages)
      return pool_fail(ASTR_ERR_INVALID, "astr_pool_slots: a page number is outside the pool");
    slots[j] = (int32_t)((int64_t)pg * ps + j % ps);
  }
  return pool_ok();
}

}  // extern "C"
