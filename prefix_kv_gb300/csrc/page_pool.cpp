// Host-side page pool for the paged prefix cache.
//
// SenseNova-U1 / Prism-Infer notes, the section on prefix KV reuse, give the
// page rules this pool keeps:
//   1. a full page joins the hit index only after its K/V has been computed
//      (bca_pool_publish is called by the owner after the write completed);
//   2. a shared tail page copies only the common prefix rows into a page of its
//      own and does not inherit the old entry's hash (a page from
//      bca_pool_alloc, filled by bca_pool_copy_rows, is unpublished);
//   3. idle cached pages may be lent to any allocation, but a page an active
//      request references is never reclaimed; when several entries share a
//      page, reclaimable capacity counts each physical page once.
// The pool only tracks page ids; the K/V data live in the caller's cache
// tensors ([layer][head][num_pages * 128][128]).  Hashes are opaque 64-bit
// keys chosen by the caller (for example chained hashes of each page's
// conditioning tokens).  All calls are thread-safe.
#include <cstdint>
#include <iterator>
#include <list>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "bca.h"

struct bca_page_pool {
  struct Page {
    int32_t refs = 0;
    bool published = false;
    uint64_t hash = 0;
    std::list<int32_t>::iterator lru;   // valid while idle and published
  };
  std::mutex mu;
  std::vector<Page> pages;
  std::vector<int32_t> free_list;              // never published, no references
  std::list<int32_t> idle;                     // published, no references; front = oldest
  std::unordered_map<uint64_t, int32_t> index; // hash -> published page

  explicit bca_page_pool(int32_t n) : pages(n) {
    free_list.reserve(n);
    for (int32_t i = n - 1; i >= 0; --i) free_list.push_back(i);
  }

  // Forget an idle cached page so it can be handed out again (rule 3).
  void evict(int32_t p) {
    Page& pg = pages[p];
    idle.erase(pg.lru);
    index.erase(pg.hash);
    pg.published = false;
    pg.hash = 0;
  }
};

extern "C" {

bca_page_pool* bca_pool_create(int32_t num_pages) {
  if (num_pages <= 0) return nullptr;
  return new bca_page_pool(num_pages);
}

void bca_pool_destroy(bca_page_pool* pool) { delete pool; }

bca_status bca_pool_alloc(bca_page_pool* pool, int32_t n, int32_t* pages_out) {
  if (pool == nullptr || n < 0 || (n > 0 && pages_out == nullptr)) return BCA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(pool->mu);
  if (static_cast<size_t>(n) > pool->free_list.size() + pool->idle.size()) return BCA_ERR_CAPACITY;
  for (int32_t i = 0; i < n; ++i) {
    int32_t p;
    if (!pool->free_list.empty()) {
      p = pool->free_list.back();
      pool->free_list.pop_back();
    } else {                                   // lend the least recently used idle page
      p = pool->idle.front();
      pool->evict(p);
    }
    pool->pages[p].refs = 1;
    pages_out[i] = p;
  }
  return BCA_OK;
}

int32_t bca_pool_match(bca_page_pool* pool, const uint64_t* hashes, int32_t n,
                       int32_t* pages_out) {
  if (pool == nullptr || n <= 0 || hashes == nullptr || pages_out == nullptr) return 0;
  std::lock_guard<std::mutex> lock(pool->mu);
  int32_t hits = 0;
  for (; hits < n; ++hits) {
    const auto it = pool->index.find(hashes[hits]);
    if (it == pool->index.end()) break;
    bca_page_pool::Page& pg = pool->pages[it->second];
    if (pg.refs == 0) pool->idle.erase(pg.lru);
    ++pg.refs;
    pages_out[hits] = it->second;
  }
  return hits;
}

bca_status bca_pool_publish(bca_page_pool* pool, int32_t page, uint64_t hash) {
  if (pool == nullptr || page < 0 || page >= static_cast<int32_t>(pool->pages.size()))
    return BCA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(pool->mu);
  bca_page_pool::Page& pg = pool->pages[page];
  if (pg.refs == 0 || pg.published) return BCA_ERR_INVALID_ARG;   // only the owner, once
  if (pool->index.count(hash)) return BCA_ERR_INVALID_ARG;         // one page per hash
  pg.published = true;
  pg.hash = hash;
  pool->index.emplace(hash, page);
  return BCA_OK;
}

bca_status bca_pool_release(bca_page_pool* pool, const int32_t* pages, int32_t n) {
  if (pool == nullptr || n < 0 || (n > 0 && pages == nullptr)) return BCA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(pool->mu);
  for (int32_t i = 0; i < n; ++i) {           // check first: a failing call changes nothing
    const int32_t p = pages[i];
    if (p < 0 || p >= static_cast<int32_t>(pool->pages.size())) return BCA_ERR_INVALID_ARG;
  }
  std::unordered_map<int32_t, int32_t> drops;
  for (int32_t i = 0; i < n; ++i) ++drops[pages[i]];
  for (const auto& d : drops)
    if (pool->pages[d.first].refs < d.second) return BCA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t p = pages[i];
    bca_page_pool::Page& pg = pool->pages[p];
    if (--pg.refs > 0) continue;
    if (pg.published) {
      pool->idle.push_back(p);                 // cached for reuse, newest at the back
      pg.lru = std::prev(pool->idle.end());
    } else {
      pool->free_list.push_back(p);
    }
  }
  return BCA_OK;
}

void bca_pool_stats(bca_page_pool* pool, int32_t* free_pages, int32_t* idle_cached,
                    int32_t* in_use) {
  if (pool == nullptr) return;
  std::lock_guard<std::mutex> lock(pool->mu);
  const int32_t f = static_cast<int32_t>(pool->free_list.size());
  const int32_t c = static_cast<int32_t>(pool->idle.size());
  if (free_pages) *free_pages = f;
  if (idle_cached) *idle_cached = c;
  if (in_use) *in_use = static_cast<int32_t>(pool->pages.size()) - f - c;
}

int32_t bca_pool_refs(bca_page_pool* pool, int32_t page) {
  if (pool == nullptr || page < 0 || page >= static_cast<int32_t>(pool->pages.size())) return -1;
  std::lock_guard<std::mutex> lock(pool->mu);
  return pool->pages[page].refs;
}

}  // extern "C"
