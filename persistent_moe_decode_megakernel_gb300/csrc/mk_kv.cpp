// mk_kv.cpp -- the paged-KV block allocator of include/mk_kv.h: a FIFO free list of pool
// pages and sequence slots (length + the pages covering it), with the per-step block tables
// built from them.  Host-only bookkeeping; every failing call leaves the pool unchanged.

#include <cstdio>
#include <deque>
#include <vector>

#include "mk.h"
#include "mk_kv.h"

namespace mk {
void set_last_error(int code, const char* text);
}

struct mk_kv_pool {
  int32_t num_pages = 0, page_size = 0, max_slots = 0, max_pages = 0;
  std::deque<int32_t> free_list;          // head: next page to hand out
  std::vector<int32_t> len;               // per slot: length in tokens, -1 when free
  std::vector<std::vector<int32_t>> pages;  // per slot: its pages, in position order
};

namespace {

int kv_fail(int code, const char* fmt, int a = 0, int b = 0) {
  char buf[256];
  std::snprintf(buf, sizeof buf, fmt, a, b);
  mk::set_last_error(code, buf);
  return code;
}

int32_t pages_for(const mk_kv_pool* p, int64_t len) {
  return static_cast<int32_t>((len + p->page_size - 1) / p->page_size);
}

bool live(const mk_kv_pool* p, int32_t slot) {
  return p && slot >= 0 && slot < p->max_slots && p->len[slot] >= 0;
}

}  // namespace

extern "C" {

int mk_kv_pool_create(int32_t num_pages, int32_t page_size, int32_t max_slots, int32_t max_pages_per_seq,
                      const int32_t* order, mk_kv_pool** out) {
  mk::set_last_error(MK_OK, "");
  if (!out) return kv_fail(MK_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (num_pages <= 0 || page_size <= 0 || max_slots <= 0 || max_pages_per_seq <= 0)
    return kv_fail(MK_ERR_INVALID_ARG, "pool sizes must be > 0");
  mk_kv_pool* p = new (std::nothrow) mk_kv_pool();
  if (!p) return kv_fail(MK_ERR_OOM, "pool");
  p->num_pages = num_pages;
  p->page_size = page_size;
  p->max_slots = max_slots;
  p->max_pages = max_pages_per_seq;
  if (order) {
    std::vector<char> seen(static_cast<size_t>(num_pages), 0);
    for (int32_t i = 0; i < num_pages; ++i) {
      const int32_t pg = order[i];
      if (pg < 0 || pg >= num_pages || seen[pg]) {
        delete p;
        return kv_fail(MK_ERR_INVALID_ARG, "order is not a permutation (entry %d = %d)", i, pg);
      }
      seen[pg] = 1;
      p->free_list.push_back(pg);
    }
  } else {
    for (int32_t i = 0; i < num_pages; ++i) p->free_list.push_back(i);
  }
  p->len.assign(static_cast<size_t>(max_slots), -1);
  p->pages.resize(static_cast<size_t>(max_slots));
  *out = p;
  return MK_OK;
}

void mk_kv_pool_destroy(mk_kv_pool* pool) { delete pool; }

int mk_kv_admit(mk_kv_pool* p, int32_t len, int32_t* slot_out) {
  mk::set_last_error(MK_OK, "");
  if (!p || !slot_out) return kv_fail(MK_ERR_INVALID_ARG, "pool or slot_out is NULL");
  if (len < 1) return kv_fail(MK_ERR_INVALID_ARG, "len %d < 1", len);
  const int32_t need = pages_for(p, len);
  if (need > p->max_pages) return kv_fail(MK_ERR_INVALID_ARG, "len %d needs %d pages, above the slot limit", len, need);
  int32_t slot = -1;
  for (int32_t s = 0; s < p->max_slots; ++s)
    if (p->len[s] < 0) { slot = s; break; }
  if (slot < 0) return kv_fail(MK_ERR_OOM, "no free slot (%d in use)", p->max_slots);
  if (static_cast<int64_t>(p->free_list.size()) < need)
    return kv_fail(MK_ERR_OOM, "%d free pages, %d needed", static_cast<int>(p->free_list.size()), need);
  std::vector<int32_t>& pg = p->pages[slot];
  pg.clear();
  for (int32_t i = 0; i < need; ++i) {
    pg.push_back(p->free_list.front());
    p->free_list.pop_front();
  }
  p->len[slot] = len;
  *slot_out = slot;
  return MK_OK;
}

int mk_kv_reserve(mk_kv_pool* p, int32_t slot, int32_t len) {
  mk::set_last_error(MK_OK, "");
  if (!live(p, slot)) return kv_fail(MK_ERR_INVALID_ARG, "slot %d is not live", slot);
  if (len < p->len[slot]) return kv_fail(MK_ERR_INVALID_ARG, "len %d below the slot's %d", len, p->len[slot]);
  const int32_t need = pages_for(p, len);
  if (need > p->max_pages) return kv_fail(MK_ERR_INVALID_ARG, "len %d needs %d pages, above the slot limit", len, need);
  std::vector<int32_t>& pg = p->pages[slot];
  const int32_t more = need - static_cast<int32_t>(pg.size());
  if (more > static_cast<int32_t>(p->free_list.size()))
    return kv_fail(MK_ERR_OOM, "%d free pages, %d needed", static_cast<int>(p->free_list.size()), more);
  for (int32_t i = 0; i < more; ++i) {
    pg.push_back(p->free_list.front());
    p->free_list.pop_front();
  }
  p->len[slot] = len;
  return MK_OK;
}

int mk_kv_evict(mk_kv_pool* p, int32_t slot) {
  mk::set_last_error(MK_OK, "");
  if (!live(p, slot)) return kv_fail(MK_ERR_INVALID_ARG, "slot %d is not live", slot);
  for (int32_t pg : p->pages[slot]) p->free_list.push_back(pg);
  p->pages[slot].clear();
  p->len[slot] = -1;
  return MK_OK;
}

int mk_kv_fill(const mk_kv_pool* p, const int32_t* slots, int32_t n, int32_t* seq_lens_out,
               int32_t* block_tables_out) {
  mk::set_last_error(MK_OK, "");
  if (!p || n < 0 || (n > 0 && (!slots || !seq_lens_out || !block_tables_out)))
    return kv_fail(MK_ERR_INVALID_ARG, "bad arguments");
  std::vector<char> used(static_cast<size_t>(p->max_slots), 0);
  for (int32_t i = 0; i < n; ++i) {
    if (!live(p, slots[i])) return kv_fail(MK_ERR_INVALID_ARG, "slots[%d] = %d is not live", i, slots[i]);
    if (used[slots[i]]) return kv_fail(MK_ERR_INVALID_ARG, "slot %d listed twice", slots[i]);
    used[slots[i]] = 1;
  }
  for (int32_t i = 0; i < n; ++i) {
    const std::vector<int32_t>& pg = p->pages[slots[i]];
    seq_lens_out[i] = p->len[slots[i]];
    int32_t* row = block_tables_out + static_cast<size_t>(i) * p->max_pages;
    for (int32_t k = 0; k < p->max_pages; ++k) row[k] = k < static_cast<int32_t>(pg.size()) ? pg[k] : -1;
  }
  return MK_OK;
}

int32_t mk_kv_free_pages(const mk_kv_pool* p) { return p ? static_cast<int32_t>(p->free_list.size()) : -1; }

int32_t mk_kv_len(const mk_kv_pool* p, int32_t slot) {
  return (p && slot >= 0 && slot < p->max_slots) ? p->len[slot] : -1;
}

}  // extern "C"
