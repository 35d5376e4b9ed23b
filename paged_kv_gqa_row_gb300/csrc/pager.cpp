// Host page allocator for the page pool (lnk_pager_*): a free set handed out
// lowest page first, a reference count per page, rows that share the pages of
// a common prefix (fork), copy on write when a row writes into a shared page,
// and release.  It owns host memory only and exports its table for upload.
//
// Source: "Mistral 7B Instruct v0.3", Entries table (prefill_paged: each
// token attends over its row's pages up to its position -- chunks, shared
// prefixes).  The pages do not say how pages are handed out; this is the
// plainest allocator that lets rows share prefix pages.
#include <cstdint>
#include <new>
#include <set>
#include <unordered_map>
#include <vector>

#include "../../include/lnk.h"

namespace {

constexpr int32_t kPageSize = 64;
constexpr int32_t kUnmapped = -1;

}  // namespace

struct lnk_pager {
  int32_t num_pages = 0, num_rows = 0, pages_per_row = 0;
  std::vector<int32_t> table;     // [num_rows][pages_per_row], -1 = unmapped
  std::vector<int32_t> refcount;  // [num_pages]: table entries mapping the page
  std::set<int32_t> free_pages;   // ordered: the lowest page is handed out first

  int32_t& entry(int32_t row, int32_t lp) { return table[static_cast<size_t>(row) * pages_per_row + lp]; }
  int32_t entry(int32_t row, int32_t lp) const { return table[static_cast<size_t>(row) * pages_per_row + lp]; }

  int32_t take() {
    const int32_t p = *free_pages.begin();
    free_pages.erase(free_pages.begin());
    refcount[p] = 1;
    return p;
  }
  void drop(int32_t p) {
    if (--refcount[p] == 0) free_pages.insert(p);
  }
};

extern "C" {

lnk_status lnk_pager_create(int32_t num_pages, int32_t num_rows, int32_t pages_per_row, lnk_pager** out) {
  if (out == nullptr) return LNK_EINVAL;
  *out = nullptr;
  if (num_pages <= 0 || num_rows <= 0 || pages_per_row <= 0) return LNK_EINVAL;
  if (static_cast<int64_t>(pages_per_row) * kPageSize > INT32_MAX) return LNK_ERANGE;
  lnk_pager* pg = new (std::nothrow) lnk_pager;
  if (pg == nullptr) return LNK_ENOSPACE;
  try {
    pg->num_pages = num_pages;
    pg->num_rows = num_rows;
    pg->pages_per_row = pages_per_row;
    pg->table.assign(static_cast<size_t>(num_rows) * pages_per_row, kUnmapped);
    pg->refcount.assign(num_pages, 0);
    for (int32_t p = 0; p < num_pages; ++p) pg->free_pages.insert(pg->free_pages.end(), p);
  } catch (...) {
    delete pg;
    return LNK_ENOSPACE;
  }
  *out = pg;
  return LNK_OK;
}

void lnk_pager_destroy(lnk_pager* pager) { delete pager; }

lnk_status lnk_pager_reserve(lnk_pager* pg, int32_t row, int32_t length) {
  if (pg == nullptr || row < 0 || row >= pg->num_rows || length < 0) return LNK_EINVAL;
  if (length > pg->pages_per_row * kPageSize) return LNK_ERANGE;
  const int32_t npages = (length + kPageSize - 1) / kPageSize;
  int32_t need = 0;
  for (int32_t lp = 0; lp < npages; ++lp) need += pg->entry(row, lp) == kUnmapped;
  if (need > static_cast<int32_t>(pg->free_pages.size())) return LNK_ENOSPACE;
  for (int32_t lp = 0; lp < npages; ++lp)
    if (pg->entry(row, lp) == kUnmapped) pg->entry(row, lp) = pg->take();
  return LNK_OK;
}

lnk_status lnk_pager_fork(lnk_pager* pg, int32_t src_row, int32_t dst_row, int32_t length) {
  if (pg == nullptr || src_row < 0 || src_row >= pg->num_rows || dst_row < 0 || dst_row >= pg->num_rows ||
      src_row == dst_row || length <= 0)
    return LNK_EINVAL;
  if (length > pg->pages_per_row * kPageSize) return LNK_ERANGE;
  const int32_t npages = (length + kPageSize - 1) / kPageSize;
  for (int32_t lp = 0; lp < pg->pages_per_row; ++lp)
    if (pg->entry(dst_row, lp) != kUnmapped) return LNK_EINVAL;  // the new row must be empty
  for (int32_t lp = 0; lp < npages; ++lp)
    if (pg->entry(src_row, lp) == kUnmapped) return LNK_EINVAL;  // the prefix must be mapped
  for (int32_t lp = 0; lp < npages; ++lp) {
    const int32_t p = pg->entry(src_row, lp);
    pg->entry(dst_row, lp) = p;
    ++pg->refcount[p];
  }
  return LNK_OK;
}

lnk_status lnk_pager_prepare_append(lnk_pager* pg, const int32_t* rows, const int32_t* positions, int32_t n,
                                    int32_t* copy_src, int32_t* copy_dst, int32_t* num_copies) {
  if (pg == nullptr || n < 0 || num_copies == nullptr) return LNK_EINVAL;
  *num_copies = 0;
  if (n == 0) return LNK_OK;
  if (rows == nullptr || positions == nullptr || copy_src == nullptr || copy_dst == nullptr) return LNK_EINVAL;
  // Pass 1: check the tokens and count the fresh pages the batch needs, so that
  // a batch that does not fit changes nothing.  A logical page is handled by
  // the first token of the batch that writes into it.
  std::unordered_map<int64_t, char> seen;
  std::unordered_map<int32_t, int32_t> moved;  // writers already moved off a shared page
  int32_t need = 0;
  for (int32_t t = 0; t < n; ++t) {
    const int32_t r = rows[t], pos = positions[t];
    if (pos < 0) continue;  // inactive token
    if (r < 0 || r >= pg->num_rows) return LNK_EINVAL;
    if (pos >= pg->pages_per_row * kPageSize) return LNK_ERANGE;
    const int32_t lp = pos / kPageSize;
    const int64_t key = static_cast<int64_t>(r) * pg->pages_per_row + lp;
    if (!seen.emplace(key, 1).second) continue;
    const int32_t p = pg->entry(r, lp);
    if (p == kUnmapped) {
      ++need;
    } else if (pg->refcount[p] - moved[p] > 1) {
      ++need;
      ++moved[p];
    }
  }
  if (need > static_cast<int32_t>(pg->free_pages.size())) return LNK_ENOSPACE;
  // Pass 2: map fresh pages and move writers off shared pages.
  seen.clear();
  int32_t nc = 0;
  for (int32_t t = 0; t < n; ++t) {
    const int32_t r = rows[t], pos = positions[t];
    if (pos < 0) continue;
    const int32_t lp = pos / kPageSize;
    const int64_t key = static_cast<int64_t>(r) * pg->pages_per_row + lp;
    if (!seen.emplace(key, 1).second) continue;
    int32_t& e = pg->entry(r, lp);
    if (e == kUnmapped) {
      e = pg->take();
    } else if (pg->refcount[e] > 1) {
      const int32_t old = e;
      e = pg->take();
      --pg->refcount[old];  // still mapped by another row, so it stays allocated
      copy_src[nc] = old;
      copy_dst[nc] = e;
      ++nc;
    }
  }
  *num_copies = nc;
  return LNK_OK;
}

lnk_status lnk_pager_release(lnk_pager* pg, int32_t row) {
  if (pg == nullptr || row < 0 || row >= pg->num_rows) return LNK_EINVAL;
  for (int32_t lp = 0; lp < pg->pages_per_row; ++lp) {
    int32_t& e = pg->entry(row, lp);
    if (e != kUnmapped) {
      pg->drop(e);
      e = kUnmapped;
    }
  }
  return LNK_OK;
}

lnk_status lnk_pager_table(const lnk_pager* pg, int32_t* table) {
  if (pg == nullptr || table == nullptr) return LNK_EINVAL;
  for (size_t i = 0; i < pg->table.size(); ++i) table[i] = pg->table[i];
  return LNK_OK;
}

int32_t lnk_pager_free_pages(const lnk_pager* pg) {
  return pg == nullptr ? -1 : static_cast<int32_t>(pg->free_pages.size());
}

int32_t lnk_pager_refcount(const lnk_pager* pg, int32_t page) {
  if (pg == nullptr || page < 0 || page >= pg->num_pages) return -1;
  return pg->refcount[page];
}

}  // extern "C"
