// Directory of the device page cache that sits in front of host-tier page
// pools (the calls oomb_offload_* in include/oomb.h): which logical page each
// cache slot holds, which KV heads of it have their K/V tiles and their
// gradient tiles loaded, which gradient tiles are modified, when each slot
// was last used, and which gradient tiles of the host pools are known to be
// zero (so that bringing one in is a fill on the device, not a copy).  Pure
// host logic without CUDA, shared by the offload calls and compiled on its
// own by the tests.
// Method: "Out of the Memory Barrier" technical summary, section 2, the fourth
// optimisation ("Async CPU offloading"): only the pages a chunk attends need
// to be on the GPU.
#pragma once

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <string>
#include <utility>
#include <vector>

namespace oomb {

// One tile move of a plan: (page, KV head) between the host pools and cache
// slot `slot`.  A write-back carries the page the slot held before.
// kZeroGrad: the host gradient tiles are zero; the cache tiles are filled
// with zeros instead of being copied.
struct TileMove {
  enum Kind : uint8_t { kFetchKV = 0, kFetchGrad = 1, kWriteGrad = 2, kZeroGrad = 3 };
  int32_t page;
  int32_t slot;
  int32_t head;
  Kind kind;
};

class PageCacheDirectory {
 public:
  PageCacheDirectory(int num_pages, int slots, int heads)
      : num_pages_(num_pages), slots_(slots), heads_(heads),
        all_heads_(heads >= 32 ? 0xFFFFFFFFu : ((1u << heads) - 1u)),
        slot_of_page_(num_pages, -1), page_of_slot_(slots, -1), kv_valid_(slots, 0),
        g_valid_(slots, 0), dirty_(slots, 0), last_use_(slots, 0), need_(num_pages, 0),
        host_zero_(num_pages, 0) {}

  // Plans one acquire: the tiles the chunk's kernels read are (sel[g][i], g)
  // for every KV head g and i < n_sel (sel is [heads][n_sel]) and every head of
  // the own pages [own0, own1).  Resident pages keep their slots; the others
  // take free slots, then the least recently used slots not used by this
  // acquire or the previous one.  Appends to `moves` the gradient write-backs
  // of the reused slots (*n_writeback of them, first), then the fetches of the
  // missing K/V tiles and, with `with_grads`, of the missing gradient tiles
  // (zero fills for those whose host tiles are known to be zero), which are
  // then marked modified.  Returns "" on success, else a message and leaves
  // the directory unchanged.
  std::string plan(const int32_t* sel, int n_sel, int own0, int own1, bool with_grads,
                   std::vector<TileMove>* moves, size_t* n_writeback, int64_t* reused) {
    std::vector<int32_t> pages;
    pages.reserve(static_cast<size_t>(std::max(n_sel, 0)) * heads_ + (own1 - own0));
    auto clear_need = [&] {
      for (int l : pages) need_[l] = 0;
    };
    auto want = [&](int l, uint32_t mask) {
      if (need_[l] == 0) pages.push_back(l);
      need_[l] |= mask;
    };
    if (own0 < 0 || own1 <= own0 || own1 > num_pages_) return "own pages out of range";
    for (int g = 0; g < heads_; ++g)
      for (int i = 0; i < n_sel; ++i) {
        const int l = sel[static_cast<size_t>(g) * n_sel + i];
        if (l < 0 || l >= own0) {
          clear_need();
          return msg("sel[%d][%d] = %d is not a page before the chunk", g, i, l);
        }
        want(l, 1u << g);
      }
    for (int l = own0; l < own1; ++l) want(l, all_heads_);
    if (static_cast<int>(pages.size()) > slots_) {
      clear_need();
      return msg("the chunk needs %zu cache slots, the cache has %d", pages.size(), slots_);
    }
    const uint64_t ep = epoch_ + 1;
    int missing = 0;
    for (int l : pages)
      if (slot_of_page_[l] < 0) ++missing;
    std::vector<std::pair<uint64_t, int>> cand;
    if (missing > 0) {
      for (int s = 0; s < slots_; ++s) {
        if (page_of_slot_[s] < 0) {
          cand.push_back({0, s});
        } else if (last_use_[s] + 1 < ep && need_[page_of_slot_[s]] == 0) {
          cand.push_back({last_use_[s], s});
        }
      }
      if (static_cast<int>(cand.size()) < missing) {
        clear_need();
        return msg("cache of %d slots: %d pages to bring in, %zu slots free or reusable "
                   "(slots of this chunk and the previous one are kept)",
                   slots_, missing, cand.size());
      }
      std::partial_sort(cand.begin(), cand.begin() + missing, cand.end());
    }
    // from here on the plan succeeds
    epoch_ = ep;
    for (int l : pages)
      if (slot_of_page_[l] >= 0) last_use_[slot_of_page_[l]] = ep;
    const size_t first = moves->size();
    int c = 0;
    for (int l : pages) {
      if (slot_of_page_[l] >= 0) continue;
      const int s = cand[c++].second;
      const int old = page_of_slot_[s];
      if (old >= 0) {                            // reuse: modified gradients go home first
        add_writebacks(s, moves);
        slot_of_page_[old] = -1;
        ++*reused;
      }
      page_of_slot_[s] = l;
      slot_of_page_[l] = s;
      kv_valid_[s] = g_valid_[s] = dirty_[s] = 0;
      last_use_[s] = ep;
    }
    *n_writeback = moves->size() - first;
    for (int l : pages) {
      const int s = slot_of_page_[l];
      const uint32_t m = need_[l];
      need_[l] = 0;
      const uint32_t kv_miss = m & ~kv_valid_[s];
      const uint32_t g_miss = with_grads ? (m & ~g_valid_[s]) : 0u;
      for (int g = 0; g < heads_; ++g) {
        if (kv_miss >> g & 1u) moves->push_back({l, s, g, TileMove::kFetchKV});
        if (g_miss >> g & 1u)
          moves->push_back({l, s, g, (host_zero_[l] >> g & 1u) ? TileMove::kZeroGrad
                                                                : TileMove::kFetchGrad});
      }
      kv_valid_[s] |= m;
      if (with_grads) {
        g_valid_[s] |= m;
        dirty_[s] |= m;                          // the backward adds into them in place
      }
    }
    return std::string();
  }

  // Appends the write-backs of every modified gradient tile of the pages
  // [first, first + n) -- of every page when n < 0 -- and marks them clean.
  void collect_writebacks(int first, int n, std::vector<TileMove>* moves) {
    if (n < 0) {
      for (int s = 0; s < slots_; ++s)
        if (page_of_slot_[s] >= 0 && dirty_[s]) add_writebacks(s, moves);
      return;
    }
    for (int l = first; l < first + n; ++l) {
      const int s = slot_of_page_[l];
      if (s >= 0 && dirty_[s]) add_writebacks(s, moves);
    }
  }

  // Appends the write-backs of every modified gradient tile of the listed
  // pages (each in [0, num_pages), checked by the caller; repeats are
  // harmless) and marks them clean.
  void collect_writebacks_of(const int32_t* pages, int n, std::vector<TileMove>* moves) {
    for (int i = 0; i < n; ++i) {
      const int s = slot_of_page_[pages[i]];
      if (s >= 0 && dirty_[s]) add_writebacks(s, moves);
    }
  }

  // The caller has set every gradient tile of the host pools to zero (a new
  // pass): the cached gradient tiles are forgotten without being written
  // back, and until a tile is written back again, bringing it in is a zero
  // fill.  The K/V tiles stay cached.
  void declare_host_grads_zero() {
    for (int l = 0; l < num_pages_; ++l) host_zero_[l] = all_heads_;
    for (int s = 0; s < slots_; ++s) g_valid_[s] = dirty_[s] = 0;
  }

  // Forgets every cached tile (after their write-backs have been collected).
  void drop() {
    for (int s = 0; s < slots_; ++s) {
      if (page_of_slot_[s] >= 0) slot_of_page_[page_of_slot_[s]] = -1;
      page_of_slot_[s] = -1;
      kv_valid_[s] = g_valid_[s] = dirty_[s] = 0;
      last_use_[s] = 0;
    }
  }

  int num_pages() const { return num_pages_; }
  int slots() const { return slots_; }
  int heads() const { return heads_; }
  // Cache slot of every logical page (-1: not resident): the device page table.
  const std::vector<int32_t>& slot_of_page() const { return slot_of_page_; }
  int page_of_slot(int s) const { return page_of_slot_[s]; }
  uint32_t dirty(int s) const { return dirty_[s]; }
  uint32_t host_zero(int l) const { return host_zero_[l]; }

 private:
  void add_writebacks(int s, std::vector<TileMove>* moves) {
    for (int g = 0; g < heads_; ++g)
      if (dirty_[s] >> g & 1u) moves->push_back({page_of_slot_[s], s, g, TileMove::kWriteGrad});
    host_zero_[page_of_slot_[s]] &= ~dirty_[s];   // the host tiles now hold sums
    dirty_[s] = 0;
  }
  template <typename... A>
  static std::string msg(const char* fmt, A... a) {
    char b[256];
    std::snprintf(b, sizeof(b), fmt, a...);
    return std::string(b);
  }

  int num_pages_, slots_, heads_;
  uint32_t all_heads_;
  std::vector<int32_t> slot_of_page_, page_of_slot_;
  std::vector<uint32_t> kv_valid_, g_valid_, dirty_;
  std::vector<uint64_t> last_use_;
  std::vector<uint32_t> need_;
  std::vector<uint32_t> host_zero_;   // per page: heads whose host gradient tiles are zero
  uint64_t epoch_ = 0;
};

}  // namespace oomb
