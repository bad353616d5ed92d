// Host-logic checks of the device page cache's directory (no GPU): slot
// assignment, reuse order, protection of the slots of the previous acquire,
// write-back of modified gradient tiles, per-KV-head tile masks, refusals,
// zero fills of gradient tiles known to be zero on the host.
// Built and run by tests/test_page_cache_directory.py.
#include <cstdio>
#include <cstdlib>
#include <string>
#include <vector>

#include "page_cache_directory.h"

using oomb::PageCacheDirectory;
using oomb::TileMove;

static int g_fail = 0;
#define CHECK(c)                                                   \
  do {                                                             \
    if (!(c)) {                                                    \
      std::printf("FAIL line %d: %s\n", __LINE__, #c);             \
      ++g_fail;                                                    \
    }                                                              \
  } while (0)

static int count(const std::vector<TileMove>& m, TileMove::Kind k) {
  int n = 0;
  for (const auto& x : m) n += x.kind == k;
  return n;
}
static bool has(const std::vector<TileMove>& m, int page, int slot, int head, TileMove::Kind k) {
  for (const auto& x : m)
    if (x.page == page && x.slot == slot && x.head == head && x.kind == k) return true;
  return false;
}

int main() {
  // 1. Fresh cache: 4 slots, 2 KV heads, 10 pages; head 0 selects page 1, head 1
  //    page 2, own pages [8, 10).  Pages get slots in the order they are met.
  {
    PageCacheDirectory d(10, 4, 2);
    const int32_t sel[2] = {1, 2};
    std::vector<TileMove> m;
    size_t nwb = 0;
    int64_t reused = 0;
    CHECK(d.plan(sel, 1, 8, 10, false, &m, &nwb, &reused).empty());
    CHECK(nwb == 0 && reused == 0);
    CHECK(m.size() == 6 && count(m, TileMove::kFetchKV) == 6);
    CHECK(has(m, 1, 0, 0, TileMove::kFetchKV) && !has(m, 1, 0, 1, TileMove::kFetchKV));
    CHECK(has(m, 2, 1, 1, TileMove::kFetchKV) && !has(m, 2, 1, 0, TileMove::kFetchKV));
    CHECK(has(m, 8, 2, 0, TileMove::kFetchKV) && has(m, 8, 2, 1, TileMove::kFetchKV));
    CHECK(has(m, 9, 3, 0, TileMove::kFetchKV) && has(m, 9, 3, 1, TileMove::kFetchKV));
    CHECK(d.slot_of_page()[1] == 0 && d.slot_of_page()[2] == 1 && d.slot_of_page()[0] == -1);
    // 2. Same chunk again with gradients: no K/V moves, gradient tiles for the
    //    same (page, head) pairs, now modified.
    m.clear();
    CHECK(d.plan(sel, 1, 8, 10, true, &m, &nwb, &reused).empty());
    CHECK(m.size() == 6 && count(m, TileMove::kFetchGrad) == 6 && nwb == 0);
    CHECK(d.dirty(0) == 1u && d.dirty(1) == 2u && d.dirty(2) == 3u);
    // 3. A chunk whose pages need new slots while every slot belongs to the
    //    previous acquire: refused, directory unchanged.
    const int32_t sel2[2] = {3, 4};
    m.clear();
    const std::string e = d.plan(sel2, 1, 6, 8, false, &m, &nwb, &reused);
    CHECK(!e.empty() && e.find("reusable") != std::string::npos && m.empty());
    CHECK(d.slot_of_page()[1] == 0 && d.dirty(2) == 3u);
    // 4. Write-backs of a page range, then of everything.
    m.clear();
    d.collect_writebacks(8, 2, &m);
    CHECK(m.size() == 4 && count(m, TileMove::kWriteGrad) == 4 && has(m, 9, 3, 1, TileMove::kWriteGrad));
    CHECK(d.dirty(2) == 0u && d.dirty(3) == 0u && d.dirty(0) == 1u);
    m.clear();
    d.collect_writebacks(8, 2, &m);
    CHECK(m.empty());
    const int32_t list[3] = {2, 5, 2};          // page 2 (slot 1, head 1); 5 not cached
    d.collect_writebacks_of(list, 3, &m);
    CHECK(m.size() == 1 && has(m, 2, 1, 1, TileMove::kWriteGrad) && d.dirty(1) == 0u);
    m.clear();
    d.collect_writebacks(0, -1, &m);
    CHECK(m.size() == 1 && has(m, 1, 0, 0, TileMove::kWriteGrad));
    // 5. drop forgets every slot.
    d.drop();
    for (int l = 0; l < 10; ++l) CHECK(d.slot_of_page()[l] == -1);
  }
  // 6. Reuse order: 6 slots, 1 KV head, no selection; acquires of own pages
  //    A = [0, 2) with gradients, B = [2, 4), C = [4, 6) (free slots), then
  //    D = [6, 8): the two least recently used slots (A's) are reused and
  //    their modified gradient tiles written back first.
  {
    PageCacheDirectory d(10, 6, 1);
    std::vector<TileMove> m;
    size_t nwb = 0;
    int64_t reused = 0;
    CHECK(d.plan(nullptr, 0, 0, 2, true, &m, &nwb, &reused).empty());
    CHECK(d.plan(nullptr, 0, 2, 4, false, &m, &nwb, &reused).empty());
    CHECK(d.plan(nullptr, 0, 4, 6, false, &m, &nwb, &reused).empty());
    CHECK(reused == 0);
    m.clear();
    CHECK(d.plan(nullptr, 0, 6, 8, false, &m, &nwb, &reused).empty());
    CHECK(reused == 2 && nwb == 2);
    CHECK(m[0].kind == TileMove::kWriteGrad && m[1].kind == TileMove::kWriteGrad);
    CHECK(has(m, 0, 0, 0, TileMove::kWriteGrad) && has(m, 1, 1, 0, TileMove::kWriteGrad));
    CHECK(has(m, 6, 0, 0, TileMove::kFetchKV) && has(m, 7, 1, 0, TileMove::kFetchKV));
    CHECK(d.slot_of_page()[0] == -1 && d.slot_of_page()[6] == 0 && d.slot_of_page()[2] == 2);
    // 7. A chunk needing a page resident in an old slot keeps that slot and
    //    moves nothing; the slot is then protected as "previous acquire".
    m.clear();
    CHECK(d.plan(nullptr, 0, 2, 4, false, &m, &nwb, &reused).empty());
    CHECK(m.empty());
    m.clear();
    CHECK(d.plan(nullptr, 0, 8, 10, false, &m, &nwb, &reused).empty());
    // C's slots (4, 5) are the oldest that are not protected: B's were just used
    CHECK(d.slot_of_page()[8] == 4 && d.slot_of_page()[9] == 5 && d.slot_of_page()[2] == 2);
  }
  // 8. Refusals leave no trace: a selected page that is not before the chunk,
  //    and a chunk larger than the cache.
  {
    PageCacheDirectory d(10, 3, 2);
    std::vector<TileMove> m;
    size_t nwb = 0;
    int64_t reused = 0;
    const int32_t bad[2] = {1, 7};
    CHECK(!d.plan(bad, 1, 6, 8, false, &m, &nwb, &reused).empty());
    CHECK(!d.plan(nullptr, 0, 4, 8, false, &m, &nwb, &reused).empty());
    CHECK(m.empty());
    const int32_t ok[2] = {1, 1};
    CHECK(d.plan(ok, 1, 6, 8, false, &m, &nwb, &reused).empty());
    // page 1 for both heads: one slot, both heads' tiles
    CHECK(m.size() == 6 && has(m, 1, 0, 0, TileMove::kFetchKV) && has(m, 1, 0, 1, TileMove::kFetchKV));
  }
  // 9. Host gradients declared zero: gradient tiles come in as zero fills
  //    (K/V tiles stay cached and move nothing) until a write-back puts sums
  //    into the host tile, after which bringing it in is a copy again.
  {
    PageCacheDirectory d(16, 8, 2);
    std::vector<TileMove> m;
    size_t nwb = 0;
    int64_t reused = 0;
    const int32_t sel[2] = {1, 2};               // A: pages 1, 2, 8, 9 -> slots 0..3
    CHECK(d.plan(sel, 1, 8, 10, true, &m, &nwb, &reused).empty());
    CHECK(count(m, TileMove::kFetchGrad) == 6 && count(m, TileMove::kZeroGrad) == 0);
    d.declare_host_grads_zero();
    CHECK(d.dirty(0) == 0u && d.dirty(2) == 0u && d.host_zero(1) == 3u);
    m.clear();                                   // B: the same chunk again
    CHECK(d.plan(sel, 1, 8, 10, true, &m, &nwb, &reused).empty());
    CHECK(m.size() == 6 && count(m, TileMove::kZeroGrad) == 6);   // no K/V moves
    CHECK(has(m, 1, 0, 0, TileMove::kZeroGrad) && has(m, 9, 3, 1, TileMove::kZeroGrad));
    CHECK(d.dirty(0) == 1u && d.dirty(2) == 3u);
    m.clear();                                   // the own pages go home: sums on the host
    d.collect_writebacks(8, 2, &m);
    CHECK(count(m, TileMove::kWriteGrad) == 4);
    CHECK(d.host_zero(8) == 0u && d.host_zero(9) == 0u && d.host_zero(1) == 3u);
    m.clear();                                   // C: pages 3, 4, 5 -> free slots 4, 5, 6
    const int32_t sel_c[2] = {3, 3};
    CHECK(d.plan(sel_c, 1, 4, 6, true, &m, &nwb, &reused).empty());
    CHECK(count(m, TileMove::kZeroGrad) == 6 && count(m, TileMove::kFetchGrad) == 0);
    m.clear();                                   // D: 12 -> free slot 7, 13 -> slot 0 (page 1 out)
    const int32_t sel_d[2] = {3, 2};
    CHECK(d.plan(sel_d, 1, 12, 14, true, &m, &nwb, &reused).empty());
    CHECK(nwb == 1 && has(m, 1, 0, 0, TileMove::kWriteGrad));
    CHECK(d.slot_of_page()[12] == 7 && d.slot_of_page()[13] == 0 && d.slot_of_page()[1] == -1);
    CHECK(has(m, 13, 0, 0, TileMove::kZeroGrad) && has(m, 12, 7, 1, TileMove::kZeroGrad));
    CHECK(d.host_zero(1) == 2u);                 // head 0 of page 1 now holds sums
    m.clear();                                   // E: page 1 back: head 0 copied, head 1 filled
    const int32_t sel_e[2] = {1, 1};
    CHECK(d.plan(sel_e, 1, 14, 16, true, &m, &nwb, &reused).empty());
    const int s1 = d.slot_of_page()[1];
    CHECK(s1 >= 0 && has(m, 1, s1, 0, TileMove::kFetchGrad) && has(m, 1, s1, 1, TileMove::kZeroGrad));
    CHECK(has(m, 8, d.slot_of_page()[8], 0, TileMove::kWriteGrad) == false);   // 8 was clean
  }
  if (g_fail == 0) std::printf("ok\n");
  return g_fail == 0 ? 0 : 1;
}
