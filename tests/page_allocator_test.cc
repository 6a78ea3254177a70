// Host-only checks of the paged cache's page allocator (csrc/paging.h): taking
// pages as positions first land in them, all-or-none reservation that leaves
// the allocator exactly as it was on failure, release, and window wrap.
// Built and run by tests/test_page_allocator.py; exits non-zero on a failure.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "paging.h"

#define CHECK(c)                                                   \
  do {                                                             \
    if (!(c)) {                                                    \
      std::fprintf(stderr, "%s:%d: %s\n", __FILE__, __LINE__, #c); \
      return 1;                                                    \
    }                                                              \
  } while (0)

using dec::PageAllocator;

static int grow_and_run_out() {
  PageAllocator a;
  a.init(/*n_seqs=*/3, /*max_seq=*/32, /*page=*/16, /*n_pages=*/5, /*window=*/false);
  std::vector<std::pair<int, int>> t;
  CHECK(a.pages_per_seq() == 2 && a.free_count() == 5);
  int32_t s0 = 0, p0 = 0;
  CHECK(a.reserve(&s0, &p0, 1, 6, t) && t.size() == 1 && a.page_of(0, 5) == 0);   // page 0 first
  int32_t s1 = 1;
  CHECK(a.reserve(&s1, &p0, 1, 20, t) && t.size() == 2 && a.free_count() == 2);
  // Positions inside held pages take nothing.
  int32_t p10 = 10;
  CHECK(a.reserve(&s1, &p10, 1, 5, t) && t.empty() && a.free_count() == 2);
  // A batch: sequence 0 crosses into its second page, sequence 2 starts.
  int32_t seqs[2] = {0, 2}, pos[2] = {16, 0};
  CHECK(a.reserve(seqs, pos, 2, 1, t) && t.size() == 2 && a.free_count() == 0);
  // Out of pages: nothing changes, not even the order of later allocations.
  int32_t s2 = 2, p16 = 16;
  CHECK(!a.reserve(&s2, &p16, 1, 1, t) && t.empty() && a.free_count() == 0 && a.page_of(2, 16) == -1);
  // Release returns a sequence's pages; the next request gets them.
  a.release(1);
  CHECK(a.free_count() == 2 && a.page_of(1, 0) == -1);
  CHECK(a.reserve(&s2, &p16, 1, 1, t) && t.size() == 1 && a.free_count() == 1);
  return 0;
}

static int all_or_none_across_a_batch() {
  PageAllocator a;
  a.init(2, 64, 16, 3, false);
  std::vector<std::pair<int, int>> t;
  int32_t seqs[2] = {0, 1}, pos[2] = {0, 0};
  // Two sequences of 32 positions need 4 pages: none is taken.
  CHECK(!a.reserve(seqs, pos, 2, 32, t) && a.free_count() == 3);
  CHECK(a.page_of(0, 0) == -1 && a.page_of(0, 16) == -1 && a.page_of(1, 0) == -1);
  // The stack order survives the undo: the first page handed out is still page 0.
  int32_t s = 1, p = 40;
  CHECK(a.reserve(&s, &p, 1, 1, t) && a.page_of(1, 40) == 0);
  return 0;
}

static int window_wrap_reuses_pages() {
  PageAllocator a;
  a.init(1, 32, 16, 2, /*window=*/true);
  std::vector<std::pair<int, int>> t;
  int32_t s = 0, p = 0;
  CHECK(a.reserve(&s, &p, 1, 40, t) && t.size() == 2 && a.free_count() == 0);   // 40 > 32: every slot
  int32_t p40 = 40;
  CHECK(a.reserve(&s, &p40, 1, 30, t) && t.empty());                            // wraps into held pages
  CHECK(a.page_of(0, 40 % 32) == a.page_of(0, 8));
  return 0;
}

int main() {
  if (grow_and_run_out() || all_or_none_across_a_batch() || window_wrap_reuses_pages()) return 1;
  std::printf("page allocator ok\n");
  return 0;
}
