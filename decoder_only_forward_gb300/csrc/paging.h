// Host side of the paged K/V cache (rml "The decoder", KV cache: pages of
// `page` positions from one arena reserved up front, a sequence taking a page
// when one of its positions first lands in it).  Plain C++ with no CUDA: the
// library keeps the device copy of the table in step with it, and a host-only
// test drives it directly.
#pragma once

#include <stdint.h>

#include <utility>
#include <vector>

namespace dec {

class PageAllocator {
 public:
  // n_seqs sequences of max_seq slots, pages of `page` slots, an arena of n_pages.
  void init(int n_seqs, int max_seq, int page, int n_pages, bool window) {
    max_seq_ = max_seq;
    page_ = page;
    window_ = window;
    pages_per_seq_ = (max_seq + page - 1) / page;
    table_.assign((size_t)n_seqs * pages_per_seq_, -1);
    free_.resize(n_pages);
    for (int i = 0; i < n_pages; ++i) free_[i] = n_pages - 1 - i;   // page 0 on top of the stack
  }

  int pages_per_seq() const { return pages_per_seq_; }
  int free_count() const { return (int)free_.size(); }

  // Physical page of (seq, slot), or -1.
  int32_t page_of(int seq, int slot) const { return table_[(size_t)seq * pages_per_seq_ + slot / page_]; }

  // Takes the pages that writing positions [p0s[i], p0s[i] + n) of sequence
  // seqs[i] needs and does not hold, for every i: all of them, or none (false,
  // the allocator exactly as before).  Under a window the slot of position p is
  // p % max_seq.  `taken` receives the new (table index, page) entries.
  bool reserve(const int32_t* seqs, const int32_t* p0s, int count, int32_t n,
               std::vector<std::pair<int, int>>& taken) {
    taken.clear();
    const int32_t span = n < max_seq_ ? n : max_seq_;   // under a window, n > max_seq repeats slots
    for (int i = 0; i < count; ++i) {
      for (int32_t t = 0; t < span; ++t) {
        const int32_t p = p0s[i] + t;
        const int32_t slot = window_ ? p % max_seq_ : p;
        const int idx = seqs[i] * pages_per_seq_ + slot / page_;
        if (table_[idx] >= 0) continue;
        if (free_.empty()) {
          for (auto it = taken.rbegin(); it != taken.rend(); ++it) {   // undo, last taken first
            free_.push_back(it->second);
            table_[it->first] = -1;
          }
          taken.clear();
          return false;
        }
        table_[idx] = free_.back();
        free_.pop_back();
        taken.emplace_back(idx, table_[idx]);
      }
    }
    return true;
  }

  // Returns every page of sequence seq to the arena.
  void release(int seq) {
    for (int i = 0; i < pages_per_seq_; ++i) {
      int32_t& e = table_[(size_t)seq * pages_per_seq_ + i];
      if (e >= 0) free_.push_back(e);
      e = -1;
    }
  }

 private:
  int max_seq_ = 0, page_ = 1, pages_per_seq_ = 0;
  bool window_ = false;
  std::vector<int32_t> table_;   // [n_seqs][pages_per_seq], -1 = none
  std::vector<int32_t> free_;    // a stack
};

}  // namespace dec
