// page_pool.h -- host-side page allocator for the paged KV layout.
//
// Paged layout ("Hybrid Sliding Window Attention (Hybrid SWA)", section
// "三、1. vLLM 中的 Hybrid KV Cache 最佳实践": global-attention layers get a
// growing set of pages, sliding-window layers a set that is recycled as tokens
// leave the window; the SWA(w, s) explainer of arXiv 2608.28444, section
// "工程落地与实践" item 1, route B: the paged cache keeps only the last w
// tokens and the sinks). K and V of every layer live in fixed-size pages of
// page_size positions drawn from one pool, [n_pages, Hkv, page_size, d] bf16
// each; a sequence's page table maps logical page lp (positions
// lp * page_size .. + page_size - 1) to a physical page, or -1.
//
// A layer with window w and s sinks needs, to append up to position p and
// attend at p, exactly the logical pages that hold a position of K(p): the
// sink pages and the pages of [p - w + 1, p]. The window only moves forward,
// so a page that no longer holds such a position is never needed again and
// goes back to the pool: a sliding-window layer holds at most
// ceil(s / page_size) + ceil((w - 1) / page_size) + 1 pages, a full-attention
// layer (w beyond every position) holds every page it has touched.
#pragma once

#include <mutex>
#include <vector>

struct swa_page_pool {
  std::mutex mu;
  std::vector<int> free_pages;  // stack of free physical pages
  std::vector<unsigned char> used;
  int n_pages = 0;
};

namespace swa_pages {

// Whether logical page lp holds a position of K(p) (positions < s, or in
// [p - w + 1, p]); only positions <= p count.
inline bool page_needed(long long lp, long long p, int w, int s, int page_size) {
  const long long first = lp * page_size, last = first + page_size - 1;
  if (first > p) return false;
  if (first < s) return true;                       // holds a sink position
  return last >= p - w + 1;                         // meets the window
}

}  // namespace swa_pages
