// Host planner: balanced split of the KV axis over a persistent grid.
//
// The decode work of a batch is the sequence of units (request, kv head) in
// request-major order, unit (i, h) costing the np_i pages of request i.
// Laid end to end, the units form one stream of total T = num_kv_heads *
// sum_i np_i pages.  The planner fixes the grid size N (at most the number of
// CTAs resident at once, and no more than T / min_pages_per_cta) and gives CTA
// c the stream positions [c*q, (c+1)*q) with q = ceil(T / N).  A unit that a
// cut falls inside is split at that page boundary; each piece becomes a
// segment that writes a partial (o, lse) state into its own slot, and a merge
// unit records which slots to combine.  Every CTA therefore streams the same
// number of pages (+-1) whatever the mix of context lengths, which is the
// load-balancing duty the page "FlashDecoding + FlashInfer" assigns to
// FlashInfer's plan step ("What FlashInfer is", item 3), and a long request
// is spread over as many CTAs as its length needs, which is the split-KV
// idea of section "FlashDecoding - the split-KV trick".
//
// Requests with no pages still get one (empty) segment per kv head so that
// their output (o = 0, lse = -inf) is written.
#include "planner.h"

#include <algorithm>

namespace fadecode {

int build_work_list(const int32_t* indptr, const int32_t* last_page_len,
                    int batch, int num_kv_heads, int page_size, int max_ctas,
                    int min_pages_per_cta, WorkList* out) {
  if (!indptr || !out || batch < 0 || num_kv_heads <= 0 || page_size <= 0 ||
      max_ctas <= 0)
    return -1;
  if (batch > 0 && !last_page_len) return -1;
  if (indptr[0] != 0) return -1;
  int64_t total_tokens = 0;
  for (int i = 0; i < batch; ++i) {
    const int64_t np = (int64_t)indptr[i + 1] - indptr[i];
    if (np < 0) return -1;
    if (np > 0) {
      if (last_page_len[i] < 1 || last_page_len[i] > page_size) return -1;
      total_tokens += (np - 1) * page_size + last_page_len[i];
    }
  }
  const int64_t total_pages = indptr[batch];
  const int64_t T = total_pages * num_kv_heads;
  if (min_pages_per_cta < 1) min_pages_per_cta = 1;

  int64_t n = max_ctas;
  if (T > 0) n = std::min<int64_t>(n, (T + min_pages_per_cta - 1) / min_pages_per_cta);
  if (n < 1) n = 1;
  const int64_t quota = T > 0 ? (T + n - 1) / n : 1;
  if (T > 0) n = (T + quota - 1) / quota;  // no CTA left without pages
  const int num_ctas = (int)n;

  WorkList wl;
  wl.num_ctas = num_ctas;
  wl.total_pages = total_pages;
  wl.total_tokens = total_tokens;
  std::vector<int32_t> seg_cta;  // owning CTA of each segment (non-decreasing)
  wl.segments.reserve((size_t)batch * num_kv_heads + num_ctas);
  seg_cta.reserve(wl.segments.capacity());

  int64_t pos = 0;
  int slots = 0;
  for (int i = 0; i < batch; ++i) {
    const int32_t pb = indptr[i], pe = indptr[i + 1];
    const int64_t np = (int64_t)pe - pb;
    for (int h = 0; h < num_kv_heads; ++h) {
      if (np == 0) {
        const int64_t cta = std::min<int64_t>(pos / quota, num_ctas - 1);
        wl.segments.push_back(Segment{i, h, pb, pb, page_size, -1, -1, 0});
        seg_cta.push_back((int32_t)cta);
        continue;
      }
      const int64_t start = pos, end = pos + np;
      const size_t first = wl.segments.size();
      const int64_t len = (np - 1) * page_size + last_page_len[i];
      for (int64_t a = start; a < end;) {
        const int64_t cta = a / quota;
        const int64_t b = std::min(end, (cta + 1) * quota);
        const int32_t last = (b == end) ? last_page_len[i] : page_size;
        wl.segments.push_back(Segment{i, h, (int32_t)(pb + (a - start)),
                                      (int32_t)(pb + (b - start)), last, -1, -1,
                                      (int32_t)(len - (a - start) * page_size)});
        seg_cta.push_back((int32_t)cta);
        a = b;
      }
      const int pieces = (int)(wl.segments.size() - first);
      if (pieces > 1) {
        const int unit = (int)wl.merge.size();
        wl.merge.push_back(MergeUnit{i, h, slots, pieces});
        for (int k = 0; k < pieces; ++k) {
          wl.segments[first + k].out_slot = slots + k;
          wl.segments[first + k].merge_unit = unit;
        }
        slots += pieces;
      }
      pos = end;
    }
  }
  wl.num_slots = slots;
  wl.cta_offsets.assign((size_t)num_ctas + 1, 0);
  for (int32_t c : seg_cta) wl.cta_offsets[(size_t)c + 1]++;
  for (int c = 0; c < num_ctas; ++c) wl.cta_offsets[c + 1] += wl.cta_offsets[c];
  *out = std::move(wl);
  return 0;
}

}  // namespace fadecode
