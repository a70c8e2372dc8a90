// Host planner: balanced split of the KV axis over a persistent grid.
//
// The decode work of a batch is the sequence of units (request, kv head) in
// request-major order, unit (i, h) costing the np_i pages of request i plus
// a fixed c0 = kSegmentCostPages for the segment's own overhead (0 for an
// empty unit).  Laid end to end, the units form one stream of total
// C = T + c0 * (non-empty units), T = num_kv_heads * sum_i np_i pages.  The
// planner fixes the grid size N (at most the number of CTAs resident at once,
// and no more than T / min_pages_per_cta) and gives CTA c the stream positions
// [c*q, (c+1)*q) with q = ceil(C / N); a page belongs to the CTA whose range
// holds its position.  A unit that a cut falls inside is split at that page
// boundary; each piece becomes a segment that writes a partial (o, lse) state
// into its own slot, and a merge unit records which slots to combine.  Every
// CTA therefore carries the same cost (+-1) whatever the mix of context
// lengths, which is the
// load-balancing duty the page "FlashDecoding + FlashInfer" assigns to
// FlashInfer's plan step ("What FlashInfer is", item 3), and a long request
// is spread over as many CTAs as its length needs, which is the split-KV
// idea of section "FlashDecoding - the split-KV trick".
//
// Equal quotas assume equal speed, but CTAs do not stream pages at exactly
// the same rate, so the slowest CTA sets the end of the launch.  With
// pool_fraction > 0 the planner hands only the first (1 - pool_fraction) of
// the stream out as quotas and cuts the rest into a pool of chunks, long ones
// first, that CTAs claim at run time (one atomic per chunk) once their quota
// is done - the fast CTAs take more of them and all CTAs finish within about
// one short chunk of each other.  The chunks are fixed here, so every chunk
// is computed the same way whichever CTA claims it.  Each chunk is one more
// piece to merge, which is why the library leaves the pool off by default.
//
// Requests with no pages still get one (empty) segment per kv head so that
// their output (o = 0, lse = -inf) is written.
#include "planner.h"

#include <algorithm>
#include <climits>

namespace fadecode {
namespace {

// Where the planner's output goes: growable vectors (WorkList) or fixed
// arrays (FixedWorkList).  Each push returns false when the output is full.
struct VectorSink {
  WorkList* wl;
  std::vector<Segment> pooled;  // pool segments, in stream order
  bool start(int num_ctas, size_t units, bool pool) {
    wl->cta_offsets.assign((size_t)num_ctas + 1, 0);
    wl->segments.reserve(units + num_ctas + 1);
    if (pool) pooled.reserve(units / 4 + 64);
    return true;
  }
  bool segment(int64_t cta, const Segment& s) {
    wl->segments.push_back(s);
    wl->cta_offsets[(size_t)cta + 1]++;
    return true;
  }
  bool pool_segment(const Segment& s) {
    pooled.push_back(s);
    return true;
  }
  bool merge(const MergeUnit& m) {
    wl->merge.push_back(m);
    return true;
  }
  void finish(int num_ctas) {
    for (int c = 0; c < num_ctas; ++c) wl->cta_offsets[c + 1] += wl->cta_offsets[c];
    wl->segments.insert(wl->segments.end(), pooled.begin(), pooled.end());
  }
};

struct FixedSink {
  FixedWorkList* wl;
  bool start(int num_ctas, size_t, bool pool) {
    if (pool || num_ctas > wl->cta_capacity) return false;
    for (int c = 0; c <= num_ctas; ++c) wl->cta_offsets[c] = 0;
    wl->num_segments = wl->num_merge = 0;
    return true;
  }
  bool segment(int64_t cta, const Segment& s) {
    if (wl->num_segments >= wl->segment_capacity) return false;
    wl->segments[wl->num_segments++] = s;
    wl->cta_offsets[cta + 1]++;
    return true;
  }
  bool pool_segment(const Segment&) { return false; }
  bool merge(const MergeUnit& m) {
    if (wl->num_merge >= wl->merge_capacity) return false;
    wl->merge[wl->num_merge++] = m;
    return true;
  }
  void finish(int num_ctas) {
    for (int c = 0; c < num_ctas; ++c) wl->cta_offsets[c + 1] += wl->cta_offsets[c];
  }
};

struct Totals {
  int num_ctas = 0, num_slots = 0;
  int64_t total_pages = 0, total_tokens = 0, pool_pages = 0;
};

// The planner proper, writing through `sink`.  Returns 0, -1 for malformed
// input, or -2 when the sink is full.
template <typename Sink>
int plan_stream(const int32_t* indptr, const int32_t* last_page_len, int batch,
                int num_kv_heads, int page_size, int max_ctas, int min_pages_per_cta,
                double pool_fraction, Sink& sink, Totals* tot) {
  if (!indptr || batch < 0 || num_kv_heads <= 0 || page_size <= 0 || max_ctas <= 0 ||
      !(pool_fraction >= 0.0 && pool_fraction < 1.0))
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
  // The pool: the last pool_pages positions of the stream, if there are
  // enough of them to give every CTA a few chunks.
  int64_t pool = (int64_t)(pool_fraction * (double)T);
  if (pool < n * kPoolMinPages * 2) pool = 0;
  // per-segment cost: without a pool, and only while a quota stays above
  // twice the cost
  int64_t busy_units = 0;
  for (int i = 0; i < batch; ++i)
    if (indptr[i + 1] > indptr[i]) busy_units += num_kv_heads;
  int64_t c0 = pool == 0 ? kSegmentCostPages : 0;
  if (c0 > 0 && (T + c0 * busy_units + n - 1) / n <= 2 * c0) c0 = 0;
  const int64_t C = T + c0 * busy_units;  // stream length in cost positions
  const int64_t S = C - pool;             // static positions [0, S)
  const int64_t quota = S > 0 ? (S + n - 1) / n : 1;
  if (pool == 0 && T > 0) n = (C + quota - 1) / quota;  // no CTA left without pages
  const int num_ctas = (int)n;

  // Pool chunk ends (absolute stream positions): tier t cuts n chunks of
  // ceil(pool / (n * 2^(t+1))) pages, so early claims take long chunks and
  // the last ones short chunks that even out the CTAs' finishing times.
  // (Empty without a pool: a plan without one allocates nothing here.)
  std::vector<int64_t> chunk_end;
  if (pool > 0) {
    int64_t a = S, size = kPoolMinPages;
    for (int t = 0; t < kPoolTiers && a < T; ++t) {
      const int64_t div = n << (t + 1);
      size = std::max<int64_t>(kPoolMinPages, (pool + div - 1) / div);
      for (int64_t c = 0; c < n && a < T; ++c) chunk_end.push_back(a = std::min(T, a + size));
      if (size == kPoolMinPages) break;
    }
    while (a < T) chunk_end.push_back(a = std::min(T, a + size));
  }

  if (!sink.start(num_ctas, (size_t)batch * num_kv_heads, pool > 0)) return -2;

  // Positions only grow, so the owning CTA and the next cut are tracked
  // incrementally (64-bit divisions per piece cost more than the rest).
  size_t ci = 0;        // first chunk end beyond the current position
  int64_t cta = 0;      // CTA of the current static position
  int64_t cut = quota;  // end of that CTA's quota
  int64_t pos = 0;
  int slots = 0, n_merge = 0;
  for (int i = 0; i < batch; ++i) {
    const int32_t pb = indptr[i], pe = indptr[i + 1];
    const int64_t np = (int64_t)pe - pb;
    const int64_t len = np > 0 ? (np - 1) * page_size + last_page_len[i] : 0;
    for (int h = 0; h < num_kv_heads; ++h) {
      // the unit's pages sit at [start, end), after its fixed cost
      const int64_t start = pos + (np > 0 ? c0 : 0), end = start + np;
      pos = end;
      while (start >= cut && cta < num_ctas - 1) {
        ++cta;
        cut += quota;
      }
      if (np == 0) {
        const Segment e{i, h, pb, pb, page_size, -1, -1, 0};
        const bool ok = (pool > 0 && start >= S) ? sink.pool_segment(e) : sink.segment(cta, e);
        if (!ok) return -2;
        continue;
      }
      // pieces: static ones cut at quota boundaries, pool ones at chunk ends
      const int64_t se = std::min(end, S);
      int pieces = 0;
      if (start < se) {
        pieces = 1;
        for (int64_t c = cut; c < se; c += quota) ++pieces;
      }
      if (end > S) {
        const int64_t a = std::max(start, S);
        while (chunk_end[ci] <= a) ++ci;
        size_t cj = ci;
        while (chunk_end[cj] < end) ++cj;
        pieces += (int)(cj - ci) + 1;
      }
      int slot = -1, unit = -1;
      if (pieces > 1) {
        unit = n_merge++;
        if (!sink.merge(MergeUnit{i, h, slots, pieces})) return -2;
        slot = slots;
        slots += pieces;
      }
      for (int64_t a = start; a < end;) {
        const bool in_pool = a >= S;
        int64_t b;
        if (!in_pool) {
          while (a >= cut) {
            ++cta;
            cut += quota;
          }
          b = std::min(se, cut);
        } else {
          while (chunk_end[ci] <= a) ++ci;
          b = std::min(end, chunk_end[ci]);
        }
        const Segment sg{i, h, (int32_t)(pb + (a - start)), (int32_t)(pb + (b - start)),
                         (b == end) ? last_page_len[i] : page_size, slot, unit,
                         (int32_t)(len - (a - start) * page_size)};
        if (!(in_pool ? sink.pool_segment(sg) : sink.segment(cta, sg))) return -2;
        if (slot >= 0) ++slot;
        a = b;
      }
    }
  }
  sink.finish(num_ctas);
  tot->num_ctas = num_ctas;
  tot->num_slots = slots;
  tot->total_pages = total_pages;
  tot->total_tokens = total_tokens;
  tot->pool_pages = pool;
  return 0;
}

// The plan in groups of num_kv_heads CTAs.  The batch's pages form one
// stream, request by request (each request preceded by the fixed cost c0);
// equal quotas of it go to the groups, and within group g CTA g * H + h
// takes the quota's pages for kv head h.  The group's CTAs therefore stream
// the same pages at the same time, each its own kv head's rows of them:
// neighbouring rows of the cache (the heads of one token are adjacent) are
// read together, which the memory streams markedly faster than rows read
// far apart in time (one kv head of an E4M3 page is 128-byte rows 1 KB
// apart).  A request a quota boundary falls inside is cut there for every
// head alike; its pieces are merged as in plan_stream.  Segments are
// produced CTA by CTA (group by group, head by head), the merge table
// first, so that both sinks receive them in order; nothing is allocated.
template <typename Sink>
int plan_heads(const int32_t* indptr, const int32_t* last_page_len, int batch,
               int num_kv_heads, int page_size, int max_ctas, int min_pages_per_cta, Sink& sink,
               Totals* tot) {
  if (!indptr || batch < 0 || num_kv_heads <= 0 || page_size <= 0 || max_ctas < num_kv_heads)
    return -1;
  if (batch > 0 && !last_page_len) return -1;
  if (indptr[0] != 0) return -1;
  const int64_t H = num_kv_heads;
  int64_t total_tokens = 0, busy = 0;
  for (int i = 0; i < batch; ++i) {
    const int64_t np = (int64_t)indptr[i + 1] - indptr[i];
    if (np < 0) return -1;
    if (np > 0) {
      if (last_page_len[i] < 1 || last_page_len[i] > page_size) return -1;
      total_tokens += (np - 1) * page_size + last_page_len[i];
      ++busy;
    }
  }
  const int64_t T = indptr[batch];  // pages of one kv head
  if (min_pages_per_cta < 1) min_pages_per_cta = 1;
  int64_t groups = max_ctas / H;
  if (T > 0) groups = std::min<int64_t>(groups, (T + min_pages_per_cta - 1) / min_pages_per_cta);
  groups = std::max<int64_t>(groups, 1);
  int64_t c0 = kSegmentCostPages;
  if ((T + c0 * busy + groups - 1) / groups <= 2 * c0) c0 = 0;
  const int64_t C = T + c0 * busy;  // stream length in cost positions
  const int64_t quota = C > 0 ? (C + groups - 1) / groups : 1;
  if (T > 0) groups = (C - 1) / quota + 1;  // every group holds a page
  const int64_t n = groups * H;
  auto group_of = [&](int64_t x) { return std::min(x / quota, groups - 1); };
  if (!sink.start((int)n, (size_t)batch * num_kv_heads, false)) return -2;

  // merge table: split requests in order, all heads of one request together
  int slots = 0;
  {
    int64_t pos = 0;
    for (int i = 0; i < batch; ++i) {
      const int64_t np = (int64_t)indptr[i + 1] - indptr[i];
      if (np == 0) continue;
      const int64_t start = pos + c0, end = start + np;
      pos = end;
      const int pieces = (int)(group_of(end - 1) - group_of(start) + 1);
      if (pieces < 2) continue;
      for (int h = 0; h < num_kv_heads; ++h) {
        if (!sink.merge(MergeUnit{i, h, slots, pieces})) return -2;
        slots += pieces;
      }
    }
  }

  // segments, CTA by CTA.  The cursor (i0, its stream position, the split
  // requests and slots before it) is the first request that may reach into
  // group g.
  int i0 = 0;
  int64_t pos0 = 0, units0 = 0, slots0 = 0;
  for (int64_t g = 0; g < groups; ++g) {
    for (int h = 0; h < num_kv_heads; ++h) {
      int64_t pos = pos0, units = units0, sl = slots0;
      for (int i = i0; i < batch; ++i) {
        const int32_t pb = indptr[i];
        const int64_t np = (int64_t)indptr[i + 1] - pb;
        if (np == 0) {  // an empty request: one empty segment per head, where it sits
          const int64_t ge = group_of(pos);
          if (ge > g) break;
          if (ge == g && !sink.segment(g * H + h, Segment{i, h, pb, pb, page_size, -1, -1, 0}))
            return -2;
          continue;
        }
        const int64_t start = pos + c0, end = start + np;
        const int64_t gs = group_of(start), gz = group_of(end - 1);
        if (gs > g) break;
        const int pieces = (int)(gz - gs + 1);
        if (gz >= g) {
          const int64_t a = std::max(start, g * quota);
          const int64_t b = g == groups - 1 ? end : std::min(end, (g + 1) * quota);
          const int64_t len = (np - 1) * page_size + last_page_len[i];
          const int k = (int)(g - gs);  // this piece's place among the request's
          const int unit = pieces > 1 ? (int)(units * H + h) : -1;
          const int slot = pieces > 1 ? (int)(sl + (int64_t)h * pieces + k) : -1;
          const Segment sg{i, h, (int32_t)(pb + (a - start)), (int32_t)(pb + (b - start)),
                           b == end ? last_page_len[i] : page_size, slot, unit,
                           (int32_t)(len - (a - start) * page_size)};
          if (!sink.segment(g * H + h, sg)) return -2;
        }
        if (pieces > 1) {
          ++units;
          sl += (int64_t)pieces * H;
        }
        pos = end;
      }
    }
    // move the cursor past the requests that end inside group g
    const int64_t next = (g + 1) * quota;
    while (i0 < batch) {
      const int64_t np = (int64_t)indptr[i0 + 1] - indptr[i0];
      if (np == 0) {
        if (group_of(pos0) > g) break;
        ++i0;
        continue;
      }
      const int64_t start = pos0 + c0, end = start + np;
      if (end > next) break;
      if (group_of(end - 1) > group_of(start)) {
        ++units0;
        slots0 += (group_of(end - 1) - group_of(start) + 1) * H;
      }
      pos0 = end;
      ++i0;
    }
  }
  sink.finish((int)n);
  tot->num_ctas = (int)n;
  tot->num_slots = slots;
  tot->total_pages = T;
  tot->total_tokens = total_tokens;
  tot->pool_pages = 0;
  return 0;
}

}  // namespace

int build_work_list(const int32_t* indptr, const int32_t* last_page_len,
                    int batch, int num_kv_heads, int page_size, int max_ctas,
                    int min_pages_per_cta, double pool_fraction, WorkList* out, bool heads) {
  if (!out) return -1;
  WorkList wl;
  VectorSink sink{&wl, {}};
  Totals tot;
  const int rc =
      heads && pool_fraction == 0.0 && max_ctas >= num_kv_heads
          ? plan_heads(indptr, last_page_len, batch, num_kv_heads, page_size, max_ctas,
                       min_pages_per_cta, sink, &tot)
          : plan_stream(indptr, last_page_len, batch, num_kv_heads, page_size, max_ctas,
                        min_pages_per_cta, pool_fraction, sink, &tot);
  if (rc != 0) return -1;
  wl.num_ctas = tot.num_ctas;
  wl.num_slots = tot.num_slots;
  wl.total_pages = tot.total_pages;
  wl.total_tokens = tot.total_tokens;
  wl.pool_pages = tot.pool_pages;
  *out = std::move(wl);
  return 0;
}

int build_work_list_fixed(const int32_t* indptr, const int32_t* last_page_len, int batch,
                          int num_kv_heads, int page_size, int max_ctas, int min_pages_per_cta,
                          FixedWorkList* out, bool heads) {
  if (!out || !out->cta_offsets || !out->segments || !out->merge) return -1;
  FixedSink sink{out};
  Totals tot;
  const int rc = heads && max_ctas >= num_kv_heads
                     ? plan_heads(indptr, last_page_len, batch, num_kv_heads, page_size,
                                  max_ctas, min_pages_per_cta, sink, &tot)
                     : plan_stream(indptr, last_page_len, batch, num_kv_heads, page_size,
                                   max_ctas, min_pages_per_cta, 0.0, sink, &tot);
  if (rc != 0) return rc;
  out->num_ctas = tot.num_ctas;
  out->num_slots = tot.num_slots;
  out->total_pages = tot.total_pages;
  out->total_tokens = tot.total_tokens;
  return 0;
}

namespace {

// Requests of a batch as a batch of their own: indptr and last_page_len
// compacted, and each one's id in the whole batch.
struct SubBatch {
  std::vector<int32_t> indptr{0}, last, ids;
  void add(const int32_t* indptr_all, const int32_t* last_all, int i) {
    ids.push_back(i);
    indptr.push_back(indptr.back() + (indptr_all[i + 1] - indptr_all[i]));
    last.push_back(last_all[i]);
  }
};

// Append the work list of a sub-batch to `out` (see build_bucket_work_list).
void append_work(const WorkList& w, const SubBatch& s, const int32_t* indptr, int64_t slot_base,
                 WorkList* out) {
  const int32_t seg0 = (int32_t)out->segments.size(), m0 = (int32_t)out->merge.size();
  if (out->cta_offsets.empty()) out->cta_offsets.push_back(0);
  for (int c = 1; c <= w.num_ctas; ++c) out->cta_offsets.push_back(seg0 + w.cta_offsets[c]);
  for (Segment sg : w.segments) {
    const int32_t shift = indptr[s.ids[sg.request]] - s.indptr[sg.request];
    sg.request = s.ids[sg.request];
    sg.page_begin += shift;
    sg.page_end += shift;
    if (sg.merge_unit >= 0) sg.merge_unit += m0;
    if (sg.out_slot >= 0) sg.out_slot += (int32_t)slot_base;
    out->segments.push_back(sg);
  }
  for (MergeUnit m : w.merge) {
    m.request = s.ids[m.request];
    m.first_slot += (int32_t)slot_base;
    out->merge.push_back(m);
  }
  out->num_ctas += w.num_ctas;
  out->total_pages += w.total_pages;
  out->total_tokens += w.total_tokens;
}

}  // namespace

int build_bucket_work_list(const int32_t* indptr, const int32_t* last_page_len,
                           const int32_t* qo_indptr, int batch, int num_kv_heads, int page_size,
                           const BucketPolicy& pol, WorkList* out, BucketList* buckets) {
  if (!indptr || !qo_indptr || !out || !buckets || batch < 0 || num_kv_heads <= 0 ||
      page_size <= 0 || pol.group < 1 || 8 % pol.group != 0 || pol.widest < 1 ||
      pol.widest > kMaxTileBuckets)
    return -1;
  if (batch > 0 && !last_page_len) return -1;
  if (indptr[0] != 0 || qo_indptr[0] != 0) return -1;
  const int G = pol.group;
  int64_t units[kMaxTileBuckets + 1] = {0};
  int count[kMaxTileBuckets + 1] = {0};
  for (int i = 0; i < batch; ++i) {
    const int64_t np = (int64_t)indptr[i + 1] - indptr[i];
    const int64_t nq = (int64_t)qo_indptr[i + 1] - qo_indptr[i];
    if (np < 0 || nq < 0) return -1;
    const int64_t t = std::max<int64_t>(1, (G * nq + 7) / 8);
    if (t > pol.widest) return -1;
    units[t] += np * num_kv_heads;
    ++count[t];
  }
  int top = 0;  // the widest tile count present
  for (int t = 1; t <= pol.widest; ++t)
    if (count[t] > 0) top = t;
  int dest[kMaxTileBuckets + 1] = {0};
  for (int t = 1; t <= pol.widest; ++t) {
    const bool own = pol.all || (t == 1 && pol.one_tile_own && units[1] >= pol.min_own_units);
    dest[t] = own ? t : top;
  }
  BucketList bl;
  for (int t = pol.widest; t >= 1; --t) {
    bool used = false;
    for (int u = 1; u <= pol.widest; ++u) used = used || (count[u] > 0 && dest[u] == t);
    if (used) bl.tiles[bl.num++] = t;
  }
  *buckets = BucketList{};
  if (bl.num == 0 || (bl.num == 1 && bl.tiles[0] == pol.widest)) return 0;
  for (int b = 0; b < bl.num; ++b)
    if (pol.max_ctas[bl.tiles[b]] < 1) return -1;

  SubBatch sub[kMaxTileBuckets];
  for (int i = 0; i < batch; ++i) {
    const int nq = qo_indptr[i + 1] - qo_indptr[i];
    const int t = dest[std::max(1, (G * nq + 7) / 8)];
    for (int b = 0; b < bl.num; ++b)
      if (bl.tiles[b] == t) sub[b].add(indptr, last_page_len, i);
  }
  WorkList w;
  int64_t cols = 0;  // partial-state columns taken by the buckets so far
  for (int b = 0; b < bl.num; ++b) {
    WorkList wb;
    if (build_work_list(sub[b].indptr.data(), sub[b].last.data(), (int)sub[b].ids.size(),
                        num_kv_heads, page_size, pol.max_ctas[bl.tiles[b]],
                        pol.min_pages_per_cta, 0.0, &wb, pol.heads) != 0)
      return -1;
    const int nc = 8 * bl.tiles[b];
    const int64_t slot_base = (cols + nc - 1) / nc;
    if (slot_base + wb.num_slots > INT32_MAX) return -1;
    bl.cta_first[b] = w.num_ctas;
    bl.num_ctas[b] = wb.num_ctas;
    bl.merge_first[b] = (int)w.merge.size();
    bl.num_merge[b] = (int)wb.merge.size();
    append_work(wb, sub[b], indptr, slot_base, &w);
    cols = (slot_base + wb.num_slots) * nc;
  }
  bl.slot_columns = cols;
  *out = std::move(w);
  *buckets = bl;
  return 0;
}

}  // namespace fadecode
