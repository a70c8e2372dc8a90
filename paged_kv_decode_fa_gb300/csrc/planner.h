// Host planner for split-KV paged decode: cuts the batch's KV work into
// per-CTA chunks of equal page count.  Pure C++, no CUDA.
#pragma once
#include <cstdint>
#include <vector>

namespace fadecode {

// One work item, eight int32 so the device can read it as two int4.
struct Segment {
  int32_t request;
  int32_t kv_head;
  int32_t page_begin;  // position in the indices array
  int32_t page_end;    // exclusive
  int32_t last_valid;  // valid slots in the segment's final page
  int32_t out_slot;    // -1: writes o/lse directly; else partial-state slot
  int32_t merge_unit;  // -1 when unsplit; else index into the merge table
  int32_t to_end;      // tokens from the segment's first token to the request end
};
static_assert(sizeof(Segment) == 32, "Segment must stay 32 bytes");

struct MergeUnit {
  int32_t request;
  int32_t kv_head;
  int32_t first_slot;
  int32_t num_slots;
};
static_assert(sizeof(MergeUnit) == 16, "MergeUnit must stay 16 bytes");

// Pool of the balanced plan: its chunk sizes halve over kPoolTiers tiers of
// one chunk per CTA each, then the rest goes in chunks of the last size; no
// chunk is shorter than kPoolMinPages pages (unless a unit ends first).
constexpr int kPoolTiers = 4;
constexpr int kPoolMinPages = 2;

// Fixed cost of a segment in the balanced plan, in pages: loading q, filling
// the ring and writing the partial state cost a CTA about as long as
// streaming two pages, so a CTA whose quota holds many short requests gets
// fewer pages.  Applied only without a pool and when a quota exceeds twice
// this cost (every CTA then still holds a page).
constexpr int kSegmentCostPages = 2;

// Upper bound of the cuts a plan makes into (request, kv head) units for a
// grid of n CTAs: n - 1 quota boundaries, the pool's start and at most
// (kPoolTiers + 2) * n chunk boundaries.  Segments <= units + cuts and
// partial slots <= 2 * cuts.
inline int64_t max_plan_cuts(int64_t n) { return n * (kPoolTiers + 3) + 1; }

struct WorkList {
  // Static part: CTA c runs segments cta_offsets[c] .. cta_offsets[c+1]-1.
  // Pool: segments cta_offsets[num_ctas] .. segments.size()-1, claimed at
  // run time, in order, by whichever CTA is free (none when pool_pages = 0).
  std::vector<int32_t> cta_offsets;  // num_ctas + 1
  std::vector<Segment> segments;
  std::vector<MergeUnit> merge;
  int num_ctas = 0;
  int num_slots = 0;
  int64_t total_pages = 0;   // sum over requests (not times kv heads)
  int64_t total_tokens = 0;  // sum of len over requests
  int64_t pool_pages = 0;    // (page, kv head) pairs left to the pool
  int pool_begin() const { return cta_offsets.empty() ? 0 : cta_offsets.back(); }
  int pool_count() const { return (int)segments.size() - pool_begin(); }
};

// Returns 0 on success, -1 for malformed input (see fa_decode.h).
// pool_fraction in [0, 1): share of the page stream left to the pool.
// heads: plan the grid in groups of num_kv_heads CTAs that take the same
// share of the page stream, one kv head each (plan_heads in planner.cpp),
// instead of cutting the stream of (request, kv head) units; applies only
// without a pool and with at least num_kv_heads CTAs.
int build_work_list(const int32_t* indptr, const int32_t* last_page_len,
                    int batch, int num_kv_heads, int page_size, int max_ctas,
                    int min_pages_per_cta, double pool_fraction, WorkList* out,
                    bool heads = false);

// The same plan without a pool, written into arrays the caller owns (no
// allocation): cta_offsets[cta_capacity + 1], segments[segment_capacity],
// merge[merge_capacity].  The counts are filled in on success.
struct FixedWorkList {
  int32_t* cta_offsets = nullptr;
  Segment* segments = nullptr;
  MergeUnit* merge = nullptr;
  int cta_capacity = 0, segment_capacity = 0, merge_capacity = 0;
  int num_ctas = 0, num_segments = 0, num_merge = 0, num_slots = 0;
  int64_t total_pages = 0, total_tokens = 0;
};

// Returns 0, -1 for malformed input, -2 when a plan does not fit the arrays.
int build_work_list_fixed(const int32_t* indptr, const int32_t* last_page_len, int batch,
                          int num_kv_heads, int page_size, int max_ctas, int min_pages_per_cta,
                          FixedWorkList* out, bool heads = false);

// Buckets of a ragged plan by 8-column tiles.  Request i of a batch with
// group G has n_i query rows and needs t_i = max(1, ceil(G n_i / 8)) tiles;
// the kernel of t tiles holds 8t / G rows a request.  policy: which tile
// counts take a launch of their own (see build_bucket_work_list).
constexpr int kMaxTileBuckets = 4;

struct BucketPolicy {
  int group = 1;                               // query heads per kv head (1, 2, 4, 8)
  int widest = kMaxTileBuckets;                // tiles the batch's one-launch kernel holds
  int max_ctas[kMaxTileBuckets + 1] = {0};     // grid bound of the kernel of t tiles [t]
  bool one_tile_own = false;                   // one-tile requests may take their own launch
  int64_t min_own_units = 0;                   // ... from this many (page, kv head) pairs
  bool all = false;                            // a launch for every tile count present
  int min_pages_per_cta = 8;
  bool heads = true;                           // head-grouped plan per bucket
};

struct BucketList {
  int num = 0;  // launches; 0: the batch stays one launch of the widest kernel
  int tiles[kMaxTileBuckets] = {0};
  int cta_first[kMaxTileBuckets] = {0}, num_ctas[kMaxTileBuckets] = {0};
  int merge_first[kMaxTileBuckets] = {0}, num_merge[kMaxTileBuckets] = {0};
  int64_t slot_columns = 0;  // partial-state columns (x head_dim floats) the buckets take
};

// Plan a ragged batch in buckets: every request goes to the kernel of the
// widest tile count present (top), except, when one_tile_own and the
// one-tile requests hold at least min_own_units (page, kv head) pairs, or
// when all, those of a tile count with a launch of its own.  One work list
// per bucket (build_work_list on the bucket's requests, its kernel's grid
// bound), concatenated widest first: a later bucket's CTAs, segments and
// merge units follow the earlier ones', its requests and page positions
// mapped back to the batch, its partial slots after the columns the
// earlier buckets' slots take, in units of its own slot (8t columns).
// Returns 0 (out and buckets filled; buckets->num = 0 and out untouched
// when one launch of the widest kernel remains) or -1 for malformed input.
int build_bucket_work_list(const int32_t* indptr, const int32_t* last_page_len,
                           const int32_t* qo_indptr, int batch, int num_kv_heads, int page_size,
                           const BucketPolicy& policy, WorkList* out, BucketList* buckets);

}  // namespace fadecode
