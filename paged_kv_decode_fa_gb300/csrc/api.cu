// C ABI of libfadecode.so (declared in include/fa_decode.h): plan handle,
// workspace layout, TMA descriptor of the KV cache and kernel launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "fa_decode.h"
#include "kernels.h"
#include "planner.h"
#include "staging.h"

using fadecode::DecodeKernel;
using fadecode::DecodeParams;
using fadecode::MergeParams;
using fadecode::WorkList;

namespace {

constexpr int kMinPagesPerCta = 8;     // smallest chunk worth a CTA of its own
constexpr int kMaxCtasPerSmBound = 4;  // grid bound (every kernel fits 3 or 4 CTAs per SM)
// Ragged plans in buckets (plan_buckets): at most one launch per number of
// 8-column tiles (1-4) a request needs; the one-tile requests of an E4M3
// batch take a launch of their own from kMinBucketUnitsPerSm (page, kv head)
// pairs per SM on (below that a launch's fixed time outweighs the gain).
constexpr int kMaxBuckets = 4;
constexpr int kMinBucketUnitsPerSm = 64;
// Share of the page stream balanced at run time.  Off: on a GB300 the
// static quotas already finish within a few percent of each other in
// back-to-back launches, and the pool's extra pieces cost more than it saves
// except on strongly mixed lengths (FADECODE_POOL=0.25: -2.7 % on the
// 256..64000-token mix); a unit whose pages all fall in the pool also ends
// up with hundreds of pieces to fold.
constexpr double kPoolFraction = 0.0;
constexpr size_t kAlign = 256;
constexpr float kLog2e = 1.4426950408889634f;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t off_err, off_umc, off_pool, off_cta, off_seg, off_merge, off_count, off_qo, meta_bytes,
      off_part_o, off_part_lse, total;
};

// Metadata (uploaded by every plan, zeros included) then the partial states.
// G is the columns of a partial state (group x query tokens); n_qo the
// entries of a ragged plan's qo_indptr copy (0 otherwise).
Layout make_layout(int64_t n_ctas, int64_t n_segments, int64_t n_merge, int64_t n_slots, int G,
                   int D, int64_t n_qo = 0) {
  Layout L;
  L.off_err = 0;
  L.off_umc = sizeof(int);  // unified-max re-centring counter
  L.off_pool = 2 * sizeof(int);  // pool claim and done counters
  L.off_cta = align_up(L.off_pool + 2 * sizeof(int));
  L.off_seg = align_up(L.off_cta + sizeof(int32_t) * (size_t)(n_ctas + 1));
  L.off_merge = align_up(L.off_seg + sizeof(fadecode::Segment) * (size_t)n_segments);
  L.off_count = align_up(L.off_merge + sizeof(fadecode::MergeUnit) * (size_t)n_merge);
  L.off_qo = align_up(L.off_count + sizeof(int32_t) * (size_t)n_merge);
  L.meta_bytes = align_up(L.off_qo + sizeof(int32_t) * (size_t)n_qo);
  L.off_part_o = L.meta_bytes;
  L.off_part_lse = align_up(L.off_part_o + sizeof(float) * (size_t)n_slots * G * D);
  L.total = align_up(L.off_part_lse + sizeof(float) * (size_t)n_slots * G);
  return L;
}

int dtype_size(fa_dtype t) {
  switch (t) {
    case FA_DTYPE_F32: return 4;
    case FA_DTYPE_BF16:
    case FA_DTYPE_F16: return 2;
    case FA_DTYPE_E4M3: return 1;
  }
  return 0;
}

// FADECODE_MERGE=kernel folds split requests in a separate merge kernel
// after the decode kernel (for comparisons); by default the last CTA to
// finish a piece of a split request folds it inside the decode kernel.
bool fused_merge_enabled() {
  const char* v = std::getenv("FADECODE_MERGE");
  return !(v && std::strcmp(v, "kernel") == 0);
}

// FADECODE_POOL=<fraction> sets the share of the page stream left to the
// run-time pool (0 turns it off, for comparisons); default kPoolFraction.
double pool_fraction() {
  const char* v = std::getenv("FADECODE_POOL");
  if (!v) return kPoolFraction;
  const double f = std::atof(v);
  return f >= 0.0 && f <= 0.5 ? f : kPoolFraction;
}

// Plans put the grid in groups of num_kv_heads CTAs that stream the same
// pages, one kv head each (the planner's plan_heads); FADECODE_PLAN=stream
// cuts the stream of (request, kv head) units instead (for comparisons, and
// what a run-time pool uses).
bool heads_plan() {
  const char* v = std::getenv("FADECODE_PLAN");
  return !(v && std::strcmp(v, "stream") == 0);
}

// Ragged plans in buckets by 8-column tiles (plan_buckets): FADECODE_BUCKETS=0
// plans a ragged batch on the one kernel its max_q needs (for comparisons);
// FADECODE_BUCKETS=all gives every tile count present a launch of its own,
// however little work it holds (for tests of every bucket kernel).
enum class BucketMode { kOff, kDefault, kAll };
BucketMode bucket_mode() {
  const char* v = std::getenv("FADECODE_BUCKETS");
  if (v && std::strcmp(v, "0") == 0) return BucketMode::kOff;
  if (v && std::strcmp(v, "all") == 0) return BucketMode::kAll;
  return BucketMode::kDefault;
}

// FADECODE_KERNEL=simt keeps every plan on the CUDA-core consumer (for
// comparisons); by default the tensor-core consumer is used where it applies.
bool tensor_cores_allowed() {
  const char* v = std::getenv("FADECODE_KERNEL");
  return !(v && std::strcmp(v, "simt") == 0);
}

bool find_kernel(fa_dtype q, fa_dtype kv, int D, int G, DecodeKernel* k) {
  const bool mma = tensor_cores_allowed();
  if (q == FA_DTYPE_F32 && kv == FA_DTYPE_F32) return fadecode::find_kernel_f32(D, G, mma, k);
  if (q == FA_DTYPE_BF16 && kv == FA_DTYPE_BF16) return fadecode::find_kernel_bf16(D, G, mma, k);
  if (q == FA_DTYPE_F16 && kv == FA_DTYPE_F16) return fadecode::find_kernel_f16(D, G, mma, k);
  if (q == FA_DTYPE_BF16 && kv == FA_DTYPE_E4M3)
    return fadecode::find_kernel_bf16_e4m3(D, G, mma, k);
  if (q == FA_DTYPE_F16 && kv == FA_DTYPE_E4M3)
    return fadecode::find_kernel_f16_e4m3(D, G, mma, k);
  return false;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct MapCache {
  CUtensorMap tmap;
  const void* base = nullptr;
  int64_t pages = -1;
};

// Encode (or reuse) the TMA descriptor of `paged_kv` for kernel `k`: the view
// [2*num_pages][P][Hkv][D], innermost first; one box = K and V rows of one
// kv head of one page (or of one 128-byte segment of those rows when the
// kernel stages them in 128-byte swizzle order).
int kv_tensor_map(MapCache* c, const DecodeKernel& k, fa_dtype kv_dtype, const void* paged_kv,
                  int64_t num_pages, int D, int Hkv, int P) {
  if (paged_kv == c->base && num_pages == c->pages) return FA_OK;
  PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_fn();
  if (!encode) return FA_ERR_CUDA;
  const size_t es = (size_t)dtype_size(kv_dtype);
  CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  switch (kv_dtype) {
    case FA_DTYPE_F32: dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT32; break;
    case FA_DTYPE_BF16: dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; break;
    case FA_DTYPE_F16: dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT16; break;
    case FA_DTYPE_E4M3: dt = CU_TENSOR_MAP_DATA_TYPE_UINT8; break;
  }
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)P,
                        (cuuint64_t)(2 * num_pages)};
  cuuint64_t strides[3] = {(cuuint64_t)(D * es), (cuuint64_t)(Hkv * D * es),
                           (cuuint64_t)(P * Hkv * D * es)};
  cuuint32_t box[4] = {(cuuint32_t)k.box_x, 1u, (cuuint32_t)P, 2u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  // Promote L2 fills to the box row length: a longer promotion would pull
  // in the neighbouring kv heads' rows, which another CTA reads much later.
  const size_t row_bytes = (size_t)k.box_x * es;
  const CUtensorMapL2promotion promo = row_bytes >= 256   ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                       : row_bytes >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                                          : CU_TENSOR_MAP_L2_PROMOTION_L2_64B;
  CUresult r = encode(&c->tmap, dt, 4, const_cast<void*>(paged_kv), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE,
                      k.swizzle_128b ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                      promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    c->base = nullptr;
    return FA_ERR_CUDA;
  }
  c->base = paged_kv;
  c->pages = num_pages;
  return FA_OK;
}

bool find_ragged_q_kernel(fa_dtype q, fa_dtype kv, int D, int G, int max_q, DecodeKernel* k) {
  if (!tensor_cores_allowed() || q != FA_DTYPE_BF16) return false;
  if (kv == FA_DTYPE_BF16) return fadecode::find_ragged_q_kernel_bf16(D, G, max_q, k);
  if (kv == FA_DTYPE_E4M3) return fadecode::find_ragged_q_kernel_bf16_e4m3(D, G, max_q, k);
  return false;
}

// The ragged kernel for requests of `tiles` 8-column tiles (1-4): the
// 8-column kernel (pages split over its warps) for one, a column split of
// `tiles` warps otherwise.
bool find_ragged_tiles_kernel(fa_dtype q, fa_dtype kv, int D, int G, int tiles, DecodeKernel* k) {
  if (G < 1 || 8 % G != 0 || tiles < 1 || tiles > 4) return false;
  if (tiles == 1 || tiles == 4)
    return find_ragged_q_kernel(q, kv, D, G, 8 * tiles / G, k) && k->q_len * G == 8 * tiles;
  if (!tensor_cores_allowed() || q != FA_DTYPE_BF16) return false;
  if (kv == FA_DTYPE_BF16) return fadecode::find_ragged_q_tiles_kernel_bf16(D, G, tiles, k);
  if (kv == FA_DTYPE_E4M3) return fadecode::find_ragged_q_tiles_kernel_bf16_e4m3(D, G, tiles, k);
  return false;
}

bool find_unified_max_kernel(fa_dtype q, fa_dtype kv, int D, int G, DecodeKernel* k) {
  if (!tensor_cores_allowed()) return false;
  if (q == FA_DTYPE_BF16 && kv == FA_DTYPE_BF16) return fadecode::find_unified_max_kernel_bf16(D, G, k);
  if (q == FA_DTYPE_F16 && kv == FA_DTYPE_F16) return fadecode::find_unified_max_kernel_f16(D, G, k);
  if (q == FA_DTYPE_BF16 && kv == FA_DTYPE_E4M3)
    return fadecode::find_unified_max_kernel_bf16_e4m3(D, G, k);
  if (q == FA_DTYPE_F16 && kv == FA_DTYPE_E4M3)
    return fadecode::find_unified_max_kernel_f16_e4m3(D, G, k);
  return false;
}

bool find_token_scale_kernel(fa_dtype q, fa_dtype kv, int D, int G, DecodeKernel* k) {
  if (kv != FA_DTYPE_E4M3) return false;
  if (q == FA_DTYPE_BF16) return fadecode::find_token_scale_kernel_bf16_e4m3(D, G, k);
  if (q == FA_DTYPE_F16) return fadecode::find_token_scale_kernel_f16_e4m3(D, G, k);
  return false;
}

// Whether a decode launch of `func` on `st` may be a programmatic dependent
// of the stream's previous kernel, and record it as the stream's last decode
// kernel.  The decode kernels let the next launch in at their start
// (griddepcontrol.launch_dependents), so a dependent launch's CTAs are
// placed on SMs that the previous launch's CTAs are still leaving.  Behind
// the same kernel each takes the slot of one that left.  Behind a decode
// kernel of another shape the launch ran up to half as long again (the
// E4M3 column split: 365 us alone, about 540 us right behind an 8-column
// launch), the mark of a persistent grid whose CTAs did not all fit at
// once: placed among departing CTAs of another size, they leave some SMs
// with fewer than the grid was sized for.  So only a launch of the same
// kernel as the stream's last decode launch is a dependent one; a stream
// not seen before (or dropped from the table) gets an ordinary launch.
// Kernels that do not let the next launch in early leave every SM empty
// before a dependent launch's CTAs are placed, whatever the table says.
bool dependent_launch_ok(cudaStream_t st, const void* func) {
  struct Entry {
    cudaStream_t stream;
    const void* func;
  };
  constexpr int kEntries = 64;  // streams remembered; the oldest entry is reused
  static std::mutex mu;
  static Entry table[kEntries];
  static int used = 0, next = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i) {
    if (table[i].stream != st) continue;
    const bool same = table[i].func == func;
    table[i].func = func;
    return same;
  }
  const int slot = used < kEntries ? used++ : next;
  if (used == kEntries) next = (slot + 1) % kEntries;
  table[slot] = Entry{st, func};
  return false;
}

// Set a kernel's shared-memory limit and return how many of its CTAs fit on
// one SM (0 on failure).  Cached per (kernel, device): a plan per decode
// step should not pay for these queries every time.
int kernel_occupancy(const DecodeKernel& k) {
  struct Entry {
    const void* func;
    int device, occ;
  };
  // a fixed table (no allocation on any call): the compiled kernels times
  // the devices in use stay far below its size; past it, queries are simply
  // not cached
  constexpr int kEntries = 256;
  static std::mutex mu;
  static Entry cache[kEntries];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].func == k.func && cache[i].device == dev) return cache[i].occ;
  int occ = 0;
  if (cudaFuncSetAttribute(k.func, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem_bytes) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k.func, k.threads, k.smem_bytes) !=
          cudaSuccess)
    return 0;
  if (used < kEntries) cache[used++] = Entry{k.func, dev, occ};
  return occ;
}

}  // namespace

// Kernel variants a plan can launch.
enum Variant { kPlain = 0, kTokenScales = 1, kUnifiedMax = 2, kNumVariants = 3 };

namespace {

// The kernels a plan of these dtypes and shape may launch (kPlain always,
// the others where built) and the persistent grid's CTAs per SM: the
// smallest occupancy among them, so that every variant fits the grid.
int select_kernels(fa_dtype q_dtype, fa_dtype kv_dtype, int head_dim, int G, int q_len,
                   DecodeKernel (&kv)[kNumVariants], bool (&has)[kNumVariants],
                   int* ctas_per_sm, bool ragged = false) {
  DecodeKernel base;
  if (ragged) {
    if (!find_ragged_q_kernel(q_dtype, kv_dtype, head_dim, G, q_len, &base))
      return FA_ERR_UNSUPPORTED;
  } else if (q_len == 1) {
    if (!find_kernel(q_dtype, kv_dtype, head_dim, G, &base)) return FA_ERR_UNSUPPORTED;
  } else {
    bool ok = false;
    if (q_dtype == FA_DTYPE_BF16 && kv_dtype == FA_DTYPE_BF16)
      ok = fadecode::find_multi_token_kernel_bf16(head_dim, G, q_len, &base);
    else if (q_dtype == FA_DTYPE_BF16 && kv_dtype == FA_DTYPE_E4M3)
      ok = fadecode::find_multi_token_kernel_bf16_e4m3(head_dim, G, q_len, &base);
    if (!ok) return FA_ERR_UNSUPPORTED;
  }
  int occ = kernel_occupancy(base);
  if (occ == 0) return FA_ERR_CUDA;
  kv[kPlain] = base;
  has[kPlain] = true;
  has[kTokenScales] = has[kUnifiedMax] = false;
  if (q_len == 1 && !ragged) {
    has[kTokenScales] = find_token_scale_kernel(q_dtype, kv_dtype, head_dim, G, &kv[kTokenScales]);
    has[kUnifiedMax] = find_unified_max_kernel(q_dtype, kv_dtype, head_dim, G, &kv[kUnifiedMax]);
  }
  for (int v = 1; v < kNumVariants; ++v) {
    if (!has[v]) continue;
    const int occ_v = kernel_occupancy(kv[v]);
    if (occ_v == 0) return FA_ERR_CUDA;
    occ = std::min(occ, occ_v);
  }
  *ctas_per_sm = std::max(1, std::min(occ, kMaxCtasPerSmBound));
  return FA_OK;
}

// Everything one decode launch needs, owned elsewhere: by a plan object, or
// by the stack of the allocation-free entry point.
struct LaunchView {
  int batch = 0, hq = 0, hkv = 0, d = 0, page_size = 0, q_len = 1;
  fa_dtype q_dtype = FA_DTYPE_F32, kv_dtype = FA_DTYPE_F32;
  const DecodeKernel* kern = nullptr;
  MapCache* map = nullptr;
  const int32_t* indices = nullptr;
  uint8_t* ws = nullptr;
  Layout layout{};
  int num_ctas = 0, num_merge = 0, pool_begin = 0, pool_count = 0;
  // this launch's first CTA entry and first merge unit in the plan's tables
  int cta_first = 0, merge_first = 0;
  bool fused_merge = true;
  bool ragged_q = false;  // query rows per request from the plan's qo_indptr copy
  cudaEvent_t ev_before = nullptr, ev_after = nullptr;
};

int launch_decode(const LaunchView& lv, const void* q, const void* paged_kv, int64_t num_pages,
                  float sm_scale, float k_scale, float v_scale, const float* k_scales,
                  const float* v_scales, float max_bound, void* o, float* lse,
                  void* cuda_stream, const float* head_k_scales = nullptr,
                  const float* head_v_scales = nullptr);

}  // namespace

struct fa_decode_plan_s;
static int run_impl(fa_decode_plan_s* plan, Variant variant, const void* q,
                    const void* paged_kv, int64_t num_pages, float sm_scale, float k_scale,
                    float v_scale, const float* k_scales, const float* v_scales,
                    float max_bound, void* o, float* lse, void* cuda_stream,
                    const float* head_k_scales = nullptr,
                    const float* head_v_scales = nullptr);

struct fa_decode_plan_s {
  int device = 0;
  int batch = 0, hq = 0, hkv = 0, d = 0, page_size = 0, group = 0;
  fa_dtype q_dtype = FA_DTYPE_F32, kv_dtype = FA_DTYPE_F32;
  // kern[kPlain] always; kern[kTokenScales] / kern[kUnifiedMax] where
  // has[...] says the plan's dtypes and shape have that variant built
  DecodeKernel kern[kNumVariants];
  bool has[kNumVariants] = {true, false, false};
  int num_sms = 0, ctas_per_sm = 0;
  WorkList wl;
  std::vector<int32_t> merge_flat;
  const int32_t* indices = nullptr;
  uint8_t* ws = nullptr;
  size_t ws_bytes = 0;
  Layout layout{};
  bool fused_merge = true;
  int q_len = 1;          // query tokens per request (ragged: the kernel's largest)
  bool ragged_q = false;  // query rows from qo_indptr
  int64_t total_q = 0;    // query rows of the batch
  // cached TMA descriptors of the KV cache, one per kernel variant
  MapCache map[kNumVariants];
  // A ragged plan in buckets (plan_buckets): launch b runs bucket[b].kern
  // over CTAs [cta_first, cta_first + num_ctas) of the work list and owns
  // merge units [merge_first, merge_first + num_merge).  0: one launch of
  // kern[variant] over the whole work list.
  struct Bucket {
    DecodeKernel kern;
    MapCache map;
    int tiles = 0, cta_first = 0, num_ctas = 0, merge_first = 0, num_merge = 0;
  };
  int num_buckets = 0;
  Bucket bucket[kMaxBuckets];
  cudaEvent_t ev_before = nullptr, ev_after = nullptr;
};

extern "C" {

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_WORKSPACE_TOO_SMALL: return "FA_ERR_WORKSPACE_TOO_SMALL";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_DEVICE_CHECK: return "FA_ERR_DEVICE_CHECK";
  }
  return "FA_UNKNOWN_STATUS";
}

size_t fa_decode_workspace_size(int batch, int num_qo_heads, int num_kv_heads, int head_dim) {
  if (batch < 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      num_qo_heads % num_kv_heads)
    return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  const int64_t max_ctas = (int64_t)sms * kMaxCtasPerSmBound;
  const int64_t cuts = fadecode::max_plan_cuts(max_ctas);
  const int64_t segs = (int64_t)batch * num_kv_heads + cuts;
  const int G = num_qo_heads / num_kv_heads;
  return make_layout(max_ctas, segs, cuts, 2 * cuts, G, head_dim, (int64_t)batch + 1).total;
}

int fa_plan_work_host_heads(const int32_t* indptr, const int32_t* last_page_len, int batch,
                            int num_kv_heads, int page_size, int max_ctas,
                            int min_pages_per_cta, int32_t* cta_offsets, int32_t* segments,
                            int32_t* merge, int* n_ctas, int* n_segments, int* n_merge,
                            int* n_slots) {
  if (!cta_offsets || !segments || !merge || !n_ctas || !n_segments || !n_merge || !n_slots)
    return FA_ERR_INVALID_ARG;
  WorkList wl;
  try {
    if (fadecode::build_work_list(indptr, last_page_len, batch, num_kv_heads, page_size,
                                  max_ctas, min_pages_per_cta, 0.0, &wl, true) != 0)
      return FA_ERR_INVALID_ARG;
  } catch (const std::bad_alloc&) {
    return FA_ERR_INVALID_ARG;
  }
  std::memcpy(cta_offsets, wl.cta_offsets.data(), sizeof(int32_t) * wl.cta_offsets.size());
  std::memcpy(segments, wl.segments.data(), sizeof(fadecode::Segment) * wl.segments.size());
  std::memcpy(merge, wl.merge.data(), sizeof(fadecode::MergeUnit) * wl.merge.size());
  *n_ctas = wl.num_ctas;
  *n_segments = (int)wl.segments.size();
  *n_merge = (int)wl.merge.size();
  *n_slots = wl.num_slots;
  return FA_OK;
}

int fa_plan_work_host_buckets(const int32_t* indptr, const int32_t* last_page_len,
                              const int32_t* qo_indptr, int batch, int group, int num_kv_heads,
                              int page_size, int widest_tiles, const int* max_ctas_by_tiles,
                              int flags, int64_t min_own_units, int32_t* cta_offsets,
                              int32_t* segments, int32_t* merge, int* n_ctas, int* n_segments,
                              int* n_merge, int* n_buckets, int* bucket_tiles,
                              int* bucket_first_cta, int64_t* slot_columns) {
  if (!max_ctas_by_tiles || !cta_offsets || !segments || !merge || !n_ctas || !n_segments ||
      !n_merge || !n_buckets || !bucket_tiles || !bucket_first_cta || !slot_columns ||
      widest_tiles < 1 || widest_tiles > fadecode::kMaxTileBuckets)
    return FA_ERR_INVALID_ARG;
  fadecode::BucketPolicy pol;
  pol.group = group;
  pol.widest = widest_tiles;
  for (int t = 1; t <= widest_tiles; ++t) pol.max_ctas[t] = max_ctas_by_tiles[t - 1];
  pol.one_tile_own = (flags & 1) != 0;
  pol.all = (flags & 2) != 0;
  pol.min_own_units = min_own_units;
  pol.min_pages_per_cta = kMinPagesPerCta;
  pol.heads = true;
  WorkList wl;
  fadecode::BucketList bl;
  try {
    if (fadecode::build_bucket_work_list(indptr, last_page_len, qo_indptr, batch, num_kv_heads,
                                         page_size, pol, &wl, &bl) != 0)
      return FA_ERR_INVALID_ARG;
  } catch (const std::bad_alloc&) {
    return FA_ERR_INVALID_ARG;
  }
  *n_buckets = bl.num;
  *slot_columns = bl.slot_columns;
  for (int b = 0; b < fadecode::kMaxTileBuckets; ++b) {
    bucket_tiles[b] = b < bl.num ? bl.tiles[b] : 0;
    bucket_first_cta[b] = b < bl.num ? bl.cta_first[b] : -1;
  }
  *n_ctas = wl.num_ctas;
  *n_segments = (int)wl.segments.size();
  *n_merge = (int)wl.merge.size();
  if (bl.num == 0) return FA_OK;
  std::memcpy(cta_offsets, wl.cta_offsets.data(), sizeof(int32_t) * wl.cta_offsets.size());
  std::memcpy(segments, wl.segments.data(), sizeof(fadecode::Segment) * wl.segments.size());
  std::memcpy(merge, wl.merge.data(), sizeof(fadecode::MergeUnit) * wl.merge.size());
  return FA_OK;
}

int fa_plan_work_host(const int32_t* indptr, const int32_t* last_page_len, int batch,
                      int num_kv_heads, int page_size, int max_ctas, int min_pages_per_cta,
                      double pool_fraction, int32_t* cta_offsets, int32_t* segments, int32_t* merge, int* n_ctas,
                      int* n_segments, int* n_merge, int* n_slots) {
  if (!cta_offsets || !segments || !merge || !n_ctas || !n_segments || !n_merge || !n_slots)
    return FA_ERR_INVALID_ARG;
  WorkList wl;
  try {
    if (fadecode::build_work_list(indptr, last_page_len, batch, num_kv_heads, page_size,
                                  max_ctas, min_pages_per_cta, pool_fraction, &wl) != 0)
      return FA_ERR_INVALID_ARG;
  } catch (const std::bad_alloc&) {
    return FA_ERR_INVALID_ARG;
  }
  std::memcpy(cta_offsets, wl.cta_offsets.data(), sizeof(int32_t) * wl.cta_offsets.size());
  std::memcpy(segments, wl.segments.data(), sizeof(fadecode::Segment) * wl.segments.size());
  std::memcpy(merge, wl.merge.data(), sizeof(fadecode::MergeUnit) * wl.merge.size());
  *n_ctas = wl.num_ctas;
  *n_segments = (int)wl.segments.size();
  *n_merge = (int)wl.merge.size();
  *n_slots = wl.num_slots;
  return FA_OK;
}

static int plan_impl(const int32_t* indptr_host, const int32_t* indices_dev,
                     const int32_t* last_page_len_host, int batch, int q_len, int num_qo_heads,
                     int num_kv_heads, int head_dim, int page_size, fa_dtype q_dtype,
                     fa_dtype kv_dtype, void* workspace_dev, size_t workspace_bytes,
                     void* cuda_stream, fa_decode_plan_t* out_plan,
                     const int32_t* qo_indptr_host = nullptr);

int fa_decode_plan(const int32_t* indptr_host, const int32_t* indices_dev,
                   const int32_t* last_page_len_host, int batch, int num_qo_heads,
                   int num_kv_heads, int head_dim, int page_size, fa_dtype q_dtype,
                   fa_dtype kv_dtype, void* workspace_dev, size_t workspace_bytes,
                   void* cuda_stream, fa_decode_plan_t* out_plan) {
  return plan_impl(indptr_host, indices_dev, last_page_len_host, batch, 1, num_qo_heads,
                   num_kv_heads, head_dim, page_size, q_dtype, kv_dtype, workspace_dev,
                   workspace_bytes, cuda_stream, out_plan);
}

int fa_decode_plan_multi_token(const int32_t* indptr_host, const int32_t* indices_dev,
                               const int32_t* last_page_len_host, int batch, int q_len,
                               int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                               fa_dtype q_dtype, fa_dtype kv_dtype, void* workspace_dev,
                               size_t workspace_bytes, void* cuda_stream,
                               fa_decode_plan_t* out_plan) {
  if (q_len < 1) return FA_ERR_INVALID_ARG;
  if (batch >= 0 && num_kv_heads > 0 && num_qo_heads % num_kv_heads == 0 &&
      (num_qo_heads / num_kv_heads) * q_len > 8) {
    // more columns than one MMA tile: the kernels with ragged query rows,
    // every request holding q_len rows (the same q / o layout)
    std::vector<int32_t> qo;
    try {
      qo.resize((size_t)batch + 1);
    } catch (const std::bad_alloc&) {
      return FA_ERR_INVALID_ARG;
    }
    for (int i = 0; i <= batch; ++i) qo[i] = i * q_len;
    return plan_impl(indptr_host, indices_dev, last_page_len_host, batch, q_len, num_qo_heads,
                     num_kv_heads, head_dim, page_size, q_dtype, kv_dtype, workspace_dev,
                     workspace_bytes, cuda_stream, out_plan, qo.data());
  }
  return plan_impl(indptr_host, indices_dev, last_page_len_host, batch, q_len, num_qo_heads,
                   num_kv_heads, head_dim, page_size, q_dtype, kv_dtype, workspace_dev,
                   workspace_bytes, cuda_stream, out_plan);
}

int fa_decode_plan_ragged_q(const int32_t* indptr_host, const int32_t* indices_dev,
                            const int32_t* last_page_len_host, const int32_t* qo_indptr_host,
                            int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                            int page_size, fa_dtype q_dtype, fa_dtype kv_dtype,
                            void* workspace_dev, size_t workspace_bytes, void* cuda_stream,
                            fa_decode_plan_t* out_plan) {
  if (!qo_indptr_host || batch < 0) return FA_ERR_INVALID_ARG;
  int max_q = 1;
  for (int i = 0; i < batch; ++i) max_q = std::max(max_q, qo_indptr_host[i + 1] - qo_indptr_host[i]);
  return plan_impl(indptr_host, indices_dev, last_page_len_host, batch, max_q, num_qo_heads,
                   num_kv_heads, head_dim, page_size, q_dtype, kv_dtype, workspace_dev,
                   workspace_bytes, cuda_stream, out_plan, qo_indptr_host);
}

size_t fa_decode_workspace_size_ragged_q(int batch, int num_qo_heads, int num_kv_heads,
                                         int head_dim) {
  if (num_kv_heads <= 0 || num_qo_heads <= 0 || num_qo_heads % num_kv_heads) return 0;
  // the widest ragged kernel holds 32 columns (group x query tokens)
  const int G = num_qo_heads / num_kv_heads;
  const int max_q = G <= 32 ? 32 / G : 1;
  return fa_decode_workspace_size(batch, num_qo_heads * max_q, num_kv_heads, head_dim);
}

}  // extern "C"

namespace {

// Buckets for a ragged batch whose widest request takes the column split
// (more than 8 columns).  Request i needs t_i = ceil(G x n_i / 8) 8-column
// tiles (1 for n_i = 0).  A column split's warps each take every page of a
// request for 8 columns of their own, so the batch runs on the column split
// of as many warps as its widest request has tiles - two or three warps a
// CTA leave room for five or four CTAs per SM (a batch of 2 or 3 tiles a
// request: -15 % on an E4M3 cache, -2 to -6 % on a 16-bit one, against
// four warps).  With E4M3 KV the column split is bound by its arithmetic,
// and a CTA streams pages at the same rate however many of its warps have
// columns, so the requests of one tile take a launch of their own on the
// 8-column kernel (pages split over its warps) when they hold enough work
// to outweigh a launch's fixed time (spec_decode_ragged: 449 -> 413 us).
// A 16-bit column split streams near the copy rate already, and the
// 8-column kernel is no faster on those requests.  The work lists are
// built by fadecode::build_bucket_work_list; buckets run one after the
// other, widest first, each grid over the whole GPU.  Returns false (and
// leaves the plan alone) when one launch of the plan's own kernel is what
// remains, a kernel is not built or the plan does not fit the workspace.
bool plan_buckets(fa_decode_plan_s* plan, const int32_t* indptr, const int32_t* last,
                  const int32_t* qo, int batch, int sms, size_t workspace_bytes,
                  BucketMode mode) {
  const int G = plan->group;
  const int nc_max = G * plan->kern[kPlain].q_len;
  if (nc_max <= 8 || nc_max % 8 != 0 || nc_max / 8 > kMaxBuckets || 8 % G != 0) return false;
  fadecode::BucketPolicy pol;
  pol.group = G;
  pol.widest = nc_max / 8;
  DecodeKernel kern[kMaxBuckets + 1];
  for (int t = 1; t <= pol.widest; ++t) {
    if (!find_ragged_tiles_kernel(plan->q_dtype, plan->kv_dtype, plan->d, G, t, &kern[t]))
      return false;
    const int occ = std::min(kernel_occupancy(kern[t]), 8);
    if (occ <= 0) return false;
    pol.max_ctas[t] = sms * occ;
  }
  pol.one_tile_own = plan->kv_dtype == FA_DTYPE_E4M3;
  pol.min_own_units = (int64_t)kMinBucketUnitsPerSm * sms;
  pol.all = mode == BucketMode::kAll;
  pol.min_pages_per_cta = kMinPagesPerCta;
  pol.heads = heads_plan();
  WorkList w;
  fadecode::BucketList bl;
  if (fadecode::build_bucket_work_list(indptr, last, qo, batch, plan->hkv, plan->page_size, pol,
                                       &w, &bl) != 0 ||
      bl.num == 0)
    return false;
  w.num_slots = (int)((bl.slot_columns + nc_max - 1) / nc_max);
  const Layout L = make_layout(w.num_ctas, (int64_t)w.segments.size(), (int64_t)w.merge.size(),
                               w.num_slots, nc_max, plan->d, (int64_t)batch + 1);
  if (L.total > workspace_bytes) return false;
  plan->wl = std::move(w);
  plan->layout = L;
  plan->num_buckets = bl.num;
  for (int b = 0; b < bl.num; ++b) {
    fa_decode_plan_s::Bucket& bk = plan->bucket[b];
    bk.kern = kern[bl.tiles[b]];
    bk.tiles = bl.tiles[b];
    bk.cta_first = bl.cta_first[b];
    bk.num_ctas = bl.num_ctas[b];
    bk.merge_first = bl.merge_first[b];
    bk.num_merge = bl.num_merge[b];
  }
  return true;
}

}  // namespace

static int plan_impl(const int32_t* indptr_host, const int32_t* indices_dev,
                     const int32_t* last_page_len_host, int batch, int q_len, int num_qo_heads,
                     int num_kv_heads, int head_dim, int page_size, fa_dtype q_dtype,
                     fa_dtype kv_dtype, void* workspace_dev, size_t workspace_bytes,
                     void* cuda_stream, fa_decode_plan_t* out_plan,
                     const int32_t* qo_indptr_host) {
  if (!out_plan) return FA_ERR_INVALID_ARG;
  *out_plan = nullptr;
  if (!indptr_host || batch < 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      page_size <= 0 || num_qo_heads % num_kv_heads || !workspace_dev)
    return FA_ERR_INVALID_ARG;
  if (batch > 0 && !last_page_len_host) return FA_ERR_INVALID_ARG;
  if (indptr_host[batch] > 0 && !indices_dev) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace_dev) % kAlign) return FA_ERR_INVALID_ARG;
  if (dtype_size(q_dtype) == 0 || dtype_size(kv_dtype) == 0) return FA_ERR_INVALID_ARG;
  const int G = num_qo_heads / num_kv_heads;
  if (page_size != fadecode::kPageSize) return FA_ERR_UNSUPPORTED;
  const bool ragged = qo_indptr_host != nullptr;
  int64_t total_q = (int64_t)batch * q_len;
  if (ragged) {
    // request i has n_i = qo_indptr[i+1] - qo_indptr[i] query tokens, the
    // last n_i positions of its cache (0 allowed: it contributes no rows)
    if (qo_indptr_host[0] != 0) return FA_ERR_INVALID_ARG;
    for (int i = 0; i < batch; ++i) {
      const int64_t nq = (int64_t)qo_indptr_host[i + 1] - qo_indptr_host[i];
      const int64_t np = (int64_t)indptr_host[i + 1] - indptr_host[i];
      if (nq < 0 || nq > q_len) return FA_ERR_INVALID_ARG;
      if (nq == 0) continue;
      if (np <= 0 || last_page_len_host[i] < 1 || last_page_len_host[i] > page_size ||
          (np - 1) * page_size + last_page_len_host[i] < nq)
        return FA_ERR_INVALID_ARG;
    }
    total_q = qo_indptr_host[batch];
  } else if (q_len > 1) {
    // every request must hold its q_len draft tokens
    for (int i = 0; i < batch; ++i) {
      const int64_t np = (int64_t)indptr_host[i + 1] - indptr_host[i];
      if (np <= 0 || last_page_len_host[i] < 1 || last_page_len_host[i] > page_size ||
          (np - 1) * page_size + last_page_len_host[i] < q_len)
        return FA_ERR_INVALID_ARG;
    }
  }
  int dev = 0, sms = 0, occ = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  // The persistent grid must fit for every variant a run may launch.
  DecodeKernel kv[kNumVariants];
  bool has[kNumVariants] = {true, false, false};
  const int sel = select_kernels(q_dtype, kv_dtype, head_dim, G, q_len, kv, has, &occ, ragged);
  if (sel != FA_OK) return sel;
  // query tokens a partial state holds columns for: the kernel's bucket
  const int ql_kernel = kv[kPlain].q_len;

  fa_decode_plan_s* plan = new (std::nothrow) fa_decode_plan_s();
  if (!plan) return FA_ERR_INVALID_ARG;
  plan->device = dev;
  plan->batch = batch;
  plan->hq = num_qo_heads;
  plan->hkv = num_kv_heads;
  plan->d = head_dim;
  plan->page_size = page_size;
  plan->group = G;
  plan->q_dtype = q_dtype;
  plan->kv_dtype = kv_dtype;
  for (int v = 0; v < kNumVariants; ++v) {
    plan->kern[v] = kv[v];
    plan->has[v] = has[v];
  }
  plan->num_sms = sms;
  plan->ctas_per_sm = occ;
  plan->indices = indices_dev;
  plan->ws = static_cast<uint8_t*>(workspace_dev);
  plan->ws_bytes = workspace_bytes;
  plan->fused_merge = fused_merge_enabled();
  plan->q_len = ragged ? ql_kernel : q_len;
  plan->ragged_q = ragged;
  plan->total_q = total_q;

  int rc = FA_OK;
  try {
    const BucketMode bm = bucket_mode();
    const bool buckets = ragged && bm != BucketMode::kOff && pool_fraction() == 0.0 &&
                         plan_buckets(plan, indptr_host, last_page_len_host, qo_indptr_host,
                                      batch, sms, workspace_bytes, bm);
    // with the run-time pool if its partial states fit the workspace, else
    // static quotas only
    const bool heads = heads_plan() && pool_fraction() == 0.0;
    const double fractions[2] = {heads ? 0.0 : pool_fraction(), 0.0};
    rc = buckets ? FA_OK : FA_ERR_WORKSPACE_TOO_SMALL;
    for (double f : fractions) {
      if (buckets) break;
      if (fadecode::build_work_list(indptr_host, last_page_len_host, batch, num_kv_heads,
                                    page_size, sms * occ, kMinPagesPerCta, f, &plan->wl,
                                    heads) != 0) {
        rc = FA_ERR_INVALID_ARG;
        break;
      }
      const WorkList& w = plan->wl;
      plan->layout = make_layout(w.num_ctas, (int64_t)w.segments.size(),
                                 (int64_t)w.merge.size(), w.num_slots, G * plan->q_len, head_dim,
                                 ragged ? (int64_t)batch + 1 : 0);
      if (plan->layout.total <= workspace_bytes) {
        rc = FA_OK;
        break;
      }
      if (f == 0.0 || w.pool_pages == 0) break;
    }
  } catch (const std::bad_alloc&) {
    rc = FA_ERR_INVALID_ARG;
  }
  if (rc != FA_OK) {
    delete plan;
    return rc;
  }
  const WorkList& wl = plan->wl;
  plan->merge_flat.resize(wl.merge.size() * FA_MERGE_INTS);
  if (!wl.merge.empty())
    std::memcpy(plan->merge_flat.data(), wl.merge.data(), wl.merge.size() * sizeof(wl.merge[0]));

  // One host image of the metadata region, one copy into the workspace.
  std::vector<uint8_t> meta(plan->layout.meta_bytes, 0);
  std::memcpy(meta.data() + plan->layout.off_cta, wl.cta_offsets.data(),
              sizeof(int32_t) * wl.cta_offsets.size());
  if (!wl.segments.empty())
    std::memcpy(meta.data() + plan->layout.off_seg, wl.segments.data(),
                sizeof(fadecode::Segment) * wl.segments.size());
  if (!wl.merge.empty())
    std::memcpy(meta.data() + plan->layout.off_merge, wl.merge.data(),
                sizeof(fadecode::MergeUnit) * wl.merge.size());
  if (ragged)
    std::memcpy(meta.data() + plan->layout.off_qo, qo_indptr_host,
                sizeof(int32_t) * ((size_t)batch + 1));
  if (fadecode::upload_async(plan->ws, meta.data(), meta.size(),
                             static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) {
    delete plan;
    return FA_ERR_CUDA;
  }
  *out_plan = plan;
  return FA_OK;
}

extern "C" {

int fa_decode_run(fa_decode_plan_t plan, const void* q, const void* paged_kv, int64_t num_pages,
                  float sm_scale, float k_scale, float v_scale, void* o, float* lse,
                  void* cuda_stream) {
  if (!plan) return FA_ERR_INVALID_ARG;
  return run_impl(plan, kPlain, q, paged_kv, num_pages, sm_scale, k_scale, v_scale, nullptr,
                  nullptr, 0.f, o, lse, cuda_stream);
}

int fa_decode_run_unified_max(fa_decode_plan_t plan, const void* q, const void* paged_kv,
                              int64_t num_pages, float sm_scale, float k_scale, float v_scale,
                              float max_bound, void* o, float* lse, void* cuda_stream) {
  if (!plan) return FA_ERR_INVALID_ARG;
  if (!plan->has[kUnifiedMax]) return FA_ERR_UNSUPPORTED;
  // the reference enters the kernel in log2 units and must stay finite there
  if (!(std::fabs(max_bound) <= 1e30f)) return FA_ERR_INVALID_ARG;
  return run_impl(plan, kUnifiedMax, q, paged_kv, num_pages, sm_scale, k_scale, v_scale,
                  nullptr, nullptr, max_bound, o, lse, cuda_stream);
}

int fa_decode_unified_max_fallbacks(fa_decode_plan_t plan, void* cuda_stream, int* count) {
  if (!plan || !count) return FA_ERR_INVALID_ARG;
  int word = 0;
  int* dword = reinterpret_cast<int*>(plan->ws + plan->layout.off_umc);
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess ||
      cudaMemcpy(&word, dword, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(dword, 0, sizeof word) != cudaSuccess)
    return FA_ERR_CUDA;
  *count = word;
  return FA_OK;
}

int fa_decode_run_token_scales(fa_decode_plan_t plan, const void* q, const void* paged_kv,
                               int64_t num_pages, float sm_scale, const float* k_scales,
                               const float* v_scales, void* o, float* lse, void* cuda_stream) {
  if (!plan) return FA_ERR_INVALID_ARG;
  if (plan->kv_dtype != FA_DTYPE_E4M3 || !plan->has[kTokenScales]) return FA_ERR_UNSUPPORTED;
  if (plan->batch > 0 && (!k_scales || !v_scales)) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(k_scales) % 16 || reinterpret_cast<uintptr_t>(v_scales) % 16)
    return FA_ERR_INVALID_ARG;
  return run_impl(plan, kTokenScales, q, paged_kv, num_pages, sm_scale, 1.f, 1.f, k_scales,
                  v_scales, 0.f, o, lse, cuda_stream);
}

int fa_decode_run_head_scales(fa_decode_plan_t plan, const void* q, const void* paged_kv,
                              int64_t num_pages, float sm_scale, const float* k_head_scales,
                              const float* v_head_scales, void* o, float* lse,
                              void* cuda_stream) {
  if (!plan) return FA_ERR_INVALID_ARG;
  if (plan->kv_dtype != FA_DTYPE_E4M3) return FA_ERR_UNSUPPORTED;
  if (plan->batch > 0 && (!k_head_scales || !v_head_scales)) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(k_head_scales) % 4 ||
      reinterpret_cast<uintptr_t>(v_head_scales) % 4)
    return FA_ERR_INVALID_ARG;
  return run_impl(plan, kPlain, q, paged_kv, num_pages, sm_scale, 1.f, 1.f, nullptr, nullptr,
                  0.f, o, lse, cuda_stream, k_head_scales, v_head_scales);
}

int fa_merge_states(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b,
                    void* o_out, float* lse_out, int n, int num_heads, int head_dim,
                    fa_dtype dtype, void* cuda_stream) {
  if (n < 0 || num_heads <= 0 || head_dim <= 0) return FA_ERR_INVALID_ARG;
  if (n == 0) return FA_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !o_out || !lse_out) return FA_ERR_INVALID_ARG;
  if (head_dim > 1024 || dtype == FA_DTYPE_E4M3 || dtype_size(dtype) == 0)
    return FA_ERR_UNSUPPORTED;
  return fadecode::launch_merge_states(o_a, lse_a, o_b, lse_b, o_out, lse_out,
                                       (int64_t)n * num_heads, head_dim, dtype, cuda_stream);
}

int fa_decode_plan_destroy(fa_decode_plan_t plan) {
  delete plan;
  return FA_OK;
}

int fa_decode_plan_get_info(fa_decode_plan_t plan, fa_plan_info* info) {
  if (!plan || !info) return FA_ERR_INVALID_ARG;
  fa_plan_info i;
  std::memset(&i, 0, sizeof i);
  i.batch = plan->batch;
  i.num_qo_heads = plan->hq;
  i.num_kv_heads = plan->hkv;
  i.head_dim = plan->d;
  i.page_size = plan->page_size;
  i.num_ctas = plan->wl.num_ctas;
  i.ctas_per_sm = plan->ctas_per_sm;
  i.num_sms = plan->num_sms;
  i.num_segments = (int)plan->wl.segments.size();
  i.num_merge_units = (int)plan->wl.merge.size();
  i.num_partial_slots = plan->wl.num_slots;
  i.threads_per_cta = plan->kern[kPlain].threads;
  i.smem_bytes_per_cta = plan->kern[kPlain].smem_bytes;
  i.stages = plan->kern[kPlain].stages;
  i.total_pages = plan->wl.total_pages;
  i.total_tokens = plan->wl.total_tokens;
  i.workspace_bytes_used = plan->layout.total;
  i.plan_upload_bytes = plan->layout.meta_bytes;
  i.tensor_cores = plan->kern[kPlain].tensor_cores ? 1 : 0;
  i.fused_merge = plan->fused_merge ? 1 : 0;
  i.q_len = plan->q_len;
  i.ragged_q = plan->ragged_q ? 1 : 0;
  i.total_q_rows = plan->total_q;
  i.unified_max = plan->has[kUnifiedMax] ? 1 : 0;
  i.num_pool_segments = plan->wl.pool_count();
  i.pool_pages = plan->wl.pool_pages;
  i.num_buckets = plan->num_buckets > 0 ? plan->num_buckets : 1;
  for (int b = 0; b < kMaxBuckets; ++b) {
    i.bucket_first_cta[b] = b < plan->num_buckets ? plan->bucket[b].cta_first : (b ? -1 : 0);
    i.bucket_q_len[b] = b < plan->num_buckets ? plan->bucket[b].kern.q_len
                                              : (b ? 0 : plan->q_len);
  }
  *info = i;
  return FA_OK;
}

int fa_decode_plan_get_work(fa_decode_plan_t plan, const int32_t** cta_offsets,
                            const int32_t** segments, const int32_t** merge) {
  if (!plan || !cta_offsets || !segments || !merge) return FA_ERR_INVALID_ARG;
  *cta_offsets = plan->wl.cta_offsets.data();
  *segments = reinterpret_cast<const int32_t*>(plan->wl.segments.data());
  *merge = plan->merge_flat.data();
  return FA_OK;
}

int fa_decode_check(fa_decode_plan_t plan, void* cuda_stream, int* flags) {
  if (!plan || !flags) return FA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int word = 0;
  int* dword = reinterpret_cast<int*>(plan->ws + plan->layout.off_err);
  if (cudaStreamSynchronize(st) != cudaSuccess ||
      cudaMemcpy(&word, dword, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(dword, 0, sizeof word) != cudaSuccess)
    return FA_ERR_CUDA;
  // A run that gave up waiting may leave the pool and merge counters short
  // of their re-armed zeros: clear them for the next run.
  if (word &&
      (cudaMemset(plan->ws + plan->layout.off_pool, 0, 2 * sizeof(int)) != cudaSuccess ||
       cudaMemset(plan->ws + plan->layout.off_count, 0,
                  sizeof(int32_t) * plan->wl.merge.size()) != cudaSuccess))
    return FA_ERR_CUDA;
  *flags = word;
  return word ? FA_ERR_DEVICE_CHECK : FA_OK;
}

int fa_decode_set_timing_events(fa_decode_plan_t plan, void* ev_before, void* ev_after) {
  if (!plan) return FA_ERR_INVALID_ARG;
  plan->ev_before = static_cast<cudaEvent_t>(ev_before);
  plan->ev_after = static_cast<cudaEvent_t>(ev_after);
  return FA_OK;
}

int fa_library_get_stats(fa_library_stats* stats) {
  if (!stats) return FA_ERR_INVALID_ARG;
  fa_library_stats s;
  std::memset(&s, 0, sizeof s);
  fadecode::staging_stats(&s.pinned_host_allocations, &s.pinned_host_bytes, &s.staged_uploads);
  *stats = s;
  return FA_OK;
}

}  // extern "C"

// ---- the allocation-free path behind fa_decode_static ---------------------
//
// The plan is built into fixed host arrays (no pool: a pool's chunk list is
// sized at run time), laid out as the workspace's metadata image in a
// file-scope host buffer, and copied into the caller-less scratch array with
// one cudaMemcpyAsync from that pageable buffer: the driver stages a copy
// from pageable memory before the call returns, so the buffer is free for
// the next call at once and nothing is pinned or allocated.  The launch
// state lives on the stack.  One mutex serialises the host side of calls.
namespace {

constexpr int kStaticMaxCtas = 8192;
constexpr int kStaticMaxSegments = (int)(FA_STATIC_SCRATCH_BYTES / sizeof(fadecode::Segment));
constexpr int kStaticMaxMerge = kStaticMaxCtas;

std::mutex g_static_mu;
int32_t g_static_cta[kStaticMaxCtas + 1];
fadecode::Segment g_static_seg[kStaticMaxSegments];
fadecode::MergeUnit g_static_merge[kStaticMaxMerge];
alignas(256) uint8_t g_static_image[FA_STATIC_SCRATCH_BYTES];

}  // namespace

namespace fadecode {

int static_decode(void* scratch, size_t scratch_bytes, const int32_t* indptr_host,
                  const int32_t* indices_dev, const int32_t* last_page_len_host, int batch,
                  int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                  fa_dtype q_dtype, fa_dtype kv_dtype, const void* q, const void* paged_kv,
                  int64_t num_pages, float sm_scale, float k_scale, float v_scale, void* o,
                  float* lse, void* cuda_stream) {
  if (!scratch || !indptr_host || batch < 0 || num_qo_heads <= 0 || num_kv_heads <= 0 ||
      head_dim <= 0 || page_size <= 0 || num_qo_heads % num_kv_heads)
    return FA_ERR_INVALID_ARG;
  if (batch > 0 && !last_page_len_host) return FA_ERR_INVALID_ARG;
  if (indptr_host[batch] > 0 && !indices_dev) return FA_ERR_INVALID_ARG;
  if (dtype_size(q_dtype) == 0 || dtype_size(kv_dtype) == 0) return FA_ERR_INVALID_ARG;
  if (page_size != fadecode::kPageSize) return FA_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  // the upload below is a copy from pageable memory, which a stream capture
  // cannot record
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return FA_ERR_CUDA;
  if (cap != cudaStreamCaptureStatusNone) return FA_ERR_UNSUPPORTED;
  const int G = num_qo_heads / num_kv_heads;

  int dev = 0, sms = 0, occ = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  DecodeKernel kv[kNumVariants];
  bool has[kNumVariants] = {true, false, false};
  // the same kernels and grid as fa_decode_plan picks, so both paths give
  // bitwise the same result
  const int sel = select_kernels(q_dtype, kv_dtype, head_dim, G, 1, kv, has, &occ);
  if (sel != FA_OK) return sel;

  std::lock_guard<std::mutex> lock(g_static_mu);
  FixedWorkList fw;
  fw.cta_offsets = g_static_cta;
  fw.segments = g_static_seg;
  fw.merge = g_static_merge;
  fw.cta_capacity = kStaticMaxCtas;
  fw.segment_capacity = kStaticMaxSegments;
  fw.merge_capacity = kStaticMaxMerge;
  const int prc = build_work_list_fixed(indptr_host, last_page_len_host, batch, num_kv_heads,
                                        page_size, std::min(sms * occ, kStaticMaxCtas),
                                        kMinPagesPerCta, &fw, heads_plan());
  if (prc == -2) return FA_ERR_WORKSPACE_TOO_SMALL;
  if (prc != 0) return FA_ERR_INVALID_ARG;
  const Layout L = make_layout(fw.num_ctas, fw.num_segments, fw.num_merge, fw.num_slots, G,
                               head_dim);
  if (L.total > scratch_bytes || L.meta_bytes > sizeof(g_static_image))
    return FA_ERR_WORKSPACE_TOO_SMALL;
  if (batch == 0) return FA_OK;

  std::memset(g_static_image, 0, L.meta_bytes);
  std::memcpy(g_static_image + L.off_cta, g_static_cta,
              sizeof(int32_t) * ((size_t)fw.num_ctas + 1));
  std::memcpy(g_static_image + L.off_seg, g_static_seg,
              sizeof(Segment) * (size_t)fw.num_segments);
  std::memcpy(g_static_image + L.off_merge, g_static_merge,
              sizeof(MergeUnit) * (size_t)fw.num_merge);
  if (cudaMemcpyAsync(scratch, g_static_image, L.meta_bytes, cudaMemcpyHostToDevice, st) !=
      cudaSuccess)
    return FA_ERR_CUDA;

  MapCache map;
  LaunchView lv;
  lv.batch = batch;
  lv.hq = num_qo_heads;
  lv.hkv = num_kv_heads;
  lv.d = head_dim;
  lv.page_size = page_size;
  lv.q_len = 1;
  lv.q_dtype = q_dtype;
  lv.kv_dtype = kv_dtype;
  lv.kern = &kv[kPlain];
  lv.map = &map;
  lv.indices = indices_dev;
  lv.ws = static_cast<uint8_t*>(scratch);
  lv.layout = L;
  lv.num_ctas = fw.num_ctas;
  lv.num_merge = fw.num_merge;
  lv.fused_merge = fused_merge_enabled();
  return launch_decode(lv, q, paged_kv, num_pages, sm_scale, k_scale, v_scale, nullptr,
                       nullptr, 0.f, o, lse, cuda_stream);
}

}  // namespace fadecode

static int run_impl(fa_decode_plan_s* plan, Variant variant, const void* q,
                    const void* paged_kv, int64_t num_pages, float sm_scale, float k_scale,
                    float v_scale, const float* k_scales, const float* v_scales,
                    float max_bound, void* o, float* lse, void* cuda_stream,
                    const float* head_k_scales, const float* head_v_scales) {
  LaunchView lv;
  lv.batch = plan->batch;
  lv.hq = plan->hq;
  lv.hkv = plan->hkv;
  lv.d = plan->d;
  lv.page_size = plan->page_size;
  lv.q_len = plan->q_len;
  lv.q_dtype = plan->q_dtype;
  lv.kv_dtype = plan->kv_dtype;
  lv.kern = &plan->kern[variant];
  lv.map = &plan->map[variant];
  lv.indices = plan->indices;
  lv.ws = plan->ws;
  lv.layout = plan->layout;
  lv.num_ctas = plan->wl.num_ctas;
  lv.num_merge = (int)plan->wl.merge.size();
  lv.pool_begin = plan->wl.pool_begin();
  lv.pool_count = plan->wl.pool_count();
  lv.fused_merge = plan->fused_merge;
  lv.ragged_q = plan->ragged_q;
  lv.ev_before = plan->ev_before;
  lv.ev_after = plan->ev_after;
  if (plan->num_buckets == 0)
    return launch_decode(lv, q, paged_kv, num_pages, sm_scale, k_scale, v_scale, k_scales,
                         v_scales, max_bound, o, lse, cuda_stream, head_k_scales,
                         head_v_scales);
  // one launch per bucket, in order; the timing events (if set) bracket all
  if (variant != kPlain) return FA_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const bool timed = plan->batch > 0 && plan->ev_before && plan->ev_after;
  if (timed && cudaEventRecord(plan->ev_before, st) != cudaSuccess) return FA_ERR_CUDA;
  lv.ev_before = lv.ev_after = nullptr;
  for (int b = 0; b < plan->num_buckets; ++b) {
    fa_decode_plan_s::Bucket& bk = plan->bucket[b];
    lv.kern = &bk.kern;
    lv.map = &bk.map;
    lv.q_len = bk.kern.q_len;
    lv.cta_first = bk.cta_first;
    lv.num_ctas = bk.num_ctas;
    lv.merge_first = bk.merge_first;
    lv.num_merge = bk.num_merge;
    const int rc = launch_decode(lv, q, paged_kv, num_pages, sm_scale, k_scale, v_scale,
                                 k_scales, v_scales, max_bound, o, lse, cuda_stream,
                                 head_k_scales, head_v_scales);
    if (rc != FA_OK) return rc;
  }
  if (timed && cudaEventRecord(plan->ev_after, st) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

namespace {

int launch_decode(const LaunchView& lv, const void* q, const void* paged_kv, int64_t num_pages,
                  float sm_scale, float k_scale, float v_scale, const float* k_scales,
                  const float* v_scales, float max_bound, void* o, float* lse,
                  void* cuda_stream, const float* head_k_scales,
                  const float* head_v_scales) {
  if (lv.batch == 0) return FA_OK;
  if (!q || !paged_kv || !o || num_pages <= 0) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(paged_kv) % 16 || reinterpret_cast<uintptr_t>(q) % 16)
    return FA_ERR_INVALID_ARG;
  if (2 * num_pages > (int64_t)0xffffffffLL) return FA_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const DecodeKernel& kern = *lv.kern;
  MapCache& mc = *lv.map;
  const int D = lv.d;
  int rc = kv_tensor_map(&mc, kern, lv.kv_dtype, paged_kv, num_pages, D, lv.hkv, lv.page_size);
  if (rc != FA_OK) return rc;

  if (!(sm_scale > 0.f)) sm_scale = 1.0f / std::sqrt((float)D);
  uint8_t* ws = lv.ws;
  const Layout& L = lv.layout;
  DecodeParams prm;
  std::memset(&prm, 0, sizeof prm);
  prm.q = q;
  prm.o = o;
  prm.lse = lse;
  prm.indices = lv.indices;
  prm.cta_offsets = reinterpret_cast<const int32_t*>(ws + L.off_cta) + lv.cta_first;
  prm.segments = reinterpret_cast<const int32_t*>(ws + L.off_seg);
  prm.part_o = reinterpret_cast<float*>(ws + L.off_part_o);
  prm.part_lse = reinterpret_cast<float*>(ws + L.off_part_lse);
  prm.err = reinterpret_cast<int*>(ws + L.off_err);
  prm.merge = reinterpret_cast<const int32_t*>(ws + L.off_merge);
  prm.merge_count = reinterpret_cast<int*>(ws + L.off_count);
  prm.fused_merge = lv.fused_merge ? 1 : 0;
  prm.k_scales = k_scales;
  prm.v_scales = v_scales;
  prm.head_k_scales = head_k_scales;
  prm.head_v_scales = head_v_scales;
  prm.num_pages = num_pages;
  prm.num_qo_heads = lv.hq;
  prm.num_kv_heads = lv.hkv;
  prm.q_len = lv.q_len;
  prm.qo_indptr = lv.ragged_q ? reinterpret_cast<const int32_t*>(ws + L.off_qo) : nullptr;
  prm.q_row_bytes = D * dtype_size(lv.q_dtype);
  prm.kv = paged_kv;
  prm.kv_row_bytes = D * dtype_size(lv.kv_dtype);
  prm.q_scale = sm_scale * k_scale * kLog2e;
  prm.v_scale = v_scale;
  prm.max_bound = max_bound * kLog2e;
  prm.um_fallbacks = reinterpret_cast<int*>(ws + L.off_umc);
  prm.pool_begin = lv.pool_begin;
  prm.pool_count = lv.pool_count;
  prm.pool_claim = reinterpret_cast<int*>(ws + L.off_pool);
  prm.pool_done = prm.pool_claim + 1;

  const bool timed = lv.ev_before && lv.ev_after;
  if (timed && cudaEventRecord(lv.ev_before, st) != cudaSuccess) return FA_ERR_CUDA;
  void* args[2] = {&mc.tmap, &prm};
  // A programmatic dependent launch where the stream's previous decode
  // launch was this kernel: its CTAs may then be placed while that launch
  // drains, each in a slot one of its CTAs left; they read nothing global
  // before it has completed (griddepcontrol.wait).  After another decode
  // kernel, an ordinary launch (see dependent_launch_ok).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(lv.num_ctas);
  cfg.blockDim = dim3(kern.threads);
  cfg.dynamicSmemBytes = (size_t)kern.smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent_launch_ok(st, kern.func) ? 1 : 0;
  if (cudaLaunchKernelExC(&cfg, kern.func, args) != cudaSuccess) return FA_ERR_CUDA;
  if (timed && cudaEventRecord(lv.ev_after, st) != cudaSuccess) return FA_ERR_CUDA;
  if (!lv.fused_merge && lv.num_merge > 0) {
    MergeParams mp;
    mp.merge = reinterpret_cast<const int32_t*>(ws + L.off_merge) +
               (size_t)lv.merge_first * FA_MERGE_INTS;
    mp.qo_indptr = prm.qo_indptr;
    mp.part_o = prm.part_o;
    mp.part_lse = prm.part_lse;
    mp.o = o;
    mp.lse = lse;
    mp.num_qo_heads = lv.hq;
    void* margs[1] = {&mp};
    if (cudaLaunchKernel(kern.merge_func, dim3((unsigned)lv.num_merge), dim3(128), margs, 0,
                         st) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace
