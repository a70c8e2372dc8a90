// Split-KV paged decode attention for sm_103a.
//
// One persistent CTA per planner chunk list (see planner.cpp).  Inside a CTA:
//  - warp NW (the producer) walks the CTA's segments (then, with a run-time
//    pool, the pool segments it claims) page by page, reads each
//    page id from the index table and issues one 4-D TMA tensor copy per page
//    that brings the page's K and V rows of one kv head ([2][16][D]) into a
//    ring of S shared-memory stages, signalled through mbarriers;
//  - warps 0..NW-1 (consumers) take the pages round-robin by their position
//    k in the CTA's page stream: page k lands in stage k % S and is consumed by
//    warp k % NW.  S is a multiple of NW, so every stage belongs to one warp,
//    which waits on that stage's phases strictly in order (a parity wait can
//    only tell the current phase from the previous one, so two consumers of
//    one stage could mistake an old phase for a new one).  For each page a
//    warp computes the scores of all G query heads of the kv head's group
//    from one read of each K row (the tile is reused across the group), folds
//    them into its running softmax state with the online-softmax recurrence,
//    and accumulates P.V from one read of each V row;
//  - at the end of a segment the NW warp states are combined with the merge
//    rule and written either as the final o/lse or as an fp32 partial state;
//    the CTA that completes a split unit folds its partial states (or, on
//    request, a separate merge kernel does).
// The online-softmax update, the warp combine and the split merge are all the
// same recurrence applied at three levels, as section "FlashDecoding - the
// split-KV trick" of the page "FlashDecoding + FlashInfer - the decode-time
// attention story" describes (tile level in the main kernel, split level in
// the reduction).  Scores are kept in the log2 domain: q is pre-multiplied by
// sm_scale * k_scale * log2(e), so exp(s - m) becomes exp2(s' - m').
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <type_traits>

#include "kernels.h"

namespace fadecode {
namespace dev {

constexpr float kLn2 = 0.693147180559945309f;
// Upper bound on any single pipeline wait; a wait that runs out sets bit 1 of
// the device-check word and the CTA finishes without waiting again.
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* addr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(addr));
}

// Fetch a TMA descriptor into the descriptor cache ahead of its first use.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Programmatic dependent launch: let the next grid in the stream begin
// launching / wait until the grid this one depends on has completed and its
// memory is visible (both no-ops for an ordinary launch).
__device__ __forceinline__ void grid_dependency_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait without the abort short-cut: true if the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
  return true;
}

// Bounded wait.  Once `aborted` is set (an earlier wait ran out) it returns
// at once so that the CTA drains instead of hanging.
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity,
                                          bool& aborted, int* err) {
  if (aborted || mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
      aborted = true;
      atomicOr(err, 2);
      return;
    }
  }
}

// Hand a ring stage back to the producer once this warp has read it with
// generic-proxy loads (ld.shared, ldmatrix).  The producer refills the stage
// with a TMA copy, an async-proxy write; without a proxy fence between the
// reads and the release, that write can land before the reads are
// performed, and the warp then reads part of the next page (seen on GB300
// as V bytes of the next page under correct K bytes, a few units per
// hundred thousand on the E4M3 consumer with thousands of short segments;
// none with the fence).
// All lanes fence, then lane 0 arrives once the warp has converged.
__device__ __forceinline__ void release_stage(uint32_t empty_bar, int lane) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
  if (lane == 0) mbar_arrive(empty_bar);
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map,
                                            int c0, int c1, int c2, int c3,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(bar), "l"(policy)
      : "memory");
}

// Contiguous global -> shared copy of `bytes` (multiple of 16, both
// addresses 16-byte aligned) completing on mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// 16 bytes global -> shared through the load path (cp.async, L1 bypassed);
// both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}

// One of the mbarrier's expected arrivals, made once this thread's earlier
// cp.async copies have landed.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- element conversion -------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t w) {
  __half2 h;
  memcpy(&h, &w, sizeof(h));
  return __half22float2(h);
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t w) {
  __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w), __NV_E4M3);
  __half2 h(hr);
  return __half22float2(h);
}

// VEC elements of type T starting at p (16 or 8 bytes), widened to float.
template <typename T, int VEC>
struct VecLoad;

template <>
struct VecLoad<float, 4> {
  static constexpr int kBytes = 16;
  __device__ __forceinline__ static void load(const void* p, float (&f)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
};

template <>
struct VecLoad<__nv_bfloat16, 8> {
  static constexpr int kBytes = 16;
  __device__ __forceinline__ static void load(const void* p, float (&f)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
  }
};

template <>
struct VecLoad<__half, 8> {
  static constexpr int kBytes = 16;
  __device__ __forceinline__ static void load(const void* p, float (&f)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    float2 a = half2_bits_to_float2(v.x), b = half2_bits_to_float2(v.y);
    float2 c = half2_bits_to_float2(v.z), d = half2_bits_to_float2(v.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
};

template <>
struct VecLoad<__nv_fp8_e4m3, 8> {
  static constexpr int kBytes = 8;
  __device__ __forceinline__ static void load(const void* p, float (&f)[8]) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    float2 a = e4m3x2_to_float2((uint16_t)(v.x & 0xffff));
    float2 b = e4m3x2_to_float2((uint16_t)(v.x >> 16));
    float2 c = e4m3x2_to_float2((uint16_t)(v.y & 0xffff));
    float2 d = e4m3x2_to_float2((uint16_t)(v.y >> 16));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
};

// q is read straight from global memory (it is small and L2-resident).
template <typename T, int VEC>
__device__ __forceinline__ void load_q(const T* p, float (&f)[VEC]) {
  static_assert(VEC * sizeof(T) == 16 || (VEC == 8 && sizeof(T) == 4),
                "q vector must be 16 or 32 bytes");
  if constexpr (sizeof(T) == 4 && VEC == 8) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  } else if constexpr (sizeof(T) == 4) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  } else {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        f[2 * i] = bf16_lo(w[i]);
        f[2 * i + 1] = bf16_hi(w[i]);
      } else {
        float2 x = half2_bits_to_float2(w[i]);
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
      }
    }
  }
}

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_float(__half x) { return __half2float(x); }

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }

// Sum v[0..G) over the LPR lanes of a row group and leave lane c holding the
// total of head c / (LPR / G): each halving step exchanges half of the
// remaining values with the partner lane instead of reducing all of them.
template <int G, int LPR>
__device__ __forceinline__ float reduce_scatter(float (&v)[G], int c) {
  static_assert(G >= 1 && G <= LPR, "group larger than a row group");
  int n = G;
#pragma unroll
  for (int off = LPR / 2; off >= LPR / G && off >= 1; off >>= 1) {
    if (n == 1) break;
    const bool upper = (c & off) != 0;
#pragma unroll
    for (int i = 0; i < G / 2; ++i) {
      if (i < n / 2) {
        const float send = upper ? v[i] : v[i + n / 2];
        const float keep = upper ? v[i + n / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
    n >>= 1;
  }
#pragma unroll
  for (int off = LPR / (2 * G); off >= 1; off >>= 1)
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
  return v[0];
}

}  // namespace dev

// Pool segments claimed at run time travel from the producer warp to the
// consumer warps through this ring in shared memory.
constexpr int kSegRing = 4;
struct SegQueue {
  uint64_t full[kSegRing];   // producer -> consumers, one arrival
  uint64_t empty[kSegRing];  // consumers -> producer, one arrival per consumer warp
  int seg[kSegRing];         // segment index, -1 once the pool is empty
};
constexpr int kSegQueueBytes = (int)((sizeof(SegQueue) + 15) / 16 * 16);

__device__ __forceinline__ void seg_queue_init(SegQueue* q, int consumer_warps) {
  for (int i = 0; i < kSegRing; ++i) {
    dev::mbar_init(dev::smem_addr(&q->full[i]), 1);
    dev::mbar_init(dev::smem_addr(&q->empty[i]), consumer_warps);
  }
}

// q rows of request `req` (first row and count): ragged from qo_indptr (plan
// data, uploaded with the work list) or q_len per request.
__device__ __forceinline__ int2 request_q_rows(const DecodeParams& p, int req) {
  if (p.qo_indptr) {
    const int a = p.qo_indptr[req];
    return make_int2(a, p.qo_indptr[req + 1] - a);
  }
  return make_int2(req * p.q_len, p.q_len);
}

// Bring one segment's q rows (G heads of each of its request's query
// tokens) into L2, 128-byte lines spread over the warp's lanes.
__device__ __forceinline__ void prefetch_q_rows(const DecodeParams& p, int req, int kvh, int lane) {
  const int G = p.num_qo_heads / p.num_kv_heads;
  const int lines = (G * p.q_row_bytes + 127) / 128;  // one query token's rows
  const int2 qr = request_q_rows(p, req);
  for (int i = 0; i < qr.y; ++i) {
    const char* rows = static_cast<const char*>(p.q) +
                       (((size_t)qr.x + i) * p.num_qo_heads + (size_t)kvh * G) * p.q_row_bytes;
    for (int l = lane; l < lines; l += 32) dev::prefetch_l2(rows + (size_t)l * 128);
  }
}

// Before a programmatic dependent launch's wait: the CTA's first segment
// record (plan data) and, into L2, the page ids of its first 64 pages, the
// K and V rows of its first two pages and its q rows - data a preceding
// kernel may still be writing.  A prefetch only warms L2, where that
// kernel's writes land, so what is read after the wait is current; the two
// page ids are read past L1 (a stale id only wastes its prefetch).  Run by
// the producer warp.
__device__ __forceinline__ void prefetch_first_segment(const DecodeParams& p, int si, int lane) {
  const int4 sa = *reinterpret_cast<const int4*>(p.segments + 8 * si);
  const int kvh = sa.y, pb = sa.z, pe = sa.w;
  if (lane < 2 && pb + 32 * lane < pe) dev::prefetch_l2(p.indices + pb + 32 * lane);
  if (p.kv != nullptr) {
    const int lines = (p.kv_row_bytes + 127) / 128;
    const int kv = lane >> 4, t = lane & 15;  // one row of K or V per lane
    for (int i = 0; i < 2 && pb + i < pe; ++i) {
      const int id = __ldcg(p.indices + pb + i);
      if (id < 0 || (int64_t)id >= p.num_pages) continue;
      const char* row = static_cast<const char*>(p.kv) +
                        ((((size_t)id * 2 + kv) * kPageSize + t) * p.num_kv_heads + kvh) *
                            (size_t)p.kv_row_bytes;
      for (int l = 0; l < lines; ++l) dev::prefetch_l2(row + (size_t)l * 128);
    }
  }
  if (p.q_row_bytes > 0) prefetch_q_rows(p, sa.x, kvh, lane);
}

// Producer warp: walks the CTA's segments page by page, reads the page ids
// through the index table (32 at a time) and issues, per page, BOXES 4-D TMA
// tensor copies (box b starts at element b * BOX_X of a row and lands at
// b * BOX_BYTES in the stage) completing on the stage's "full" barrier.  Page
// k of the stream goes to stage k % S once the stage's previous page has been
// released.  Ends by waiting (bounded) for its last copies to land.
// With a queue, after its static segments the warp claims pool segments one
// at a time and passes each (then -1) to the consumers through the queue; a
// pool segment starts on a stream position that is a multiple of `align`
// (empty stages fill the gap), so that the consumer warps split its pages the
// same way whichever CTA claims it.
// With SCALES, each page also brings the 16 per-token K scales and the 16 V
// scales of its kv head (64 contiguous bytes each) into scales[stage][0..31]:
// lanes 0-7 copy 16 bytes each with cp.async (the load path, which keeps
// these small rows off the copy engine the page itself goes through), and
// the stage's "full" barrier counts their arrivals as well (kScaleLanes + 1).
constexpr int kScaleLanes = 8;  // producer lanes that copy a page's scales

template <int S, int STAGE_BYTES, int BOXES, int BOX_X, int BOX_BYTES, bool SCALES = false>
__device__ __forceinline__ void produce_pages(const CUtensorMap* map, const DecodeParams& p,
                                              int seg_begin, int seg_end, uint8_t* ring,
                                              uint64_t* full, uint64_t* empty, int lane,
                                              float* scales = nullptr, SegQueue* queue = nullptr,
                                              int align = 1) {
  bool aborted = false;
  // the descriptor loads while the first segment and its page ids are read
  if (lane == 0) dev::prefetch_tensormap(map);
  const uint64_t policy = dev::evict_first_policy();
  int k = 0, claimed = 0;
  // lane 0 claims one pool segment ahead - the first while it issues the
  // copies of its last static segment - so that a claim's round trip
  // overlaps the copies of the segment before it
  const bool pooled = queue && p.pool_count > 0;
  int ahead = -1;
  bool claiming = false;
  for (int si = seg_begin;; ++si) {
    if (pooled && !claiming && si >= seg_end - 1) {
      claiming = true;
      if (lane == 0) ahead = atomicAdd(p.pool_claim, 1);
    }
    if (si >= seg_end) {
      if (!pooled) break;
      int idx = p.pool_count;
      if (lane == 0 && !aborted) {
        idx = ahead;
        if (idx < p.pool_count) ahead = atomicAdd(p.pool_claim, 1);
      }
      idx = __shfl_sync(0xffffffffu, idx, 0);
      const int cur = idx < p.pool_count ? p.pool_begin + idx : -1;
      if (lane == 0) {
        const int slot = claimed % kSegRing;
        dev::mbar_wait(dev::smem_addr(&queue->empty[slot]),
                       (uint32_t)(((claimed / kSegRing) & 1) ^ 1), aborted, p.err);
        *reinterpret_cast<volatile int*>(&queue->seg[slot]) = cur;
        dev::mbar_arrive(dev::smem_addr(&queue->full[slot]));
      }
      ++claimed;
      if (cur < 0) break;
      si = cur;
      const int pad = (align - k % align) % align;
      if (lane == 0)
        for (int i = 0; i < pad; ++i) {  // empty stages: released at once by their warp
          const int kk = k + i;
          dev::mbar_wait(dev::smem_addr(&empty[kk % S]), (uint32_t)(((kk / S) & 1) ^ 1), aborted,
                         p.err);
          dev::mbar_arrive_n(dev::smem_addr(&full[kk % S]), SCALES ? kScaleLanes + 1 : 1);
        }
      k += pad;
    }
    const int4 sa = *reinterpret_cast<const int4*>(p.segments + 8 * si);
    const int kvh = sa.y, pb = sa.z, pe = sa.w;
    // The consumers read this segment's q rows when they reach it, several
    // pages from now: bring them into L2 while the pages are in flight.
    if (p.q_row_bytes > 0) prefetch_q_rows(p, sa.x, kvh, lane);
    for (int p0 = pb; p0 < pe; p0 += 32) {
      const int cnt = min(32, pe - p0);
      int id = lane < cnt ? __ldg(p.indices + p0 + lane) : 0;
      const bool bad = lane < cnt && (id < 0 || (int64_t)id >= p.num_pages);
      if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.err, 1);
      for (int i = 0; i < cnt; ++i, ++k) {
        const int page = __shfl_sync(0xffffffffu, id, i);
        if (lane == 0) {
          const int stage = k % S;
          const uint32_t round = (uint32_t)(k / S);
          dev::mbar_wait(dev::smem_addr(&empty[stage]), (round & 1u) ^ 1u, aborted, p.err);
          const uint32_t fb = dev::smem_addr(&full[stage]);
          dev::mbar_arrive_expect_tx(fb, STAGE_BYTES);
          // Out-of-range ids (already flagged) land outside the tensor map
          // and read zeros.
#pragma unroll
          for (int b = 0; b < BOXES; ++b)
            dev::tma_load_4d(dev::smem_addr(ring + stage * STAGE_BYTES + b * BOX_BYTES), map,
                             b * BOX_X, kvh, 0, 2 * page, fb, policy);
        }
        if constexpr (SCALES) {
          // lane 0 found the stage free; the scale rows have no bounds check
          // of their own: a flagged out-of-range page reads page 0's scales
          __syncwarp();
          if (lane < kScaleLanes) {
            const int stage = k % S;
            const int64_t pg = (page < 0 || (int64_t)page >= p.num_pages) ? 0 : page;
            const size_t row = ((size_t)pg * p.num_kv_heads + kvh) * kPageSize;
            const float* src = (lane < 4 ? p.k_scales : p.v_scales) + row + 4 * (lane & 3);
            dev::cp_async16(dev::smem_addr(scales + stage * 2 * kPageSize + 4 * lane), src);
            dev::cp_async_arrive(dev::smem_addr(&full[stage]));
          }
        }
      }
    }
    if (si >= seg_end) si = seg_end;  // a pool segment: the next one is claimed again
  }
  // No copy may still be landing in shared memory when the CTA exits (only
  // possible if a consumer gave up waiting).
  if constexpr (SCALES) dev::cp_async_wait_all();
  if (lane == 0) {
    const int first = k > S ? k - S : 0;
    for (int kk = first; kk < k; ++kk)
      if (!dev::mbar_wait_bounded(dev::smem_addr(&full[kk % S]), (uint32_t)((kk / S) & 1)))
        atomicOr(p.err, 2);
  }
}

// Next segment for a consumer warp: the CTA's static segments in order, then
// the pool segments its producer claimed, -1 when none is left.  A pool
// segment first consumes the empty stages the producer inserted before it
// (those of this warp) and moves kbase to the aligned start.  With the
// column split (CS) every warp consumes every page and pool segments need no
// alignment.  Warp-uniform.
template <int S, int NW, bool CS = false>
__device__ __forceinline__ int next_segment(const DecodeParams& p, SegQueue* queue, int& si,
                                            int seg_end, int& taken, int& kbase,
                                            uint64_t* full, uint64_t* empty, int warp, int lane,
                                            bool& aborted) {
  if (si < seg_end) return si++;
  if (p.pool_count == 0) return -1;
  const int slot = taken % kSegRing;
  dev::mbar_wait(dev::smem_addr(&queue->full[slot]), (uint32_t)((taken / kSegRing) & 1), aborted,
                 p.err);
  int cur = aborted ? -1 : *reinterpret_cast<volatile int*>(&queue->seg[slot]);
  cur = __shfl_sync(0xffffffffu, cur, 0);
  __syncwarp();
  if (lane == 0) dev::mbar_arrive(dev::smem_addr(&queue->empty[slot]));
  ++taken;
  if (cur < 0) return -1;
  const int ka = CS ? kbase : (kbase + NW - 1) / NW * NW;
  for (int k = kbase; k < ka; ++k) {
    if (k % NW != warp) continue;
    dev::mbar_wait(dev::smem_addr(&full[k % S]), (uint32_t)((k / S) & 1), aborted, p.err);
    __syncwarp();
    if (lane == 0) dev::mbar_arrive(dev::smem_addr(&empty[k % S]));
  }
  kbase = ka;
  return cur;
}

// End of a CTA's run (one thread): count it; the last CTA re-arms the pool
// counters for the next run.  Every claim of this CTA's producer happened
// before the end marker the consumers saw, so after the last count nobody
// claims any more.
__device__ __forceinline__ void pool_finish(const DecodeParams& p) {
  if (p.pool_count == 0) return;
  __threadfence();
  if (atomicAdd(p.pool_done, 1) == (int)gridDim.x - 1) {
    atomicExch(p.pool_claim, 0);
    atomicExch(p.pool_done, 0);
  }
}

// Fold the partial states of one split unit u = {request, kv_head,
// first_slot, num_slots} with the merge rule (log2 domain) and write o and
// lse.  The per-head weights are computed once, in `scratch` (at least
// num_slots * G floats, else a slower path reads the lse values per
// element); then every output element issues its num_slots loads at once.
// Runs on `nthreads` threads numbered `tid`, which synchronise on named
// barrier `bar` (0 = __syncthreads).
// Query rows of a request: the first row q0 of q / o / lse and the number
// of columns in use, G heads x its query tokens.  Ragged (RQ): request i owns
// rows qo_indptr[i] .. qo_indptr[i+1] (section "Ragged attention" of the page
// "FlashDecoding + FlashInfer" applied to the queries); otherwise every
// request has QL rows.
struct QRows {
  int q0, ncols;
};
template <int G, int QL, bool RQ>
__device__ __forceinline__ QRows query_rows(const int32_t* qo_indptr, int req) {
  if constexpr (RQ) {
    const int a = __ldg(qo_indptr + req);
    return QRows{a, G * (__ldg(qo_indptr + req + 1) - a)};
  } else {
    return QRows{req * QL, G * QL};
  }
}

// Output row of column n of a (request, kv head) unit: the unit's columns
// are the G heads of the group times its query tokens, token-major.
template <int G>
__device__ __forceinline__ size_t out_row(int q0, int kvh, int n, int num_qo_heads) {
  return ((size_t)q0 + n / G) * num_qo_heads + kvh * G + n % G;
}

template <typename QT, int D, int NC, int G, int QL, bool RQ = false>
__device__ __forceinline__ void fold_split_unit(const float* part_o, const float* part_lse,
                                                int4 u, QT* obase, float* lse_out, int num_qo_heads,
                                                const int32_t* qo_indptr,
                                                float* scratch, int scratch_floats, int tid,
                                                int nthreads, int bar) {
  static_assert(NC == G * QL, "columns = heads of the group x query tokens");
  const int kvh = u.y, s0 = u.z, ns = u.w;
  const QRows qr = query_rows<G, QL, RQ>(qo_indptr, u.x);
  if (ns * NC <= scratch_floats) {
    auto sync = [&]() {
      if (bar == 0) __syncthreads(); else dev::named_barrier(bar, nthreads);
    };
    // the unit's slots are consecutive: all ns * NC lse values in one pass
    for (int i = tid; i < ns * NC; i += nthreads)
      scratch[i] = __ldcg(part_lse + (size_t)s0 * NC + i);
    sync();
    // weights w[k][h] = 2^(lse_k - M_h) / den_h in place, and lse
    for (int h = tid; h < NC; h += nthreads) {
      float M = -INFINITY;
      for (int k = 0; k < ns; ++k) M = fmaxf(M, scratch[k * NC + h]);
      float den = 0.f;
      if (M != -INFINITY)
        for (int k = 0; k < ns; ++k) {
          const float w = dev::fast_exp2(scratch[k * NC + h] - M);
          scratch[k * NC + h] = w;
          den += w;
        }
      const float inv = den > 0.f ? 1.f / den : 0.f;
      for (int k = 0; k < ns; ++k) scratch[k * NC + h] = M != -INFINITY ? scratch[k * NC + h] * inv : 0.f;
      if (lse_out && h < qr.ncols)
        lse_out[out_row<G>(qr.q0, kvh, h, num_qo_heads)] =
            M != -INFINITY ? (M + dev::fast_log2(den)) * dev::kLn2 : -INFINITY;
    }
    sync();
    // four consecutive dims per thread (16-byte loads), eight pieces in
    // flight: a unit of many pieces is bound by load latency otherwise
    static_assert(D % 4 == 0, "float4 rows");
    for (int e = tid; e < qr.ncols * D / 4; e += nthreads) {
      const int h = e / (D / 4), d4 = (e % (D / 4)) * 4;
      const float4* po = reinterpret_cast<const float4*>(part_o + ((size_t)s0 * NC + h) * D + d4);
      const size_t stride = (size_t)NC * D / 4;  // float4s between pieces
      float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
      int k = 0;
      for (; k + 8 <= ns; k += 8) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = __ldcg(po + (size_t)(k + j) * stride);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float w = scratch[(k + j) * NC + h];
          num.x = fmaf(v[j].x, w, num.x);
          num.y = fmaf(v[j].y, w, num.y);
          num.z = fmaf(v[j].z, w, num.z);
          num.w = fmaf(v[j].w, w, num.w);
        }
      }
      for (; k < ns; ++k) {
        const float4 v = __ldcg(po + (size_t)k * stride);
        const float w = scratch[k * NC + h];
        num.x = fmaf(v.x, w, num.x);
        num.y = fmaf(v.y, w, num.y);
        num.z = fmaf(v.z, w, num.z);
        num.w = fmaf(v.w, w, num.w);
      }
      QT* orow = obase + out_row<G>(qr.q0, kvh, h, num_qo_heads) * D + d4;
      orow[0] = dev::from_float<QT>(num.x);
      orow[1] = dev::from_float<QT>(num.y);
      orow[2] = dev::from_float<QT>(num.z);
      orow[3] = dev::from_float<QT>(num.w);
    }
    return;
  }
  for (int e = tid; e < qr.ncols * D; e += nthreads) {
    const int h = e / D, dd = e % D;
    float M = -INFINITY;
    for (int k = 0; k < ns; ++k) M = fmaxf(M, __ldcg(part_lse + (size_t)(s0 + k) * NC + h));
    float out = 0.f, lse2 = -INFINITY;
    if (M != -INFINITY) {
      float den = 0.f, num = 0.f;
      for (int k = 0; k < ns; ++k) {
        const float w = dev::fast_exp2(__ldcg(part_lse + (size_t)(s0 + k) * NC + h) - M);
        den += w;
        num = fmaf(__ldcg(part_o + ((size_t)(s0 + k) * NC + h) * D + dd), w, num);
      }
      out = num / den;
      lse2 = M + dev::fast_log2(den);
    }
    const size_t row = out_row<G>(qr.q0, kvh, h, num_qo_heads);
    obase[row * D + dd] = dev::from_float<QT>(out);
    if (dd == 0 && lse_out) lse_out[row] = lse2 * dev::kLn2;
  }
}

// Split units whose last piece this CTA completed; it folds them after its
// last segment.  Filled by consumer thread 0 only.
constexpr int kMaxFolds = 60;
struct FoldList {
  int n;
  int unit[kMaxFolds];
  int pad[3];
};
constexpr int kFoldListBytes = (int)((sizeof(FoldList) + 15) / 16 * 16);

// Fold the units on the fold list now, with `scratch` (free while the CTA is
// between segments) for the weights; a unit whose weights do not fit stays
// on the list for fold_pending.  All consumer threads, between consumer
// barriers.  Folding here, with the producer's copies of the next pages in
// flight, keeps the folds out of the launch's tail.
template <typename QT, int D, int G, int NW, int QL = 1, bool RQ = false>
__device__ __forceinline__ void fold_listed(const DecodeParams& p, FoldList* folds,
                                            float* scratch, int scratch_floats) {
  constexpr int CT = NW * 32;
  constexpr int NC = G * QL;
  const int n = folds->n;
  if (n == 0) return;
  int kept = 0;
  for (int i = 0; i < n; ++i) {
    const int unit = folds->unit[i];
    const int4 u = reinterpret_cast<const int4*>(p.merge)[unit];
    if (u.w * NC > scratch_floats) {
      kept += 1;  // same decision in every thread
      continue;
    }
    fold_split_unit<QT, D, NC, G, QL, RQ>(p.part_o, p.part_lse, u, static_cast<QT*>(p.o), p.lse,
                                          p.num_qo_heads, p.qo_indptr, scratch, scratch_floats,
                                          threadIdx.x, CT, 1);
    dev::named_barrier(1, CT);  // scratch free for the next unit
  }
  if (kept) {  // compact the list (thread 0; the others have read it above)
    dev::named_barrier(1, CT);
    if (threadIdx.x == 0) {
      int w = 0;
      for (int i = 0; i < n; ++i) {
        const int4 u = reinterpret_cast<const int4*>(p.merge)[folds->unit[i]];
        if (u.w * NC > scratch_floats) folds->unit[w++] = folds->unit[i];
      }
      folds->n = w;
    }
  } else if (threadIdx.x == 0) {
    folds->n = 0;
  }
  dev::named_barrier(1, CT);
}

// Combine the NS states of one segment for all NC columns (unnormalised o in
// mo[w][h][d] against the state's max mm[w][h], sum md[w][h], all log2
// domain; NS = NW when the warps split the pages, 1 when each warp owns its
// columns) with the merge rule and write either the final o (q dtype) and
// lse of the columns in use, or an fp32 partial slot.  Runs on the NW*32 consumer
// threads after a consumer barrier and ends with one (mo is free again).
// A split piece is then counted by thread 0 alone while the other warps go
// on: the piece that completes its unit puts the unit on the CTA's fold list,
// folded at the next segment's combine (fold_listed, with `scratch`) or
// after the CTA's last segment (fold_pending), so no warp waits for the
// count's round trip.
template <typename QT, int D, int G, int NW, int QL = 1, bool RQ = false, int NS = NW>
__device__ __forceinline__ void combine_and_emit(const DecodeParams& p, const float* mo,
                                                 const float* mm, const float* md, QRows qr,
                                                 int kvh, int out_slot, int merge_unit,
                                                 FoldList* folds, float* scratch,
                                                 int scratch_floats) {
  constexpr int CT = NW * 32;
  constexpr int NC = G * QL;  // columns: heads of the group x query tokens
  QT* __restrict__ obase = static_cast<QT*>(p.o);
  fold_listed<QT, D, G, NW, QL, RQ>(p, folds, scratch, scratch_floats);
  // a split piece stores every column of its slot; final rows only the
  // columns in use
  const int cols = out_slot < 0 ? qr.ncols : NC;
  // the per-tensor V scale, times the kv head's own (per-head scales)
  const float v_scale =
      p.head_v_scales ? p.v_scale * __ldg(p.head_v_scales + kvh) : p.v_scale;
  for (int e = threadIdx.x; e < cols * D; e += CT) {
    const int h = e / D, dd = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NS; ++w) M = fmaxf(M, mm[w * NC + h]);
    float out = 0.f, lse2 = -INFINITY;
    if (M != -INFINITY) {
      float den = 0.f, num = 0.f;
#pragma unroll
      for (int w = 0; w < NS; ++w) {
        const float sw = dev::fast_exp2(mm[w * NC + h] - M);
        den = fmaf(md[w * NC + h], sw, den);
        num = fmaf(mo[(w * NC + h) * D + dd], sw, num);
      }
      out = num / den * v_scale;
      lse2 = M + dev::fast_log2(den);
    }
    if (out_slot < 0) {
      const size_t row = out_row<G>(qr.q0, kvh, h, p.num_qo_heads);
      obase[row * D + dd] = dev::from_float<QT>(out);
      if (dd == 0 && p.lse) p.lse[row] = lse2 * dev::kLn2;
    } else {
      p.part_o[((size_t)out_slot * NC + h) * D + dd] = out;
      if (dd == 0) p.part_lse[(size_t)out_slot * NC + h] = lse2;
    }
  }
  dev::named_barrier(1, CT);  // all reads of mo and all writes of this CTA done
  if (out_slot < 0 || !p.fused_merge || threadIdx.x != 0) return;
  const int4 u = reinterpret_cast<const int4*>(p.merge)[merge_unit];
  // one fence after the barrier publishes the whole CTA's writes (fences
  // are cumulative) before the arrival is counted
  __threadfence();
  const int prev = atomicAdd(&p.merge_count[merge_unit], 1);
  if (prev != u.w - 1) return;
  __threadfence();
  p.merge_count[merge_unit] = 0;  // re-armed for the next run of the plan
  if (folds->n < kMaxFolds) {
    folds->unit[folds->n++] = merge_unit;
    return;
  }
  // list full (a CTA that completed very many units): fold this one now,
  // on this thread alone
  fold_split_unit<QT, D, NC, G, QL, RQ>(p.part_o, p.part_lse, u, obase, p.lse, p.num_qo_heads,
                                        p.qo_indptr, nullptr, 0, 0, 1, 1);
}

// After a CTA's last segment: fold the split units it completed, in the
// order it completed them; each fold combines the unit's pieces in slot
// order, so the result does not depend on which CTA folds.  Consumer
// threads only; mo serves as scratch.
template <typename QT, int D, int G, int NW, int QL = 1, bool RQ = false>
__device__ __forceinline__ void fold_pending(const DecodeParams& p, float* mo, FoldList* folds,
                                             int scratch_floats) {
  constexpr int CT = NW * 32;
  constexpr int NC = G * QL;
  dev::named_barrier(1, CT);  // thread 0's list is complete
  const int n = folds->n;
  for (int i = 0; i < n; ++i) {
    const int4 u = reinterpret_cast<const int4*>(p.merge)[folds->unit[i]];
    fold_split_unit<QT, D, NC, G, QL, RQ>(p.part_o, p.part_lse, u, static_cast<QT*>(p.o), p.lse,
                                          p.num_qo_heads, p.qo_indptr, mo, scratch_floats,
                                          threadIdx.x, CT, 1);
    dev::named_barrier(1, CT);  // scratch free for the next unit
  }
}

template <typename QT, typename KVT, int D, int G, int NW>
struct DecodeCfg {
  static constexpr int P = kPageSize;
  static constexpr int KV_ES = sizeof(KVT);
  static constexpr int VEC_BYTES = KV_ES == 1 ? 8 : 16;
  static constexpr int VEC = VEC_BYTES / KV_ES;
  static constexpr int LPR = D / VEC;  // lanes that share one K/V row
  static constexpr int RPS = 32 / LPR;  // rows a warp covers per step
  static constexpr int STEPS = P / RPS;
  static constexpr int HPL = LPR / G;   // lanes holding the same head's score
  static constexpr int ROW_BYTES = D * KV_ES;
  static constexpr int STAGE_BYTES = 2 * P * ROW_BYTES;
  // ring of about 64 KB, a whole number of stages per consumer warp
  static constexpr int SPW0 = 65536 / STAGE_BYTES / NW;
  static constexpr int SPW = SPW0 < 1 ? 1 : (SPW0 > 4 ? 4 : SPW0);
  static constexpr int S = SPW * NW;
  static constexpr int THREADS = (NW + 1) * 32;
  static constexpr int OFF_FULL = S * STAGE_BYTES;
  static constexpr int OFF_EMPTY = OFF_FULL + 8 * S;
  static constexpr int OFF_P = OFF_EMPTY + 8 * S;
  static constexpr int OFF_MO = OFF_P + 4 * NW * P * G;
  static constexpr int OFF_MM = OFF_MO + 4 * NW * G * D;
  static constexpr int OFF_MD = OFF_MM + 4 * NW * G;
  static constexpr int OFF_FOLDS = OFF_MD + 4 * NW * G;
  static constexpr int OFF_QUEUE = OFF_FOLDS + kFoldListBytes;
  static constexpr int SMEM = OFF_QUEUE + kSegQueueBytes;
  static_assert(LPR <= 32 && 32 % LPR == 0 && P % RPS == 0, "row mapping");
  static_assert(G <= LPR, "group size larger than lanes per row");
  static_assert(STAGE_BYTES % 128 == 0, "stage alignment");
  static_assert(S % NW == 0, "each ring stage must belong to exactly one consumer warp");
};

template <typename QT, typename KVT, int D, int G, int NW>
__global__ void __launch_bounds__(DecodeCfg<QT, KVT, D, G, NW>::THREADS)
    fa_decode_split_kernel(const __grid_constant__ CUtensorMap kv_map,
                           const DecodeParams p) {
  using C = DecodeCfg<QT, KVT, D, G, NW>;
  constexpr int P = C::P, VEC = C::VEC, LPR = C::LPR, RPS = C::RPS,
                STEPS = C::STEPS, HPL = C::HPL, S = C::S;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_FULL);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + C::OFF_EMPTY);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  SegQueue* queue = reinterpret_cast<SegQueue*>(smem + C::OFF_QUEUE);
  FoldList* folds = reinterpret_cast<FoldList*>(smem + C::OFF_FOLDS);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      dev::mbar_init(dev::smem_addr(&full[s]), 1);
      dev::mbar_init(dev::smem_addr(&empty[s]), 1);
    }
    seg_queue_init(queue, NW);
    folds->n = 0;
    dev::fence_barrier_init();
  }
  __syncthreads();
  // Launched as a programmatic dependent (fa_decode_run): the next launch
  // may start placing its CTAs now.  Until the grid this one depends on has
  // completed, the CTA reads only plan data (written by the plan's upload,
  // a copy the launch is fully ordered after) and brings its first page ids
  // and q rows into L2, the GPU's point of coherence; everything else waits.
  dev::grid_dependency_launch();
  const int seg_begin = p.cta_offsets[blockIdx.x];
  const int seg_end = p.cta_offsets[blockIdx.x + 1];
  if (warp == NW && seg_begin < seg_end) prefetch_first_segment(p, seg_begin, lane);
  dev::grid_dependency_wait();

  if (warp == NW) {
    produce_pages<S, C::STAGE_BYTES, 1, 0, C::STAGE_BYTES>(&kv_map, p, seg_begin, seg_end, ring,
                                                          full, empty, lane, nullptr, queue, NW);
    return;
  }

  // ------------------ consumers ----------------------------------------
  float* pw = reinterpret_cast<float*>(smem + C::OFF_P) + warp * P * G;
  float* mo = reinterpret_cast<float*>(smem + C::OFF_MO);
  float* mm = reinterpret_cast<float*>(smem + C::OFF_MM);
  float* md = reinterpret_cast<float*>(smem + C::OFF_MD);
  const int rs = lane / LPR;  // row within a step
  const int c = lane % LPR;   // column chunk
  const int hl = c / HPL;     // head whose score this lane ends up holding
  const QT* __restrict__ qbase = static_cast<const QT*>(p.q);
  constexpr int CT = NW * 32;

  bool aborted = false;  // a timed-out wait makes every later wait return at once
  int kbase = 0, next_si = seg_begin, taken = 0;
  for (;;) {
    const int si = next_segment<S, NW>(p, queue, next_si, seg_end, taken, kbase, full, empty,
                                       warp, lane, aborted);
    if (si < 0) break;
    const int4 sa = *reinterpret_cast<const int4*>(p.segments + 8 * si);
    const int4 sb = *reinterpret_cast<const int4*>(p.segments + 8 * si + 4);
    const int req = sa.x, kvh = sa.y, npg = sa.w - sa.z;
    const int last_valid = sb.x, out_slot = sb.y;
    const float q_scale =
        p.head_k_scales ? p.q_scale * __ldg(p.head_k_scales + kvh) : p.q_scale;

    float qf[G][VEC];
    float acc[G][VEC];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const QT* qp = qbase + ((size_t)req * p.num_qo_heads + kvh * G + h) * D + c * VEC;
      dev::load_q<QT, VEC>(qp, qf[h]);
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        qf[h][v] *= q_scale;
        acc[h][v] = 0.f;
      }
    }
    float m_l = -INFINITY, d_l = 0.f;

    // this warp's pages of the segment: stream positions k with k % NW == warp
    for (int k = kbase + (warp - kbase % NW + NW) % NW; k < kbase + npg; k += NW) {
      const int lp = k - kbase;
      const int stage = k % S;
      dev::mbar_wait(dev::smem_addr(&full[stage]), (uint32_t)((k / S) & 1), aborted, p.err);
      const uint8_t* kt = ring + stage * C::STAGE_BYTES;
      const uint8_t* vt = kt + P * C::ROW_BYTES;
      const int valid = (lp == npg - 1) ? last_valid : P;

      float sc[STEPS];
#pragma unroll
      for (int st = 0; st < STEPS; ++st) {
        const int j = st * RPS + rs;
        float kf[VEC];
        dev::VecLoad<KVT, VEC>::load(kt + j * C::ROW_BYTES + c * C::VEC_BYTES, kf);
        float part[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float a = 0.f;
#pragma unroll
          for (int v = 0; v < VEC; ++v) a = fmaf(qf[h][v], kf[v], a);
          part[h] = a;
        }
        const float s = dev::reduce_scatter<G, LPR>(part, c);
        sc[st] = j < valid ? s : -INFINITY;
      }
      float mx = sc[0];
#pragma unroll
      for (int st = 1; st < STEPS; ++st) mx = fmaxf(mx, sc[st]);
#pragma unroll
      for (int off = LPR; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m_l, mx);
      const float alpha = dev::fast_exp2(m_l - m_new);
      float ps = 0.f;
#pragma unroll
      for (int st = 0; st < STEPS; ++st) {
        sc[st] = dev::fast_exp2(sc[st] - m_new);
        ps += sc[st];
      }
#pragma unroll
      for (int off = LPR; off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      d_l = d_l * alpha + ps;
      m_l = m_new;
      if (c % HPL == 0) {
#pragma unroll
        for (int st = 0; st < STEPS; ++st) pw[(st * RPS + rs) * G + hl] = sc[st];
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float a = __shfl_sync(0xffffffffu, alpha, h * HPL);
#pragma unroll
        for (int v = 0; v < VEC; ++v) acc[h][v] *= a;
      }
      __syncwarp();
#pragma unroll
      for (int st = 0; st < STEPS; ++st) {
        const int j = st * RPS + rs;
        if (j < valid) {
          float vf[VEC];
          dev::VecLoad<KVT, VEC>::load(vt + j * C::ROW_BYTES + c * C::VEC_BYTES, vf);
          float pj[G];
#pragma unroll
          for (int h = 0; h < G; ++h) pj[h] = pw[j * G + h];
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int v = 0; v < VEC; ++v) acc[h][v] = fmaf(pj[h], vf[v], acc[h][v]);
        }
      }
      dev::release_stage(dev::smem_addr(&empty[stage]), lane);
    }

    // Sum the row groups of this warp (they share m and d).
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int v = 0; v < VEC; ++v)
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1)
          acc[h][v] += __shfl_xor_sync(0xffffffffu, acc[h][v], off);
    if (rs == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int v = 0; v < VEC; ++v) mo[(warp * G + h) * D + c * VEC + v] = acc[h][v];
      if (c % HPL == 0) {
        mm[warp * G + hl] = m_l;
        md[warp * G + hl] = d_l;
      }
    }
    dev::named_barrier(1, CT);

    // Merge the NW warp states of this segment and emit.
    combine_and_emit<QT, D, G, NW>(p, mo, mm, md, QRows{req, G}, kvh, out_slot, sb.z, folds,
                                   reinterpret_cast<float*>(smem + C::OFF_P), NW * P * G);
    kbase += npg;
  }
  fold_pending<QT, D, G, NW>(p, mo, folds, NW * G * D);
  if (threadIdx.x == 0) pool_finish(p);
}

// Split-level merge as a separate kernel: one CTA per (request, kv head)
// that the planner split folds its partial states with the merge rule.
template <typename QT, int D, int G, int QL = 1, bool RQ = false>
__global__ void __launch_bounds__(128) fa_merge_partials_kernel(const MergeParams p) {
  __shared__ float weights[2048];
  const int4 u = reinterpret_cast<const int4*>(p.merge)[blockIdx.x];
  fold_split_unit<QT, D, G * QL, G, QL, RQ>(p.part_o, p.part_lse, u, static_cast<QT*>(p.o),
                                            p.lse, p.num_qo_heads, p.qo_indptr, weights, 2048,
                                            threadIdx.x, blockDim.x, 0);
}

template <typename QT, typename KVT, int D, int G, int NW = 4>
inline void fill_kernel(DecodeKernel* k) {
  using C = DecodeCfg<QT, KVT, D, G, NW>;
  k->func = reinterpret_cast<const void*>(&fa_decode_split_kernel<QT, KVT, D, G, NW>);
  k->merge_func = reinterpret_cast<const void*>(&fa_merge_partials_kernel<QT, D, G>);
  k->threads = C::THREADS;
  k->smem_bytes = C::SMEM;
  k->stages = C::S;
  k->stage_bytes = C::STAGE_BYTES;
  k->group = G;
  k->head_dim = D;
  k->box_x = D;
  k->swizzle_128b = false;
  k->tensor_cores = false;
}

}  // namespace fadecode
