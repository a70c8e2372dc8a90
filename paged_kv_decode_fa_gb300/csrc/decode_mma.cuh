// Split-KV paged decode with the per-page products on the tensor cores
// (mma.sync m16n8k16, fp32 accumulate), for groups of 2..8 query heads per
// kv head over 16-bit or E4M3 KV.
//
// Same pipeline, planner contract and epilogue as fa_decode_split_kernel
// (decode_kernel.cuh); only the consumer arithmetic differs.  With a group
// of G heads a page is a tiny contraction - scores S^T[16 tokens x G] =
// K[16 x D] . q^T, then O^T[D x G] += V^T[D x 16] . P^T - and doing it as
// per-lane FMAs with shuffle reductions costs about 1100 warp instructions
// per (page, kv head) at G = 4, which keeps the issue slots busy enough to
// cap the HBM rate.  Here each page costs D/16 MMAs for the scores and D/16
// for P.V, with tokens on the M side (no padding whatever G is):
//
//  - the stage holds each 128-byte row segment of K/V in TMA "128B swizzle"
//    order (16-byte granule c of row r stored at c ^ (r & 7)), one box per
//    128 bytes of row, so that both fragment loads below are free of bank
//    conflicts;
//  - scores: lane (g, t) loads K rows g and g+8, granules 2t and 2t+1 of each
//    row segment, with 128-bit loads; the reduction index of the MMA is
//    permuted so that these are exactly the lane's A-fragment elements, and
//    q's B fragment (held in registers for the whole segment) uses the same
//    permutation; E4M3 K is widened to f16 in registers;
//  - softmax on the C fragment (tokens g, g+8 x heads 2t, 2t+1): weights
//    against a per-column reference that moves only when a page's maximum
//    passes it by more than 2^8 (or against a caller's static bound, the
//    unified max), so a page costs one warp vote; the column reduction (three
//    shuffles) and the exact rescale of the state run only when it moves;
//    each lane keeps its own share of the denominator, summed over the column
//    once per segment;
//  - P.V: P is rounded to the MMA type, transposed through a 256-byte
//    per-warp buffer into B fragments, V^T fragments come straight from the
//    stage with ldmatrix.trans (for E4M3, pairs of bytes are transposed as
//    16-bit elements and split with one byte permute; the page split loads
//    them right after the scores and hands the stage back before the
//    softmax).
//
// Up to 8 columns (query heads x query tokens) the warps split the pages
// (page k to warp k % NW).  With more, each warp owns 8 columns and takes
// every page of the segment (the column split), several pages a step so that
// their independent loads and MMA chains overlap.
#pragma once
#include <type_traits>

#include "decode_kernel.cuh"

namespace fadecode {
namespace mma {

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <bool kBf16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (kBf16)
    mma_bf16(c, a0, a1, a2, a3, b0, b1);
  else
    mma_f16(c, a0, a1, a2, a3, b0, b1);
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// The two E4M3 codes in the low 16 bits (low byte first) -> f16x2 (low
// half first), exact; one hardware conversion.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t out;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
      : "=r"(out)
      : "r"(two_codes));
  return out;
}

// Both halves of a word of four E4M3 codes -> two f16x2.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four_codes, uint32_t& lo,
                                                  uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(four_codes));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
  if (bf16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack2(uint32_t w, bool bf16) {
  if (bf16) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  __half2 h;
  memcpy(&h, &w, sizeof h);
  return __half22float2(h);
}

}  // namespace mma

template <typename QT, typename KVT, int D, int G, int NW, bool TS = false, int QL = 1>
struct MmaCfg {
  static constexpr int NC = G * QL;  // MMA columns: heads of the group x query tokens
  // Column split: with more than 8 columns every consumer warp takes every
  // page of a segment and owns 8 columns of its own (warp w: columns
  // 8w .. 8w+7), so no warp holds more than one 8-column accumulator tile
  // and a column's state never needs merging across warps.  With at most 8
  // columns the warps split the pages instead (page k to warp k % NW).
  static constexpr bool CS = NC > 8;
  static constexpr int NS = CS ? 1 : NW;  // partial states per column at a segment's end
  // pages a consumer warp takes per step: two or three (E4M3) for the
  // column split (every warp takes every page), one for the page split
  static constexpr int NPP = CS ? (sizeof(KVT) == 1 ? 3 : 2) : 1;
  static constexpr int P = kPageSize;
  static constexpr int KV_ES = sizeof(KVT);
  static constexpr bool kFp8 = KV_ES == 1;
  // MMA operand type: bf16 for bf16 KV, f16 for f16 and E4M3 KV.
  static constexpr bool kBf16 = std::is_same<KVT, __nv_bfloat16>::value;
  static constexpr int ROW_BYTES = D * KV_ES;
  static constexpr int SEGS = ROW_BYTES / 128;    // 128-byte row segments = TMA boxes
  static constexpr int BOX_X = 128 / KV_ES;       // elements per box row
  static constexpr int BOX_BYTES = 2 * P * 128;   // K and V rows of one segment
  static constexpr int STAGE_BYTES = SEGS * BOX_BYTES;
  static constexpr int E = 16 / KV_ES;            // elements per 16-byte granule
  static constexpr int KSTEPS = D / 16;
  static constexpr int MTILES = D / 16;
  // Ring size, whole stages per consumer warp.  16-bit KV: 64 KB (48 KB at
  // G = 8, whose larger epilogue buffer would otherwise leave room for only
  // two CTAs per SM), three CTAs per SM.  E4M3 KV: 32 KB (two 4 KB pages per
  // warp) so that four CTAs fit per SM - its denser per-byte arithmetic needs
  // the extra warps to hide each page's dependent chain; the E4M3 column
  // split (three pages a warp step) 48 KB at three CTAs per SM.  A column
  // split of two or three warps (16 or 24 columns) takes 32 KB, so that five
  // or four CTAs fit per SM.
  static constexpr int RING_BYTES =
      CS && NW < 4 ? 32768
                   : (KV_ES == 1 ? (CS ? 49152 : 32768) : (NC >= 8 ? 49152 : 65536));
  static constexpr int SPW0 = RING_BYTES / STAGE_BYTES / NW;
  static constexpr int SPW = SPW0 < 1 ? 1 : (SPW0 > 4 ? 4 : SPW0);
  // column split: every warp reads every stage, any number of stages works
  static constexpr int S = CS ? RING_BYTES / STAGE_BYTES : SPW * NW;
  static constexpr int THREADS = (NW + 1) * 32;
  // CTAs per SM the ring size is chosen for; the register budget must allow
  // it (column split: 480 or 512 threads per SM at two or three warps)
  static constexpr int MIN_CTAS = CS ? (NW <= 2 ? 5 : NW == 3 ? 4 : 3) : (KV_ES == 1 ? 4 : 3);
  static constexpr int OFF_FULL = S * STAGE_BYTES;
  static constexpr int OFF_EMPTY = OFF_FULL + 8 * S;
  static constexpr int OFF_PT = OFF_EMPTY + 8 * S;  // [NW][NPP][8 heads][16 tokens] 16-bit
  static constexpr int OFF_MO = OFF_PT + NW * NPP * 8 * P * 2;
  static constexpr int OFF_MM = OFF_MO + 4 * NS * NC * D;
  static constexpr int OFF_MD = OFF_MM + 4 * NS * NC;
  static constexpr int OFF_FOLDS = OFF_MD + 4 * NS * NC;
  static constexpr int OFF_QUEUE = OFF_FOLDS + kFoldListBytes;
  static constexpr int OFF_SCALES = OFF_QUEUE + kSegQueueBytes;    // [S][32] fp32 if TS
  static constexpr int SMEM = OFF_SCALES + (TS ? S * 2 * P * 4 : 0);
  static_assert(!TS || kFp8, "per-token scales are for E4M3 KV");
  static_assert(ROW_BYTES % 128 == 0, "rows must be whole 128-byte swizzle rows");
  static_assert(NC >= 1 && (NC <= 8 || NC <= 8 * NW), "8 columns (the MMA N side) per warp");
  static_assert(STAGE_BYTES % 1024 == 0, "swizzled boxes need 1024-byte alignment");
  static_assert(CS || S % NW == 0, "each ring stage must belong to exactly one consumer warp");
  static_assert(!kFp8 || D % 32 == 0, "E4M3 V is transposed two granules at a time");
};

// Unified-max softmax window (log2 units): while a column's running maximum
// m stays within [ref - below, ref + above] of the static reference, its
// weights are exp2(s - ref) with no running-max bookkeeping.  bf16 weights:
// above 16 - a weight stays below 2^16 and a sum over 2^31 tokens below 2^47
// (fp32 and bf16 hold both); below 64 - ex2.approx flushes weights under
// 2^-126 to zero, so a flushed token weighs under 2^(64-126) relative to the
// maximum one.  f16 weights (f16 and E4M3 KV) have a 5-bit exponent: above
// 15 keeps every weight under 2^15 (f16 tops out at 65504); below 8 keeps the
// largest weight at 2^-8 or more, so the tokens that matter (weights down to
// 2^-6 of it) stay normal f16 numbers (2^-14 and up) and the ones that go
// subnormal or flush (under 2^-24) weigh under 2^-6 and 2^-16 of it.
constexpr float kUmAboveBf16 = 16.f, kUmBelowBf16 = 64.f;
constexpr float kUmAboveF16 = 15.f, kUmBelowF16 = 8.f;
// Without a static bound the reference of a column is its first observed
// maximum, re-centred (exactly) only when a later page's maximum exceeds it
// by more than 2^8: weights stay below 256, inside bf16 and f16 alike, and
// the largest weight of a column is at least 1, so the weights that the
// f16 conversion flushes (below 2^-24) weigh nothing next to it.
constexpr float kLazyAbove = 8.f;
// E4M3 page split: load a page's V fragments into registers right after its
// scores and release the stage then, instead of after P.V.
constexpr bool kEarlyVRelease = true;

template <typename QT, typename KVT, int D, int G, int NW, bool TS, int QL, bool UM,
          bool RQ = false>
__global__ void __launch_bounds__(MmaCfg<QT, KVT, D, G, NW, TS, QL>::THREADS,
                                  MmaCfg<QT, KVT, D, G, NW, TS, QL>::MIN_CTAS)
    fa_decode_mma_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p) {
  using C = MmaCfg<QT, KVT, D, G, NW, TS, QL>;
  constexpr int NC = C::NC;
  constexpr bool CS = C::CS;
  // causal masking among the query tokens (multi-token and ragged plans)
  constexpr bool kCausal = QL > 1 || RQ;
  constexpr int P = C::P, S = C::S, SEGS = C::SEGS, KSTEPS = C::KSTEPS, MTILES = C::MTILES;
  constexpr bool kBf16 = C::kBf16, kFp8 = C::kFp8;
  static_assert(kBf16 ? std::is_same<QT, __nv_bfloat16>::value
                      : (std::is_same<QT, __half>::value || kFp8),
                "q type must match the MMA type (or be widened for E4M3 KV)");
  // bf16 q with E4M3 KV runs the MMA in f16: q is scaled by a power of two
  // per segment to sit well inside the f16 range.
  constexpr bool kConvertQ = kFp8 && std::is_same<QT, __nv_bfloat16>::value;
  // the unified-max window relies on the 8-bit exponent of bf16 weights
  static_assert(!UM || (!TS && QL == 1 && !RQ), "unified max: plain decode");
  constexpr float kUmAbove = kBf16 ? kUmAboveBf16 : kUmAboveF16;
  constexpr float kUmBelow = kBf16 ? kUmBelowBf16 : kUmBelowF16;
  static_assert(!RQ || !TS, "ragged q: no per-token scales");

  // Swizzled TMA destinations must sit on 1024-byte boundaries: the launch
  // reserves 1 KB more than the layout so the base can be rounded up.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (dev::smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_FULL);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + C::OFF_EMPTY);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  SegQueue* queue = reinterpret_cast<SegQueue*>(smem + C::OFF_QUEUE);
  FoldList* folds = reinterpret_cast<FoldList*>(smem + C::OFF_FOLDS);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      dev::mbar_init(dev::smem_addr(&full[s]), TS ? kScaleLanes + 1 : 1);
      dev::mbar_init(dev::smem_addr(&empty[s]), CS ? NW : 1);  // its consumer warps
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
    produce_pages<S, C::STAGE_BYTES, SEGS, C::BOX_X, C::BOX_BYTES, TS>(
        &kv_map, p, seg_begin, seg_end, ring, full, empty, lane,
        reinterpret_cast<float*>(smem + C::OFF_SCALES), queue, CS ? 1 : NW);
    return;
  }

  uint16_t* pT = reinterpret_cast<uint16_t*>(smem + C::OFF_PT) + warp * C::NPP * 8 * P;
  float* mo = reinterpret_cast<float*>(smem + C::OFF_MO);
  float* mm = reinterpret_cast<float*>(smem + C::OFF_MM);
  float* md = reinterpret_cast<float*>(smem + C::OFF_MD);
  const int g = lane >> 2;  // MMA group id: token row g (and g+8), q/P column g
  const int t = lane & 3;   // thread in group: columns 2t, 2t+1 of the C fragment
  // column n <-> query token n / G, head n % G of the group
  const QT* __restrict__ qbase = static_cast<const QT*>(p.q);
  constexpr int CT = NW * 32;
  const uint32_t ring_addr = dev::smem_addr(ring);

  bool aborted = false;  // a timed-out wait makes every later wait return at once
  int kbase = 0, next_si = seg_begin, taken = 0;
  for (;;) {
    const int si = next_segment<S, NW, CS>(p, queue, next_si, seg_end, taken, kbase, full, empty,
                                           warp, lane, aborted);
    if (si < 0) break;
    const int4 sa = *reinterpret_cast<const int4*>(p.segments + 8 * si);
    const int4 sb = *reinterpret_cast<const int4*>(p.segments + 8 * si + 4);
    const int req = sa.x, kvh = sa.y, npg = sa.w - sa.z;
    const int last_valid = sb.x, out_slot = sb.y, to_end = sb.w;
    const QRows qr = query_rows<G, QL, RQ>(p.qo_indptr, req);
    const int nq = qr.ncols / G;  // this request's query tokens
    // this warp's columns: cb .. cb + 7 (the column split), else 0 .. 7
    const int cb = CS ? 8 * warp : 0;
    // a warp whose columns are all past the request's still takes its pages
    // (every warp releases every stage) but computes nothing
    const bool active = !CS || cb < qr.ncols;
    // causal limits of columns cb+2t, cb+2t+1: token position (from the
    // segment start) after which query token n / G must not look; columns
    // past the request's see nothing
    int lim[2] = {0x7fffffff, 0x7fffffff};
    if constexpr (kCausal) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int n = cb + 2 * t + e;
        lim[e] = n < qr.ncols ? to_end - nq + n / G : -1;
      }
    }

    // ---- q as the B fragment of the score MMA, for the whole segment.
    // Reduction step j uses, in lane t, the four dims base(j) .. base(j)+3:
    // b0 <- dims base, base+1 and b1 <- base+2, base+3, where base(j) walks
    // granules 2t and 2t+1 of each 128-byte row segment (the same elements
    // the lane loads from K).
    uint32_t qb[KSTEPS][2];
    // per-kv-head scales (fa_decode_run_head_scales) join the per-tensor ones
    const float seg_q_scale = p.head_k_scales ? p.q_scale * __ldg(p.head_k_scales + kvh)
                                              : p.q_scale;
    float qscale = seg_q_scale;
    {
      float qf[KSTEPS][4];
#pragma unroll
      for (int j = 0; j < KSTEPS; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) qf[j][e] = 0.f;
      uint32_t raw[KSTEPS][2];
      if (cb + g < qr.ncols) {
        const int n = cb + g;  // this lane's column of the B fragment
        const QT* qrow = qbase + (((size_t)qr.q0 + n / G) * p.num_qo_heads + kvh * G + n % G) * D;
        // Load L (16 bytes, 8 consecutive elements) feeds reduction steps 2L
        // and 2L+1.  16-bit KV: step j = 4*seg + 2*half + u covers dims
        // seg*BOX_X + (2t + half)*8 + 4u .. +3.  E4M3 KV: step j = 4*half + w
        // covers dims (2t + half)*16 + 4w .. +3.
#pragma unroll
        for (int L = 0; L < KSTEPS / 2; ++L) {
          int d0;
          if constexpr (kFp8)
            d0 = (2 * t + (L >> 1)) * 16 + (L & 1) * 8;
          else
            d0 = (L >> 1) * C::BOX_X + (2 * t + (L & 1)) * 8;
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(qrow + d0));
          raw[2 * L][0] = v.x;
          raw[2 * L][1] = v.y;
          raw[2 * L + 1][0] = v.z;
          raw[2 * L + 1][1] = v.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < KSTEPS; ++j) raw[j][0] = raw[j][1] = 0u;
      }
      if constexpr (kConvertQ) {
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < KSTEPS; ++j) {
          const float2 lo = mma::unpack2(raw[j][0], true), hi = mma::unpack2(raw[j][1], true);
          qf[j][0] = lo.x; qf[j][1] = lo.y; qf[j][2] = hi.x; qf[j][3] = hi.y;
#pragma unroll
          for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(qf[j][e]));
        }
        const unsigned bits = __reduce_max_sync(0xffffffffu, __float_as_uint(amax));
        int shift = 0;
        if (bits != 0u && bits < 0x7f800000u) {
          const int ex = (int)((bits >> 23) & 0xff) - 127;  // amax in [2^ex, 2^(ex+1))
          shift = min(max(14 - ex, -120), 120);
        }
        const float up = ldexpf(1.f, shift);
        qscale = seg_q_scale * ldexpf(1.f, -shift);
#pragma unroll
        for (int j = 0; j < KSTEPS; ++j) {
          qb[j][0] = mma::pack2(qf[j][0] * up, qf[j][1] * up, false);
          qb[j][1] = mma::pack2(qf[j][2] * up, qf[j][3] * up, false);
        }
      } else {
#pragma unroll
        for (int j = 0; j < KSTEPS; ++j) {
          qb[j][0] = raw[j][0];
          qb[j][1] = raw[j][1];
        }
      }
    }

    float o[MTILES][4];
#pragma unroll
    for (int mt = 0; mt < MTILES; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
    // m_h: the column's reference (running max, or the static bound when
    // UM); d_h: this lane's share of the column's denominator, summed over
    // the column's 8 lanes once the segment is done
    float m_h[2] = {-INFINITY, -INFINITY}, d_h[2] = {0.f, 0.f};
    float tmx[2] = {-INFINITY, -INFINITY};  // this lane's running maxima of the columns
    bool um_first = true, um_moved = false;
    if constexpr (UM) m_h[0] = m_h[1] = p.max_bound;
    // the reference the weights are taken against: m_h, or 0 for a column
    // that has seen nothing yet (every token so far masked), whose weights
    // exp2(-inf - 0) = 0 keep its state empty; it changes only on a rescale
    float mref[2] = {0.f, 0.f};

    // ---- O^T[dim][head] += V^T . P^T for one page (stage address st).
    // Slots past the last valid token may hold anything (NaN included): a
    // zero weight would not cancel them in the MMA, so on a segment's
    // partial last page their V elements are cleared in the A fragments,
    // in registers (a full page takes the same step without the masks).
    // The stage itself is never written by the consumers: it belongs to
    // the copy engine, which refills it for a later page as soon as this
    // warp releases it.  Each fragment register holds two consecutive
    // tokens (low half 2t, high half 2t+1; +8 for the upper token block).
    // E4M3 V fragments of one page, as loaded (four 8x8 matrices of byte
    // pairs per 16 dims x 16 tokens, transposed by ldmatrix)
    auto load_v_fp8 = [&](uint32_t st, uint32_t (&vf)[MTILES / 2][4]) {
#pragma unroll
      for (int c2 = 0; c2 < MTILES / 2; ++c2) {
        const int mi = lane >> 3, r = lane & 7;
        const int gran = 2 * c2 + (mi >> 1), tok = (mi & 1) * 8 + r;
        mma::ldsm_x4_trans(st + (P + tok) * 128 + ((gran ^ (tok & 7)) * 16), vf[c2][0],
                           vf[c2][1], vf[c2][2], vf[c2][3]);
      }
    };
    auto pv_step = [&](auto masked, uint32_t st, uint32_t pb0, uint32_t pb1, int valid,
                       const uint32_t* vf_loaded = nullptr) {
      constexpr bool kMask = decltype(masked)::value;
      uint32_t vmask_lo = 0xffffffffu, vmask_hi = 0xffffffffu;
      if constexpr (kMask) {
        vmask_lo = (2 * t < valid ? 0x0000ffffu : 0u) | (2 * t + 1 < valid ? 0xffff0000u : 0u);
        vmask_hi = (2 * t + 8 < valid ? 0x0000ffffu : 0u) | (2 * t + 9 < valid ? 0xffff0000u : 0u);
      }
      if constexpr (kFp8) {
        uint32_t vf[MTILES / 2][4];
        if (vf_loaded) {
#pragma unroll
          for (int c2 = 0; c2 < MTILES / 2; ++c2)
#pragma unroll
            for (int e = 0; e < 4; ++e) vf[c2][e] = vf_loaded[4 * c2 + e];
        } else {
          load_v_fp8(st, vf);
        }
#pragma unroll
        for (int c2 = 0; c2 < MTILES / 2; ++c2) {
          uint32_t d0 = vf[c2][0], d1 = vf[c2][1], d2 = vf[c2][2], d3 = vf[c2][3];
          // matrices 0 and 2 hold tokens 2t, 2t+1; 1 and 3 tokens 2t+8, 2t+9
          if constexpr (kMask) {
            d0 &= vmask_lo;
            d2 &= vmask_lo;
            d1 &= vmask_hi;
            d3 &= vmask_hi;
          }
          uint32_t a[4][2];
          mma::e4m3x4_to_f16x2x2(__byte_perm(d0, 0u, 0x3120), a[0][0], a[0][1]);
          mma::e4m3x4_to_f16x2x2(__byte_perm(d1, 0u, 0x3120), a[1][0], a[1][1]);
          mma::e4m3x4_to_f16x2x2(__byte_perm(d2, 0u, 0x3120), a[2][0], a[2][1]);
          mma::e4m3x4_to_f16x2x2(__byte_perm(d3, 0u, 0x3120), a[3][0], a[3][1]);
          mma::mma16816<false>(o[2 * c2], a[0][0], a[0][1], a[1][0], a[1][1], pb0, pb1);
          mma::mma16816<false>(o[2 * c2 + 1], a[2][0], a[2][1], a[3][0], a[3][1], pb0, pb1);
        }
      } else {
#pragma unroll
        for (int mt = 0; mt < MTILES; ++mt) {
          const int mi = lane >> 3, r = lane & 7;
          const int sgi = (mt * 16) / C::BOX_X;
          const int gran = ((mt * 16) % C::BOX_X) / 8 + (mi & 1);
          const int tok = (mi >> 1) * 8 + r;
          uint32_t a0, a1, a2, a3;
          mma::ldsm_x4_trans(
              st + sgi * C::BOX_BYTES + (P + tok) * 128 + ((gran ^ (tok & 7)) * 16), a0, a1,
              a2, a3);
          // matrices 0 and 1 hold tokens 2t, 2t+1; 2 and 3 tokens 2t+8, 2t+9
          if constexpr (kMask) {
            a0 &= vmask_lo;
            a1 &= vmask_lo;
            a2 &= vmask_hi;
            a3 &= vmask_hi;
          }
          mma::mma16816<kBf16>(o[mt], a0, a1, a2, a3, pb0, pb1);
        }
      }
    };

    // One step over NPP of the warp's pages, k, k + PS, ..., of the segment
    // (PS: the distance between the warp's pages, 1 for the column split,
    // NW for the page split): scores, one softmax update over all of them,
    // P.V.  Several pages a step keep their independent loads and MMA chains
    // in flight in the warp at once.
    constexpr int PS = CS ? 1 : NW;
    auto step = [&](auto npp_tag, int k) {
      constexpr int NPP = decltype(npp_tag)::value;
      int stage[NPP], lp[NPP], valid[NPP];
      uint32_t st[NPP];
#pragma unroll
      for (int u = 0; u < NPP; ++u) {
        const int ku = k + u * PS;
        lp[u] = ku - kbase;
        stage[u] = ku % S;
        dev::mbar_wait(dev::smem_addr(&full[stage[u]]), (uint32_t)((ku / S) & 1), aborted, p.err);
        st[u] = ring_addr + stage[u] * C::STAGE_BYTES;
        valid[u] = (lp[u] == npg - 1) ? last_valid : P;
      }
      if (CS && !active) {  // nothing to compute: release the stages
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int u = 0; u < NPP; ++u) dev::mbar_arrive(dev::smem_addr(&empty[stage[u]]));
        }
        return;
      }

      // ---- scores S^T[token][head] = K . q^T (two accumulators a page to halve the chain)
      float s[NPP][4], vs_lo[NPP], vs_hi[NPP];  // vs: per-token V scales of tokens g, g+8
      const int sw = g & 7;  // swizzle of rows g and g+8
#pragma unroll
      for (int u = 0; u < NPP; ++u) {
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int sgi = 0; sgi < SEGS; ++sgi) {
#pragma unroll
          for (int qq = 0; qq < 2; ++qq) {
            const uint32_t gran = (uint32_t)(((2 * t + qq) ^ sw) * 16);
            const uint4 ka = mma::lds128(st[u] + sgi * C::BOX_BYTES + g * 128 + gran);
            const uint4 kb = mma::lds128(st[u] + sgi * C::BOX_BYTES + (g + 8) * 128 + gran);
            const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w};
            const uint32_t wb[4] = {kb.x, kb.y, kb.z, kb.w};
            if constexpr (kFp8) {
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                const int j = qq * 4 + w;
                uint32_t a0, a1, a2, a3;
                mma::e4m3x4_to_f16x2x2(wa[w], a0, a2);
                mma::e4m3x4_to_f16x2x2(wb[w], a1, a3);
                mma::mma16816<false>(sc[j & 1], a0, a1, a2, a3, qb[j][0], qb[j][1]);
              }
            } else {
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                const int j = sgi * 4 + qq * 2 + h2;
                mma::mma16816<kBf16>(sc[j & 1], wa[2 * h2], wb[2 * h2], wa[2 * h2 + 1],
                                     wb[2 * h2 + 1], qb[j][0], qb[j][1]);
              }
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) s[u][e] = (sc[0][e] + sc[1][e]) * qscale;
        vs_lo[u] = vs_hi[u] = 1.f;
        if constexpr (TS) {
          const float* scl =
              reinterpret_cast<const float*>(smem + C::OFF_SCALES) + stage[u] * 2 * P;
          const float ks_lo = scl[g], ks_hi = scl[g + 8];
          vs_lo[u] = scl[P + g];
          vs_hi[u] = scl[P + g + 8];
          s[u][0] *= ks_lo;
          s[u][1] *= ks_lo;
          s[u][2] *= ks_hi;
          s[u][3] *= ks_hi;
        }
        if (valid[u] < P) {
          if (g >= valid[u]) s[u][0] = s[u][1] = -INFINITY;
          if (g + 8 >= valid[u]) s[u][2] = s[u][3] = -INFINITY;
        }
        if constexpr (kCausal) {
          const int pos = lp[u] * P + g;  // token position from the segment start
          if (pos > lim[0]) s[u][0] = -INFINITY;
          if (pos > lim[1]) s[u][1] = -INFINITY;
          if (pos + 8 > lim[0]) s[u][2] = -INFINITY;
          if (pos + 8 > lim[1]) s[u][3] = -INFINITY;
        }
      }

      // E4M3 page split: V's fragments go to registers now and the stage goes
      // back to the copy engine before the softmax, so the ring holds a page
      // only while its bytes are read (16 registers a page)
      constexpr bool kEarlyV = kFp8 && !CS && kEarlyVRelease;
      uint32_t vfrag[kEarlyV ? NPP : 1][MTILES / 2][4];
      if constexpr (kEarlyV) {
#pragma unroll
        for (int u = 0; u < NPP; ++u) {
          load_v_fp8(st[u], vfrag[u]);
          dev::release_stage(dev::smem_addr(&empty[stage[u]]), lane);
        }
      }

      // ---- softmax for heads 2t (s[.][0], s[.][2]) and 2t+1 (s[.][1], s[.][3])
      // The weights use a reference per column that moves only rarely, so a
      // step needs no column reduction - only a vote on whether some lane's
      // running maximum rose past the window above the reference.  Unified
      // max (UM): the reference starts at the caller's static bound, and the
      // first step of a segment also checks the window's lower edge (the
      // running maximum never falls, so once a column is inside it stays
      // inside).  Otherwise it starts empty and takes the column's first
      // observed maximum.  A column leaving its window is re-centred on its
      // true maximum (an exact rescale of its state).
      float alpha[2] = {1.f, 1.f};
      bool rescale;
      {
        constexpr float kAbove = UM ? kUmAbove : kLazyAbove;
#pragma unroll
        for (int u = 0; u < NPP; ++u) {
          tmx[0] = fmaxf(tmx[0], fmaxf(s[u][0], s[u][2]));
          tmx[1] = fmaxf(tmx[1], fmaxf(s[u][1], s[u][3]));
        }
        const bool first = um_first;
        um_first = false;
        rescale = first ||
                  __any_sync(0xffffffffu, tmx[0] > m_h[0] + kAbove || tmx[1] > m_h[1] + kAbove);
        if (rescale) {
          float mx[2] = {tmx[0], tmx[1]};
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], off));
            mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], off));
          }
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool outside =
                mx[e] > m_h[e] + kAbove || (UM && mx[e] < m_h[e] - kUmBelow);
            if (outside && mx[e] != -INFINITY) {
              // nothing accumulated before the first step (and a lowered
              // reference could make this factor overflow); a column still
              // empty gets 0, which keeps its empty state
              alpha[e] = first ? 1.f : dev::fast_exp2(m_h[e] - mx[e]);
              m_h[e] = mx[e];
              um_moved = true;
            }
            mref[e] = m_h[e] == -INFINITY ? 0.f : m_h[e];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < NPP; ++u) {
        const uint32_t p01 = mma::pack2(dev::fast_exp2(s[u][0] - mref[0]),
                                        dev::fast_exp2(s[u][1] - mref[1]), kBf16);
        const uint32_t p23 = mma::pack2(dev::fast_exp2(s[u][2] - mref[0]),
                                        dev::fast_exp2(s[u][3] - mref[1]), kBf16);
        // sums from the rounded weights, so numerator and denominator agree
        const float2 a = mma::unpack2(p01, kBf16), b = mma::unpack2(p23, kBf16);
        uint32_t pv01 = p01, pv23 = p23;  // weights times the per-token V scale
        if constexpr (TS) {
          pv01 = mma::pack2(a.x * vs_lo[u], a.y * vs_lo[u], kBf16);
          pv23 = mma::pack2(b.x * vs_hi[u], b.y * vs_hi[u], kBf16);
        }
        if (u == 0) {
          d_h[0] = fmaf(d_h[0], alpha[0], a.x + b.x);
          d_h[1] = fmaf(d_h[1], alpha[1], a.y + b.y);
        } else {
          d_h[0] += a.x + b.x;
          d_h[1] += a.y + b.y;
        }
        // P^T B fragments: transpose [token][head] -> [head][token] through smem
        uint16_t* pu = pT + u * 8 * P;
        pu[(2 * t) * P + g] = (uint16_t)(pv01 & 0xffffu);
        pu[(2 * t + 1) * P + g] = (uint16_t)(pv01 >> 16);
        pu[(2 * t) * P + g + 8] = (uint16_t)(pv23 & 0xffffu);
        pu[(2 * t + 1) * P + g + 8] = (uint16_t)(pv23 >> 16);
      }
      // once the running maxima settle, most steps leave them unchanged
      if (rescale && __any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
        for (int mt = 0; mt < MTILES; ++mt) {
          o[mt][0] *= alpha[0];
          o[mt][1] *= alpha[1];
          o[mt][2] *= alpha[0];
          o[mt][3] *= alpha[1];
        }
      }
      __syncwarp();
#pragma unroll
      for (int u = 0; u < NPP; ++u) {
        const uint16_t* pu = pT + u * 8 * P;
        const uint32_t pb0 = *reinterpret_cast<const uint32_t*>(pu + g * P + 2 * t);
        const uint32_t pb1 = *reinterpret_cast<const uint32_t*>(pu + g * P + 2 * t + 8);
        const uint32_t* vf = kEarlyV ? &vfrag[kEarlyV ? u : 0][0][0] : nullptr;
        if (valid[u] < P)
          pv_step(std::true_type{}, st[u], pb0, pb1, valid[u], vf);
        else
          pv_step(std::false_type{}, st[u], pb0, pb1, valid[u], vf);
        if constexpr (!kEarlyV) dev::release_stage(dev::smem_addr(&empty[stage[u]]), lane);
      }
    };

    // page split: page k to warp k % NW, one page a step; column split:
    // every page to every warp, NPP pages a step (the rest one at a time)
    {
      int k = CS ? kbase : kbase + (warp - kbase % NW + NW) % NW;
      if constexpr (C::NPP > 1) {
        for (; k + (C::NPP - 1) * PS < kbase + npg; k += C::NPP * PS)
          step(std::integral_constant<int, C::NPP>{}, k);
      }
      for (; k < kbase + npg; k += PS) step(std::integral_constant<int, 1>{}, k);
    }

    // ---- this warp's state: O^T rows -> dims, heads 2t and 2t+1
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      d_h[0] += __shfl_xor_sync(0xffffffffu, d_h[0], off);
      d_h[1] += __shfl_xor_sync(0xffffffffu, d_h[1], off);
    }
    if constexpr (UM) {
      if (__any_sync(0xffffffffu, um_moved) && lane == 0 && p.um_fallbacks)
        atomicAdd(p.um_fallbacks, 1);
      // a warp that drew no page holds no state: its reference must not
      // outweigh the others' in the combine
      if (um_first) m_h[0] = m_h[1] = -INFINITY;
    }
    // state slot of this warp's columns: its own row (page split) or the
    // columns' only state (column split); an idle warp of the column split
    // leaves its columns empty (m = -inf, d = 0, o = 0: what it holds)
    const int srow = CS ? 0 : warp;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int h = cb + 2 * t + e;  // column
      if (h < NC) {
#pragma unroll
        for (int mt = 0; mt < MTILES; ++mt) {
          const int dlo = kFp8 ? mt * 16 + 2 * g : mt * 16 + g;
          const int dhi = kFp8 ? mt * 16 + 2 * g + 1 : mt * 16 + g + 8;
          mo[(srow * NC + h) * D + dlo] = o[mt][e];
          mo[(srow * NC + h) * D + dhi] = o[mt][2 + e];
        }
        if (g == 0) {
          mm[srow * NC + h] = m_h[e];
          md[srow * NC + h] = d_h[e];
        }
      }
    }
    dev::named_barrier(1, CT);
    // the P^T buffers (NW x 256 bytes) are free between segments
    combine_and_emit<QT, D, G, NW, QL, RQ, C::NS>(p, mo, mm, md, qr, kvh, out_slot, sb.z, folds,
                                                  reinterpret_cast<float*>(smem + C::OFF_PT),
                                                  NW * 8 * P / 2);
    kbase += npg;
  }
  fold_pending<QT, D, G, NW, QL, RQ>(p, mo, folds, C::NS * NC * D);
  if (threadIdx.x == 0) pool_finish(p);
}

template <typename QT, typename KVT, int D, int G, int NW = 4, bool TS = false, int QL = 1,
          bool UM = false, bool RQ = false>
inline void fill_mma_kernel(DecodeKernel* k) {
  using C = MmaCfg<QT, KVT, D, G, NW, TS, QL>;
  k->func = reinterpret_cast<const void*>(&fa_decode_mma_kernel<QT, KVT, D, G, NW, TS, QL, UM, RQ>);
  k->merge_func = reinterpret_cast<const void*>(&fa_merge_partials_kernel<QT, D, G, QL, RQ>);
  k->threads = C::THREADS;
  k->smem_bytes = C::SMEM + 1024;  // room to align the ring to 1024 bytes
  k->stages = C::S;
  k->stage_bytes = C::STAGE_BYTES;
  k->group = G;
  k->head_dim = D;
  k->box_x = C::BOX_X;
  k->swizzle_128b = true;
  k->tensor_cores = true;
  k->token_scales = TS;
  k->q_len = QL;
  k->unified_max = UM;
  k->ragged_q = RQ;
}

}  // namespace fadecode

namespace fadecode {

// Dispatch over the compiled head_dim x group grid for one dtype pair: the
// tensor-core consumer where it applies and is allowed, the CUDA-core one
// otherwise.
template <typename QT, typename KVT>
inline bool find_kernel_for(int head_dim, int group, bool allow_mma, DecodeKernel* k) {
  constexpr bool kMmaTypes = sizeof(KVT) <= 2;
#define FA_CASE(DD, GG)                                                              \
  if (head_dim == DD && group == GG) {                                               \
    if constexpr (kMmaTypes && GG >= 2 && (DD * sizeof(KVT)) % 128 == 0) {           \
      if (allow_mma) {                                                               \
        fill_mma_kernel<QT, KVT, DD, GG>(k);                                         \
        return true;                                                                 \
      }                                                                              \
    }                                                                                \
    fill_kernel<QT, KVT, DD, GG>(k);                                                 \
    return true;                                                                     \
  }
  FA_CASE(64, 1) FA_CASE(64, 2) FA_CASE(64, 4) FA_CASE(64, 8)
  FA_CASE(128, 1) FA_CASE(128, 2) FA_CASE(128, 4) FA_CASE(128, 8)
#undef FA_CASE
  return false;
}

// Multi-token decode: tensor-core consumer, head_dim 128, group * q_len <= 8.
template <typename QT, typename KVT>
inline bool find_multi_token_kernel_for(int head_dim, int group, int q_len, DecodeKernel* k) {
  if (head_dim != 128) return false;
#define FA_QL_CASE(GG, QQ)                                 \
  if (group == GG && q_len == QQ) {                        \
    fill_mma_kernel<QT, KVT, 128, GG, 4, false, QQ>(k);    \
    return true;                                           \
  }
  FA_QL_CASE(1, 2) FA_QL_CASE(1, 4) FA_QL_CASE(1, 8)
  FA_QL_CASE(2, 2) FA_QL_CASE(2, 4) FA_QL_CASE(4, 2)
#undef FA_QL_CASE
  return false;
}

// Ragged query rows (qo_indptr): tensor-core consumer, head_dim 128, the
// smallest built bucket of query tokens per request that holds max_q: at most
// 8 columns (group x tokens) with the pages split over the warps, else up to
// 32 columns split over the warps (8 each).
template <typename QT, typename KVT>
inline bool find_ragged_q_kernel_for(int head_dim, int group, int max_q, DecodeKernel* k) {
  if (head_dim != 128 || max_q < 1) return false;
#define FA_RQ_CASE(GG, QQ)                                          \
  if (group == GG && max_q <= QQ) {                                 \
    fill_mma_kernel<QT, KVT, 128, GG, 4, false, QQ, false, true>(k); \
    return true;                                                    \
  }
  FA_RQ_CASE(1, 8) FA_RQ_CASE(1, 32) FA_RQ_CASE(2, 4) FA_RQ_CASE(2, 16)
  FA_RQ_CASE(4, 2) FA_RQ_CASE(4, 8) FA_RQ_CASE(8, 1) FA_RQ_CASE(8, 4)
#undef FA_RQ_CASE
  return false;
}

// Ragged query rows on the kernel of a request's 8-column tiles: a column
// split of `tiles` warps (8 x tiles columns: 2 or 3), each warp one tile.
template <typename QT, typename KVT>
inline bool find_ragged_q_tiles_kernel_for(int head_dim, int group, int tiles, DecodeKernel* k) {
  if (head_dim != 128) return false;
#define FA_RT_CASE(GG, TT)                                                           \
  if (group == GG && tiles == TT) {                                                  \
    fill_mma_kernel<QT, KVT, 128, GG, TT, false, 8 * TT / GG, false, true>(k);       \
    return true;                                                                     \
  }
  FA_RT_CASE(1, 2) FA_RT_CASE(1, 3) FA_RT_CASE(2, 2) FA_RT_CASE(2, 3)
  FA_RT_CASE(4, 2) FA_RT_CASE(4, 3) FA_RT_CASE(8, 2) FA_RT_CASE(8, 3)
#undef FA_RT_CASE
  return false;
}

// Unified-max softmax: tensor-core consumer, groups 2, 4, 8, rows of a
// whole number of 128 bytes (E4M3: head_dim 128).
template <typename QT, typename KVT>
inline bool find_unified_max_kernel_for(int head_dim, int group, DecodeKernel* k) {
#define FA_UM_CASE(DD, GG)                                       \
  if (head_dim == DD && group == GG) {                           \
    if constexpr ((DD * sizeof(KVT)) % 128 == 0) {               \
      fill_mma_kernel<QT, KVT, DD, GG, 4, false, 1, true>(k);    \
      return true;                                               \
    }                                                            \
    return false;                                                \
  }
  FA_UM_CASE(64, 2) FA_UM_CASE(64, 4) FA_UM_CASE(64, 8)
  FA_UM_CASE(128, 2) FA_UM_CASE(128, 4) FA_UM_CASE(128, 8)
#undef FA_UM_CASE
  return false;
}

// E4M3 KV with per-token scales: tensor-core consumer, head_dim 128, group 2..8.
template <typename QT>
inline bool find_token_scale_kernel_for(int head_dim, int group, DecodeKernel* k) {
  if (head_dim != 128) return false;
  if (group == 2) { fill_mma_kernel<QT, __nv_fp8_e4m3, 128, 2, 4, true>(k); return true; }
  if (group == 4) { fill_mma_kernel<QT, __nv_fp8_e4m3, 128, 4, 4, true>(k); return true; }
  if (group == 8) { fill_mma_kernel<QT, __nv_fp8_e4m3, 128, 8, 4, true>(k); return true; }
  return false;
}

}  // namespace fadecode
