// Cascade prefix attention on the fifth-generation tensor cores (tcgen05).
//
// The prefix pass is a real contraction: 128 query rows (the query heads of
// every request that reads one kv head) against every token of the shared
// prefix.  fa_prefix_kernel (cascade.cu) runs it on warp-level mma.sync,
// where the legacy tensor pipe and nine warps per SM bound it far below the
// GB300's tensor rate.  Here one CTA per SM works on one (kv head, 128-row
// block, prefix chunk) item, 64 tokens (4 pages) at a time:
//
//  - warp 4 (TMA): per tile, 16 tensor copies of 2 KB (4 pages x {K, V} x two
//    64-dim halves) into a 4-stage ring, each half-block a [64 tokens][64
//    dims] 128-byte-swizzled matrix.  Pages past the chunk are fetched from
//    an out-of-range page index, so the copy fills them with zeros;
//  - warp 5 (MMA, one lane): S[b] = Q K^T (M 128, N 64, K 128: 8 MMAs, Q and
//    K K-major) into one of two TMEM score buffers, then, once the softmax
//    has written P for the previous tile, O += P V (M 128, N 128, K 64: 4
//    MMAs, V read MN-major straight from the ring) into the TMEM output
//    accumulator; tcgen05.commit signals each step's mbarrier;
//  - warps 0-3 (softmax): thread r owns query row r = TMEM lane r.  It loads
//    its 64 scores with tcgen05.ld, keeps the row maximum and sum in
//    registers (no shuffles), writes its row of P as bf16/f16 into a
//    swizzled shared-memory tile for the next MMA, and rescales its row of
//    O in TMEM (tcgen05.ld / st) only when the maximum has grown by more than
//    2^8 - between rescales the weights stay below 256, far inside the
//    bf16/f16 and fp32 ranges.  At the end it normalises O and writes the
//    row's partial state (o, log2-sum-exp) for fa_cascade_combine_kernel.
//
// TMEM: 256 columns - S0 [0, 64), S1 [64, 128), O [128, 256).  Every wait is
// bounded (2 s); a wait that runs out sets bit 1 of the device-check word and
// the CTA drains, still freeing its TMEM.
#pragma once

namespace fadecode {
namespace tc {

constexpr int kD = 128;
constexpr int kTok = 64;                   // tokens per tile
constexpr int kPages = kTok / kPageSize;   // 4
constexpr int kStages = 4;
constexpr int kBlock = kTok * 128;         // [64 rows][128 bytes]
constexpr int kStageBytes = 4 * kBlock;    // K lo, K hi, V lo, V hi
constexpr int kQBytes = 2 * kPrefixRows * 128;
constexpr int kPBytes = kPrefixRows * 128;
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kQBytes;
constexpr int kOffP = kOffKV + kStages * kStageBytes;
constexpr int kOffBar = kOffP + 2 * kPBytes;
// kv_full[4], kv_empty[4], s_full[2], s_free[2], p_full[2], p_free[2], o_done, q_ready
constexpr int kNumBars = 2 * kStages + 10;
constexpr int kOffTmem = kOffBar + 8 * kNumBars;
constexpr int kSmem = kOffTmem + 16;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr float kRescaleAbove = 8.f;       // log2 units

static_assert(32 % kPages == 0, "a warp's page-id load covers whole tiles");
static_assert(kOffKV % 1024 == 0 && kStageBytes % 1024 == 0 && kOffP % 1024 == 0,
              "swizzled operands need 1024-byte alignment");

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  // tcgen05 shared-memory matrix descriptor: start, leading and stride byte
  // offsets (16-byte units), version 1, 128-byte swizzle
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f16 instruction descriptor: fp32 accumulator, A and B both bf16 or
// both f16, A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1).
__host__ __device__ constexpr uint32_t instr_desc(bool bf16, int m, int n, int b_mn) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     bool accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate));
}

__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          dev::smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

}  // namespace tc

template <typename QT>
__global__ void __launch_bounds__(tc::kThreads, 1)
    fa_prefix_tc_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p,
                        const PrefixParams pp) {
  using namespace tc;
  constexpr bool kBf16 = std::is_same<QT, __nv_bfloat16>::value;
  constexpr uint32_t kIdescQK = instr_desc(kBf16, 128, kTok, 0);
  constexpr uint32_t kIdescPV = instr_desc(kBf16, 128, kD, 1);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (dev::smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + kStages;
  uint64_t* s_full = bars + 2 * kStages;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* p_free = p_full + 2;
  uint64_t* o_done = p_free + 2;
  uint64_t* q_ready = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x;
  const int4 sa = *reinterpret_cast<const int4*>(p.segments + 8 * item);
  const int4 sb = *reinterpret_cast<const int4*>(p.segments + 8 * item + 4);
  const int row0 = sa.x, kvh = sa.y, pb = sa.z, npg = sa.w - sa.z, row_count = sb.x;
  const int out_item = sb.y;
  const int tiles = (npg + kPages - 1) / kPages;
  const uint32_t sbase = dev::smem_addr(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      dev::mbar_init(dev::smem_addr(&kv_full[s]), 1);
      dev::mbar_init(dev::smem_addr(&kv_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      dev::mbar_init(dev::smem_addr(&s_full[b]), 1);
      dev::mbar_init(dev::smem_addr(&s_free[b]), 4);
      dev::mbar_init(dev::smem_addr(&p_full[b]), 4);
      dev::mbar_init(dev::smem_addr(&p_free[b]), 1);
    }
    dev::mbar_init(dev::smem_addr(o_done), 1);
    dev::mbar_init(dev::smem_addr(q_ready), 4);
    dev::fence_barrier_init();
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dev::smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 2 * kTok;
  bool aborted = false;

  if (warp == 4) {
    // ---------------------------------------------------------------- TMA
    // The warp reads the page ids 32 at a time (eight tiles' worth, one per
    // lane); lane 0 waits for ring stages and issues the copies.
    if (lane == 0) dev::prefetch_tensormap(&kv_map);
    const uint64_t policy = dev::evict_first_policy();
    const int oob = (int)(2 * p.num_pages);  // beyond the last page: zero fill
    int ids = 0;
    for (int j = 0; j < tiles; ++j) {
      const int first = j * kPages;  // page position within the chunk
      if (first % 32 == 0) {
        const int pos = first + lane;
        int id = -1;
        if (pos < npg) {
          id = __ldg(p.indices + pb + pos);
          if (id < 0 || (int64_t)id >= p.num_pages) {
            atomicOr(p.err, 1);
            id = -1;
          }
        }
        ids = id;
      }
      int c3[kPages];
#pragma unroll
      for (int i = 0; i < kPages; ++i) {
        const int id = __shfl_sync(0xffffffffu, ids, (first + i) % 32);
        c3[i] = id < 0 ? oob : 2 * id;
      }
      if (lane == 0) {
        const int s = j % kStages;
        dev::mbar_wait(dev::smem_addr(&kv_empty[s]), (uint32_t)(((j / kStages) & 1) ^ 1),
                       aborted, p.err);
        const uint32_t fb = dev::smem_addr(&kv_full[s]);
        dev::mbar_arrive_expect_tx(fb, kStageBytes);
        const uint32_t st = sbase + kOffKV + s * kStageBytes;
#pragma unroll
        for (int i = 0; i < kPages; ++i) {
          const uint32_t row = (uint32_t)i * (kPageSize * 128);
          dev::tma_load_4d(st + 0 * kBlock + row, &kv_map, 0, kvh, 0, c3[i], fb, policy);
          dev::tma_load_4d(st + 1 * kBlock + row, &kv_map, 64, kvh, 0, c3[i], fb, policy);
          dev::tma_load_4d(st + 2 * kBlock + row, &kv_map, 0, kvh, 0, c3[i] + 1, fb, policy);
          dev::tma_load_4d(st + 3 * kBlock + row, &kv_map, 64, kvh, 0, c3[i] + 1, fb, policy);
        }
      }
      __syncwarp();
    }
    // no copy may still be landing when the CTA exits
    if (lane == 0)
      for (int j = tiles > kStages ? tiles - kStages : 0; j < tiles; ++j)
        if (!dev::mbar_wait_bounded(dev::smem_addr(&kv_full[j % kStages]),
                                    (uint32_t)((j / kStages) & 1)))
          atomicOr(p.err, 2);
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t q_addr = sbase + kOffQ, p_addr = sbase + kOffP;
      auto pv = [&](int i) {
        const int b = i & 1, s = i % kStages;
        dev::mbar_wait(dev::smem_addr(&p_full[b]), (uint32_t)((i >> 1) & 1), aborted, p.err);
        fence_after();
        const uint32_t v_addr = sbase + kOffKV + s * kStageBytes + 2 * kBlock;
#pragma unroll
        for (int k = 0; k < kTok / 16; ++k)  // 16 tokens per MMA
          umma(tO, smem_desc(p_addr + b * kPBytes + k * 32, 16, 1024),
              smem_desc(v_addr + k * 16 * 128, kBlock, 1024), kIdescPV, i > 0 || k > 0);
        commit(&p_free[b]);
        commit(&kv_empty[s]);
      };
      dev::mbar_wait(dev::smem_addr(q_ready), 0u, aborted, p.err);
      fence_after();
      for (int j = 0; j < tiles; ++j) {
        const int s = j % kStages, b = j & 1;
        dev::mbar_wait(dev::smem_addr(&kv_full[s]), (uint32_t)((j / kStages) & 1), aborted,
                       p.err);
        if (j >= 2)
          dev::mbar_wait(dev::smem_addr(&s_free[b]), (uint32_t)(((j - 2) >> 1) & 1), aborted,
                         p.err);
        fence_after();
        const uint32_t k_addr = sbase + kOffKV + s * kStageBytes;
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) {  // 16 dims per MMA, 64 per 128-byte block
          const uint32_t off = (uint32_t)(k % 4) * 32;  // 32 bytes = 16 dims into the row
          umma(tS + b * kTok, smem_desc(q_addr + (k / 4) * (kPrefixRows * 128) + off, 16, 1024),
              smem_desc(k_addr + (k / 4) * kBlock + off, 16, 1024), kIdescQK, k > 0);
        }
        commit(&s_full[b]);
        if (j >= 1) pv(j - 1);
      }
      if (tiles > 0) pv(tiles - 1);
      commit(o_done);
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int r = threadIdx.x;  // query row of the block = TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    // Q row into the swizzled A tile: granule c8 (8 elements) of row r lands
    // in block c8 / 8 at granule (c8 % 8) ^ (r % 8)
    {
      const int G = pp.group;
      const int rho = row0 + r;
      const bool live = r < row_count;
      const QT* qrow = static_cast<const QT*>(pp.q) +
                       ((size_t)(rho / G) * p.num_qo_heads + (size_t)kvh * G + rho % G) * kD;
#pragma unroll
      for (int c8 = 0; c8 < kD / 8; ++c8) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (live) v = __ldg(reinterpret_cast<const uint4*>(qrow + c8 * 8));
        const uint32_t a = sbase + kOffQ + (c8 / 8) * (kPrefixRows * 128) + r * 128 +
                           (uint32_t)(((c8 % 8) ^ (r & 7)) * 16);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(dev::smem_addr(q_ready));
    }
    float m_ref = -INFINITY, d = 0.f;
    for (int j = 0; j < tiles; ++j) {
      const int b = j & 1;
      dev::mbar_wait(dev::smem_addr(&s_full[b]), (uint32_t)((j >> 1) & 1), aborted, p.err);
      fence_after();
      float s[kTok];
      {
        float lo[32], hi[32];
        ld32(tS + lane_off + b * kTok, lo);
        ld32(tS + lane_off + b * kTok + 32, hi);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = lo[i];
          s[32 + i] = hi[i];
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(dev::smem_addr(&s_free[b]));
      const int valid = min(kTok, (npg - j * kPages) * kPageSize);
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < kTok; ++i) {
        s[i] = i < valid ? s[i] * pp.q_scale : -INFINITY;
        mt = fmaxf(mt, s[i]);
      }
      // re-reference the row only when its maximum rose by more than 2^8
      const bool rebase = mt > m_ref + kRescaleAbove;
      const float m_new = rebase ? mt : m_ref;
      const float alpha = m_ref == -INFINITY ? 0.f : dev::fast_exp2(m_ref - m_new);
      if (j >= 1 && __any_sync(0xffffffffu, rebase)) {
        // O holds the tiles before j: wait for P.V of tile j-1, then scale
        dev::mbar_wait(dev::smem_addr(&p_free[(j - 1) & 1]), (uint32_t)(((j - 1) >> 1) & 1),
                       aborted, p.err);
        fence_after();
        const float f = rebase ? alpha : 1.f;
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          float v[32];
          ld32(tO + lane_off + c * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= f;
          st32(tO + lane_off + c * 32, v);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      if (rebase) {
        d *= alpha;
        m_ref = m_new;
      }
      // P row: weights rounded to the MMA type, sums from the rounded values
      uint32_t pk[kTok / 2];
#pragma unroll
      for (int i = 0; i < kTok / 2; ++i) {
        const float a0 = dev::fast_exp2(s[2 * i] - m_ref), a1 = dev::fast_exp2(s[2 * i + 1] - m_ref);
        pk[i] = mma::pack2(a0, a1, kBf16);
        const float2 back = mma::unpack2(pk[i], kBf16);
        d += back.x + back.y;
      }
      if (j >= 2)  // P buffer b was read by P.V of tile j-2
        dev::mbar_wait(dev::smem_addr(&p_free[b]), (uint32_t)(((j - 2) >> 1) & 1), aborted,
                       p.err);
      const uint32_t prow = sbase + kOffP + b * kPBytes + r * 128;
#pragma unroll
      for (int g8 = 0; g8 < kTok / 8; ++g8) {
        const uint32_t a = prow + (uint32_t)((g8 ^ (r & 7)) * 16);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(pk[4 * g8]),
                     "r"(pk[4 * g8 + 1]), "r"(pk[4 * g8 + 2]), "r"(pk[4 * g8 + 3])
                     : "memory");
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      fence_before();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(dev::smem_addr(&p_full[b]));
    }
    // ---- this row's partial state: o / d and log2-sum-exp
    dev::mbar_wait(dev::smem_addr(o_done), 0u, aborted, p.err);
    fence_after();
    const float inv = d > 0.f ? 1.f / d : 0.f;
    float* dst = pp.part_o + ((size_t)out_item * kPrefixRows + r) * kD;
#pragma unroll
    for (int c = 0; c < kD / 32; ++c) {
      float v[32];
      if (tiles > 0) {
        ld32(tO + lane_off + c * 32, v);  // every lane of the warp takes part
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;  // no tile: O was never written
      }
      if (r < row_count) {
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(dst + c * 32 + i) =
              make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv, v[i + 3] * inv);
      }
    }
    if (r < row_count)
      pp.part_lse[(size_t)out_item * kPrefixRows + r] =
          d > 0.f ? m_ref + dev::fast_log2(d) : -INFINITY;
  }
  fence_before();
  __syncthreads();
  if (warp == 5) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace fadecode
