// Cascade prefix attention on the fifth-generation tensor cores (tcgen05).
//
// The prefix pass is a real contraction: the query rows of one kv head (its
// query heads in every request, 128 rows a block) against every token of the
// shared prefix.  fa_prefix_kernel (cascade.cu) runs it on warp-level mma.sync,
// where the legacy tensor pipe and nine warps per SM bound it far below the
// GB300's tensor rate.  Here one CTA per SM works on one (kv head, prefix
// chunk) and on two 128-row blocks of that kv head's query rows at once (A
// and B, 256 rows; B is absent when the kv head has a single block), 64
// tokens (4 pages) at a time.  The two blocks share every K/V tile and give
// the tensor cores independent work: while the softmax of block A runs, the
// MMAs of block B proceed, and the other way round.
//
//  - warps 8 and 11 (TMA): K and V of a tile go into separate 5-slot rings,
//    filled by one warp each, each slot 8 tensor copies of 2 KB (4 pages x
//    two 64-dim halves), each half a [64 tokens][64 dims] 128-byte-swizzled
//    matrix.  A K slot comes free as soon as both blocks' Q K^T of it
//    completed, a V slot once both blocks' P V did.  Two issuing threads
//    keep twice the copies in flight that one does (a thread's copy
//    instructions stall while the memory system is busy).  Pages past the
//    chunk are fetched from an out-of-range page index, so the copy fills
//    them with zeros;
//  - warps 9 and 10 (MMA, one per block, one elected lane issuing): S = Q K^T
//    (M 128, N 64, K 128: 8 MMAs, Q and K K-major) into one of the block's
//    two TMEM score buffers, and O += P V (M 128, N 128, K 64: 4 MMAs, P read
//    from TMEM, V MN-major straight from its ring slot) into the block's
//    TMEM output accumulator.  The order is fixed: S(0), S(1), then per tile
//    j: P V(j) once P(j) is written, then S(j + 2) into the buffer P(j) just
//    left (MMAs of one thread run in issue order);
//  - warps 0-3 (block A) and 4-7 (block B), the softmax: thread r of a
//    warpgroup owns query row r of its block = TMEM lane r.  It loads its 64
//    scores with tcgen05.ld, keeps the row maximum and sum in registers (no
//    shuffles), writes its row of P as bf16/f16 over the first 32 columns of
//    the same score buffer (tcgen05.st), and rescales its row of O in TMEM
//    only when the maximum has grown by more than 2^8 - between rescales the
//    weights stay below 256, far inside the bf16/f16 and fp32 ranges.  At the
//    end it normalises O and writes the row's partial state (o,
//    log2-sum-exp) for fa_cascade_combine_kernel: o staged in the then idle
//    K/V ring and copied out with one bulk copy per row.
//
// The CTA's work item (kv head, chunk pages, rows) follows from its block
// index and the plan's sizes, so the first global loads - the TMA warps' page
// ids, the softmax threads' q rows - go out before the CTA-wide barrier.
//
// TMEM: all 512 columns - per block two score/P buffers of 64 columns and an
// output accumulator of 128 (A: S [0, 128), O [256, 384); B: S [128, 256),
// O [384, 512)).  Every wait is bounded (2 s); a wait that runs out sets bit
// 1 of the device-check word and the CTA drains, still freeing its TMEM.
#pragma once

namespace fadecode {
namespace tc {

constexpr int kD = 128;
constexpr int kTok = 64;                   // tokens per tile
constexpr int kPages = kTok / kPageSize;   // 4
constexpr int kSlots = 5;                  // depth of the K ring and of the V ring
constexpr int kHalf = kTok * 128;          // [64 tokens][64 dims], 128-byte rows
constexpr int kSlotBytes = 2 * kHalf;      // one tile of K (or V): both halves
constexpr int kQBytes = 2 * kPrefixRows * 128;  // one block's Q: two [128][64] halves
constexpr int kOffQ = 0;                        // Q of block A, then of block B
constexpr int kOffK = kOffQ + 2 * kQBytes;
constexpr int kOffV = kOffK + kSlots * kSlotBytes;
constexpr int kOffBar = kOffV + kSlots * kSlotBytes;
// k_full[n], k_empty[n], v_full[n], v_empty[n]; per block s_full[2],
// p_full[2], pv_done[2]; o_done[2], q_ready
constexpr int kBlockBars = 6;
constexpr int kNumBars = 4 * kSlots + 2 * kBlockBars + 3;
constexpr int kOffTmem = kOffBar + 8 * kNumBars;
constexpr int kSmem = kOffTmem + 16;
constexpr int kThreads = 384;  // 8 softmax warps, K and V TMA warps, an MMA warp per block
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleAbove = 8.f;       // log2 units

static_assert(32 % kPages == 0, "a warp's page-id load covers whole tiles");
static_assert(kOffK % 1024 == 0 && kSlotBytes % 1024 == 0 && kOffV % 1024 == 0,
              "swizzled operands need 1024-byte alignment");
static_assert(kSmem + 1024 <= 227 * 1024, "shared memory per CTA");
static_assert(256 * (kD * 4 + 16) <= 2 * kSlots * kSlotBytes,
              "the K/V ring holds the output rows of both blocks");

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

// Executed by a whole converged warp (warp-uniform operands); one elected
// lane issues.
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     bool accumulate) {
  asm volatile(
      "{\n.reg .pred e, p;\nelect.sync _|e, 0xffffffff;\nsetp.ne.b32 p, %4, 0;\n"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate));
}

__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile(
      "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(
          dev::smem_addr(bar))
      : "memory");
}

// Non-blocking probe of an mbarrier phase (try_wait may suspend the thread
// for a while, which would stall a scheduler polling several barriers).
// Called by a whole warp: lane 0's answer is everyone's.
__device__ __forceinline__ bool ready(const uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(dev::smem_addr(bar)), "r"(parity)
      : "memory");
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
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

// max(a, b, c) in one instruction
__device__ __forceinline__ float max3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}

// Two fp32 lanes in one 64-bit register, for the paired add / fma
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
  return v;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// O += P V with P (M x K, K-major, packed pairs per 32-bit column) in TMEM
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                        uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n.reg .pred e, p;\nelect.sync _|e, 0xffffffff;\nsetp.ne.b32 p, %4, 0;\n"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"((uint32_t)accumulate));
}

// 32 consecutive 32-bit columns of this thread's TMEM lane from packed words
__device__ __forceinline__ void st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

}  // namespace tc

// Prefix work of one CTA: the chunk of kv head h and row-block pair q:
// item_a = (h * row_blocks + 2q) * chunks + c and item_b = item_a + chunks
// (the next row block) when that block exists.
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
  uint64_t* k_full = bars;
  uint64_t* k_empty = bars + kSlots;
  uint64_t* v_full = bars + 2 * kSlots;
  uint64_t* v_empty = bars + 3 * kSlots;
  // per block X: s_full[2], p_full[2], pv_done[2]
  auto blk_bar = [&](int X, int which, int b) -> uint64_t* {
    return bars + 4 * kSlots + X * kBlockBars + 2 * which + b;
  };
  uint64_t* o_done = bars + 4 * kSlots + 2 * kBlockBars;  // [2], one per block
  uint64_t* q_ready = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int c = blockIdx.x % pp.chunks;
  const int pair = blockIdx.x / pp.chunks;
  const int h_kv = pair / pp.pair_blocks, rbp = pair % pp.pair_blocks;
  const int item_a = (h_kv * pp.row_blocks + 2 * rbp) * pp.chunks + c;
  const int nblk = (2 * rbp + 1 < pp.row_blocks) ? 2 : 1;
  // the plan's work items, derived here instead of read: chunk c holds
  // prefix pages [pb, pb + npg)
  const int kvh = h_kv;
  const int pb = (int)((int64_t)pp.prefix_pages * c / pp.chunks);
  const int npg = (int)((int64_t)pp.prefix_pages * (c + 1) / pp.chunks) - pb;
  const int tiles = (npg + kPages - 1) / kPages;
  const uint32_t sbase = dev::smem_addr(smem);

  // Loads that need no shared memory go out before the CTA-wide barrier
  // (they overlap the barrier set-up and the TMEM allocation): the TMA
  // warps' first window of page ids, the softmax threads' query rows.
  const int kv = warp == 11 ? 1 : 0;  // TMA warps: 8 loads K, 11 loads V
  auto load_ids = [&](int first) -> int {
    const int pos = first + lane;
    int id = -1;
    if (pos < npg) {
      id = __ldg(p.indices + pb + pos);
      if (id < 0 || (int64_t)id >= p.num_pages) {
        if (kv == 0) atomicOr(p.err, 1);
        id = -1;
      }
    }
    return id;
  };
  int ids = 0;
  if (warp == 8 || warp == 11) ids = load_ids(0);
  const int X = (warp / 4) & 1;       // softmax: block of this warpgroup
  const int r = threadIdx.x % 128;    // softmax: query row of the block = TMEM lane
  int row0 = 0, row_count = 0, out_item = 0;
  uint4 qv[kD / 8];
  if (warp < 8 && X < nblk) {
    row0 = (2 * rbp + X) * kPrefixRows;
    row_count = min(kPrefixRows, pp.rows - row0);
    out_item = item_a + X * pp.chunks;
    const int G = pp.group;
    const int rho = row0 + r;
    const QT* qrow = static_cast<const QT*>(pp.q) +
                     ((size_t)(rho / G) * p.num_qo_heads + (size_t)kvh * G + rho % G) * kD;
#pragma unroll
    for (int c8 = 0; c8 < kD / 8; ++c8)
      qv[c8] = r < row_count ? __ldg(reinterpret_cast<const uint4*>(qrow + c8 * 8))
                             : make_uint4(0u, 0u, 0u, 0u);
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      dev::mbar_init(dev::smem_addr(&k_full[s]), 1);
      dev::mbar_init(dev::smem_addr(&k_empty[s]), nblk);  // every block's Q K^T of the tile
      dev::mbar_init(dev::smem_addr(&v_full[s]), 1);
      dev::mbar_init(dev::smem_addr(&v_empty[s]), nblk);  // every block's P V of the tile
    }
    for (int X = 0; X < 2; ++X)
      for (int b = 0; b < 2; ++b) {
        dev::mbar_init(dev::smem_addr(blk_bar(X, 0, b)), 1);  // s_full
        dev::mbar_init(dev::smem_addr(blk_bar(X, 1, b)), 4);  // p_full
        dev::mbar_init(dev::smem_addr(blk_bar(X, 2, b)), 1);  // pv_done
      }
    dev::mbar_init(dev::smem_addr(&o_done[0]), 1);
    dev::mbar_init(dev::smem_addr(&o_done[1]), 1);
    dev::mbar_init(dev::smem_addr(q_ready), 4 * nblk);
    dev::fence_barrier_init();
  }
  if (warp == 9) {
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
  // block X: score/P buffers at columns X*128 + b*64, output at 256 + X*128
  bool aborted = false;

  if (warp == 8 || warp == 11) {
    // ---------------------------------------------------------------- TMA
    // Warp 8 fills the K ring, warp 11 the V ring.  Each lane holds one page
    // id of a 32-page window (eight tiles); lane 0 waits for ring slots and
    // issues the copies.
    if (lane == 0) dev::prefetch_tensormap(&kv_map);
    const uint64_t policy = dev::evict_first_policy();
    const int oob = (int)(2 * p.num_pages);  // beyond the last page: zero fill
    auto issue = [&](int t, int ids, uint64_t* full, uint64_t* empty, uint32_t ring, int kv) {
      int c3[kPages];
#pragma unroll
      for (int i = 0; i < kPages; ++i) {
        const int id = __shfl_sync(0xffffffffu, ids, (t * kPages + i) % 32);
        c3[i] = id < 0 ? oob : 2 * id + kv;
      }
      if (lane == 0) {
        const int s = t % kSlots;
        dev::mbar_wait(dev::smem_addr(&empty[s]), (uint32_t)(((t / kSlots) & 1) ^ 1), aborted,
                       p.err);
        const uint32_t fb = dev::smem_addr(&full[s]);
        dev::mbar_arrive_expect_tx(fb, kSlotBytes);
        const uint32_t st = ring + s * kSlotBytes;
#pragma unroll
        for (int i = 0; i < kPages; ++i) {
          const uint32_t row = (uint32_t)i * (kPageSize * 128);
          dev::tma_load_4d(st + row, &kv_map, 0, kvh, 0, c3[i], fb, policy);
          dev::tma_load_4d(st + kHalf + row, &kv_map, 64, kvh, 0, c3[i], fb, policy);
        }
      }
      __syncwarp();
    };
    uint64_t* full = kv ? v_full : k_full;
    uint64_t* empty = kv ? v_empty : k_empty;
    const uint32_t ring = sbase + (kv ? kOffV : kOffK);
    for (int t = 0; t < tiles; ++t) {
      if (t > 0 && (t * kPages) % 32 == 0) ids = load_ids(t * kPages);
      issue(t, ids, full, empty, ring, kv);
    }
    // no copy may still be landing when the CTA exits
    if (lane == 0)
      for (int t = tiles > kSlots ? tiles - kSlots : 0; t < tiles; ++t)
        if (!dev::mbar_wait_bounded(dev::smem_addr(&full[t % kSlots]),
                                    (uint32_t)((t / kSlots) & 1)))
          atomicOr(p.err, 2);
  } else if (warp == 9 || warp == 10) {
    // ---------------------------------------------------------------- MMA
    // Warp 9 issues block A's MMAs, warp 10 block B's: a converged warp, one
    // elected lane issuing, blocking waits.
    const int X = warp - 9;
    if (X < nblk) {
      dev::mbar_wait(dev::smem_addr(q_ready), 0u, aborted, p.err);
      aborted = __any_sync(0xffffffffu, aborted);
      fence_after();
      const uint32_t q_addr = sbase + kOffQ + X * kQBytes;
      const uint32_t tO = tmem + 256 + X * 128;
      auto qk = [&](int j) {
        const int s = j % kSlots, b = j & 1;
        dev::mbar_wait(dev::smem_addr(&k_full[s]), (uint32_t)((j / kSlots) & 1), aborted, p.err);
        fence_after();
        const uint32_t k_addr = sbase + kOffK + s * kSlotBytes;
        const uint32_t tS = tmem + X * 128 + b * kTok;
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) {  // 16 dims per MMA, 64 per 128-byte half
          const uint32_t off = (uint32_t)(k % 4) * 32;  // 32 bytes = 16 dims into the row
          umma(tS, smem_desc(q_addr + (k / 4) * (kPrefixRows * 128) + off, 16, 1024),
               smem_desc(k_addr + (k / 4) * kHalf + off, 16, 1024), kIdescQK, k > 0);
        }
        commit(blk_bar(X, 0, b));  // s_full
        commit(&k_empty[s]);
      };
      if (tiles > 0) qk(0);
      if (tiles > 1) qk(1);
      for (int j = 0; j < tiles; ++j) {
        const int s = j % kSlots, b = j & 1;
        dev::mbar_wait(dev::smem_addr(blk_bar(X, 1, b)), (uint32_t)((j >> 1) & 1), aborted,
                       p.err);
        dev::mbar_wait(dev::smem_addr(&v_full[s]), (uint32_t)((j / kSlots) & 1), aborted, p.err);
        fence_after();
        const uint32_t v_addr = sbase + kOffV + s * kSlotBytes;
        const uint32_t tP = tmem + X * 128 + b * kTok;  // P(j): 32 columns of packed pairs
#pragma unroll
        for (int k = 0; k < kTok / 16; ++k)  // 16 tokens (8 columns of P) per MMA
          umma_ts(tO, tP + k * 8, smem_desc(v_addr + k * 16 * 128, kHalf, 1024), kIdescPV,
                  j > 0 || k > 0);
        commit(blk_bar(X, 2, b));  // pv_done
        commit(&v_empty[s]);
        if (j + 2 < tiles) qk(j + 2);
        aborted = __any_sync(0xffffffffu, aborted);
      }
      commit(&o_done[X]);
      // TMEM is freed only after this block's last MMA completed
      if (!dev::mbar_wait_bounded(dev::smem_addr(&o_done[X]), 0u) && lane == 0) atomicOr(p.err, 2);
    }
  } else if (warp / 4 < nblk) {
    // ---------------------------------------------------------------- softmax
    const uint32_t lane_off = (uint32_t)(32 * (warp % 4)) << 16;
    const uint32_t tS0 = tmem + X * 128 + lane_off, tO = tmem + 256 + X * 128 + lane_off;
    uint64_t* s_full = blk_bar(X, 0, 0);
    uint64_t* p_full = blk_bar(X, 1, 0);
    uint64_t* pv_done = blk_bar(X, 2, 0);
    // Q row into the swizzled A tile: granule c8 (8 elements) of row r lands
    // in half c8 / 8 at granule (c8 % 8) ^ (r % 8)
    {
#pragma unroll
      for (int c8 = 0; c8 < kD / 8; ++c8) {
        const uint4 v = qv[c8];
        const uint32_t a = sbase + kOffQ + X * kQBytes + (c8 / 8) * (kPrefixRows * 128) +
                           r * 128 + (uint32_t)(((c8 % 8) ^ (r & 7)) * 16);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(dev::smem_addr(q_ready));
    }
    const float scale = pp.q_scale;  // log2-domain score scale (> 0)
    float m_ref = -INFINITY, d = 0.f;
    for (int j = 0; j < tiles; ++j) {
      const int b = j & 1;
      dev::mbar_wait(dev::smem_addr(&s_full[b]), (uint32_t)((j >> 1) & 1), aborted, p.err);
      fence_after();
      float s[kTok];
      {
        float lo[32], hi[32];
        ld32(tS0 + b * kTok, lo);
        ld32(tS0 + b * kTok + 32, hi);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = lo[i];
          s[32 + i] = hi[i];
        }
      }
      const int valid = min(kTok, (npg - j * kPages) * kPageSize);
      if (valid < kTok) {  // last tile of a ragged chunk
#pragma unroll
        for (int i = 0; i < kTok; ++i)
          if (i >= valid) s[i] = -INFINITY;
      }
      // row maximum of the raw scores: four chains of three-input maxima
      float m4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float m = s[16 * k];
#pragma unroll
        for (int i = 1; i < 15; i += 2) m = max3(m, s[16 * k + i], s[16 * k + i + 1]);
        m4[k] = fmaxf(m, s[16 * k + 15]);
      }
      const float mt = fmaxf(max3(m4[0], m4[1], m4[2]), m4[3]) * scale;
      // re-reference the row only when its maximum rose by more than 2^8
      const bool rebase = mt > m_ref + kRescaleAbove;
      const float m_new = rebase ? mt : m_ref;
      const float alpha = m_ref == -INFINITY ? 0.f : dev::fast_exp2(m_ref - m_new);
      if (j >= 1 && __any_sync(0xffffffffu, rebase)) {
        // O holds the tiles before j: wait for P V of tile j-1, then scale
        dev::mbar_wait(dev::smem_addr(&pv_done[(j - 1) & 1]), (uint32_t)(((j - 1) >> 1) & 1),
                       aborted, p.err);
        fence_after();
        const float f = rebase ? alpha : 1.f;
#pragma unroll
        for (int cc = 0; cc < kD / 32; ++cc) {
          float v[32];
          ld32(tO + cc * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= f;
          st32(tO + cc * 32, v);
        }
      }
      if (rebase) {
        d *= alpha;
        m_ref = m_new;
      }
      // P row: weights 2^(s * scale - m) for pairs of scores (paired fma),
      // rounded to the MMA type for P V; the row sum takes the fp32 weights
      // (paired adds, four accumulators)
      const uint64_t scale2 = f2(scale, scale), neg_m2 = f2(-m_ref, -m_ref);
      uint32_t pk[kTok / 2];
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};  // +0.0f in both lanes
#pragma unroll
      for (int i = 0; i < kTok / 2; ++i) {
        float x0, x1;
        f2_split(fma2(f2(s[2 * i], s[2 * i + 1]), scale2, neg_m2), x0, x1);
        const float a0 = dev::fast_exp2(x0), a1 = dev::fast_exp2(x1);
        pk[i] = mma::pack2(a0, a1, kBf16);
        acc[i % 4] = add2(acc[i % 4], f2(a0, a1));
      }
      {
        float lo, hi;
        f2_split(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])), lo, hi);
        d += lo + hi;
      }
      // P over the first 32 columns of the score buffer it came from
      st32u(tS0 + b * kTok, pk);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      fence_before();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(dev::smem_addr(&p_full[b]));
    }
    // ---- this row's partial state: o / d and log2-sum-exp
    // Both blocks' MMAs are done once both o_done fired; from then on the
    // K/V ring is idle and stages the rows: each thread writes its row of o
    // (rows 528 bytes apart, so that a warp's 16-byte stores fall in distinct
    // banks) and copies it out with one 512-byte bulk copy.
    dev::mbar_wait(dev::smem_addr(&o_done[0]), 0u, aborted, p.err);
    if (nblk > 1) dev::mbar_wait(dev::smem_addr(&o_done[1]), 0u, aborted, p.err);
    fence_after();
    const float inv = d > 0.f ? 1.f / d : 0.f;
    constexpr uint32_t kRowPitch = kD * 4 + 16;
    const uint32_t srow = sbase + kOffK + (uint32_t)threadIdx.x * kRowPitch;
#pragma unroll
    for (int cc = 0; cc < kD / 32; ++cc) {
      float v[32];
      if (tiles > 0) {
        ld32(tO + cc * 32, v);  // every lane of the warp takes part
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;  // no tile: O was never written
      }
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(srow + (cc * 32 + i) * 4),
                     "f"(v[i] * inv), "f"(v[i + 1] * inv), "f"(v[i + 2] * inv),
                     "f"(v[i + 3] * inv)
                     : "memory");
    }
    if (r < row_count) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      float* dst = pp.part_o + ((size_t)out_item * kPrefixRows + r) * kD;
      asm volatile(
          "cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n\t"
          "cp.async.bulk.commit_group;\n\t"
          "cp.async.bulk.wait_group.read 0;" ::"l"(dst),
          "r"(srow), "n"(kD * 4)
          : "memory");
      pp.part_lse[(size_t)out_item * kPrefixRows + r] =
          d > 0.f ? m_ref + dev::fast_log2(d) : -INFINITY;
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 9) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace fadecode
