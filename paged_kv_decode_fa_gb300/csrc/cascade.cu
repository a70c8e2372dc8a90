// Cascade decode: a batch whose requests all start with the same shared
// prefix (whole pages, e.g. a system prompt) plus a suffix of their own.
//
// Page "GitHub Spotlight: FlashInfer" (sections "Core Superpowers" and
// "Scenario A: Enterprise Retrieval-Augmented Generation") describes cascade
// attention: the shared prefix is attended once for all the requests that
// share it and the result is combined with each request's own part; the
// combination is the merge rule of section "FlashDecoding - the split-KV
// trick" on the page "FlashDecoding + FlashInfer".  Plain decode reads the
// prefix once per request; here it is read once per kv head and row block:
//
//  1. suffix: the regular split-KV decode over each request's own pages
//     (fa_decode_plan / fa_decode_run), into workspace buffers;
//  2. prefix: fa_prefix_kernel - for one kv head, the rows are the query
//     heads of every request that read it (request b, head j -> row b*G + j);
//     each consumer warp owns 16 rows and every warp consumes every staged
//     page, so a page is fetched from HBM once per 128 rows.  Per page a warp
//     computes S[16 rows x 16 tokens] = Q K^T and O += P V with m16n8k16 MMAs;
//     the score C fragments are reused directly as the A fragment of P.V.
//     The prefix is cut into page chunks for parallelism; each (kv head, row
//     block, chunk) writes an fp32 partial state per row;
//  3. fa_cascade_combine_kernel folds, per (request, qo head), the prefix
//     chunks and the suffix state with the merge rule.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "decode_mma.cuh"
#include "fa_decode.h"
#include "staging.h"

namespace fadecode {

struct PrefixParams {
  const void* q;        // [B, Hq, D]
  float* part_o;        // [items][128 rows][D], normalised
  float* part_lse;      // [items][128 rows], log2 domain
  int group;            // query heads per kv head
  float q_scale;        // sm_scale * k_scale * log2(e)
  float v_scale;        // applied to the partial outputs (E4M3 KV; 1 otherwise)
  int row_blocks;       // 128-row blocks per kv head
  int pair_blocks;      // pairs of row blocks per kv head (tcgen05 kernel)
  int chunks;           // prefix chunks
  int rows;             // query rows per kv head (batch x group)
  int prefix_pages;     // pages of the shared prefix
};

struct CombineParams {
  const float* part_o;
  const float* part_lse;
  const void* suffix_o;   // [B, Hq, D] q dtype
  const float* suffix_lse;  // [B, Hq], natural log
  void* o;                // [B, Hq, D] q dtype
  float* lse;             // [B, Hq] or nullptr
  int batch, num_qo_heads, group, row_blocks, chunks;
};

constexpr int kPrefixRows = 128;  // rows per CTA: 8 consumer warps x 16

template <typename KVT, int D, int NW>
struct PrefixCfg {
  static constexpr int P = kPageSize;
  static constexpr int KV_ES = sizeof(KVT);
  static constexpr bool kFp8 = KV_ES == 1;
  static constexpr int SEGS = D * KV_ES / 128;    // 128-byte row segments
  static constexpr int BOX_X = 128 / KV_ES;       // elements per box row
  static constexpr int BOX_BYTES = 2 * P * 128;
  static constexpr int STAGE_BYTES = SEGS * BOX_BYTES;
  static constexpr int KSTEPS = D / 16;
  static constexpr int NT = D / 8;                // output n-tiles of 8 dims
  static constexpr int S = 8;
  static constexpr int THREADS = (NW + 1) * 32;
  static constexpr int OFF_FULL = S * STAGE_BYTES;
  static constexpr int OFF_EMPTY = OFF_FULL + 8 * S;
  static constexpr int SMEM = OFF_EMPTY + 8 * S;
  static_assert(NW * 16 == kPrefixRows, "16 rows per consumer warp");
  static_assert((D * KV_ES) % 128 == 0, "rows must be whole 128-byte swizzle rows");
  static_assert(!kFp8 || D == 128, "E4M3 prefix rows are laid out for head_dim 128");
};

// The prefix pass on warp-level MMAs.  16-bit KV: the MMA type is the KV
// type and q is its A fragment as stored.  E4M3 KV: the MMAs run in f16 -
// K and V are widened in registers (exact), q is scaled by a power of two
// per warp into f16 range (the scores are scaled back), k_scale is folded
// into q_scale and v_scale into the partial outputs.
template <typename QT, typename KVT, int D, int NW>
__global__ void __launch_bounds__(PrefixCfg<KVT, D, NW>::THREADS)
    fa_prefix_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p,
                     const PrefixParams pp) {
  using C = PrefixCfg<KVT, D, NW>;
  constexpr int P = C::P, S = C::S, SEGS = C::SEGS, KSTEPS = C::KSTEPS, NT = C::NT;
  constexpr bool kFp8 = C::kFp8;
  constexpr bool kQBf16 = std::is_same<QT, __nv_bfloat16>::value;
  // MMA operand type: the KV type for 16-bit KV, f16 for E4M3
  constexpr bool kBf16 = !kFp8 && kQBf16;
  static_assert(kFp8 || std::is_same<QT, KVT>::value, "16-bit KV: q of the same type");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (dev::smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_FULL);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + C::OFF_EMPTY);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      dev::mbar_init(dev::smem_addr(&full[s]), 1);
      dev::mbar_init(dev::smem_addr(&empty[s]), NW);  // every consumer warp releases
    }
    dev::fence_barrier_init();
  }
  __syncthreads();
  if (warp == NW) {
    produce_pages<S, C::STAGE_BYTES, SEGS, C::BOX_X, C::BOX_BYTES>(&kv_map, p, item, item + 1,
                                                                   ring, full, empty, lane);
    return;
  }

  const int4 sa = *reinterpret_cast<const int4*>(p.segments + 8 * item);
  const int4 sb = *reinterpret_cast<const int4*>(p.segments + 8 * item + 4);
  const int row0 = sa.x, kvh = sa.y, npg = sa.w - sa.z, row_count = sb.x;
  const int G = pp.group;
  const int g = lane >> 2, t = lane & 3;
  const int r_lo = warp * 16 + g, r_hi = r_lo + 8;  // rows within the block

  // Q as the A fragment for the whole chunk, reduction index permuted as in
  // the decode kernels.  16-bit KV: step j = 4*seg + 2*half + u covers dims
  // seg*64 + (2t + half)*8 + 4u .. +3 (a0/a1 the first two, a2/a3 the last).
  // E4M3 KV: step j covers dims 32t + 4j .. +3, the four bytes word j%4 of
  // granule 2t + j/4 of a K row holds.
  uint32_t qa[KSTEPS][4];
  float qscale = pp.q_scale;
  {
    const QT* qbase = static_cast<const QT*>(pp.q);
    const int rows[2] = {r_lo, r_hi};
    uint32_t raw[2][KSTEPS][2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int rho = row0 + rows[rr];
      const bool live = rows[rr] < row_count;
      const QT* qrow = qbase + ((size_t)(rho / G) * p.num_qo_heads + kvh * G + rho % G) * D;
#pragma unroll
      for (int L = 0; L < KSTEPS / 2; ++L) {
        const int d0 = kFp8 ? 32 * t + 8 * L : (L >> 1) * 64 + (2 * t + (L & 1)) * 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (live) v = __ldg(reinterpret_cast<const uint4*>(qrow + d0));
        raw[rr][2 * L][0] = v.x;
        raw[rr][2 * L][1] = v.y;
        raw[rr][2 * L + 1][0] = v.z;
        raw[rr][2 * L + 1][1] = v.w;
      }
    }
    if constexpr (kFp8) {
      // f16 MMAs: q times 2^shift (one shift per warp) with its largest
      // magnitude in [2^14, 2^15); the scores are scaled back by qscale
      float amax = 0.f;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int j = 0; j < KSTEPS; ++j)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float2 f = mma::unpack2(raw[rr][j][h], kQBf16);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
      const unsigned bits = __reduce_max_sync(0xffffffffu, __float_as_uint(amax));
      int shift = 0;
      if (bits != 0u && bits < 0x7f800000u) {
        const int ex = (int)((bits >> 23) & 0xff) - 127;
        shift = min(max(14 - ex, -120), 120);
      }
      const float up = ldexpf(1.f, shift);
      qscale = pp.q_scale * ldexpf(1.f, -shift);
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int j = 0; j < KSTEPS; ++j)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float2 f = mma::unpack2(raw[rr][j][h], kQBf16);
            raw[rr][j][h] = mma::pack2(f.x * up, f.y * up, false);
          }
    }
#pragma unroll
    for (int j = 0; j < KSTEPS; ++j) {
      qa[j][0] = raw[0][j][0];
      qa[j][1] = raw[1][j][0];
      qa[j][2] = raw[0][j][1];
      qa[j][3] = raw[1][j][1];
    }
  }

  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, d_r[2] = {0.f, 0.f};  // rows g, g+8
  bool aborted = false;
  const uint32_t ring_addr = dev::smem_addr(ring);

  for (int k = 0; k < npg; ++k) {
    const int stage = k % S;
    dev::mbar_wait(dev::smem_addr(&full[stage]), (uint32_t)((k / S) & 1), aborted, p.err);
    const uint32_t st = ring_addr + stage * C::STAGE_BYTES;

    // ---- S[rows][tokens]: n-tile 0 = tokens 0..7 (K row g), 1 = tokens 8..15;
    // two accumulators per n-tile (even / odd reduction steps) halve the
    // dependent MMA chain
    float acc[2][2][4] = {};
    const int sw = g & 7;
#pragma unroll
    for (int sgi = 0; sgi < SEGS; ++sgi) {
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        const uint32_t gran = (uint32_t)(((2 * t + qq) ^ sw) * 16);
        const uint4 k0 = mma::lds128(st + sgi * C::BOX_BYTES + g * 128 + gran);
        const uint4 k1 = mma::lds128(st + sgi * C::BOX_BYTES + (g + 8) * 128 + gran);
        const uint32_t w0[4] = {k0.x, k0.y, k0.z, k0.w};
        const uint32_t w1[4] = {k1.x, k1.y, k1.z, k1.w};
        if constexpr (kFp8) {
          // word w: dims 32t + 16qq + 4w .. +3 of K rows g / g+8, widened to
          // the B fragment (b0: the first two dims, b1: the last two)
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int j = qq * 4 + w;
            uint32_t b0, b1, c0, c1;
            mma::e4m3x4_to_f16x2x2(w0[w], b0, b1);
            mma::e4m3x4_to_f16x2x2(w1[w], c0, c1);
            mma::mma16816<false>(acc[0][j & 1], qa[j][0], qa[j][1], qa[j][2], qa[j][3], b0, b1);
            mma::mma16816<false>(acc[1][j & 1], qa[j][0], qa[j][1], qa[j][2], qa[j][3], c0, c1);
          }
        } else {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int j = sgi * 4 + qq * 2 + u;
            mma::mma16816<kBf16>(acc[0][u], qa[j][0], qa[j][1], qa[j][2], qa[j][3], w0[2 * u],
                                 w0[2 * u + 1]);
            mma::mma16816<kBf16>(acc[1][u], qa[j][0], qa[j][1], qa[j][2], qa[j][3], w1[2 * u],
                                 w1[2 * u + 1]);
          }
        }
      }
    }
    float sc[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[n][e] = acc[n][0][e] + acc[n][1][e];
    // lane holds rows g (e = 0, 1) and g+8 (e = 2, 3) x tokens 2t, 2t+1 (+8)
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[n][e] *= qscale;
    float mx[2] = {fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1])),
                   fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]))};
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], off));
      mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], off));
    }
    float alpha[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float mn = fmaxf(m_r[r], mx[r]);
      alpha[r] = dev::fast_exp2(m_r[r] - mn);
      m_r[r] = mn;
    }
    // P as the A fragment of P.V: a0 = row g tokens 2t..(n-tile 0),
    // a1 = row g+8, a2/a3 the same for tokens 8+2t..
    uint32_t pa[4];
    float ps[2] = {0.f, 0.f};
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      const uint32_t lo = mma::pack2(dev::fast_exp2(sc[n][0] - m_r[0]),
                                     dev::fast_exp2(sc[n][1] - m_r[0]), kBf16);
      const uint32_t hi = mma::pack2(dev::fast_exp2(sc[n][2] - m_r[1]),
                                     dev::fast_exp2(sc[n][3] - m_r[1]), kBf16);
      pa[2 * n] = lo;
      pa[2 * n + 1] = hi;
      const float2 a = mma::unpack2(lo, kBf16), b = mma::unpack2(hi, kBf16);
      ps[0] += a.x + a.y;
      ps[1] += b.x + b.y;
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      ps[0] += __shfl_xor_sync(0xffffffffu, ps[0], off);
      ps[1] += __shfl_xor_sync(0xffffffffu, ps[1], off);
    }
    d_r[0] = d_r[0] * alpha[0] + ps[0];
    d_r[1] = d_r[1] * alpha[1] + ps[1];
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][0] *= alpha[0];
        o[n][1] *= alpha[0];
        o[n][2] *= alpha[1];
        o[n][3] *= alpha[1];
      }
    }
    // ---- O[rows][dims] += P V: B fragments of V from ldmatrix.trans
    if constexpr (kFp8) {
      // a granule holds 16 dims of 8 tokens as 8 byte pairs; transposed as
      // 16-bit elements, a lane gets dim pair g of tokens 2t, 2t+1 (and of
      // 8+2t, 9+2t), split with one byte permute into the f16 B fragments of
      // dim 2g (n-tile 2*gran) and dim 2g+1 (n-tile 2*gran+1): n-tile
      // 2*gran + e, column c holds dim 16*gran + 2c + e
#pragma unroll
      for (int g2 = 0; g2 < NT / 4; ++g2) {
        const int mi = lane >> 3, r = lane & 7;
        const int gran = 2 * g2 + (mi >> 1);
        const int tok = (mi & 1) * 8 + r;
        uint32_t d0, d1, d2, d3;
        mma::ldsm_x4_trans(st + (P + tok) * 128 + ((gran ^ (tok & 7)) * 16), d0, d1, d2, d3);
        uint32_t lo0, hi0, lo1, hi1, lo2, hi2, lo3, hi3;
        mma::e4m3x4_to_f16x2x2(__byte_perm(d0, 0u, 0x3120), lo0, hi0);
        mma::e4m3x4_to_f16x2x2(__byte_perm(d1, 0u, 0x3120), lo1, hi1);
        mma::e4m3x4_to_f16x2x2(__byte_perm(d2, 0u, 0x3120), lo2, hi2);
        mma::e4m3x4_to_f16x2x2(__byte_perm(d3, 0u, 0x3120), lo3, hi3);
        // matrices 0/1: granule 2*g2, tokens 0..7 / 8..15; 2/3: granule 2*g2+1
        mma::mma16816<false>(o[4 * g2], pa[0], pa[1], pa[2], pa[3], lo0, lo1);
        mma::mma16816<false>(o[4 * g2 + 1], pa[0], pa[1], pa[2], pa[3], hi0, hi1);
        mma::mma16816<false>(o[4 * g2 + 2], pa[0], pa[1], pa[2], pa[3], lo2, lo3);
        mma::mma16816<false>(o[4 * g2 + 3], pa[0], pa[1], pa[2], pa[3], hi2, hi3);
      }
    } else {
#pragma unroll
      for (int n2 = 0; n2 < NT / 2; ++n2) {
        const int mi = lane >> 3, r = lane & 7;
        const int sgi = (n2 * 16) / C::BOX_X;
        const int gran = ((n2 * 16) % C::BOX_X) / 8 + (mi >> 1);
        const int tok = (mi & 1) * 8 + r;
        uint32_t b0, b1, b2, b3;
        mma::ldsm_x4_trans(st + sgi * C::BOX_BYTES + (P + tok) * 128 + ((gran ^ (tok & 7)) * 16),
                           b0, b1, b2, b3);
        // b0/b1: dims 16*n2 + 0..7, tokens 0..7 / 8..15; b2/b3: dims + 8..15
        mma::mma16816<kBf16>(o[2 * n2], pa[0], pa[1], pa[2], pa[3], b0, b1);
        mma::mma16816<kBf16>(o[2 * n2 + 1], pa[0], pa[1], pa[2], pa[3], b2, b3);
      }
    }
    dev::release_stage(dev::smem_addr(&empty[stage]), lane);
  }

  // ---- partial state of this chunk, per row: o / d and log2-sum-exp
  const int out_item = sb.y;
  const int rows[2] = {r_lo, r_hi};
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    if (rows[rr] >= row_count) continue;
    const float inv = d_r[rr] > 0.f ? pp.v_scale / d_r[rr] : 0.f;
    float* dst = pp.part_o + ((size_t)out_item * kPrefixRows + rows[rr]) * D;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      if constexpr (kFp8) {
        // n-tile n = 2*gran + e, column c: dim 16*gran + 2c + e
        const int base = 16 * (n >> 1) + (n & 1);
        dst[base + 2 * (2 * t)] = o[n][2 * rr] * inv;
        dst[base + 2 * (2 * t + 1)] = o[n][2 * rr + 1] * inv;
      } else {
        const float2 v = make_float2(o[n][2 * rr] * inv, o[n][2 * rr + 1] * inv);
        *reinterpret_cast<float2*>(dst + n * 8 + 2 * t) = v;
      }
    }
    if (t == 0)
      pp.part_lse[(size_t)out_item * kPrefixRows + rows[rr]] =
          d_r[rr] > 0.f ? m_r[rr] + dev::fast_log2(d_r[rr]) : -INFINITY;
  }
}

}  // namespace fadecode

#include "cascade_tc.cuh"

namespace fadecode {

// One warp per (request, qo head): fold the prefix chunks' states and the
// suffix state with the merge rule.  Lane k holds chunk k's log2-sum-exp
// (32 chunks at a time) and lane l the dims [V*l, V*l + V) of the output
// (V = D / 32); the chunk loop keeps several loads of partial outputs in
// flight.
template <typename QT, int D>
__global__ void __launch_bounds__(256) fa_cascade_combine_kernel(const CombineParams c) {
  static_assert(D == 128 || D == 64, "four or two dims per lane");
  constexpr int V = D / 32;
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (int64_t)c.batch * c.num_qo_heads) return;
  const int b = (int)(wid / c.num_qo_heads), h = (int)(wid % c.num_qo_heads);
  const int kvh = h / c.group, rho = b * c.group + h % c.group;
  const int rb = rho / kPrefixRows, row = rho % kPrefixRows;
  const int item0 = (kvh * c.row_blocks + rb) * c.chunks;
  constexpr float kLog2e = 1.4426950408889634f;
  auto chunk_lse = [&](int k) -> float {
    return k < c.chunks ? __ldg(c.part_lse + (size_t)(item0 + k) * kPrefixRows + row) : -INFINITY;
  };
  const float ls = c.suffix_lse[wid] * kLog2e;
  float M = ls;
  for (int k0 = 0; k0 < c.chunks; k0 += 32) M = fmaxf(M, chunk_lse(k0 + lane));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float num[V] = {};
  float den = 0.f, lse2 = -INFINITY;
  const bool bf = std::is_same<QT, __nv_bfloat16>::value;
  if (M != -INFINITY) {
    for (int k0 = 0; k0 < c.chunks; k0 += 32) {
      const float wl = dev::fast_exp2(chunk_lse(k0 + lane) - M);  // 0 past the last chunk
      den += wl;
      const int n = min(32, c.chunks - k0);
      const float* src = c.part_o + ((size_t)(item0 + k0) * kPrefixRows + row) * D + V * lane;
#pragma unroll 4
      for (int i = 0; i < n; ++i) {
        const float w = __shfl_sync(0xffffffffu, wl, i);
        const float* s = src + (size_t)i * kPrefixRows * D;
        if constexpr (V == 4) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(s));
          num[0] = fmaf(x.x, w, num[0]);
          num[1] = fmaf(x.y, w, num[1]);
          num[2] = fmaf(x.z, w, num[2]);
          num[3] = fmaf(x.w, w, num[3]);
        } else {
          const float2 x = __ldg(reinterpret_cast<const float2*>(s));
          num[0] = fmaf(x.x, w, num[0]);
          num[1] = fmaf(x.y, w, num[1]);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    const float ws = dev::fast_exp2(ls - M);
    den += ws;
    const QT* sv = static_cast<const QT*>(c.suffix_o) + wid * D + V * lane;
#pragma unroll
    for (int v = 0; v < V; v += 2) {
      const float2 s01 = mma::unpack2(*reinterpret_cast<const uint32_t*>(sv + v), bf);
      num[v] = fmaf(s01.x, ws, num[v]);
      num[v + 1] = fmaf(s01.y, ws, num[v + 1]);
    }
    lse2 = M + dev::fast_log2(den);
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  QT* ov = static_cast<QT*>(c.o) + wid * D + V * lane;
#pragma unroll
  for (int v = 0; v < V; v += 2)
    *reinterpret_cast<uint32_t*>(ov + v) = mma::pack2(num[v] * inv, num[v + 1] * inv, bf);
  if (lane == 0 && c.lse) c.lse[wid] = lse2 * 0.693147180559945309f;
}

}  // namespace fadecode

// ------------------------------------------------------------------ host side

using fadecode::DecodeParams;

namespace {

constexpr size_t kCAlign = 256;
size_t calign(size_t x) { return (x + kCAlign - 1) / kCAlign * kCAlign; }

struct CascadeKernels {
  const void* prefix = nullptr;
  const void* combine = nullptr;
  int threads = 0, smem = 0;
  bool tcgen05 = false;  // prefix on the tcgen05 tensor cores (K and V boxes apart)
};

// FADECODE_CASCADE=mma keeps the prefix pass on the warp-level mma.sync
// kernel (for comparisons); by default it runs on tcgen05.
bool cascade_tcgen05() {
  const char* v = std::getenv("FADECODE_CASCADE");
  return !(v && std::strcmp(v, "mma") == 0);
}

// The prefix pass on tcgen05 for 16-bit KV at head_dim 128 (unless
// FADECODE_CASCADE=mma), on the mma.sync kernel otherwise (head_dim 64,
// E4M3 KV).
template <typename QT, typename KVT, int D>
CascadeKernels cascade_kernels() {
  CascadeKernels k;
  k.combine = reinterpret_cast<const void*>(&fadecode::fa_cascade_combine_kernel<QT, D>);
  if constexpr (std::is_same<QT, KVT>::value && D == 128) {
    if (cascade_tcgen05()) {
      k.prefix = reinterpret_cast<const void*>(&fadecode::fa_prefix_tc_kernel<QT>);
      k.threads = fadecode::tc::kThreads;
      k.smem = fadecode::tc::kSmem + 1024;
      k.tcgen05 = true;
      return k;
    }
  }
  using C = fadecode::PrefixCfg<KVT, D, 8>;
  k.prefix = reinterpret_cast<const void*>(&fadecode::fa_prefix_kernel<QT, KVT, D, 8>);
  k.threads = C::THREADS;
  k.smem = C::SMEM + 1024;
  return k;
}

// The kernels of a (q, kv, head_dim) combination; false if not built.
bool find_cascade_kernels(fa_dtype q, fa_dtype kv, int D, CascadeKernels* k) {
  const bool e4m3 = kv == FA_DTYPE_E4M3;
  if (q == FA_DTYPE_BF16 && kv == FA_DTYPE_BF16) {
    *k = D == 128 ? cascade_kernels<__nv_bfloat16, __nv_bfloat16, 128>()
                  : cascade_kernels<__nv_bfloat16, __nv_bfloat16, 64>();
  } else if (q == FA_DTYPE_F16 && kv == FA_DTYPE_F16) {
    *k = D == 128 ? cascade_kernels<__half, __half, 128>() : cascade_kernels<__half, __half, 64>();
  } else if (e4m3 && D == 128 && q == FA_DTYPE_BF16) {
    *k = cascade_kernels<__nv_bfloat16, __nv_fp8_e4m3, 128>();
  } else if (e4m3 && D == 128 && q == FA_DTYPE_F16) {
    *k = cascade_kernels<__half, __nv_fp8_e4m3, 128>();
  } else {
    return false;
  }
  return true;
}

// kv_rows = 2: one box brings a page's K and V rows together (mma.sync
// kernel); 1: K and V in separate boxes (tcgen05 kernel, whose operands are
// [tokens][dims] blocks of K or of V).
int encode_prefix_map(CUtensorMap* map, fa_dtype dt, const void* paged_kv, int64_t num_pages,
                      int D, int Hkv, int P, int kv_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return FA_ERR_CUDA;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  const size_t es = dt == FA_DTYPE_E4M3 ? 1 : 2;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)P,
                        (cuuint64_t)(2 * num_pages)};
  cuuint64_t strides[3] = {(cuuint64_t)(D * es), (cuuint64_t)(Hkv * D * es),
                           (cuuint64_t)(P * Hkv * D * es)};
  // one box row is 128 bytes of a K or V row (the 128-byte swizzle span)
  cuuint32_t box[4] = {(cuuint32_t)(128 / es), 1u, (cuuint32_t)P, (cuuint32_t)kv_rows};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUtensorMapDataType type = dt == FA_DTYPE_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : dt == FA_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUresult r = fn(map, type, 4, const_cast<void*>(paged_kv), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// Most prefix work items a plan makes (its partial states are sized by it):
// at least one chunk per (kv head, row block), else up to 4 per SM.
int64_t prefix_items_cap(int num_kv_heads, int64_t row_blocks, int sms) {
  return std::max<int64_t>((int64_t)num_kv_heads * row_blocks, 4 * (int64_t)sms);
}

struct CascadeLayout {
  size_t off_suffix_ws, suffix_ws_bytes, off_err, off_items, off_cta, meta_bytes, off_part_o,
      off_part_lse, off_so, off_slse, total;
};

CascadeLayout cascade_layout(size_t suffix_ws, int64_t items, int batch, int Hq, int D) {
  CascadeLayout L;
  L.off_suffix_ws = 0;
  L.suffix_ws_bytes = calign(suffix_ws);
  L.off_err = L.suffix_ws_bytes;
  L.off_items = calign(L.off_err + sizeof(int));
  L.off_cta = calign(L.off_items + 32 * (size_t)items);
  L.meta_bytes = calign(L.off_cta + sizeof(int32_t) * (size_t)(items + 1)) - L.off_err;
  L.off_part_o = L.off_err + L.meta_bytes;
  L.off_part_lse = calign(L.off_part_o + sizeof(float) * (size_t)items * fadecode::kPrefixRows * D);
  L.off_so = calign(L.off_part_lse + sizeof(float) * (size_t)items * fadecode::kPrefixRows);
  L.off_slse = calign(L.off_so + 2 * (size_t)batch * Hq * D);
  L.total = calign(L.off_slse + sizeof(float) * (size_t)batch * Hq);
  return L;
}

}  // namespace

struct fa_cascade_plan_s {
  fa_decode_plan_t suffix = nullptr;
  int batch = 0, hq = 0, hkv = 0, d = 0, group = 0, row_blocks = 0, chunks = 0, items = 0;
  int prefix_pages = 0;
  int grid = 0;  // prefix CTAs: one per item, or per item pair on tcgen05
  fa_dtype dtype = FA_DTYPE_BF16;     // q
  fa_dtype kv_dtype = FA_DTYPE_BF16;
  const int32_t* prefix_indices = nullptr;
  uint8_t* ws = nullptr;
  CascadeLayout L{};
  CascadeKernels k;
  CUtensorMap map;
  const void* map_base = nullptr;
  int64_t map_pages = -1;
  cudaEvent_t ev_before = nullptr, ev_after = nullptr;  // around the prefix kernel
  // The prefix kernel runs on a side stream, forked before and joined after
  // the suffix decode, so that its CTAs take each SM as the decode's CTAs
  // leave it (null: both on the caller's stream).  The stream is the
  // device's (shared by all plans, made once); the events are the plan's.
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  int device = 0;
  ~fa_cascade_plan_s();
};

namespace {
// FADECODE_CASCADE_OVERLAP=0 keeps the two passes in order on one stream.
bool cascade_overlap() {
  const char* v = std::getenv("FADECODE_CASCADE_OVERLAP");
  return !(v && v[0] == '0');
}

// Shared-memory attribute and occupancy of a prefix kernel, set and queried
// once per kernel and device.
int prefix_occupancy(const CascadeKernels& k, int dev) {
  struct Entry {
    const void* func;
    int device, occ;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : cache)
    if (e.func == k.prefix && e.device == dev) return e.occ;
  int occ = 0;
  if (cudaFuncSetAttribute(k.prefix, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k.prefix, k.threads, k.smem) !=
          cudaSuccess)
    return 0;
  cache.push_back(Entry{k.prefix, dev, occ});
  return occ;
}

// Fork / join events of cascade plans: a free list per device, so that
// planning every step creates none once warm.
constexpr int kMaxEventDevices = 64;
std::mutex g_event_mu;
std::vector<cudaEvent_t> g_free_events[kMaxEventDevices];

bool take_event(int dev, cudaEvent_t* ev) {
  if (dev < 0 || dev >= kMaxEventDevices) return false;
  {
    std::lock_guard<std::mutex> lock(g_event_mu);
    if (!g_free_events[dev].empty()) {
      *ev = g_free_events[dev].back();
      g_free_events[dev].pop_back();
      return true;
    }
  }
  return cudaEventCreateWithFlags(ev, cudaEventDisableTiming) == cudaSuccess;
}

void give_event(int dev, cudaEvent_t ev) {
  if (!ev) return;
  if (dev < 0 || dev >= kMaxEventDevices) {
    cudaEventDestroy(ev);
    return;
  }
  std::lock_guard<std::mutex> lock(g_event_mu);
  g_free_events[dev].push_back(ev);
}

// One non-blocking stream per device for the prefix pass, created on first
// use and kept for the life of the process.
cudaStream_t device_side_stream(int dev) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static cudaStream_t streams[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!streams[dev] && cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) !=
                           cudaSuccess)
    streams[dev] = nullptr;
  return streams[dev];
}
}  // namespace

extern "C" {

size_t fa_cascade_workspace_size(int batch, int num_qo_heads, int num_kv_heads, int head_dim) {
  const size_t sw = fa_decode_workspace_size(batch, num_qo_heads, num_kv_heads, head_dim);
  if (sw == 0) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  const int G = num_qo_heads / num_kv_heads;
  const int64_t rows = (int64_t)batch * G;
  const int64_t rb = (rows + fadecode::kPrefixRows - 1) / fadecode::kPrefixRows;
  return cascade_layout(sw, prefix_items_cap(num_kv_heads, rb, sms), batch, num_qo_heads,
                        head_dim).total;
}

int fa_cascade_plan(const int32_t* prefix_indices_dev, int num_prefix_pages,
                    const int32_t* indptr_host, const int32_t* indices_dev,
                    const int32_t* last_page_len_host, int batch, int num_qo_heads,
                    int num_kv_heads, int head_dim, int page_size, fa_dtype q_dtype,
                    fa_dtype kv_dtype, void* workspace_dev, size_t workspace_bytes,
                    void* cuda_stream, fa_cascade_plan_t* out_plan) {
  if (!out_plan) return FA_ERR_INVALID_ARG;
  *out_plan = nullptr;
  if (!prefix_indices_dev || num_prefix_pages < 1 || !indptr_host || batch < 1 ||
      num_qo_heads <= 0 || num_kv_heads <= 0 || num_qo_heads % num_kv_heads || !workspace_dev ||
      reinterpret_cast<uintptr_t>(workspace_dev) % kCAlign)
    return FA_ERR_INVALID_ARG;
  CascadeKernels k;
  if (page_size != fadecode::kPageSize || (head_dim != 128 && head_dim != 64) ||
      !find_cascade_kernels(q_dtype, kv_dtype, head_dim, &k))
    return FA_ERR_UNSUPPORTED;
  const size_t sw = fa_decode_workspace_size(batch, num_qo_heads, num_kv_heads, head_dim);
  if (sw == 0) return FA_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  const int occ = prefix_occupancy(k, dev);
  if (occ < 1) return FA_ERR_CUDA;

  fa_cascade_plan_s* plan = new (std::nothrow) fa_cascade_plan_s();
  if (!plan) return FA_ERR_INVALID_ARG;
  plan->device = dev;
  if (cascade_overlap() &&
      (!(plan->side = device_side_stream(dev)) || !take_event(dev, &plan->ev_fork) ||
       !take_event(dev, &plan->ev_join))) {
    delete plan;
    return FA_ERR_CUDA;
  }
  plan->batch = batch;
  plan->hq = num_qo_heads;
  plan->hkv = num_kv_heads;
  plan->d = head_dim;
  plan->group = num_qo_heads / num_kv_heads;
  plan->dtype = q_dtype;
  plan->kv_dtype = kv_dtype;
  plan->prefix_indices = prefix_indices_dev;
  plan->ws = static_cast<uint8_t*>(workspace_dev);
  plan->k = k;
  // prefix work: (kv head, row block, page chunk), about one wave of CTAs
  const int64_t rows = (int64_t)batch * plan->group;
  plan->row_blocks = (int)((rows + fadecode::kPrefixRows - 1) / fadecode::kPrefixRows);
  // the tcgen05 kernel takes two row blocks of a kv head per CTA
  const int64_t base = (int64_t)num_kv_heads *
                       (k.tcgen05 ? (plan->row_blocks + 1) / 2 : plan->row_blocks);
  // chunk count with the fewest waves x pages per chunk (at least 4 pages a
  // chunk), so that every SM gets work and the last wave is not a straggler
  const int64_t slots = (int64_t)sms * occ;
  int chunks = 1;
  int64_t best = INT64_MAX;
  const int64_t cap = prefix_items_cap(num_kv_heads, plan->row_blocks, sms);
  for (int c = 1; c <= std::max(1, num_prefix_pages / 4); ++c) {
    if (c > 1 && (int64_t)num_kv_heads * plan->row_blocks * c > cap) break;
    const int64_t waves = (base * c + slots - 1) / slots;
    const int64_t cost = waves * ((num_prefix_pages + c - 1) / c);
    if (cost < best) {
      best = cost;
      chunks = c;
    }
    if (base * c > 8 * slots) break;
  }
  plan->chunks = chunks;
  plan->prefix_pages = num_prefix_pages;
  plan->items = (int)((int64_t)num_kv_heads * plan->row_blocks * chunks);
  plan->grid = (int)(base * chunks);
  plan->L = cascade_layout(sw, plan->items, batch, num_qo_heads, head_dim);
  if (plan->L.total > workspace_bytes) {
    delete plan;
    return FA_ERR_WORKSPACE_TOO_SMALL;
  }
  // suffix plan in the first part of the workspace
  int rc = fa_decode_plan(indptr_host, indices_dev, last_page_len_host, batch, num_qo_heads,
                          num_kv_heads, head_dim, page_size, q_dtype, kv_dtype,
                          plan->ws + plan->L.off_suffix_ws, plan->L.suffix_ws_bytes, cuda_stream,
                          &plan->suffix);
  if (rc != FA_OK) {
    delete plan;
    return rc;
  }
  // The tcgen05 kernel derives its work from its block index: only the
  // error word is reset, in stream order, with no host image to build.
  if (k.tcgen05) {
    if (cudaMemsetAsync(plan->ws + plan->L.off_err, 0, sizeof(int),
                        static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) {
      fa_decode_plan_destroy(plan->suffix);
      delete plan;
      return FA_ERR_CUDA;
    }
    *out_plan = plan;
    return FA_OK;
  }
  // prefix work items in the decode segment format the producer reads:
  // {row_begin, kv_head, page_begin, page_end, row_count, item, 0, 0}
  std::vector<uint8_t> meta(plan->L.meta_bytes, 0);
  int32_t* items = reinterpret_cast<int32_t*>(meta.data() + (plan->L.off_items - plan->L.off_err));
  int32_t* cta = reinterpret_cast<int32_t*>(meta.data() + (plan->L.off_cta - plan->L.off_err));
  for (int h = 0; h < num_kv_heads; ++h)
    for (int rb = 0; rb < plan->row_blocks; ++rb)
      for (int c = 0; c < chunks; ++c) {
        const int it = (h * plan->row_blocks + rb) * chunks + c;
        const int pb = (int)((int64_t)num_prefix_pages * c / chunks);
        const int pe = (int)((int64_t)num_prefix_pages * (c + 1) / chunks);
        const int r0 = rb * fadecode::kPrefixRows;
        const int nrows = (int)std::min<int64_t>(fadecode::kPrefixRows, rows - r0);
        int32_t* s = items + 8 * it;
        s[0] = r0; s[1] = h; s[2] = pb; s[3] = pe; s[4] = nrows; s[5] = it; s[6] = 0; s[7] = 0;
      }
  for (int i = 0; i <= plan->items; ++i) cta[i] = i;
  if (fadecode::upload_async(plan->ws + plan->L.off_err, meta.data(), meta.size(),
                             static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) {
    fa_decode_plan_destroy(plan->suffix);
    delete plan;
    return FA_ERR_CUDA;
  }
  *out_plan = plan;
  return FA_OK;
}

int fa_cascade_run(fa_cascade_plan_t plan, const void* q, const void* paged_kv,
                   int64_t num_pages, float sm_scale, void* o, float* lse, void* cuda_stream) {
  return fa_cascade_run_scaled(plan, q, paged_kv, num_pages, sm_scale, 1.f, 1.f, o, lse,
                               cuda_stream);
}

int fa_cascade_run_scaled(fa_cascade_plan_t plan, const void* q, const void* paged_kv,
                          int64_t num_pages, float sm_scale, float k_scale, float v_scale,
                          void* o, float* lse, void* cuda_stream) {
  if (!plan || !q || !paged_kv || !o || num_pages <= 0) return FA_ERR_INVALID_ARG;
  // per-tensor scales belong to an E4M3 cache; a 16-bit one is used as stored
  if (plan->kv_dtype != FA_DTYPE_E4M3 && (k_scale != 1.f || v_scale != 1.f))
    return FA_ERR_INVALID_ARG;
  if (!(k_scale > 0.f) || !(v_scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(paged_kv) % 16 || reinterpret_cast<uintptr_t>(q) % 16)
    return FA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const int D = plan->d;
  if (!(sm_scale > 0.f)) sm_scale = 1.0f / std::sqrt((float)D);
  uint8_t* ws = plan->ws;
  void* so = ws + plan->L.off_so;
  float* slse = reinterpret_cast<float*>(ws + plan->L.off_slse);
  const bool timed = plan->ev_before && plan->ev_after;
  // a timed run keeps the prefix kernel alone on the GPU
  const bool fork = plan->side && !timed;
  cudaStream_t pst = fork ? plan->side : st;
  if (fork && (cudaEventRecord(plan->ev_fork, st) != cudaSuccess ||
               cudaStreamWaitEvent(plan->side, plan->ev_fork, 0) != cudaSuccess))
    return FA_ERR_CUDA;
  // 1. each request's own pages
  int rc = fa_decode_run(plan->suffix, q, paged_kv, num_pages, sm_scale, k_scale, v_scale, so,
                         slse, cuda_stream);
  if (rc != FA_OK) return rc;
  // 2. the shared prefix, once per kv head and row block
  if (paged_kv != plan->map_base || num_pages != plan->map_pages) {
    rc = encode_prefix_map(&plan->map, plan->kv_dtype, paged_kv, num_pages, D, plan->hkv,
                           fadecode::kPageSize, plan->k.tcgen05 ? 1 : 2);
    if (rc != FA_OK) return rc;
    plan->map_base = paged_kv;
    plan->map_pages = num_pages;
  }
  DecodeParams prm;
  std::memset(&prm, 0, sizeof prm);
  prm.q = q;
  prm.indices = plan->prefix_indices;
  prm.cta_offsets = reinterpret_cast<const int32_t*>(ws + plan->L.off_cta);
  prm.segments = reinterpret_cast<const int32_t*>(ws + plan->L.off_items);
  prm.err = reinterpret_cast<int*>(ws + plan->L.off_err);
  prm.num_pages = num_pages;
  prm.num_qo_heads = plan->hq;
  prm.num_kv_heads = plan->hkv;
  prm.q_len = 1;
  fadecode::PrefixParams pp;
  pp.q = q;
  pp.part_o = reinterpret_cast<float*>(ws + plan->L.off_part_o);
  pp.part_lse = reinterpret_cast<float*>(ws + plan->L.off_part_lse);
  pp.group = plan->group;
  pp.q_scale = sm_scale * k_scale * 1.4426950408889634f;
  pp.v_scale = v_scale;
  pp.row_blocks = plan->row_blocks;
  pp.pair_blocks = (plan->row_blocks + 1) / 2;
  pp.chunks = plan->chunks;
  pp.rows = plan->batch * plan->group;
  pp.prefix_pages = plan->prefix_pages;
  void* args[3] = {&plan->map, &prm, &pp};
  if (timed && cudaEventRecord(plan->ev_before, st) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaLaunchKernel(plan->k.prefix, dim3(plan->grid), dim3(plan->k.threads), args,
                       (size_t)plan->k.smem, pst) != cudaSuccess)
    return FA_ERR_CUDA;
  if (timed && cudaEventRecord(plan->ev_after, st) != cudaSuccess) return FA_ERR_CUDA;
  if (fork && (cudaEventRecord(plan->ev_join, plan->side) != cudaSuccess ||
               cudaStreamWaitEvent(st, plan->ev_join, 0) != cudaSuccess))
    return FA_ERR_CUDA;
  // 3. fold prefix chunks and suffix
  fadecode::CombineParams c;
  c.part_o = pp.part_o;
  c.part_lse = pp.part_lse;
  c.suffix_o = so;
  c.suffix_lse = slse;
  c.o = o;
  c.lse = lse;
  c.batch = plan->batch;
  c.num_qo_heads = plan->hq;
  c.group = plan->group;
  c.row_blocks = plan->row_blocks;
  c.chunks = plan->chunks;
  void* cargs[1] = {&c};
  const int64_t warps = (int64_t)plan->batch * plan->hq;
  if (cudaLaunchKernel(plan->k.combine, dim3((unsigned)((warps * 32 + 255) / 256)), dim3(256),
                       cargs, 0, st) != cudaSuccess)
    return FA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"

fa_cascade_plan_s::~fa_cascade_plan_s() {
  give_event(device, ev_fork);
  give_event(device, ev_join);
}

extern "C" {

int fa_cascade_plan_destroy(fa_cascade_plan_t plan) {
  if (plan) {
    fa_decode_plan_destroy(plan->suffix);
    delete plan;
  }
  return FA_OK;
}

int fa_cascade_set_timing_events(fa_cascade_plan_t plan, void* ev_before, void* ev_after) {
  if (!plan) return FA_ERR_INVALID_ARG;
  plan->ev_before = static_cast<cudaEvent_t>(ev_before);
  plan->ev_after = static_cast<cudaEvent_t>(ev_after);
  return FA_OK;
}

int fa_cascade_check(fa_cascade_plan_t plan, void* cuda_stream, int* flags) {
  if (!plan || !flags) return FA_ERR_INVALID_ARG;
  int f1 = 0;
  const int rc = fa_decode_check(plan->suffix, cuda_stream, &f1);
  if (rc != FA_OK && rc != FA_ERR_DEVICE_CHECK) return rc;
  int word = 0;
  int* dword = reinterpret_cast<int*>(plan->ws + plan->L.off_err);
  if (cudaMemcpy(&word, dword, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(dword, 0, sizeof word) != cudaSuccess)
    return FA_ERR_CUDA;
  *flags = f1 | word;
  return *flags ? FA_ERR_DEVICE_CHECK : FA_OK;
}

}  // extern "C"
