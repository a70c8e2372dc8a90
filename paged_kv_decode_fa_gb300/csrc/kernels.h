// Host-side view of the CUDA kernels: parameter blocks and the registry that
// maps (q dtype, kv dtype, head_dim, group size) to a compiled instance.
#pragma once
#include <cstddef>
#include <cstdint>

#include "fa_decode.h"

namespace fadecode {

constexpr int kPageSize = 16;

// Kernel parameters of the split-KV decode kernel (the TMA descriptor of the
// KV cache travels beside it as a __grid_constant__ argument).
struct DecodeParams {
  const void* q;               // [B, Hq, D] q dtype
  void* o;                     // [B, Hq, D] q dtype
  float* lse;                  // [B, Hq] or nullptr
  const int32_t* indices;      // page ids
  const int32_t* cta_offsets;  // [num_ctas + 1]
  const int32_t* segments;     // [num_segments * 8]
  float* part_o;               // [slots, G, D] fp32, normalised partial outputs
  float* part_lse;             // [slots, G] fp32, log2-domain log-sum-exp
  int* err;                    // device-check word
  const int32_t* merge;        // [n_merge * 4] {request, kv_head, first_slot, num_slots}
  int* merge_count;            // [n_merge] arrivals per split unit, zero between runs
  int fused_merge;             // 1: the last CTA of a split unit merges it
  const float* k_scales;       // [num_pages, Hkv, page_size] per-token scales, or nullptr
  const float* v_scales;       // same for V
  const float* head_k_scales;  // [Hkv] one K scale per kv head (times q_scale), or nullptr
  const float* head_v_scales;  // [Hkv] one V scale per kv head (times v_scale), or nullptr
  int64_t num_pages;
  int num_qo_heads;
  int num_kv_heads;
  int q_len;                   // query tokens per request (1 for plain decode); with
                               // qo_indptr, the most a request may have
  const int32_t* qo_indptr;    // [B + 1] query rows per request (ragged q), or nullptr
  int q_row_bytes;             // head_dim * q element size (0: no q prefetch)
  const void* kv;              // paged KV base (for L2 prefetches), or nullptr
  int kv_row_bytes;            // head_dim * KV element size
  float q_scale;  // sm_scale * k_scale * log2(e), folded into q
  float v_scale;
  float max_bound;    // unified-max kernels: static reference of the logits, log2 units
  int* um_fallbacks;  // unified-max kernels: count of (segment, warp) re-centrings, or nullptr
  // Pool of the plan: segments pool_begin .. pool_begin + pool_count - 1,
  // claimed in order through *pool_claim; *pool_done counts finished CTAs
  // and the last one re-arms both (zero between runs).
  int pool_begin;
  int pool_count;
  int* pool_claim;
  int* pool_done;
};

struct MergeParams {
  const int32_t* merge;  // [n_merge * 4]
  const int32_t* qo_indptr;  // [B + 1] for ragged q, else nullptr
  const float* part_o;
  const float* part_lse;
  void* o;
  float* lse;
  int num_qo_heads;
};

// One compiled decode kernel instance and its launch shape.
struct DecodeKernel {
  const void* func = nullptr;      // __global__ (CUtensorMap, DecodeParams)
  const void* merge_func = nullptr;  // __global__ (MergeParams)
  int threads = 0;
  int smem_bytes = 0;
  int stages = 0;
  int stage_bytes = 0;
  int group = 0;
  int head_dim = 0;
  int box_x = 0;              // elements per TMA box row (D, or 128 bytes' worth)
  bool swizzle_128b = false;  // stage rows in TMA 128-byte swizzle order
  bool tensor_cores = false;  // per-page products on mma.sync
  bool token_scales = false;  // reads per-token K/V scales (E4M3 only)
  int q_len = 1;              // query tokens per request the kernel was built for (ragged:
                              // the most a request may have)
  bool unified_max = false;   // softmax against a static bound (no running max)
  bool ragged_q = false;      // query rows per request from qo_indptr
};

// Each returns false when the combination is not compiled.  allow_mma
// selects the tensor-core consumer where it applies (group >= 2, 16-bit or
// E4M3 KV, rows a multiple of 128 bytes); otherwise the CUDA-core one.
bool find_kernel_f32(int head_dim, int group, bool allow_mma, DecodeKernel* k);
bool find_kernel_bf16(int head_dim, int group, bool allow_mma, DecodeKernel* k);
bool find_kernel_f16(int head_dim, int group, bool allow_mma, DecodeKernel* k);
bool find_kernel_bf16_e4m3(int head_dim, int group, bool allow_mma, DecodeKernel* k);
bool find_kernel_f16_e4m3(int head_dim, int group, bool allow_mma, DecodeKernel* k);
// Multi-token decode (q_len query tokens per request, causal among them):
// tensor-core consumer, head_dim 128, group * q_len <= 8.
bool find_multi_token_kernel_bf16(int head_dim, int group, int q_len, DecodeKernel* k);
bool find_multi_token_kernel_bf16_e4m3(int head_dim, int group, int q_len, DecodeKernel* k);
// Ragged query rows: request i has qo_indptr[i+1] - qo_indptr[i] <= max_q
// query tokens (head_dim 128; group x max_q <= 32).
bool find_ragged_q_kernel_bf16(int head_dim, int group, int max_q, DecodeKernel* k);
bool find_ragged_q_kernel_bf16_e4m3(int head_dim, int group, int max_q, DecodeKernel* k);
// The same for requests of `tiles` (2 or 3) 8-column tiles: a column split
// of that many consumer warps, with more CTAs per SM than four warps allow.
bool find_ragged_q_tiles_kernel_bf16(int head_dim, int group, int tiles, DecodeKernel* k);
bool find_ragged_q_tiles_kernel_bf16_e4m3(int head_dim, int group, int tiles, DecodeKernel* k);
// Unified-max softmax (groups 2, 4, 8; bf16 q and KV at head_dim 64 or 128).
bool find_unified_max_kernel_bf16(int head_dim, int group, DecodeKernel* k);
// The same with f16 weights: f16 q and KV, or E4M3 KV (head_dim 128 for E4M3).
bool find_unified_max_kernel_f16(int head_dim, int group, DecodeKernel* k);
bool find_unified_max_kernel_bf16_e4m3(int head_dim, int group, DecodeKernel* k);
bool find_unified_max_kernel_f16_e4m3(int head_dim, int group, DecodeKernel* k);
// E4M3 KV with per-token, per-kv-head scales (tensor-core consumer only).
bool find_token_scale_kernel_bf16_e4m3(int head_dim, int group, DecodeKernel* k);
bool find_token_scale_kernel_f16_e4m3(int head_dim, int group, DecodeKernel* k);

// Plan + run of one batch with the workspace replaced by `scratch` (the
// library's own device array) and no allocation of any kind: the path
// behind fa_decode_static (api.cu).  Returns an fa_status.
int static_decode(void* scratch, size_t scratch_bytes, const int32_t* indptr_host,
                  const int32_t* indices_dev, const int32_t* last_page_len_host, int batch,
                  int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                  fa_dtype q_dtype, fa_dtype kv_dtype, const void* q, const void* paged_kv,
                  int64_t num_pages, float sm_scale, float k_scale, float v_scale, void* o,
                  float* lse, void* cuda_stream);

// fa_merge_states kernels (merge.cu).
int launch_merge_states(const void* o_a, const float* lse_a, const void* o_b,
                        const float* lse_b, void* o_out, float* lse_out,
                        int64_t n_states, int head_dim, fa_dtype dtype,
                        void* stream);

}  // namespace fadecode
