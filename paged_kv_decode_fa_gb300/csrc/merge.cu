// fa_merge_states: elementwise merge of two sets of partial attention states
// with the rule of section "FlashDecoding - the split-KV trick" (page
// "FlashDecoding + FlashInfer - the decode-time attention story"):
//   m = max(m_a, m_b), d = d_a e^(m_a-m) + d_b e^(m_b-m), o likewise,
// applied to normalised states (m = lse, d = 1) and normalised again.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace fadecode {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.693147180559945309f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }

// One warp per state.  Every lane reads both lse values before lane 0 writes
// the merged one, and each output element is written by the lane that read
// its inputs, so o_out/lse_out may alias o_a/lse_a.
template <typename T>
__global__ void __launch_bounds__(256)
    merge_states_kernel(const T* o_a, const float* lse_a, const T* o_b,
                        const float* lse_b, T* o_out, float* lse_out, int64_t n, int D) {
  const int64_t s = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (s >= n) return;
  const float la = lse_a[s], lb = lse_b[s];
  const float m = fmaxf(la, lb);
  const bool empty = (m == -INFINITY);
  float wa = 0.f, wb = 0.f, lse = -INFINITY;
  if (!empty) {
    wa = ex2((la - m) * kLog2e);
    wb = ex2((lb - m) * kLog2e);
    lse = m + lg2(wa + wb) * kLn2;
  }
  const float inv = empty ? 0.f : 1.f / (wa + wb);
  __syncwarp();
  for (int d = lane; d < D; d += 32) {
    const int64_t i = s * D + d;
    const float x = empty ? 0.f : (to_f(o_a[i]) * wa + to_f(o_b[i]) * wb) * inv;
    o_out[i] = from_f<T>(x);
  }
  __syncwarp();
  if (lane == 0) lse_out[s] = lse;
}

template <typename T>
int launch(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o_out,
           float* lse_out, int64_t n, int D, cudaStream_t st) {
  const int threads = 256;
  const int64_t blocks = (n * 32 + threads - 1) / threads;
  if (blocks > 0x7fffffff) return FA_ERR_UNSUPPORTED;
  merge_states_kernel<T><<<(unsigned)blocks, threads, 0, st>>>(
      static_cast<const T*>(o_a), lse_a, static_cast<const T*>(o_b), lse_b,
      static_cast<T*>(o_out), lse_out, n, D);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

int launch_merge_states(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b,
                        void* o_out, float* lse_out, int64_t n_states, int head_dim,
                        fa_dtype dtype, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (dtype) {
    case FA_DTYPE_F32:
      return launch<float>(o_a, lse_a, o_b, lse_b, o_out, lse_out, n_states, head_dim, st);
    case FA_DTYPE_BF16:
      return launch<__nv_bfloat16>(o_a, lse_a, o_b, lse_b, o_out, lse_out, n_states, head_dim, st);
    case FA_DTYPE_F16:
      return launch<__half>(o_a, lse_a, o_b, lse_b, o_out, lse_out, n_states, head_dim, st);
    default:
      return FA_ERR_UNSUPPORTED;
  }
}

}  // namespace fadecode
