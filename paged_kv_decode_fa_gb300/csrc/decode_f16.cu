// Compiled instances of the split-KV decode kernel for q = __half, kv = __half
// (one translation unit per dtype pair so the build runs in parallel).
#include "decode_mma.cuh"

namespace fadecode {
bool find_kernel_f16(int head_dim, int group, bool allow_mma, DecodeKernel* k) {
  return find_kernel_for<__half, __half>(head_dim, group, allow_mma, k);
}
bool find_unified_max_kernel_f16(int head_dim, int group, DecodeKernel* k) {
  return find_unified_max_kernel_for<__half, __half>(head_dim, group, k);
}
}  // namespace fadecode
