// Compiled instances of the decode kernel with ragged query rows for requests
// of two or three 8-column tiles (a column split of two or three warps), for
// q = __nv_bfloat16, kv = __nv_fp8_e4m3 (a translation unit of their own so the
// build runs in parallel).
#include "decode_mma.cuh"

namespace fadecode {
bool find_ragged_q_tiles_kernel_bf16_e4m3(int head_dim, int group, int tiles, DecodeKernel* k) {
  return find_ragged_q_tiles_kernel_for<__nv_bfloat16, __nv_fp8_e4m3>(head_dim, group, tiles, k);
}
}  // namespace fadecode
