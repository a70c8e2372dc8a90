// fa_decode_static: plan + run of one decode batch with the work list and the
// partial softmax states kept in a fixed array that the library itself owns,
// so that the call allocates nothing: no device memory, no page-locked host
// memory, no events, no heap objects.
//
// Who needs this: code that is handed only input and output pointers and is
// not allowed to allocate - a custom operator inside a host framework that
// owns all device memory through its own pool, an out-of-memory or
// allocator callback, or a latency-critical loop where cudaMalloc (which can
// synchronise the whole device) is not acceptable.  Everyone else should use
// fa_decode_plan / fa_decode_run with a workspace of their own.
//
// The array below lives in every GPU that loads this library, for the life
// of the process.  In host code its name is only a host-side stand-in, not a
// device address, so the address is looked up with cudaGetSymbolAddress,
// once per device, while that device is current.
#include <cuda_runtime.h>

#include <mutex>

#include "fa_decode.h"
#include "kernels.h"

static_assert(FA_STATIC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

// The work list, the device-check word and the fp32 partial states of a call.
static __device__ __align__(256) unsigned char g_static_scratch[FA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (looked up on the
// first call for that device).
int static_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return FA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_decode_static(const int32_t* indptr_host, const int32_t* indices_dev,
                                const int32_t* last_page_len_host, int batch, int num_qo_heads,
                                int num_kv_heads, int head_dim, int page_size, fa_dtype q_dtype,
                                fa_dtype kv_dtype, const void* q, const void* paged_kv,
                                int64_t num_pages, float sm_scale, float k_scale, float v_scale,
                                void* o, float* lse, void* cuda_stream) {
  void* scratch = nullptr;
  int rc = static_scratch_address(&scratch);
  if (rc != FA_OK) return rc;
  // Plans into fixed host arrays, copies the work list (and a zeroed
  // device-check word) into the scratch on the stream and launches; a batch
  // whose plan does not fit is refused with FA_ERR_WORKSPACE_TOO_SMALL
  // before anything is enqueued.
  return fadecode::static_decode(scratch, FA_STATIC_SCRATCH_BYTES, indptr_host, indices_dev,
                                 last_page_len_host, batch, num_qo_heads, num_kv_heads,
                                 head_dim, page_size, q_dtype, kv_dtype, q, paged_kv, num_pages,
                                 sm_scale, k_scale, v_scale, o, lse, cuda_stream);
}

extern "C" int fa_decode_static_check(void* cuda_stream, int* flags) {
  if (!flags) return FA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  int rc = static_scratch_address(&scratch);
  if (rc != FA_OK) return rc;
  // the device-check word is the first int of the scratch (the work list's
  // layout starts with it)
  int word = 0;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (cudaStreamSynchronize(st) != cudaSuccess ||
      cudaMemcpy(&word, scratch, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemsetAsync(scratch, 0, sizeof word, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return FA_ERR_CUDA;
  *flags = word;
  return word ? FA_ERR_DEVICE_CHECK : FA_OK;
}
