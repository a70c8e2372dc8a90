// Asynchronous upload of small host buffers (plan metadata).
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace fadecode {

// Copy `bytes` from host memory `src` to device memory `dst` on `stream`
// without waiting for the stream: a copy straight from pageable memory would
// first wait for the work already queued on the stream to finish, which
// serialises planning on the host with the decode kernels on the device.
// The bytes go through one of a few page-locked staging buffers that the
// library owns (reused round-robin, each once its previous copy is done).
// Returns cudaSuccess or the failing call's error.
cudaError_t upload_async(void* dst, const void* src, size_t bytes, cudaStream_t stream);

// Page-locked staging buffers allocated so far (count and bytes) and
// uploads made through the ring, since the library was loaded.
void staging_stats(int64_t* allocations, int64_t* bytes, int64_t* uploads);

}  // namespace fadecode
