// Page-locked staging ring for plan uploads (see staging.h).
#include "staging.h"

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

namespace fadecode {
namespace {

constexpr int kSlots = 8;
constexpr size_t kMinSlotBytes = 64 << 10;

struct Slot {
  void* buf = nullptr;
  size_t cap = 0;
  cudaEvent_t done = nullptr;  // recorded after the slot's last copy
  int device = -1;             // device the event belongs to
  bool pending = false;
};

std::mutex g_mu;
Slot g_slots[kSlots];
int g_next = 0;
std::atomic<int64_t> g_allocs{0}, g_alloc_bytes{0}, g_uploads{0};

}  // namespace

cudaError_t upload_async(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
  if (bytes == 0) return cudaSuccess;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  Slot& s = g_slots[g_next];
  g_next = (g_next + 1) % kSlots;
  if (s.pending) {  // the slot's previous copy must have left the buffer
    if ((e = cudaEventSynchronize(s.done)) != cudaSuccess) return e;
    s.pending = false;
  }
  if (s.done && s.device != device) {
    cudaEventDestroy(s.done);
    s.done = nullptr;
  }
  if (!s.done) {
    if ((e = cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming)) != cudaSuccess) return e;
    s.device = device;
  }
  if (s.cap < bytes) {
    if (s.buf) cudaFreeHost(s.buf);
    s.buf = nullptr;
    s.cap = 0;
    size_t cap = kMinSlotBytes;
    while (cap < bytes) cap *= 2;
    if ((e = cudaMallocHost(&s.buf, cap)) != cudaSuccess) return e;
    s.cap = cap;
    g_allocs.fetch_add(1);
    g_alloc_bytes.fetch_add((int64_t)cap);
  }
  std::memcpy(s.buf, src, bytes);
  if ((e = cudaMemcpyAsync(dst, s.buf, bytes, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
    return e;
  if ((e = cudaEventRecord(s.done, stream)) != cudaSuccess) return e;
  s.pending = true;
  g_uploads.fetch_add(1);
  return cudaSuccess;
}

void staging_stats(int64_t* allocations, int64_t* bytes, int64_t* uploads) {
  *allocations = g_allocs.load();
  *bytes = g_alloc_bytes.load();
  *uploads = g_uploads.load();
}

}  // namespace fadecode
