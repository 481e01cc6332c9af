// The library's cached per-device scratch: the doc-scan word and the
// cost-ranked slot order that forward launches with documents read.
//
// One buffer per device, grown on demand and never shrunk.  Growth frees the
// old buffer and allocates the new one in stream order (cudaFreeAsync /
// cudaMallocAsync on the caller's stream), so a call that fits the current
// buffer allocates nothing.  Calls on one stream are ordered by the stream;
// a call on another stream first waits for an event recorded after the
// previous user's work, so two launches never use the buffer at once.  The
// per-device lock is held only while a call enqueues its work.
#include <cuda_runtime_api.h>

#include <algorithm>
#include <mutex>

#include "internal.h"

namespace cpring {
namespace {

struct DeviceScratch {
  std::mutex mu;
  void* ptr = nullptr;
  size_t cap = 0;
  cudaEvent_t released = nullptr;  // recorded after the last lease's work
  cudaStream_t last_stream = nullptr;
  bool used = false;
};

constexpr int kMaxDevices = 64;
DeviceScratch g_scratch[kMaxDevices];

}  // namespace

ScratchLease::ScratchLease(size_t bytes, cudaStream_t stream) : stream_(stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
  DeviceScratch& s = g_scratch[dev];
  s.mu.lock();
  dev_ = dev;
  if (!s.released && cudaEventCreateWithFlags(&s.released, cudaEventDisableTiming) != cudaSuccess) {
    s.released = nullptr;
    return;
  }
  if (s.used && s.last_stream != stream &&
      cudaStreamWaitEvent(stream, s.released, 0) != cudaSuccess)
    return;
  if (s.cap < bytes) {
    const size_t want = std::max<size_t>({bytes, 4096, 2 * s.cap});
    const size_t rounded = (want + 255) / 256 * 256;
    if (s.ptr) cudaFreeAsync(s.ptr, stream);
    s.ptr = nullptr;
    s.cap = 0;
    if (cudaMallocAsync(&s.ptr, rounded, stream) != cudaSuccess) {
      s.ptr = nullptr;
      return;
    }
    s.cap = rounded;
  }
  ptr_ = s.ptr;
  ok_ = true;
}

ScratchLease::~ScratchLease() {
  if (dev_ < 0) return;
  DeviceScratch& s = g_scratch[dev_];
  if (s.released && cudaEventRecord(s.released, stream_) == cudaSuccess) {
    s.last_stream = stream_;
    s.used = true;
  }
  s.mu.unlock();
}

}  // namespace cpring
