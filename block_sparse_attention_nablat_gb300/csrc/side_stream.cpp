// The library's own second stream per device.  The mask builder forks work onto
// it from the caller's stream with an event and joins back the same way, so
// the caller sees one ordered sequence on its stream (this also holds inside a
// stream capture: the fork and join become graph edges).
#include <mutex>

#include "internal.h"

namespace nabla {
namespace {

constexpr int kMaxDevices = 64;
SideStream g_side[kMaxDevices];
bool g_side_ready[kMaxDevices];
std::mutex g_side_mutex;  // guards creation and each fork-join sequence

}  // namespace

void side_stream_lock() { g_side_mutex.lock(); }
void side_stream_unlock() { g_side_mutex.unlock(); }

// Call with the lock held.
cudaError_t side_stream(SideStream *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!g_side_ready[dev]) {
    int least = 0, greatest = 0;
    if ((e = cudaDeviceGetStreamPriorityRange(&least, &greatest)) != cudaSuccess) return e;
    SideStream s{};
    if ((e = cudaStreamCreateWithPriority(&s.stream, cudaStreamNonBlocking, greatest)) !=
        cudaSuccess)
      return e;
    if ((e = cudaEventCreateWithFlags(&s.event, cudaEventDisableTiming)) != cudaSuccess) {
      cudaStreamDestroy(s.stream);
      return e;
    }
    g_side[dev] = s;
    g_side_ready[dev] = true;
  }
  *out = g_side[dev];
  return cudaSuccess;
}

}  // namespace nabla
