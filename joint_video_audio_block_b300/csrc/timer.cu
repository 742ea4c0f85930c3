// Launch timer for measurement: brackets the attention launches of the block / trunk calls
// with CUDA events recorded on the launching stream, so a benchmark can time the dominant
// kernel inside a real trunk step instead of in isolation.  Host-side state only; the events
// are the only resources it creates (no device memory).
#include <vector>

#include "../../include/h3.h"
#include "kernels.h"

namespace h3 {

namespace {
struct TimerState {
  std::vector<cudaEvent_t> start, stop;
  int used = 0;
  int device = -1;
};
TimerState g_timer;

void destroy_events() {
  for (cudaEvent_t e : g_timer.start) cudaEventDestroy(e);
  for (cudaEvent_t e : g_timer.stop) cudaEventDestroy(e);
  g_timer.start.clear();
  g_timer.stop.clear();
  g_timer.used = 0;
}
}  // namespace

void timer_mark_begin(cudaStream_t st) {
  if (g_timer.used < static_cast<int>(g_timer.start.size())) cudaEventRecord(g_timer.start[g_timer.used], st);
}

void timer_mark_end(cudaStream_t st) {
  if (g_timer.used < static_cast<int>(g_timer.stop.size())) {
    cudaEventRecord(g_timer.stop[g_timer.used], st);
    ++g_timer.used;
  }
}

}  // namespace h3

using namespace h3;

extern "C" h3_status h3_kernel_timer_start(int capacity) {
  if (capacity < 0 || capacity > (1 << 20)) return H3_EINVAL;
  destroy_events();
  if (capacity == 0) return H3_OK;
  if (cudaGetDevice(&g_timer.device) != cudaSuccess) return H3_ECUDA;
  g_timer.start.reserve(capacity);
  g_timer.stop.reserve(capacity);
  for (int i = 0; i < capacity; ++i) {
    cudaEvent_t a = nullptr, b = nullptr;
    if (cudaEventCreate(&a) != cudaSuccess) {
      destroy_events();
      return H3_ECUDA;
    }
    if (cudaEventCreate(&b) != cudaSuccess) {
      cudaEventDestroy(a);
      destroy_events();
      return H3_ECUDA;
    }
    g_timer.start.push_back(a);
    g_timer.stop.push_back(b);
  }
  return H3_OK;
}

extern "C" h3_status h3_kernel_timer_read(float* ms, int capacity, int* n_recorded) {
  if (!n_recorded || capacity < 0 || (capacity > 0 && !ms)) return H3_EINVAL;
  const int n = g_timer.used;
  *n_recorded = n;
  for (int i = 0; i < n && i < capacity; ++i) {
    if (cudaEventSynchronize(g_timer.stop[i]) != cudaSuccess) return H3_ECUDA;
    if (cudaEventElapsedTime(&ms[i], g_timer.start[i], g_timer.stop[i]) != cudaSuccess) return H3_ECUDA;
  }
  destroy_events();
  return H3_OK;
}
