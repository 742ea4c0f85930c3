// Diagnostic for the library's failure path: a kernel whose pipeline wait can never complete.
//
// Every mbarrier wait in the library's kernels is bounded (mbar_wait): when it runs out it
// records a site code in the device error word and the kernel leaves its loop and tears down
// normally, so the GPU context stays usable and h3_last_device_error reports H3_ETIMEOUT.
// This kernel exercises exactly that path on purpose -- one warp initialises an mbarrier that
// expects one arrival, nothing ever arrives, and the bounded wait gives up after the caller's
// time limit -- so the path can be tested without any fault, trap or hang.
#include "../../include/h3.h"
#include "kernels.h"

namespace h3 {

__global__ void expire_wait_kernel(unsigned long long timeout_ns, unsigned* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // phase 0 never completes: no thread arrives
  const bool ok = mbar_wait(b, 0, err_ctx(err), kErrDiagWait, timeout_ns);
  (void)ok;
  __syncthreads();
}

}  // namespace h3

using namespace h3;

extern "C" h3_status h3_diag_expire_wait(unsigned timeout_us, void* stream) {
  if (timeout_us == 0 || timeout_us > 1000000u) return H3_EINVAL;
  unsigned* err = h3_error_word_ptr();
  if (!err) return H3_ECUDA;
  expire_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<unsigned long long>(timeout_us) * 1000ull, err);
  return cudaGetLastError() == cudaSuccess ? H3_OK : H3_ECUDA;
}
