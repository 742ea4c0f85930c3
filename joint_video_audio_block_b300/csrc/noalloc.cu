// h3_qknorm_rope_static: the QK-norm + RoPE step with its scratch in a fixed device array.
//
// h3_qknorm_rope needs a per-row cos/sin table as scratch and takes it from the caller's
// workspace.  Some callers have no way to hand over extra device memory at that point: an
// embedder whose device memory is owned by a pool or allocator it cannot reach from the call
// site, or a latency-critical loop that must not pay for cudaMalloc's implicit device
// synchronisation.  This entry point serves them: the table lives in the file-scope array
// below, which the library's module holds on every device that loads it until the process
// exits.  Nothing here calls cudaMalloc, cudaFree or any allocating routine.
//
// Sharing: every call (on any stream) writes the same array.  Calls whose GPU work overlaps
// race on it; the caller must order them (one stream, or events).  The table is fully
// rewritten for the rows a call uses before it is read, so no part needs to start at zero.
#include <atomic>

#include "../../include/h3.h"
#include "kernels.h"

namespace h3 {

// cos/sin pairs for up to H3_QKROPE_STATIC_MAX_PAIRS (row, frequency) entries: 16 MiB.
static __device__ __align__(256) float2 g_rope_scratch[H3_QKROPE_STATIC_MAX_PAIRS];

// Device address of g_rope_scratch on the current device.  In host code the array's name is
// only a host-side stand-in, so the address is looked up once per device (with that device
// current) and cached; host threads may race on the first lookup and all store the same
// address.  Returns nullptr if the lookup fails.
static float2* rope_scratch_ptr() {
  static std::atomic<float2*> ptr[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  float2* a = ptr[dev].load(std::memory_order_acquire);
  if (!a) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_rope_scratch) != cudaSuccess || !p) return nullptr;
    a = static_cast<float2*>(p);
    ptr[dev].store(a, std::memory_order_release);
  }
  return a;
}

// argument checks shared with h3_qknorm_rope (api.cu)
bool qknorm_rope_args_ok(const h3_dims* d, const void* qkv, const float* pos, const void* q_norm,
                         const void* k_norm, const void* q_out, const void* k_out, const void* vt_out, int ld_vt,
                         int n_rows);

}  // namespace h3

using namespace h3;

extern "C" h3_status h3_qknorm_rope_static(const h3_dims* dims, const void* qkv, const float* pos,
                                           const void* q_norm, const void* k_norm, void* q_out, void* k_out,
                                           void* vt_out, int ld_vt, int n_rows, void* stream) {
  if (!qknorm_rope_args_ok(dims, qkv, pos, q_norm, k_norm, q_out, k_out, vt_out, ld_vt, n_rows)) return H3_EINVAL;
  const long long pairs = static_cast<long long>(n_rows) * (dims->head_dim / 2);
  if (pairs > H3_QKROPE_STATIC_MAX_PAIRS) return H3_EINVAL;  // beyond the fixed scratch array
  if (n_rows == 0) return H3_OK;
  float2* cs = rope_scratch_ptr();
  if (!cs) return H3_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_rope_table(pos, cs, n_rows, dims->head_dim, dims->rope_sections, dims->rope_theta, st);
  if (e == cudaSuccess)
    e = launch_qknorm_rope(static_cast<const bf16*>(qkv), cs, static_cast<const bf16*>(q_norm),
                           static_cast<const bf16*>(k_norm), dims->qk_eps, static_cast<bf16*>(q_out),
                           static_cast<bf16*>(k_out), static_cast<bf16*>(vt_out), ld_vt, n_rows, dims->heads,
                           dims->head_dim, st);
  return e == cudaSuccess ? H3_OK : (e == cudaErrorInvalidValue ? H3_EINVAL : H3_ECUDA);
}
