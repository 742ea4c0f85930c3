// Diagnostic of how fast one issuing thread can feed the tensor pipe (no counterpart on the
// pages; it measures the sm_103a property the attention and GEMM pipelines are designed around).
//
// Each CTA (one per SM: its shared-memory request leaves room for no second one) allocates all
// 512 tensor-memory columns and one thread issues `batches` batches of 16 bf16 MMAs of
// 128 x 128 x 16: 8 with both operands in shared memory into columns 0..127, then 8 with the A
// operand in tensor memory (columns 384..447) into columns 128..255 -- the attention kernel's
// S = Q K^T and O += P V shapes.  The operands are whatever the memories hold and nothing is
// read back; only the cycle count from the first issue to the completion of the last MMA is kept.
//   mode 0  batches back to back
//   mode 1  between the 8 shared-memory-operand MMAs and the 8 tensor-memory-operand MMAs of
//           each batch the thread polls an mbarrier whose phase is already complete and uses
//           the answer at once (what a pipeline's wait for a ready stage costs there)
//   mode 2  the same poll at the same point as a non-blocking test whose answer is read only
//           after the tensor-memory-operand MMAs
//   mode 3  the blocking poll of mode 1 placed after the tensor-memory-operand MMAs instead
//   mode 4  mode 0 while eight more warps (two on every SM sub-partition, the issuer's
//           included, as the attention kernel's softmax warps are) run a dependent chain of
//           FMA and SFU exp2 until the MMAs are done
// A full-rate pipe takes 64 cycles per MMA (8,192 FLOP per cycle per SM).
#include <algorithm>
#include <vector>

#include "../../include/h3.h"
#include "kernels.h"

namespace h3 {

constexpr unsigned kErrDiagIssue = 0x302;
constexpr int kIssueSmem = 120 * 1024;

__device__ unsigned long long g_issue_cycles[H3_DIAG_MAX_CTAS];
__device__ float g_issue_sink;  // keeps the busy warps' arithmetic alive

__device__ __forceinline__ void mma_ts_diag(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ uint32_t mbar_test_diag(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok;
}

template <int MODE>
__global__ void __launch_bounds__(384, 1) issue_rate_kernel(int batches, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s = smem_u32(smem);  // operands: A atoms at s, s + 16K; B atoms at s + 32K, s + 48K
  const uint32_t bar = s + 65536;     // [0] completion of the MMAs; [1] a barrier polled in modes 1, 2
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + 65536 + 64);
  volatile uint32_t* done = reinterpret_cast<volatile uint32_t*>(smem + 65536 + 128);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_init(bar + 8, 1);
    *done = 0;
    fence_barrier_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(smem_u32(slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  if (threadIdx.x == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
    const unsigned long long t0 = clock64();
    // on a freshly initialised barrier the phase of parity 1 counts as complete
    for (int g = 0; g < batches; ++g) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        umma_bf16_ss(tmem, sdesc_k_sw128(s + off), sdesc_k_sw128(s + 32768 + off), idesc, kk != 0);
      }
      uint32_t early = 1;
      if (MODE == 1 && !mbar_wait(bar + 8, 1, err, kErrDiagIssue)) break;
      if (MODE == 2) early = mbar_test_diag(bar + 8, 1);
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_ts_diag(tmem + 128, tmem + 384 + kk * 8, sdesc_k_sw128(s + 32768 + off), idesc, kk != 0);
      }
      if (MODE == 2 && !early) record_error(err, kErrDiagIssue);
      if (MODE == 3) {
        if (!mbar_wait(bar + 8, 1, err, kErrDiagIssue)) break;
        tc_fence_after();
      }
    }
    umma_commit(bar);
    mbar_wait(bar, 0, err, kErrDiagIssue);
    g_issue_cycles[blockIdx.x] = clock64() - t0;
    *done = 1;
  }
  if (MODE == 4 && threadIdx.x >= 128) {
    float a = 1.0f + 1e-3f * threadIdx.x;
    for (int it = 0; it < (1 << 22) && *done == 0u; ++it) {
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        float e;
        asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(a * -1e-3f));
        a = fmaf(a, 0.999f, e);
      }
    }
    if (a == -1.0f) g_issue_sink = a;
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int MODE>
static cudaError_t launch_issue_rate(int batches, int ctas, unsigned* err, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(issue_rate_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kIssueSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  issue_rate_kernel<MODE><<<ctas, MODE == 4 ? 384 : 128, kIssueSmem, st>>>(batches, err);
  return cudaGetLastError();
}

}  // namespace h3

using namespace h3;

extern "C" h3_status h3_diag_issue_rate(int mode, int batches, int ctas, double* cycles_per_mma, void* stream) {
  if (mode < 0 || mode > 4 || batches < 1 || batches > 100000 || ctas < 1 || ctas > H3_DIAG_MAX_CTAS ||
      !cycles_per_mma)
    return H3_EINVAL;
  unsigned* err = h3_error_word_ptr();
  if (!err) return H3_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = mode == 0   ? launch_issue_rate<0>(batches, ctas, err, st)
                  : mode == 1 ? launch_issue_rate<1>(batches, ctas, err, st)
                  : mode == 2 ? launch_issue_rate<2>(batches, ctas, err, st)
                  : mode == 3 ? launch_issue_rate<3>(batches, ctas, err, st)
                              : launch_issue_rate<4>(batches, ctas, err, st);
  if (e != cudaSuccess) return H3_ECUDA;
  std::vector<unsigned long long> cyc(ctas);
  if (cudaMemcpyFromSymbolAsync(cyc.data(), g_issue_cycles, sizeof(unsigned long long) * ctas, 0,
                                cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return H3_ECUDA;
  std::sort(cyc.begin(), cyc.end());
  *cycles_per_mma = static_cast<double>(cyc[ctas / 2]) / (16.0 * batches);
  return H3_OK;
}
