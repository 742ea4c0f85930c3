// a0: ModulationCache build -- table[t][j] = bf16(sum_k W[j][k] * temb[t][k] + b[j]).
//
// "minimax-h3-mlx" README, "AdaLN precompute": adaln_proj of each block reads only the
// timestep embedding, so every modulation vector of a run is computed once up front and the
// projection dropped; the table is built from the float32 timestep embedding through the
// unquantised projection.  The product is kept in fp32 (fp32 temb x bf16 weight, fp32 FMA
// accumulation) so the table carries no extra rounding of the embedding.
//
// Tiling: a CTA owns 128 weight rows; timesteps are processed 16 at a time, the reduction in
// 64-wide chunks staged through shared memory (weights widened to fp32 once per chunk).
#include "kernels.h"

namespace h3 {

constexpr int MC_ROWS = 128, MC_T = 16, MC_K = 64;

__global__ void __launch_bounds__(256) modcache_kernel(const float* __restrict__ temb, int T, int Dt,
                                                       const bf16* __restrict__ W, const bf16* __restrict__ bias,
                                                       int n_out, bf16* __restrict__ table_b, long long t_stride) {
  __shared__ float sw[MC_ROWS][MC_K + 1];
  __shared__ float st[MC_T][MC_K + 1];
  const int j0 = blockIdx.x * MC_ROWS;
  const int tl = threadIdx.x % MC_T;         // timestep within the chunk
  const int jb = (threadIdx.x / MC_T) * 8;   // 8 rows per thread
  for (int t0 = 0; t0 < T; t0 += MC_T) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int k0 = 0; k0 < Dt; k0 += MC_K) {
      __syncthreads();
      for (int idx = threadIdx.x; idx < MC_ROWS * MC_K; idx += 256) {
        const int rr = idx / MC_K, kk = idx % MC_K;
        const int j = j0 + rr, kx = k0 + kk;
        sw[rr][kk] = (j < n_out && kx < Dt) ? bf2f(W[static_cast<size_t>(j) * Dt + kx]) : 0.f;
      }
      for (int idx = threadIdx.x; idx < MC_T * MC_K; idx += 256) {
        const int tt = idx / MC_K, kk = idx % MC_K;
        const int t = t0 + tt, kx = k0 + kk;
        st[tt][kk] = (t < T && kx < Dt) ? temb[static_cast<size_t>(t) * Dt + kx] : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < MC_K; ++kk) {
        const float tv = st[tl][kk];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(sw[jb + i][kk], tv, acc[i]);
      }
    }
    const int t = t0 + tl;
    if (t < T) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = j0 + jb + i;
        if (j < n_out) {
          const float b = bias ? bf2f(bias[j]) : 0.f;
          table_b[static_cast<long long>(t) * t_stride + j] = f2bf(acc[i] + b);
        }
      }
    }
  }
}

cudaError_t launch_modcache(const float* temb, int T, int Dt, const bf16* W, const bf16* bias, int n_out,
                            bf16* table_b, long long t_stride, cudaStream_t st) {
  if (T <= 0 || n_out <= 0) return cudaSuccess;
  modcache_kernel<<<cdiv(n_out, MC_ROWS), 256, 0, st>>>(temb, T, Dt, W, bias, n_out, table_b, t_stride);
  return cudaGetLastError();
}

}  // namespace h3
