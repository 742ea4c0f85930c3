// a0: ModulationCache build -- table[t][j] = bf16(sum_k W[j][k] * temb[t][k] + b[j]).
//
// "minimax-h3-mlx" README, "AdaLN precompute": adaln_proj of each block reads only the
// timestep embedding, so every modulation vector of a run is computed once up front and the
// projection dropped; the table is built from the float32 timestep embedding through the
// unquantised projection.  The product is kept in fp32 (fp32 temb x bf16 weight, fp32 FMA
// accumulation) so the table carries no extra rounding of the embedding; that rules out the
// bf16 tensor cores, so this is a CUDA-core kernel bound by fp32 FMA throughput
// (2 T 18H Dt FLOP per block) with every weight read from HBM exactly once.
//
// Tiling: a CTA owns 128 weight rows and up to MC_TMAX timesteps (all of them for T <= 80);
// the reduction runs in 32-wide chunks staged through shared memory (weights widened to fp32
// once per chunk with 16-byte loads).  256 threads, each accumulating 8 rows x 5 timesteps.
#include "kernels.h"

namespace h3 {

constexpr int MC_ROWS = 128, MC_K = 32, MC_TT = 5, MC_TMAX = 16 * MC_TT;

__global__ void __launch_bounds__(256) modcache_kernel(const float* __restrict__ temb, int T, int Dt,
                                                       const bf16* __restrict__ W, const bf16* __restrict__ bias,
                                                       int n_out, bf16* __restrict__ table_b, long long t_stride) {
  // k-major: a thread's 8 rows are 8 consecutive floats; the odd row pitches (129, 81 words)
  // keep the transposing stores of the staging loops free of bank conflicts
  __shared__ float sw[MC_K][MC_ROWS + 1];
  __shared__ float st[MC_K][MC_TMAX + 1];
  const int j0 = blockIdx.x * MC_ROWS;
  const int t_base = blockIdx.y * MC_TMAX;
  const int tr = threadIdx.x & 15;          // timesteps t_base + tr + 16 i, i < 5
  const int jr = (threadIdx.x >> 4) * 8;    // rows j0 + jr .. + 7
  float acc[8][MC_TT];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < MC_TT; ++b) acc[a][b] = 0.f;

  for (int k0 = 0; k0 < Dt; k0 += MC_K) {
    __syncthreads();
    // weights: 128 rows x 32 k = 512 vectors of 8 bf16; Dt % 8 == 0 keeps every vector whole
    for (int v = threadIdx.x; v < MC_ROWS * MC_K / 8; v += 256) {
      const int rr = v >> 2, kk = (v & 3) * 8;
      const int j = j0 + rr, kx = k0 + kk;
      float f[8];
      if (j < n_out && kx < Dt) {
        const int4 u = ld_nc_v4(W + static_cast<size_t>(j) * Dt + kx);
        const uint32_t w[4] = {(uint32_t)u.x, (uint32_t)u.y, (uint32_t)u.z, (uint32_t)u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          f[2 * e] = bf16lo(w[e]);
          f[2 * e + 1] = bf16hi(w[e]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) sw[kk + e][rr] = f[e];
    }
    for (int v = threadIdx.x; v < MC_TMAX * MC_K; v += 256) {
      const int tt = v / MC_K, kk = v % MC_K;
      const int t = t_base + tt, kx = k0 + kk;
      st[kk][tt] = (t < T && kx < Dt) ? temb[static_cast<size_t>(t) * Dt + kx] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < MC_K; ++kk) {
      float wv[8], tv[MC_TT];
#pragma unroll
      for (int a = 0; a < 8; ++a) wv[a] = sw[kk][jr + a];
#pragma unroll
      for (int b = 0; b < MC_TT; ++b) tv[b] = st[kk][tr + 16 * b];
#pragma unroll
      for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < MC_TT; ++b) acc[a][b] = fmaf(wv[a], tv[b], acc[a][b]);
    }
  }
  float bj[8];
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    const int j = j0 + jr + a;
    bj[a] = (bias && j < n_out) ? bf2f(bias[j]) : 0.f;
  }
#pragma unroll
  for (int b = 0; b < MC_TT; ++b) {
    const int t = t_base + tr + 16 * b;
    if (t >= T) continue;
    bf16* dst = table_b + static_cast<long long>(t) * t_stride + j0 + jr;
    if (j0 + jr + 8 <= n_out && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(acc[2 * e][b] + bj[2 * e], acc[2 * e + 1][b] + bj[2 * e + 1]);
      *reinterpret_cast<int4*>(dst) = make_int4(w[0], w[1], w[2], w[3]);
    } else {
#pragma unroll
      for (int a = 0; a < 8; ++a)
        if (j0 + jr + a < n_out) dst[a] = f2bf(acc[a][b] + bj[a]);
    }
  }
}

cudaError_t launch_modcache(const float* temb, int T, int Dt, const bf16* W, const bf16* bias, int n_out,
                            bf16* table_b, long long t_stride, cudaStream_t st) {
  if (T <= 0 || n_out <= 0) return cudaSuccess;
  if (Dt % 8) return cudaErrorInvalidValue;
  dim3 grid(cdiv(n_out, MC_ROWS), cdiv(T, MC_TMAX));
  modcache_kernel<<<grid, 256, 0, st>>>(temb, T, Dt, W, bias, n_out, table_b, t_stride);
  return cudaGetLastError();
}

}  // namespace h3
