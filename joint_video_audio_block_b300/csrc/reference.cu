// Plain CUDA-core kernels for the contractions (the H3_F_UNFUSED path).
//
// These are the in-library "two-kernel oracle" counterpart of the tcgen05 kernels, in the
// spirit of the per-fusion A/B switches of the "H3-metal" README ("Exact DiT fusions"): same
// inputs, same layouts, same epilogue arithmetic, no tensor cores, no TMA.  They exist for
// A/B checks and for bring-up, not for speed.
#include "kernels.h"

namespace h3 {

// ------------------------------------------------------------------------------ linear

__device__ __forceinline__ float load_weight(const LinearArgs& a, int row, int kx) {
  if (!a.int8) return bf2f(static_cast<const bf16*>(a.w)[static_cast<size_t>(row) * a.K + kx]);
  const uint8_t qv = static_cast<const uint8_t*>(a.w)[static_cast<size_t>(row) * a.K + kx];
  const size_t g = static_cast<size_t>(row) * (a.K / 32) + kx / 32;
  const float w = __fmaf_rn(bf2f(a.wscale[g]), static_cast<float>(qv), bf2f(a.wqbias[g]));
  return bf2f(f2bf(w));
}

__device__ __forceinline__ float epilogue_value(const LinearArgs& a, int row, int col, float acc0, float acc1) {
  if (a.epi == kEpiSwiglu) {
    const float g = acc0 + (a.bias ? bf2f(a.bias[col]) : 0.f);
    const float v = acc1 + (a.bias ? bf2f(a.bias[a.n_y + col]) : 0.f);
    return g / (1.f + expf(-g)) * v;
  }
  const float y = acc0 + (a.bias ? bf2f(a.bias[col]) : 0.f);
  if (a.epi == kEpiGateRes) {
    const TableRef& t = a.gate;
    const float gate = bf2f(t.table_b[static_cast<long long>(t.tidx[row]) * t.t_stride +
                                      static_cast<long long>(6 * t.tag[row] + a.m_gate) * a.n_y + col]);
    return bf2f(a.res[static_cast<size_t>(row) * a.ldy + col]) + gate * y;
  }
  return y;
}

__global__ void __launch_bounds__(256) linear_ref_kernel(LinearArgs a) {
  __shared__ float sx[64][33];
  __shared__ float sw[2][64][33];
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int nw = (a.epi == kEpiSwiglu) ? 2 : 1;
  float acc[2][4][4];
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[p][i][j] = 0.f;

  for (int k0 = 0; k0 < a.K; k0 += 32) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < 64 * 32; idx += 256) {
      const int rr = idx / 32, kk = idx % 32;
      const int row = m0 + rr, kx = k0 + kk;
      sx[rr][kk] = (row < a.M && kx < a.K) ? bf2f(a.x[static_cast<size_t>(row) * a.lda + kx]) : 0.f;
    }
    for (int p = 0; p < nw; ++p) {
      for (int idx = threadIdx.x; idx < 64 * 32; idx += 256) {
        const int rr = idx / 32, kk = idx % 32;
        const int col = n0 + rr, kx = k0 + kk;
        sw[p][rr][kk] = (col < a.n_y && kx < a.K) ? load_weight(a, p * a.n_y + col, kx) : 0.f;
      }
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < 32; ++kk) {
      float xv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = sx[ty * 4 + i][kk];
      for (int p = 0; p < nw; ++p) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float wv = sw[p][tx * 4 + j][kk];
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[p][i][j] = fmaf(xv[i], wv, acc[p][i][j]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = m0 + ty * 4 + i;
    if (row >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = n0 + tx * 4 + j;
      if (col >= a.n_y) continue;
      a.y[static_cast<size_t>(row) * a.ldy + col] = f2bf(epilogue_value(a, row, col, acc[0][i][j], acc[1][i][j]));
    }
  }
}

cudaError_t launch_linear_ref(const LinearArgs& a, cudaStream_t st) {
  if (a.M <= 0) return cudaSuccess;
  dim3 grid(cdiv(a.n_y, 64), cdiv(a.M, 64));
  linear_ref_kernel<<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------ attention

// One CTA = 64 queries of one head; two threads per query, each owning half of head_dim.
template <int HD>
__global__ void __launch_bounds__(128) attention_ref_kernel(const bf16* __restrict__ q, const bf16* __restrict__ k,
                                                            const bf16* __restrict__ vt, int ld_vt, bf16* __restrict__ o,
                                                            int n_rows, int nh) {
  constexpr int HH = HD / 2;
  constexpr int KT = 32;  // keys per tile
  __shared__ float sk[KT][HD + 1];
  __shared__ float sv[KT][HD + 1];
  const int h = blockIdx.y;
  const int qi = blockIdx.x * 64 + threadIdx.x / 2;
  const int part = threadIdx.x & 1;
  const bool valid = qi < n_rows;
  const float scale = rsqrtf(static_cast<float>(HD));
  float qv[HH], ov[HH];
#pragma unroll
  for (int d = 0; d < HH; ++d) {
    qv[d] = valid ? bf2f(q[(static_cast<size_t>(h) * n_rows + qi) * HD + part * HH + d]) * scale : 0.f;
    ov[d] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int j0 = 0; j0 < n_rows; j0 += KT) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < KT * HD; idx += 128) {
      const int jj = idx / HD, d = idx % HD;
      const int j = j0 + jj;
      sk[jj][d] = j < n_rows ? bf2f(k[(static_cast<size_t>(h) * n_rows + j) * HD + d]) : 0.f;
    }
    for (int idx = threadIdx.x; idx < KT * HD; idx += 128) {
      const int d = idx / KT, jj = idx % KT;
      const int j = j0 + jj;
      sv[jj][d] = j < n_rows ? bf2f(vt[(static_cast<size_t>(h) * HD + d) * ld_vt + j]) : 0.f;
    }
    __syncthreads();
    float s[KT];
    float mt = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < KT; ++jj) {
      float a = 0.f;
#pragma unroll
      for (int d = 0; d < HH; ++d) a = fmaf(qv[d], sk[jj][part * HH + d], a);
      a += __shfl_xor_sync(0xffffffffu, a, 1);
      s[jj] = (j0 + jj < n_rows) ? a : -INFINITY;
      mt = fmaxf(mt, s[jj]);
    }
    const float mn = fmaxf(m, mt);
    const float corr = expf(m - mn);
    l *= corr;
#pragma unroll
    for (int d = 0; d < HH; ++d) ov[d] *= corr;
#pragma unroll
    for (int jj = 0; jj < KT; ++jj) {
      const float p = expf(s[jj] - mn);
      l += p;
#pragma unroll
      for (int d = 0; d < HH; ++d) ov[d] = fmaf(p, sv[jj][part * HH + d], ov[d]);
    }
    m = mn;
  }
  if (valid) {
    const float inv = 1.f / l;
    bf16* dst = o + static_cast<size_t>(qi) * nh * HD + h * HD + part * HH;
#pragma unroll
    for (int d = 0; d < HH; ++d) dst[d] = f2bf(ov[d] * inv);
  }
}

cudaError_t launch_attention_ref(const bf16* q, const bf16* k, const bf16* vt, int ld_vt, bf16* o, int n_rows, int nh,
                                 int hd, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  dim3 grid(cdiv(n_rows, 64), nh);
  if (hd == 128)
    attention_ref_kernel<128><<<grid, 128, 0, st>>>(q, k, vt, ld_vt, o, n_rows, nh);
  else if (hd == 64)
    attention_ref_kernel<64><<<grid, 128, 0, st>>>(q, k, vt, ld_vt, o, n_rows, nh);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace h3
