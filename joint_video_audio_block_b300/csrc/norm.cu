// a1 / a6: per-row gather of the AdaLN modulation + LayerNorm + modulate.
//
// "minimax-h3-mlx" README, "AdaLN: measure, do not reason": the norms are modulated as
// x * (1 + scale) + shift; "Architecture": the row's modality tag selects its modulation.
// One CTA per row keeps the whole row in registers (128-bit loads, 8 bf16 per vector), so x
// is read from HBM once and xn written once: 4*H bytes per row.  Statistics are two-pass
// (mean, then centred variance) in fp32 with warp-shuffle + shared-memory reductions.
#include "kernels.h"

namespace h3 {

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();  // red[] may still be read from a previous reduction
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  return warp_sum(t);
}

__device__ __forceinline__ void unpack8(const int4& u, float* f) {
  const uint32_t w[4] = {(uint32_t)u.x, (uint32_t)u.y, (uint32_t)u.z, (uint32_t)u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16lo(w[i]);
    f[2 * i + 1] = bf16hi(w[i]);
  }
}

template <int VPT>
__global__ void __launch_bounds__(1024) adaln_modulate_kernel(const bf16* __restrict__ x, bf16* __restrict__ xn, int H,
                                                               float eps, TableRef tr, int m_shift, int m_scale) {
  __shared__ float red[32];
  const int r = blockIdx.x;
  const int nvec = H >> 3;
  const int4* xr = reinterpret_cast<const int4*>(x + static_cast<size_t>(r) * H);
  float v[VPT][8];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int vi = threadIdx.x + i * blockDim.x;
    if (vi < nvec) {
      unpack8(ld_nc_v4(xr + vi), v[i]);
#pragma unroll
      for (int e = 0; e < 8; ++e) s += v[i][e];
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[i][e] = 0.f;
    }
  }
  const float mean = block_sum(s, red) / static_cast<float>(H);
  float s2 = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int vi = threadIdx.x + i * blockDim.x;
    if (vi < nvec) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float d = v[i][e] - mean;
        s2 += d * d;
      }
    }
  }
  const float var = block_sum(s2, red) / static_cast<float>(H);
  const float rstd = rsqrtf(var + eps);

  const int tg = tr.tag[r];
  const long long base = static_cast<long long>(tr.tidx[r]) * tr.t_stride;
  const int4* sh = reinterpret_cast<const int4*>(tr.table_b + base + static_cast<long long>(6 * tg + m_shift) * H);
  const int4* sc = reinterpret_cast<const int4*>(tr.table_b + base + static_cast<long long>(6 * tg + m_scale) * H);
  int4* out = reinterpret_cast<int4*>(xn + static_cast<size_t>(r) * H);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int vi = threadIdx.x + i * blockDim.x;
    if (vi < nvec) {
      float fs[8], fc[8];
      unpack8(ld_nc_v4(sh + vi), fs);
      unpack8(ld_nc_v4(sc + vi), fc);
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = (v[i][2 * e] - mean) * rstd * (1.f + fc[2 * e]) + fs[2 * e];
        const float b = (v[i][2 * e + 1] - mean) * rstd * (1.f + fc[2 * e + 1]) + fs[2 * e + 1];
        o[e] = pack_bf16x2(a, b);
      }
      out[vi] = make_int4(o[0], o[1], o[2], o[3]);
    }
  }
}

cudaError_t launch_adaln_modulate(const bf16* x, bf16* xn, int n_rows, int H, float eps, TableRef tr, int m_shift,
                                  int m_scale, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  const int nvec = H / 8;
  int vpt = cdiv(nvec, 256);
  if (vpt < 1) vpt = 1;
  if (vpt > 4) return cudaErrorInvalidValue;  // H > 8192
  int threads = cdiv(cdiv(nvec, vpt), 32) * 32;
  dim3 grid(n_rows);
  switch (vpt) {
    case 1: adaln_modulate_kernel<1><<<grid, threads, 0, st>>>(x, xn, H, eps, tr, m_shift, m_scale); break;
    case 2: adaln_modulate_kernel<2><<<grid, threads, 0, st>>>(x, xn, H, eps, tr, m_shift, m_scale); break;
    case 3: adaln_modulate_kernel<3><<<grid, threads, 0, st>>>(x, xn, H, eps, tr, m_shift, m_scale); break;
    default: adaln_modulate_kernel<4><<<grid, threads, 0, st>>>(x, xn, H, eps, tr, m_shift, m_scale); break;
  }
  return cudaGetLastError();
}

}  // namespace h3
