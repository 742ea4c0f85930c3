// a1 / a6: per-row gather of the AdaLN modulation + LayerNorm + modulate.
//
// "minimax-h3-mlx" README, "AdaLN: measure, do not reason": the norms are modulated as
// x * (1 + scale) + shift; "Architecture": the row's modality tag selects its modulation.
// The whole row stays in registers (128-bit loads, 8 bf16 per vector), so x is read from HBM
// once and xn written once: 4*H bytes per row.
#include "kernels.h"

namespace h3 {

__device__ __forceinline__ void unpack8(const int4& u, float* f) {
  const uint32_t w[4] = {(uint32_t)u.x, (uint32_t)u.y, (uint32_t)u.z, (uint32_t)u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16lo(w[i]);
    f[2 * i + 1] = bf16hi(w[i]);
  }
}

// a pair of block-wide sums (every thread receives both)
__device__ __forceinline__ float2 block_sum2(float a, float b, float2* red) {
  a = warp_sum(a);
  b = warp_sum(b);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (lane == 0) red[warp] = make_float2(a, b);
  __syncthreads();
  float2 t = lane < nw ? red[lane] : make_float2(0.f, 0.f);
  return make_float2(warp_sum(t.x), warp_sum(t.y));
}

// One CTA per row.  The row (VPT 16-byte vectors per thread) and the row's shift and scale
// vectors are all loaded up front as packed bf16, so the gather's latency overlaps the
// statistics.  The statistics take one block reduction: the sums of d and d^2 for
// d = x - x[0] (shifting by an element of the row keeps E[d^2] - E[d]^2 free of the
// cancellation a large mean would cause), accumulated in fp32.
template <int VPT>
__global__ void __launch_bounds__(1024) adaln_modulate_kernel(const bf16* __restrict__ x, bf16* __restrict__ xn, int H,
                                                               float eps, TableRef tr, int m_shift, int m_scale) {
  __shared__ float2 red[32];
  const int r = blockIdx.x;
  const int nvec = H >> 3;
  const int4* xr = reinterpret_cast<const int4*>(x + static_cast<size_t>(r) * H);
  const int tg = tr.tag[r];
  const long long base = static_cast<long long>(tr.tidx[r]) * tr.t_stride;
  const int4* sh = reinterpret_cast<const int4*>(tr.table_b + base + static_cast<long long>(6 * tg + m_shift) * H);
  const int4* sc = reinterpret_cast<const int4*>(tr.table_b + base + static_cast<long long>(6 * tg + m_scale) * H);
  int4 v[VPT], vs[VPT], vc[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int vi = threadIdx.x + i * blockDim.x;
    const bool ok = vi < nvec;
    v[i] = ok ? ld_nc_v4(xr + vi) : make_int4(0, 0, 0, 0);
    vs[i] = ok ? ld_nc_v4(sh + vi) : make_int4(0, 0, 0, 0);
    vc[i] = ok ? ld_nc_v4(sc + vi) : make_int4(0, 0, 0, 0);
  }
  const float x0 = bf2f(x[static_cast<size_t>(r) * H]);
  float s1 = 0.f, s2 = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    if (threadIdx.x + i * blockDim.x < nvec) {
      float f[8];
      unpack8(v[i], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float d = f[e] - x0;
        s1 += d;
        s2 = fmaf(d, d, s2);
      }
    }
  }
  const float2 tot = block_sum2(s1, s2, red);
  const float md = tot.x / static_cast<float>(H);
  const float mean = x0 + md;
  const float var = fmaxf(tot.y / static_cast<float>(H) - md * md, 0.f);
  const float rstd = rsqrtf(var + eps);
  int4* out = reinterpret_cast<int4*>(xn + static_cast<size_t>(r) * H);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int vi = threadIdx.x + i * blockDim.x;
    if (vi < nvec) {
      float f[8], fs[8], fc[8];
      unpack8(v[i], f);
      unpack8(vs[i], fs);
      unpack8(vc[i], fc);
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = (f[2 * e] - mean) * rstd * (1.f + fc[2 * e]) + fs[2 * e];
        const float b = (f[2 * e + 1] - mean) * rstd * (1.f + fc[2 * e + 1]) + fs[2 * e + 1];
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
