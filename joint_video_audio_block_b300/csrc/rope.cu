// a3: QK RMSNorm + 3D MM-RoPE on the per-head interleaved QKV projection.
//
// "H3-metal" README, "Checkpoint layout and media pipeline": the checkpoint stores qkv rows
// interleaved per head and a fused QK-normalisation/RoPE kernel consumes that layout
// directly.  "minimax-h3-mlx" README, "Validation": the projection reshapes to
// (rows, heads, 3, head_dim).  Rotary reading: rotate-half pairs (i, i + hd/2), frequency
// theta^(-2i/hd), pairs split into contiguous (t, h, w) sections.
//
// Outputs are laid out for the attention kernel: q and k head-major [nh][N][hd] (K-major
// operands of S = Q K^T) and v transposed per head [nh][hd][ld_vt] (K-major operand of O = P V).
#include <type_traits>

#include "kernels.h"

namespace h3 {

// cs[r][i] = (cos, sin) of pos[r][axis(i)] * theta^(-2i/hd), evaluated in double once per forward.
__global__ void rope_table_kernel(const float* __restrict__ pos, float2* __restrict__ cs, int n_rows, int hd, int s0,
                                  int s1, float theta) {
  const int half = hd / 2;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(n_rows) * half) return;
  const int r = static_cast<int>(idx / half), i = static_cast<int>(idx % half);
  const int axis = i < s0 ? 0 : (i < s0 + s1 ? 1 : 2);
  const double omega = pow(static_cast<double>(theta), -2.0 * i / hd);
  const double phi = static_cast<double>(pos[3 * r + axis]) * omega;
  double s, c;
  sincos(phi, &s, &c);
  cs[idx] = make_float2(static_cast<float>(c), static_cast<float>(s));
}

cudaError_t launch_rope_table(const float* pos, float2* cs, int n_rows, int hd, const int sections[3], float theta,
                              cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  const long long n = static_cast<long long>(n_rows) * (hd / 2);
  rope_table_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(pos, cs, n_rows, hd, sections[0],
                                                                            sections[1], theta);
  return cudaGetLastError();
}

// One CTA = 64 rows x 1 head; each warp handles 8 rows, each lane hd/32 elements of q, k, v.
template <int HD>
__global__ void __launch_bounds__(256) qknorm_rope_kernel(const bf16* __restrict__ qkv, const float2* __restrict__ cs,
                                                          const bf16* __restrict__ qn, const bf16* __restrict__ kn,
                                                          float eps, bf16* __restrict__ q, bf16* __restrict__ k,
                                                          bf16* __restrict__ vt, int ld_vt, int n_rows, int nh) {
  constexpr int EPL = HD / 32;     // elements per lane (4 or 2)
  constexpr int HALF = HD / 2;
  constexpr int PART = HALF / EPL;  // lane distance between the two halves of a rotary pair
  __shared__ __align__(16) bf16 sv[64][HD + 8];
  const int h = blockIdx.y, r0 = blockIdx.x * 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool has_norm = (qn != nullptr) && (kn != nullptr);
  float wq[EPL], wk[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    wq[e] = has_norm ? bf2f(qn[lane * EPL + e]) : 1.f;
    wk[e] = has_norm ? bf2f(kn[lane * EPL + e]) : 1.f;
  }
  const int pi = (lane % PART) * EPL;  // pair index of this lane's first element
  const bool first_half = lane < PART;
  const size_t row_stride = static_cast<size_t>(3) * nh * HD;

  // EPL consecutive bf16 per lane move as one 4- or 8-byte word; two rows per iteration keep
  // twice the loads in flight
  using Vec = typename std::conditional<EPL == 4, uint2, uint32_t>::type;
  auto unpack = [](const Vec& u, float* f) {
    if constexpr (EPL == 4) {
      f[0] = bf16lo(u.x);
      f[1] = bf16hi(u.x);
      f[2] = bf16lo(u.y);
      f[3] = bf16hi(u.y);
    } else {
      f[0] = bf16lo(u);
      f[1] = bf16hi(u);
    }
  };
  auto pack = [](const float* f) -> Vec {
    if constexpr (EPL == 4) {
      return make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
    } else {
      return pack_bf16x2(f[0], f[1]);
    }
  };
#pragma unroll 1
  for (int rb = warp; rb < 64; rb += 16) {
    Vec in[2][3];
    float2 cr[2][EPL];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r = r0 + rb + 8 * u;
      if (r < n_rows) {
        const bf16* base = qkv + static_cast<size_t>(r) * row_stride + static_cast<size_t>(h) * 3 * HD + lane * EPL;
#pragma unroll
        for (int which = 0; which < 3; ++which) in[u][which] = *reinterpret_cast<const Vec*>(base + which * HD);
#pragma unroll
        for (int e = 0; e < EPL; ++e) cr[u][e] = cs[static_cast<size_t>(r) * HALF + pi + e];
      } else {
#pragma unroll
        for (int which = 0; which < 3; ++which) in[u][which] = Vec{};
#pragma unroll
        for (int e = 0; e < EPL; ++e) cr[u][e] = make_float2(1.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int rr = rb + 8 * u;
      const int r = r0 + rr;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        float a[EPL];
        unpack(in[u][which], a);
        if (has_norm) {
          float ss = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) ss += a[e] * a[e];
          ss = warp_sum(ss);
          const float rinv = rsqrtf(ss / HD + eps);
#pragma unroll
          for (int e = 0; e < EPL; ++e) a[e] = a[e] * rinv * (which ? wk[e] : wq[e]);
        }
        float out[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          const float b = __shfl_xor_sync(0xffffffffu, a[e], PART);
          const float2 c = cr[u][e];
          // first half holds x_i, partner x_{i+hd/2}: x_i cos - x_{i+hd/2} sin
          // second half holds x_{i+hd/2}, partner x_i: x_i sin + x_{i+hd/2} cos
          out[e] = first_half ? (a[e] * c.x - b * c.y) : (b * c.y + a[e] * c.x);
        }
        if (r < n_rows)
          *reinterpret_cast<Vec*>((which ? k : q) + (static_cast<size_t>(h) * n_rows + r) * HD + lane * EPL) = pack(out);
      }
      *reinterpret_cast<Vec*>(&sv[rr][lane * EPL]) = in[u][2];  // zeros for rows past the end
    }
  }
  __syncthreads();
  // transposed store of v: 16-byte chunks of 8 consecutive rows for one d
  for (int c = threadIdx.x; c < HD * 8; c += 256) {
    const int d = c >> 3, j0 = (c & 7) * 8;
    if (r0 + j0 >= n_rows) continue;
    uint32_t w[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const uint32_t lo = __bfloat16_as_ushort(sv[j0 + 2 * jj][d]);
      const uint32_t hi = __bfloat16_as_ushort(sv[j0 + 2 * jj + 1][d]);
      w[jj] = lo | (hi << 16);
    }
    *reinterpret_cast<int4*>(vt + (static_cast<size_t>(h) * HD + d) * ld_vt + r0 + j0) = make_int4(w[0], w[1], w[2], w[3]);
  }
}

cudaError_t launch_qknorm_rope(const bf16* qkv, const float2* cs, const bf16* qn, const bf16* kn, float eps, bf16* q,
                               bf16* k, bf16* vt, int ld_vt, int n_rows, int nh, int hd, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  dim3 grid(cdiv(n_rows, 64), nh);
  if (hd == 128)
    qknorm_rope_kernel<128><<<grid, 256, 0, st>>>(qkv, cs, qn, kn, eps, q, k, vt, ld_vt, n_rows, nh);
  else if (hd == 64)
    qknorm_rope_kernel<64><<<grid, 256, 0, st>>>(qkv, cs, qn, kn, eps, q, k, vt, ld_vt, n_rows, nh);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace h3
