// Trunk entry and exit, and the sampler's transitions (Euler and second-order res_multistep).
//
// "minimax-h3-mlx" README, "Architecture": modality-specific behaviour comes only from the two
// input patch projections, the per-row AdaLN tag and the two output heads; "Porting notes":
// the patch projections and output heads ship as float32 tensors; "Layout": the scheduler is
// rectified-flow Euler with an exponential sigma shift.  "H3-metal" README, "Specialized
// projection kernels": the close-reference head keeps the F32 weights; "Scheduling and
// activation memory": the sampler keeps its float32 latents on the GPU.
//
//   embed_kernel   x[r] = bf16(W z[r] + b) for one modality's rows: float32 weights [H, K]
//                  (K = 96 video / 32 audio latent features), float32 accumulation, written
//                  straight into the rows of the packed bf16 hidden stream.
//   head_kernel    v[r] = W (LN(x[r]) (1 + scale) + shift) + b for one modality's rows, the
//                  final AdaLN gathered per row from a [T][3 tags][2][H] table; float32
//                  weights [K_out, H] (K_out <= 128) and float32 arithmetic throughout;
//                  optionally also the sampler update of the float32 latent rows: the Euler
//                  transition z[r] += dsigma * v[r], or a res_multistep step (mlx-h3 README,
//                  "Why mlx-h3": the sampler's second-order solver; the page names it without
//                  defining it, and the step here is the multistep form of the refined
//                  exponential solver of Zhang, Song and Chen, 2023): with the data prediction
//                  D = z - sigma v, z <- a z + c_now D + c_prev D_prev, D_prev <- D, the weights
//                  from h3_res_multistep_step.
#include <algorithm>
#include <cmath>
#include <functional>
#include <vector>

#include "../../include/h3.h"
#include "kernels.h"

namespace h3 {

// ------------------------------------------------------------------------------ embed

constexpr int EM_ROWS = 64, EM_COLS = 128, EM_K = 32;

__global__ void __launch_bounds__(256) embed_kernel(const float* __restrict__ z, int K, const float* __restrict__ w,
                                                    const float* __restrict__ b, int n_rows, int H,
                                                    bf16* __restrict__ x) {
  __shared__ float zs[EM_K][EM_ROWS + 1];
  __shared__ float ws[EM_K][EM_COLS + 1];
  const int r0 = blockIdx.y * EM_ROWS, c0 = blockIdx.x * EM_COLS;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;  // rows ty*4 .. +3, cols tx*8 .. +7
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < K; k0 += EM_K) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < EM_ROWS * EM_K; idx += 256) {
      const int rr = idx / EM_K, kk = idx % EM_K;
      const int r = r0 + rr, k = k0 + kk;
      zs[kk][rr] = (r < n_rows && k < K) ? z[static_cast<size_t>(r) * K + k] : 0.f;
    }
    for (int idx = threadIdx.x; idx < EM_COLS * EM_K; idx += 256) {
      const int cc = idx / EM_K, kk = idx % EM_K;
      const int c = c0 + cc, k = k0 + kk;
      ws[kk][cc] = (c < H && k < K) ? w[static_cast<size_t>(c) * K + k] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < EM_K; ++kk) {
      float a[4], bw[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = zs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 8; ++j) bw[j] = ws[kk][tx * 8 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], bw[j], acc[i][j]);
    }
  }
  const int c = c0 + tx * 8;
  if (c >= H) return;  // H % 64 == 0, so a group of 8 columns is all in or all out
  float bias[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) bias[j] = b ? b[c + j] : 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + ty * 4 + i;
    if (r >= n_rows) continue;
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = pack_bf16x2(acc[i][2 * e] + bias[2 * e], acc[i][2 * e + 1] + bias[2 * e + 1]);
    *reinterpret_cast<int4*>(x + static_cast<size_t>(r) * H + c) = make_int4(o[0], o[1], o[2], o[3]);
  }
}

// ------------------------------------------------------------------------------ head

// A CTA owns HD_ROWS rows and all K_out (<= HD_NMAX) outputs: the row statistics first (one
// warp per row), then a register-tiled float32 GEMM over H in chunks of HD_K, the normalised
// and modulated activations formed while the A chunk is staged into shared memory (the row
// was just read, so the second read hits L2).  Thread (ty, tx) accumulates rows ty*4 .. +3 and
// outputs tx + 16 j, j < HD_NMAX / 16.
constexpr int HD_ROWS = 64, HD_K = 32, HD_NMAX = 128, HD_NJ = HD_NMAX / 16;

struct HeadArgs {
  const bf16* x;  // [n_rows, H] (the modality's rows of the hidden stream)
  int n_rows, H;
  const uint8_t* tag;
  const int32_t* tidx;
  const bf16* table_f;  // [T][6H] at t = 0, row stride t_stride
  long long t_stride;
  const float* w;  // [K_out, H]
  const float* b;  // [K_out] or null
  int K_out;
  float eps;
  float* v;  // [n_rows, K_out] or null
  float* z;  // [n_rows, K_out] or null: the sampler update of the latent rows
  float dsigma;
  int ms;           // 0: Euler, z += dsigma v; 1: res_multistep
  float sigma, ca, cn, cp;  // res_multistep: D = z - sigma v, z <- ca z + cn D + cp D_prev
  float* dprev;     // res_multistep: [n_rows, K_out], read when cp != 0, then overwritten with D
};

__global__ void __launch_bounds__(256) head_kernel(const HeadArgs a) {
  __shared__ float s_mean[HD_ROWS], s_rstd[HD_ROWS];
  __shared__ const bf16* s_mod[HD_ROWS];  // the row's shift vector (scale follows at + H)
  __shared__ float as[HD_K][HD_ROWS + 1];
  __shared__ float bs[HD_K][HD_NMAX + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * HD_ROWS;
  const int H = a.H;
  // 1. row statistics (fp32, two passes over the bf16 row), one warp per row
  for (int rr = warp; rr < HD_ROWS; rr += 8) {
    const int r = r0 + rr;
    float mean = 0.f, rstd = 0.f;
    const bf16* mod = a.table_f;
    if (r < a.n_rows) {
      const bf16* xr = a.x + static_cast<size_t>(r) * H;
      float s = 0.f;
      for (int c = lane * 8; c < H; c += 256) {
        const int4 u = ld_nc_v4(xr + c);
        const uint32_t wv[4] = {(uint32_t)u.x, (uint32_t)u.y, (uint32_t)u.z, (uint32_t)u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) s += bf16lo(wv[e]) + bf16hi(wv[e]);
      }
      mean = warp_sum(s) / static_cast<float>(H);
      float s2 = 0.f;
      for (int c = lane * 8; c < H; c += 256) {
        const int4 u = ld_nc_v4(xr + c);
        const uint32_t wv[4] = {(uint32_t)u.x, (uint32_t)u.y, (uint32_t)u.z, (uint32_t)u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float d0 = bf16lo(wv[e]) - mean, d1 = bf16hi(wv[e]) - mean;
          s2 = fmaf(d0, d0, fmaf(d1, d1, s2));
        }
      }
      rstd = rsqrtf(warp_sum(s2) / static_cast<float>(H) + a.eps);
      mod = a.table_f + static_cast<long long>(a.tidx[r]) * a.t_stride + static_cast<long long>(2 * a.tag[r]) * H;
    }
    if (lane == 0) {
      s_mean[rr] = mean;
      s_rstd[rr] = rstd;
      s_mod[rr] = mod;
    }
  }
  __syncthreads();
  // 2. v = W xn + b, register-tiled
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  float acc[4][HD_NJ];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < HD_NJ; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < H; k0 += HD_K) {
    __syncthreads();
    // A chunk: xn[row][k0 .. k0+31] = (x - mean) rstd (1 + scale) + shift
    for (int idx = threadIdx.x; idx < HD_ROWS * HD_K; idx += 256) {
      const int rr = idx / HD_K, kk = idx % HD_K;
      const int r = r0 + rr, k = k0 + kk;
      float val = 0.f;
      if (r < a.n_rows && k < H) {
        const bf16* mod = s_mod[rr];
        const float xv = bf2f(a.x[static_cast<size_t>(r) * H + k]);
        val = (xv - s_mean[rr]) * s_rstd[rr] * (1.f + bf2f(mod[H + k])) + bf2f(mod[k]);
      }
      as[kk][rr] = val;
    }
    // B chunk: W^T[k0 .. k0+31][o]
    for (int idx = threadIdx.x; idx < HD_NMAX * HD_K; idx += 256) {
      const int o = idx / HD_K, kk = idx % HD_K;
      const int k = k0 + kk;
      bs[kk][o] = (o < a.K_out && k < H) ? __ldg(a.w + static_cast<size_t>(o) * H + k) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < HD_K; ++kk) {
      float av[4], bv[HD_NJ];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = as[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < HD_NJ; ++j) bv[j] = bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < HD_NJ; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
  }
  // 3. bias, optional v, optional sampler update of the latent rows
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + ty * 4 + i;
    if (r >= a.n_rows) continue;
#pragma unroll
    for (int j = 0; j < HD_NJ; ++j) {
      const int o = tx + 16 * j;
      if (o >= a.K_out) continue;
      const float v = acc[i][j] + (a.b ? a.b[o] : 0.f);
      const size_t idx = static_cast<size_t>(r) * a.K_out + o;
      if (a.v) a.v[idx] = v;
      if (a.z) {
        const float z = a.z[idx];
        if (a.ms) {
          const float dn = fmaf(-a.sigma, v, z);
          float zn = fmaf(a.cn, dn, a.ca * z);
          if (a.cp != 0.f) zn = fmaf(a.cp, a.dprev[idx], zn);
          a.z[idx] = zn;
          a.dprev[idx] = dn;
        } else {
          a.z[idx] = fmaf(a.dsigma, v, z);
        }
      }
    }
  }
}

}  // namespace h3

using namespace h3;

namespace {
bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool a4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }  // float32 / int32 arrays
}  // namespace

extern "C" h3_status h3_embed_rows(const h3_dims* dims, const float* z, int K, const float* w, const float* b,
                                   int n_rows, void* x_rows, void* stream) {
  if (!dims || !z || !w || !x_rows || K <= 0 || K > 4096 || n_rows < 0) return H3_EINVAL;
  const int H = dims->hidden;
  if (H <= 0 || H % 64 || !a16(x_rows) || !a4(z) || !a4(w) || !a4(b)) return H3_EINVAL;
  if (n_rows == 0) return H3_OK;
  dim3 grid(cdiv(H, EM_COLS), cdiv(n_rows, EM_ROWS));
  embed_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(z, K, w, b, n_rows, H, static_cast<bf16*>(x_rows));
  return cudaGetLastError() == cudaSuccess ? H3_OK : H3_ECUDA;
}

namespace {
h3_status launch_head(const h3_dims* dims, const void* x_rows, int n_rows, const uint8_t* tag, const int32_t* tidx,
                      const void* table_f, long long t_stride, const float* w, const float* b, int K_out, float* v_out,
                      float* z_inout, float dsigma, const h3_ms_step* ms, float* d_prev, void* stream) {
  if (!dims || !x_rows || !tag || !tidx || !table_f || !w || K_out <= 0 || K_out > HD_NMAX || n_rows < 0)
    return H3_EINVAL;
  if (!v_out && !z_inout) return H3_EINVAL;
  const int H = dims->hidden;
  if (H <= 0 || H % 64 || !a16(x_rows) || t_stride < 6LL * H) return H3_EINVAL;
  if (!a4(tidx) || !a4(w) || !a4(b) || !a4(v_out) || !a4(z_inout) || !a4(d_prev) ||
      (reinterpret_cast<uintptr_t>(table_f) & 1))
    return H3_EINVAL;
  if (ms && (!z_inout || !d_prev || !(ms->sigma > 0.f))) return H3_EINVAL;
  if (n_rows == 0) return H3_OK;
  HeadArgs a{static_cast<const bf16*>(x_rows), n_rows, H, tag, tidx, static_cast<const bf16*>(table_f), t_stride,
             w, b, K_out, dims->ln_eps, v_out, z_inout, dsigma, ms ? 1 : 0, ms ? ms->sigma : 0.f, ms ? ms->a : 0.f,
             ms ? ms->c_now : 0.f, ms ? ms->c_prev : 0.f, d_prev};
  head_kernel<<<cdiv(n_rows, HD_ROWS), 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? H3_OK : H3_ECUDA;
}
}  // namespace

extern "C" h3_status h3_head_forward(const h3_dims* dims, const void* x_rows, int n_rows, const uint8_t* tag,
                                     const int32_t* tidx, const void* table_f, long long t_stride, const float* w,
                                     const float* b, int K_out, float* v_out, float* z_inout, float dsigma,
                                     void* stream) {
  return launch_head(dims, x_rows, n_rows, tag, tidx, table_f, t_stride, w, b, K_out, v_out, z_inout, dsigma, nullptr,
                     nullptr, stream);
}

extern "C" h3_status h3_head_forward_ms(const h3_dims* dims, const void* x_rows, int n_rows, const uint8_t* tag,
                                        const int32_t* tidx, const void* table_f, long long t_stride, const float* w,
                                        const float* b, int K_out, const h3_ms_step* step, float* v_out,
                                        float* z_inout, float* d_prev_inout, void* stream) {
  if (!step) return H3_EINVAL;
  return launch_head(dims, x_rows, n_rows, tag, tidx, table_f, t_stride, w, b, K_out, v_out, z_inout, 0.f, step,
                     d_prev_inout, stream);
}

// The weights of one res_multistep step, in double precision, rounded once to float.  In
// log-noise time t = -ln(sigma) the sampling ODE is dz/dt = D - z; over a step of length
// h = ln(sigma / sigma_next), with D linear in t through D_now and D_prev (at r h,
// r = ln(sigma / sigma_prev) / h < 0), variation of constants gives
//   a = e^-h,  c_now = h (phi1 - phi2 / r),  c_prev = h phi2 / r,
// phi1 = (1 - e^-h) / h and phi2 = (1 - phi1) / h.  The first step (no previous prediction)
// takes D constant: a = sigma_next / sigma, c_now = 1 - a (the Euler step); a step to 0
// returns D (a = 0, c_now = 1).
extern "C" h3_status h3_res_multistep_step(float sigma_prev, float sigma, float sigma_next, h3_ms_step* out) {
  if (!out || !(sigma > 0.f) || !(sigma_next >= 0.f) || !(sigma_next < sigma) || std::isnan(sigma_prev))
    return H3_EINVAL;
  const bool first = !(sigma_prev > 0.f);
  if (!first && !(sigma_prev > sigma)) return H3_EINVAL;
  const double s = sigma, sn = sigma_next, sp = sigma_prev;
  double a = 0.0, cn = 1.0, cp = 0.0;
  if (sn > 0.0) {
    a = sn / s;
    cn = 1.0 - a;
    if (!first) {
      const double h = std::log(s / sn), r = std::log(s / sp) / h;
      const double phi1 = -std::expm1(-h) / h, phi2 = (1.0 - phi1) / h;
      cn = h * (phi1 - phi2 / r);
      cp = h * phi2 / r;
    }
  }
  out->sigma = sigma;
  out->a = static_cast<float>(a);
  out->c_now = static_cast<float>(cn);
  out->c_prev = static_cast<float>(cp);
  return H3_OK;
}

extern "C" h3_status h3_final_modcache_build(const h3_dims* dims, const float* temb, int T, int Dt, const void* w,
                                             const void* b, void* table_f, void* stream) {
  if (!dims || !temb || !a16(temb) || !w || !table_f || T <= 0 || Dt <= 0 || Dt % 8 || !a16(w)) return H3_EINVAL;
  const int n_out = 6 * dims->hidden;
  if (dims->hidden <= 0 || dims->hidden % 64) return H3_EINVAL;
  const bf16* wp = static_cast<const bf16*>(w);
  const bf16* bp = static_cast<const bf16*>(b);
  const cudaError_t e = launch_modcache(temb, T, Dt, &wp, &bp, 1, n_out, static_cast<bf16*>(table_f), n_out,
                                        h3_error_word_ptr(), static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) return H3_OK;
  return e == cudaErrorInvalidValue ? H3_EINVAL : H3_ECUDA;
}

// float32 linspace the way the scheduler's reference evaluates it (a float32 step; the first
// half from the start, the second half back from the end, each point one fused multiply-add),
// then the time shift s sigma / (1 + (s - 1) sigma) in float32.
extern "C" h3_status h3_sigma_schedule(int steps, float shift, float* sigma_out) {
  if (steps < 1 || !sigma_out || !(shift > 0.f)) return H3_EINVAL;
  const int n = steps + 1;
  const float start = 1.f, end = 0.f;
  const float step = (end - start) / static_cast<float>(n - 1);
  const int half = n / 2;
  for (int i = 0; i < n; ++i) {
    const float s = i < half ? std::fma(step, static_cast<float>(i), start)
                             : std::fma(-step, static_cast<float>(n - 1 - i), end);
    sigma_out[i] = shift * s / (1.f + (shift - 1.f) * s);
  }
  return H3_OK;
}

// The plan of a run: both schedules' grids (h3_sigma_schedule), the distinct timesteps 1000 sigma
// (float32) their transitions evaluate, in descending order -- the rows of the modulation
// tables -- and each transition's row for video and for audio.  Exact equality decides
// "distinct": the table must hold the very values the sampler evaluates.
extern "C" h3_status h3_sampler_plan(int steps, float shift_video, float shift_audio, float* timesteps,
                                     int* n_timesteps, int32_t* vidx, int32_t* aidx) {
  if (steps < 1 || !timesteps || !n_timesteps || !vidx || !aidx) return H3_EINVAL;
  std::vector<float> sv(steps + 1), sa(steps + 1);
  h3_status st = h3_sigma_schedule(steps, shift_video, sv.data());
  if (st != H3_OK) return st;
  if ((st = h3_sigma_schedule(steps, shift_audio, sa.data())) != H3_OK) return st;
  std::vector<float> tv(steps), ta(steps), all;
  all.reserve(2 * steps);
  for (int i = 0; i < steps; ++i) {
    tv[i] = 1000.f * sv[i];
    ta[i] = 1000.f * sa[i];
    all.push_back(tv[i]);
    all.push_back(ta[i]);
  }
  std::sort(all.begin(), all.end(), std::greater<float>());
  all.erase(std::unique(all.begin(), all.end()), all.end());
  auto row = [&](float t) {
    return static_cast<int32_t>(std::lower_bound(all.begin(), all.end(), t, std::greater<float>()) - all.begin());
  };
  for (int i = 0; i < steps; ++i) {
    vidx[i] = row(tv[i]);
    aidx[i] = row(ta[i]);
  }
  std::copy(all.begin(), all.end(), timesteps);
  *n_timesteps = static_cast<int>(all.size());
  return H3_OK;
}
