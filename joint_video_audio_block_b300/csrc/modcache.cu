// a0: ModulationCache build -- table[t][b][j] = bf16(sum_k W_b[j][k] * temb[t][k] + bias_b[j]).
//
// "minimax-h3-mlx" README, "AdaLN precompute": adaln_proj of each block reads only the
// timestep embedding, so every modulation vector of a run is computed once up front and the
// projection dropped; the table is built from the float32 timestep embedding through the
// unquantised projection.  Reading the 50 x [96768, 2688] bf16 weights (26 GB) is the whole
// cost, so the kernel is built to stream each weight from HBM exactly once.
//
// On the tensor cores, exactly.  A float32 embedding value x splits into three bf16 terms
// with x = hi + mid + lo exactly: hi = bf16(x); x - hi is exact in float32 and below half an
// ulp of bf16 at x's scale, so mid = bf16(x - hi) takes the next 8 significant bits, and
// (x - hi) - mid, exact again, has at most 6 significant bits left and is a bf16 value (lo).
// Each bf16 x bf16 product is exact in fp32, so three accumulating MMAs (W hi + W mid + W lo)
// with fp32 accumulation form sum_k W[j][k] x[k] with the products of the CUDA-core kernel
// this replaces and the same fp32 accumulation error class; the bias is added in fp32 and the
// sum rounded once to bf16.
//
// GEMM shape: the weight rows are the M dimension (128-row tiles, TMA, 128-byte swizzle), the
// timesteps the N dimension (T rounded up to a multiple of 16, at most 128 per pass; 80 for a
// 40-step run's 77), Dt the reduction.  One CTA per SM, persistent over the row tiles of up to
// MC_GROUP blocks per launch (their tensor maps travel as kernel parameters).  Two rings: the
// weight tiles stream from HBM through a deep ring (8 x 16 KB at N = 80, enough bytes in
// flight per SM to cover HBM latency under load), the split embedding tiles -- the same for
// every row tile -- through a short one:
//   warp 0      TMA producer of the weight tile (128 rows x 64 k) per step
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer (3 x 4 MMAs of M128 N K16)
//   warps 2..5  epilogue: tcgen05.ld, + bias, bf16, table[t][b][j] for every t < T
//   warps 6..13 split producers: temb[t][k] (float32, L2-resident) -> the hi / mid / lo bf16
//               tiles of the stage in the swizzled K-major layout the MMA reads; each stage's
//               values are loaded into registers three stages ahead of their use
// Two accumulators in TMEM let the epilogue of one tile overlap the mainloop of the next.
#include <cudaTypedefs.h>

#include "kernels.h"

namespace h3 {

constexpr int MC_BM = 128, MC_BK = 64, MC_NMAX = 128, MC_GROUP = 16;
constexpr int MC_SPLIT_WARPS = 8;
constexpr int MC_THREADS = 192 + 32 * MC_SPLIT_WARPS;
constexpr int MC_A_BYTES = MC_BM * MC_BK * 2;  // 16 KB
constexpr int MC_SMEM_CAP = 227 * 1024;
constexpr int MC_UNITS = MC_NMAX * 8 / (32 * MC_SPLIT_WARPS);  // 8-value units per split thread at N = 128

constexpr int MC_MAX_A_STAGES = 12, MC_B_STAGES = 3;

struct McParams {
  CUtensorMap w[MC_GROUP];      // weights of the group's blocks, bf16 [n_out, Dt]
  const bf16* bias[MC_GROUP];   // [n_out] or null
  const float* temb;            // [T, Dt], 16-byte aligned rows
  bf16* table;                  // first block of the group, t = 0
  long long t_stride;
  int T, t0, N;                 // timesteps, first of this pass, padded width of this pass
  int Dt, kb_count, n_out, row_tiles, num_tiles, stages_a, stages_b;
  unsigned* err;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__global__ void __launch_bounds__(MC_THREADS, 1) modcache_tc_kernel(const __grid_constant__ McParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int SA = p.stages_a, SB = p.stages_b, N = p.N;
  const int b_bytes = N * 128;                        // one split tile: N rows x 64 k bf16
  const int b_stage = 3 * b_bytes;                    // hi, mid, lo
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SA * MC_A_BYTES + SB * b_stage);
  const uint32_t bar_full = smem_u32(bars);           // SA: weight tile landed
  const uint32_t bar_aempty = bar_full + 8 * SA;      // SA: MMA done with the weight tile
  const uint32_t bar_ready = bar_aempty + 8 * SA;     // SB: split tiles written (split warps)
  const uint32_t bar_bempty = bar_ready + 8 * SB;     // SB: MMA done with the split tiles
  const uint32_t bar_tfull = bar_bempty + 8 * SB;     // 2: accumulator complete
  const uint32_t bar_tempty = bar_tfull + 16;         // 2: accumulator drained (4 warps)
  const uint32_t bar_drain = bar_tempty + 16;         // failure path: the issuer's MMAs completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * SA + 2 * SB + 5);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ErrCtx ec = err_ctx(p.err);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_aempty + 8 * s, 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(bar_ready + 8 * s, MC_SPLIT_WARPS);
      mbar_init(bar_bempty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, 4);
    }
    mbar_init(bar_drain, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 2 * MC_NMAX);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t a_base = smem_u32(smem);
  const uint32_t b_base = a_base + SA * MC_A_BYTES;

  if (warp == 0) {
    if (lane == 0) {
      for (int g = 0; g < p.num_tiles / p.row_tiles; ++g) tma_prefetch_desc(&p.w[g]);
      int s = 0, issued = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const int blk = tile / p.row_tiles, rt = tile % p.row_tiles;
        for (int kb = 0; kb < p.kb_count; ++kb, ++issued) {
          if (!mbar_wait(bar_aempty + 8 * s, ph ^ 1, ec, kErrModcacheProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_full + 8 * s, MC_A_BYTES);
          tma_load_2d(a_base + s * MC_A_BYTES, &p.w[blk], bar_full + 8 * s, kb * MC_BK, rt * MC_BM);
          if (++s == SA) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok)  // let the copies still in flight land before the shared memory is released
        for (int i = issued > SA ? issued - SA : 0; i < issued; ++i)
          mbar_drain(bar_full + 8 * (i % SA), (i / SA) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(MC_BM, N);
      int sa = 0, sb = 0, acc = 0;
      uint32_t pha = 0, phb = 0, aph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        if (!mbar_wait(bar_tempty + 8 * acc, aph ^ 1, ec, kErrModcacheMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + acc * MC_NMAX;
        for (int kb = 0; kb < p.kb_count; ++kb) {
          if (!mbar_wait(bar_full + 8 * sa, pha, ec, kErrModcacheMma) ||
              !mbar_wait(bar_ready + 8 * sb, phb, ec, kErrModcacheMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = a_base + sa * MC_A_BYTES, b0 = b_base + sb * b_stage;
#pragma unroll
          for (int kk = 0; kk < MC_BK / 16; ++kk)
#pragma unroll
            for (int sp = 0; sp < 3; ++sp)
              umma_bf16_ss(d, sdesc_k_sw128(a0 + 32 * kk), sdesc_k_sw128(b0 + sp * b_bytes + 32 * kk), idesc,
                           (kb | kk | sp) != 0);
          umma_commit(bar_aempty + 8 * sa);
          umma_commit(bar_bempty + 8 * sb);
          if (++sa == SA) {
            sa = 0;
            pha ^= 1;
          }
          if (++sb == SB) {
            sb = 0;
            phb ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(bar_tfull + 8 * acc);
        if (++acc == 2) {
          acc = 0;
          aph ^= 1;
        }
      }
      if (!ok) {  // the MMAs already issued finish before TMEM is released
        umma_commit(bar_drain);
        mbar_drain(bar_drain, 0);
      }
    }
  } else if (warp < 6) {
    // epilogue: this warp's 32 TMEM lanes are 32 weight rows; columns are timesteps t0 + c
    const int quad = warp & 3;
    int acc = 0;
    uint32_t aph = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      const int blk = tile / p.row_tiles, rt = tile % p.row_tiles;
      const int j = rt * MC_BM + quad * 32 + lane;
      const bool row_ok = j < p.n_out;
      const float bj = (row_ok && p.bias[blk]) ? bf2f(p.bias[blk][j]) : 0.f;
      bf16* dst = p.table + static_cast<long long>(blk) * p.n_out + j;
      if (!mbar_wait(bar_tfull + 8 * acc, aph, ec, kErrModcacheEpilogue)) break;
      tc_fence_after();
      const uint32_t t_acc = tmem + acc * MC_NMAX + (static_cast<uint32_t>(quad * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < N / 16; ++c) {
        uint32_t r[16];
        tmem_ld16(t_acc + c * 16, r);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int t = p.t0 + c * 16 + e;
            if (t < p.T) dst[static_cast<long long>(t) * p.t_stride] = f2bf(__uint_as_float(r[e]) + bj);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        aph ^= 1;
      }
    }
  } else {
    // split producers: thread u handles units u + 256 i, unit = (row t of the pass, 8-wide k
    // chunk c of the stage).  A stage's float32 values depend on its k-block only (they recur
    // for every row tile), and are loaded into one of three register slots three stages ahead
    // of their use; the loop is unrolled over the slots so no slot is ever copied.
    const int tid = threadIdx.x - 192;
    const int n_units = N * 8;  // (row, chunk) units of a stage, at most MC_UNITS per thread
    float v0[MC_UNITS][8], v1[MC_UNITS][8], v2[MC_UNITS][8];
    auto load = [&](float (&v)[MC_UNITS][8], int kb) {
#pragma unroll
      for (int i = 0; i < MC_UNITS; ++i) {
        const int u = tid + 32 * MC_SPLIT_WARPS * i, row = u >> 3, c = u & 7;
        if (u >= n_units) break;
        const int t = p.t0 + row, k = kb * MC_BK + 8 * c;
        if (t < p.T && k < p.Dt) {  // Dt % 8 == 0: a chunk is all in or all out
          const float4* src = reinterpret_cast<const float4*>(p.temb + static_cast<size_t>(t) * p.Dt + k);
          const float4 a = __ldg(src), b = __ldg(src + 1);
          v[i][0] = a.x, v[i][1] = a.y, v[i][2] = a.z, v[i][3] = a.w;
          v[i][4] = b.x, v[i][5] = b.y, v[i][6] = b.z, v[i][7] = b.w;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) v[i][e] = 0.f;
        }
      }
    };
    int s = 0, kb = 0, tile = blockIdx.x;
    uint32_t ph = 0;
    bool ok = tile < p.num_tiles;
    load(v0, 0);
    load(v1, 1 % p.kb_count);
    load(v2, 2 % p.kb_count);
    // one stage: wait until the MMA has released slot s, write the split of `v` into it, then
    // refill `v` with the values of the stage three ahead
    auto stage = [&](float (&v)[MC_UNITS][8]) {
      if (!ok) return;
      if (!mbar_wait(bar_bempty + 8 * s, ph ^ 1, ec, kErrModcacheSplit)) {
        ok = false;
        return;
      }
      const uint32_t b0 = b_base + s * b_stage;
#pragma unroll
      for (int i = 0; i < MC_UNITS; ++i) {
        const int u = tid + 32 * MC_SPLIT_WARPS * i, row = u >> 3, c = u & 7;
        if (u >= n_units) break;
        uint32_t hi[4], mi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = v[i][2 * e], x1 = v[i][2 * e + 1];
          const uint32_t h = pack_bf16x2(x0, x1);
          const float r0 = x0 - bf16lo(h), r1 = x1 - bf16hi(h);  // exact
          const uint32_t m = pack_bf16x2(r0, r1);
          const float q0 = r0 - bf16lo(m), q1 = r1 - bf16hi(m);  // exact, and a bf16 value
          hi[e] = h;
          mi[e] = m;
          lo[e] = pack_bf16x2(q0, q1);
        }
        const uint32_t off = row * 128 + ((c ^ (row & 7)) << 4);  // 128-byte swizzle
        st_shared_v4(b0 + off, hi[0], hi[1], hi[2], hi[3]);
        st_shared_v4(b0 + b_bytes + off, mi[0], mi[1], mi[2], mi[3]);
        st_shared_v4(b0 + 2 * b_bytes + off, lo[0], lo[1], lo[2], lo[3]);
      }
      fence_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ready + 8 * s);
      if (++s == SB) {
        s = 0;
        ph ^= 1;
      }
      load(v, (kb + 3) % p.kb_count);
      if (++kb == p.kb_count) {
        kb = 0;
        tile += gridDim.x;
        ok = tile < p.num_tiles;
      }
    };
    while (ok) {
      stage(v0);
      stage(v1);
      stage(v2);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * MC_NMAX);
  }
}

cudaError_t launch_modcache(const float* temb, int T, int Dt, const bf16* const* W, const bf16* const* bias,
                            int n_blocks, int n_out, bf16* table, long long t_stride, unsigned* err,
                            cudaStream_t st) {
  if (T <= 0 || n_out <= 0 || n_blocks <= 0) return cudaSuccess;
  if (Dt <= 0 || Dt % 8 || (reinterpret_cast<uintptr_t>(temb) & 15)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(modcache_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MC_SMEM_CAP);
  if (e != cudaSuccess) return e;
  const int row_tiles = cdiv(n_out, MC_BM);
  const int groups = cdiv(n_blocks, MC_GROUP);
  const int per_group = cdiv(n_blocks, groups);  // balanced groups of <= MC_GROUP blocks
  for (int t0 = 0; t0 < T; t0 += MC_NMAX) {
    const int N = cdiv(T - t0 < MC_NMAX ? T - t0 : MC_NMAX, 16) * 16;
    const int b_stage = 3 * N * 128;
    int stages_a = (MC_SMEM_CAP - 1024 - 512 - MC_B_STAGES * b_stage) / MC_A_BYTES;
    stages_a = stages_a > MC_MAX_A_STAGES ? MC_MAX_A_STAGES : stages_a;  // >= 5 for N <= 128
    const int smem = 1024 + stages_a * MC_A_BYTES + MC_B_STAGES * b_stage + 512;
    for (int b0 = 0; b0 < n_blocks; b0 += per_group) {
      const int nb = n_blocks - b0 < per_group ? n_blocks - b0 : per_group;
      McParams p{};
      for (int i = 0; i < nb; ++i) {
        if (!W[b0 + i]) return cudaErrorInvalidValue;
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(Dt), static_cast<cuuint64_t>(n_out)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(Dt) * 2};
        cuuint32_t box[2] = {MC_BK, MC_BM};
        cuuint32_t estr[2] = {1, 1};
        if (tensor_map_encode_tiled(&p.w[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<bf16*>(W[b0 + i]), dims,
                                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
          return cudaErrorInvalidValue;
        p.bias[i] = bias ? bias[b0 + i] : nullptr;
      }
      p.temb = temb;
      p.table = table + static_cast<long long>(b0) * n_out;
      p.t_stride = t_stride;
      p.T = T;
      p.t0 = t0;
      p.N = N;
      p.Dt = Dt;
      p.kb_count = cdiv(Dt, MC_BK);
      p.n_out = n_out;
      p.row_tiles = row_tiles;
      p.num_tiles = row_tiles * nb;
      p.stages_a = stages_a;
      p.stages_b = MC_B_STAGES;
      p.err = err;
      const int grid = p.num_tiles < num_sms() ? p.num_tiles : num_sms();
      modcache_tc_kernel<<<grid, MC_THREADS, smem, st>>>(p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace h3
