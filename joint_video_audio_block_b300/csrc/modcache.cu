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
// Each bf16 x bf16 product is exact in fp32.  The three tiles sit one after another in shared
// memory, so one MMA of N = 3 x (padded T) multiplies the weight tile by all of them: its
// accumulator holds W.hi, W.mid and W.lo as three column groups, each an exact-product fp32
// dot product, and the epilogue forms (W.hi + W.mid) + W.lo + bias in fp32 and rounds once to
// bf16 -- the products of a float32 CUDA-core dot product and the same fp32 error class.  One
// wide MMA instead of three narrow ones keeps a single issuing thread ahead of the tensor pipe.
//
// GEMM shape: the weight rows are the M dimension (256-row tiles: two 128-row MMAs per k-step
// share each split tile, TMA, 128-byte swizzle), the timesteps the N dimension (T rounded up to
// a multiple of 16, at most 80 per pass, so that 3 x 80 fits one MMA; a 40-step run's 77
// timesteps are one pass), Dt the reduction, 64 k per step.  One CTA per SM, persistent over
// the row tiles of up to MC_GROUP blocks per launch (their tensor maps travel as kernel
// parameters).  Three rings of shared memory:
//   weights   W tile, 256 rows x 64 k bf16 (TMA from HBM), 3+ slots -- the stream that sets
//             the kernel's speed;
//   embedding temb tile, N rows x 64 k float32 (TMA from L2), 3 slots;
//   split     the hi / mid / lo bf16 tiles of the step, N rows x 64 k each, back to back in the
//             swizzled K-major layout the MMA reads, 2 slots.
// The embedding reaches the split warps through shared memory, not through loads into their
// registers: the proxy fence a split warp issues before releasing its tiles to the tensor core
// then has no global load of its own to wait for.  The embedding and split work per weight
// byte is what limits this kernel (measured: with it removed, the same pipeline streams the
// weights at the HBM copy rate), hence the 256-row tiles that halve it and the three
// embedding slots that cover the L2 latency of its loads.
//   warp 0      TMA producer: the weight tile and the embedding tile of each step
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer (2 x 4 MMAs of M128 N3N K16
//               per step)
//   warps 2..5  epilogue: tcgen05.ld, + bias, bf16, table[t][b][j] for every t < T
//   warps 6..13 split producers: embedding tile -> hi / mid / lo tiles
// The two 128-row accumulators fill TMEM; each is released as soon as the epilogue has read
// it, so the next tile's first MMAs into the first overlap the epilogue of the second.
#include <cudaTypedefs.h>

#include "kernels.h"

namespace h3 {

constexpr int MC_BM = 256, MC_BK = 64, MC_NMAX = 80, MC_GROUP = 16;
constexpr int MC_ACC_COLS = 256;  // one 128-row accumulator: 3 x N <= 240 columns
constexpr int MC_SPLIT_WARPS = 8;
constexpr int MC_THREADS = 192 + 32 * MC_SPLIT_WARPS;
constexpr int MC_A_BYTES = MC_BM * MC_BK * 2;  // 32 KB: two 128-row halves of 16 KB
constexpr int MC_SMEM_CAP = 227 * 1024;
constexpr int MC_MAX_A_STAGES = 8, MC_T_STAGES = 3, MC_B_STAGES = 2;
constexpr int MC_UNITS = (MC_NMAX * 8 + 32 * MC_SPLIT_WARPS - 1) / (32 * MC_SPLIT_WARPS);  // 8-value units per split thread

struct McParams {
  CUtensorMap w[MC_GROUP];      // weights of the group's blocks, bf16 [n_out, Dt]
  CUtensorMap temb;             // float32 [T, Dt], box 64 k x N rows
  const bf16* bias[MC_GROUP];   // [n_out] or null
  bf16* table;                  // first block of the group, t = 0
  long long t_stride;
  int T, t0, N;                 // timesteps, first of this pass, padded width of this pass
  int Dt, kb_count, n_out, row_tiles, num_tiles, stages_a;
  unsigned* err;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
               : "memory");
  return v;
}

__global__ void __launch_bounds__(MC_THREADS, 1) modcache_tc_kernel(const __grid_constant__ McParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int SA = p.stages_a, SB = MC_B_STAGES, ST = MC_T_STAGES, N = p.N;
  const int t_bytes = N * MC_BK * 4;                  // one embedding tile: N rows x 64 k float32
  const int b_bytes = N * 128;                        // one split tile: N rows x 64 k bf16
  const int b_stage = 3 * b_bytes;                    // hi, mid, lo
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SA * MC_A_BYTES + ST * t_bytes + SB * b_stage);
  const uint32_t bar_afull = smem_u32(bars);          // SA: weight tile landed
  const uint32_t bar_aempty = bar_afull + 8 * SA;     // SA: MMA done with the weight tile
  const uint32_t bar_tfull = bar_aempty + 8 * SA;     // ST: embedding tile landed
  const uint32_t bar_tempty = bar_tfull + 8 * ST;     // ST: split warps done reading it
  const uint32_t bar_ready = bar_tempty + 8 * ST;     // SB: split tiles written (split warps)
  const uint32_t bar_bempty = bar_ready + 8 * SB;     // SB: MMA done with the split tiles
  const uint32_t bar_accfull = bar_bempty + 8 * SB;   // the tile's accumulators complete
  const uint32_t bar_accempty = bar_accfull + 8;      // 2: accumulator h (rows 128h..) read (4 warps)
  const uint32_t bar_drain = bar_accempty + 16;       // failure path: the issuer's MMAs completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * SA + 2 * ST + 2 * SB + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ErrCtx ec = err_ctx(p.err);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(bar_afull + 8 * s, 1);
      mbar_init(bar_aempty + 8 * s, 1);
    }
    for (int s = 0; s < ST; ++s) {
      mbar_init(bar_tfull + 8 * s, 1);
      mbar_init(bar_tempty + 8 * s, MC_SPLIT_WARPS);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(bar_ready + 8 * s, MC_SPLIT_WARPS);
      mbar_init(bar_bempty + 8 * s, 1);
    }
    mbar_init(bar_accfull, 1);
    for (int a = 0; a < 2; ++a) mbar_init(bar_accempty + 8 * a, 4);
    mbar_init(bar_drain, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 2 * MC_ACC_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t a_base = smem_u32(smem);
  const uint32_t t_base = a_base + SA * MC_A_BYTES;
  const uint32_t b_base = t_base + ST * t_bytes;

  if (warp == 0) {
    if (lane == 0) {
      for (int g = 0; g < p.num_tiles / p.row_tiles; ++g) tma_prefetch_desc(&p.w[g]);
      tma_prefetch_desc(&p.temb);
      int sa = 0, st = 0, issued = 0;
      uint32_t pha = 0, pht = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const int blk = tile / p.row_tiles, rt = tile % p.row_tiles;
        for (int kb = 0; kb < p.kb_count; ++kb, ++issued) {
          if (!mbar_wait(bar_aempty + 8 * sa, pha ^ 1, ec, kErrModcacheProducer) ||
              !mbar_wait(bar_tempty + 8 * st, pht ^ 1, ec, kErrModcacheProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_afull + 8 * sa, MC_A_BYTES);
          tma_load_2d(a_base + sa * MC_A_BYTES, &p.w[blk], bar_afull + 8 * sa, kb * MC_BK, rt * MC_BM);  // 256 rows
          mbar_arrive_expect_tx(bar_tfull + 8 * st, t_bytes);
          tma_load_2d(t_base + st * t_bytes, &p.temb, bar_tfull + 8 * st, kb * MC_BK, p.t0);
          if (++sa == SA) {
            sa = 0;
            pha ^= 1;
          }
          if (++st == ST) {
            st = 0;
            pht ^= 1;
          }
        }
      }
      if (!ok) {  // let the copies still in flight land before the shared memory is released
        for (int i = issued > SA ? issued - SA : 0; i < issued; ++i)
          mbar_drain(bar_afull + 8 * (i % SA), (i / SA) & 1);
        for (int i = issued > ST ? issued - ST : 0; i < issued; ++i)
          mbar_drain(bar_tfull + 8 * (i % ST), (i / ST) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 3 * N);
      int sa = 0, sb = 0;
      uint32_t pha = 0, phb = 0, aph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, aph ^= 1) {
        for (int kb = 0; kb < p.kb_count; ++kb) {
          if (!mbar_wait(bar_afull + 8 * sa, pha, ec, kErrModcacheMma) ||
              !mbar_wait(bar_ready + 8 * sb, phb, ec, kErrModcacheMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = a_base + sa * MC_A_BYTES, b0 = b_base + sb * b_stage;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // the first k-step of a tile writes accumulator h afresh: the epilogue must have
            // read the previous tile's
            if (kb == 0) {
              if (!mbar_wait(bar_accempty + 8 * h, aph ^ 1, ec, kErrModcacheMma)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
#pragma unroll
            for (int kk = 0; kk < MC_BK / 16; ++kk)  // B: the hi, mid, lo tiles as one 3N-row operand
              umma_bf16_ss(tmem + h * MC_ACC_COLS, sdesc_k_sw128(a0 + h * (MC_A_BYTES / 2) + 32 * kk),
                           sdesc_k_sw128(b0 + 32 * kk), idesc, (kb | kk) != 0);
          }
          if (!ok) break;
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
        umma_commit(bar_accfull);
      }
      if (!ok) {  // the MMAs already issued finish before TMEM is released
        umma_commit(bar_drain);
        mbar_drain(bar_drain, 0);
      }
    }
  } else if (warp < 6) {
    // epilogue: this warp's 32 TMEM lanes are 32 weight rows of each 128-row half; columns are
    // timesteps t0 + c in three groups (W.hi, W.mid, W.lo).  A half is read out of TMEM and
    // rounded to bf16 in registers, released to the MMA issuer, and only then stored, so the
    // next tile's MMAs wait for the TMEM reads alone, not for the table stores.
    const int quad = warp & 3;
    uint32_t aph = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, aph ^= 1) {
      const int blk = tile / p.row_tiles, rt = tile % p.row_tiles;
      if (!mbar_wait(bar_accfull, aph, ec, kErrModcacheEpilogue)) break;
      tc_fence_after();
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        const int j = rt * MC_BM + h * 128 + quad * 32 + lane;
        const bool row_ok = j < p.n_out;
        const float bj = (row_ok && p.bias[blk]) ? bf2f(p.bias[blk][j]) : 0.f;
        const uint32_t t_acc = tmem + h * MC_ACC_COLS + (static_cast<uint32_t>(quad * 32) << 16);
        uint32_t out[MC_NMAX / 2];  // bf16 pairs (t, t + 1) of this row
#pragma unroll
        for (int c = 0; c < MC_NMAX / 16; ++c) {
          if (c < N / 16) {
            uint32_t rh[16], rm[16], rl[16];
            tmem_ld16(t_acc + c * 16, rh);
            tmem_ld16(t_acc + N + c * 16, rm);
            tmem_ld16(t_acc + 2 * N + c * 16, rl);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const float v0 = (__uint_as_float(rh[e]) + __uint_as_float(rm[e])) + __uint_as_float(rl[e]);
              const float v1 = (__uint_as_float(rh[e + 1]) + __uint_as_float(rm[e + 1])) + __uint_as_float(rl[e + 1]);
              out[c * 8 + e / 2] = pack_bf16x2(v0 + bj, v1 + bj);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_accempty + 8 * h);
        if (row_ok) {
          bf16* dst = p.table + static_cast<long long>(blk) * p.n_out + j;
#pragma unroll
          for (int c = 0; c < MC_NMAX / 16; ++c)
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int t = p.t0 + c * 16 + e;
              if (c < N / 16 && t < p.T) {
                const uint32_t pr = out[c * 8 + e / 2];
                dst[static_cast<long long>(t) * p.t_stride] =
                    __ushort_as_bfloat16(static_cast<unsigned short>((e & 1) ? (pr >> 16) : (pr & 0xffffu)));
              }
            }
        }
      }
    }
  } else {
    // split producers: thread u handles units u + 256 i, unit = (row of the pass, 8-wide k chunk
    // c of the step).  Rows past T and k past Dt arrive as zeros (TMA fill).
    const int tid = threadIdx.x - 192;
    const int n_units = N * 8;
    int st = 0, sb = 0;
    uint32_t pht = 0, phb = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      for (int kb = 0; kb < p.kb_count; ++kb) {
        if (!mbar_wait(bar_tfull + 8 * st, pht, ec, kErrModcacheSplit) ||
            !mbar_wait(bar_bempty + 8 * sb, phb ^ 1, ec, kErrModcacheSplit)) {
          ok = false;
          break;
        }
        const uint32_t t0 = t_base + st * t_bytes, b0 = b_base + sb * b_stage;
#pragma unroll
        for (int i = 0; i < MC_UNITS; ++i) {
          const int u = tid + 32 * MC_SPLIT_WARPS * i, row = u >> 3, c = u & 7;
          if (u >= n_units) break;
          const float4 xa = ld_shared_f4(t0 + row * (MC_BK * 4) + c * 32);
          const float4 xb = ld_shared_f4(t0 + row * (MC_BK * 4) + c * 32 + 16);
          const float x[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
          uint32_t hi[4], mi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = x[2 * e], x1 = x[2 * e + 1];
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
        if (lane == 0) {
          mbar_arrive(bar_ready + 8 * sb);
          mbar_arrive(bar_tempty + 8 * st);
        }
        if (++st == ST) {
          st = 0;
          pht ^= 1;
        }
        if (++sb == SB) {
          sb = 0;
          phb ^= 1;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * MC_ACC_COLS);
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
  const cuuint32_t estr[2] = {1, 1};
  for (int t0 = 0; t0 < T; t0 += MC_NMAX) {
    const int N = cdiv(T - t0 < MC_NMAX ? T - t0 : MC_NMAX, 16) * 16;
    const int t_bytes = N * MC_BK * 4, b_stage = 3 * N * 128;
    int stages_a = (MC_SMEM_CAP - 1024 - 512 - MC_T_STAGES * t_bytes - MC_B_STAGES * b_stage) / MC_A_BYTES;
    stages_a = stages_a > MC_MAX_A_STAGES ? MC_MAX_A_STAGES : stages_a;  // >= 3 for N <= 80
    const int smem = 1024 + stages_a * MC_A_BYTES + MC_T_STAGES * t_bytes + MC_B_STAGES * b_stage + 512;
    McParams p{};
    {
      const cuuint64_t dims[2] = {static_cast<cuuint64_t>(Dt), static_cast<cuuint64_t>(T)};
      const cuuint64_t strides[1] = {static_cast<cuuint64_t>(Dt) * 4};
      const cuuint32_t box[2] = {MC_BK, static_cast<cuuint32_t>(N)};
      if (tensor_map_encode_tiled(&p.temb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(temb), dims, strides,
                                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    for (int b0 = 0; b0 < n_blocks; b0 += per_group) {
      const int nb = n_blocks - b0 < per_group ? n_blocks - b0 : per_group;
      for (int i = 0; i < nb; ++i) {
        if (!W[b0 + i]) return cudaErrorInvalidValue;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(Dt), static_cast<cuuint64_t>(n_out)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(Dt) * 2};
        const cuuint32_t box[2] = {MC_BK, MC_BM};
        if (tensor_map_encode_tiled(&p.w[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<bf16*>(W[b0 + i]), dims,
                                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
          return cudaErrorInvalidValue;
        p.bias[i] = bias ? bias[b0 + i] : nullptr;
      }
      for (int i = nb; i < MC_GROUP; ++i) p.bias[i] = nullptr;
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
      p.err = err;
      const int grid = p.num_tiles < num_sms() ? p.num_tiles : num_sms();
      modcache_tc_kernel<<<grid, MC_THREADS, smem, st>>>(p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace h3
