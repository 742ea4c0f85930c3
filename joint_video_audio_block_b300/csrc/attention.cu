// a4: full unmasked self-attention over the packed sequence, FlashAttention-style, on tcgen05.
//
// "minimax-h3-mlx" README, "Architecture": attention is full self-attention over the whole
// packed sequence (no cross-attention, no mask); "Performance": it is flash-style (the score
// matrix is never materialised) and dominates the work at realistic lengths.
//
// One CTA = one head x 128 query rows.  Roles:
//   warp 0      TMA producer: Q once, then K and V^T tiles of 128 keys (2-stage ring)
//   warp 1      TMEM allocator + single-thread MMA issuer:
//                 S_j  = Q K_j^T        -> TMEM (two 128-column buffers, so S_{j+1} runs
//                                          while the softmax reads S_j)
//                 O   += P_j V_j        -> TMEM (128 columns), A = P from shared memory,
//                                          B = V^T tile (keys contiguous: K-major)
//   warps 2..5  softmax: one thread per query row (its TMEM lane), online max / sum in fp32,
//               P rounded to bf16 into the 128-byte-swizzled A-operand layout; O is rescaled
//               in TMEM only when the running max grew by more than 2^8 (the stale max keeps
//               every exponent <= 2^8, and l and O share it, so the result is unchanged).
// Keys beyond n_rows in the last tile get a score of -inf (TMA fills them with zeros).
#include <cudaTypedefs.h>

#include "kernels.h"

namespace h3 {

constexpr int AT_BM = 128, AT_BN = 128;
constexpr int AT_ATOM = 128 * 128;            // one 128-row x 128-byte swizzle atom
constexpr int AT_THREADS = 192;
constexpr float AT_RESCALE_THRESHOLD = 8.0f;  // log2 units

// Shared-memory plan for head_dim HD: Q and K tiles are 128 rows x HD (HD/64 atoms along d),
// V^T tiles are HD rows x 128 keys (2 atoms along keys, HD*128 bytes each), P is 128 x 128.
template <int HD>
struct AtCfg {
  static constexpr int QK_TILE = 128 * HD * 2;
  static constexpr int V_ATOM = HD * 128;
  static constexpr int V_TILE = 2 * V_ATOM;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = QK_TILE;               // 2 stages
  static constexpr int V_OFF = K_OFF + 2 * QK_TILE;   // 2 stages
  static constexpr int P_OFF = V_OFF + 2 * V_TILE;
  static constexpr int BAR_OFF = P_OFF + 2 * AT_ATOM;
  static constexpr int SMEM = BAR_OFF + 256 + 1024;
};

template <int HD>
__global__ void __launch_bounds__(AT_THREADS, 1)
    attention_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, bf16* __restrict__ o, int n_rows, int nh,
                        float scale_log2, unsigned* err) {
  using C = AtCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  const uint32_t b_q = smem_u32(bars);
  const uint32_t b_kfull = b_q + 8;        // [2]
  const uint32_t b_vfull = b_kfull + 16;   // [2]
  const uint32_t b_kvempty = b_vfull + 16; // [2]
  const uint32_t b_sfull = b_kvempty + 16; // [2]
  const uint32_t b_pfull = b_sfull + 16;
  const uint32_t b_odone = b_pfull + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int q0 = blockIdx.x * AT_BM;
  const int nt = cdiv(n_rows, AT_BN);

  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(b_kfull + 8 * s, 1);
      mbar_init(b_vfull + 8 * s, 1);
      mbar_init(b_kvempty + 8 * s, 1);
      mbar_init(b_sfull + 8 * s, 1);
    }
    mbar_init(b_pfull, 4);
    mbar_init(b_odone, 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s0 = tmem, t_o = tmem + 256;

  const uint32_t sQ = smem_u32(smem + C::Q_OFF);
  const uint32_t sK = smem_u32(smem + C::K_OFF);
  const uint32_t sV = smem_u32(smem + C::V_OFF);
  const uint32_t sP = smem_u32(smem + C::P_OFF);

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(b_q, C::QK_TILE);
      for (int a = 0; a < HD / 64; ++a) tma_load_3d(sQ + a * AT_ATOM, &tmQ, b_q, 64 * a, q0, h);
      for (int j = 0; j < nt; ++j) {
        const int s = j & 1;
        if (!mbar_wait(b_kvempty + 8 * s, ((j >> 1) & 1) ^ 1, err, kErrAttnProducer)) break;
        const uint32_t kd = sK + s * C::QK_TILE, vd = sV + s * C::V_TILE;
        mbar_arrive_expect_tx(b_kfull + 8 * s, C::QK_TILE);
        for (int a = 0; a < HD / 64; ++a) tma_load_3d(kd + a * AT_ATOM, &tmK, b_kfull + 8 * s, 64 * a, j * AT_BN, h);
        mbar_arrive_expect_tx(b_vfull + 8 * s, C::V_TILE);
        tma_load_3d(vd, &tmV, b_vfull + 8 * s, j * AT_BN, 0, h);
        tma_load_3d(vd + C::V_ATOM, &tmV, b_vfull + 8 * s, j * AT_BN + 64, 0, h);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, HD);
      bool ok = mbar_wait(b_q, 0, err, kErrAttnMma);
      // S_0
      if (ok) ok = mbar_wait(b_kfull, 0, err, kErrAttnMma);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * AT_ATOM + (kk & 3) * 32;
          umma_bf16_ss(t_s0, sdesc_k_sw128(sQ + off), sdesc_k_sw128(sK + off), idesc_s, kk != 0);
        }
        umma_commit(b_sfull);
      }
      for (int j = 0; ok && j < nt; ++j) {
        const int s = j & 1;
        if (j + 1 < nt) {
          const int s1 = (j + 1) & 1;
          if (!mbar_wait(b_kfull + 8 * s1, ((j + 1) >> 1) & 1, err, kErrAttnMma)) break;
          tc_fence_after();
          const uint32_t kb = sK + s1 * C::QK_TILE;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * AT_ATOM + (kk & 3) * 32;
            umma_bf16_ss(t_s0 + s1 * 128, sdesc_k_sw128(sQ + off), sdesc_k_sw128(kb + off), idesc_s, kk != 0);
          }
          umma_commit(b_sfull + 8 * s1);
        }
        if (!mbar_wait(b_pfull, j & 1, err, kErrAttnMma)) break;
        if (!mbar_wait(b_vfull + 8 * s, (j >> 1) & 1, err, kErrAttnMma)) break;
        tc_fence_after();
        const uint32_t vb = sV + s * C::V_TILE;
#pragma unroll
        for (int kk = 0; kk < AT_BN / 16; ++kk) {
          const uint32_t inner = (kk & 3) * 32;
          umma_bf16_ss(t_o, sdesc_k_sw128(sP + (kk >> 2) * AT_ATOM + inner),
                       sdesc_k_sw128(vb + (kk >> 2) * C::V_ATOM + inner), idesc_o, (j | kk) != 0);
        }
        umma_commit(b_kvempty + 8 * s);
        umma_commit(b_odone);
      }
    }
  } else {
    // softmax warps 2..5: TMEM lane quadrant = warp % 4, one query row per thread
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    uint8_t* prow = smem + C::P_OFF + r * 128;
    for (int j = 0; j < nt; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(b_sfull + 8 * sb, (j >> 1) & 1, err, kErrAttnSoftmax)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t u[32];
        tmem_ld32(t_s0 + sb * 128 + lane_off + c * 32, u);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[c * 32 + i] = __uint_as_float(u[i]) * scale_log2;
      }
      const int valid = n_rows - j * AT_BN;  // keys of this tile that exist
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        if (i >= valid) sv[i] = -INFINITY;
        mt = fmaxf(mt, sv[i]);
      }
      float alpha = 1.f;
      bool rescale = false;
      if (j == 0) {
        m_used = mt;
      } else if (mt > m_used + AT_RESCALE_THRESHOLD) {
        alpha = exp2f(m_used - mt);
        m_used = mt;
        rescale = true;
      }
      float rs = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float p0 = exp2f(sv[2 * i] - m_used);
        const float p1 = exp2f(sv[2 * i + 1] - m_used);
        rs += p0 + p1;
        pk[i] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + rs;
      // PV_{j-1} must be complete before P is overwritten and O is touched
      if (j > 0 && !mbar_wait(b_odone, (j - 1) & 1, err, kErrAttnSoftmax)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t u[32];
          tmem_ld32(t_o + lane_off + c * 32, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
          tmem_st32(t_o + lane_off + c * 32, u);
        }
        tmem_wait_st();
      }
      // P row -> two swizzle atoms (keys 0..63, 64..127); 16-byte chunk c at c ^ (r & 7)
#pragma unroll
      for (int a = 0; a < 2; ++a) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int w0 = a * 32 + c * 4;
          *reinterpret_cast<int4*>(prow + a * AT_ATOM + ((c ^ (r & 7)) << 4)) =
              make_int4(pk[w0], pk[w0 + 1], pk[w0 + 2], pk[w0 + 3]);
        }
      }
      fence_async_shared();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_pfull);
    }
    if (ok && mbar_wait(b_odone, (nt - 1) & 1, err, kErrAttnSoftmax)) {
      tc_fence_after();
      const int row = q0 + r;
      const float inv = 1.f / l;
      bf16* dst = o + static_cast<size_t>(row) * nh * HD + h * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(t_o + lane_off + c * 32, u);
        tmem_wait_ld();
        if (row < n_rows) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(u[8 * q + 2 * e]) * inv, __uint_as_float(u[8 * q + 2 * e + 1]) * inv);
            reinterpret_cast<int4*>(dst + c * 32)[q] = make_int4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

static bool encode_3d(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
                      uint64_t s2_bytes, uint32_t b0, uint32_t b1) {
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return tensor_map_encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int HD>
static cudaError_t launch_at(const bf16* q, const bf16* k, const bf16* vt, int ld_vt, bf16* o, int n_rows, int nh,
                             unsigned* err, cudaStream_t st) {
  using C = AtCfg<HD>;
  CUtensorMap tq, tk, tv;
  const uint64_t rs = static_cast<uint64_t>(HD) * 2;
  if (!encode_3d(&tq, q, HD, n_rows, nh, rs, rs * n_rows, 64, AT_BM)) return cudaErrorInvalidValue;
  if (!encode_3d(&tk, k, HD, n_rows, nh, rs, rs * n_rows, 64, AT_BN)) return cudaErrorInvalidValue;
  if (!encode_3d(&tv, vt, n_rows, HD, nh, static_cast<uint64_t>(ld_vt) * 2, static_cast<uint64_t>(ld_vt) * 2 * HD, 64,
                 HD))
    return cudaErrorInvalidValue;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  dim3 grid(cdiv(n_rows, AT_BM), nh);
  attention_tc_kernel<HD><<<grid, AT_THREADS, C::SMEM, st>>>(tq, tk, tv, o, n_rows, nh, scale_log2, err);
  return cudaGetLastError();
}

cudaError_t launch_attention_tc(const bf16* q, const bf16* k, const bf16* vt, int ld_vt, bf16* o, int n_rows, int nh,
                                int hd, unsigned* err, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  if (hd == 128) return launch_at<128>(q, k, vt, ld_vt, o, n_rows, nh, err, st);
  if (hd == 64) return launch_at<64>(q, k, vt, ld_vt, o, n_rows, nh, err, st);
  return cudaErrorInvalidValue;
}

}  // namespace h3
