// a4: full unmasked self-attention over the packed sequence, FlashAttention-style, on tcgen05.
//
// "minimax-h3-mlx" README, "Architecture": attention is full self-attention over the whole
// packed sequence (no cross-attention, no mask); "Performance": it is flash-style (the score
// matrix is never materialised) and dominates the work at realistic lengths.
//
// One CTA = one head x two 128-row query tiles (A and B) that share every K/V tile, so the
// tensor core always has the other tile's work while one tile's softmax runs:
//   warp 0       TMA producer: Q_A, Q_B once, then K_j and V_j^T tiles of 128 keys (ring)
//   warp 1       TMEM allocator + single-thread MMA issuer, per key tile j:
//                  O_A += P_A(j) V_j   (A operand P from TMEM)      S_A(j+1) = Q_A K_{j+1}^T
//                  O_B += P_B(j) V_j                                S_B(j+1) = Q_B K_{j+1}^T
//                each a run of 8 MMAs issued as one asm block; the issuer shares its
//                sub-partition with two softmax warps, so its own instruction count shows in
//                the kernel's time
//   warps 4..7   softmax of tile A, warps 8..11 softmax of tile B: one thread per query row
//                (its TMEM lane); the row of S is read with tcgen05.ld, the online max / sum
//                kept in fp32, and P rounded to bf16 written back over the front half of the
//                same S columns with tcgen05.st, where the P.V MMA reads it.
// TMEM (512 columns): S_A 0..127, S_B 128..255, O_A 256.., O_B 256+HD.. (fp32).  tcgen05.mma
// from one thread complete in issue order, so S_X(j+1) (issued after PV_X(j)) may overwrite
// P_X(j), and the completion of S_X(j+1) also means PV_X(j) is done: the softmax may then
// rescale O_X in TMEM before releasing P_X(j+1).  O is rescaled only when the running max grew
// by more than 2^8 (the stale max bounds every exponent by 2^8 and l and O share it, so the
// normalised result is unchanged).  Keys beyond n_rows in the last tile get a score of -inf
// (TMA fills them with zeros).
#include <cudaTypedefs.h>

#include "kernels.h"

namespace h3 {

constexpr int AT_BM = 128, AT_BN = 128;
constexpr int AT_ATOM = 128 * 128;            // one 128-row x 128-byte swizzle atom
constexpr int AT_THREADS = 384;
// Register split (setmaxnreg): the kernel launches at AT_LAUNCH_REGS per thread (checked on the
// host before every launch); warps 0..3 then give back down to AT_REGS_CTRL and the eight
// softmax warps take AT_REGS_SOFTMAX.  128 * 72 + 256 * 216 = 384 * 168, so the increase is
// always covered by the block's own launch allocation.
constexpr int AT_LAUNCH_REGS = 168, AT_REGS_CTRL = 72, AT_REGS_SOFTMAX = 216;
static_assert(128 * AT_REGS_CTRL + 256 * AT_REGS_SOFTMAX <= AT_THREADS * AT_LAUNCH_REGS, "register split");
constexpr float AT_RESCALE_THRESHOLD = 8.0f;  // log2 units

// Shared-memory plan for head_dim HD: each Q and K tile is 128 rows x HD (HD/64 atoms along
// d); each V^T tile is HD rows x 128 keys (2 atoms along keys, HD*128 bytes each).
template <int HD>
struct AtCfg {
  static constexpr int STAGES = HD == 64 ? 4 : 2;
  static constexpr int QK_TILE = 128 * HD * 2;
  static constexpr int V_ATOM = HD * 128;
  static constexpr int V_TILE = 2 * V_ATOM;
  static constexpr int Q_OFF = 0;                         // Q_A, Q_B
  static constexpr int K_OFF = 2 * QK_TILE;               // STAGES
  static constexpr int V_OFF = K_OFF + STAGES * QK_TILE;  // STAGES
  static constexpr int BAR_OFF = V_OFF + STAGES * V_TILE;
  static constexpr int SMEM = BAR_OFF + 256 + 1024;
};

// softmax arithmetic helpers: 3-input max, the SFU base-2 exponential (flushes results below
// 2^-126 to zero, which only drops probabilities that bf16 P cannot carry anyway), and
// paired fp32 FMA / add on two lanes of a 64-bit register
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint64_t pack_u32x2(uint32_t lo, uint32_t hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
  return d;
}
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  return pack_u32x2(__float_as_uint(lo), __float_as_uint(hi));
}
__device__ __forceinline__ float lo_f32(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi_f32(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// The 128-byte-swizzled K-major shared-memory descriptor split in two 32-bit words: the low
// word carries the start address (16-byte units) and the unused leading offset, the high word
// the 1024-byte stride, the descriptor version and the swizzle mode, and is the same for every
// operand here.  The issuer keeps only low words and steps them by each k slice's offset.
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr) { return ((saddr & 0x3FFFFu) >> 4) | (1u << 16); }
constexpr uint32_t AT_SDESC_HI = (1024u >> 4) | (1u << 14) | (2u << 29);

// A run of MMAs over consecutive 16-wide k slices of one tile pair, in one asm block: one
// predicate for the first MMA (accumulate or overwrite), the rest accumulate; slice i steps the
// descriptors' low words by O_i (16-byte units, compile-time).  SS: A and B in shared memory,
// with the same offsets (Q and K tiles share their layout).  TS: A (P) in TMEM, 8 columns per
// slice, B (V^T) in shared memory.
#define AT_SS_STEP(o)                                                                      \
  "add.u32 ra, %1, " #o ";\n\tadd.u32 rb, %2, " #o ";\n\t"                               \
  "mov.b64 da, {ra, %5};\n\tmov.b64 db, {rb, %5};\n\t"                                  \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, pt;\n\t"
#define AT_TS_STEP(ta, o)                                                                  \
  "add.u32 ra, %1, " #ta ";\n\tadd.u32 rb, %2, " #o ";\n\t"                              \
  "mov.b64 db, {rb, %5};\n\t"                                                            \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], db, %3, pt;\n\t"
#define AT_RUN_HEAD                                                                        \
  "{\n\t.reg .pred p, pt;\n\t.reg .b32 ra, rb;\n\t.reg .b64 da, db;\n\t"                 \
  "setp.ne.u32 p, %4, 0;\n\tsetp.eq.u32 pt, %4, %4;\n\t"

// S = Q K^T over head_dim 128 (8 slices; the second four in the next 64-column swizzle atom)
__device__ __forceinline__ void umma_ss_run8(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(AT_RUN_HEAD
               "mov.b64 da, {%1, %5};\n\tmov.b64 db, {%2, %5};\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n\t"
               AT_SS_STEP(2) AT_SS_STEP(4) AT_SS_STEP(6) AT_SS_STEP(1024) AT_SS_STEP(1026) AT_SS_STEP(1028)
               AT_SS_STEP(1030) "}"
               ::"r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(AT_SDESC_HI)
               : "memory");
}
// S = Q K^T over head_dim 64 (4 slices)
__device__ __forceinline__ void umma_ss_run4(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(AT_RUN_HEAD
               "mov.b64 da, {%1, %5};\n\tmov.b64 db, {%2, %5};\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n\t"
               AT_SS_STEP(2) AT_SS_STEP(4) AT_SS_STEP(6) "}"
               ::"r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(AT_SDESC_HI)
               : "memory");
}
// O += P V over 128 keys (8 slices); the V^T tile's second 64-key atom starts VA units on
template <int VA>
__device__ __forceinline__ void umma_ts_run8(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc,
                                             uint32_t accumulate);
template <>
__device__ __forceinline__ void umma_ts_run8<1024>(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc,
                                                   uint32_t accumulate) {
  asm volatile(AT_RUN_HEAD
               "mov.b64 db, {%2, %5};\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p;\n\t"
               AT_TS_STEP(8, 2) AT_TS_STEP(16, 4) AT_TS_STEP(24, 6) AT_TS_STEP(32, 1024) AT_TS_STEP(40, 1026)
               AT_TS_STEP(48, 1028) AT_TS_STEP(56, 1030) "}"
               ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(AT_SDESC_HI)
               : "memory");
}
template <>
__device__ __forceinline__ void umma_ts_run8<512>(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(AT_RUN_HEAD
               "mov.b64 db, {%2, %5};\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p;\n\t"
               AT_TS_STEP(8, 2) AT_TS_STEP(16, 4) AT_TS_STEP(24, 6) AT_TS_STEP(32, 512) AT_TS_STEP(40, 514)
               AT_TS_STEP(48, 516) AT_TS_STEP(56, 518) "}"
               ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(AT_SDESC_HI)
               : "memory");
}

// SPARSE: block-sparse attention over 128 x 128 (query tile, key tile) blocks.  mask[h][qi][kj]
// != 0 keeps key tile kj for query tile qi of head h; every other score is -inf.  The CTA
// loads the key tiles either of its two query tiles keeps, and each query tile multiplies and
// normalises only the ones it keeps.  A query row that keeps no key tile gets a zero output.
template <int HD, bool SPARSE>
__global__ void __launch_bounds__(AT_THREADS, 1)
    attention_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, bf16* __restrict__ o, int n_rows, int nh,
                        float scale_log2, const uint8_t* __restrict__ mask, unsigned* err) {
  using C = AtCfg<HD>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  const uint32_t b_q = smem_u32(bars);
  const uint32_t b_kfull = b_q + 8;               // [ST]
  const uint32_t b_vfull = b_kfull + 8 * ST;      // [ST]
  const uint32_t b_kvempty = b_vfull + 8 * ST;    // [ST]
  const uint32_t b_sfull = b_kvempty + 8 * ST;    // [2] (tile A, tile B)
  const uint32_t b_pfull = b_sfull + 16;          // [2]
  const uint32_t b_odone = b_pfull + 16;
  const uint32_t b_drain = b_odone + 8;           // failure path: the issuer's MMAs have completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 1 + 3 * ST + 6);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ErrCtx ec = err_ctx(err);
  const int h = blockIdx.y;
  const int q0 = blockIdx.x * 2 * AT_BM;
  const int nt = cdiv(n_rows, AT_BN);
  // key-tile masks of this CTA's two query tiles (dense: every tile kept)
  const int qt = cdiv(n_rows, AT_BM);
  const uint8_t* mask_a = SPARSE ? mask + (static_cast<size_t>(h) * qt + 2 * blockIdx.x) * nt : nullptr;
  const uint8_t* mask_b = (SPARSE && 2 * blockIdx.x + 1 < qt) ? mask_a + nt : nullptr;
  auto keep = [&](int x, int j) -> bool {
    if (!SPARSE) return true;
    const uint8_t* m = x ? mask_b : mask_a;
    return m != nullptr && m[j] != 0;
  };
  // the key tiles the CTA visits, in order: next_tile(j) = first kept tile >= j (nt if none)
  auto next_tile = [&](int j) -> int {
    if (SPARSE)
      while (j < nt && !keep(0, j) && !keep(1, j)) ++j;
    return j;
  };

  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(b_kfull + 8 * s, 1);
      mbar_init(b_vfull + 8 * s, 1);
      mbar_init(b_kvempty + 8 * s, 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(b_sfull + 8 * x, 1);
      mbar_init(b_pfull + 8 * x, 4);
    }
    mbar_init(b_odone, 1);
    mbar_init(b_drain, 1);
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

  if (warp < 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(AT_REGS_CTRL));

  const uint32_t sQ = smem_u32(smem + C::Q_OFF);
  const uint32_t sK = smem_u32(smem + C::K_OFF);
  const uint32_t sV = smem_u32(smem + C::V_OFF);

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(b_q, 2 * C::QK_TILE);
      for (int x = 0; x < 2; ++x)
        for (int a = 0; a < HD / 64; ++a)
          tma_load_3d(sQ + x * C::QK_TILE + a * AT_ATOM, &tmQ, b_q, 64 * a, q0 + x * AT_BM, h);
      int issued = 0;
      bool ok = true;
      for (int it = 0, j = next_tile(0); j < nt; ++it, j = next_tile(j + 1)) {
        const int s = it % ST;
        if (!mbar_wait(b_kvempty + 8 * s, ((it / ST) & 1) ^ 1, ec, kErrAttnProducer)) {
          ok = false;
          break;
        }
        const uint32_t kd = sK + s * C::QK_TILE, vd = sV + s * C::V_TILE;
        mbar_arrive_expect_tx(b_kfull + 8 * s, C::QK_TILE);
        for (int a = 0; a < HD / 64; ++a) tma_load_3d(kd + a * AT_ATOM, &tmK, b_kfull + 8 * s, 64 * a, j * AT_BN, h);
        mbar_arrive_expect_tx(b_vfull + 8 * s, C::V_TILE);
        tma_load_3d(vd, &tmV, b_vfull + 8 * s, j * AT_BN, 0, h);
        tma_load_3d(vd + C::V_ATOM, &tmV, b_vfull + 8 * s, j * AT_BN + 64, 0, h);
        issued = it + 1;
      }
      if (!ok) {  // let the copies still in flight land before the shared memory is released
        mbar_drain(b_q, 0);
        for (int i = issued > ST ? issued - ST : 0; i < issued; ++i) {
          mbar_drain(b_kfull + 8 * (i % ST), (i / ST) & 1);
          mbar_drain(b_vfull + 8 * (i % ST), (i / ST) & 1);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, HD);
      // Descriptors are built once per operand tile (their low words) and stepped inside the MMA
      // runs by the compile-time offset of each 16-wide k slice: the start-address field holds
      // the shared address in 16-byte units, and no tile crosses 256 KB, so the step is a plain
      // add.  it = position of the key tile in the CTA's visiting order (ring stage and phase).
      static_assert(AT_ATOM >> 4 == 1024 && (HD == 128 || HD == 64), "offsets in the MMA runs");
      auto issue_s = [&](int x, int it) {  // S_x = Q_x K^T for visited tile it
        const uint32_t dq = sdesc_lo(sQ + x * C::QK_TILE), dk = sdesc_lo(sK + (it % ST) * C::QK_TILE);
        if constexpr (HD == 128) umma_ss_run8(tmem + x * 128, dq, dk, idesc_s, 0);
        else umma_ss_run4(tmem + x * 128, dq, dk, idesc_s, 0);
        umma_commit(b_sfull + 8 * x);
      };
      auto issue_pv = [&](int x, int it, int first) {  // O_x (+)= P_x V for visited tile it
        const uint32_t dv = sdesc_lo(sV + (it % ST) * C::V_TILE);
        umma_ts_run8<(C::V_ATOM >> 4)>(tmem + 256 + x * HD, tmem + x * 128, dv, idesc_o, !first);
      };
      // Each query tile runs its own sequence over the key tiles it keeps (all of them when
      // dense); cnt[x] counts tile x's S / P phases.  S_x of the next kept tile is issued right
      // after PV_x of the current one, so it may overwrite P_x in TMEM (in-order execution).
      int j = next_tile(0);
      int cnt[2] = {0, 0};
      bool ok = mbar_wait(b_q, 0, ec, kErrAttnMma);
      if (ok && j < nt) {
        ok = mbar_wait(b_kfull, 0, ec, kErrAttnMma);
        if (ok) {
          tc_fence_after();
          if (keep(0, j)) issue_s(0, 0);
          if (keep(1, j)) issue_s(1, 0);
        }
      }
      for (int it = 0; ok && j < nt; ++it) {
        const int s = it % ST;
        const uint32_t par = (it / ST) & 1;
        const int jn = next_tile(j + 1);
        const bool more = jn < nt;
        bool v_ready = false, k_ready = false;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (keep(x, j)) {  // P_x V for this tile
            if (!mbar_wait(b_pfull + 8 * x, cnt[x] & 1, ec, kErrAttnMma)) {
              ok = false;
              break;
            }
            if (!v_ready && !mbar_wait(b_vfull + 8 * s, par, ec, kErrAttnMma)) {
              ok = false;
              break;
            }
            v_ready = true;
            tc_fence_after();
            issue_pv(x, it, cnt[x] == 0);
            ++cnt[x];
          }
          if (x == 1) umma_commit(b_kvempty + 8 * s);  // K / V of this stage are no longer read
          if (more && keep(x, jn)) {  // S_x of the next visited tile
            if (!k_ready && !mbar_wait(b_kfull + 8 * ((it + 1) % ST), ((it + 1) / ST) & 1, ec, kErrAttnMma)) {
              ok = false;
              break;
            }
            k_ready = true;
            tc_fence_after();
            issue_s(x, it + 1);
          }
        }
        j = jn;
      }
      if (ok) {
        umma_commit(b_odone);
      } else {  // the MMAs already issued finish before TMEM is released
        umma_commit(b_drain);
        mbar_drain(b_drain, 0);
      }
    }
  } else if (warp >= 4) {
    // softmax warps: tile x = 0 (warps 4..7) or 1 (warps 8..11); TMEM lane quadrant = warp % 4
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(AT_REGS_SOFTMAX));
    const int x = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_off + x * 128;
    const uint32_t t_o = tmem + lane_off + 256 + x * HD;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    int cnt = 0;  // S / P phases of this query tile = key tiles it keeps
    for (int j = next_tile(0); j < nt; j = next_tile(j + 1)) {
      if (SPARSE && !keep(x, j)) continue;  // visited for the other query tile only
      if (!mbar_wait(b_sfull + 8 * x, cnt & 1, ec, kErrAttnSoftmax)) {
        ok = false;
        break;
      }
      ++cnt;
      tc_fence_after();
      uint32_t sv[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t(&chunk)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c]);
        tmem_ld32(t_s + c * 32, chunk);
      }
      tmem_wait_ld();
      const int valid = n_rows - j * AT_BN;  // keys of this tile that exist
      if (valid < AT_BN) {
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= valid) sv[i] = __float_as_uint(-INFINITY);
      }
      // row max with 3-input max (tree of 43 + 1 instructions for 128 values)
      float mq[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float m = __uint_as_float(sv[32 * c]);
#pragma unroll
        for (int i = 1; i < 31; i += 2) m = fmax3f(m, __uint_as_float(sv[32 * c + i]), __uint_as_float(sv[32 * c + i + 1]));
        mq[c] = fmaxf(m, __uint_as_float(sv[32 * c + 31]));
      }
      const float mt = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * scale_log2;
      float alpha = 1.f;
      bool rescale = false;
      if (m_used == -INFINITY) {  // first tile this query tile keeps
        m_used = mt;
      } else if (mt > m_used + AT_RESCALE_THRESHOLD) {
        alpha = ex2f(m_used - mt);
        m_used = mt;
        rescale = true;
      }
      // p = 2^(s * scale - m): paired f32x2 FMA and add, ex2 on the SFU, bf16x2 pack
      const uint64_t c2 = pack_f32x2(scale_log2, scale_log2);
      const uint64_t nm2 = pack_f32x2(-m_used, -m_used);
      uint64_t rs2 = pack_f32x2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint64_t e2 = fma_f32x2(pack_u32x2(sv[32 * c + 2 * i], sv[32 * c + 2 * i + 1]), c2, nm2);
          const float p0 = ex2f(lo_f32(e2)), p1 = ex2f(hi_f32(e2));
          rs2 = add_f32x2(rs2, pack_f32x2(p0, p1));
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(t_s + c * 16, pk);  // keys 32c..32c+31 -> bf16 pairs in columns 16c..16c+15
      }
      const float rs = lo_f32(rs2) + hi_f32(rs2);
      l = l * alpha + rs;
      // O_x is quiescent until P_x(j) is released (PV_x(j-1) completed before S_x(j)):
      // rescale it now if the max grew
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t u[32];
          tmem_ld32(t_o + c * 32, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
          tmem_st32(t_o + c * 32, u);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_pfull + 8 * x);
    }
    if (ok && mbar_wait(b_odone, 0, ec, kErrAttnSoftmax)) {
      tc_fence_after();
      const int row = q0 + x * AT_BM + r;
      const float inv = l > 0.f ? 1.f / l : 0.f;  // a row that kept no key tile outputs zeros
      bf16* dst = o + static_cast<size_t>(row) * nh * HD + h * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(t_o + c * 32, u);
        tmem_wait_ld();
        if (row < n_rows) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = l > 0.f ? pack_bf16x2(__uint_as_float(u[8 * q + 2 * e]) * inv,
                                           __uint_as_float(u[8 * q + 2 * e + 1]) * inv)
                             : 0u;  // O was never written (or is all zero): do not read it
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

template <int HD, bool SPARSE>
static cudaError_t launch_at(const bf16* q, const bf16* k, const bf16* vt, int ld_vt, bf16* o, int n_rows, int nh,
                             const uint8_t* mask, unsigned* err, cudaStream_t st) {
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
    cudaError_t e =
        cudaFuncSetAttribute(attention_tc_kernel<HD, SPARSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    // the register split above is only sound if the kernel launches with exactly this count
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, attention_tc_kernel<HD, SPARSE>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != AT_LAUNCH_REGS) return cudaErrorInvalidConfiguration;
    configured = true;
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  dim3 grid(cdiv(n_rows, 2 * AT_BM), nh);
  attention_tc_kernel<HD, SPARSE><<<grid, AT_THREADS, C::SMEM, st>>>(tq, tk, tv, o, n_rows, nh, scale_log2, mask, err);
  return cudaGetLastError();
}

cudaError_t launch_attention_tc(const bf16* q, const bf16* k, const bf16* vt, int ld_vt, bf16* o, int n_rows, int nh,
                                int hd, unsigned* err, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  if (hd == 128) return launch_at<128, false>(q, k, vt, ld_vt, o, n_rows, nh, nullptr, err, st);
  if (hd == 64) return launch_at<64, false>(q, k, vt, ld_vt, o, n_rows, nh, nullptr, err, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attention_sparse_tc(const bf16* q, const bf16* k, const bf16* vt, int ld_vt, bf16* o, int n_rows,
                                       int nh, int hd, const uint8_t* mask, unsigned* err, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  if (hd == 128) return launch_at<128, true>(q, k, vt, ld_vt, o, n_rows, nh, mask, err, st);
  if (hd == 64) return launch_at<64, true>(q, k, vt, ld_vt, o, n_rows, nh, mask, err, st);
  return cudaErrorInvalidValue;
}

}  // namespace h3
