// a2 / a5 / a7 / a8 / a9: the trunk linears on the 5th-generation tensor cores.
//
// y[M, n] = epilogue(x[M, K] . W[n, K]^T + b), x and W both K-major bf16 (or W as weight-only
// INT8 group-32 codes, "mlx-h3" README, "Local model layout"), fp32 accumulation in TMEM.
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles; 128 x 192 for the plain and
// gate+residual linears when that fills the last wave of SMs better):
//   warp 0      TMA producer: A tile 128x64 and B tile 256x64 per stage (128-byte swizzle)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer (M=128, N=256, K=16 steps)
//   warps 2..5  epilogue: tcgen05.ld 32 columns at a time, bias / SwiGLU / gate+residual, store
//   warps 6..21 (INT8 only) two groups of eight that take the stages in turn: a warp loads
//               the u8 codes, scales and qbias of its group's next stage from global memory
//               into registers right after handing the current stage to the tensor core, and
//               writes them dequantised into the swizzled bf16 B tile.  With no load in flight
//               when a warp issues its proxy fence, the fence waits for the shared stores
//               alone (measured on the INT8 GEMMs at 12,936 rows: 8 - 17% faster than sixteen
//               warps each keeping three stages of loads in flight across their fences)
// Two 256-column accumulators in TMEM let the epilogue of tile i overlap the mainloop of i+1.
//
// Epilogues ("minimax-h3-mlx" README, "Validation" and "AdaLN: measure, do not reason";
// "H3-metal" README, "Metal 4 and TensorOps paths" for the paired gate/up tiles):
//   BIAS     y = acc + b
//   SWIGLU   the B tile is the gate rows j..j+127 and the value rows F+j..F+j+127, so one
//            256-wide accumulator holds both halves and y = silu(g + b_g) * (v + b_v) is
//            formed on-chip; only the F-wide activation is written
//   GATE_RES y = res + gate[tag, t] * (acc + b), the AdaLN gate gathered per row
#include <cudaTypedefs.h>

#include "kernels.h"

namespace h3 {

constexpr int G_BM = 128, G_BN = 256, G_BK = 64;
constexpr int G_A_BYTES = G_BM * G_BK * 2;   // 16 KB
// Tile raster: column sweeps over groups of group_m row-blocks.  The host sizes group_m so a
// group's A rows (group_m x 128 x K x 2 bytes) take about 24 MB of the 126 MB L2 and stay
// resident while the sweep streams B once per group: B is read from HBM m_tiles / group_m
// times, A once.  Measured on fc1 at 33,720 rows (one launch, DRAM bytes read): 5.0 GB with
// 24 MB groups, 6.4 GB with 48 MB and 19.9 GB with 96 MB, where the larger groups no longer
// stay resident beside the B stream; the 50-block step time is the same at 24 and 48 MB.
constexpr size_t kRasterABytes = size_t(24) << 20;

// bf16 weights: 128 x 256 tiles, two TMEM accumulators so the epilogue of one tile overlaps the
// mainloop of the next.  INT8 weights: 256 x 256 tiles (two 128-row MMAs per k-step share each
// dequantised B tile, halving the dequantisation per FLOP); the two accumulators fill TMEM, so
// the epilogue does not overlap the next tile's mainloop.
// bf16 weights with the plain or gate+residual epilogue may also run 128 x 192 tiles (BN = 192):
// chosen on the host when they fill the last wave of SMs better (small row counts against the
// 5376-wide projections), with a fifth ring stage in the shared memory the narrower B tile frees.
template <bool INT8, int BN = G_BN>
struct GemmCfg {
  static constexpr int BM = INT8 ? 256 : 128;
  static constexpr int MSUB = BM / 128;        // 128-row MMAs per k-step
  static constexpr int NBUF = INT8 ? 1 : 2;    // accumulator buffers
  static constexpr int A_BYTES = BM * G_BK * 2;
  static constexpr int B_BYTES = BN * G_BK * 2;  // INT8: the dequantised 256-row tile
  static constexpr int STAGES = INT8 ? 3 : (BN == G_BN ? 4 : 5);
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int THREADS = INT8 ? 192 + 32 * 16 : 192;  // INT8: 2 groups of 8 dequant warps
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + 256;
};

struct GemmParams {
  int M, K, n_y;
  int m_tiles, n_tiles, num_tiles, kb_count;
  int group_m;      // row-blocks per raster group
  int b_row_step;   // B rows per column tile: 256 (plain) or 128 (SwiGLU)
  int b_row1_off;   // row offset of the second 128-row half of a B tile: 128, or n_y for SwiGLU
  const bf16* bias;
  bf16* y;
  int ldy;
  const bf16* res;
  TableRef gate;
  int m_gate;
  const void* wcodes;  // INT8: u8 [rows, K]
  const bf16* wscale;  // INT8: [rows, K/32]
  const bf16* wqbias;
  int groups;          // K / 32
  int w_rows;          // rows of W (codes beyond it are TMA zero fill; their scales are not read)
  // QKV epilogue (head_dim 128): column tile nb < nh holds head nb's q and k rows, tile
  // nb >= nh the v rows of heads 2(nb - nh) and 2(nb - nh) + 1
  int nh;
  const float2* cs;    // [M][64] rotary (cos, sin)
  const bf16* qn;      // [128] RMSNorm weights or null
  const bf16* kn;
  float qk_eps;
  bf16* q;             // [nh][M][128]
  bf16* k;
  bf16* vt;            // [nh][128][ld_vt]
  int ld_vt;
  unsigned* err;
};

// First row of each 128-row half of the B tile of column tile nb.
template <int EPI>
__device__ __forceinline__ void b_tile_rows(const GemmParams& p, int nb, int& r0, int& r1) {
  if (EPI == kEpiQkv) {
    if (nb < p.nh) {
      r0 = nb * 384;          // q rows of head nb; its k rows follow
      r1 = r0 + 128;
    } else {
      const int h0 = 2 * (nb - p.nh);
      r0 = h0 * 384 + 256;    // v rows of heads h0 and h0 + 1
      r1 = r0 + 384;
    }
  } else {
    r0 = nb * p.b_row_step;
    r1 = r0 + p.b_row1_off;
  }
}

__device__ __forceinline__ void tile_coords(int tile, int m_tiles, int n_tiles, int group_m, int& mb, int& nb) {
  const int per_group = group_m * n_tiles;
  const int g = tile / per_group;
  const int first_m = g * group_m;
  const int gm = min(m_tiles - first_m, group_m);
  const int local = tile % per_group;
  mb = first_m + local % gm;
  nb = local / gm;
}

__device__ __forceinline__ void load8(const bf16* p, float* f) {
  const int4 u = ld_nc_v4(p);
  const uint32_t w[4] = {(uint32_t)u.x, (uint32_t)u.y, (uint32_t)u.z, (uint32_t)u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16lo(w[i]);
    f[2 * i + 1] = bf16hi(w[i]);
  }
}

// CW consecutive values of a row: 16-byte stores when the chunk is whole, element stores at the
// ragged end of the row
template <int CW>
__device__ __forceinline__ void store_row(bf16* dst, const float* v, int valid) {
  if (valid >= CW) {
#pragma unroll
    for (int c = 0; c < CW / 8; ++c) {
      const int4 o = make_int4(pack_bf16x2(v[8 * c], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                               pack_bf16x2(v[8 * c + 4], v[8 * c + 5]), pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
      reinterpret_cast<int4*>(dst)[c] = o;
    }
  } else {
#pragma unroll
    for (int i = 0; i < CW; ++i)
      if (i < valid) dst[i] = f2bf(v[i]);
  }
}

template <int CW>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[CW]) {
  if constexpr (CW == 32) {
    tmem_ld32(taddr, r);
  } else {
    static_assert(CW == 16, "16- or 32-column chunks");
    tmem_ld16(taddr, r);
  }
}

__device__ __forceinline__ void load16_f32(const bf16* p, float* f) {
  load8(p, f);
  load8(p + 8, f + 8);
}

// QKV epilogue of one tile for the calling thread's row ("H3-metal" README, "Checkpoint layout
// and media pipeline": QK normalisation and RoPE consume the per-head interleaved projection).
// q|k tile (nb < nh): columns 0..127 are head nb's q, 128..255 its k.  Each thread owns one row,
// so the RMS over 128 values and the rotary pairs (i, i + 64) stay in the thread: pass 1 reads
// the accumulator for the two sums of squares, pass 2 re-reads it 8 pairs at a time, applies
// bias, norm weight and rotation, and writes 256 contiguous bytes per head row.  v tile: two
// heads' v rows, written transposed (warp lanes = consecutive rows, so each store instruction
// covers 64 contiguous bytes).
__device__ __forceinline__ void qkv_epilogue(const GemmParams& p, uint32_t tacc, int row, int nb) {
  const bool row_ok = row < p.M;
  if (nb < p.nh) {
    const int h = nb;
    const bf16* bh = p.bias ? p.bias + static_cast<size_t>(h) * 384 : nullptr;
    float ssq = 0.f, ssk = 0.f;
#pragma unroll 1
    for (int c = 0; c < 16; ++c) {
      uint32_t r[16];
      tmem_ld16(tacc + c * 16, r);
      tmem_wait_ld();
      float b[16];
      if (bh) {
        load16_f32(bh + c * 16, b);
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) b[e] = 0.f;
      }
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float v = __uint_as_float(r[e]) + b[e];
        acc = fmaf(v, v, acc);
      }
      if (c < 8) ssq += acc;
      else ssk += acc;
    }
    const bool has_norm = p.qn != nullptr && p.kn != nullptr;
    const float rnq = has_norm ? rsqrtf(ssq / 128.f + p.qk_eps) : 1.f;
    const float rnk = has_norm ? rsqrtf(ssk / 128.f + p.qk_eps) : 1.f;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {  // rotary pairs i = 8c .. 8c + 7
      float cs_c[8], cs_s[8];
      if (row_ok) {
        const float4* src = reinterpret_cast<const float4*>(p.cs + static_cast<size_t>(row) * 64 + 8 * c);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float4 v = __ldg(src + e);
          cs_c[2 * e] = v.x;
          cs_s[2 * e] = v.y;
          cs_c[2 * e + 1] = v.z;
          cs_s[2 * e + 1] = v.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) cs_c[e] = cs_s[e] = 0.f;
      }
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {
        uint32_t ra[8], rb[8];
        tmem_ld8(tacc + part * 128 + 8 * c, ra);
        tmem_ld8(tacc + part * 128 + 64 + 8 * c, rb);
        tmem_wait_ld();
        float ba[8], bb[8], wa[8], wb[8];
        if (bh) {
          load8(bh + part * 128 + 8 * c, ba);
          load8(bh + part * 128 + 64 + 8 * c, bb);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) ba[e] = bb[e] = 0.f;
        }
        if (has_norm) {
          const bf16* wn = part ? p.kn : p.qn;
          load8(wn + 8 * c, wa);
          load8(wn + 64 + 8 * c, wb);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) wa[e] = wb[e] = 1.f;
        }
        const float rn = part ? rnk : rnq;
        uint32_t oa[4], ob[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float ya[2], yb[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int i = 2 * e + u;
            const float xa = (__uint_as_float(ra[i]) + ba[i]) * rn * wa[i];
            const float xb = (__uint_as_float(rb[i]) + bb[i]) * rn * wb[i];
            ya[u] = xa * cs_c[i] - xb * cs_s[i];
            yb[u] = xa * cs_s[i] + xb * cs_c[i];
          }
          oa[e] = pack_bf16x2(ya[0], ya[1]);
          ob[e] = pack_bf16x2(yb[0], yb[1]);
        }
        if (row_ok) {
          bf16* dst = (part ? p.k : p.q) + (static_cast<size_t>(h) * p.M + row) * 128;
          *reinterpret_cast<int4*>(dst + 8 * c) = make_int4(oa[0], oa[1], oa[2], oa[3]);
          *reinterpret_cast<int4*>(dst + 64 + 8 * c) = make_int4(ob[0], ob[1], ob[2], ob[3]);
        }
      }
    }
  } else {
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
      const int h = 2 * (nb - p.nh) + hh;
      const bf16* bh = (p.bias && h < p.nh) ? p.bias + static_cast<size_t>(h) * 384 + 256 : nullptr;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tacc + hh * 128 + c * 32, r);
        tmem_wait_ld();
        if (!row_ok || h >= p.nh) continue;
        float b[32];
        if (bh) {
          load16_f32(bh + c * 32, b);
          load16_f32(bh + c * 32 + 16, b + 16);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) b[e] = 0.f;
        }
        bf16* dst = p.vt + (static_cast<size_t>(h) * 128 + c * 32) * p.ld_vt + row;
#pragma unroll
        for (int e = 0; e < 32; ++e) dst[static_cast<size_t>(e) * p.ld_vt] = f2bf(__uint_as_float(r[e]) + b[e]);
      }
    }
  }
}

// Epilogue of one tile for the calling thread's row (TMEM lane = row within the tile), CW
// accumulator columns at a time (16 in the INT8 kernels, whose 22 warps leave 80 registers a
// thread; 32 otherwise).
template <int EPI, int CW, int BN>
__device__ __forceinline__ void gemm_epilogue(const GemmParams& p, uint32_t tacc, int row, int nb) {
  const bool row_ok = row < p.M;
  if (EPI == kEpiQkv) {
    qkv_epilogue(p, tacc, row, nb);
  } else if (EPI == kEpiSwiglu) {
#pragma unroll 1
    for (int c = 0; c < 128 / CW; ++c) {
      uint32_t rg[CW], rv[CW];
      tmem_ld_cols<CW>(tacc + c * CW, rg);
      tmem_ld_cols<CW>(tacc + 128 + c * CW, rv);
      tmem_wait_ld();
      const int col0 = nb * 128 + c * CW;
      if (row_ok && col0 < p.n_y) {
        float v[CW];
        const int valid = min(CW, p.n_y - col0);
#pragma unroll
        for (int q = 0; q < CW / 8; ++q) {
          float bg[8], bv[8];
          if (p.bias && valid >= CW) {
            load8(p.bias + col0 + 8 * q, bg);
            load8(p.bias + p.n_y + col0 + 8 * q, bv);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int cc = col0 + 8 * q + e;
              bg[e] = (p.bias && cc < p.n_y) ? bf2f(p.bias[cc]) : 0.f;
              bv[e] = (p.bias && cc < p.n_y) ? bf2f(p.bias[p.n_y + cc]) : 0.f;
            }
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float g = __uint_as_float(rg[8 * q + e]) + bg[e];
            const float u = __uint_as_float(rv[8 * q + e]) + bv[e];
            // silu(g) u with the SFU exponential and a fast reciprocal: a few fp32 ulps,
            // far below the bf16 rounding of the stored activation; for g below ~-88 the
            // reciprocal of an infinite 1 + e^-g gives 0
            v[8 * q + e] = g * __fdividef(1.f, 1.f + __expf(-g)) * u;
          }
        }
        store_row<CW>(p.y + static_cast<size_t>(row) * p.ldy + col0, v, valid);
      }
    }
  } else {
    const bf16* gate_row = nullptr;
    if (EPI == kEpiGateRes && row_ok) {
      const TableRef& t = p.gate;
      gate_row = t.table_b + static_cast<long long>(t.tidx[row]) * t.t_stride +
                 static_cast<long long>(6 * t.tag[row] + p.m_gate) * p.n_y;
    }
#pragma unroll 1
    for (int c = 0; c < BN / CW; ++c) {
      uint32_t r[CW];
      tmem_ld_cols<CW>(tacc + c * CW, r);
      tmem_wait_ld();
      const int col0 = nb * BN + c * CW;
      if (row_ok && col0 < p.n_y) {
        const int valid = min(CW, p.n_y - col0);
        float v[CW];
#pragma unroll
        for (int q = 0; q < CW / 8; ++q) {
          float b[8], rs[8], g[8];
          if (valid >= CW) {
            if (p.bias) load8(p.bias + col0 + 8 * q, b);
            else {
#pragma unroll
              for (int e = 0; e < 8; ++e) b[e] = 0.f;
            }
            if (EPI == kEpiGateRes) {
              load8(p.res + static_cast<size_t>(row) * p.ldy + col0 + 8 * q, rs);
              load8(gate_row + col0 + 8 * q, g);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int cc = col0 + 8 * q + e;
              const bool ok = cc < p.n_y;
              b[e] = (p.bias && ok) ? bf2f(p.bias[cc]) : 0.f;
              if (EPI == kEpiGateRes) {
                rs[e] = ok ? bf2f(p.res[static_cast<size_t>(row) * p.ldy + cc]) : 0.f;
                g[e] = ok ? bf2f(gate_row[cc]) : 0.f;
              }
            }
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float a = __uint_as_float(r[8 * q + e]) + b[e];
            v[8 * q + e] = (EPI == kEpiGateRes) ? rs[e] + g[e] * a : a;
          }
        }
        store_row<CW>(p.y + static_cast<size_t>(row) * p.ldy + col0, v, valid);
      }
    }
  }
}

// Dequant warp groups taking the stages in turn.  A group's wait for B slot q % S reads the
// barrier's phase parity, so the barrier must be at most one phase behind: the group's own
// previous stage q - DQ_GROUPS needed stage q - DQ_GROUPS - S released, which covers q - 2S only
// when DQ_GROUPS <= S.
constexpr int DQ_GROUPS = 2;
static_assert(DQ_GROUPS <= GemmCfg<true>::STAGES, "a dequant group could run a whole ring cycle ahead");
constexpr int DQ_THREADS = 512 / DQ_GROUPS;     // threads of one group
constexpr int DQ_ROWS = 256 / (DQ_THREADS / 4);  // B-tile rows per thread (four threads per row)

// One dequant stage of the calling thread: its rows' 16-code chunk (k-chunk t & 3 of the
// stage's 64 k) and the scale and qbias of the group that chunk belongs to.
struct DqStage {
  int4 codes[DQ_ROWS];
  float sc[DQ_ROWS], qb[DQ_ROWS];
};

__device__ __forceinline__ void dq_load_stage(const GemmParams& p, const uint8_t* w, int brow0, int brow1, int kb,
                                              int t, DqStage& d) {
  const int kc = t & 3;
  const int g = kb * 2 + (kc >> 1);
  const int k0 = kb * 64 + kc * 16;
#pragma unroll
  for (int i = 0; i < DQ_ROWS; ++i) {
    const int n = (t >> 2) + (DQ_THREADS / 4) * i;  // row within the 256-row tile
    const int grow = (n < 128) ? brow0 + n : brow1 + (n - 128);
    const bool ok = grow < p.w_rows && k0 < p.K;  // K % 32 == 0: a 16-code chunk is all in or all out
    const size_t gi = static_cast<size_t>(grow) * p.groups + g;
    d.codes[i] = ok ? ld_nc_v4(w + static_cast<size_t>(grow) * p.K + k0) : make_int4(0, 0, 0, 0);
    d.sc[i] = ok ? bf2f(p.wscale[gi]) : 0.f;
    d.qb[i] = ok ? bf2f(p.wqbias[gi]) : 0.f;
  }
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Two codes (given as the f32 bit patterns 2^23 + code) -> bf16x2 of fma_f32(sc, code, qb):
// the subtraction of 2^23 is exact, the fused multiply-add rounds once to f32 per lane, then
// each lane is rounded to bf16 (nearest even).
__device__ __forceinline__ uint32_t dq_pair(uint32_t m0, uint32_t m1, uint64_t sc2, uint64_t qb2) {
  uint64_t v, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(m0), "r"(m1));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(v), "l"(0xCB000000CB000000ull));  // - 2^23
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(v) : "l"(r), "l"(sc2), "l"(qb2));
  uint32_t lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
  return pack_bf16x2(__uint_as_float(lo), __uint_as_float(hi));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Dequantise one stage: the thread's codes -> bf16 [256][64] in the 128-byte swizzled K-major
// layout (row n at n*128 bytes, 16-byte chunk c at c ^ (n & 7)).  Thread t of the DQ_THREADS
// threads of a dequant warp group handles k-chunk (t & 3) (16 codes, one group) of rows
// t/4 + (DQ_THREADS/4) i.  Each
// 16-byte chunk goes out as one 128-bit shared store: a quarter warp (two rows, eight chunks)
// then covers all 32 banks once.
__device__ __forceinline__ void dequant_stage(uint32_t sb, const DqStage& d, int t) {
  const int kc = t & 3;
#pragma unroll
  for (int i = 0; i < DQ_ROWS; ++i) {
    const int n = (t >> 2) + (DQ_THREADS / 4) * i;
    const uint64_t sc2 = (static_cast<uint64_t>(__float_as_uint(d.sc[i])) << 32) | __float_as_uint(d.sc[i]);
    const uint64_t qb2 = (static_cast<uint64_t>(__float_as_uint(d.qb[i])) << 32) | __float_as_uint(d.qb[i]);
    const uint32_t cw[4] = {(uint32_t)d.codes[i].x, (uint32_t)d.codes[i].y, (uint32_t)d.codes[i].z,
                            (uint32_t)d.codes[i].w};
    uint32_t o[8];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // bytes 2h, 2h+1 of the word under the exponent byte of 2^23: exact u8 -> f32 pattern
        const uint32_t m0 = prmt(cw[w], 0x4B000000u, 0x7540u + 2 * h);
        const uint32_t m1 = prmt(cw[w], 0x4B000000u, 0x7541u + 2 * h);
        o[2 * w + h] = dq_pair(m0, m1, sc2, qb2);
      }
    }
    const uint32_t rowp = sb + n * 128;
    const int c0 = 2 * kc, c1 = 2 * kc + 1;
    st_shared_v4(rowp + ((c0 ^ (n & 7)) << 4), o[0], o[1], o[2], o[3]);
    st_shared_v4(rowp + ((c1 ^ (n & 7)) << 4), o[4], o[5], o[6], o[7]);
  }
}

template <int EPI, bool INT8, int BN = G_BN>
__global__ void __launch_bounds__(GemmCfg<INT8>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
  static_assert(BN == G_BN || (!INT8 && (EPI == kEpiBias || EPI == kEpiGateRes) && BN % 64 == 0),
                "narrow column tiles only for bf16 weights with the plain or gate epilogue");
  using C = GemmCfg<INT8, BN>;
  constexpr int S = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::STAGE_BYTES);
  const uint32_t bar_full = smem_u32(bars);          // S barriers: TMA landed
  const uint32_t bar_empty = bar_full + 8 * S;       // S barriers: MMA done with the stage
  const uint32_t bar_ready = bar_empty + 8 * S;      // S barriers: INT8 dequant done
  const uint32_t bar_tfull = bar_ready + 8 * S;      // 2 barriers: accumulator complete
  const uint32_t bar_tempty = bar_tfull + 16;        // 2 barriers: accumulator drained
  const uint32_t bar_drain = bar_tempty + 16;        // failure path: the issuer's MMAs have completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * S + 5);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ErrCtx ec = err_ctx(p.err);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_ready + 8 * s, DQ_THREADS / 32);  // the warps of the group that dequantises the stage
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, 4);
    }
    mbar_init(bar_drain, 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto sA = [&](int s) { return smem + s * C::STAGE_BYTES; };
  auto sB = [&](int s) { return smem + s * C::STAGE_BYTES + C::A_BYTES; };

  if (warp == 0) {
    if (lane == 0) {
      int s = 0, issued = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, p.m_tiles, p.n_tiles, p.group_m, mb, nb);
        int brow0, brow1;
        b_tile_rows<EPI>(p, nb, brow0, brow1);
        for (int kb = 0; kb < p.kb_count; ++kb, ++issued) {
          if (!mbar_wait(bar_empty + 8 * s, ph ^ 1, ec, kErrGemmProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * s;
          mbar_arrive_expect_tx(fb, C::A_BYTES + (INT8 ? 0 : C::B_BYTES));
#pragma unroll
          for (int a = 0; a < C::MSUB; ++a)
            tma_load_2d(smem_u32(sA(s)) + a * G_A_BYTES, &tmA, fb, kb * G_BK, mb * C::BM + a * 128);
          if (!INT8 && BN == G_BN) {  // two 128-row boxes (SwiGLU: gate rows, then value rows)
            tma_load_2d(smem_u32(sB(s)), &tmB, fb, kb * G_BK, brow0);
            tma_load_2d(smem_u32(sB(s)) + 128 * 128, &tmB, fb, kb * G_BK, brow1);
          } else if (!INT8) {  // BN / 64 boxes of 64 consecutive rows
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
              tma_load_2d(smem_u32(sB(s)) + i * 64 * 128, &tmB, fb, kb * G_BK, brow0 + 64 * i);
          }
          if (++s == S) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok)  // let the copies still in flight land before the shared memory is released
        for (int i = issued > S ? issued - S : 0; i < issued; ++i) mbar_drain(bar_full + 8 * (i % S), (i / S) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(G_BM, BN);
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        if (!mbar_wait(bar_tempty + 8 * acc, aph ^ 1, ec, kErrGemmMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * C::MSUB * G_BN;  // accumulators 256 columns apart
        for (int kb = 0; kb < p.kb_count; ++kb) {
          if (!mbar_wait(bar_full + 8 * s, ph, ec, kErrGemmMma) ||
              (INT8 && !mbar_wait(bar_ready + 8 * s, ph, ec, kErrGemmMma))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA(s)), b0 = smem_u32(sB(s));
#pragma unroll
          for (int k = 0; k < G_BK / 16; ++k)
#pragma unroll
            for (int a = 0; a < C::MSUB; ++a)
              umma_bf16_ss(d + a * G_BN, sdesc_k_sw128(a0 + a * G_A_BYTES + 32 * k), sdesc_k_sw128(b0 + 32 * k),
                           idesc, (kb | k) != 0);
          umma_commit(bar_empty + 8 * s);
          if (++s == S) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(bar_tfull + 8 * acc);
        if (++acc == C::NBUF) {
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
    const int quad = warp & 3;
    int acc = 0;
    uint32_t aph = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      int mb, nb;
      tile_coords(tile, p.m_tiles, p.n_tiles, p.group_m, mb, nb);
      if (!mbar_wait(bar_tfull + 8 * acc, aph, ec, kErrGemmEpilogue)) break;
      tc_fence_after();
#pragma unroll 1
      for (int a = 0; a < C::MSUB; ++a) {
        const int row = mb * C::BM + a * 128 + quad * 32 + lane;
        gemm_epilogue<EPI, INT8 ? 16 : 32, BN>(p, tmem_base + (acc * C::MSUB + a) * G_BN + ((quad * 32) << 16), row,
                                               nb);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
      if (++acc == C::NBUF) {
        acc = 0;
        aph ^= 1;
      }
    }
  } else if (INT8) {
    // DQ_GROUPS groups of dequant warps take the CTA's (tile, kb) stages in turn: group g
    // dequantises stages g, g + DQ_GROUPS, g + 2 DQ_GROUPS, ...  A warp loads the codes, scales and qbias of its
    // next stage right after the proxy fence of the current one, into the registers it has just
    // consumed, and they arrive while the other group works.  So no load is in flight when a
    // warp issues its fence: the fence that hands a B tile to the tensor core waits for the
    // warp's shared stores alone.
    const int grp = (threadIdx.x - 192) / DQ_THREADS;
    const int t = (threadIdx.x - 192) % DQ_THREADS;
    struct Cursor {
      int tile, kb, nb;
    };
    auto advance = [&](Cursor& c) {
      if (++c.kb == p.kb_count) {
        c.kb = 0;
        c.tile += gridDim.x;
        int mb;
        if (c.tile < p.num_tiles) tile_coords(c.tile, p.m_tiles, p.n_tiles, p.group_m, mb, c.nb);
      }
    };
    const uint8_t* wcodes = static_cast<const uint8_t*>(p.wcodes);
    auto prefetch = [&](const Cursor& c, DqStage& d) {
      if (c.tile < p.num_tiles) {
        int r0, r1;
        b_tile_rows<EPI>(p, c.nb, r0, r1);
        dq_load_stage(p, wcodes, r0, r1, c.kb, t, d);
      }
    };
    Cursor cur{static_cast<int>(blockIdx.x), 0, 0};
    if (cur.tile < p.num_tiles) {
      int mb;
      tile_coords(cur.tile, p.m_tiles, p.n_tiles, p.group_m, mb, cur.nb);
    }
    int q = grp;  // stage index in the CTA's sequence: ring slot q % S, phase (q / S) & 1
    for (int i = 0; i < grp; ++i) advance(cur);
    DqStage d;
    prefetch(cur, d);
    bool ok = true;
    while (cur.tile < p.num_tiles) {
      const int s = q % S;
      if (!mbar_wait(bar_empty + 8 * s, ((q / S) & 1) ^ 1, ec, kErrGemmDequant)) {
        ok = false;
        break;
      }
      dequant_stage(smem_u32(sB(s)), d, t);
      fence_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ready + 8 * s);
      for (int i = 0; i < DQ_GROUPS; ++i) advance(cur);
      q += DQ_GROUPS;
      prefetch(cur, d);
    }
    (void)ok;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------------------ host side

CUresult tensor_map_encode_tiled(CUtensorMap* m, CUtensorMapDataType dt, cuuint32_t rank, void* addr,
                                 const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                                 const cuuint32_t* estr, CUtensorMapInterleave il, CUtensorMapSwizzle sw,
                                 CUtensorMapL2promotion l2, CUtensorMapFloatOOBfill oob) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return CUDA_ERROR_NOT_FOUND;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn(m, dt, rank, addr, dims, strides, box, estr, il, sw, l2, oob);
}

static bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
                      uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = tensor_map_encode_tiled(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                                      CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

template <int EPI, bool INT8, int BN = G_BN>
static cudaError_t launch_tc(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, cudaStream_t st) {
  using C = GemmCfg<INT8, BN>;
  static bool configured = false;  // per instantiation; the attribute is per function, not per device
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_tc_kernel<EPI, INT8, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int grid = min(p.num_tiles, num_sms());
  gemm_tc_kernel<EPI, INT8, BN><<<grid, C::THREADS, C::SMEM, st>>>(ta, tb, p);
  return cudaGetLastError();
}

cudaError_t launch_linear_tc(const LinearArgs& a, cudaStream_t st) {
  if (a.M <= 0) return cudaSuccess;
  GemmParams p{};
  p.M = a.M;
  p.K = a.K;
  p.n_y = a.n_y;
  p.m_tiles = cdiv(a.M, a.int8 ? GemmCfg<true>::BM : GemmCfg<false>::BM);
  const bool sw = a.epi == kEpiSwiglu;
  // Column-tile width: 256, or 192 for the bf16 plain / gate+residual linears when that fills
  // the SMs' last wave clearly better -- fewer column-width units per SM over the whole launch,
  // (whole waves of 148 tiles) x width, by more than 3% (the narrower tile costs some per-tile
  // overhead).  1,829 rows x 5376 columns: 315 tiles of 256 = 3 waves (768) against 420 of
  // 192 = 3 waves (576).
  int bn = G_BN;
  if (!a.int8 && (a.epi == kEpiBias || a.epi == kEpiGateRes)) {
    const long long nsm = num_sms();
    auto cost = [&](int w) { return cdiv(static_cast<long long>(p.m_tiles) * cdiv(a.n_y, w), nsm) * w; };
    if (cost(192) * 100 < cost(G_BN) * 97) bn = 192;
  }
  p.b_row_step = sw ? 128 : bn;
  p.b_row1_off = sw ? a.n_y : 128;
  p.n_tiles = cdiv(a.n_y, p.b_row_step);
  p.num_tiles = p.m_tiles * p.n_tiles;
  p.kb_count = cdiv(a.K, G_BK);
  {
    const int bm = a.int8 ? GemmCfg<true>::BM : GemmCfg<false>::BM;
    const size_t a_rows_bytes = static_cast<size_t>(bm) * a.K * 2;
    int gm = static_cast<int>(kRasterABytes / (a_rows_bytes > 0 ? a_rows_bytes : 1));
    p.group_m = gm < 4 ? 4 : (gm > p.m_tiles ? p.m_tiles : gm);
    if (p.group_m < 1) p.group_m = 1;
  }
  p.bias = a.bias;
  p.y = a.y;
  p.ldy = a.ldy;
  p.res = a.res;
  p.gate = a.gate;
  p.m_gate = a.m_gate;
  p.wcodes = a.w;
  p.wscale = a.wscale;
  p.wqbias = a.wqbias;
  p.groups = a.K / 32;
  p.err = a.err;
  int w_rows = sw ? 2 * a.n_y : a.n_y;
  if (a.epi == kEpiQkv) {
    // n_y = 3 * nh * 128 weight rows, tiled as nh q|k tiles and ceil(nh / 2) v tiles
    p.nh = a.qkv.nh;
    p.n_tiles = a.qkv.nh + (a.qkv.nh + 1) / 2;
    p.num_tiles = p.m_tiles * p.n_tiles;
    p.cs = a.qkv.cs;
    p.qn = a.qkv.qn;
    p.kn = a.qkv.kn;
    p.qk_eps = a.qkv.eps;
    p.q = a.qkv.q;
    p.k = a.qkv.k;
    p.vt = a.qkv.vt;
    p.ld_vt = a.qkv.ld_vt;
    w_rows = a.n_y;
  }
  p.w_rows = w_rows;

  CUtensorMap ta, tb;
  if (!encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, a.K, a.M, static_cast<uint64_t>(a.lda) * 2, G_BK, G_BM,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (a.int8) {
    if (!encode_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w, a.K, w_rows, static_cast<uint64_t>(a.K), G_BK, 128,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    if (!encode_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.w, a.K, w_rows, static_cast<uint64_t>(a.K) * 2, G_BK,
                   bn == G_BN ? 128 : 64, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  if (bn == 192) return a.epi == kEpiBias ? launch_tc<kEpiBias, false, 192>(ta, tb, p, st)
                                          : launch_tc<kEpiGateRes, false, 192>(ta, tb, p, st);
  switch (a.epi * 2 + (a.int8 ? 1 : 0)) {
    case kEpiBias * 2: return launch_tc<kEpiBias, false>(ta, tb, p, st);
    case kEpiBias * 2 + 1: return launch_tc<kEpiBias, true>(ta, tb, p, st);
    case kEpiSwiglu * 2: return launch_tc<kEpiSwiglu, false>(ta, tb, p, st);
    case kEpiSwiglu * 2 + 1: return launch_tc<kEpiSwiglu, true>(ta, tb, p, st);
    case kEpiGateRes * 2: return launch_tc<kEpiGateRes, false>(ta, tb, p, st);
    case kEpiGateRes * 2 + 1: return launch_tc<kEpiGateRes, true>(ta, tb, p, st);
    case kEpiQkv * 2: return launch_tc<kEpiQkv, false>(ta, tb, p, st);
    case kEpiQkv * 2 + 1: return launch_tc<kEpiQkv, true>(ta, tb, p, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace h3
