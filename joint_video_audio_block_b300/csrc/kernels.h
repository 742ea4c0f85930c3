// Internal launcher declarations shared by the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include "common.cuh"

namespace h3 {

// A row's modulation vector m lives at table_b[tidx[r]*t_stride + (6*tag[r] + m)*H + c].
struct TableRef {
  const bf16* table_b;
  long long t_stride;
  const uint8_t* tag;
  const int32_t* tidx;
};

enum Epilogue : int { kEpiBias = 0, kEpiSwiglu = 1, kEpiGateRes = 2, kEpiQkv = 3 };

// Fused QKV epilogue (head_dim 128): per-head RMSNorm of q and k (optional), rotary embedding
// from the per-row cos/sin table, q and k written head-major, v written transposed.
struct QkvOut {
  int nh;
  const float2* cs;  // [M][64]
  const bf16* qn;    // [128] or null
  const bf16* kn;
  float eps;
  bf16* q;           // [nh][M][128]
  bf16* k;
  bf16* vt;          // [nh][128][ld_vt]
  int ld_vt;
};

// y = epilogue(x W^T + b).  W is bf16 [n_w_rows, K] or INT8-g32 codes + per-group scale/qbias.
struct LinearArgs {
  const bf16* x;
  int lda;
  int M;        // rows of x
  int K;        // reduction length
  int n_y;      // output columns (n_out, or n_out/2 for SwiGLU)
  bool int8;
  const void* w;         // bf16 [n_w_rows, K] or u8 [n_w_rows, K]
  const bf16* wscale;    // int8: [n_w_rows, K/32]
  const bf16* wqbias;    // int8: [n_w_rows, K/32]
  const bf16* bias;      // [n_w_rows] or null
  bf16* y;
  int ldy;
  int epi;
  const bf16* res;       // gate-residual input (stride ldy)
  TableRef gate;         // gate-residual gate
  int m_gate;
  QkvOut qkv;            // kEpiQkv outputs
  unsigned* err;
};

cudaError_t launch_adaln_modulate(const bf16* x, bf16* xn, int n_rows, int H, float eps, TableRef tr, int m_shift,
                                  int m_scale, cudaStream_t st);

cudaError_t launch_rope_table(const float* pos, float2* cs, int n_rows, int hd, const int sections[3], float theta,
                              cudaStream_t st);

cudaError_t launch_qknorm_rope(const bf16* qkv, const float2* cs, const bf16* qn, const bf16* kn, float eps, bf16* q,
                               bf16* k, bf16* vt, int ld_vt, int n_rows, int nh, int hd, cudaStream_t st);

// table[t * t_stride + b * n_out + j] = bf16(W[b][j] . temb[t] + bias[b][j]) for b < n_blocks
// (bias may be null, or hold null entries); temb 16-byte aligned, Dt % 8 == 0.
cudaError_t launch_modcache(const float* temb, int T, int Dt, const bf16* const* W, const bf16* const* bias,
                            int n_blocks, int n_out, bf16* table, long long t_stride, unsigned* err,
                            cudaStream_t st);

cudaError_t launch_linear_ref(const LinearArgs& a, cudaStream_t st);
cudaError_t launch_linear_tc(const LinearArgs& a, cudaStream_t st);

cudaError_t launch_attention_ref(const bf16* q, const bf16* k, const bf16* vt, int ld_vt, bf16* o, int n_rows, int nh,
                                 int hd, cudaStream_t st);
cudaError_t launch_attention_tc(const bf16* q, const bf16* k, const bf16* vt, int ld_vt, bf16* o, int n_rows, int nh,
                                int hd, unsigned* err, cudaStream_t st);
// block-sparse: mask u8 [nh][ceil(n/128)][ceil(n/128)], nonzero = keep (query tile, key tile)
cudaError_t launch_attention_sparse_tc(const bf16* q, const bf16* k, const bf16* vt, int ld_vt, bf16* o, int n_rows,
                                       int nh, int hd, const uint8_t* mask, unsigned* err, cudaStream_t st);

int num_sms();

// device address of the library's error word on the current device (api.cu)
unsigned* h3_error_word_ptr();

// measurement hooks (timer.cu): record the armed start / stop events around one launch
void timer_mark_begin(cudaStream_t st);
void timer_mark_end(cudaStream_t st);

// cuTensorMapEncodeTiled fetched through the runtime's driver entry point (the library does not
// link libcuda directly, so it loads on machines without a driver).
CUresult tensor_map_encode_tiled(CUtensorMap* m, CUtensorMapDataType dt, cuuint32_t rank, void* addr,
                                 const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                                 const cuuint32_t* estr, CUtensorMapInterleave il, CUtensorMapSwizzle sw,
                                 CUtensorMapL2promotion l2, CUtensorMapFloatOOBfill oob);

}  // namespace h3
