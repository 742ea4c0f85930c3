// C ABI of libh3 (declared in include/h3.h): argument checks, workspace plan, kernel order.
//
// The block follows "minimax-h3-mlx" README, "Architecture" / "AdaLN: measure, do not
// reason" / "Validation":
//   xn = LN(x)(1 + scale_msa) + shift_msa            adaln_modulate
//   qkv = xn Wqkv^T + b                               tcgen05 GEMM
//   q, k = RoPE(RMSNorm(.)), v^T                      in that GEMM's epilogue (head_dim 128), else
//                                                     a bias epilogue + qknorm_rope
//   o = softmax(q k^T / sqrt(hd)) v                   tcgen05 attention
//   x' = x + gate_msa (o Wo^T + bo)                   tcgen05 GEMM, gate+residual epilogue
//   xn = LN(x')(1 + scale_mlp) + shift_mlp            adaln_modulate
//   h = silu(g) v, [g | v] = xn W1^T + b1             tcgen05 GEMM, SwiGLU epilogue
//   x'' = x' + gate_mlp (h W2^T + b2)                 tcgen05 GEMM, gate+residual epilogue
// Activation arenas follow their lifetimes inside the block ("H3-metal" README, "Scheduling
// and activation memory"): the QKV arena is reused for the SwiGLU activation, and the
// attention-branch output x' is written straight into x_out.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <vector>

#include "../../include/h3.h"
#include "kernels.h"

namespace h3 {

__device__ unsigned g_error_word;  // first error site recorded by a bounded device wait

unsigned* error_word();
unsigned* h3_error_word_ptr() { return error_word(); }

// Device address of g_error_word on the current device, looked up once per device and cached
// (host threads may race on the first lookup; they all store the same address).
unsigned* error_word() {
  static std::atomic<unsigned*> ptr[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  unsigned* w = ptr[dev].load(std::memory_order_acquire);
  if (!w) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess || !p) return nullptr;
    w = static_cast<unsigned*>(p);
    ptr[dev].store(w, std::memory_order_release);
  }
  return w;
}

static size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
// int32 / float32 arrays the kernels read element-wise (tidx, pos, latents): 4-byte aligned
static bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }
static int ld_vt_for(int n_rows) { return (n_rows + 63) / 64 * 64; }

struct Workspace {
  float2* cs;
  bf16* xn;
  bf16* qkv;  // also the SwiGLU activation
  bf16* q;
  bf16* k;
  bf16* vt;
  bf16* o;
  size_t bytes;
};

static Workspace plan(const h3_dims& d, int n, void* base) {
  const size_t N = static_cast<size_t>(n);
  const size_t H = d.hidden, I = static_cast<size_t>(d.heads) * d.head_dim, F = d.ffn, hd = d.head_dim;
  const size_t wide = (3 * I > F ? 3 * I : F);
  size_t off = 0;
  Workspace w{};
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += align256(bytes);
    return o;
  };
  const size_t o_cs = take(N * (hd / 2) * sizeof(float2));
  const size_t o_xn = take(N * H * 2);
  const size_t o_qkv = take(N * wide * 2);
  const size_t o_q = take(N * I * 2);
  const size_t o_k = take(N * I * 2);
  const size_t o_vt = take(static_cast<size_t>(d.heads) * hd * ld_vt_for(n) * 2);
  const size_t o_o = take(N * I * 2);
  w.bytes = off;
  if (base) {
    char* b = static_cast<char*>(base);
    w.cs = reinterpret_cast<float2*>(b + o_cs);
    w.xn = reinterpret_cast<bf16*>(b + o_xn);
    w.qkv = reinterpret_cast<bf16*>(b + o_qkv);
    w.q = reinterpret_cast<bf16*>(b + o_q);
    w.k = reinterpret_cast<bf16*>(b + o_k);
    w.vt = reinterpret_cast<bf16*>(b + o_vt);
    w.o = reinterpret_cast<bf16*>(b + o_o);
  }
  return w;
}

static bool dims_ok(const h3_dims* d) {
  if (!d) return false;
  if (d->hidden <= 0 || d->hidden % 64 || d->hidden > 8192) return false;
  if (d->heads <= 0 || (d->head_dim != 64 && d->head_dim != 128)) return false;
  if ((d->heads * d->head_dim) % 64) return false;
  if (d->ffn <= 0 || d->ffn % 128) return false;
  if (d->n_tags <= 0 || d->n_tags > 255) return false;
  const int* s = d->rope_sections;
  if (s[0] < 0 || s[1] < 0 || s[2] < 0 || s[0] + s[1] + s[2] != d->head_dim / 2) return false;
  if (!(d->rope_theta > 0.f) || !(d->ln_eps >= 0.f) || !(d->qk_eps >= 0.f)) return false;
  return true;
}

// Host checks shared by h3_qknorm_rope and h3_qknorm_rope_static: the geometry, null pointers,
// and the alignment qknorm_rope_kernel's vector accesses need -- qkv, q_out and k_out 16 bytes
// (8-byte word loads / stores per lane at head_dim 128), vt_out 16 bytes with ld_vt % 8 == 0
// (16-byte transposed stores), pos 4 bytes, the norm weights 2 bytes.
bool qknorm_rope_args_ok(const h3_dims* d, const void* qkv, const float* pos, const void* q_norm,
                         const void* k_norm, const void* q_out, const void* k_out, const void* vt_out, int ld_vt,
                         int n_rows) {
  if (!dims_ok(d) || !qkv || !pos || !q_out || !k_out || !vt_out || n_rows < 0) return false;
  if (ld_vt < n_rows || ld_vt % 8 || ((q_norm == nullptr) != (k_norm == nullptr))) return false;
  if (!aligned16(qkv) || !aligned16(q_out) || !aligned16(k_out) || !aligned16(vt_out)) return false;
  if ((reinterpret_cast<uintptr_t>(pos) & 3) || (reinterpret_cast<uintptr_t>(q_norm) & 1) ||
      (reinterpret_cast<uintptr_t>(k_norm) & 1))
    return false;
  return true;
}

static bool linear_ok(const h3_linear& l, int n_out, int k) {
  if (l.n_out != n_out || l.k != k || !l.w || !aligned16(l.w)) return false;
  if (l.bias && !aligned16(l.bias)) return false;
  if (l.fmt == H3_W_BF16) return k % 8 == 0;
  if (l.fmt == H3_W_INT8_G32) return k % 32 == 0 && l.scale && l.qbias;
  return false;
}

static h3_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return H3_OK;
  if (e == cudaErrorInvalidValue) return H3_EINVAL;
  return H3_ECUDA;
}

static LinearArgs make_linear(const h3_linear& l, int epi, const bf16* x, int lda, bf16* y, int ldy, int M) {
  LinearArgs a{};
  a.x = x;
  a.lda = lda;
  a.M = M;
  a.K = l.k;
  a.n_y = epi == kEpiSwiglu ? l.n_out / 2 : l.n_out;
  a.int8 = l.fmt == H3_W_INT8_G32;
  a.w = l.w;
  a.wscale = static_cast<const bf16*>(l.scale);
  a.wqbias = static_cast<const bf16*>(l.qbias);
  a.bias = static_cast<const bf16*>(l.bias);
  a.y = y;
  a.ldy = ldy;
  a.epi = epi;
  a.err = error_word();
  return a;
}

static cudaError_t run_linear(const LinearArgs& a, unsigned flags, cudaStream_t st) {
  return (flags & H3_F_UNFUSED) ? launch_linear_ref(a, st) : launch_linear_tc(a, st);
}

static bool check_indices(const uint8_t* tag, const int32_t* tidx, int n, int n_tags, int T) {
  std::vector<uint8_t> ht(n);
  std::vector<int32_t> hi(n);
  if (cudaMemcpy(ht.data(), tag, n, cudaMemcpyDeviceToHost) != cudaSuccess) return false;
  if (cudaMemcpy(hi.data(), tidx, sizeof(int32_t) * n, cudaMemcpyDeviceToHost) != cudaSuccess) return false;
  for (int i = 0; i < n; ++i)
    if (ht[i] >= n_tags || hi[i] < 0 || hi[i] >= T) return false;
  return true;
}

// a2 + a3: QKV projection, QK-norm and rotary embedding, q / k head-major and v transposed.
// head_dim 128 on the tensor-core path: one GEMM whose epilogue does the norm and rotation
// (the projection never goes to memory); otherwise the projection is written to `qkv_tmp`
// ([n, 3 nh hd] bf16) and a second kernel does the norm and rotation.
static cudaError_t qkv_step(const h3_dims& d, const h3_linear& wqkv, const bf16* xn, const float2* cs, const bf16* qn,
                            const bf16* kn, bf16* q, bf16* k, bf16* vt, int ld_vt, int n, bf16* qkv_tmp,
                            unsigned flags, cudaStream_t st) {
  const int H = d.hidden, I = d.heads * d.head_dim;
  if (!(flags & H3_F_UNFUSED) && d.head_dim == 128) {
    LinearArgs a = make_linear(wqkv, kEpiQkv, xn, H, nullptr, 0, n);
    a.qkv = QkvOut{d.heads, cs, qn, kn, d.qk_eps, q, k, vt, ld_vt};
    return launch_linear_tc(a, st);
  }
  LinearArgs a = make_linear(wqkv, kEpiBias, xn, H, qkv_tmp, 3 * I, n);
  cudaError_t e = run_linear(a, flags, st);
  if (e != cudaSuccess) return e;
  return launch_qknorm_rope(qkv_tmp, cs, qn, kn, d.qk_eps, q, k, vt, ld_vt, n, d.heads, d.head_dim, st);
}

// one block given a planned workspace whose rotary table is already filled
static h3_status block_core(const h3_dims& d, const h3_block_w& w, const bf16* table_b, long long t_stride,
                            const bf16* x_in, bf16* x_out, int n, const uint8_t* tag, const int32_t* tidx,
                            const Workspace& ws, unsigned flags, cudaStream_t st) {
  const int H = d.hidden, I = d.heads * d.head_dim, F = d.ffn;
  TableRef tr{table_b, t_stride, tag, tidx};
  cudaError_t e;
  // a1
  if ((e = launch_adaln_modulate(x_in, ws.xn, n, H, d.ln_eps, tr, 0, 1, st)) != cudaSuccess) return cuda_status(e);
  // a2 + a3
  const bool qk = !(flags & H3_F_NO_QKNORM) && w.q_norm && w.k_norm;
  if ((e = qkv_step(d, w.qkv, ws.xn, ws.cs, qk ? static_cast<const bf16*>(w.q_norm) : nullptr,
                    qk ? static_cast<const bf16*>(w.k_norm) : nullptr, ws.q, ws.k, ws.vt, ld_vt_for(n), n, ws.qkv,
                    flags, st)) != cudaSuccess)
    return cuda_status(e);
  LinearArgs a;
  // a4
  timer_mark_begin(st);
  e = (flags & H3_F_UNFUSED)
          ? launch_attention_ref(ws.q, ws.k, ws.vt, ld_vt_for(n), ws.o, n, d.heads, d.head_dim, st)
          : launch_attention_tc(ws.q, ws.k, ws.vt, ld_vt_for(n), ws.o, n, d.heads, d.head_dim, error_word(), st);
  if (e != cudaSuccess) return cuda_status(e);
  timer_mark_end(st);
  // a5: x_out = x_in + gate_msa * (o Wo^T + bo)
  a = make_linear(w.o, kEpiGateRes, ws.o, I, x_out, H, n);
  a.res = x_in;
  a.gate = tr;
  a.m_gate = 2;
  if ((e = run_linear(a, flags, st)) != cudaSuccess) return cuda_status(e);
  // a6
  if ((e = launch_adaln_modulate(x_out, ws.xn, n, H, d.ln_eps, tr, 3, 4, st)) != cudaSuccess) return cuda_status(e);
  // a7: h = silu(g) * v into the QKV arena
  a = make_linear(w.fc1, kEpiSwiglu, ws.xn, H, ws.qkv, F, n);
  if ((e = run_linear(a, flags, st)) != cudaSuccess) return cuda_status(e);
  // a8: x_out += gate_mlp * (h W2^T + b2)
  a = make_linear(w.fc2, kEpiGateRes, ws.qkv, F, x_out, H, n);
  a.res = x_out;
  a.gate = tr;
  a.m_gate = 5;
  if ((e = run_linear(a, flags, st)) != cudaSuccess) return cuda_status(e);
  return H3_OK;
}

static bool block_w_ok(const h3_dims& d, const h3_block_w* w) {
  if (!w) return false;
  const int H = d.hidden, I = d.heads * d.head_dim, F = d.ffn;
  if (!linear_ok(w->qkv, 3 * I, H) || !linear_ok(w->o, H, I) || !linear_ok(w->fc1, 2 * F, H) ||
      !linear_ok(w->fc2, H, F))
    return false;
  if ((w->q_norm == nullptr) != (w->k_norm == nullptr)) return false;
  return true;
}

}  // namespace h3

using namespace h3;

extern "C" {

size_t h3_workspace_size(const h3_dims* dims, int n_rows) {
  if (!dims_ok(dims) || n_rows < 0) return 0;
  return plan(*dims, n_rows, nullptr).bytes;
}

const char* h3_status_str(h3_status s) {
  switch (s) {
    case H3_OK: return "ok";
    case H3_EINVAL: return "invalid argument";
    case H3_EUNSUPPORTED: return "unsupported";
    case H3_ECUDA: return "CUDA error";
    case H3_ETIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

h3_status h3_last_device_error(void* stream, unsigned* site) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return H3_ECUDA;
  unsigned* w = error_word();
  if (!w) return H3_ECUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return H3_ECUDA;
  if (site) *site = v;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return H3_ECUDA;
    return H3_ETIMEOUT;
  }
  return H3_OK;
}

h3_status h3_modcache_build(const h3_dims* dims, const float* temb, int T, int Dt, const void* const* adaln_w,
                            const void* const* adaln_b, int n_blocks, void* table, void* stream) {
  if (!dims_ok(dims) || !temb || !aligned16(temb) || T <= 0 || Dt <= 0 || Dt % 8 || !adaln_w || n_blocks <= 0 ||
      !table)
    return H3_EINVAL;
  for (int b = 0; b < n_blocks; ++b)
    if (!adaln_w[b] || !aligned16(adaln_w[b]) || (adaln_b && adaln_b[b] && (reinterpret_cast<uintptr_t>(adaln_b[b]) & 1)))
      return H3_EINVAL;
  const int n_out = 18 * dims->hidden;
  const long long t_stride = static_cast<long long>(n_blocks) * n_out;
  return cuda_status(launch_modcache(temb, T, Dt, reinterpret_cast<const bf16* const*>(adaln_w),
                                     reinterpret_cast<const bf16* const*>(adaln_b), n_blocks, n_out,
                                     static_cast<bf16*>(table), t_stride, error_word(),
                                     static_cast<cudaStream_t>(stream)));
}

h3_status h3_adaln_modulate(const h3_dims* dims, const void* x, void* xn, int n_rows, const void* table_b,
                            long long t_stride, int m_shift, int m_scale, const uint8_t* tag, const int32_t* tidx,
                            void* stream) {
  if (!dims_ok(dims) || n_rows < 0 || !x || !xn || x == xn || !table_b || !tag || !tidx) return H3_EINVAL;
  if (m_shift < 0 || m_shift > 5 || m_scale < 0 || m_scale > 5 || !aligned16(x) || !aligned16(xn) ||
      !aligned16(table_b) || t_stride % 8 || !aligned4(tidx))
    return H3_EINVAL;
  TableRef tr{static_cast<const bf16*>(table_b), t_stride, tag, tidx};
  return cuda_status(launch_adaln_modulate(static_cast<const bf16*>(x), static_cast<bf16*>(xn), n_rows,
                                           dims->hidden, dims->ln_eps, tr, m_shift, m_scale,
                                           static_cast<cudaStream_t>(stream)));
}

h3_status h3_linear_forward(const h3_linear* lin, int epilogue, const void* x, int lda, void* y, int ldy, int n_rows,
                            const void* res, const void* table_b, long long t_stride, int m_gate, const uint8_t* tag,
                            const int32_t* tidx, unsigned flags, void* stream) {
  if (!lin || !x || !y || n_rows < 0 || epilogue < 0 || epilogue > 2) return H3_EINVAL;
  if (!linear_ok(*lin, lin->n_out, lin->k) || lin->n_out <= 0 || lin->k <= 0) return H3_EINVAL;
  const int n_y = epilogue == H3_EPI_SWIGLU ? lin->n_out / 2 : lin->n_out;
  if (epilogue == H3_EPI_SWIGLU && lin->n_out % 2) return H3_EINVAL;
  if (lda < lin->k || lda % 8 || ldy < n_y || ldy % 8 || !aligned16(x) || !aligned16(y)) return H3_EINVAL;
  if (n_y % 8) return H3_EINVAL;
  LinearArgs a = make_linear(*lin, epilogue, static_cast<const bf16*>(x), lda, static_cast<bf16*>(y), ldy, n_rows);
  if (epilogue == H3_EPI_GATE_RES) {
    if (!res || !table_b || !tag || !tidx || m_gate < 0 || m_gate > 5 || !aligned16(res) || !aligned16(table_b) ||
        t_stride % 8 || !aligned4(tidx))
      return H3_EINVAL;
    a.res = static_cast<const bf16*>(res);
    a.gate = TableRef{static_cast<const bf16*>(table_b), t_stride, tag, tidx};
    a.m_gate = m_gate;
  }
  return cuda_status(run_linear(a, flags, static_cast<cudaStream_t>(stream)));
}

h3_status h3_qknorm_rope(const h3_dims* dims, const void* qkv, const float* pos, const void* q_norm,
                         const void* k_norm, void* q_out, void* k_out, void* vt_out, int ld_vt, int n_rows,
                         void* workspace, size_t ws_bytes, void* stream) {
  if (!qknorm_rope_args_ok(dims, qkv, pos, q_norm, k_norm, q_out, k_out, vt_out, ld_vt, n_rows) || !workspace)
    return H3_EINVAL;
  const size_t need = static_cast<size_t>(n_rows) * (dims->head_dim / 2) * sizeof(float2);
  if (ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15)) return H3_EINVAL;
  if (n_rows == 0) return H3_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float2* cs = static_cast<float2*>(workspace);
  cudaError_t e = launch_rope_table(pos, cs, n_rows, dims->head_dim, dims->rope_sections, dims->rope_theta, st);
  if (e == cudaSuccess)
    e = launch_qknorm_rope(static_cast<const bf16*>(qkv), cs, static_cast<const bf16*>(q_norm),
                           static_cast<const bf16*>(k_norm), dims->qk_eps, static_cast<bf16*>(q_out),
                           static_cast<bf16*>(k_out), static_cast<bf16*>(vt_out), ld_vt, n_rows, dims->heads,
                           dims->head_dim, st);
  return cuda_status(e);
}

size_t h3_qkv_project_workspace_size(const h3_dims* dims, int n_rows) {
  if (!dims_ok(dims) || n_rows < 0) return 0;
  const size_t N = static_cast<size_t>(n_rows);
  return align256(N * (dims->head_dim / 2) * sizeof(float2)) +
         N * 3 * static_cast<size_t>(dims->heads) * dims->head_dim * 2;
}

h3_status h3_qkv_project(const h3_dims* dims, const h3_linear* wqkv, const void* xn, const float* pos,
                         const void* q_norm, const void* k_norm, void* q_out, void* k_out, void* vt_out, int ld_vt,
                         int n_rows, void* workspace, size_t ws_bytes, unsigned flags, void* stream) {
  if (!dims_ok(dims) || !wqkv || !xn || !pos || !q_out || !k_out || !vt_out || n_rows < 0 || !workspace)
    return H3_EINVAL;
  const int H = dims->hidden, I = dims->heads * dims->head_dim;
  if (!linear_ok(*wqkv, 3 * I, H) || ld_vt < n_rows || ld_vt % 8 || !aligned16(xn) || !aligned16(q_out) ||
      !aligned16(k_out) || !aligned16(vt_out) || ((q_norm == nullptr) != (k_norm == nullptr)) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255))
    return H3_EINVAL;
  if (ws_bytes < h3_qkv_project_workspace_size(dims, n_rows)) return H3_EINVAL;
  if (n_rows == 0) return H3_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float2* cs = static_cast<float2*>(workspace);
  bf16* tmp = reinterpret_cast<bf16*>(static_cast<char*>(workspace) +
                                      align256(static_cast<size_t>(n_rows) * (dims->head_dim / 2) * sizeof(float2)));
  cudaError_t e = launch_rope_table(pos, cs, n_rows, dims->head_dim, dims->rope_sections, dims->rope_theta, st);
  if (e == cudaSuccess)
    e = qkv_step(*dims, *wqkv, static_cast<const bf16*>(xn), cs, static_cast<const bf16*>(q_norm),
                 static_cast<const bf16*>(k_norm), static_cast<bf16*>(q_out), static_cast<bf16*>(k_out),
                 static_cast<bf16*>(vt_out), ld_vt, n_rows, tmp, flags, st);
  return cuda_status(e);
}

h3_status h3_attention(const h3_dims* dims, const void* q, const void* k, const void* vt, int ld_vt, void* o,
                       int n_rows, unsigned flags, void* stream) {
  if (!dims_ok(dims) || !q || !k || !vt || !o || n_rows < 0 || ld_vt < n_rows || ld_vt % 8) return H3_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o)) return H3_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bf16 *qb = static_cast<const bf16*>(q), *kb = static_cast<const bf16*>(k), *vb = static_cast<const bf16*>(vt);
  cudaError_t e = (flags & H3_F_UNFUSED)
                      ? launch_attention_ref(qb, kb, vb, ld_vt, static_cast<bf16*>(o), n_rows, dims->heads,
                                             dims->head_dim, st)
                      : launch_attention_tc(qb, kb, vb, ld_vt, static_cast<bf16*>(o), n_rows, dims->heads,
                                            dims->head_dim, error_word(), st);
  return cuda_status(e);
}

h3_status h3_attention_sparse(const h3_dims* dims, const void* q, const void* k, const void* vt, int ld_vt, void* o,
                              int n_rows, const uint8_t* tile_mask, void* stream) {
  if (!dims_ok(dims) || !q || !k || !vt || !o || !tile_mask || n_rows < 0 || ld_vt < n_rows || ld_vt % 8)
    return H3_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o)) return H3_EINVAL;
  return cuda_status(launch_attention_sparse_tc(static_cast<const bf16*>(q), static_cast<const bf16*>(k),
                                                static_cast<const bf16*>(vt), ld_vt, static_cast<bf16*>(o), n_rows,
                                                dims->heads, dims->head_dim, tile_mask, error_word(),
                                                static_cast<cudaStream_t>(stream)));
}

h3_status h3_block_forward(const h3_dims* dims, const h3_block_w* w, const void* table_b, long long t_stride, int T,
                           const void* x_in, void* x_out, int n_rows, const uint8_t* tag, const int32_t* tidx,
                           const float* pos, void* workspace, size_t ws_bytes, unsigned flags, void* stream) {
  if (!dims_ok(dims) || !block_w_ok(*dims, w) || !table_b || T <= 0 || t_stride % 8 || !x_in || !x_out ||
      n_rows < 0 || !tag || !tidx || !pos || !workspace)
    return H3_EINVAL;
  if (!aligned16(x_in) || !aligned16(x_out) || !aligned16(table_b) || !aligned4(tidx) || !aligned4(pos) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255))
    return H3_EINVAL;
  if (x_in != x_out) {
    const char *a = static_cast<const char*>(x_in), *b = static_cast<const char*>(x_out);
    const size_t len = static_cast<size_t>(n_rows) * dims->hidden * 2;
    if (a < b + len && b < a + len) return H3_EINVAL;
  }
  const Workspace ws = plan(*dims, n_rows, workspace);
  if (ws_bytes < ws.bytes) return H3_EINVAL;
  if (n_rows == 0) return H3_OK;
  if ((flags & H3_F_CHECK_INDEX) && !check_indices(tag, tidx, n_rows, dims->n_tags, T)) return H3_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_rope_table(pos, ws.cs, n_rows, dims->head_dim, dims->rope_sections, dims->rope_theta, st);
  if (e != cudaSuccess) return cuda_status(e);
  return block_core(*dims, *w, static_cast<const bf16*>(table_b), t_stride, static_cast<const bf16*>(x_in),
                    static_cast<bf16*>(x_out), n_rows, tag, tidx, ws, flags, st);
}

h3_status h3_trunk_forward(const h3_dims* dims, const h3_block_w* blocks, int n_blocks, const void* table, int T,
                           void* x, int n_rows, const uint8_t* tag, const int32_t* tidx, const float* pos,
                           void* workspace, size_t ws_bytes, unsigned flags, void* stream) {
  if (!dims_ok(dims) || !blocks || n_blocks <= 0 || !table || T <= 0 || !x || n_rows < 0 || !tag || !tidx || !pos ||
      !workspace)
    return H3_EINVAL;
  if (!aligned16(x) || !aligned16(table) || !aligned4(tidx) || !aligned4(pos) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255))
    return H3_EINVAL;
  for (int b = 0; b < n_blocks; ++b)
    if (!block_w_ok(*dims, &blocks[b])) return H3_EINVAL;
  const Workspace ws = plan(*dims, n_rows, workspace);
  if (ws_bytes < ws.bytes) return H3_EINVAL;
  if (n_rows == 0) return H3_OK;
  if ((flags & H3_F_CHECK_INDEX) && !check_indices(tag, tidx, n_rows, dims->n_tags, T)) return H3_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_rope_table(pos, ws.cs, n_rows, dims->head_dim, dims->rope_sections, dims->rope_theta, st);
  if (e != cudaSuccess) return cuda_status(e);
  const long long n18 = 18LL * dims->hidden;
  const long long t_stride = n18 * n_blocks;
  bf16* xb = static_cast<bf16*>(x);
  for (int b = 0; b < n_blocks; ++b) {
    const bf16* tb = static_cast<const bf16*>(table) + b * n18;
    h3_status s = block_core(*dims, blocks[b], tb, t_stride, xb, xb, n_rows, tag, tidx, ws, flags, st);
    if (s != H3_OK) return s;
  }
  return H3_OK;
}

}  // extern "C"

namespace {
// The model evaluation shared by both sampler transitions: the latent rows enter the hidden
// stream through their patch projections (text rows are copied in), then the trunk runs.
h3_status denoise_entry_trunk(const h3_dims* dims, const h3_block_w* blocks, int n_blocks, const void* table,
                              const void* table_f, int T, const h3_io_w* io, const void* text_x, const float* z_cond,
                              const float* z_video, const float* z_audio, void* x, const uint8_t* tag,
                              const int32_t* tidx, const float* pos, void* workspace, size_t ws_bytes, unsigned flags,
                              void* stream) {
  if (!dims_ok(dims) || !io || !x || !table_f || !tag || !tidx) return H3_EINVAL;
  const int H = dims->hidden;
  const int L = io->text_rows, C = io->cond_rows, A = io->audio_rows, V = io->video_rows;
  if (L < 0 || C < 0 || A < 0 || V < 0 || (L && !text_x) || (C && !z_cond) || (A && !z_audio) || (V && !z_video))
    return H3_EINVAL;
  // everything the entry projections and heads read, checked before the first launch
  const void* f32s[] = {z_cond, z_video, z_audio, io->patch_v, io->patch_v_b, io->patch_a, io->patch_a_b,
                        io->head_v, io->head_v_b, io->head_a, io->head_a_b};
  for (const void* f : f32s)
    if (!aligned4(f)) return H3_EINVAL;
  if (((C || V) && (!io->patch_v || !io->head_v)) || (A && (!io->patch_a || !io->head_a))) return H3_EINVAL;
  if (io->k_video <= 0 || io->k_video > 128 || io->k_audio <= 0 || io->k_audio > 128) return H3_EINVAL;
  if (!aligned16(table_f) || (L && !aligned16(text_x))) return H3_EINVAL;
  const int n = L + C + A + V;
  const size_t row_bytes = static_cast<size_t>(H) * 2;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* xb = static_cast<char*>(x);
  h3_status s = H3_OK;
  if (L && cudaMemcpyAsync(xb, text_x, L * row_bytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess) return H3_ECUDA;
  if (C && (s = h3_embed_rows(dims, z_cond, io->k_video, io->patch_v, io->patch_v_b, C, xb + L * row_bytes, stream)))
    return s;
  if (A && (s = h3_embed_rows(dims, z_audio, io->k_audio, io->patch_a, io->patch_a_b, A,
                              xb + static_cast<size_t>(L + C) * row_bytes, stream)))
    return s;
  if (V && (s = h3_embed_rows(dims, z_video, io->k_video, io->patch_v, io->patch_v_b, V,
                              xb + static_cast<size_t>(L + C + A) * row_bytes, stream)))
    return s;
  return h3_trunk_forward(dims, blocks, n_blocks, table, T, x, n, tag, tidx, pos, workspace, ws_bytes, flags, stream);
}
}  // namespace

extern "C" {

h3_status h3_denoise_step(const h3_dims* dims, const h3_block_w* blocks, int n_blocks, const void* table,
                          const void* table_f, int T, const h3_io_w* io, const void* text_x, const float* z_cond,
                          float* z_video, float* z_audio, void* x, const uint8_t* tag, const int32_t* tidx,
                          const float* pos, float dsigma_video, float dsigma_audio, void* workspace, size_t ws_bytes,
                          unsigned flags, void* stream) {
  h3_status s = denoise_entry_trunk(dims, blocks, n_blocks, table, table_f, T, io, text_x, z_cond, z_video, z_audio,
                                    x, tag, tidx, pos, workspace, ws_bytes, flags, stream);
  if (s) return s;
  const int L = io->text_rows, C = io->cond_rows, A = io->audio_rows, V = io->video_rows;
  const size_t row_bytes = static_cast<size_t>(dims->hidden) * 2;
  char* xb = static_cast<char*>(x);
  const long long tf_stride = 6LL * dims->hidden;
  // exit + Euler transition
  if (A && (s = h3_head_forward(dims, xb + static_cast<size_t>(L + C) * row_bytes, A, tag + (L + C), tidx + (L + C),
                                table_f, tf_stride, io->head_a, io->head_a_b, io->k_audio, nullptr, z_audio,
                                dsigma_audio, stream)))
    return s;
  if (V && (s = h3_head_forward(dims, xb + static_cast<size_t>(L + C + A) * row_bytes, V, tag + (L + C + A),
                                tidx + (L + C + A), table_f, tf_stride, io->head_v, io->head_v_b, io->k_video,
                                nullptr, z_video, dsigma_video, stream)))
    return s;
  return H3_OK;
}

h3_status h3_denoise_step_ms(const h3_dims* dims, const h3_block_w* blocks, int n_blocks, const void* table,
                             const void* table_f, int T, const h3_io_w* io, const void* text_x, const float* z_cond,
                             float* z_video, float* z_audio, float* d_prev_video, float* d_prev_audio, void* x,
                             const uint8_t* tag, const int32_t* tidx, const float* pos, const h3_ms_step* step_video,
                             const h3_ms_step* step_audio, void* workspace, size_t ws_bytes, unsigned flags,
                             void* stream) {
  if (!io || !step_video || !step_audio || (io->audio_rows && !d_prev_audio) || (io->video_rows && !d_prev_video))
    return H3_EINVAL;
  if (!aligned4(d_prev_video) || !aligned4(d_prev_audio) || !(step_video->sigma > 0.f) || !(step_audio->sigma > 0.f))
    return H3_EINVAL;
  h3_status s = denoise_entry_trunk(dims, blocks, n_blocks, table, table_f, T, io, text_x, z_cond, z_video, z_audio,
                                    x, tag, tidx, pos, workspace, ws_bytes, flags, stream);
  if (s) return s;
  const int L = io->text_rows, C = io->cond_rows, A = io->audio_rows, V = io->video_rows;
  const size_t row_bytes = static_cast<size_t>(dims->hidden) * 2;
  char* xb = static_cast<char*>(x);
  const long long tf_stride = 6LL * dims->hidden;
  // exit + res_multistep transition
  if (A && (s = h3_head_forward_ms(dims, xb + static_cast<size_t>(L + C) * row_bytes, A, tag + (L + C),
                                   tidx + (L + C), table_f, tf_stride, io->head_a, io->head_a_b, io->k_audio,
                                   step_audio, nullptr, z_audio, d_prev_audio, stream)))
    return s;
  if (V && (s = h3_head_forward_ms(dims, xb + static_cast<size_t>(L + C + A) * row_bytes, V, tag + (L + C + A),
                                   tidx + (L + C + A), table_f, tf_stride, io->head_v, io->head_v_b, io->k_video,
                                   step_video, nullptr, z_video, d_prev_video, stream)))
    return s;
  return H3_OK;
}

}  // extern "C"
