/*
 * libh3 -- the denoiser forward of the H3 joint audio+video DiT trunk on one B300 (sm_103a).
 *
 * C ABI.  Every pointer argument named "device" is a CUDA device pointer owned by the caller;
 * pointers named "host" are host memory.  The library allocates no device memory: scratch
 * space comes from the caller's workspace (the one exception, h3_qknorm_rope_static, uses a
 * fixed array that is part of the loaded library).  All compute calls are asynchronous on `stream`
 * (a cudaStream_t passed as void*; NULL = the legacy default stream) and return before the
 * GPU work finishes.  Tensors are dense and row-major unless a stride is given; "bf16" means
 * IEEE bfloat16 bit patterns (2 bytes), "f32" float32.
 *
 * Errors: every call returns an h3_status.  Shape, alignment and null-pointer violations are
 * detected on the host and return H3_EINVAL before anything is launched (bf16 tensors the
 * kernels move in 16-byte vectors must be 16-byte aligned where an entry point says so; every
 * f32 and i32 array must be 4-byte aligned); a CUDA launch error
 * returns H3_ECUDA.  Kernels never trap: a pipeline wait that exceeds its time limit records a
 * site code in the library's device error word and ends the launch; h3_last_device_error()
 * reports it.  Nothing aborts the process.
 *
 * Sources (page and section): "minimax-h3-mlx" README -- "Architecture" (packed sequence
 * [text | conditions | audio | video], per-row AdaLN modality tag, 50 blocks, hidden 5376,
 * 56 x 128 heads, SwiGLU 14336, 3D MM-RoPE), "AdaLN precompute" (ModulationCache,
 * adaln_proj 50 x [96768, 2688]), "AdaLN: measure, do not reason" (six modulation tensors,
 * x*(1+scale)+shift, x + gate*f(x)), "Validation" (per-head interleaved qkv rows, fused
 * [gate; value] fc1); "H3-metal" README -- "Exact DiT fusions", "Checkpoint layout and media
 * pipeline" (fused QK-norm + RoPE on interleaved qkv); "mlx-h3" README -- "Local model
 * layout" (weight-only INT8 group 32).
 */
#ifndef H3_H
#define H3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  H3_OK = 0,
  H3_EINVAL = 1,        /* bad shape, alignment, pointer or argument */
  H3_EUNSUPPORTED = 2,  /* valid request this build does not implement */
  H3_ECUDA = 3,         /* CUDA runtime / driver call failed */
  H3_ETIMEOUT = 4       /* a device pipeline wait ran out (see h3_last_device_error) */
} h3_status;

typedef enum { H3_W_BF16 = 0, H3_W_INT8_G32 = 1 } h3_wfmt;

/* flags for the block / trunk calls */
#define H3_F_UNFUSED 0x1u      /* run the plain CUDA-core reference kernels instead of tcgen05 */
#define H3_F_NO_QKNORM 0x2u    /* skip QK RMSNorm even if weights are given */
#define H3_F_CHECK_INDEX 0x4u  /* copy tag/tidx to the host and range-check them first (synchronises) */

/* Block geometry.  hidden H, heads nh, head_dim hd (64 or 128), ffn F, n_tags modality tags.
 * rope_sections: frequency pairs given to the (t, h, w) position axes, summing to hd/2.
 * Requirements: H % 64 == 0 and H <= 8192, (nh*hd) % 64 == 0, F % 128 == 0, 1 <= n_tags <= 255,
 * rope_theta > 0, ln_eps >= 0, qk_eps >= 0. */
typedef struct {
  int hidden, heads, head_dim, ffn, n_tags;
  int rope_sections[3];
  float rope_theta; /* 1e4 */
  float ln_eps;     /* LayerNorm eps, 1e-6 */
  float qk_eps;     /* QK RMSNorm eps, 1e-6 */
} h3_dims;

/* One linear layer y = x W^T + b with W [n_out, k] (checkpoint orientation).
 * H3_W_BF16:     w = device bf16 [n_out, k].
 * H3_W_INT8_G32: w = device u8 codes [n_out, k]; scale, qbias = device bf16 [n_out, k/32];
 *                W[o][c] = bf16(fma_f32(scale[o][c/32], w[o][c], qbias[o][c/32])); k % 32 == 0.
 * bias: device bf16 [n_out] or NULL.  Row strides must be multiples of 16 bytes. */
typedef struct {
  int fmt;
  const void* w;
  const void* scale;
  const void* qbias;
  const void* bias;
  int n_out, k;
} h3_linear;

/* One block's weights.  qkv: [3*nh*hd, H], rows interleaved per head ([h: q, k, v]);
 * o: [H, nh*hd]; fc1: [2F, H], first F rows = gate; fc2: [H, F].
 * q_norm, k_norm: device bf16 [hd] RMSNorm weights or NULL (no QK-norm). */
typedef struct {
  h3_linear qkv, o, fc1, fc2;
  const void* q_norm;
  const void* k_norm;
} h3_block_w;

/* Modulation table addressing.  The table holds, per timestep t and block b, 18*H bf16 values
 * read as 3 modality tags x 6 tensors x H, tensor order (shift_msa, scale_msa, gate_msa,
 * shift_mlp, scale_mlp, gate_mlp): entry (t, b, tag, m, c) is at
 *   table[t*t_stride + b*18*H + (6*tag + m)*H + c].
 * h3_modcache_build writes the packed layout [T][B][18][H] (t_stride = B*18*H). */

/* Bytes of workspace h3_block_forward / h3_trunk_forward need for n_rows rows. */
size_t h3_workspace_size(const h3_dims* dims, int n_rows);

/* a0 -- ModulationCache build ("minimax-h3-mlx" README, "AdaLN precompute").
 *   table[t][b][j] = bf16( sum_k adaln_w[b][j][k] * temb[t][k] + adaln_b[b][j] ),
 * fp32 accumulation, j < 18*H.
 * On the tensor cores: temb splits exactly into three bf16 terms and the three products
 * accumulate in fp32, so every product is exact and only the fp32 accumulation rounds.
 * temb: device f32 [T, Dt], 16-byte aligned; adaln_w: HOST array of n_blocks device pointers (16-byte aligned) to bf16 [18H, Dt];
 * adaln_b: HOST array of n_blocks device pointers to bf16 [18H] (array or entries may be NULL);
 * table: device bf16 [T][n_blocks][18H], written.  Dt % 8 == 0. */
h3_status h3_modcache_build(const h3_dims* dims, const float* temb, int T, int Dt, const void* const* adaln_w,
                            const void* const* adaln_b, int n_blocks, void* table, void* stream);

/* a1..a8 -- one DiT block over the packed sequence.
 * table_b: device pointer to this block's slice at t = 0 (table + b*18*H), t_stride as above,
 * T timesteps.  x_in, x_out: device bf16 [n_rows, H] (x_out may equal x_in; otherwise they must
 * not overlap).  tag: device u8 [n_rows] (< n_tags); tidx: device i32 [n_rows] (< T);
 * pos: device f32 [n_rows, 3] = (t, h, w) rotary position (1-D rows pass (p, p, p)).
 * workspace: device, >= h3_workspace_size bytes, 256-byte aligned. */
h3_status h3_block_forward(const h3_dims* dims, const h3_block_w* w, const void* table_b, long long t_stride, int T,
                           const void* x_in, void* x_out, int n_rows, const uint8_t* tag, const int32_t* tidx,
                           const float* pos, void* workspace, size_t ws_bytes, unsigned flags, void* stream);

/* a10 -- the trunk: for b < n_blocks, x = block_b(x; table[:, b]).  blocks: HOST array of
 * n_blocks weight sets; table: device bf16 [T][n_blocks][18H] as written by h3_modcache_build;
 * x: device bf16 [n_rows, H], updated in place.  Other arguments as h3_block_forward.  The
 * rotary cos/sin table is computed once per call and shared by all blocks. */
h3_status h3_trunk_forward(const h3_dims* dims, const h3_block_w* blocks, int n_blocks, const void* table, int T,
                           void* x, int n_rows, const uint8_t* tag, const int32_t* tidx, const float* pos,
                           void* workspace, size_t ws_bytes, unsigned flags, void* stream);

/* ---- trunk entry and exit, and the sampler ("minimax-h3-mlx" README, "Architecture": two
 * input patch projections and two output heads around the trunk; "Porting notes": those ship
 * as float32 tensors; "Layout": rectified-flow Euler with an exponential sigma shift) ---- */

/* x_rows[r] = bf16(W z[r] + b), r < n_rows, float32 weights and arithmetic: the input
 * projection of one modality's rows (video or condition latents: K = 96 patch features;
 * audio: K = 32).  z: device f32 [n_rows, K]; w: device f32 [H, K] (checkpoint orientation);
 * b: device f32 [H] or NULL; x_rows: device bf16, the first of the modality's n_rows rows of
 * the packed hidden stream [N, H] (16-byte aligned).  Text rows enter through a bf16 linear
 * (h3_linear_forward, condition_proj [H, 5120]). */
h3_status h3_embed_rows(const h3_dims* dims, const float* z, int K, const float* w, const float* b, int n_rows,
                        void* x_rows, void* stream);

/* Final-layer modulation table: table_f[t][j] = bf16(sum_k w[j][k] temb[t][k] + b[j]),
 * j < 6H, read as 3 modality tags x (shift, scale) x H (the kernel of h3_modcache_build).
 * temb: device f32 [T, Dt], 16-byte aligned; w: device
 * bf16 [6H, Dt] (16-byte aligned); b: device bf16 [6H] or NULL; table_f: device bf16 [T][6H]. */
h3_status h3_final_modcache_build(const h3_dims* dims, const float* temb, int T, int Dt, const void* w, const void* b,
                                  void* table_f, void* stream);

/* Output head of one modality's rows, in float32:
 *   v[r] = W (LN(x[r]) (1 + scale) + shift) + b,  (shift, scale) = table_f[tidx[r]*t_stride + (2 tag[r] + {0,1}) H]
 * and, when z_inout is given, the Euler transition z[r] += dsigma * v[r] (dsigma = sigma_next -
 * sigma_now of the modality's schedule).  x_rows: device bf16 [n_rows, H] (16-byte aligned);
 * tag, tidx: device, of these rows; table_f: device bf16 (t_stride >= 6H); w: device f32
 * [K_out, H]; b: device f32 [K_out] or NULL; v_out: device f32 [n_rows, K_out] or NULL;
 * z_inout: device f32 [n_rows, K_out] or NULL (not both NULL).  K_out <= 128. */
h3_status h3_head_forward(const h3_dims* dims, const void* x_rows, int n_rows, const uint8_t* tag, const int32_t* tidx,
                          const void* table_f, long long t_stride, const float* w, const float* b, int K_out,
                          float* v_out, float* z_inout, float dsigma, void* stream);

/* ---- the second-order sampler (mlx-h3 README, "Why mlx-h3": 20 schedule steps of the
 * res_multistep solver).  The page names the solver without defining it; this is the multistep
 * form of the refined exponential solver (Zhang, Song and Chen, "Improved Order Analysis and
 * Design of Exponential Integrator for Diffusion Models Sampling", 2023).  With the data
 * prediction D = z - sigma v of a rectified-flow velocity v, one step is
 *   z_next = a z + c_now D + c_prev D_prev,
 * D_prev being the previous step's prediction of the same modality. ---- */
typedef struct {
  float sigma;   /* the noise level the velocity is evaluated at (> 0) */
  float a, c_now, c_prev;
} h3_ms_step;

/* HOST: the weights of one res_multistep step from sigma to sigma_next (0 <= sigma_next <
 * sigma), sigma_prev being the previous step's sigma (> sigma), or <= 0 for the first step,
 * which is then first order (c_prev = 0; the Euler step).  A step to sigma_next = 0 returns D
 * (a = 0, c_now = 1).  Computed in double precision, rounded once to float.  Anything else
 * (a NaN anywhere included) returns H3_EINVAL. */
h3_status h3_res_multistep_step(float sigma_prev, float sigma, float sigma_next, h3_ms_step* out);

/* h3_head_forward with a res_multistep update instead of the Euler one: v as there, then per
 * element D = z - step->sigma * v, z = a z + c_now D + c_prev d_prev, d_prev = D (float32).
 * step: HOST; z_inout, d_prev_inout: device f32 [n_rows, K_out], both required; d_prev_inout is
 * read only when step->c_prev != 0 (it may hold anything on the first step) and always
 * written.  v_out: device f32 [n_rows, K_out] or NULL. */
h3_status h3_head_forward_ms(const h3_dims* dims, const void* x_rows, int n_rows, const uint8_t* tag,
                             const int32_t* tidx, const void* table_f, long long t_stride, const float* w,
                             const float* b, int K_out, const h3_ms_step* step, float* v_out, float* z_inout,
                             float* d_prev_inout, void* stream);

/* HOST: the sampling grid of one schedule, steps + 1 values from 1 to 0: a float32 linspace
 * (float32 step; first half start + step*i, second half end - step*(n-1-i), each one fused
 * multiply-add) followed by the time shift s sigma / (1 + (s - 1) sigma) in float32.
 * sigma_out: host f32 [steps + 1]. */
h3_status h3_sigma_schedule(int steps, float shift, float* sigma_out);

/* HOST: the plan of a run with video and audio on their own grids (h3_sigma_schedule with
 * shift_video, shift_audio): the distinct timesteps 1000 sigma (float32) that its `steps`
 * transitions evaluate, in descending order -- the rows of the modulation tables -- and, per
 * transition i, the row of the video (vidx[i]) and audio (aidx[i]) timestep.  Values are
 * distinct by exact float32 equality.  timesteps: host f32 with room for 2*steps values;
 * n_timesteps: host int, written; vidx, aidx: host i32 [steps]. */
h3_status h3_sampler_plan(int steps, float shift_video, float shift_audio, float* timesteps, int* n_timesteps,
                          int32_t* vidx, int32_t* aidx);

/* One denoiser transition of the sampler over the packed sequence [text | cond | audio | video]:
 *   x[text rows]  = text_x (the projected conditioner rows, computed once by the caller)
 *   x[cond rows]  = embed(z_cond; patch_v),  x[audio rows] = embed(z_audio; patch_a),
 *   x[video rows] = embed(z_video; patch_v)                      (h3_embed_rows)
 *   x = trunk(x)                                                 (h3_trunk_forward)
 *   z_video += dsigma_video * head_v(x[video rows]),  z_audio += dsigma_audio * head_a(x[audio rows])
 *                                                                (h3_head_forward)
 * io: the entry / exit weights (device f32) and segment sizes; table: the blocks' table as for
 * h3_trunk_forward; table_f: the final table [T][6H] (h3_final_modcache_build); tag, tidx, pos:
 * this transition's per-row tags, table rows and positions; x: device bf16 [N, H] scratch of
 * the hidden stream (overwritten).  The latents stay on the device across transitions. */
typedef struct {
  int text_rows, cond_rows, audio_rows, video_rows;
  int k_video, k_audio;                      /* latent features per row: 96 and 32 */
  const float* patch_v; const float* patch_v_b;  /* [H, k_video], [H] (bias nullable) */
  const float* patch_a; const float* patch_a_b;  /* [H, k_audio], [H] */
  const float* head_v; const float* head_v_b;    /* [k_video, H], [k_video] */
  const float* head_a; const float* head_a_b;    /* [k_audio, H], [k_audio] */
} h3_io_w;

h3_status h3_denoise_step(const h3_dims* dims, const h3_block_w* blocks, int n_blocks, const void* table,
                          const void* table_f, int T, const h3_io_w* io, const void* text_x, const float* z_cond,
                          float* z_video, float* z_audio, void* x, const uint8_t* tag, const int32_t* tidx,
                          const float* pos, float dsigma_video, float dsigma_audio, void* workspace, size_t ws_bytes,
                          unsigned flags, void* stream);

/* h3_denoise_step with res_multistep updates: the same entry, trunk and heads, then each
 * modality's latents take the step of h3_head_forward_ms with its own weights (step_video,
 * step_audio: HOST, from h3_res_multistep_step on the modality's grid) and its own previous
 * prediction (d_prev_video: device f32 [video_rows, k_video], d_prev_audio: [audio_rows,
 * k_audio]; read when c_prev != 0, always overwritten with this step's prediction). */
h3_status h3_denoise_step_ms(const h3_dims* dims, const h3_block_w* blocks, int n_blocks, const void* table,
                             const void* table_f, int T, const h3_io_w* io, const void* text_x, const float* z_cond,
                             float* z_video, float* z_audio, float* d_prev_video, float* d_prev_audio, void* x,
                             const uint8_t* tag, const int32_t* tidx, const float* pos, const h3_ms_step* step_video,
                             const h3_ms_step* step_audio, void* workspace, size_t ws_bytes, unsigned flags,
                             void* stream);

/* ---- step entry points (each row of the block on its own; used for per-step parity) ---- */

/* a1 / a6 -- gather + LayerNorm + modulate ("minimax-h3-mlx" README, "AdaLN: measure, do not
 * reason"): xn[r] = LN(x[r]) * (1 + table_b[tidx[r]*t_stride + (6 tag[r] + m_scale) H])
 *                            + table_b[tidx[r]*t_stride + (6 tag[r] + m_shift) H].
 * LayerNorm without affine, biased variance, eps = dims->ln_eps; statistics in fp32.
 * x, xn: device bf16 [n_rows, H] (distinct). */
h3_status h3_adaln_modulate(const h3_dims* dims, const void* x, void* xn, int n_rows, const void* table_b,
                            long long t_stride, int m_shift, int m_scale, const uint8_t* tag, const int32_t* tidx,
                            void* stream);

/* epilogues of h3_linear_forward */
#define H3_EPI_BIAS 0      /* y = x W^T + b                                                   */
#define H3_EPI_SWIGLU 1    /* y = silu(g) * v, [g | v] = x W^T + b; W has 2*n_y rows (gate rows first) */
#define H3_EPI_GATE_RES 2  /* y = res + gate(r) * (x W^T + b), gate from the modulation table */

/* a2 / a5 / a7 / a8 / a9 -- one linear with a fused epilogue on the tcgen05 tensor cores.
 * x: device bf16 [n_rows, lin->k] (row stride lda elements); y: device bf16 [n_rows, n_y]
 * (row stride ldy), n_y = lin->n_out except SWIGLU where n_y = lin->n_out / 2.
 * GATE_RES: res device bf16 [n_rows, n_y] (stride ldy; may equal y), the gate of row r and
 * column c is table_b[tidx[r]*t_stride + (6 tag[r] + m_gate) n_y + c].  Unused arguments may
 * be NULL / 0.  flags: H3_F_UNFUSED selects the CUDA-core reference GEMM. */
h3_status h3_linear_forward(const h3_linear* lin, int epilogue, const void* x, int lda, void* y, int ldy,
                            int n_rows, const void* res, const void* table_b, long long t_stride, int m_gate,
                            const uint8_t* tag, const int32_t* tidx, unsigned flags, void* stream);

/* a3 -- QK RMSNorm + 3D MM-RoPE on the interleaved projection ("H3-metal" README,
 * "Checkpoint layout and media pipeline"): for row r, head h, q = qkv[r, h*3hd + 0..hd),
 * k = qkv[r, h*3hd + hd..2hd), v = qkv[r, h*3hd + 2hd..3hd); q, k <- RMSNorm(.) * w (if weights
 * given), then rotate-half RoPE with angle pos[r][axis(i)] * theta^(-2i/hd) for pair (i, i+hd/2),
 * axis(i) by rope_sections.  Outputs head-major q_out, k_out: device bf16 [nh][n_rows][hd];
 * vt_out: device bf16 [nh][hd][ld_vt] (v transposed, ld_vt >= n_rows, ld_vt % 8 == 0).
 * qkv, q_out, k_out, vt_out and workspace must be 16-byte aligned, pos 4-byte aligned;
 * anything else returns H3_EINVAL before a launch.
 * workspace: device scratch of >= n_rows * hd/2 * 8 bytes (the per-row cos/sin table). */
h3_status h3_qknorm_rope(const h3_dims* dims, const void* qkv, const float* pos, const void* q_norm,
                         const void* k_norm, void* q_out, void* k_out, void* vt_out, int ld_vt, int n_rows,
                         void* workspace, size_t ws_bytes, void* stream);

/* a2 + a3 -- the QKV projection with QK-norm and rotary embedding as one step, as the block
 * runs it: q_out, k_out = RoPE(RMSNorm(.)) of xn Wqkv^T + b in the layout of h3_qknorm_rope,
 * vt_out = v transposed.  With head_dim 128 (and without H3_F_UNFUSED) the norm and rotation
 * run in the GEMM's epilogue and the projection never reaches memory; otherwise the projection
 * goes to the workspace and h3_qknorm_rope's kernel follows.  xn: device bf16 [n_rows, H];
 * wqkv: [3 nh hd, H] rows interleaved per head; workspace: device, 256-byte aligned, at least
 * h3_qkv_project_workspace_size bytes (the per-row cos/sin table + room for the projection). */
size_t h3_qkv_project_workspace_size(const h3_dims* dims, int n_rows);
h3_status h3_qkv_project(const h3_dims* dims, const h3_linear* wqkv, const void* xn, const float* pos,
                         const void* q_norm, const void* k_norm, void* q_out, void* k_out, void* vt_out, int ld_vt,
                         int n_rows, void* workspace, size_t ws_bytes, unsigned flags, void* stream);

/* a4 -- full unmasked self-attention ("minimax-h3-mlx" README, "Architecture"): per head,
 * o[r, h*hd + d] = sum_j softmax_j(q[h][r] . k[h][j] / sqrt(hd)) vt[h][d][j] over all j < n_rows.
 * q, k: device bf16 [nh][n_rows][hd]; vt: device bf16 [nh][hd][ld_vt]; o: device bf16
 * [n_rows, nh*hd].  hd must be 128 on the tcgen05 path.  flags: H3_F_UNFUSED = reference kernel. */
h3_status h3_attention(const h3_dims* dims, const void* q, const void* k, const void* vt, int ld_vt, void* o,
                       int n_rows, unsigned flags, void* stream);

/* Block-sparse variant of h3_attention (video sparse attention style: attention restricted to
 * selected tiles; the pages' own sparse backend uses trained tile masks, which are not part of
 * this library -- the caller supplies the mask).  The sequence is cut into 128-row tiles,
 * nt = ceil(n_rows / 128) query tiles and as many key tiles; tile_mask: device u8
 * [nh][nt][nt], tile_mask[h][qi][kj] != 0 keeps key tile kj for query tile qi of head h, and
 * every score outside the kept tiles counts as -inf.  A query row that keeps no key tile gets an
 * all-zero output row.  Work scales with the kept tiles (the kernel skips a key tile that both
 * query tiles of its 256-row pair drop).  Other arguments and layouts as h3_attention. */
h3_status h3_attention_sparse(const h3_dims* dims, const void* q, const void* k, const void* vt, int ld_vt, void* o,
                              int n_rows, const uint8_t* tile_mask, void* stream);

/* h3_qknorm_rope without a caller-supplied workspace.  The pages have no counterpart: this
 * entry point exists for callers that cannot allocate device memory at the call site (an
 * embedder whose device memory belongs to a pool or allocator it cannot reach there, or a
 * latency-critical loop that must not take cudaMalloc's implicit device synchronisation).
 * It computes exactly what h3_qknorm_rope computes, with the same arguments minus
 * workspace/ws_bytes, and allocates nothing: the cos/sin scratch is a fixed device array
 * inside the library (16 MiB, held on every device that loads the library until the process
 * exits) holding up to H3_QKROPE_STATIC_MAX_PAIRS (row, frequency) pairs.
 *   n_rows * head_dim / 2 > H3_QKROPE_STATIC_MAX_PAIRS (32768 rows at head_dim 128, 65536 at
 *   64) returns H3_EINVAL before any launch; so do the argument errors of h3_qknorm_rope.
 * The first call on a device looks up the array's device address (once per device, with that
 * device current) and caches it; make that first call before any stream capture.  The cached
 * address does not survive cudaDeviceReset (the library's module is reloaded afterwards).  Every call shares the
 * array: calls whose GPU work overlaps (different streams without ordering) race on it and
 * must be serialised by the caller.  Each call rewrites the part it reads, so the array needs
 * no clearing. */
#define H3_QKROPE_STATIC_MAX_PAIRS (1 << 21)
h3_status h3_qknorm_rope_static(const h3_dims* dims, const void* qkv, const float* pos, const void* q_norm,
                                const void* k_norm, void* q_out, void* k_out, void* vt_out, int ld_vt, int n_rows,
                                void* stream);

/* Measurement hook.  h3_kernel_timer_start(capacity) creates `capacity` pairs of CUDA events
 * (no device memory); from then on the first `capacity` attention launches made by
 * h3_block_forward / h3_trunk_forward are each bracketed by an event pair recorded on the
 * launching stream.  h3_kernel_timer_read waits for the recorded events, writes up to
 * `capacity` per-launch durations in milliseconds to the host array `ms`, the number recorded
 * to *n_recorded, and releases the events.  capacity 0 disarms.  Host-side state shared by
 * every caller in the process (not thread-safe); meant for benchmarks. */
h3_status h3_kernel_timer_start(int capacity);
h3_status h3_kernel_timer_read(float* ms, int capacity, int* n_recorded);

/* Diagnostic of the failure path: launches one kernel whose mbarrier wait can never complete
 * (nothing arrives), bounded by timeout_us (1 .. 1,000,000 microseconds).  The wait runs out,
 * records site 0x301 in the device error word and the kernel ends normally, exactly as a
 * stalled pipeline in any of the library's kernels would; the next h3_last_device_error then
 * reports H3_ETIMEOUT with that site and the context stays usable.  No fault or trap is
 * involved.  timeout_us outside the range returns H3_EINVAL. */
h3_status h3_diag_expire_wait(unsigned timeout_us, void* stream);

/* Synchronises `stream`, then reads and clears the device error word.  Returns H3_OK, or
 * H3_ETIMEOUT when a bounded device wait ran out since the last call (*site, if not NULL,
 * receives the site code), or H3_ECUDA if the stream reports a CUDA error. */
h3_status h3_last_device_error(void* stream, unsigned* site);

const char* h3_status_str(h3_status s);

#ifdef __cplusplus
}
#endif
#endif /* H3_H */
