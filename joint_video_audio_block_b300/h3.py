"""ctypes binding of libh3 (include/h3.h): argument marshalling only.

Every function here has the name of the C entry point it calls and takes raw device
pointers (ints) and plain sizes; the compute happens in the library's CUDA kernels.  The
helpers at the end only turn torch tensors into those pointers and structs.  Loading fails
loudly if libh3.so has not been built: there is no other implementation to fall back to.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libh3.so")

H3_OK, H3_EINVAL, H3_EUNSUPPORTED, H3_ECUDA, H3_ETIMEOUT = range(5)
H3_W_BF16, H3_W_INT8_G32 = 0, 1
H3_F_UNFUSED, H3_F_NO_QKNORM, H3_F_CHECK_INDEX = 0x1, 0x2, 0x4
H3_EPI_BIAS, H3_EPI_SWIGLU, H3_EPI_GATE_RES = 0, 1, 2

# every symbol include/h3.h declares
EXPORTS = (
    "h3_workspace_size", "h3_modcache_build", "h3_block_forward", "h3_trunk_forward", "h3_adaln_modulate",
    "h3_linear_forward", "h3_qknorm_rope", "h3_qknorm_rope_static", "h3_attention", "h3_last_device_error",
    "h3_status_str", "h3_kernel_timer_start", "h3_kernel_timer_read", "h3_qkv_project",
    "h3_qkv_project_workspace_size", "h3_diag_expire_wait", "h3_attention_sparse", "h3_embed_rows",
    "h3_final_modcache_build", "h3_head_forward", "h3_sigma_schedule", "h3_denoise_step",
    "h3_res_multistep_step", "h3_head_forward_ms", "h3_denoise_step_ms", "h3_sampler_plan",
)

# largest n_rows * head_dim / 2 that h3_qknorm_rope_static's fixed scratch array holds
H3_QKROPE_STATIC_MAX_PAIRS = 1 << 21


class H3Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {h3_status_str(status)} ({status})")
        self.status = status


class h3_dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("n_tags", ctypes.c_int), ("rope_sections", ctypes.c_int * 3), ("rope_theta", ctypes.c_float),
                ("ln_eps", ctypes.c_float), ("qk_eps", ctypes.c_float)]


class h3_linear(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("w", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("qbias", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("n_out", ctypes.c_int), ("k", ctypes.c_int)]


class h3_block_w(ctypes.Structure):
    _fields_ = [("qkv", h3_linear), ("o", h3_linear), ("fc1", h3_linear), ("fc2", h3_linear),
                ("q_norm", ctypes.c_void_p), ("k_norm", ctypes.c_void_p)]


class h3_io_w(ctypes.Structure):
    _fields_ = [("text_rows", ctypes.c_int), ("cond_rows", ctypes.c_int), ("audio_rows", ctypes.c_int),
                ("video_rows", ctypes.c_int), ("k_video", ctypes.c_int), ("k_audio", ctypes.c_int),
                ("patch_v", ctypes.c_void_p), ("patch_v_b", ctypes.c_void_p), ("patch_a", ctypes.c_void_p),
                ("patch_a_b", ctypes.c_void_p), ("head_v", ctypes.c_void_p), ("head_v_b", ctypes.c_void_p),
                ("head_a", ctypes.c_void_p), ("head_a_b", ctypes.c_void_p)]


class h3_ms_step(ctypes.Structure):
    _fields_ = [("sigma", ctypes.c_float), ("a", ctypes.c_float), ("c_now", ctypes.c_float), ("c_prev", ctypes.c_float)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libh3.so not built at {LIB_PATH}; run joint_video_audio_block_b300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, u32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_uint, ctypes.c_size_t
        D, LW, BW = ctypes.POINTER(h3_dims), ctypes.POINTER(h3_linear), ctypes.POINTER(h3_block_w)
        MS = ctypes.POINTER(h3_ms_step)
        sig = {
            "h3_workspace_size": (sz, [D, i32]),
            "h3_modcache_build": (i32, [D, vp, i32, i32, ctypes.POINTER(vp), ctypes.POINTER(vp), i32, vp, vp]),
            "h3_block_forward": (i32, [D, BW, vp, i64, i32, vp, vp, i32, vp, vp, vp, vp, sz, u32, vp]),
            "h3_trunk_forward": (i32, [D, BW, i32, vp, i32, vp, i32, vp, vp, vp, vp, sz, u32, vp]),
            "h3_adaln_modulate": (i32, [D, vp, vp, i32, vp, i64, i32, i32, vp, vp, vp]),
            "h3_linear_forward": (i32, [LW, i32, vp, i32, vp, i32, i32, vp, vp, i64, i32, vp, vp, u32, vp]),
            "h3_qknorm_rope": (i32, [D, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, sz, vp]),
            "h3_qknorm_rope_static": (i32, [D, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp]),
            "h3_qkv_project_workspace_size": (sz, [D, i32]),
            "h3_qkv_project": (i32, [D, LW, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, sz, u32, vp]),
            "h3_attention": (i32, [D, vp, vp, vp, i32, vp, i32, u32, vp]),
            "h3_attention_sparse": (i32, [D, vp, vp, vp, i32, vp, i32, vp, vp]),
            "h3_embed_rows": (i32, [D, vp, i32, vp, vp, i32, vp, vp]),
            "h3_final_modcache_build": (i32, [D, vp, i32, i32, vp, vp, vp, vp]),
            "h3_head_forward": (i32, [D, vp, i32, vp, vp, vp, i64, vp, vp, i32, vp, vp, ctypes.c_float, vp]),
            "h3_sigma_schedule": (i32, [i32, ctypes.c_float, ctypes.POINTER(ctypes.c_float)]),
            "h3_denoise_step": (i32, [D, BW, i32, vp, vp, i32, ctypes.POINTER(h3_io_w), vp, vp, vp, vp, vp, vp, vp, vp,
                                      ctypes.c_float, ctypes.c_float, vp, sz, u32, vp]),
            "h3_res_multistep_step": (i32, [ctypes.c_float, ctypes.c_float, ctypes.c_float, MS]),
            "h3_sampler_plan": (i32, [i32, ctypes.c_float, ctypes.c_float, ctypes.POINTER(ctypes.c_float),
                                      ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i32)]),
            "h3_head_forward_ms": (i32, [D, vp, i32, vp, vp, vp, i64, vp, vp, i32, MS, vp, vp, vp, vp]),
            "h3_denoise_step_ms": (i32, [D, BW, i32, vp, vp, i32, ctypes.POINTER(h3_io_w), vp, vp, vp, vp, vp, vp, vp,
                                         vp, vp, vp, MS, MS, vp, sz, u32, vp]),
            "h3_last_device_error": (i32, [vp, ctypes.POINTER(u32)]),
            "h3_kernel_timer_start": (i32, [i32]),
            "h3_diag_expire_wait": (i32, [u32, vp]),
            "h3_kernel_timer_read": (i32, [ctypes.POINTER(ctypes.c_float), i32, ctypes.POINTER(i32)]),
            "h3_status_str": (ctypes.c_char_p, [i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != H3_OK:
        raise H3Error(status, what)


# ------------------------------------------------------------------ the C entry points


def h3_status_str(status: int) -> str:
    return lib().h3_status_str(status).decode()


def h3_workspace_size(dims: h3_dims, n_rows: int) -> int:
    return lib().h3_workspace_size(ctypes.byref(dims), n_rows)


def h3_modcache_build(dims, temb, T, Dt, adaln_w_ptrs, adaln_b_ptrs, n_blocks, table, stream):
    W = (ctypes.c_void_p * n_blocks)(*adaln_w_ptrs)
    B = (ctypes.c_void_p * n_blocks)(*adaln_b_ptrs) if adaln_b_ptrs is not None else None
    _check(lib().h3_modcache_build(ctypes.byref(dims), temb, T, Dt, W, B, n_blocks, table, stream),
           "h3_modcache_build")


def h3_block_forward(dims, w, table_b, t_stride, T, x_in, x_out, n_rows, tag, tidx, pos, workspace, ws_bytes, flags,
                     stream):
    _check(lib().h3_block_forward(ctypes.byref(dims), ctypes.byref(w), table_b, t_stride, T, x_in, x_out, n_rows, tag,
                                  tidx, pos, workspace, ws_bytes, flags, stream), "h3_block_forward")


def h3_trunk_forward(dims, blocks, n_blocks, table, T, x, n_rows, tag, tidx, pos, workspace, ws_bytes, flags, stream):
    arr = (h3_block_w * n_blocks)(*blocks)
    _check(lib().h3_trunk_forward(ctypes.byref(dims), arr, n_blocks, table, T, x, n_rows, tag, tidx, pos, workspace,
                                  ws_bytes, flags, stream), "h3_trunk_forward")


def h3_adaln_modulate(dims, x, xn, n_rows, table_b, t_stride, m_shift, m_scale, tag, tidx, stream):
    _check(lib().h3_adaln_modulate(ctypes.byref(dims), x, xn, n_rows, table_b, t_stride, m_shift, m_scale, tag, tidx,
                                   stream), "h3_adaln_modulate")


def h3_linear_forward(lin, epilogue, x, lda, y, ldy, n_rows, res=None, table_b=None, t_stride=0, m_gate=0, tag=None,
                      tidx=None, flags=0, stream=None):
    _check(lib().h3_linear_forward(ctypes.byref(lin), epilogue, x, lda, y, ldy, n_rows, res, table_b, t_stride, m_gate,
                                   tag, tidx, flags, stream), "h3_linear_forward")


def h3_qknorm_rope(dims, qkv, pos, q_norm, k_norm, q_out, k_out, vt_out, ld_vt, n_rows, workspace, ws_bytes, stream):
    _check(lib().h3_qknorm_rope(ctypes.byref(dims), qkv, pos, q_norm, k_norm, q_out, k_out, vt_out, ld_vt, n_rows,
                                workspace, ws_bytes, stream), "h3_qknorm_rope")


def h3_qknorm_rope_static(dims, qkv, pos, q_norm, k_norm, q_out, k_out, vt_out, ld_vt, n_rows, stream):
    """h3_qknorm_rope with the library's fixed scratch array instead of a workspace (for callers
    that cannot allocate device memory at the call site); n_rows * head_dim / 2 must not exceed
    H3_QKROPE_STATIC_MAX_PAIRS."""
    _check(lib().h3_qknorm_rope_static(ctypes.byref(dims), qkv, pos, q_norm, k_norm, q_out, k_out, vt_out, ld_vt,
                                       n_rows, stream), "h3_qknorm_rope_static")


def h3_qkv_project_workspace_size(dims, n_rows: int) -> int:
    return lib().h3_qkv_project_workspace_size(ctypes.byref(dims), n_rows)


def h3_qkv_project(dims, wqkv, xn, pos, q_norm, k_norm, q_out, k_out, vt_out, ld_vt, n_rows, workspace, ws_bytes,
                   flags, stream):
    _check(lib().h3_qkv_project(ctypes.byref(dims), ctypes.byref(wqkv), xn, pos, q_norm, k_norm, q_out, k_out, vt_out,
                                ld_vt, n_rows, workspace, ws_bytes, flags, stream), "h3_qkv_project")


def h3_attention(dims, q, k, vt, ld_vt, o, n_rows, flags, stream):
    _check(lib().h3_attention(ctypes.byref(dims), q, k, vt, ld_vt, o, n_rows, flags, stream), "h3_attention")


def h3_kernel_timer_start(capacity: int):
    _check(lib().h3_kernel_timer_start(capacity), "h3_kernel_timer_start")


def h3_kernel_timer_read(capacity: int) -> list:
    """Per-launch attention durations (ms) recorded since h3_kernel_timer_start."""
    buf = (ctypes.c_float * max(capacity, 1))()
    n = ctypes.c_int(0)
    _check(lib().h3_kernel_timer_read(buf, capacity, ctypes.byref(n)), "h3_kernel_timer_read")
    return [buf[i] for i in range(min(n.value, capacity))]


def h3_diag_expire_wait(timeout_us: int, stream):
    _check(lib().h3_diag_expire_wait(timeout_us, stream), "h3_diag_expire_wait")


def h3_attention_sparse(dims, q, k, vt, ld_vt, o, n_rows, tile_mask, stream):
    _check(lib().h3_attention_sparse(ctypes.byref(dims), q, k, vt, ld_vt, o, n_rows, tile_mask, stream),
           "h3_attention_sparse")


def h3_embed_rows(dims, z, K, w, b, n_rows, x_rows, stream):
    _check(lib().h3_embed_rows(ctypes.byref(dims), z, K, w, b, n_rows, x_rows, stream), "h3_embed_rows")


def h3_final_modcache_build(dims, temb, T, Dt, w, b, table_f, stream):
    _check(lib().h3_final_modcache_build(ctypes.byref(dims), temb, T, Dt, w, b, table_f, stream),
           "h3_final_modcache_build")


def h3_head_forward(dims, x_rows, n_rows, tag, tidx, table_f, t_stride, w, b, K_out, v_out, z_inout, dsigma, stream):
    _check(lib().h3_head_forward(ctypes.byref(dims), x_rows, n_rows, tag, tidx, table_f, t_stride, w, b, K_out, v_out,
                                 z_inout, dsigma, stream), "h3_head_forward")


def h3_sigma_schedule(steps: int, shift: float) -> list:
    """Host-side sampling grid (steps + 1 float32 values from 1 to 0) of one shifted schedule."""
    buf = (ctypes.c_float * (steps + 1))()
    _check(lib().h3_sigma_schedule(steps, shift, buf), "h3_sigma_schedule")
    return [buf[i] for i in range(steps + 1)]


def h3_denoise_step(dims, blocks, n_blocks, table, table_f, T, io, text_x, z_cond, z_video, z_audio, x, tag, tidx, pos,
                    dsigma_video, dsigma_audio, workspace, ws_bytes, flags, stream):
    arr = (h3_block_w * n_blocks)(*blocks)
    _check(lib().h3_denoise_step(ctypes.byref(dims), arr, n_blocks, table, table_f, T, ctypes.byref(io), text_x, z_cond,
                                 z_video, z_audio, x, tag, tidx, pos, dsigma_video, dsigma_audio, workspace, ws_bytes,
                                 flags, stream), "h3_denoise_step")


def h3_sampler_plan(steps: int, shift_video: float, shift_audio: float):
    """Host-side run plan: (distinct timesteps descending, video row per step, audio row per step)."""
    ts = (ctypes.c_float * (2 * steps))()
    n = ctypes.c_int()
    vi = (ctypes.c_int * steps)()
    ai = (ctypes.c_int * steps)()
    _check(lib().h3_sampler_plan(steps, shift_video, shift_audio, ts, ctypes.byref(n), vi, ai), "h3_sampler_plan")
    return [ts[i] for i in range(n.value)], list(vi), list(ai)


def h3_res_multistep_step(sigma_prev, sigma, sigma_next) -> h3_ms_step:
    """Host-side weights of one res_multistep step (sigma_prev <= 0 or None: the first step)."""
    out = h3_ms_step()
    _check(lib().h3_res_multistep_step(-1.0 if sigma_prev is None else sigma_prev, sigma, sigma_next,
                                       ctypes.byref(out)), "h3_res_multistep_step")
    return out


def h3_head_forward_ms(dims, x_rows, n_rows, tag, tidx, table_f, t_stride, w, b, K_out, step, v_out, z_inout,
                       d_prev_inout, stream):
    _check(lib().h3_head_forward_ms(ctypes.byref(dims), x_rows, n_rows, tag, tidx, table_f, t_stride, w, b, K_out,
                                    ctypes.byref(step), v_out, z_inout, d_prev_inout, stream), "h3_head_forward_ms")


def h3_denoise_step_ms(dims, blocks, n_blocks, table, table_f, T, io, text_x, z_cond, z_video, z_audio, d_prev_video,
                       d_prev_audio, x, tag, tidx, pos, step_video, step_audio, workspace, ws_bytes, flags, stream):
    arr = (h3_block_w * n_blocks)(*blocks)
    _check(lib().h3_denoise_step_ms(ctypes.byref(dims), arr, n_blocks, table, table_f, T, ctypes.byref(io), text_x,
                                    z_cond, z_video, z_audio, d_prev_video, d_prev_audio, x, tag, tidx, pos,
                                    ctypes.byref(step_video), ctypes.byref(step_audio), workspace, ws_bytes, flags,
                                    stream), "h3_denoise_step_ms")


def make_io_w(t: dict, text_rows, cond_rows, audio_rows, video_rows, k_video=96, k_audio=32):
    """h3_io_w over device float32 tensors named like synth.io_weights()."""
    io = h3_io_w()
    io.text_rows, io.cond_rows, io.audio_rows, io.video_rows = text_rows, cond_rows, audio_rows, video_rows
    io.k_video, io.k_audio = k_video, k_audio
    for f in ("patch_v", "patch_v_b", "patch_a", "patch_a_b", "head_v", "head_v_b", "head_a", "head_a_b"):
        setattr(io, f, ptr(t.get(f)))
    io._refs = dict(t)
    return io


def h3_last_device_error(stream):
    site = ctypes.c_uint(0)
    st = lib().h3_last_device_error(stream, ctypes.byref(site))
    return st, site.value


# ------------------------------------------------------------------ torch helpers


def ptr(t) -> int | None:
    """Device pointer of a tensor, or None."""
    return None if t is None else t.data_ptr()


def stream_ptr(stream=None) -> int:
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def make_dims(hidden, heads, head_dim, ffn, rope_sections, n_tags=3, rope_theta=1e4, ln_eps=1e-6, qk_eps=1e-6):
    d = h3_dims()
    d.hidden, d.heads, d.head_dim, d.ffn, d.n_tags = hidden, heads, head_dim, ffn, n_tags
    d.rope_sections[:] = list(rope_sections)
    d.rope_theta, d.ln_eps, d.qk_eps = rope_theta, ln_eps, qk_eps
    return d


def make_linear(w, bias=None, scale=None, qbias=None):
    """h3_linear over device tensors: bf16 w [n_out, k], or u8 codes with bf16 scale/qbias."""
    import torch

    lw = h3_linear()
    lw.fmt = H3_W_INT8_G32 if w.dtype == torch.uint8 else H3_W_BF16
    lw.w, lw.scale, lw.qbias, lw.bias = ptr(w), ptr(scale), ptr(qbias), ptr(bias)
    lw.n_out, lw.k = int(w.shape[0]), int(w.shape[1])
    lw._refs = (w, bias, scale, qbias)  # the struct holds raw pointers: keep the tensors alive with it
    return lw


def make_block_w(t: dict):
    """h3_block_w from a dict of device tensors named like the checkpoint's linears."""
    bw = h3_block_w()
    for name, lname in (("qkv", "wqkv"), ("o", "wo"), ("fc1", "w1"), ("fc2", "w2")):
        bname = "b" + lname[1:]
        setattr(bw, name, make_linear(t[lname], t.get(bname), t.get(lname + "_scale"), t.get(lname + "_qbias")))
    bw.q_norm, bw.k_norm = ptr(t.get("qnorm")), ptr(t.get("knorm"))
    bw._refs = dict(t)  # keep every tensor the struct points at alive with it
    return bw
