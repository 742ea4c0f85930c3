"""CPU oracle for the H3 joint audio+video DiT block -- TEST INFRASTRUCTURE ONLY.

This module is the plain, slow, obviously-correct statement of what the block computes.  It
exists to check the CUDA library; the library never imports or calls it, and only the test
suite, the smoke check and the CPU-baseline leg of the benchmark may use it.  It shares no
code with the CUDA path: inputs come from the seeded generators in ``synth`` (which hold no
block arithmetic), everything else is here.

Arithmetic is float64 throughout (numpy; a matrix product is used as a library step).  Inputs
are the bf16 values the GPU receives, widened exactly.  Each function names the page and
section it follows.  Sources:

- "minimax-h3-mlx" README (PipeNetwork): sections "Architecture" (packed sequence, per-row
  modality tag, 50 blocks, hidden 5376, 56x128 heads, SwiGLU 14336, 3D MM-RoPE), "AdaLN
  precompute" (ModulationCache built from the timestep embedding through adaln_proj,
  [96768, 2688] per block), "AdaLN: measure, do not reason" (x*(1+scale)+shift for the
  norms, x + gate*f(x) for the residual branches, names such as shift_mlp), "Validation"
  (per-head interleaved qkv rows [h: q, k, v]; fused fc1 [gate; value] with
  fc2(silu(gate)*value)), "Performance" (dense full attention, linear share of the work).
- "H3-metal" README (antirez/h3.c): "Checkpoint layout and media pipeline" (fused
  QK-normalisation + RoPE on the interleaved qkv), "Exact DiT fusions".
- "mlx-h3" README: "Local model layout" (weight-only INT8 group 32, a8g32); "Why mlx-h3"
  (the sampler: 20 schedule steps of the second-order res_multistep solver, which the page
  names without defining; res_multistep_coefficients follows the published refined
  exponential solver of Zhang, Song and Chen, 2023, in its multistep form).

Readings where the pages are silent (each also listed in the design notes):
- the 18 in 18*H is 3 modality tags x 6 modulation tensors, tag-major, tensor order
  (shift_msa, scale_msa, gate_msa, shift_mlp, scale_mlp, gate_mlp);
- the norm is LayerNorm without affine, biased variance, eps 1e-6;
- QK-norm is a per-head RMSNorm with a learned [head_dim] weight, eps 1e-6, before RoPE;
- MM-RoPE: rotate-half pairs (i, i + hd/2), frequencies theta^(-2i/hd) with theta 1e4, the
  hd/2 pairs split into contiguous (t, h, w) sections of hd/8, 3hd/16, 3hd/16 pairs;
- attention is unmasked softmax(q k^T / sqrt(hd)) v over every row;
- linears carry biases; no nonlinearity is applied to temb inside the library.
- res_multistep: data prediction D = z - sigma v, log-noise time t = -ln(sigma), D linear in t
  through the current and previous predictions; first step first-order, a step to sigma 0
  returns D.

Parity status: the whole block and trunk are "parity unpinned" against the real model (the
pages print no worked example and no weights are available); each step is pinned separately
by the tests in tests/test_oracle_pins.py.
"""

from __future__ import annotations

import math

import numpy as np

# modulation tensor order inside one tag's group of six
SHIFT_MSA, SCALE_MSA, GATE_MSA, SHIFT_MLP, SCALE_MLP, GATE_MLP = range(6)


# ----------------------------------------------------------------------------------------
# storage helpers
# ----------------------------------------------------------------------------------------


def widen_bf16(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values, exact."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def round_bf16(x) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even); returns float64 holding bf16 values.

    The value is first rounded to float32 (the storage the GPU rounds from), then its low 16
    mantissa bits are rounded away.
    """
    x = np.asarray(x, dtype=np.float64)
    f = np.ascontiguousarray(x.astype(np.float32)).reshape(-1)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32).astype(np.float64)
    return np.where(np.isfinite(f), out, f.astype(np.float64)).reshape(x.shape)


def to_bf16_bits(x) -> np.ndarray:
    """bf16 bit patterns of round_bf16(x)."""
    r = round_bf16(x)
    f = np.ascontiguousarray(r.astype(np.float32)).reshape(-1)
    return (f.view(np.uint32) >> 16).astype(np.uint16).reshape(r.shape)


# ----------------------------------------------------------------------------------------
# a0: ModulationCache
# ----------------------------------------------------------------------------------------


def modcache(temb, adaln_w, adaln_b):
    """ModulationCache table for every (timestep, block).

    minimax-h3-mlx README, "AdaLN precompute": adaln_proj.linear of each block maps only the
    timestep embedding to 96768 = 18*H outputs, so the table for all timesteps of a run can be
    built once and the projection dropped.  The table is built from the float32 timestep
    embedding through unquantised (bf16) projections and stored as bf16.

    temb: float32 [T, Dt]; adaln_w: list of bf16 bits [18H, Dt]; adaln_b: list of bf16 bits
    [18H] or None.  Returns (table64 [T, B, 18H] float64, table_bf16 [T, B, 18H] float64
    holding bf16 values).
    """
    te = np.asarray(temb, dtype=np.float32).astype(np.float64)
    T = te.shape[0]
    B = len(adaln_w)
    n_out = np.asarray(adaln_w[0]).shape[0]
    table = np.empty((T, B, n_out), dtype=np.float64)
    for b in range(B):
        W = widen_bf16(adaln_w[b])
        y = te @ W.T
        if adaln_b is not None and adaln_b[b] is not None:
            y = y + widen_bf16(adaln_b[b])[None, :]
        table[:, b, :] = y
    return table, round_bf16(table)


def table_bytes(n_timesteps: int, n_blocks: int, hidden: int) -> int:
    """Size of the bf16 table: T x B x 18H x 2 bytes."""
    return n_timesteps * n_blocks * 18 * hidden * 2


def modulation(table_b, tag, tidx, m: int, hidden: int) -> np.ndarray:
    """Per-row modulation vector m of one block: table_b[tidx[r], 6*tag[r] + m, :].

    minimax-h3-mlx README, "Architecture": the per-row modality tag is the only
    modality-specific input to a block; it selects the row's AdaLN modulation.
    table_b: [T, 18H] (one block's slice).  Returns float64 [N, H].
    """
    tb = np.asarray(table_b, dtype=np.float64).reshape(table_b.shape[0], 18, hidden)
    tag = np.asarray(tag, dtype=np.int64)
    tidx = np.asarray(tidx, dtype=np.int64)
    return tb[tidx, 6 * tag + m, :]


# ----------------------------------------------------------------------------------------
# a1 / a6: LayerNorm + modulate
# ----------------------------------------------------------------------------------------


def layernorm(x, eps: float) -> np.ndarray:
    """Row LayerNorm without affine: (x - mean) / sqrt(biased var + eps)."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def adaln_modulate(x, shift, scale, eps: float) -> np.ndarray:
    """minimax-h3-mlx README, "AdaLN: measure, do not reason": norm(x) * (1 + scale) + shift."""
    return layernorm(x, eps) * (1.0 + scale) + shift


# ----------------------------------------------------------------------------------------
# linears, SwiGLU, INT8 dequant
# ----------------------------------------------------------------------------------------


def linear(x, w, b=None) -> np.ndarray:
    """y = x W^T (+ b); W is [out, in] as stored in the checkpoint."""
    y = np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T
    if b is not None:
        y = y + np.asarray(b, dtype=np.float64)[None, :]
    return y


def silu(g) -> np.ndarray:
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def swiglu(y, ffn: int) -> np.ndarray:
    """minimax-h3-mlx README, "Validation": fc1 is a fused [gate; value] projection and the MLP
    computes fc2(silu(gate) * value); gate = the first `ffn` outputs."""
    y = np.asarray(y, dtype=np.float64)
    return silu(y[:, :ffn]) * y[:, ffn:2 * ffn]


def dequant_int8_g32(q, scale_bits, qb_bits) -> np.ndarray:
    """Weight-only INT8 group-32 unpack: w' = bf16(fma_f32(scale[o, k/32], q[o, k], qbias[o, k/32])).

    mlx-h3 README, "Local model layout" names the a8g32 format (8-bit codes, group 32, per
    group scale and bias).  The product scale*q (8 + 8 significant bits) and its sum with the
    bias are exact in float64, so rounding that exact value to float32 once reproduces a fused
    multiply-add; the float32 result is then rounded to bf16.  Exactness is asserted.
    """
    q = np.asarray(q, dtype=np.uint8).astype(np.float64)
    n, k = q.shape
    sc = np.repeat(widen_bf16(scale_bits), 32, axis=1)[:, :k]
    qb = np.repeat(widen_bf16(qb_bits), 32, axis=1)[:, :k]
    p = sc * q
    s = p + qb
    # TwoSum error term: zero iff the float64 sum is exact
    bb = s - p
    err = (p - (s - bb)) + (qb - bb)
    assert not np.any(err != 0.0), "scale*q + qbias not exact in float64"
    return round_bf16(s.astype(np.float32).astype(np.float64))


# ----------------------------------------------------------------------------------------
# a3: QK-norm + 3D MM-RoPE
# ----------------------------------------------------------------------------------------


def split_qkv(y, heads: int, head_dim: int):
    """minimax-h3-mlx README, "Validation": qkv rows are interleaved per head, [h0: q,k,v][h1: ...],
    so the projection output reshapes to (rows, heads, 3, head_dim)."""
    y = np.asarray(y, dtype=np.float64).reshape(y.shape[0], heads, 3, head_dim)
    return y[:, :, 0, :], y[:, :, 1, :], y[:, :, 2, :]


def rms_norm(x, w, eps: float) -> np.ndarray:
    """Per-head RMSNorm over the last axis with learned weight w: x / sqrt(mean(x^2) + eps) * w."""
    x = np.asarray(x, dtype=np.float64)
    r = np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)
    return x / r * np.asarray(w, dtype=np.float64)


def rope_angles(pos, head_dim: int, theta: float, sections) -> np.ndarray:
    """Rotation angle of every frequency pair: phi[r, i] = pos[r, axis(i)] * theta^(-2i/hd).

    Pairs 0..s_t-1 follow the t axis, the next s_h pairs the h axis, the last s_w the w axis.
    """
    half = head_dim // 2
    assert sum(sections) == half
    i = np.arange(half, dtype=np.float64)
    omega = theta ** (-2.0 * i / head_dim)
    axis = np.concatenate([np.full(s, a, dtype=np.int64) for a, s in enumerate(sections)])
    p = np.asarray(pos, dtype=np.float32).astype(np.float64)
    return p[:, axis] * omega[None, :]


def rope(x, pos, head_dim: int, theta: float, sections) -> np.ndarray:
    """Rotate-half RoPE: element i pairs with i + hd/2, (a, b) -> (a cos - b sin, a sin + b cos).

    x: [N, heads, hd].  "3D MM-RoPE" (minimax-h3-mlx README, "Architecture") is read as the
    sectioned rotary above; a row with position (p, p, p) gets plain 1-D RoPE.
    """
    x = np.asarray(x, dtype=np.float64)
    half = head_dim // 2
    phi = rope_angles(pos, head_dim, theta, sections)[:, None, :]
    c, s = np.cos(phi), np.sin(phi)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


# ----------------------------------------------------------------------------------------
# a4: full self-attention
# ----------------------------------------------------------------------------------------


def attention(q, k, v, rows=None) -> np.ndarray:
    """Unmasked softmax attention of every query row over all rows, per head.

    minimax-h3-mlx README, "Architecture": full self-attention over the whole packed
    sequence, no cross-attention; "Performance": dense attention over all rows.
    q, k, v: [N, heads, hd].  rows: optional subset of query rows.  Returns [len(rows), heads, hd].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if rows is not None:
        q = q[rows]
    nh, hd = q.shape[1], q.shape[2]
    out = np.empty_like(q)
    inv = 1.0 / math.sqrt(hd)
    for h in range(nh):
        s = (q[:, h, :] @ k[:, h, :].T) * inv
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, h, :]
    return out


def attention_tile_sparse(q, k, v, tile_mask, tile: int = 128, rows=None) -> np.ndarray:
    """Block-sparse attention: the unmasked attention above restricted, per head, to the
    (query tile, key tile) blocks a tile mask keeps -- the video sparse attention form of the
    "FastH3 OmniRef (Ref2VA) on Apple Silicon MLX" page, section "Opt-in M5 attention backend"
    (a VSA tile mask selects tiles of 64 or 128 with head dimension 128; there the mask comes
    from trained gates, here it is given).  Scores outside the kept tiles are -inf; a query row
    that keeps no tile outputs 0.

    q, k, v: [N, heads, hd]; tile_mask: [heads, ceil(N/tile), ceil(N/tile)], nonzero = keep.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n = q.shape[0]
    sel = np.arange(n) if rows is None else np.asarray(rows)
    nh, hd = q.shape[1], q.shape[2]
    out = np.zeros((len(sel), nh, hd))
    inv = 1.0 / math.sqrt(hd)
    key_tile = np.arange(n) // tile
    for h in range(nh):
        keep = np.asarray(tile_mask[h], dtype=bool)[(sel // tile)[:, None], key_tile[None, :]]  # [rows, N]
        s = (q[sel, h, :] @ k[:, h, :].T) * inv
        s = np.where(keep, s, -np.inf)
        live = keep.any(axis=1)
        m = np.where(live, s.max(axis=1), 0.0)
        p = np.where(keep, np.exp(s - m[:, None]), 0.0)
        den = p.sum(axis=1)
        o = (p @ v[:, h, :]) / np.where(live, den, 1.0)[:, None]
        out[:, h, :] = np.where(live[:, None], o, 0.0)
    return out


# ----------------------------------------------------------------------------------------
# a1..a8: one block; a10: the trunk
# ----------------------------------------------------------------------------------------


def _w(wd, name):
    v = wd.get(name)
    return None if v is None else widen_bf16(v)


def block_forward(x, weights, table_b, tag, tidx, pos, dims, *, rows=None, emulate_bf16=False,
                  dequant=None, return_parts=False):
    """One DiT block over the packed sequence.

    x: bf16 bits or float64 [N, H]; weights: dict of bf16 bits (synth.block_weights layout);
    table_b: this block's bf16 table slice [T, 18H] (float64 holding bf16 values).
    rows: compute outputs only for these rows (keys and values still use every row).
    emulate_bf16: round to bf16 where the GPU stores activations (xn, q/k/v, o, x after the
    attention branch, the SwiGLU activation h, the output) -- a diagnostic only.
    dequant: optional dict name -> float64 weight replacing the bf16 one (INT8 path).

    Steps (minimax-h3-mlx README, "Architecture", "AdaLN: measure, do not reason",
    "Validation"):
      xn = LN(x)(1 + scale_msa) + shift_msa; qkv = xn Wqkv^T + b; q, k = RMSNorm (optional),
      then RoPE; o = softmax(q k^T/sqrt(hd)) v; x = x + gate_msa * (o Wo^T + bo);
      xn = LN(x)(1 + scale_mlp) + shift_mlp; h = silu(g) * v of [g; v] = xn W1^T + b1;
      x = x + gate_mlp * (h W2^T + b2).
    """
    H, nh, hd, F = dims.hidden, dims.heads, dims.head_dim, dims.ffn
    rnd = round_bf16 if emulate_bf16 else (lambda a: a)
    x = np.asarray(x)
    x = widen_bf16(x) if x.dtype == np.uint16 else np.asarray(x, dtype=np.float64)
    N = x.shape[0]
    sel = np.arange(N) if rows is None else np.asarray(rows)

    def W(name):
        if dequant is not None and name in dequant:
            return dequant[name]
        return _w(weights, name)

    def mod(m, r):
        return modulation(table_b, np.asarray(tag)[r], np.asarray(tidx)[r], m, H)

    # attention branch: every row feeds keys/values
    xn = rnd(adaln_modulate(x, mod(SHIFT_MSA, slice(None)), mod(SCALE_MSA, slice(None)), dims.ln_eps))
    wqkv, bqkv = W("wqkv"), _w(weights, "bqkv")
    y = linear(xn, wqkv, bqkv)
    q, k, v = split_qkv(y, nh, hd)
    if weights.get("qnorm") is not None:
        q = rms_norm(q, _w(weights, "qnorm"), dims.qk_eps)
        k = rms_norm(k, _w(weights, "knorm"), dims.qk_eps)
    q = rnd(rope(q, pos, hd, dims.rope_theta, dims.rope_sections))
    k = rnd(rope(k, pos, hd, dims.rope_theta, dims.rope_sections))
    v = rnd(v)
    o = rnd(attention(q, k, v, rows=sel).reshape(len(sel), nh * hd))
    xs = x[sel]
    x1 = rnd(xs + mod(GATE_MSA, sel) * linear(o, W("wo"), _w(weights, "bo")))

    # MLP branch on the selected rows
    xn2 = rnd(adaln_modulate(x1, mod(SHIFT_MLP, sel), mod(SCALE_MLP, sel), dims.ln_eps))
    hact = rnd(swiglu(linear(xn2, W("w1"), _w(weights, "b1")), F))
    out = rnd(x1 + mod(GATE_MLP, sel) * linear(hact, W("w2"), _w(weights, "b2")))
    if return_parts:
        return out, dict(xn=xn, q=q, k=k, v=v, o=o, x1=x1, xn2=xn2, h=hact)
    return out


def trunk_forward(x, block_weight_list, table_bf16, tag, tidx, pos, dims, *, emulate_bf16=False):
    """minimax-h3-mlx README, "Architecture": 50 identical blocks applied in sequence over the
    packed sequence; block b reads table[:, b].  table_bf16: [T, B, 18H]."""
    h = x
    for b, wb in enumerate(block_weight_list):
        h = block_forward(h, wb, table_bf16[:, b, :], tag, tidx, pos, dims, emulate_bf16=emulate_bf16)
    return h


# ----------------------------------------------------------------------------------------
# trunk entry and exit; the sampler
# ----------------------------------------------------------------------------------------


def embed_rows(z, w, b) -> np.ndarray:
    """Input projection of one modality's rows into the hidden stream: x = z W^T + b.

    minimax-h3-mlx README, "Architecture": modality-specific behaviour comes only from the two
    input patch projections (video, audio), the per-row tag and the two output heads; the
    conditioner's hidden state enters through condition_proj (section "Encoder truncation").
    "Porting notes" / "Validation": the patch projections ship as float32 tensors, so the
    projection is float32 weights on float32 latents; the result joins the bf16 hidden stream.
    z: [rows, K]; w: [H, K] float32; b: [H].  Returns float64 (the exact value).
    """
    return linear(np.asarray(z, dtype=np.float64), np.asarray(w, dtype=np.float64), b)


def final_modulation(table_f, tag, tidx, m: int, hidden: int) -> np.ndarray:
    """Per-row final-layer modulation: table_f[tidx[r], 2*tag[r] + m, :] with m = 0 shift, 1 scale.

    Reading: the timestep-aware output head ("H3-metal" README, "Sampler and DiT controls":
    the patch projection and timestep-aware head stay fresh) is an AdaLN with its own two
    tensors per modality tag, tabulated from the timestep embedding like the blocks' six.
    table_f: [T, 6H]."""
    tf = np.asarray(table_f, dtype=np.float64).reshape(table_f.shape[0], 6, hidden)
    return tf[np.asarray(tidx, np.int64), 2 * np.asarray(tag, np.int64) + m, :]


def head_forward(x, shift, scale, w, b, eps: float) -> np.ndarray:
    """Output head of one modality's rows: v = (LN(x)(1 + scale) + shift) W^T + b.

    minimax-h3-mlx README, "Architecture": two output heads; "Porting notes": they ship as
    float32 tensors ("H3-metal" README, "Specialized projection kernels": the close-reference
    head keeps them in F32).  x: bf16 values [rows, H]; w: [K_out, H] float32."""
    xn = adaln_modulate(np.asarray(x, dtype=np.float64), shift, scale, eps)
    return linear(xn, np.asarray(w, dtype=np.float64), b)


def linspace_f32(start: float, end: float, steps: int) -> np.ndarray:
    """torch.linspace in float32 as the minimax-h3-mlx README ("Porting notes", "Validation")
    describes ATen's: a float32 step (end - start) / (steps - 1); the first half evaluated as
    start + step * i, the second half as end - step * (steps - 1 - i), each with one fused
    multiply-add rounded to float32.  (The fused result equals rounding the exact float64
    value of the product-sum once, since step and i are exact and the float64 product of a
    24-bit and a <= 24-bit integer is exact.)"""
    f32 = np.float32
    if steps == 1:
        return np.array([start], np.float32)
    step = f32((f32(end) - f32(start)) / f32(steps - 1))
    half = steps // 2
    out = np.empty(steps, np.float32)
    for i in range(steps):
        if i < half:
            out[i] = f32(np.float64(f32(start)) + np.float64(step) * i)
        else:
            out[i] = f32(np.float64(f32(end)) - np.float64(step) * (steps - 1 - i))
    return out


def shifted_sigmas(steps: int, shift: float) -> np.ndarray:
    """Rectified-flow sampling grid for `steps` Euler transitions: sigma_i from 1 to 0 on the
    float32 linspace grid, then the time shift sigma' = s sigma / (1 + (s - 1) sigma) in float32
    (minimax-h3-mlx README, "AdaLN precompute": separate video and audio shifts, 12.0 and 3.0;
    "Porting notes": scheduler scalars in float32).  Returns float32 [steps + 1]."""
    f32 = np.float32
    sig = linspace_f32(1.0, 0.0, steps + 1)
    s = f32(shift)
    return (s * sig / (f32(1.0) + (s - f32(1.0)) * sig)).astype(np.float32)


def euler_step(z, v, sigma_now: float, sigma_next: float) -> np.ndarray:
    """One rectified-flow Euler transition: z <- z + (sigma_next - sigma_now) v
    (minimax-h3-mlx README, "Layout": the scheduler is rectified-flow Euler)."""
    return np.asarray(z, dtype=np.float64) + (float(sigma_next) - float(sigma_now)) * np.asarray(v, dtype=np.float64)


def data_prediction(z, v, sigma: float) -> np.ndarray:
    """The clean-latent estimate behind a rectified-flow velocity: z_sigma = (1 - sigma) x0 +
    sigma eps and v = eps - x0 give x0 = z - sigma v."""
    return np.asarray(z, dtype=np.float64) - float(sigma) * np.asarray(v, dtype=np.float64)


def res_multistep_coefficients(sigma_prev, sigma: float, sigma_next: float) -> tuple:
    """Weights (a, c_now, c_prev) of one step z_next = a z + c_now D_now + c_prev D_prev of the
    second-order multistep exponential integrator that the mlx-h3 README ("Why mlx-h3") names as
    the sampler (res_multistep).  The pages name the solver but do not define it; this follows
    the published method it is named for: the refined exponential solver (RES) of Zhang, Song
    and Chen, "Improved Order Analysis and Design of Exponential Integrator for Diffusion
    Models Sampling" (2023), in its multistep form.

    Derivation.  With the data prediction D(z, sigma) = z - sigma v, the sampling ODE
    dz/dsigma = v reads dz/dsigma = (z - D)/sigma; in log-noise time t = -ln(sigma) it is
    dz/dt = D - z, so over one step of length h = t_next - t = ln(sigma / sigma_next),
        z(t + h) = e^-h z(t) + integral_0^h e^-(h - u) D(t + u) du.
    D is taken linear in u through D_now (u = 0) and D_prev (u = r h, r = (t_prev - t) / h < 0),
    and the two integrals are h phi1(-h) and h^2 phi2(-h) with phi1(x) = (e^x - 1)/x and
    phi2(x) = (phi1(x) - 1)/x, which gives
        a = e^-h = sigma_next / sigma,
        c_now = h (phi1 - phi2 / r),  c_prev = h phi2 / r.
    Without a previous prediction (sigma_prev None: the first step) D is taken constant: the
    first-order step a = sigma_next / sigma, c_now = 1 - a, which equals the Euler step
    z + (sigma_next - sigma) v.  A step to sigma_next = 0 returns D_now (a = 0, c_now = 1), the
    limit of both forms and the Euler step to zero.  float64 throughout."""
    sigma = float(sigma)
    sigma_next = float(sigma_next)
    if not sigma > 0.0:
        raise ValueError("sigma must be positive")
    if sigma_next == 0.0:
        return 0.0, 1.0, 0.0
    a = sigma_next / sigma
    if sigma_prev is None:
        return a, 1.0 - a, 0.0
    h = math.log(sigma / sigma_next)
    r = math.log(sigma / float(sigma_prev)) / h
    phi1 = -math.expm1(-h) / h
    phi2 = (1.0 - phi1) / h
    return a, h * (phi1 - phi2 / r), h * phi2 / r


def res_multistep_step(z, v, sigma_prev, sigma: float, sigma_next: float, d_prev=None):
    """One res_multistep transition of a modality's latents (coefficients above).  Returns
    (z_next, D_now); D_now is the d_prev of the next step.  d_prev is needed unless sigma_prev
    is None."""
    d_now = data_prediction(z, v, sigma)
    a, c_now, c_prev = res_multistep_coefficients(sigma_prev, sigma, sigma_next)
    z_next = a * np.asarray(z, dtype=np.float64) + c_now * d_now
    if c_prev != 0.0:
        z_next = z_next + c_prev * np.asarray(d_prev, dtype=np.float64)
    return z_next, d_now


def denoise_velocities(text_x, z_cond, z_audio, z_video, io, block_weight_list, table_bf16, table_f, tag, tidx, pos,
                       dims):
    """The model evaluation of one sampler transition over the packed sequence [text | cond |
    audio | video] (minimax-h3-mlx README, "Architecture" and "Layout"): the entry projections
    write the latent rows into the hidden stream (stored as bf16, as the stream is), the trunk
    runs, and the output heads give each modality's velocity.  Returns (v_audio, v_video).
    io: synth.io_weights() layout; text_x: the projected text rows (bf16 values)."""
    H = dims.hidden
    parts = [np.asarray(text_x, dtype=np.float64)]
    if len(z_cond):
        parts.append(round_bf16(embed_rows(z_cond, io["patch_v"], io["patch_v_b"])))
    parts.append(round_bf16(embed_rows(z_audio, io["patch_a"], io["patch_a_b"])))
    parts.append(round_bf16(embed_rows(z_video, io["patch_v"], io["patch_v_b"])))
    x = np.concatenate(parts, axis=0)
    x = trunk_forward(x, block_weight_list, table_bf16, tag, tidx, pos, dims)
    a0 = len(text_x) + len(z_cond)
    v0 = a0 + len(z_audio)
    out = []
    for r0, n, w, b in ((a0, len(z_audio), io["head_a"], io["head_a_b"]), (v0, len(z_video), io["head_v"], io["head_v_b"])):
        rows = slice(r0, r0 + n)
        shift = final_modulation(table_f, tag[rows], tidx[rows], 0, H)
        scale = final_modulation(table_f, tag[rows], tidx[rows], 1, H)
        out.append(head_forward(x[rows], shift, scale, w, b, dims.ln_eps))
    return out[0], out[1]


def denoise_step(text_x, z_cond, z_audio, z_video, io, block_weight_list, table_bf16, table_f, tag, tidx, pos, dims,
                 dsigma_video: float, dsigma_audio: float):
    """One Euler sampler transition (minimax-h3-mlx README, "Layout"; mlx-h3 README,
    "Generate": video and audio advance on their own sigma grids): the velocities of
    denoise_velocities move each modality's latents by its own dsigma.  Returns
    (z_audio, z_video)."""
    v_a, v_v = denoise_velocities(text_x, z_cond, z_audio, z_video, io, block_weight_list, table_bf16, table_f, tag,
                                  tidx, pos, dims)
    return euler_step(z_audio, v_a, 0.0, dsigma_audio), euler_step(z_video, v_v, 0.0, dsigma_video)


def denoise_step_multistep(text_x, z_cond, z_audio, z_video, io, block_weight_list, table_bf16, table_f, tag, tidx,
                           pos, dims, sig_video, sig_audio, d_prev_video=None, d_prev_audio=None):
    """One res_multistep sampler transition (mlx-h3 README, "Why mlx-h3"): the velocities of
    denoise_velocities, then res_multistep_step per modality on its own grid.  sig_video,
    sig_audio: (sigma_prev or None, sigma, sigma_next).  Returns (z_audio, z_video, D_audio,
    D_video), the D's being the next step's d_prev."""
    v_a, v_v = denoise_velocities(text_x, z_cond, z_audio, z_video, io, block_weight_list, table_bf16, table_f, tag,
                                  tidx, pos, dims)
    za, da = res_multistep_step(z_audio, v_a, *sig_audio, d_prev=d_prev_audio)
    zv, dv = res_multistep_step(z_video, v_v, *sig_video, d_prev=d_prev_video)
    return za, zv, da, dv


# ----------------------------------------------------------------------------------------
# work model
# ----------------------------------------------------------------------------------------


def block_linear_params(dims) -> int:
    """Weights of the four trunk linears of one block (qkv, o, fc1, fc2)."""
    H, I, F = dims.hidden, dims.inner, dims.ffn
    return 3 * I * H + H * I + 2 * F * H + H * F


def block_flops(dims, n_rows: int) -> tuple:
    """(linear FLOP, attention FLOP) of one block: 2 N P_lin and 4 N^2 I (QK^T and PV)."""
    return 2 * n_rows * block_linear_params(dims), 4 * n_rows * n_rows * dims.inner
