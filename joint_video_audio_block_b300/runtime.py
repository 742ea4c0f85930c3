"""Torch-side plumbing around libh3: device buffers, uploads, streams.

PyTorch only allocates device memory and provides streams here; every step of the block runs
in libh3's kernels through the binding in h3.py.
"""

from __future__ import annotations

import numpy as np
import torch

from . import h3 as _h3


def dims_of(d) -> _h3.h3_dims:
    """h3_dims from any object with hidden/heads/head_dim/ffn/rope_sections (e.g. synth.Dims)."""
    return _h3.make_dims(d.hidden, d.heads, d.head_dim, d.ffn, d.rope_sections, n_tags=getattr(d, "n_tags", 3),
                         rope_theta=getattr(d, "rope_theta", 1e4), ln_eps=getattr(d, "ln_eps", 1e-6),
                         qk_eps=getattr(d, "qk_eps", 1e-6))


def bf16_from_bits(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """Upload raw bf16 bit patterns (uint16 numpy) as a bfloat16 tensor."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def bits_from_bf16(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a bfloat16 tensor as uint16 numpy (exact)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32_from_bf16(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def upload_block(weights: dict, device="cuda", int8: bool = False, quantize=None) -> dict:
    """Device tensors for one block from synth-style bf16-bit arrays.

    With int8=True each linear is stored as weight-only INT8 group-32 codes produced by the
    given `quantize` callable (bits -> (q, scale_bits, qbias_bits)); biases stay bf16.
    """
    out = {}
    for name, arr in weights.items():
        if int8 and name in ("wqkv", "wo", "w1", "w2"):
            q, s, b = quantize(arr)
            out[name] = torch.from_numpy(q).to(device)
            out[name + "_scale"] = bf16_from_bits(s, device)
            out[name + "_qbias"] = bf16_from_bits(b, device)
        else:
            out[name] = bf16_from_bits(arr, device)
    return out


def workspace(dims: _h3.h3_dims, n_rows: int, device="cuda") -> torch.Tensor:
    nbytes = _h3.h3_workspace_size(dims, n_rows)
    if nbytes == 0 and n_rows > 0:
        raise _h3.H3Error(_h3.H3_EINVAL, "h3_workspace_size")
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def sampler_plan(steps: int, video_shift: float = 12.0, audio_shift: float = 3.0):
    """Host-side plan of a run: the video and audio sampling grids (h3_sigma_schedule), the
    distinct timesteps (1000 sigma, float32) of the transitions in descending order -- the rows
    of the modulation tables -- and, per transition, the table row of each schedule
    (h3_sampler_plan)."""
    sv = np.asarray(_h3.h3_sigma_schedule(steps, video_shift), np.float32)
    sa = np.asarray(_h3.h3_sigma_schedule(steps, audio_shift), np.float32)
    values, vidx, aidx = _h3.h3_sampler_plan(steps, video_shift, audio_shift)
    return np.asarray(values, np.float32), sv, sa, vidx, aidx


def step_tidx(tidx: torch.Tensor, audio_rows: slice, vidx: int, aidx: int) -> torch.Tensor:
    """Per-row table rows of one transition: the audio rows follow the audio schedule, every
    other row (text, conditions, video) the video schedule."""
    tidx.fill_(vidx)
    tidx[audio_rows] = aidx
    return tidx
