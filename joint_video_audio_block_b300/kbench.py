"""Per-step microbenchmark of the block's kernels through the C ABI.

    python -m joint_video_audio_block_b300.kbench --kernel attention --rows 12936 [--reps 10]

Runs one step of the block (attention, a linear with its epilogue, AdaLN modulate, QK-norm +
RoPE, or the modulation-table build) on seeded device inputs of the full-width H3 geometry
(hidden 5376, 56 x 128 heads, SwiGLU 14336, timestep embedding 2688), times it with CUDA
events on the launching stream after warm-up, and prints one JSON line with the duration,
the algorithmic FLOP and bytes of one launch, and the achieved rates.  Every input of the
timed kernels is larger than L2 except where stated in the output.  Also the command the
kernel profiles are captured with.
"""

from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from joint_video_audio_block_b300 import h3  # noqa: E402
from joint_video_audio_block_b300 import runtime as R  # noqa: E402

KERNELS = ("block", "attention", "attention_sparse", "qkv", "o", "fc1", "fc2", "adaln", "qkrope", "qkvrope",
           "modcache", "embed", "head")


def _normal(shape, std=1.0, mean=0.0, stream=1):
    return synth.device_normal_bf16(7, stream, shape, mean, std)


def setup(kernel: str, n: int, int8: bool, density: float = 0.25, blocks: int = 1):
    """Returns (launch(), flop, bytes, note) for one launch of `kernel` over n rows."""
    d = synth.H3
    H, I, F, hd, nh = d.hidden, d.inner, d.ffn, d.head_dim, d.heads
    dims = R.dims_of(d)
    st = h3.stream_ptr()
    keep = []

    if kernel == "block":
        # one whole DiT block (h3_block_forward: a1..a8) on the packed layout of the nearest
        # configuration; FLOP = the MMA work of the block (linears + attention)
        cfg = min(synth.CONFIGS.values(), key=lambda c: abs(c.layout.n_rows - n) if c.dims is d else 1 << 30)
        tag, tidx, pos = (np.resize(a, (n,) + a.shape[1:]) for a in synth.packed_rows(cfg))
        w = synth.device_block_weights(synth.CONFIGS["block12936"], 0)
        if int8:
            raise ValueError("block timing is bf16 only")
        bw = h3.make_block_w(w)
        x = _normal((n, H), stream=30)
        out = torch.empty_like(x)
        table = _normal((1, 18 * H), 0.5, stream=31)
        tag_d = torch.from_numpy(np.ascontiguousarray(tag)).cuda()
        tidx_d = torch.zeros(n, dtype=torch.int32, device="cuda")
        pos_d = torch.from_numpy(np.ascontiguousarray(pos)).cuda()
        ws = R.workspace(dims, n)
        keep += [w, bw, x, out, table, tag_d, tidx_d, pos_d, ws]

        def launch():
            h3.h3_block_forward(dims, bw, table.data_ptr(), 18 * H, 1, x.data_ptr(), out.data_ptr(), n, tag_d.data_ptr(),
                                tidx_d.data_ptr(), pos_d.data_ptr(), ws.data_ptr(), ws.numel(), 0, st)

        lin = 2.0 * n * (3 * I * H + H * I + 2 * F * H + H * F)
        return launch, lin + 4.0 * n * n * I, 0.0, f"packed layout of {cfg.name}; FLOP = linears + attention", keep

    if kernel == "attention":
        ld = (n + 63) // 64 * 64
        q, k = _normal((nh, n, hd), stream=1), _normal((nh, n, hd), stream=2)
        vt, o = _normal((nh, hd, ld), stream=3), torch.empty(n, I, dtype=torch.bfloat16, device="cuda")
        keep += [q, k, vt, o]

        def launch():
            h3.h3_attention(dims, q.data_ptr(), k.data_ptr(), vt.data_ptr(), ld, o.data_ptr(), n, 0, st)

        return launch, 4.0 * n * n * I, 4.0 * n * I * 2, "", keep

    if kernel == "attention_sparse":
        # random (query tile, key tile) mask of the given density; FLOP counted on kept tiles only
        ld = (n + 63) // 64 * 64
        nt = (n + 127) // 128
        q, k = _normal((nh, n, hd), stream=1), _normal((nh, n, hd), stream=2)
        vt, o = _normal((nh, hd, ld), stream=3), torch.empty(n, I, dtype=torch.bfloat16, device="cuda")
        mask = (np.random.default_rng(0).random((nh, nt, nt)) < density).astype(np.uint8)
        rows_in = np.minimum(np.arange(nt) * 128 + 128, n) - np.arange(nt) * 128
        kept = float((mask * rows_in[None, :, None] * rows_in[None, None, :]).sum())
        md = torch.from_numpy(mask).cuda()
        keep += [q, k, vt, o, md]

        def launch():
            h3.h3_attention_sparse(dims, q.data_ptr(), k.data_ptr(), vt.data_ptr(), ld, o.data_ptr(), n, md.data_ptr(),
                                   st)

        return launch, 4.0 * kept * hd, 4.0 * n * I * 2, f"tile density {density}: FLOP of kept tiles only", keep

    if kernel in ("qkv", "o", "fc1", "fc2"):
        K, n_out, epi = {"qkv": (H, 3 * I, h3.H3_EPI_BIAS), "o": (I, H, h3.H3_EPI_GATE_RES),
                         "fc1": (H, 2 * F, h3.H3_EPI_SWIGLU), "fc2": (F, H, h3.H3_EPI_GATE_RES)}[kernel]
        n_y = n_out // 2 if epi == h3.H3_EPI_SWIGLU else n_out
        x = _normal((n, K), stream=4)
        w = _normal((n_out, K), 0.02, stream=5)
        b = _normal((n_out,), 0.02, stream=6)
        wbytes = 2.0
        if int8:
            q = torch.randint(0, 256, (n_out, K), dtype=torch.uint8, device="cuda")
            sc = _normal((n_out, K // 32), 1e-3, stream=7)
            qb = _normal((n_out, K // 32), 0.02, stream=8)
            lin = h3.make_linear(q, b, sc, qb)
            wbytes = 1.0 + 4.0 / 32
        else:
            lin = h3.make_linear(w, b)
        y = _normal((n, n_y), stream=9)
        tag, tidx, _ = synth.packed_rows(synth.CONFIGS["block12936"])
        tag_d = torch.from_numpy(np.resize(tag, n)).cuda()
        tidx_d = torch.zeros(n, dtype=torch.int32, device="cuda")
        table = _normal((1, 18 * H), 0.5, stream=10)
        keep += [x, w, b, y, tag_d, tidx_d, table, lin]
        gate = epi == h3.H3_EPI_GATE_RES

        def launch():
            h3.h3_linear_forward(lin, epi, x.data_ptr(), K, y.data_ptr(), n_y, n,
                                 res=y.data_ptr() if gate else None, table_b=table.data_ptr() if gate else None,
                                 t_stride=18 * H, m_gate=2 if kernel == "o" else 5,
                                 tag=tag_d.data_ptr() if gate else None, tidx=tidx_d.data_ptr() if gate else None,
                                 stream=st)

        byts = n * K * 2.0 + n_out * K * wbytes + n_y * n * 2.0 * (2 if gate else 1)
        return launch, 2.0 * n * K * n_out, byts, "", keep

    if kernel == "adaln":
        x = _normal((n, H), stream=11)
        xn = torch.empty_like(x)
        tag_d = torch.full((n,), 2, dtype=torch.uint8, device="cuda")
        tidx_d = torch.zeros(n, dtype=torch.int32, device="cuda")
        table = _normal((1, 18 * H), 0.5, stream=12)
        keep += [x, xn, tag_d, tidx_d, table]

        def launch():
            h3.h3_adaln_modulate(dims, x.data_ptr(), xn.data_ptr(), n, table.data_ptr(), 18 * H, 0, 1,
                                 tag_d.data_ptr(), tidx_d.data_ptr(), st)

        return launch, 0.0, 4.0 * n * H, "table rows are L2-resident (one (tag, t) vector pair)", keep

    if kernel == "qkrope":
        qkv = _normal((n, 3 * I), stream=13)
        _, _, pos = synth.packed_rows(synth.CONFIGS["block12936"])
        pos_d = torch.from_numpy(np.ascontiguousarray(np.resize(pos, (n, 3)))).cuda()
        ld = (n + 63) // 64 * 64
        q = torch.empty(nh, n, hd, dtype=torch.bfloat16, device="cuda")
        k, vt = torch.empty_like(q), torch.empty(nh, hd, ld, dtype=torch.bfloat16, device="cuda")
        qn, kn = _normal((hd,), 0.02, 1.0, stream=14), _normal((hd,), 0.02, 1.0, stream=15)
        ws = torch.empty(n * hd * 4, dtype=torch.uint8, device="cuda")
        keep += [qkv, pos_d, q, k, vt, qn, kn, ws]

        def launch():
            h3.h3_qknorm_rope(dims, qkv.data_ptr(), pos_d.data_ptr(), qn.data_ptr(), kn.data_ptr(), q.data_ptr(),
                              k.data_ptr(), vt.data_ptr(), ld, n, ws.data_ptr(), ws.numel(), st)

        return launch, 0.0, 12.0 * n * I + 12.0 * n + n * hd * 4.0 * 2, "includes the per-row cos/sin table", keep

    if kernel == "qkvrope":
        # a2 + a3 as the block runs them: the QKV GEMM with QK-norm + RoPE in its epilogue
        xn = _normal((n, H), stream=18)
        w = _normal((3 * I, H), 0.02, stream=19)
        b = _normal((3 * I,), 0.02, stream=20)
        wbytes = 2.0
        if int8:
            qc = torch.randint(0, 256, (3 * I, H), dtype=torch.uint8, device="cuda")
            sc = _normal((3 * I, H // 32), 1e-3, stream=21)
            qb = _normal((3 * I, H // 32), 0.02, stream=22)
            lin = h3.make_linear(qc, b, sc, qb)
            keep.append((qc, sc, qb))
            wbytes = 1.0 + 4.0 / 32
        else:
            lin = h3.make_linear(w, b)
        _, _, pos = synth.packed_rows(synth.CONFIGS["block12936"])
        pos_d = torch.from_numpy(np.ascontiguousarray(np.resize(pos, (n, 3)))).cuda()
        ld = (n + 63) // 64 * 64
        q = torch.empty(nh, n, hd, dtype=torch.bfloat16, device="cuda")
        k, vt = torch.empty_like(q), torch.empty(nh, hd, ld, dtype=torch.bfloat16, device="cuda")
        qn, kn = _normal((hd,), 0.02, 1.0, stream=23), _normal((hd,), 0.02, 1.0, stream=24)
        ws = torch.empty(h3.h3_qkv_project_workspace_size(dims, n), dtype=torch.uint8, device="cuda")
        keep += [xn, w, b, lin, pos_d, q, k, vt, qn, kn, ws]

        def launch():
            h3.h3_qkv_project(dims, lin, xn.data_ptr(), pos_d.data_ptr(), qn.data_ptr(), kn.data_ptr(), q.data_ptr(),
                              k.data_ptr(), vt.data_ptr(), ld, n, ws.data_ptr(), ws.numel(), 0, st)

        byts = n * H * 2.0 + 3 * I * H * wbytes + 3.0 * n * I * 2 + n * hd * 4.0
        return launch, 2.0 * n * H * 3 * I, byts, "includes the per-row cos/sin table kernel", keep

    if kernel in ("embed", "head"):
        # video-latent rows: the input patch projection (96 -> H) or the final AdaLN + output head
        # (H -> 96) with the Euler update of the float32 latents, float32 weights
        K = synth.VIDEO_FEATURES
        f32 = lambda shape, s_, std=1.0: torch.randn(shape, generator=torch.Generator("cuda").manual_seed(s_),  # noqa
                                                     device="cuda") * std
        x = _normal((n, H), stream=40)
        z = f32((n, K), 41)
        if kernel == "embed":
            w, b = f32((H, K), 42, 0.02), f32((H,), 43, 0.02)
            keep += [x, z, w, b]

            def launch():
                h3.h3_embed_rows(dims, z.data_ptr(), K, w.data_ptr(), b.data_ptr(), n, x.data_ptr(), st)

            return launch, 2.0 * n * H * K, n * K * 4.0 + H * K * 4.0 + n * H * 2.0, "float32 CUDA-core", keep
        w, b = f32((K, H), 44, 0.02), f32((K,), 45, 0.02)
        table = _normal((1, 6 * H), 0.5, stream=46)
        tag_d = torch.full((n,), 2, dtype=torch.uint8, device="cuda")
        tidx_d = torch.zeros(n, dtype=torch.int32, device="cuda")
        keep += [x, z, w, b, table, tag_d, tidx_d]

        def launch():
            h3.h3_head_forward(dims, x.data_ptr(), n, tag_d.data_ptr(), tidx_d.data_ptr(), table.data_ptr(), 6 * H,
                               w.data_ptr(), b.data_ptr(), K, None, z.data_ptr(), -0.01, st)

        return launch, 2.0 * n * H * K, n * H * 2.0 + 2 * n * K * 4.0, "float32 CUDA-core; with the Euler update", keep

    if kernel == "modcache":
        T = n
        temb = torch.from_numpy(synth.sinusoidal_temb(list(range(T)), d.temb_dim)).cuda()
        Ws = [_normal((18 * H, d.temb_dim), 0.02, stream=16 + 2 * i) for i in range(blocks)]
        bs = [_normal((18 * H,), 0.02, stream=17 + 2 * i) for i in range(blocks)]
        table = torch.empty(T, blocks, 18 * H, dtype=torch.bfloat16, device="cuda")
        keep += [temb, table] + Ws + bs

        def launch():
            h3.h3_modcache_build(dims, temb.data_ptr(), T, d.temb_dim, [W.data_ptr() for W in Ws],
                                 [b.data_ptr() for b in bs], blocks, table.data_ptr(), st)

        byts = blocks * (18.0 * H * d.temb_dim * 2 + 18 * H * 2) + T * d.temb_dim * 4 + T * blocks * 18 * H * 2
        return (launch, 2.0 * T * blocks * 18 * H * d.temb_dim, byts,
                f"rows = timesteps T; {blocks} blocks' adaln_proj", keep)

    raise ValueError(kernel)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", choices=KERNELS, required=True)
    ap.add_argument("--rows", type=int, default=12936)
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--int8", action="store_true")
    ap.add_argument("--density", type=float, default=0.25, help="attention_sparse: fraction of kept tiles")
    ap.add_argument("--blocks", type=int, default=1, help="modcache: blocks whose tables one call builds")
    a = ap.parse_args(argv)
    torch.cuda.set_device(0)
    launch, flop, byts, note, _keep = setup(a.kernel, a.rows, a.int8, a.density, a.blocks)
    for _ in range(a.warmup):
        launch()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.reps):
        launch()
    e1.record()
    torch.cuda.synchronize()
    st, site = h3.h3_last_device_error(h3.stream_ptr())
    if st != h3.H3_OK:
        raise RuntimeError(f"device error word set: site {site:#x}")
    ms = e0.elapsed_time(e1) / a.reps
    out = {"kernel": a.kernel, "rows": a.rows, "int8": a.int8, "ms": ms, "flop": flop, "bytes": byts,
           "tflops": flop / ms / 1e9, "gbs": byts / ms / 1e6, "note": note}
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
