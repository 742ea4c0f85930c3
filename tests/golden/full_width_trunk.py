"""Inputs and stored oracle values of the full-width 50-block trunk parity test.

The workload: the H3 block geometry at full width (hidden 5376, 56 heads of 128, SwiGLU 14336;
"minimax-h3-mlx" README, "Architecture"), 50 blocks deep, over the 1,829 packed rows of the
512x512 22-frame canvas (text 256, audio 37, video 6x16x16), per-row modality tags, and the
video and audio rows at the two different timesteps one sampling step of a 40-step run uses
(video shift 12.0, audio shift 3.0; "AdaLN precompute").  Seeded synthetic weights (synth,
config "trunk50x1829").

The modulation table holds the two timesteps this step reads (the 77-entry table's rows for
them, built by the oracle's ModulationCache from the sinusoidal timestep embedding), so tidx is
renumbered 0 / 1 into it.  Building all 77 rows would change nothing the trunk reads.

Run as a script, this file writes `trunk50x1829_golden.npz` beside it: the exact oracle trunk
(float64 arithmetic, 50 blocks over every row) at 32 seeded rows, and the distance of the
bf16-storage oracle (bf16 rounding at the GPU's storage points, exact arithmetic elsewhere)
from it on the same rows.  It calls only oracle/ and synth; nothing in it comes from the CUDA
library.  About 20 minutes of fp64 on 8 host cores.
"""

from __future__ import annotations

import json
import os
import sys
import time

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(os.path.dirname(_HERE))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

import oracle.h3_oracle as O  # noqa: E402
import synth  # noqa: E402

CONFIG = "trunk50x1829"
STEP = 3                      # sampling step whose two timesteps the rows use
GOLDEN = os.path.join(_HERE, "trunk50x1829_golden.npz")
GOLDEN_ROWS = 32


def inputs():
    """(cfg, x bits [N, H], tag, tidx renumbered into the table, pos, table_bf [2, 50, 18H])."""
    cfg = synth.CONFIGS[CONFIG]
    x = synth.activations(cfg)
    tag, tidx, pos = synth.packed_rows(cfg, step=STEP)
    used = np.unique(tidx)
    temb = synth.temb(cfg)[used]
    tables = []
    for b in range(cfg.n_blocks):
        w, bias = synth.adaln_weights(cfg, b)
        _, tb = O.modcache(temb, [w], [bias])
        tables.append(tb[:, 0, :])
    table_bf = np.stack(tables, axis=1)
    tidx_r = np.searchsorted(used, tidx).astype(np.int32)
    return cfg, x, tag, tidx_r, pos, table_bf


def golden_rows(n_rows: int) -> np.ndarray:
    return np.sort(np.random.default_rng(13).choice(n_rows, GOLDEN_ROWS, replace=False))


def rel_errors(got, ref):
    """(relative L2, max-abs / max|ref|) of got against ref."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    mx = float(np.abs(got - ref).max()) / max(float(np.abs(ref).max()), 1e-300)
    return float(rel), mx


def main():
    t0 = time.time()
    cfg, x, tag, tidx, pos, table_bf = inputs()
    d = cfg.dims
    xe = x  # exact chain
    xb = x  # bf16-storage chain
    for b in range(cfg.n_blocks):
        w = synth.block_weights(cfg, b)
        xe = O.block_forward(xe, w, table_bf[:, b, :], tag, tidx, pos, d)
        xb = O.block_forward(xb, w, table_bf[:, b, :], tag, tidx, pos, d, emulate_bf16=True)
        print(f"block {b}: {time.time() - t0:.0f} s, max|x| {np.abs(xe).max():.3g}", flush=True)
    rows = golden_rows(xe.shape[0])
    r_rows, m_rows = rel_errors(xb[rows], xe[rows])
    r_all, m_all = rel_errors(xb, xe)
    meta = {
        "config": CONFIG, "step": STEP, "rows": GOLDEN_ROWS,
        "bf16_storage_rel_l2_rows": r_rows, "bf16_storage_max_abs_rows": m_rows,
        "bf16_storage_rel_l2_all": r_all, "bf16_storage_max_abs_all": m_all,
        "max_abs_ref": float(np.abs(xe).max()),
        "written_by": "tests/golden/full_width_trunk.py (oracle/ and synth only)",
    }
    np.savez_compressed(GOLDEN, rows=rows, ref=xe[rows].astype(np.float32), meta=json.dumps(meta))
    print(json.dumps(meta, indent=1))


if __name__ == "__main__":
    main()
