#!/usr/bin/env python
"""Benchmark: DiT trunk tokens/s per denoiser step on one B300 (plus attn+GEMM % of bf16 peak).

A step is one denoiser evaluation of the 50-block H3 trunk (h3_trunk_forward) over the packed
33,720-row sequence of a 768p 5 s Ref2VA request (text 256, one image condition 1,008, audio
200, video 32x24x42), bf16 weights and activations, all inputs resident in HBM.  The
modulation table (77 timesteps) is built once by h3_modcache_build before timing, as a run
does.  Weights are random (seeded), so `data` is synthetic.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the same workload (the path
has no data-parallel split inside one forward); value is the whole-job tokens/s.
`--impl reference` times the CPU oracle (the only reference implementation of this path) on a
bounded sample of the same workload, on rank 0.
"""

from __future__ import annotations

import argparse
import functools
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "DiT trunk tokens/s per denoiser step"
UNIT = "tokens/s"
CPU_SAMPLE_ROWS = 384


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6400.0, 1800.0, 1400.0, "fallback"


def _attention_traffic(n_rows):
    """DRAM bytes per attention launch at n_rows, from the ncu capture recorded in
    profiles/attention_traffic.json, scaled by rows (Q, K, V and O are each read or written once
    per launch while K/V tiles stay L2-resident, so traffic grows with N); None when there is no
    capture or the kernel source has changed since it was taken."""
    import hashlib

    try:
        with open(os.path.join(ROOT, "profiles", "attention_traffic.json")) as f:
            rec = json.load(f)
        src = open(os.path.join(ROOT, rec["source"]), "rb").read()
        if hashlib.sha256(src).hexdigest() != rec["source_sha256"]:
            return None
        return int(rec["traffic_bytes_per_launch"]) * n_rows / int(rec["rows"])
    except (OSError, KeyError, ValueError):
        return None


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The largest value of x over all ranks (x itself without a process group): the job's
    time is the slowest replica's."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, rows: int, steps: int, seconds: float) -> float:
    """Tokens per second of the whole job: every replica processes `rows` tokens per step."""
    return world * rows * steps / seconds


def _flops(cfg, n_rows):
    """(linear, attention) MMA FLOP of one block."""
    d = cfg.dims
    lin = 2 * n_rows * (3 * d.inner * d.hidden + d.hidden * d.inner + 2 * d.ffn * d.hidden + d.hidden * d.ffn)
    return lin, 4 * n_rows * n_rows * d.inner


# ------------------------------------------------------------------------------ clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id, rank, path=None):
        import tempfile

        self.bus = bus_id
        self.proc = None
        self.path = path or os.path.join(tempfile.gettempdir(), f"h3_bench_clocks_rank{rank}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            sel = ["-i", self.bus] if self.bus else []
            self.proc = subprocess.Popen(["nvidia-smi"] + sel + [f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------ CPU oracle leg


@functools.lru_cache(maxsize=2)
def _oracle_inputs(cfg, rows, step):
    """The sampled rows' inputs for the oracle leg, drawn once per process (generating a
    full-width block's weights takes longer than the timed block forward itself)."""
    import oracle.h3_oracle as O

    tag, tidx, pos = synth.packed_rows(cfg, step=step)
    sel = np.sort(np.random.default_rng(0).choice(cfg.layout.n_rows, rows, replace=False))
    sub = synth.Config(cfg.name + "_sample", cfg.dims, cfg.layout, cfg.seed, timesteps=cfg.timesteps,
                       n_timesteps=cfg.n_timesteps)
    x = synth.normal_bf16(cfg.seed, 0xABCD, (rows, cfg.dims.hidden))
    w = synth.block_weights(sub, 0)
    aw, ab = synth.adaln_weights(sub, 0)
    used = np.unique(tidx[sel])
    temb = synth.sinusoidal_temb(np.asarray(cfg.timesteps)[used], cfg.dims.temb_dim)
    _, tbf = O.modcache(temb, [aw], [ab])
    remap = {int(t): i for i, t in enumerate(used)}
    tl = np.array([remap[int(t)] for t in tidx[sel]], np.int32)
    return x, w, tbf[:, 0, :], tag[sel], tl, pos[sel]


def cpu_oracle_sample(cfg, rows=CPU_SAMPLE_ROWS, step=10):
    """Time the CPU oracle on one full-width block over `rows` rows sampled from the packed
    sequence (same tags, positions and timestep mix), then scale by the FLOP model to the
    whole trunk.  Returns (tokens/s, seconds, threads, description)."""
    import oracle.h3_oracle as O

    try:
        from threadpoolctl import threadpool_info

        threads = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        threads = os.cpu_count() or 1
    rows = min(rows, cfg.layout.n_rows)
    x, w, tb, tag, tl, pos = _oracle_inputs(cfg, rows, step)
    t0 = time.perf_counter()
    O.block_forward(x, w, tb, tag, tl, pos, cfg.dims)
    dt = time.perf_counter() - t0
    lin_s, att_s = _flops(cfg, rows)
    rate = (lin_s + att_s) / dt
    lin, att = _flops(cfg, cfg.layout.n_rows)
    trunk_s = cfg.n_blocks * (lin + att) / rate
    desc = (f"one full-width block over {rows} rows sampled from the {cfg.layout.n_rows}-row sequence, "
            f"{dt:.2f} s ({rate / 1e9:.1f} GFLOP/s fp64); scaled by the FLOP model to {cfg.n_blocks} blocks "
            f"at {cfg.layout.n_rows} rows")
    return cfg.layout.n_rows / trunk_s, dt, threads, desc


def run_reference(args, cfg, rank):
    if rank != 0:
        return
    vals = []
    for i in range(args.warmup + args.steps):
        v, dt, threads, desc = cpu_oracle_sample(cfg)
        if i >= args.warmup:
            vals.append((v, dt))
    value = statistics.median(v for v, _ in vals)
    ms = statistics.median(cfg.layout.n_rows / v * 1e3 for v, _ in vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "rows": cfg.layout.n_rows, "blocks": cfg.n_blocks},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ GPU arm


BLOCK_WORKLOADS = ("block1829", "block12936", "block12936_int8")


def time_single_blocks(dev, sp, reps=20, warmup=5):
    """One full-width DiT block (h3_block_forward) per configuration: 1,829 and 12,936 packed
    rows with bf16 weights, and 12,936 rows with weight-only INT8-g32 weights.  Device-drawn
    weights (seeded), the block's table built by h3_modcache_build, CUDA events around `reps`
    back-to-back launches after `warmup`; the block's 0.77 GB of weights (0.43 GB as INT8)
    exceed L2, so every launch streams them from HBM."""
    import torch

    from joint_video_audio_block_b300 import h3
    from joint_video_audio_block_b300 import runtime as R

    _, bf16_peak, _, peak_kind = _peaks()
    out = {}
    for name in BLOCK_WORKLOADS:
        cfg = synth.CONFIGS[name]
        d = cfg.dims
        dims = R.dims_of(d)
        N = cfg.layout.n_rows
        w = synth.device_block_weights(cfg, 0)
        if cfg.int8:
            for lname in ("wqkv", "wo", "w1", "w2"):
                w[lname], w[lname + "_scale"], w[lname + "_qbias"] = synth.device_quantize_int8_g32(w[lname])
        bw = h3.make_block_w(w)
        aw, ab = synth.device_adaln_weights(cfg, 0)
        temb = torch.from_numpy(synth.temb(cfg)).to(dev)
        T = temb.shape[0]
        table = torch.empty(T, 1, 18 * d.hidden, dtype=torch.bfloat16, device=dev)
        h3.h3_modcache_build(dims, temb.data_ptr(), T, d.temb_dim, [aw.data_ptr()], [ab.data_ptr()], 1,
                             table.data_ptr(), sp)
        del aw, ab
        tag, tidx, pos = (torch.from_numpy(a).to(dev) for a in synth.packed_rows(cfg))
        x = synth.device_normal_bf16(cfg.seed, 0xFFFF02, (N, d.hidden))
        y = torch.empty_like(x)
        ws = R.workspace(dims, N)

        def launch():
            h3.h3_block_forward(dims, bw, table.data_ptr(), 18 * d.hidden, T, x.data_ptr(), y.data_ptr(), N,
                                tag.data_ptr(), tidx.data_ptr(), pos.data_ptr(), ws.data_ptr(), ws.numel(), 0, sp)

        for _ in range(warmup):
            launch()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            launch()
        e1.record()
        torch.cuda.synchronize()
        st, site = h3.h3_last_device_error(sp)
        if st != h3.H3_OK:
            raise RuntimeError(f"device error timing {name}: site {site:#x}")
        ms = e0.elapsed_time(e1) / reps
        lin, att = _flops(cfg, N)
        out[name] = {"rows": N, "weights": "int8_g32" if cfg.int8 else "bf16", "ms_per_block": ms,
                     "tflops": (lin + att) / ms / 1e9, "frac_of_burst": (lin + att) / ms / 1e9 / bf16_peak,
                     "ms_at_60pct_of_burst": (lin + att) / (0.6 * bf16_peak * 1e12) * 1e3, "reps": reps,
                     "peak_kind": peak_kind}
        del w, bw, table, x, y, ws
        torch.cuda.empty_cache()
    return out


# The pages' own figure for the 37,966-row request: 8.8 min per 50-block denoising step on an M3
# Ultra (MLX, bf16, one block timed and multiplied by 50; "minimax-h3-mlx" README, "Performance").
# Another machine's number: context for the page-faithful canvas, not a target.
PAGES_M3_ULTRA_STEP_S = 8.8 * 60


def time_page_canvas(dev, sp, dims, bws, B, table, T, steps=2, warmup=1):
    """The same 50-block trunk (the resident weights and modulation table of the main workload)
    over the pages' 5 s, 1344x768 request: 37,966 packed rows, tokens/s per denoiser step, next
    to the pages' M3 Ultra figure for that request."""
    import torch

    from joint_video_audio_block_b300 import h3
    from joint_video_audio_block_b300 import runtime as R

    cfg = synth.CONFIGS["trunk37966"]
    d = cfg.dims
    N = cfg.layout.n_rows
    tag, tidx, pos = (torch.from_numpy(a).to(dev) for a in synth.packed_rows(cfg, step=10))
    x0 = synth.device_normal_bf16(cfg.seed, 0xFFFF03, (N, d.hidden))
    x = torch.empty_like(x0)
    ws = R.workspace(dims, N)

    def step():
        x.copy_(x0)
        h3.h3_trunk_forward(dims, bws, B, table.data_ptr(), T, x.data_ptr(), N, tag.data_ptr(), tidx.data_ptr(),
                            pos.data_ptr(), ws.data_ptr(), ws.numel(), 0, sp)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    st, site = h3.h3_last_device_error(sp)
    if st != h3.H3_OK:
        raise RuntimeError(f"device error timing the page canvas: site {site:#x}")
    s_per_step = e0.elapsed_time(e1) / 1e3 / steps
    lay = cfg.layout
    out = {"workload": cfg.name, "rows": N,
           "layout": f"text {lay.text} | audio {lay.audio} | video {'x'.join(map(str, lay.video))} "
                     "(a reading: the pages give only the total)",
           "blocks": B, "steps": steps, "ms_per_step": s_per_step * 1e3, "tokens_per_s": N / s_per_step,
           "pages_figure": {"s_per_step": PAGES_M3_ULTRA_STEP_S, "tokens_per_s": N / PAGES_M3_ULTRA_STEP_S,
                            "hardware": "M3 Ultra, MLX, bf16", "use": "context, another machine"}}
    del x0, x, ws
    torch.cuda.empty_cache()
    return out


def run_ours(args, cfg, rank, world, local_rank):
    import torch

    from joint_video_audio_block_b300 import h3
    from joint_video_audio_block_b300 import runtime as R

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    d = cfg.dims
    dims = R.dims_of(d)
    N, B, T = cfg.layout.n_rows, args.blocks or cfg.n_blocks, cfg.n_timesteps
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    # weights (device-side seeded draws), modulation table built once, adaln weights dropped
    blocks = [synth.device_block_weights(cfg, b) for b in range(B)]
    temb = torch.from_numpy(synth.temb(cfg)).cuda()
    table = torch.empty(T, B, 18 * d.hidden, dtype=torch.bfloat16, device=dev)
    adaln = [synth.device_adaln_weights(cfg, b) for b in range(B)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    h3.h3_modcache_build(dims, temb.data_ptr(), T, d.temb_dim, [w.data_ptr() for w, _ in adaln],
                         [b.data_ptr() for _, b in adaln], B, table.data_ptr(), sp)
    e1.record()
    torch.cuda.synchronize()
    modcache_ms = e0.elapsed_time(e1)
    modcache_bytes = B * 18 * d.hidden * (d.temb_dim + 1) * 2 + table.numel() * 2
    del adaln
    torch.cuda.empty_cache()

    tag, tidx, pos = synth.packed_rows(cfg, step=10)
    tag_d, tidx_d, pos_d = (torch.from_numpy(a).to(dev) for a in (tag, tidx, pos))
    x0 = synth.device_normal_bf16(cfg.seed, 0xFFFF01, (N, d.hidden))
    x = torch.empty_like(x0)
    ws = R.workspace(dims, N)
    bws = [h3.make_block_w(w) for w in blocks]

    def step():
        x.copy_(x0)
        h3.h3_trunk_forward(dims, bws, B, table.data_ptr(), T, x.data_ptr(), N, tag_d.data_ptr(), tidx_d.data_ptr(),
                            pos_d.data_ptr(), ws.data_ptr(), ws.numel(), 0, sp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, site = h3.h3_last_device_error(sp)
    if st != h3.H3_OK:
        raise RuntimeError(f"device error after warm-up: {h3.h3_status_str(st)} site {site:#x}")

    try:
        pr = torch.cuda.get_device_properties(dev)
        bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
    except Exception:
        bus = None
    clocks = ClockSampler(bus, rank, args.clocks_csv.replace("{rank}", str(rank)) if args.clocks_csv else None)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    h3.h3_kernel_timer_start(B * args.steps)  # events around every attention launch of the timed steps
    ta, tb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ta.record()
    for _ in range(args.steps):
        step()
    tb.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    att_durations = h3.h3_kernel_timer_read(B * args.steps)
    if dist:
        dist.barrier()
    elapsed = max_over_ranks(ta.elapsed_time(tb) / 1e3, dist, dev)
    st, site = h3.h3_last_device_error(sp)
    if st != h3.H3_OK:
        raise RuntimeError(f"device error in timed region: site {site:#x}")
    ms_per_step = elapsed / args.steps * 1e3
    value = whole_job_rate(world, N, args.steps, elapsed)

    # end to end: host (pinned) inputs in, result out, every step
    xh = x0.cpu().pin_memory()
    out_h = torch.empty_like(xh).pin_memory()
    tag_h, tidx_h, pos_h = (torch.from_numpy(a).pin_memory() for a in (tag, tidx, pos))
    h2d = xh.numel() * 2 + tag_h.numel() + tidx_h.numel() * 4 + pos_h.numel() * 4
    d2h = out_h.numel() * 2

    def e2e_step():
        x.copy_(xh, non_blocking=True)
        tag_d.copy_(tag_h, non_blocking=True)
        tidx_d.copy_(tidx_h, non_blocking=True)
        pos_d.copy_(pos_h, non_blocking=True)
        h3.h3_trunk_forward(dims, bws, B, table.data_ptr(), T, x.data_ptr(), N, tag_d.data_ptr(), tidx_d.data_ptr(),
                            pos_d.data_ptr(), ws.data_ptr(), ws.numel(), 0, sp)
        out_h.copy_(x, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist, dev)
    e2e_value = whole_job_rate(world, N, args.steps, e2e_s)

    # one whole sampler transition at the same workload: entry projections, the trunk, the
    # output heads and the Euler update of the float32 latents (h3_denoise_step)
    lay = cfg.layout
    L, C, A, V = lay.text, lay.n_cond, lay.audio, lay.n_video
    g = torch.Generator(device=dev)
    g.manual_seed(cfg.seed + 77)
    rnd = lambda *shape, std=1.0: torch.randn(*shape, generator=g, device=dev) * std  # noqa: E731
    kv, ka = synth.VIDEO_FEATURES, synth.AUDIO_FEATURES
    io_d = {"patch_v": rnd(d.hidden, kv, std=0.02), "patch_v_b": rnd(d.hidden, std=0.02),
            "patch_a": rnd(d.hidden, ka, std=0.02), "patch_a_b": rnd(d.hidden, std=0.02),
            "head_v": rnd(kv, d.hidden, std=0.02), "head_v_b": rnd(kv, std=0.02),
            "head_a": rnd(ka, d.hidden, std=0.02), "head_a_b": rnd(ka, std=0.02)}
    iow = h3.make_io_w(io_d, L, C, A, V, kv, ka)
    table_f = (rnd(T, 6 * d.hidden, std=0.5)).to(torch.bfloat16)
    text_x = x0[:L].clone()
    zc, zv, za = rnd(C, kv), rnd(V, kv), rnd(A, ka)

    def transition():
        h3.h3_denoise_step(dims, bws, B, table.data_ptr(), table_f.data_ptr(), T, iow, text_x.data_ptr(),
                           zc.data_ptr() if C else None, zv.data_ptr(), za.data_ptr(), x.data_ptr(), tag_d.data_ptr(),
                           tidx_d.data_ptr(), pos_d.data_ptr(), -0.01, -0.01, ws.data_ptr(), ws.numel(), 0, sp)

    transition()
    torch.cuda.synchronize()
    tc, td = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tc.record()
    for _ in range(2):
        transition()
    td.record()
    torch.cuda.synchronize()
    transition_ms = tc.elapsed_time(td) / 2

    hbm_peak, bf16_peak, bf16_sus, peak_kind = _peaks()
    lin_f, att_f = _flops(cfg, N)
    att_ms = statistics.mean(att_durations) if att_durations else float("nan")
    att_tflops = att_f / (att_ms / 1e3) / 1e12
    mma_tflops = B * (lin_f + att_f) / (ms_per_step / 1e3) / 1e12  # per GPU (each replica)
    traffic = _attention_traffic(N)

    canvas = None
    if not args.no_page_canvas and cfg.name == "trunk33720" and B == cfg.n_blocks:
        canvas = time_page_canvas(dev, sp, dims, bws, B, table, T)
    blocks_timed = None if args.no_block_workloads else time_single_blocks(dev, sp)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, threads, desc = cpu_oracle_sample(cfg)
        cpu = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": cfg.name, "rows": N, "blocks": B, "hidden": d.hidden, "heads": d.heads,
                       "head_dim": d.head_dim, "ffn": d.ffn, "timesteps_in_table": T,
                       "l2": "inputs larger than L2 (38.5 GB of weights streamed per step)",
                       "parallelism": f"replicas{world}"},
            "mma_frac_of_bf16_peak": {"tflops": mma_tflops, "burst": mma_tflops / bf16_peak,
                                      "sustained": mma_tflops / bf16_sus, "peak_kind": peak_kind},
            "roofline": {"kernel": "attention_tc_kernel<128>", "bound": "tensor", "achieved": att_tflops,
                         "peak": bf16_sus, "unit": "TFLOP/s", "frac": att_tflops / bf16_sus,
                         "peak_kind": f"{peak_kind} bf16 sustained (kernel timed inside the trunk step)",
                         "frac_of_burst": att_tflops / bf16_peak, "traffic": traffic,
                         "flop_per_launch": att_f, "ms_per_launch": att_ms, "launches_timed": len(att_durations)},
            "modcache": {"ms": modcache_ms, "timesteps": T, "blocks": B,
                         "GB_per_s": modcache_bytes / (modcache_ms / 1e3) / 1e9},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "sampler_transition": {"ms": transition_ms, "tokens_per_s": N / (transition_ms / 1e3),
                                   "what": "entry projections + trunk + output heads + Euler (h3_denoise_step)"},
            "single_block_workloads": blocks_timed,
            "page_canvas": canvas,
            "gpu_launches": args.steps * (1 + 7 * B),  # rope table + 7 kernels per block
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="trunk33720")
    ap.add_argument("--blocks", type=int, default=0, help="override the block count (diagnostics only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-block-workloads", action="store_true",
                    help="skip the per-block timings of the 1,829- and 12,936-row configurations")
    ap.add_argument("--no-page-canvas", action="store_true",
                    help="skip the pages' 37,966-row request (timed after the main workload)")
    ap.add_argument("--clocks-csv", default=None, help="where to keep the raw clock samples ({rank} is replaced)")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = synth.CONFIGS[args.workload]
    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return
    run_ours(args, cfg, rank, world, local_rank)


if __name__ == "__main__":
    main()
