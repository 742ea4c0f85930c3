"""GPU parity of the trunk's entry and exit and of the sampler's Euler transition, through the
C ABI against the CPU oracle on the same seeded inputs.

All three are float32 arithmetic on the GPU (float32 weights, as the released checkpoint ships
the patch projections and output heads).  Bounds: the bf16 output of the input projection is
within one bf16 ulp of the exact value plus the float32 accumulation bound K 2^-24 sum|w z|; the
float32 head output is within the float32 accumulation bound H 2^-24 sum|w xn| plus the
LayerNorm's own float32 error (the same bound again, generously); the Euler update adds its
own rounding of z."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA device", allow_module_level=True)

import oracle.h3_oracle as O  # noqa: E402
import synth  # noqa: E402
from joint_video_audio_block_b300 import h3, runtime as R  # noqa: E402

pytestmark = pytest.mark.gpu


def _sync():
    torch.cuda.synchronize()
    st, site = h3.h3_last_device_error(h3.stream_ptr())
    assert st == h3.H3_OK, f"device error {site:#x}"


def _segments(cfg):
    """(first row, rows) of the video-latent rows (conditions + video) and of the audio rows."""
    lay = cfg.layout
    cond0 = lay.text
    audio0 = cond0 + lay.n_cond
    video0 = audio0 + lay.audio
    return (cond0, lay.n_cond, video0, lay.n_video), (audio0, lay.audio)


@pytest.mark.parametrize("name", ["tiny", "block1829", "trunk33720"])
def test_embed_rows(name):
    cfg = synth.CONFIGS[name]
    d, n = cfg.dims, cfg.layout.n_rows
    H = d.hidden
    dims = R.dims_of(d)
    w = synth.io_weights(cfg)
    zv, za = synth.latents(cfg)
    (c0, nc, v0, nv), (a0, na) = _segments(cfg)
    x = torch.full((n, H), 7.0, dtype=torch.bfloat16, device="cuda")  # sentinel
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    pv, pvb, pa, pab = dev(w["patch_v"]), dev(w["patch_v_b"]), dev(w["patch_a"]), dev(w["patch_a_b"])
    zv_d, za_d = dev(zv), dev(za)
    st = h3.stream_ptr()
    row = lambda r: x.data_ptr() + r * H * 2  # noqa: E731
    if nc:
        h3.h3_embed_rows(dims, zv_d.data_ptr(), synth.VIDEO_FEATURES, pv.data_ptr(), pvb.data_ptr(), nc, row(c0), st)
    h3.h3_embed_rows(dims, zv_d[nc:].data_ptr(), synth.VIDEO_FEATURES, pv.data_ptr(), pvb.data_ptr(), nv, row(v0), st)
    h3.h3_embed_rows(dims, za_d.data_ptr(), synth.AUDIO_FEATURES, pa.data_ptr(), pab.data_ptr(), na, row(a0), st)
    _sync()
    got = R.f32_from_bf16(x).astype(np.float64)
    assert np.all(got[:c0] == 7.0)  # text rows untouched
    for z, W, b, r0, rows in ((zv[:nc], w["patch_v"], w["patch_v_b"], c0, nc), (zv[nc:], w["patch_v"], w["patch_v_b"], v0, nv),
                              (za, w["patch_a"], w["patch_a_b"], a0, na)):
        if rows == 0:
            continue
        ref = O.embed_rows(z, W, b)
        absum = np.abs(z.astype(np.float64)) @ np.abs(W.astype(np.float64)).T + np.abs(b.astype(np.float64))
        bound = 2.0 ** -8 * np.abs(ref) + z.shape[1] * 2.0 ** -24 * absum
        err = np.abs(got[r0:r0 + rows] - ref)
        assert np.all(err <= bound), f"{name} rows {r0}+{rows}: excess {np.max(err - bound):.3e}"


def _final_table(cfg):
    w = synth.io_weights(cfg)
    temb = synth.temb(cfg)
    t64, tbf = O.modcache(temb, [w["final_w"]], [w["final_b"]])
    return w, temb, t64[:, 0, :], tbf[:, 0, :]


@pytest.mark.parametrize("name", ["tiny", "trunk33720"])
def test_final_modcache_build(name):
    cfg = synth.CONFIGS[name]
    d = cfg.dims
    w, temb, t64, tbf = _final_table(cfg)
    T = t64.shape[0]
    table = torch.empty(T, 6 * d.hidden, dtype=torch.bfloat16, device="cuda")
    temb_d, w_d, b_d = torch.from_numpy(temb).cuda(), R.bf16_from_bits(w["final_w"]), R.bf16_from_bits(w["final_b"])
    h3.h3_final_modcache_build(R.dims_of(d), temb_d.data_ptr(), T, d.temb_dim, w_d.data_ptr(), b_d.data_ptr(),
                               table.data_ptr(), h3.stream_ptr())
    _sync()
    got = R.f32_from_bf16(table).astype(np.float64)
    absum = np.abs(temb.astype(np.float64)) @ np.abs(O.widen_bf16(w["final_w"])).T + np.abs(O.widen_bf16(w["final_b"]))
    excess = np.abs(got - t64) - (2.0 ** -8 * np.abs(t64) + 2.0 ** -20 * absum)
    assert np.all(excess <= 0), excess.max()


@pytest.mark.parametrize("name", ["tiny", "block1829", "trunk33720"])
@pytest.mark.parametrize("modality", ["video", "audio"])
def test_head_forward_and_euler(name, modality):
    cfg = synth.CONFIGS[name]
    d, n = cfg.dims, cfg.layout.n_rows
    H = d.hidden
    dims = R.dims_of(d)
    w, _, _, tbf = _final_table(cfg)
    (c0, nc, v0, nv), (a0, na) = _segments(cfg)
    r0, rows = (v0, nv) if modality == "video" else (a0, na)
    K = synth.VIDEO_FEATURES if modality == "video" else synth.AUDIO_FEATURES
    W, b = w["head_v" if modality == "video" else "head_a"], w["head_v_b" if modality == "video" else "head_a_b"]
    x_bits = synth.activations(cfg)[r0:r0 + rows]
    tag, tidx, _ = synth.packed_rows(cfg, step=3)
    tag, tidx = tag[r0:r0 + rows], tidx[r0:r0 + rows]
    T = tbf.shape[0]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    x = R.bf16_from_bits(x_bits)
    table = R.bf16_from_bits(O.to_bf16_bits(tbf))
    Wd, bd, tag_d, tidx_d = dev(W), dev(b), dev(tag), dev(tidx)
    z0 = synth.normal_f32(cfg.seed, 0xBEEF, (rows, K))
    z = dev(z0)
    v = torch.empty(rows, K, dtype=torch.float32, device="cuda")
    sig = O.shifted_sigmas(40, 12.0 if modality == "video" else 3.0)
    dsig = float(np.float32(sig[4]) - np.float32(sig[3]))
    h3.h3_head_forward(dims, x.data_ptr(), rows, tag_d.data_ptr(), tidx_d.data_ptr(), table.data_ptr(), 6 * H,
                       Wd.data_ptr(), bd.data_ptr(), K, v.data_ptr(), z.data_ptr(), dsig, h3.stream_ptr())
    _sync()
    assert T >= 1
    shift = O.final_modulation(tbf, tag, tidx, 0, H)
    scale = O.final_modulation(tbf, tag, tidx, 1, H)
    ref = O.head_forward(O.widen_bf16(x_bits), shift, scale, W, b, d.ln_eps)
    xn = O.adaln_modulate(O.widen_bf16(x_bits), shift, scale, d.ln_eps)
    absum = np.abs(xn) @ np.abs(W.astype(np.float64)).T + np.abs(b.astype(np.float64))
    bound = 2 * H * 2.0 ** -24 * absum
    got_v = v.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got_v - ref) <= bound), f"head: excess {np.max(np.abs(got_v - ref) - bound):.3e}"
    rel = np.linalg.norm(got_v - ref) / np.linalg.norm(ref)
    print(f"head {name} {modality}: rel_l2={rel:.3e}")
    z_ref = O.euler_step(z0, ref, 0.0, dsig)
    bound_z = abs(dsig) * bound + 2.0 ** -24 * np.abs(z_ref) * 2
    assert np.all(np.abs(z.cpu().numpy() - z_ref) <= bound_z)


def test_denoise_steps_tiny():
    """Three sampler transitions of a 2-block tiny model end to end through h3_denoise_step
    against the oracle's composition (entry -> trunk -> heads -> Euler), with the run's own
    video (shift 12) and audio (shift 3) grids and per-row table rows per transition."""
    cfg = synth.CONFIGS["tiny"]
    d = cfg.dims
    H, n, B, S = d.hidden, cfg.layout.n_rows, 2, 3
    dims = R.dims_of(d)
    lay = cfg.layout
    L, C, A, V = lay.text, lay.n_cond, lay.audio, lay.n_video
    values, sv, sa, vidx, aidx = R.sampler_plan(S)
    # tables for the run's distinct timesteps (oracle-built bf16 values feed both sides)
    temb = synth.sinusoidal_temb(values, d.temb_dim)
    blocks = [synth.block_weights(cfg, b) for b in range(B)]
    aw = [synth.adaln_weights(cfg, b) for b in range(B)]
    _, tbf = O.modcache(temb, [a for a, _ in aw], [b for _, b in aw])
    io = synth.io_weights(cfg)
    _, tf = O.modcache(temb, [io["final_w"]], [io["final_b"]])
    tf = tf[:, 0, :]
    tag, _, pos = synth.packed_rows(cfg)
    text_bits = synth.activations(cfg)[:L]
    zv0, za0 = synth.latents(cfg)
    z_cond, z_video = zv0[:C], zv0[C:]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    # device state
    wts = [R.upload_block(w) for w in blocks]
    bws = [h3.make_block_w(w) for w in wts]
    io_d = {k: dev(v) for k, v in io.items() if k.startswith(("patch", "head"))}
    iow = h3.make_io_w(io_d, L, C, A, V)
    table = R.bf16_from_bits(O.to_bf16_bits(tbf))
    table_f = R.bf16_from_bits(O.to_bf16_bits(tf))
    text_x = R.bf16_from_bits(text_bits)
    zc_d, zv_d, za_d = dev(z_cond), dev(z_video), dev(za0)
    x = torch.empty(n, H, dtype=torch.bfloat16, device="cuda")
    tag_d, pos_d = dev(tag), dev(pos)
    tidx_d = torch.empty(n, dtype=torch.int32, device="cuda")
    ws = R.workspace(dims, n)
    T = len(values)
    # oracle state
    zv_ref, za_ref = z_video.astype(np.float64), za0.astype(np.float64)
    audio = slice(L + C, L + C + A)
    for i in range(S):
        R.step_tidx(tidx_d, audio, vidx[i], aidx[i])
        dsv, dsa = float(sv[i + 1] - sv[i]), float(sa[i + 1] - sa[i])
        h3.h3_denoise_step(dims, bws, B, table.data_ptr(), table_f.data_ptr(), T, iow, text_x.data_ptr(),
                           zc_d.data_ptr() if C else None, zv_d.data_ptr(), za_d.data_ptr(), x.data_ptr(),
                           tag_d.data_ptr(), tidx_d.data_ptr(), pos_d.data_ptr(), dsv, dsa, ws.data_ptr(), ws.numel(),
                           0, h3.stream_ptr())
        tidx = np.full(n, vidx[i], np.int32)
        tidx[audio] = aidx[i]
        za_ref, zv_ref = O.denoise_step(O.widen_bf16(text_bits), z_cond, za_ref, zv_ref, io, blocks, tbf, tf, tag, tidx,
                                        pos, d, dsv, dsa)
    _sync()
    # compare the distance the latents travelled (z itself is dominated by the initial noise)
    for got, ref, z0, what in ((zv_d, zv_ref, z_video, "video"), (za_d, za_ref, za0, "audio")):
        g = got.cpu().numpy().astype(np.float64) - z0
        r = ref - z0
        rel = np.linalg.norm(g - r) / np.linalg.norm(r)
        mx = np.abs(g - r).max() / np.abs(r).max()
        print(f"denoise {what}: moved rms {np.sqrt(np.mean(r * r)):.3e}; rel_l2={rel:.3e} max_abs/max|ref|={mx:.3e}")
        assert rel <= 1e-2 and mx <= 5e-2


def _head_case(name, modality):
    cfg = synth.CONFIGS[name]
    d, n = cfg.dims, cfg.layout.n_rows
    w, _, _, tbf = _final_table(cfg)
    (c0, nc, v0, nv), (a0, na) = _segments(cfg)
    r0, rows = (v0, nv) if modality == "video" else (a0, na)
    K = synth.VIDEO_FEATURES if modality == "video" else synth.AUDIO_FEATURES
    W, b = w["head_v" if modality == "video" else "head_a"], w["head_v_b" if modality == "video" else "head_a_b"]
    x_bits = synth.activations(cfg)[r0:r0 + rows]
    tag, tidx, _ = synth.packed_rows(cfg, step=3)
    return cfg, d, tbf, rows, K, W, b, x_bits, tag[r0:r0 + rows], tidx[r0:r0 + rows]


@pytest.mark.parametrize("name", ["tiny", "block1829"])
@pytest.mark.parametrize("modality", ["video", "audio"])
@pytest.mark.parametrize("where", ["first", "interior", "last"])
def test_head_forward_res_multistep(name, modality, where):
    """The output head with the res_multistep update against the oracle's head and step, on
    the run's own 20-step grid: the first step (first order; the previous-prediction buffer
    holds NaN and must not be read), an interior second-order step, and the step to 0 (which
    returns the prediction).  float32 on the GPU: the head's bound, carried through
    D = z - sigma v, plus the rounding of the three-term update and of the float32 weights."""
    cfg, d, tbf, rows, K, W, b, x_bits, tag, tidx = _head_case(name, modality)
    H = d.hidden
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    x = R.bf16_from_bits(x_bits)
    table = R.bf16_from_bits(O.to_bf16_bits(tbf))
    Wd, bd, tag_d, tidx_d = dev(W), dev(b), dev(tag), dev(tidx)
    sig = O.shifted_sigmas(20, 12.0 if modality == "video" else 3.0).astype(np.float64)
    i = {"first": 0, "interior": 7, "last": 19}[where]
    prev = None if i == 0 else float(sig[i - 1])
    step = h3.h3_res_multistep_step(prev, float(sig[i]), float(sig[i + 1]))
    z0 = synth.normal_f32(cfg.seed, 0xBEEF, (rows, K))
    dp0 = synth.normal_f32(cfg.seed, 0xD0D0, (rows, K))
    z = dev(z0)
    dp = torch.full((rows, K), float("nan"), device="cuda") if prev is None else dev(dp0)
    v = torch.empty(rows, K, dtype=torch.float32, device="cuda")
    h3.h3_head_forward_ms(R.dims_of(d), x.data_ptr(), rows, tag_d.data_ptr(), tidx_d.data_ptr(), table.data_ptr(),
                          6 * H, Wd.data_ptr(), bd.data_ptr(), K, step, v.data_ptr(), z.data_ptr(), dp.data_ptr(),
                          h3.stream_ptr())
    _sync()
    shift = O.final_modulation(tbf, tag, tidx, 0, H)
    scale = O.final_modulation(tbf, tag, tidx, 1, H)
    ref_v = O.head_forward(O.widen_bf16(x_bits), shift, scale, W, b, d.ln_eps)
    xn = O.adaln_modulate(O.widen_bf16(x_bits), shift, scale, d.ln_eps)
    bound_v = 2 * H * 2.0 ** -24 * (np.abs(xn) @ np.abs(W.astype(np.float64)).T + np.abs(b.astype(np.float64)))
    got_v = v.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got_v - ref_v) <= bound_v)
    z_ref, d_ref = O.res_multistep_step(z0, ref_v, prev, float(sig[i]), float(sig[i + 1]),
                                        d_prev=None if prev is None else dp0)
    a, cn, cp = O.res_multistep_coefficients(prev, float(sig[i]), float(sig[i + 1]))
    s = float(sig[i])
    bound_d = s * bound_v + 2.0 ** -23 * (np.abs(z0) + s * np.abs(ref_v))
    np.testing.assert_array_less(np.abs(dp.cpu().numpy() - d_ref), bound_d + 1e-30)
    mag = abs(a) * np.abs(z0) + abs(cn) * np.abs(d_ref) + (abs(cp) * np.abs(dp0) if cp else 0.0)
    bound_z = abs(cn) * bound_d + 2.0 ** -21 * mag
    err = np.abs(z.cpu().numpy() - z_ref)
    assert np.all(np.isfinite(z.cpu().numpy()))
    assert np.all(err <= bound_z), f"excess {np.max(err - bound_z):.3e}"
    if where == "last":  # the step to 0 is the prediction itself, bit for bit
        np.testing.assert_array_equal(z.cpu().numpy(), dp.cpu().numpy())


def test_denoise_run_res_multistep_tiny():
    """A whole 4-step run of a 2-block tiny model through h3_denoise_step_ms -- the first
    (first-order) step, two second-order steps and the step to 0 -- against the oracle's
    composition with the same grids (video shift 12, audio shift 3) and table rows."""
    cfg = synth.CONFIGS["tiny"]
    d = cfg.dims
    H, n, B, S = d.hidden, cfg.layout.n_rows, 2, 4
    dims = R.dims_of(d)
    lay = cfg.layout
    L, C, A, V = lay.text, lay.n_cond, lay.audio, lay.n_video
    values, sv, sa, vidx, aidx = R.sampler_plan(S)
    temb = synth.sinusoidal_temb(values, d.temb_dim)
    blocks = [synth.block_weights(cfg, b) for b in range(B)]
    aw = [synth.adaln_weights(cfg, b) for b in range(B)]
    _, tbf = O.modcache(temb, [a for a, _ in aw], [b for _, b in aw])
    io = synth.io_weights(cfg)
    _, tf = O.modcache(temb, [io["final_w"]], [io["final_b"]])
    tf = tf[:, 0, :]
    tag, _, pos = synth.packed_rows(cfg)
    text_bits = synth.activations(cfg)[:L]
    zv0, za0 = synth.latents(cfg)
    z_cond, z_video = zv0[:C], zv0[C:]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    wts = [R.upload_block(w) for w in blocks]
    bws = [h3.make_block_w(w) for w in wts]
    io_d = {k: dev(v) for k, v in io.items() if k.startswith(("patch", "head"))}
    iow = h3.make_io_w(io_d, L, C, A, V)
    table = R.bf16_from_bits(O.to_bf16_bits(tbf))
    table_f = R.bf16_from_bits(O.to_bf16_bits(tf))
    text_x = R.bf16_from_bits(text_bits)
    zc_d, zv_d, za_d = dev(z_cond), dev(z_video), dev(za0)
    dv_d = torch.empty_like(zv_d)
    da_d = torch.empty_like(za_d)
    x = torch.empty(n, H, dtype=torch.bfloat16, device="cuda")
    tag_d, pos_d = dev(tag), dev(pos)
    tidx_d = torch.empty(n, dtype=torch.int32, device="cuda")
    ws = R.workspace(dims, n)
    T = len(values)
    zv_ref, za_ref = z_video.astype(np.float64), za0.astype(np.float64)
    dv_ref = da_ref = None
    audio = slice(L + C, L + C + A)
    svd, sad = sv.astype(np.float64), sa.astype(np.float64)
    for i in range(S):
        R.step_tidx(tidx_d, audio, vidx[i], aidx[i])
        pv = None if i == 0 else float(svd[i - 1])
        pa = None if i == 0 else float(sad[i - 1])
        stv = h3.h3_res_multistep_step(pv, float(svd[i]), float(svd[i + 1]))
        sta = h3.h3_res_multistep_step(pa, float(sad[i]), float(sad[i + 1]))
        h3.h3_denoise_step_ms(dims, bws, B, table.data_ptr(), table_f.data_ptr(), T, iow, text_x.data_ptr(),
                              zc_d.data_ptr() if C else None, zv_d.data_ptr(), za_d.data_ptr(), dv_d.data_ptr(),
                              da_d.data_ptr(), x.data_ptr(), tag_d.data_ptr(), tidx_d.data_ptr(), pos_d.data_ptr(),
                              stv, sta, ws.data_ptr(), ws.numel(), 0, h3.stream_ptr())
        tidx = np.full(n, vidx[i], np.int32)
        tidx[audio] = aidx[i]
        za_ref, zv_ref, da_ref, dv_ref = O.denoise_step_multistep(
            O.widen_bf16(text_bits), z_cond, za_ref, zv_ref, io, blocks, tbf, tf, tag, tidx, pos, d,
            (pv, float(svd[i]), float(svd[i + 1])), (pa, float(sad[i]), float(sad[i + 1])),
            d_prev_video=dv_ref, d_prev_audio=da_ref)
    _sync()
    for got, ref, z0, what in ((zv_d, zv_ref, z_video, "video"), (za_d, za_ref, za0, "audio")):
        g = got.cpu().numpy().astype(np.float64) - z0
        r = ref - z0
        rel = np.linalg.norm(g - r) / np.linalg.norm(r)
        mx = np.abs(g - r).max() / np.abs(r).max()
        print(f"res_multistep run {what}: moved rms {np.sqrt(np.mean(r * r)):.3e}; rel_l2={rel:.3e} "
              f"max_abs/max|ref|={mx:.3e}")
        assert rel <= 1e-2 and mx <= 5e-2
