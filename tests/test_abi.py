"""The C-ABI library without a GPU: it loads, exports every entry point include/h3.h declares,
and its host-side logic (workspace plan, argument checks, status strings) behaves."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "h3.h")


@pytest.fixture(scope="module")
def h3mod():
    from joint_video_audio_block_b300 import build

    build.build()
    from joint_video_audio_block_b300 import h3

    h3.lib()
    return h3


def _no_gpu() -> bool:
    try:
        import torch

        return not torch.cuda.is_available()
    except ImportError:  # pragma: no cover
        return True


# Tests that hand the library fake device addresses rely on the host checks refusing the call
# before any launch; they run only where no GPU exists, so a regressed check can never turn
# into a launch on those addresses.
fake_addresses = pytest.mark.skipif(not _no_gpu(), reason="fake device addresses: host-only test")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:h3_status|size_t|const char\s*\*)\s+(h3_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("h3_modcache_build", "h3_block_forward", "h3_trunk_forward"):
        assert n in names
    assert len(names) >= 10


def test_library_exports_every_declared_symbol(h3mod):
    L = h3mod.lib()
    for name in _declared():
        assert hasattr(L, name), name
    assert sorted(h3mod.EXPORTS) == _declared()


def test_status_strings(h3mod):
    assert h3mod.h3_status_str(0) == "ok"
    assert "invalid" in h3mod.h3_status_str(1)
    assert h3mod.h3_status_str(99) == "unknown status"


def _tiny_dims(h3mod):
    import synth

    from joint_video_audio_block_b300 import runtime as R

    return R.dims_of(synth.TINY)


def test_workspace_plan(h3mod):
    import synth

    d = _tiny_dims(h3mod)
    n = 72
    D = synth.TINY
    a = lambda b: (b + 255) // 256 * 256  # noqa: E731
    ld_vt = (n + 63) // 64 * 64
    expect = (a(n * D.head_dim // 2 * 8) + a(n * D.hidden * 2) + a(n * max(3 * D.inner, D.ffn) * 2)
              + 2 * a(n * D.inner * 2) + a(D.heads * D.head_dim * ld_vt * 2) + a(n * D.inner * 2))
    assert h3mod.h3_workspace_size(d, n) == expect
    assert h3mod.h3_workspace_size(d, 0) == 0
    # grows with rows; invalid dims give 0
    assert h3mod.h3_workspace_size(d, 1000) > h3mod.h3_workspace_size(d, 72)
    bad = h3mod.make_dims(100, 4, 64, 512, (8, 12, 12))
    assert h3mod.h3_workspace_size(bad, 72) == 0
    bad = h3mod.make_dims(192, 4, 64, 512, (8, 12, 11))  # sections must sum to hd/2
    assert h3mod.h3_workspace_size(bad, 72) == 0


@fake_addresses
def test_invalid_arguments_rejected_before_launch(h3mod):
    """Null pointers and inconsistent shapes return H3_EINVAL on the host: no CUDA call runs."""
    L = h3mod.lib()
    d = _tiny_dims(h3mod)
    bw = h3mod.h3_block_w()
    st = L.h3_block_forward(ctypes.byref(d), ctypes.byref(bw), None, 0, 1, None, None, 72, None, None, None, None, 0,
                            0, None)
    assert st == h3mod.H3_EINVAL
    st = L.h3_trunk_forward(ctypes.byref(d), None, 0, None, 1, None, 72, None, None, None, None, 0, 0, None)
    assert st == h3mod.H3_EINVAL
    st = L.h3_modcache_build(ctypes.byref(d), None, 1, 96, None, None, 1, None, None)
    assert st == h3mod.H3_EINVAL
    lin = h3mod.h3_linear()
    st = L.h3_linear_forward(ctypes.byref(lin), 0, None, 0, None, 0, 1, None, None, 0, 0, None, None, 0, None)
    assert st == h3mod.H3_EINVAL
    st = L.h3_attention(ctypes.byref(d), None, None, None, 72, None, 72, 0, None)
    assert st == h3mod.H3_EINVAL


def test_sigma_schedule_is_the_oracle_grid(h3mod):
    """Host-only entry point (no GPU): the library's sampling grid equals the oracle's float32
    linspace + time shift bit for bit."""
    import numpy as np

    import oracle.h3_oracle as O

    for steps, shift in ((40, 12.0), (40, 3.0), (8, 12.0), (77, 1.0), (1, 3.0)):
        got = np.asarray(h3mod.h3_sigma_schedule(steps, shift), np.float32)
        np.testing.assert_array_equal(got, O.shifted_sigmas(steps, shift))


@fake_addresses
def test_more_invalid_arguments_rejected_before_launch(h3mod):
    """Misalignment and range errors of the newer entry points are refused on the host."""
    L = h3mod.lib()
    d = _tiny_dims(h3mod)
    odd = 0x1000 + 2  # not 16-byte aligned (never dereferenced: the call must refuse first)
    al = 0x2000
    # attention: misaligned q; sparse attention: no mask
    assert L.h3_attention(ctypes.byref(d), odd, al, al, 72, al, 72, 0, None) == h3mod.H3_EINVAL
    assert L.h3_attention_sparse(ctypes.byref(d), al, al, al, 72, al, 72, None, None) == h3mod.H3_EINVAL
    # ld_vt must cover the rows and be a multiple of 8
    assert L.h3_attention(ctypes.byref(d), al, al, al, 70, al, 72, 0, None) == h3mod.H3_EINVAL
    # entry / exit: bad widths, both outputs missing, misaligned rows
    assert L.h3_embed_rows(ctypes.byref(d), al, 0, al, None, 8, al, None) == h3mod.H3_EINVAL
    assert L.h3_embed_rows(ctypes.byref(d), al, 96, al, None, 8, odd, None) == h3mod.H3_EINVAL
    assert L.h3_head_forward(ctypes.byref(d), al, 8, al, al, al, 6 * 192, al, None, 96, None, None,
                             ctypes.c_float(0.0), None) == h3mod.H3_EINVAL
    assert L.h3_head_forward(ctypes.byref(d), al, 8, al, al, al, 6 * 192, al, None, 129, al, None,
                             ctypes.c_float(0.0), None) == h3mod.H3_EINVAL
    assert L.h3_head_forward(ctypes.byref(d), al, 8, al, al, al, 5 * 192, al, None, 96, al, None,
                             ctypes.c_float(0.0), None) == h3mod.H3_EINVAL
    # sampler grid: no steps / non-positive shift
    buf = (ctypes.c_float * 4)()
    assert L.h3_sigma_schedule(0, ctypes.c_float(3.0), buf) == h3mod.H3_EINVAL
    assert L.h3_sigma_schedule(3, ctypes.c_float(0.0), buf) == h3mod.H3_EINVAL
    # the static-scratch variant refuses sizes beyond its array, and the wait diagnostic its range
    n = h3mod.H3_QKROPE_STATIC_MAX_PAIRS // 32 + 1  # head_dim 64 -> 32 pairs per row
    assert L.h3_qknorm_rope_static(ctypes.byref(d), al, al, None, None, al, al, al, (n + 63) // 64 * 64, n,
                                   None) == h3mod.H3_EINVAL
    assert L.h3_diag_expire_wait(0, None) == h3mod.H3_EINVAL
    assert L.h3_diag_expire_wait(2_000_000, None) == h3mod.H3_EINVAL
    # the timer: negative capacity
    assert L.h3_kernel_timer_start(-1) == h3mod.H3_EINVAL


@fake_addresses
def test_qknorm_rope_entry_points_refuse_misaligned_pointers(h3mod):
    """Both QK-norm + RoPE entry points refuse, on the host, any pointer the kernel would access
    with a vector width it is not aligned to (qkv, q_out, k_out, vt_out: 16 bytes; pos: 4), and
    the allocation-free one refuses the same geometry errors as the workspace one."""
    L = h3mod.lib()
    d = _tiny_dims(h3mod)
    al, ws = 0x10000, 0x20000
    n, ld = 0, 128  # zero rows: a valid call returns H3_OK right after its checks, launching nothing
    base = [al, al, None, None, al, al, al, ld, n]

    def call(args, static):
        qkv, pos, qn, kn, q, k, vt, ldv, rows = args
        if static:
            return L.h3_qknorm_rope_static(ctypes.byref(d), qkv, pos, qn, kn, q, k, vt, ldv, rows, None)
        return L.h3_qknorm_rope(ctypes.byref(d), qkv, pos, qn, kn, q, k, vt, ldv, rows, ws, 1 << 20, None)

    for static in (False, True):
        assert call(base, static) == h3mod.H3_OK
        for slot, off in ((0, 2), (0, 8), (4, 2), (4, 8), (5, 4), (5, 8), (6, 8), (1, 2)):
            bad = list(base)
            bad[slot] = al + off
            assert call(bad, static) == h3mod.H3_EINVAL, (static, slot, off)
        bad = list(base)
        bad[7] = 76  # ld_vt not a multiple of 8
        assert call(bad, static) == h3mod.H3_EINVAL
        bad = list(base)
        bad[2] = al  # one norm weight without the other
        assert call(bad, static) == h3mod.H3_EINVAL
    # geometry the workspace entry point refuses is refused by the static one too
    for field, value in (("n_tags", 0), ("hidden", 0), ("ln_eps", -1.0)):
        dd = h3mod.make_dims(192, 4, 64, 512, (8, 12, 12))
        setattr(dd, field, value)
        assert L.h3_qknorm_rope_static(ctypes.byref(dd), al, al, None, None, al, al, al, ld, n, None) == \
            h3mod.H3_EINVAL
        assert L.h3_qknorm_rope(ctypes.byref(dd), al, al, None, None, al, al, al, ld, n, ws, 1 << 20, None) == \
            h3mod.H3_EINVAL


@fake_addresses
def test_modcache_build_refuses_misaligned_inputs(h3mod):
    """The table build reads the embedding by TMA (16-byte aligned rows) and the weights by TMA
    (16-byte aligned base): a misaligned embedding, weight or bias pointer, or an embedding
    width that is not a multiple of 8, is refused on the host."""
    L = h3mod.lib()
    d = _tiny_dims(h3mod)
    al, odd = 0x40000, 0x40000 + 4
    W = (ctypes.c_void_p * 2)(al, al)
    B = (ctypes.c_void_p * 2)(al, al)
    # valid arguments up to the launch would reach CUDA; every case below must stop before it
    assert L.h3_modcache_build(ctypes.byref(d), odd, 77, 96, W, B, 2, al, None) == h3mod.H3_EINVAL
    assert L.h3_modcache_build(ctypes.byref(d), al, 77, 92, W, B, 2, al, None) == h3mod.H3_EINVAL
    Wbad = (ctypes.c_void_p * 2)(al, odd)
    assert L.h3_modcache_build(ctypes.byref(d), al, 77, 96, Wbad, B, 2, al, None) == h3mod.H3_EINVAL
    Bbad = (ctypes.c_void_p * 2)(al, al + 1)
    assert L.h3_modcache_build(ctypes.byref(d), al, 77, 96, W, Bbad, 2, al, None) == h3mod.H3_EINVAL
    assert L.h3_final_modcache_build(ctypes.byref(d), odd, 77, 96, al, al, al, None) == h3mod.H3_EINVAL


def test_res_multistep_weights_are_the_oracle_s_rounded_to_float(h3mod):
    """Host-only entry point: the library's res_multistep weights are the oracle's float64
    weights rounded once to float32, on the grids a run uses (video shift 12, audio shift 3,
    20 and 40 steps): first step (no previous sigma), interior steps, and the step to 0."""
    import numpy as np

    import oracle.h3_oracle as O

    for steps, shift in ((20, 12.0), (20, 3.0), (40, 12.0), (40, 3.0)):
        sig = O.shifted_sigmas(steps, shift).astype(np.float64)
        for i in range(steps):
            prev = None if i == 0 else float(sig[i - 1])
            got = h3mod.h3_res_multistep_step(prev, float(sig[i]), float(sig[i + 1]))
            want = O.res_multistep_coefficients(prev, float(sig[i]), float(sig[i + 1]))
            assert got.sigma == np.float32(sig[i])
            for g, w in zip((got.a, got.c_now, got.c_prev), want):
                # double-precision weights rounded once: within one float32 ulp of the oracle's
                assert abs(g - w) <= np.spacing(np.float32(abs(w))) + 1e-12, (steps, shift, i, g, w)
            if i + 1 == steps:
                assert (got.a, got.c_now, got.c_prev) == (0.0, 1.0, 0.0)
            if i == 0:
                assert got.c_prev == 0.0


@fake_addresses
def test_res_multistep_arguments_refused(h3mod):
    L = h3mod.lib()
    out = h3mod.h3_ms_step()
    f = ctypes.c_float
    nan = float("nan")
    bad = ((0.9, 0.0, 0.0), (0.9, 0.5, 0.5), (0.9, 0.5, 0.6), (0.9, 0.5, -0.1), (0.4, 0.5, 0.25),
           (nan, 0.5, 0.25), (0.9, nan, 0.25), (0.9, 0.5, nan))
    for sp, s, sn in bad:
        assert L.h3_res_multistep_step(f(sp), f(s), f(sn), ctypes.byref(out)) == h3mod.H3_EINVAL, (sp, s, sn)
    assert L.h3_res_multistep_step(f(-1.0), f(0.5), f(0.25), None) == h3mod.H3_EINVAL
    d = _tiny_dims(h3mod)
    al = 0x2000
    step = h3mod.h3_res_multistep_step(None, 0.5, 0.25)
    # the multistep head needs both the latents and the previous-prediction buffer
    assert L.h3_head_forward_ms(ctypes.byref(d), al, 8, al, al, al, 6 * 192, al, None, 96, ctypes.byref(step), None,
                                al, None, None) == h3mod.H3_EINVAL
    assert L.h3_head_forward_ms(ctypes.byref(d), al, 8, al, al, al, 6 * 192, al, None, 96, ctypes.byref(step), al,
                                None, al, None) == h3mod.H3_EINVAL
    assert L.h3_head_forward_ms(ctypes.byref(d), al, 8, al, al, al, 6 * 192, al, None, 96, None, None, al, al,
                                None) == h3mod.H3_EINVAL


@fake_addresses
def test_misaligned_int32_and_float32_arrays_refused(h3mod):
    """Every f32 / i32 array a kernel reads element by element must be 4-byte aligned; an array
    that is not returns H3_EINVAL on the host (the fake addresses below are never touched: each
    call must refuse first).  Covers tidx and pos of the block and trunk, the gate's tidx, the
    AdaLN tidx, the entry projection and head arrays, and both sampler transitions."""
    L = h3mod.lib()
    d = _tiny_dims(h3mod)
    al, odd = 0x40000, 0x40002  # 16-byte aligned; 2 bytes off
    H, I, F = 192, 256, 512

    def lin(n_out, k):
        x = h3mod.h3_linear()
        x.fmt, x.w, x.n_out, x.k = 0, al, n_out, k
        return x

    bw = h3mod.h3_block_w()
    bw.qkv, bw.o, bw.fc1, bw.fc2 = lin(3 * I, H), lin(H, I), lin(2 * F, H), lin(H, F)
    ws = 0x100000
    big = 1 << 30
    for tidx, pos in ((odd, al), (al, odd)):
        assert L.h3_block_forward(ctypes.byref(d), ctypes.byref(bw), al, 18 * H, 1, al, al, 72, al, tidx, pos, ws, big,
                                  0, None) == h3mod.H3_EINVAL
        assert L.h3_trunk_forward(ctypes.byref(d), ctypes.byref(bw), 1, al, 1, al, 72, al, tidx, pos, ws, big, 0,
                                  None) == h3mod.H3_EINVAL
    assert L.h3_adaln_modulate(ctypes.byref(d), al, al + 0x10000, 72, al, 18 * H, 0, 1, al, odd, None) == h3mod.H3_EINVAL
    lo = lin(H, I)
    assert L.h3_linear_forward(ctypes.byref(lo), h3mod.H3_EPI_GATE_RES, al, I, al, H, 72, al, al, 18 * H, 2, al, odd, 0,
                               None) == h3mod.H3_EINVAL
    f = ctypes.c_float
    # entry projection: latents, weights, bias
    for z, w, b in ((odd, al, al), (al, odd, al), (al, al, odd)):
        assert L.h3_embed_rows(ctypes.byref(d), z, 96, w, b, 8, al, None) == h3mod.H3_EINVAL
    # head: tidx, weights, bias, v, z (Euler); and the previous prediction (res_multistep)
    for tidx, w, b, v, z in ((odd, al, al, al, al), (al, odd, al, al, al), (al, al, odd, al, al),
                             (al, al, al, odd, al), (al, al, al, al, odd)):
        assert L.h3_head_forward(ctypes.byref(d), al, 8, al, tidx, al, 6 * H, w, b, 96, v, z, f(-0.1),
                                 None) == h3mod.H3_EINVAL
    step = h3mod.h3_res_multistep_step(None, 0.5, 0.25)
    assert L.h3_head_forward_ms(ctypes.byref(d), al, 8, al, al, al, 6 * H, al, al, 96, ctypes.byref(step), None, al,
                                odd, None) == h3mod.H3_EINVAL
    # sampler transitions: a misaligned latent array or weight is refused before the entry
    # projections or the trunk launch
    io = h3mod.h3_io_w()
    io.text_rows, io.cond_rows, io.audio_rows, io.video_rows, io.k_video, io.k_audio = 8, 0, 8, 8, 96, 32
    for fld in ("patch_v", "patch_v_b", "patch_a", "patch_a_b", "head_v", "head_v_b", "head_a", "head_a_b"):
        setattr(io, fld, al)
    arr = (h3mod.h3_block_w * 1)(bw)
    for zv, za in ((odd, al), (al, odd)):
        assert L.h3_denoise_step(ctypes.byref(d), arr, 1, al, al, 1, ctypes.byref(io), al, None, zv, za, al, al, al,
                                 al, f(-0.1), f(-0.1), ws, big, 0, None) == h3mod.H3_EINVAL
        assert L.h3_denoise_step_ms(ctypes.byref(d), arr, 1, al, al, 1, ctypes.byref(io), al, None, zv, za, al, al,
                                    al, al, al, al, ctypes.byref(step), ctypes.byref(step), ws, big, 0,
                                    None) == h3mod.H3_EINVAL
    io.head_a = odd
    assert L.h3_denoise_step(ctypes.byref(d), arr, 1, al, al, 1, ctypes.byref(io), al, None, al, al, al, al, al, al,
                             f(-0.1), f(-0.1), ws, big, 0, None) == h3mod.H3_EINVAL
    io.head_a = al
    assert L.h3_denoise_step_ms(ctypes.byref(d), arr, 1, al, al, 1, ctypes.byref(io), al, None, al, al, odd, al, al,
                                al, al, al, ctypes.byref(step), ctypes.byref(step), ws, big, 0,
                                None) == h3mod.H3_EINVAL


def test_sampler_plan_is_the_oracle_grids_deduplicated(h3mod):
    """Host-only entry point: the run plan's table rows are the distinct float32 values
    1000 sigma of both schedules' first `steps` grid points (the oracle's shifted_sigmas),
    descending, and each transition's rows point at its own values; a 40-step run has 78 rows
    in float32 (the 12/13 pair of the two grids differs by one ulp; exact arithmetic gives the
    pages' 77, pinned in the oracle tests)."""
    import numpy as np

    import oracle.h3_oracle as O

    for steps in (1, 2, 8, 20, 40):
        tv = np.float32(1000.0) * O.shifted_sigmas(steps, 12.0)[:steps]
        ta = np.float32(1000.0) * O.shifted_sigmas(steps, 3.0)[:steps]
        want = sorted(set(tv.tolist()) | set(ta.tolist()), reverse=True)
        vals, vi, ai = h3mod.h3_sampler_plan(steps, 12.0, 3.0)
        assert vals == want
        assert [vals[i] for i in vi] == tv.tolist() and [vals[i] for i in ai] == ta.tolist()
    assert len(h3mod.h3_sampler_plan(40, 12.0, 3.0)[0]) == 78
    assert len(h3mod.h3_sampler_plan(8, 12.0, 3.0)[0]) == 15
    L = h3mod.lib()
    buf = (ctypes.c_float * 8)()
    n = ctypes.c_int()
    idx = (ctypes.c_int * 4)()
    f = ctypes.c_float
    assert L.h3_sampler_plan(0, f(12.0), f(3.0), buf, ctypes.byref(n), idx, idx) == h3mod.H3_EINVAL
    assert L.h3_sampler_plan(4, f(12.0), f(0.0), buf, ctypes.byref(n), idx, idx) == h3mod.H3_EINVAL
    assert L.h3_sampler_plan(4, f(12.0), f(3.0), None, ctypes.byref(n), idx, idx) == h3mod.H3_EINVAL
