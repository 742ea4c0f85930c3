"""Pins of the CPU oracle to facts outside itself: closed forms, hand-worked values,
brute force on tiny inputs, invariants, and figures printed on the pages.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a swapped
modulation tensor, a wrong RoPE pairing or frequency, a transposed weight) fails it.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle.h3_oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _page(name):
    with open(os.path.join(GOLDEN, "page_figures.json")) as f:
        return json.load(f)[name]


# ------------------------------------------------------------------------ bf16 rounding


def test_round_bf16_known_values():
    # 1 + 2^-8 is exactly half-way between bf16 neighbours 1 and 1 + 2^-7: ties to even -> 1
    assert O.round_bf16(1.0 + 2 ** -8) == 1.0
    # 1 + 3*2^-8 is half-way between 1 + 2^-7 (odd mantissa) and 1 + 2^-6: ties to even -> 1 + 2^-6
    assert O.round_bf16(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6
    assert O.round_bf16(1.0 + 2 ** -8 + 2 ** -20) == 1.0 + 2 ** -7
    assert O.round_bf16(-3.0) == -3.0
    assert O.round_bf16(0.1) == 0.10009765625  # 0x3DCD
    b = O.to_bf16_bits(np.array([1.0, -2.0, 0.5]))
    assert list(b) == [0x3F80, 0xC000, 0x3F00]


# ------------------------------------------------------------------------ LayerNorm + modulate


def test_layernorm_worked_example():
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    # mean 2.5, biased variance 1.25
    expect = np.array([-1.5, -0.5, 0.5, 1.5]) / math.sqrt(1.25)
    np.testing.assert_allclose(O.layernorm(x, 0.0)[0], expect, rtol=0, atol=1e-15)
    shift = np.full((1, 4), 0.1)
    scale = np.full((1, 4), 1.0)
    np.testing.assert_allclose(O.adaln_modulate(x, shift, scale, 0.0)[0], 2 * expect + 0.1, atol=1e-15)


def test_layernorm_zero_modulation_gives_unit_rows():
    rng = np.random.default_rng(0)
    x = rng.normal(3.0, 2.0, size=(5, 64))
    eps = 1e-6
    y = O.adaln_modulate(x, np.zeros_like(x), np.zeros_like(x), eps)
    var = x.var(axis=1)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-13)
    np.testing.assert_allclose(y.var(axis=1), var / (var + eps), rtol=1e-12)


def test_modulate_is_affine_in_scale_and_shift():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(3, 16))
    n = O.layernorm(x, 1e-6)
    sc = rng.normal(size=(3, 16))
    sh = rng.normal(size=(3, 16))
    y = O.adaln_modulate(x, sh, sc, 1e-6)
    # scale = -1 annihilates the normalised input, leaving only the shift
    np.testing.assert_allclose(O.adaln_modulate(x, sh, -np.ones_like(x), 1e-6), sh, atol=1e-15)
    np.testing.assert_allclose(y - sh, n * (1 + sc), atol=1e-13)


# ------------------------------------------------------------------------ table + gather


def test_modcache_equals_exact_live_projection():
    """The table entry equals the live adaln projection of the row's timestep embedding,
    here evaluated with an exactly rounded sum (math.fsum) on a separate code path."""
    cfg = synth.CONFIGS["tiny"]
    te = synth.sinusoidal_temb([0.5, 700.0], cfg.dims.temb_dim)
    W, b = synth.adaln_weights(cfg, 0)
    W2, b2 = synth.adaln_weights(cfg, 1)
    t64, tbf = O.modcache(te, [W, W2], [b, b2])
    assert t64.shape == (2, 2, 18 * 192)
    Wf = [synth.bf16_bits_to_f32(W).astype(float), synth.bf16_bits_to_f32(W2).astype(float)]
    bf = [synth.bf16_bits_to_f32(b).astype(float), synth.bf16_bits_to_f32(b2).astype(float)]
    rng = np.random.default_rng(2)
    for t, blk in itertools.product(range(2), range(2)):
        for j in rng.choice(18 * 192, 40, replace=False):
            terms = [Wf[blk][j, kk] * float(te[t, kk]) for kk in range(cfg.dims.temb_dim)] + [bf[blk][j]]
            exact = math.fsum(terms)
            assert abs(t64[t, blk, j] - exact) <= 1e-15 * max(1.0, abs(exact)) * 8
            assert tbf[t, blk, j] == O.round_bf16(exact)


def test_table_size_matches_pages():
    shp = _page("adaln_proj_shape")["value"]
    B, n_out, dt = shp
    assert n_out == 18 * 5376 and dt == 2688
    assert round(B * n_out * dt / 1e9, 2) == _page("adaln_params_billion")["value"]
    assert round(B * n_out * dt * 2 / 1e9, 1) == _page("adaln_resident_gb")["value"]
    for key in ("cache_mb_40_step_run", "cache_mb_15s_run"):
        g = _page(key)
        mb = O.table_bytes(g["timesteps"], g["blocks"], g["hidden"]) / 1e6
        assert round(mb) == g["value"], (key, mb)


def test_gather_selects_tag_and_timestep():
    H, T = 8, 3
    # code every entry by (t, j, c) so a wrong index shows up as a wrong code
    tb = np.zeros((T, 18 * H))
    for t in range(T):
        for j in range(18):
            tb[t, j * H:(j + 1) * H] = 1000 * t + 10 * j + np.arange(H) / 100
    tag = np.array([0, 1, 2, 2, 1])
    tidx = np.array([2, 0, 1, 0, 2])
    for m in range(6):
        g = O.modulation(tb, tag, tidx, m, H)
        for r in range(5):
            j = 6 * tag[r] + m
            assert np.all(g[r] == 1000 * tidx[r] + 10 * j + np.arange(H) / 100)


# ------------------------------------------------------------------------ QK-norm + RoPE


def test_rms_norm_closed_form():
    x = np.array([[[3.0, 4.0]]])  # mean square 12.5
    y = O.rms_norm(x, np.array([1.0, 2.0]), 0.0)
    np.testing.assert_allclose(y[0, 0], [3 / math.sqrt(12.5), 8 / math.sqrt(12.5)], atol=1e-15)


def _unit(hd, i):
    x = np.zeros((1, 1, hd))
    x[0, 0, i] = 1.0
    return x


def test_rope_hand_worked_hd16():
    """hd = 16: 8 pairs (i, i+8), sections (t, h, w) = (2, 3, 3) pairs, omega_i = 1e4^(-2i/16)."""
    hd, th, sec = 16, 1e4, (2, 3, 3)
    assert synth.Dims(16, 1, 16, 16, 16).rope_sections == sec
    # pair 0 on the t axis, omega 1, pos t = 1: e_0 -> (cos 1) e_0 + (sin 1) e_8
    y = O.rope(_unit(hd, 0), np.array([[1.0, 0, 0]]), hd, th, sec)[0, 0]
    assert y[0] == pytest.approx(math.cos(1.0), abs=1e-15) and y[8] == pytest.approx(math.sin(1.0), abs=1e-15)
    assert np.count_nonzero(np.abs(y) > 1e-15) == 2
    # pair 1 on the t axis, omega = 10^-0.5, pos t = 2
    y = O.rope(_unit(hd, 1), np.array([[2.0, 0, 0]]), hd, th, sec)[0, 0]
    a = 2.0 * 10 ** -0.5
    assert y[1] == pytest.approx(math.cos(a), abs=1e-15) and y[9] == pytest.approx(math.sin(a), abs=1e-15)
    # pair 2 is the first h-axis pair, omega = 0.1; the second half of a pair rotates as (-sin, cos)
    y = O.rope(_unit(hd, 10), np.array([[5.0, 3.0, 7.0]]), hd, th, sec)[0, 0]
    assert y[2] == pytest.approx(-math.sin(0.3), abs=1e-15) and y[10] == pytest.approx(math.cos(0.3), abs=1e-15)
    # pair 5 is the first w-axis pair, omega = 10^-2.5
    y = O.rope(_unit(hd, 5), np.array([[9.0, 9.0, 1.0]]), hd, th, sec)[0, 0]
    a = 10 ** -2.5
    assert y[5] == pytest.approx(math.cos(a), abs=1e-15) and y[13] == pytest.approx(math.sin(a), abs=1e-15)


def test_rope_invariants():
    rng = np.random.default_rng(3)
    hd, th = 64, 1e4
    sec = synth.TINY.rope_sections
    q = rng.normal(size=(6, 2, hd))
    k = rng.normal(size=(6, 2, hd))
    # integer positions so that the shifted positions stay exact in float32
    pos = rng.integers(0, 50, size=(6, 3)).astype(np.float32)
    rq = O.rope(q, pos, hd, th, sec)
    # pair norms preserved
    half = hd // 2
    np.testing.assert_allclose(rq[..., :half] ** 2 + rq[..., half:] ** 2, q[..., :half] ** 2 + q[..., half:] ** 2,
                               rtol=1e-12)
    # zero position is the identity
    np.testing.assert_allclose(O.rope(q, np.zeros((6, 3), np.float32), hd, th, sec), q, atol=0)
    # scores depend on relative position only: shifting every row by one offset per axis
    shift = np.array([7.0, -3.0, 11.0], np.float32)
    rk = O.rope(k, pos, hd, th, sec)
    s0 = np.einsum("nhd,mhd->hnm", rq, rk)
    rq2 = O.rope(q, pos + shift, hd, th, sec)
    rk2 = O.rope(k, pos + shift, hd, th, sec)
    s1 = np.einsum("nhd,mhd->hnm", rq2, rk2)
    np.testing.assert_allclose(s1, s0, rtol=1e-9, atol=1e-9)
    # shifting only the keys changes the scores (the rotation is not a no-op)
    rk3 = O.rope(k, pos + shift, hd, th, sec)
    assert np.abs(np.einsum("nhd,mhd->hnm", rq, rk3) - s0).max() > 1e-3


def test_rope_1d_rows_are_textbook_rope():
    """(p, p, p) rows: every pair rotates by p * omega_i, as a complex multiplication."""
    hd = 64
    rng = np.random.default_rng(4)
    x = rng.normal(size=(5, 1, hd))
    p = np.arange(5, dtype=np.float32) * 3.0
    y = O.rope(x, np.stack([p, p, p], 1), hd, 1e4, synth.TINY.rope_sections)
    half = hd // 2
    z = x[:, 0, :half] + 1j * x[:, 0, half:]
    for r in range(5):
        for i in range(half):
            ang = float(p[r]) * 1e4 ** (-2 * i / hd)
            w = z[r, i] * complex(math.cos(ang), math.sin(ang))
            assert y[r, 0, i] == pytest.approx(w.real, abs=1e-12)
            assert y[r, 0, half + i] == pytest.approx(w.imag, abs=1e-12)


def test_split_qkv_interleaved_rows():
    heads, hd = 3, 2
    y = np.arange(heads * 3 * hd, dtype=float)[None, :]
    q, k, v = O.split_qkv(y, heads, hd)
    # head h occupies columns [h*3hd, (h+1)*3hd) as q | k | v
    assert q[0].tolist() == [[0, 1], [6, 7], [12, 13]]
    assert k[0].tolist() == [[2, 3], [8, 9], [14, 15]]
    assert v[0].tolist() == [[4, 5], [10, 11], [16, 17]]


# ------------------------------------------------------------------------ attention


def _brute_attention(q, k, v):
    """Pure-Python softmax attention with exactly rounded sums (tiny inputs only)."""
    n, nh, hd = q.shape
    out = np.zeros_like(q)
    for h in range(nh):
        for r in range(n):
            s = [math.fsum(q[r, h, d] * k[j, h, d] for d in range(hd)) / math.sqrt(hd) for j in range(n)]
            m = max(s)
            e = [math.exp(a - m) for a in s]
            z = math.fsum(e)
            for d in range(hd):
                out[r, h, d] = math.fsum(e[j] * v[j, h, d] for j in range(n)) / z
    return out


@pytest.mark.parametrize("n", [1, 2, 5, 16])
def test_attention_brute_force(n):
    rng = np.random.default_rng(10 + n)
    q, k, v = (rng.normal(size=(n, 2, 4)) * 2 for _ in range(3))
    np.testing.assert_allclose(O.attention(q, k, v), _brute_attention(q, k, v), rtol=1e-12, atol=1e-13)


def test_attention_invariants():
    rng = np.random.default_rng(5)
    n, nh, hd = 12, 2, 8
    q, k, v = (rng.normal(size=(n, nh, hd)) for _ in range(3))
    o = O.attention(q, k, v)
    perm = rng.permutation(n)
    np.testing.assert_allclose(O.attention(q, k[perm], v[perm]), o, rtol=1e-12, atol=1e-14)
    # identical keys: uniform weights, output = mean of values
    kk = np.broadcast_to(k[:1], k.shape)
    np.testing.assert_allclose(O.attention(q, kk, v), np.broadcast_to(v.mean(0), o.shape), atol=1e-14)
    # one dominant key selects its value
    k2 = k.copy() * 0
    k2[3] = q[0] * 1e3
    np.testing.assert_allclose(O.attention(q[:1], k2, v)[0], v[3], atol=1e-12)
    # query subset equals the same rows of the full result
    np.testing.assert_allclose(O.attention(q, k, v, rows=[4, 0, 7]), o[[4, 0, 7]], atol=0)


# ------------------------------------------------------------------------ linears / SwiGLU


def test_linear_orientation_and_identity():
    x = np.array([[1.0, 2.0, 3.0]])
    w = np.array([[1.0, 0, 0], [0, 0, 1.0]])  # [out=2, in=3]
    assert O.linear(x, w, np.array([10.0, 20.0])).tolist() == [[11.0, 23.0]]
    rng = np.random.default_rng(6)
    xx = rng.normal(size=(4, 7))
    np.testing.assert_array_equal(O.linear(xx, np.eye(7)), xx)


def test_swiglu_closed_form():
    y = np.array([[0.0, 1.0, -30.0, 5.0, 2.0, 3.0]])  # F = 3: gates [0, 1, -30], values [5, 2, 3]
    h = O.swiglu(y, 3)[0]
    assert h[0] == 0.0
    assert h[1] == pytest.approx(2.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    assert abs(h[2]) < 1e-11
    # silu(x) -> x for large x
    assert O.silu(np.array([40.0]))[0] == pytest.approx(40.0, rel=1e-15)


# ------------------------------------------------------------------------ INT8 group 32


def test_int8_roundtrip_bound_and_grid_points():
    cfg = synth.CONFIGS["tiny"]
    w = synth.block_weights(cfg)["wo"]  # [192, 256]
    q, sc, qb = synth.quantize_int8_g32(w)
    wd = O.dequant_int8_g32(q, sc, qb)
    wm = O.widen_bf16(w)
    s = np.repeat(O.widen_bf16(sc), 32, axis=1)
    ulp = np.abs(wd) * 2.0 ** -8  # >= half a bf16 ulp of w'
    assert np.all(np.abs(wm - wd) <= s / 2 + ulp + 1e-30)
    # points on the grid qb + j*scale (exactly representable here) come back as j
    scale_bits = np.array([[O.to_bf16_bits(2.0 ** -7)]], np.uint16)
    qb_bits = np.array([[O.to_bf16_bits(-0.5)]], np.uint16)
    j = np.arange(0, 256, 8)[:32]
    grid = -0.5 + j * 2.0 ** -7
    gb = O.to_bf16_bits(grid).reshape(1, 32)
    assert np.all(O.widen_bf16(gb) == grid)
    q2, s2, b2 = synth.quantize_int8_g32(gb)
    assert s2[0, 0] == O.to_bf16_bits((grid.max() - grid.min()) / 255)[()]
    # dequantising the generator's own output of a grid with scale 2^-7 reproduces it
    qq = j.astype(np.uint8).reshape(1, 32)
    np.testing.assert_array_equal(O.dequant_int8_g32(qq, scale_bits, qb_bits)[0], grid)


def test_int8_constant_group():
    w = O.to_bf16_bits(np.full((1, 32), 0.25))
    q, sc, qb = synth.quantize_int8_g32(w)
    assert np.all(q == 0) and O.widen_bf16(sc)[0, 0] == 0.0
    assert np.all(O.dequant_int8_g32(q, sc, qb) == 0.25)


# ------------------------------------------------------------------------ block structure


def _tiny_inputs(seed_block=0):
    cfg = synth.CONFIGS["tiny"]
    d = cfg.dims
    x = synth.activations(cfg)
    w = synth.block_weights(cfg, seed_block)
    te = synth.temb(cfg)
    W, b = synth.adaln_weights(cfg, seed_block)
    _, tbf = O.modcache(te, [W], [b])
    tag, tidx, pos = synth.packed_rows(cfg)
    return cfg, d, x, w, tbf[:, 0, :], tag, tidx, pos


def _set_mod(tb, H, m, value, tags=(0, 1, 2)):
    tb = tb.copy().reshape(tb.shape[0], 18, H)
    for t in tags:
        tb[:, 6 * t + m, :] = value
    return tb.reshape(tb.shape[0], 18 * H)


def test_block_zero_gates_is_identity():
    cfg, d, x, w, tb, tag, tidx, pos = _tiny_inputs()
    tb0 = _set_mod(_set_mod(tb, d.hidden, O.GATE_MSA, 0.0), d.hidden, O.GATE_MLP, 0.0)
    out = O.block_forward(x, w, tb0, tag, tidx, pos, d)
    np.testing.assert_array_equal(out, O.widen_bf16(x))


def test_block_branch_wiring():
    """With gate_mlp = 0 the output is the attention branch alone: it must not move with the
    MLP-branch shift, and must move with the attention-branch shift.  With gate_msa = 0 the
    output must not depend on the attention weights."""
    cfg, d, x, w, tb, tag, tidx, pos = _tiny_inputs()
    H = d.hidden
    a = O.block_forward(x, w, _set_mod(tb, H, O.GATE_MLP, 0.0), tag, tidx, pos, d)
    b = O.block_forward(x, w, _set_mod(_set_mod(tb, H, O.GATE_MLP, 0.0), H, O.SHIFT_MLP, 5.0), tag, tidx, pos, d)
    np.testing.assert_array_equal(a, b)
    c = O.block_forward(x, w, _set_mod(_set_mod(tb, H, O.GATE_MLP, 0.0), H, O.SHIFT_MSA, 5.0), tag, tidx, pos, d)
    assert np.abs(c - a).max() > 1e-3
    w2 = dict(w)
    w2["wqkv"] = synth.block_weights(cfg, 7)["wqkv"]
    e = O.block_forward(x, w, _set_mod(tb, H, O.GATE_MSA, 0.0), tag, tidx, pos, d)
    f = O.block_forward(x, w2, _set_mod(tb, H, O.GATE_MSA, 0.0), tag, tidx, pos, d)
    np.testing.assert_array_equal(e, f)


def test_block_tag_selects_its_own_modulation():
    """Rows tagged text read only table entries 0..5: changing the audio/video entries leaves
    text rows' attention-branch input unchanged."""
    cfg, d, x, w, tb, tag, tidx, pos = _tiny_inputs()
    H = d.hidden
    _, parts = O.block_forward(x, w, tb, tag, tidx, pos, d, return_parts=True)
    tb2 = _set_mod(tb, H, O.SHIFT_MSA, 3.0, tags=(1, 2))
    _, parts2 = O.block_forward(x, w, tb2, tag, tidx, pos, d, return_parts=True)
    text = tag == synth.TAG_TEXT
    np.testing.assert_array_equal(parts["xn"][text], parts2["xn"][text])
    assert np.abs(parts["xn"][~text] - parts2["xn"][~text]).min() > 1.0


def test_block_rows_subset_matches_full():
    cfg, d, x, w, tb, tag, tidx, pos = _tiny_inputs()
    full = O.block_forward(x, w, tb, tag, tidx, pos, d)
    rows = np.array([0, 17, 40, 71])
    sub = O.block_forward(x, w, tb, tag, tidx, pos, d, rows=rows)
    np.testing.assert_allclose(sub, full[rows], rtol=0, atol=1e-12)


def test_block_bf16_emulation_close_to_exact():
    cfg, d, x, w, tb, tag, tidx, pos = _tiny_inputs()
    a = O.block_forward(x, w, tb, tag, tidx, pos, d)
    b = O.block_forward(x, w, tb, tag, tidx, pos, d, emulate_bf16=True)
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 0 < rel < 1e-2


# ------------------------------------------------------------------------ work model


def test_flop_model_matches_linear_share_on_the_pages():
    g = _page("linear_share")
    geo = _page("block_geometry")["value"]
    assert (synth.H3.hidden, synth.H3.heads, synth.H3.head_dim, synth.H3.inner, synth.H3.ffn) == (
        geo["hidden"], geo["heads"], geo["head_dim"], geo["inner"], geo["ffn"])
    assert O.block_linear_params(synth.H3) == 385_351_680
    for n, share in zip(g["rows"], g["value"]):
        lin, att = O.block_flops(synth.H3, n)
        assert abs(lin / (lin + att) - share) <= g["tolerance"], (n, lin / (lin + att))


# ----------------------------------------------------------------------------- block-sparse attention


def _qkv(n, nh, hd, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, nh, hd)), rng.standard_normal((n, nh, hd)), rng.standard_normal((n, nh, hd)))


def test_sparse_attention_all_kept_is_dense():
    q, k, v = _qkv(37, 2, 8, 1)
    nt = -(-37 // 8)
    full = np.ones((2, nt, nt), np.uint8)
    np.testing.assert_allclose(O.attention_tile_sparse(q, k, v, full, tile=8), O.attention(q, k, v), rtol=0, atol=1e-13)


def test_sparse_attention_single_tile_is_attention_over_that_tile():
    """Keeping one key tile is plain attention over just those keys (computed by slicing)."""
    q, k, v = _qkv(40, 1, 4, 2)
    mask = np.zeros((1, 5, 5), np.uint8)
    mask[0, :, 3] = 1  # every query tile keeps key tile 3 = keys 24..31
    got = O.attention_tile_sparse(q, k, v, mask, tile=8)
    # brute force with explicit loops over the kept keys
    ref = np.zeros_like(q)
    for r in range(40):
        s = np.array([q[r, 0] @ k[j, 0] for j in range(24, 32)]) / 2.0
        p = np.exp(s - s.max())
        ref[r, 0] = (p[:, None] * v[24:32, 0]).sum(0) / p.sum()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_sparse_attention_row_without_kept_tiles_is_zero():
    q, k, v = _qkv(24, 1, 4, 3)
    mask = np.ones((1, 3, 3), np.uint8)
    mask[0, 1, :] = 0  # query tile 1 (rows 8..15) keeps nothing
    got = O.attention_tile_sparse(q, k, v, mask, tile=8)
    assert np.all(got[8:16] == 0)
    np.testing.assert_allclose(got[:8], O.attention(q, k, v)[:8], rtol=0, atol=1e-13)


def test_sparse_attention_tiny_brute_force():
    """Exhaustive loop over a random mask: each row's softmax over exactly its kept keys."""
    rng = np.random.default_rng(4)
    n, nh, hd, tile = 12, 2, 3, 4
    q, k, v = _qkv(n, nh, hd, 5)
    mask = (rng.random((nh, 3, 3)) < 0.5).astype(np.uint8)
    got = O.attention_tile_sparse(q, k, v, mask, tile=tile)
    for h in range(nh):
        for r in range(n):
            keys = [j for j in range(n) if mask[h, r // tile, j // tile]]
            if not keys:
                assert np.all(got[r, h] == 0)
                continue
            s = np.array([q[r, h] @ k[j, h] for j in keys]) / math.sqrt(hd)
            p = np.exp(s - s.max())
            ref = sum(p[i] * v[j, h] for i, j in enumerate(keys)) / p.sum()
            np.testing.assert_allclose(got[r, h], ref, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- trunk entry / exit, sampler


def test_embed_rows_selector_weights_copy_the_latent():
    """A 0/1 selector W (column c reads latent feature c mod K) turns the projection into a copy."""
    rng = np.random.default_rng(6)
    z = rng.standard_normal((5, 12)).astype(np.float32)
    H = 40
    w = np.zeros((H, 12), np.float32)
    w[np.arange(H), np.arange(H) % 12] = 1.0
    b = rng.standard_normal(H).astype(np.float32)
    got = O.embed_rows(z, w, b)
    np.testing.assert_array_equal(got, z[:, np.arange(H) % 12].astype(np.float64) + b.astype(np.float64))


def test_head_on_constant_rows_is_the_projected_shift():
    """A constant row normalises to zero, so the head's output is W shift + b exactly."""
    H, K = 64, 6
    rng = np.random.default_rng(7)
    x = np.full((3, H), 0.625)
    shift = rng.standard_normal((3, H))
    scale = rng.standard_normal((3, H))
    w = rng.standard_normal((K, H)).astype(np.float32)
    b = rng.standard_normal(K).astype(np.float32)
    np.testing.assert_allclose(O.head_forward(x, shift, scale, w, b, 1e-6),
                               shift @ w.astype(np.float64).T + b, rtol=0, atol=1e-12)


def test_final_modulation_indexing():
    T, H = 3, 8
    tf = np.arange(T * 6 * H, dtype=np.float64).reshape(T, 6 * H)
    tag = np.array([0, 1, 2, 2])
    tidx = np.array([2, 0, 1, 2])
    for m in (0, 1):
        got = O.final_modulation(tf, tag, tidx, m, H)
        for r in range(4):
            np.testing.assert_array_equal(got[r], tf[tidx[r], (2 * tag[r] + m) * H:(2 * tag[r] + m + 1) * H])


@pytest.mark.parametrize("steps", [2, 7, 8, 20, 40, 41, 50, 77])
def test_linspace_matches_aten(steps):
    """The pages name ATen's float32 linspace as the grid the scheduler must reproduce."""
    torch = pytest.importorskip("torch")
    ref = torch.linspace(1.0, 0.0, steps, dtype=torch.float32).numpy()
    np.testing.assert_array_equal(O.linspace_f32(1.0, 0.0, steps), ref)


def test_shifted_sigmas_endpoints_monotone_and_identity_shift():
    for shift in (1.0, 3.0, 12.0):
        s = O.shifted_sigmas(40, shift)
        assert s[0] == 1.0 and s[-1] == 0.0 and np.all(np.diff(s) < 0)
    np.testing.assert_array_equal(O.shifted_sigmas(40, 1.0), O.linspace_f32(1.0, 0.0, 41))
    # a larger shift keeps more of the grid at high noise
    assert np.all(O.shifted_sigmas(40, 12.0)[1:-1] > O.shifted_sigmas(40, 3.0)[1:-1])


def test_euler_integrates_a_constant_velocity_exactly():
    rng = np.random.default_rng(8)
    z0 = rng.standard_normal(10)
    v = rng.standard_normal(10)
    sig = O.shifted_sigmas(20, 12.0).astype(np.float64)
    z = z0
    for i in range(20):
        z = O.euler_step(z, v, sig[i], sig[i + 1])
    np.testing.assert_allclose(z, z0 + (sig[-1] - sig[0]) * v, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(O.euler_step(z0, v, 0.5, 0.5), z0)


def test_shifted_sigmas_hand_worked_values():
    """Hand-worked points of the shift s sigma / (1 + (s - 1) sigma) ("minimax-h3-mlx" README,
    "AdaLN precompute": video shift 12.0, audio shift 3.0).  On a 4-step grid sigma runs
    1, 0.75, 0.5, 0.25, 0, and every point below is one correctly rounded float32 division of
    exact operands:
      shift 3:  0.75 -> 2.25 / 2.5 = 0.9;   0.5 -> 1.5 / 2 = 0.75;  0.25 -> 0.75 / 1.5 = 0.5
      shift 12: 0.75 -> 9 / 9.25 = 36/37;   0.5 -> 6 / 6.5 = 12/13;  0.25 -> 3 / 3.75 = 0.8
    A plausible slip such as sigma^(1/s) gives 0.794 / 0.976 at sigma = 0.5 instead."""
    f32 = np.float32
    np.testing.assert_array_equal(O.shifted_sigmas(4, 3.0), np.array([1, 0.9, 0.75, 0.5, 0], np.float32))
    np.testing.assert_array_equal(O.shifted_sigmas(4, 12.0),
                                  np.array([1, f32(36 / 37), f32(12 / 13), f32(0.8), 0], np.float32))
    np.testing.assert_array_equal(O.shifted_sigmas(2, 12.0)[1], f32(12 / 13))


@pytest.mark.parametrize("shift", [3.0, 12.0, 5.5])
def test_shifted_sigmas_equal_the_exponential_time_shift(shift):
    """The same grid written as the exponential time shift of rectified-flow samplers ("Layout":
    Euler with an exponential sigma shift): sigma' = e^mu / (e^mu + (1/sigma - 1)) with
    mu = ln s.  Evaluated here in float64 from that form; the oracle's float32 result must sit
    within two float32 ulps of it at every interior grid point."""
    steps = 40
    sig = O.linspace_f32(1.0, 0.0, steps + 1).astype(np.float64)[1:-1]
    mu = math.log(shift)
    want = math.exp(mu) / (math.exp(mu) + (1.0 / sig - 1.0))
    got = O.shifted_sigmas(steps, shift).astype(np.float64)[1:-1]
    ulp = np.spacing(want.astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(got - want) <= 2 * ulp), np.max(np.abs(got - want) / ulp)


def _wiring_case():
    """A small packed sequence [text 3 | cond 2x2 | audio 5 | video 1x2x3] with every gate of
    every block zero, so the trunk is exactly the identity (the residual branches add 0)."""
    d = synth.Dims(hidden=128, heads=4, head_dim=32, ffn=128, temb_dim=16)
    cfg = synth.Config("wiring", d, synth.Layout(3, (2, 2), 5, (1, 2, 3)), seed=21, n_blocks=2)
    lay = cfg.layout
    n = lay.n_rows
    tag, _, pos = synth.packed_rows(cfg)
    tidx = np.arange(n, dtype=np.int32)  # one table row per packed row
    H = d.hidden
    rng = np.random.default_rng(22)
    table = rng.standard_normal((n, cfg.n_blocks, 18 * H))
    t4 = table.reshape(n, cfg.n_blocks, 18, H)
    t4[:, :, [2, 5, 8, 11, 14, 17], :] = 0.0  # gate_msa, gate_mlp of every tag
    blocks = [synth.block_weights(cfg, b) for b in range(cfg.n_blocks)]
    text_x = O.round_bf16(rng.standard_normal((lay.text, H)))
    return cfg, d, tag, tidx, pos, table, blocks, text_x


def _wiring_io(H, kv, ka):
    return {k: np.zeros(s, np.float32) for k, s in (
        ("patch_v", (H, kv)), ("patch_v_b", (H,)), ("patch_a", (H, ka)), ("patch_a_b", (H,)),
        ("head_v", (kv, H)), ("head_v_b", (kv,)), ("head_a", (ka, H)), ("head_a_b", (ka,)))}


def test_denoise_step_exit_wiring_closed_form():
    """Which head, which rows and which d sigma: with the final scale at -1 every row's head
    input is its final shift alone, and with one table row per packed row (tidx = r) and shift
    (r + 1)(tag + 1) in every channel, selector heads (output k reads channel k) with biases
    0.5 (audio) and 0.25 (video) give, for packed row r of a segment,
      z_new = z + dsigma_seg ((r + 1)(tag + 1) + b_seg).
    Worked out here, not by the oracle's own steps; swapping the heads, the segment offsets,
    the tags or the two d sigma values changes the result."""
    cfg, d, tag, tidx, pos, table, blocks, text_x = _wiring_case()
    lay, H, n = cfg.layout, d.hidden, cfg.layout.n_rows
    kv, ka = synth.VIDEO_FEATURES, synth.AUDIO_FEATURES
    io = _wiring_io(H, kv, ka)
    io["head_v"][np.arange(kv), np.arange(kv)] = 1.0
    io["head_a"][np.arange(ka), np.arange(ka)] = 1.0
    io["head_v_b"][:] = 0.25
    io["head_a_b"][:] = 0.5
    table_f = np.zeros((n, 6 * H))
    tf = table_f.reshape(n, 3, 2, H)
    for r in range(n):
        for tg in range(3):
            tf[r, tg, 0, :] = (r + 1) * (tg + 1)  # shift
            tf[r, tg, 1, :] = -1.0                # scale: (1 + scale) = 0
    rng = np.random.default_rng(23)
    zc = rng.standard_normal((lay.n_cond, kv))
    za = rng.standard_normal((lay.audio, ka))
    zv = rng.standard_normal((lay.n_video, kv))
    ds_v, ds_a = -0.0625, -0.125
    za2, zv2 = O.denoise_step(text_x, zc, za, zv, io, blocks, table, table_f, tag, tidx, pos, d, ds_v, ds_a)
    a0 = lay.text + lay.n_cond
    v0 = a0 + lay.audio
    ra = np.arange(a0, v0)[:, None]
    rv = np.arange(v0, n)[:, None]
    assert np.all(tag[a0:v0] == synth.TAG_AUDIO) and np.all(tag[v0:] == synth.TAG_VIDEO)
    np.testing.assert_allclose(za2, za + ds_a * ((ra + 1) * (synth.TAG_AUDIO + 1) + 0.5), rtol=0, atol=1e-12)
    np.testing.assert_allclose(zv2, zv + ds_v * ((rv + 1) * (synth.TAG_VIDEO + 1) + 0.25), rtol=0, atol=1e-12)


def test_denoise_step_entry_wiring_closed_form():
    """Which patch projection and which rows: the entry weights write channels 0 and 1 of a
    row's latent as the hidden pattern [z0, -z0, z1, -z1, ...] (exact in bf16 for the eighths
    drawn here), whose LayerNorm is worked out by hand -- mean 0, variance (z0^2 + z1^2) / 2 --
    so with zero final modulation and heads reading hidden channels 0 and 2 the row's velocity
    is (z0, z1) / sqrt((z0^2 + z1^2) / 2 + eps) in its first two outputs and 0 elsewhere.
    A latent row embedded at another row's place, or a segment read from the wrong offset,
    breaks it (the condition rows carry other latents)."""
    cfg, d, tag, tidx, pos, table, blocks, text_x = _wiring_case()
    lay, H, n = cfg.layout, d.hidden, cfg.layout.n_rows
    kv, ka = synth.VIDEO_FEATURES, synth.AUDIO_FEATURES
    io = _wiring_io(H, kv, ka)
    c = np.arange(H)
    sign = np.where(c % 2 == 0, 1.0, -1.0)
    for pw in (io["patch_v"], io["patch_a"]):
        pw[c, (c // 2) % 2] = sign  # hidden c reads latent channel (c // 2) % 2 with sign (-1)^c
    for hw in (io["head_v"], io["head_a"]):
        hw[0, 0] = 1.0
        hw[1, 2] = 1.0
    table_f = np.zeros((n, 6 * H))
    rng = np.random.default_rng(24)
    eighths = lambda shape: rng.integers(-24, 25, shape) / 8.0  # noqa: E731
    zc, za, zv = eighths((lay.n_cond, kv)), eighths((lay.audio, ka)), eighths((lay.n_video, kv))
    za[:, :2] = np.where(za[:, :2] == 0, 0.5, za[:, :2])
    zv[:, :2] = np.where(zv[:, :2] == 0, 0.5, zv[:, :2])
    ds_v, ds_a = -0.0625, -0.125
    eps = d.ln_eps
    za2, zv2 = O.denoise_step(text_x, zc, za, zv, io, blocks, table, table_f, tag, tidx, pos, d, ds_v, ds_a)
    for z, z2, ds in ((za, za2, ds_a), (zv, zv2, ds_v)):
        den = np.sqrt((z[:, 0] ** 2 + z[:, 1] ** 2) / 2.0 + eps)
        want = z.copy()
        want[:, 0] += ds * z[:, 0] / den
        want[:, 1] += ds * z[:, 1] / den
        np.testing.assert_allclose(z2, want, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ res_multistep sampler
#
# The second-order multistep exponential integrator the mlx-h3 README ("Why mlx-h3") names as
# the sampler.  Pinned by hand-worked weights, by the cases that reduce to the Euler step, by
# exactness where the method is exact (a data prediction linear in t = -ln sigma), and by its
# order of convergence against scipy's adaptive integrator on a nonlinear problem.


@pytest.mark.parametrize("sig, want", [
    # equal log-steps (r = -1): c_now = h (phi1 + phi2), c_prev = -h phi2, h phi1 = 1 - a
    ((1.0, 0.5, 0.25), (0.5, 1.5 - 1.0 / (2.0 * math.log(2.0)), -(1.0 - 1.0 / (2.0 * math.log(2.0))))),
    ((1.0, 1.0 / 3.0, 1.0 / 9.0), (1.0 / 3.0, 5.0 / 3.0 - 2.0 / (3.0 * math.log(3.0)),
                                   -(1.0 - 2.0 / (3.0 * math.log(3.0))))),
    # a step twice as long in log-sigma as the previous one (r = -1/2): c_now = h phi1 + 2 h phi2
    ((1.0, 0.5, 0.125), (0.125 * 2.0, 11.0 / 4.0 - 3.0 / (4.0 * math.log(2.0)), -2.0 + 3.0 / (4.0 * math.log(2.0)))),
])
def test_res_multistep_hand_worked_weights(sig, want):
    got = O.res_multistep_coefficients(*sig)
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-15)
    # a constant prediction is carried exactly: a + c_now + c_prev = 1
    assert abs(sum(got) - 1.0) < 1e-14


def test_data_prediction_recovers_the_clean_latent():
    """Rectified flow: z = (1 - sigma) x0 + sigma eps moves with velocity v = eps - x0, so the
    prediction z - sigma v is x0 itself, at every sigma (and a wrong sign or a (1 - sigma)
    factor would miss it)."""
    rng = np.random.default_rng(34)
    x0, eps = rng.standard_normal((5, 7)), rng.standard_normal((5, 7))
    for sigma in (1.0, 0.73, 0.2, 1e-3):
        z = (1.0 - sigma) * x0 + sigma * eps
        np.testing.assert_allclose(O.data_prediction(z, eps - x0, sigma), x0, rtol=0, atol=1e-14)


def test_res_multistep_first_step_is_euler_and_last_step_is_the_prediction():
    rng = np.random.default_rng(31)
    z, v = rng.standard_normal((7, 5)), rng.standard_normal((7, 5))
    z1, d = O.res_multistep_step(z, v, None, 0.8, 0.55)
    np.testing.assert_allclose(z1, z + (0.55 - 0.8) * v, rtol=0, atol=1e-14)
    np.testing.assert_array_equal(d, z - 0.8 * v)
    z2, _ = O.res_multistep_step(z, v, 0.9, 0.3, 0.0, d_prev=rng.standard_normal((7, 5)))
    np.testing.assert_allclose(z2, z - 0.3 * v, rtol=0, atol=1e-15)


def test_res_multistep_is_exact_for_a_prediction_linear_in_log_sigma():
    """dz/dt = D(t) - z with D(t) = A + B t (t = -ln sigma) has the solution
    z(t) = A + B (t - 1) + C e^-t.  The second-order step, fed the exact z and predictions at
    t_prev and t, must land on z(t_next) to rounding for any step lengths; the first-order step
    must not (B != 0)."""
    rng = np.random.default_rng(32)
    A, B, C = rng.standard_normal(6), rng.standard_normal(6), rng.standard_normal(6)
    zt = lambda t: A + B * (t - 1.0) + C * math.exp(-t)  # noqa: E731
    Dt = lambda t: A + B * t  # noqa: E731
    for _ in range(20):
        s_prev, s, s_next = np.sort(rng.uniform(0.02, 1.0, 3))[::-1]
        t_prev, t, t_next = -math.log(s_prev), -math.log(s), -math.log(s_next)
        z = zt(t)
        v = (z - Dt(t)) / s  # so that z - sigma v is the exact prediction at t
        z_next, d_now = O.res_multistep_step(z, v, s_prev, s, s_next, d_prev=Dt(t_prev))
        np.testing.assert_allclose(d_now, Dt(t), rtol=0, atol=1e-13)
        np.testing.assert_allclose(z_next, zt(t_next), rtol=0, atol=1e-12)
        z_first, _ = O.res_multistep_step(z, v, None, s, s_next)
        assert np.abs(z_first - zt(t_next)).max() > 1e-8


def _solve_multistep(sigmas, z0, pred, second_order=True):
    z, d_prev, s_prev = z0.copy(), None, None
    for s, s_next in zip(sigmas[:-1], sigmas[1:]):
        d = pred(z, s)
        v = (z - d) / s
        z, d_prev = O.res_multistep_step(z, v, s_prev if second_order else None, s, s_next, d_prev=d_prev)
        s_prev = s
    return z


def test_res_multistep_converges_at_second_order():
    """On dz/dsigma = (z - D(z, sigma)) / sigma with a nonlinear D, halving the log-sigma step
    divides the error against scipy's integrator (rtol 1e-12) by about 4; the Euler steps of
    the same grids (first order) only by about 2."""
    from scipy.integrate import solve_ivp

    pred = lambda z, s: np.tanh(z) * math.cos(3.0 * s) + 0.5 * s  # noqa: E731
    z0 = np.array([0.7, -1.3, 2.1])
    s0, s1 = 1.0, 0.05

    def rhs(t, z):
        s = math.exp(-t)
        return pred(z, s) - z

    ref = solve_ivp(rhs, (-math.log(s0), -math.log(s1)), z0, rtol=1e-12, atol=1e-14, method="DOP853").y[:, -1]
    errs = {}
    for order in (True, False):
        errs[order] = []
        for n in (40, 80, 160):
            sig = np.exp(-np.linspace(-math.log(s0), -math.log(s1), n + 1))
            errs[order].append(np.abs(_solve_multistep(sig, z0, pred, order) - ref).max())
    for e in (errs[True],):
        rates = [math.log2(e[i] / e[i + 1]) for i in range(2)]
        assert all(1.8 < r < 2.3 for r in rates), rates
    rates1 = [math.log2(errs[False][i] / errs[False][i + 1]) for i in range(2)]
    assert all(0.8 < r < 1.2 for r in rates1), rates1


def test_denoise_step_multistep_uses_each_modality_s_own_grid():
    """The zero-gate trunk and selector heads of the Euler wiring pins give every latent row a
    known velocity v = (r + 1)(tag + 1) + b_seg; each modality must then move by its own sigma
    triple and its own previous prediction:
      z_new = a z + c_now (z - sigma v) + c_prev D_prev,
    with (a, c_now, c_prev) from that modality's grid.  Swapped grids or previous predictions
    fail it (the triples differ)."""
    cfg, d, tag, tidx, pos, table, blocks, text_x = _wiring_case()
    lay, H, n = cfg.layout, d.hidden, cfg.layout.n_rows
    kv, ka = synth.VIDEO_FEATURES, synth.AUDIO_FEATURES
    io = _wiring_io(H, kv, ka)
    io["head_v"][np.arange(kv), np.arange(kv)] = 1.0
    io["head_a"][np.arange(ka), np.arange(ka)] = 1.0
    io["head_v_b"][:] = 0.25
    io["head_a_b"][:] = 0.5
    table_f = np.zeros((n, 6 * H))
    tf = table_f.reshape(n, 3, 2, H)
    for r in range(n):
        for tg in range(3):
            tf[r, tg, 0, :] = (r + 1) * (tg + 1)
            tf[r, tg, 1, :] = -1.0
    rng = np.random.default_rng(33)
    zc = rng.standard_normal((lay.n_cond, kv))
    za = rng.standard_normal((lay.audio, ka))
    zv = rng.standard_normal((lay.n_video, kv))
    da_prev = rng.standard_normal((lay.audio, ka))
    dv_prev = rng.standard_normal((lay.n_video, kv))
    sig_v, sig_a = (0.97, 0.9, 0.7), (0.8, 0.6, 0.45)
    za2, zv2, da, dv = O.denoise_step_multistep(text_x, zc, za, zv, io, blocks, table, table_f, tag, tidx, pos, d,
                                                sig_v, sig_a, d_prev_video=dv_prev, d_prev_audio=da_prev)
    a0 = lay.text + lay.n_cond
    v0 = a0 + lay.audio
    for z, z2, dn, dp, rows, tg, b, sig in ((za, za2, da, da_prev, np.arange(a0, v0), synth.TAG_AUDIO, 0.5, sig_a),
                                            (zv, zv2, dv, dv_prev, np.arange(v0, n), synth.TAG_VIDEO, 0.25, sig_v)):
        v = (rows[:, None] + 1.0) * (tg + 1) + b
        a, cn, cp = O.res_multistep_coefficients(*sig)
        want_d = z - sig[1] * v
        np.testing.assert_allclose(dn, want_d, rtol=0, atol=1e-12)
        np.testing.assert_allclose(z2, a * z + cn * want_d + cp * dp, rtol=0, atol=1e-11)


def test_two_shifted_grids_give_the_pages_distinct_timestep_counts():
    """The pages count 77 distinct timesteps for a 40-step run ("AdaLN precompute") and
    8 + 8 - 1 = 15 for 8 forwards ("Full-resolution 15 s generation").  The reading -- each
    schedule's first `steps` points of the even grid from 1 to 0, shifted by
    s sigma / (1 + (s - 1) sigma) with s = 12 (video) and 3 (audio) -- reproduces both in exact
    rational arithmetic: the grids meet at sigma' = 1, 12/13 and 3/4 for 40 steps, only at 1
    for 8."""
    from fractions import Fraction as Fr

    def grid(steps, s):
        return [Fr(s) * x / (1 + (Fr(s) - 1) * x) for x in (1 - Fr(i, steps) for i in range(steps))]

    for name, steps in (("cache_mb_40_step_run", 40), ("cache_mb_15s_run", 8)):
        v, a = grid(steps, 12), grid(steps, 3)
        assert len(set(v) | set(a)) == _page(name)["timesteps"]
    v, a = set(grid(40, 12)), set(grid(40, 3))
    assert v & a == {Fr(1), Fr(12, 13), Fr(3, 4)}
