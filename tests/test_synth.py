"""The seeded input generator: determinism, stream independence, distribution, layouts."""

import numpy as np

import synth


def _splitmix64_first(state):
    """Published SplitMix64 step from state 0 (Steele, Lea & Flood 2014), written out here."""
    m = (1 << 64) - 1
    z = (state + 0x9E3779B97F4A7C15) & m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def test_splitmix_known_value():
    # the first output of SplitMix64 seeded with 0 is 0xE220A8397B1DCDAF
    assert _splitmix64_first(0) == 0xE220A8397B1DCDAF


def test_deterministic_and_streams_differ():
    a = synth.normal_bf16(5, 3, (1000,))
    b = synth.normal_bf16(5, 3, (1000,))
    c = synth.normal_bf16(5, 4, (1000,))
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    # threaded and single-threaded generation agree (chunking keeps Box-Muller pairs intact)
    big = synth.normal_f32(9, 1, (300001,))
    assert np.array_equal(big[:1000], synth.normal_f32(9, 1, (1000,)))


def test_distribution():
    x = synth.normal_f64(1, 2, (400000,), 0.5, 2.0)
    assert abs(x.mean() - 0.5) < 0.02 and abs(x.std() - 2.0) < 0.02
    b = synth.bf16_bits_to_f32(synth.normal_bf16(1, 2, (400000,), 0.5, 2.0))
    assert np.max(np.abs(b - x)) <= np.max(np.abs(x)) * 2 ** -8


def test_layouts_and_sizes():
    for name, n in [("tiny", 72), ("block1829", 1829), ("block12936", 12936), ("trunk33720", 33720),
                    ("trunk50x1829_narrow", 1829)]:
        cfg = synth.CONFIGS[name]
        tag, tidx, pos = synth.packed_rows(cfg)
        assert len(tag) == n and pos.shape == (n, 3)
        assert set(np.unique(tag)) <= {0, 1, 2}
        assert tidx.min() >= 0 and tidx.max() < cfg.n_timesteps
    assert len(synth.CONFIGS["trunk33720"].timesteps) == 77
    narrow = synth.CONFIGS["trunk50x1829_narrow"]
    assert narrow.dims.head_dim == synth.H3.head_dim and narrow.dims.rope_sections == synth.H3.rope_sections
    assert narrow.n_blocks == 50 and len(narrow.timesteps) == 77
    tag, tidx, pos = synth.packed_rows(synth.CONFIGS["trunk33720"], step=5)
    assert len(np.unique(tidx)) == 2  # video and audio schedules differ away from sigma = 1


def test_quantizer_codes_in_range():
    w = synth.normal_bf16(3, 1, (64, 128), 0.0, 0.02)
    q, s, b = synth.quantize_int8_g32(w)
    assert q.shape == (64, 128) and s.shape == (64, 4) and b.shape == (64, 4)
    # every group uses both ends of the code range
    g = q.reshape(64, 4, 32)
    assert np.all(g.min(axis=2) == 0) and np.all(g.max(axis=2) >= 254)


def test_device_quantizer_matches_the_host_recipe():
    """The torch quantizer that prepares the benchmark's INT8 weights follows the host recipe
    bit for bit (run here on CPU tensors)."""
    torch = __import__("pytest").importorskip("torch")
    w = synth.normal_bf16(3, 2, (96, 256), 0.0, 0.02)
    w[5, :32] = w[5, 0]  # a constant group: scale 0, every code 0
    q, s, b = synth.quantize_int8_g32(w)
    t = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16)
    qd, sd, bd = synth.device_quantize_int8_g32(t)
    assert np.array_equal(qd.numpy(), q)
    assert np.array_equal(sd.view(torch.int16).numpy().view(np.uint16), s)
    assert np.array_equal(bd.view(torch.int16).numpy().view(np.uint16), b)
