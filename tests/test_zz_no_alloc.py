"""h3_qknorm_rope_static -- the QK-norm + RoPE step for callers that cannot allocate.

Callers that cannot hand the library extra device memory at the call site (their memory
belongs to a pool they cannot reach there, or they must avoid cudaMalloc's implicit
synchronisation) use this entry point; its scratch is a fixed array inside the library.
It must give exactly what h3_qknorm_rope gives with a caller workspace, call after call,
and refuse sizes its array cannot hold.  This file is collected last on purpose.
"""

import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA device", allow_module_level=True)

import synth  # noqa: E402
from joint_video_audio_block_b300 import h3, runtime as R  # noqa: E402

pytestmark = pytest.mark.gpu


def _inputs(name, seed):
    cfg = synth.CONFIGS[name]
    d = cfg.dims
    n = cfg.layout.n_rows
    qkv = R.bf16_from_bits(synth.normal_bf16(seed, 911, (n, 3 * d.inner), 0.0, 1.5))
    _, _, pos = synth.packed_rows(cfg)
    w = R.upload_block(synth.block_weights(cfg, 0))
    return R.dims_of(d), d, n, qkv, torch.from_numpy(pos).cuda(), w


def _outputs(d, n):
    ld_vt = (n + 63) // 64 * 64
    q = torch.empty(d.heads, n, d.head_dim, dtype=torch.bfloat16, device="cuda")
    return q, torch.empty_like(q), torch.zeros(d.heads, d.head_dim, ld_vt, dtype=torch.bfloat16, device="cuda"), ld_vt


def _run_both(name, seed):
    dims, d, n, qkv, pos, w = _inputs(name, seed)
    qn, kn = h3.ptr(w["qnorm"]), h3.ptr(w["knorm"])
    st = h3.stream_ptr()
    # the existing entry point, with a caller workspace
    q0, k0, v0, ld_vt = _outputs(d, n)
    ws = torch.empty(n * d.head_dim * 4, dtype=torch.uint8, device="cuda")
    h3.h3_qknorm_rope(dims, qkv.data_ptr(), pos.data_ptr(), qn, kn, q0.data_ptr(), k0.data_ptr(), v0.data_ptr(), ld_vt,
                      n, ws.data_ptr(), ws.numel(), st)
    # the allocation-free entry point
    q1, k1, v1, _ = _outputs(d, n)
    h3.h3_qknorm_rope_static(dims, qkv.data_ptr(), pos.data_ptr(), qn, kn, q1.data_ptr(), k1.data_ptr(), v1.data_ptr(),
                             ld_vt, n, st)
    torch.cuda.synchronize()
    status, site = h3.h3_last_device_error(st)
    assert status == h3.H3_OK, f"device error word set: site {site:#x}"
    # same kernels on the same inputs: the tolerance is zero difference
    for a, b, what in ((q0, q1, "q"), (k0, k1, "k"), (v0, v1, "v^T")):
        diff = float((a.float() - b.float()).abs().max())
        assert diff == 0.0, f"{name} {what}: static-scratch result differs from workspace result by {diff}"
        assert torch.equal(a, b)


def test_static_scratch_matches_workspace_twice():
    # two calls in a row on different shapes: the second reuses the array the first filled
    _run_both("block1829", seed=21)
    _run_both("tiny", seed=22)
    _run_both("block1829", seed=23)


def test_static_scratch_rejects_oversize():
    d = synth.H3
    dims = R.dims_of(d)
    n = h3.H3_QKROPE_STATIC_MAX_PAIRS // (d.head_dim // 2) + 1
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(h3.H3Error) as e:
        h3.h3_qknorm_rope_static(dims, dummy.data_ptr(), dummy.data_ptr(), None, None, dummy.data_ptr(),
                                 dummy.data_ptr(), dummy.data_ptr(), (n + 63) // 64 * 64, n, h3.stream_ptr())
    assert e.value.status == h3.H3_EINVAL  # refused on the host, before any launch
