"""Pins of the oracle's training-path RoPE (oracle.rope_apply): the forward rotation with no
cache write, and its backward, the rotation by -theta.

AstrAI internals, "Rotary Position Embedding (RoPE)", and inference guide, "Rotary Embedding
Backend": training applies RoPE as a torch complex multiply of adjacent pairs by the table
entry, and autograd differentiates it. The pins compare against torch's own autograd of that
complex multiply in float64, against exactly representable rotations, and against the
separately-rounded f32 evaluation written out with numpy scalars.
"""
import numpy as np
import pytest

import oracle
from paged_kv_cache_apply_gb300 import workloads as W

torch = pytest.importorskip("torch")


def _wid(a):
    return W.f32_from_bf16_bits(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


def _torch_complex_rope(x64, fr, pos):
    """The torch complex path in float64: view_as_complex pairs times the table entry."""
    T, nh, D = x64.shape
    f = torch.view_as_complex(torch.from_numpy(fr[pos].astype(np.float64)).contiguous())  # [T, D/2]
    z = torch.view_as_complex(x64.reshape(T, nh, D // 2, 2))
    return torch.view_as_real(z * f[:, None, :]).reshape(T, nh, D)


def _bound(a, b, c, s):
    # |fl(fl(a c) op fl(b s)) - exact| for one f32 pair, with room for the sign of s
    u = 2.0 ** -24
    return (u * (abs(a * c) + abs(b * s) + abs(a * c + b * s)) * 1.001 + 1e-45,
            u * (abs(b * c) + abs(a * s) + abs(b * c - a * s)) * 1.001 + 1e-45)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_is_torch_autograd_of_the_complex_multiply(dtype):
    rng = np.random.default_rng(41)
    T, nh, D = 29, 3, 64
    fr = W.rope_freqs_cis(512, D)
    pos = rng.integers(0, 512, T).astype(np.int32)
    x = torch.from_numpy(_wid(W.normal_values((T, nh, D), dtype, 9, 1))).requires_grad_(True)
    g_bits = W.normal_values((T, nh, D), dtype, 9, 2)  # the gradient arriving at the rotated x
    g = _wid(g_bits)
    y = _torch_complex_rope(x, fr, pos)
    (gx,) = torch.autograd.grad(y, x, grad_outputs=torch.from_numpy(g))
    exact = gx.numpy()
    got = _wid(oracle.rope_apply(g_bits, fr, pos, inverse=True))
    a, b = g[..., 0::2], g[..., 1::2]
    c = fr[pos][:, None, :, 0].astype(np.float64)
    s = fr[pos][:, None, :, 1].astype(np.float64)
    br, bi = _bound(a, b, c, s)
    if dtype == "bf16":  # the final rounding to bf16 adds half an ulp of bf16
        br = br + 2.0 ** -8 * np.abs(exact[..., 0::2]) * 1.01
        bi = bi + 2.0 ** -8 * np.abs(exact[..., 1::2]) * 1.01
    assert np.all(np.abs(got[..., 0::2] - exact[..., 0::2]) <= br)
    assert np.all(np.abs(got[..., 1::2] - exact[..., 1::2]) <= bi)
    # the forward of the same path, against the same torch expression
    fwd = _wid(oracle.rope_apply(W.normal_values((T, nh, D), dtype, 9, 1), fr, pos))
    ref = y.detach().numpy()
    a, b = x.detach().numpy()[..., 0::2], x.detach().numpy()[..., 1::2]
    br, bi = _bound(a, b, c, -s)
    if dtype == "bf16":
        br = br + 2.0 ** -8 * np.abs(ref[..., 0::2]) * 1.01
        bi = bi + 2.0 ** -8 * np.abs(ref[..., 1::2]) * 1.01
    assert np.all(np.abs(fwd[..., 0::2] - ref[..., 0::2]) <= br)
    assert np.all(np.abs(fwd[..., 1::2] - ref[..., 1::2]) <= bi)


def test_exact_quarter_turns():
    # table rows (1,0), (0,1), (-1,0), (0,-1): the rotations are exact, so are their transposes
    D = 8
    fr = np.zeros((4, D // 2, 2), np.float32)
    fr[0, :, 0] = 1
    fr[1, :, 1] = 1
    fr[2, :, 0] = -1
    fr[3, :, 1] = -1
    x = W.normal_values((4, 2, D), "f32", 11, 1)
    pos = np.arange(4, dtype=np.int32)
    a, b = x[..., 0::2], x[..., 1::2]
    fwd = oracle.rope_apply(x, fr, pos)
    bwd = oracle.rope_apply(x, fr, pos, inverse=True)
    want_f = [(a[0], b[0]), (-b[1], a[1]), (-a[2], -b[2]), (b[3], -a[3])]
    want_b = [(a[0], b[0]), (b[1], -a[1]), (-a[2], -b[2]), (-b[3], a[3])]
    for p in range(4):
        assert np.array_equal(fwd[p, :, 0::2], want_f[p][0]) and np.array_equal(fwd[p, :, 1::2], want_f[p][1])
        assert np.array_equal(bwd[p, :, 0::2], want_b[p][0]) and np.array_equal(bwd[p, :, 1::2], want_b[p][1])


def test_backward_spec_is_separately_rounded_products():
    # R5 with the conjugate entry, written out with numpy float32 scalars (IEEE, never fused):
    # re = RN(RN(a c) + RN(b s)), im = RN(RN(b c) - RN(a s))
    rng = np.random.default_rng(43)
    T, nh, D = 7, 2, 32
    x = W.normal_values((T, nh, D), "f32", 12, 1) * np.float32(5.0)
    fr = W.rope_freqs_cis(64, D)
    pos = rng.integers(0, 64, T).astype(np.int32)
    got = oracle.rope_apply(x, fr, pos, inverse=True)
    a, b = x[..., 0::2], x[..., 1::2]
    c = fr[pos][:, None, :, 0]
    s = fr[pos][:, None, :, 1]
    re = (a * c).astype(np.float32) + (b * s).astype(np.float32)
    im = (b * c).astype(np.float32) - (a * s).astype(np.float32)
    assert np.array_equal(got[..., 0::2], re) and np.array_equal(got[..., 1::2], im)


def test_round_trip_recovers_the_input_within_rounding():
    rng = np.random.default_rng(44)
    T, nh, D = 40, 2, 128
    x = W.normal_values((T, nh, D), "f32", 13, 1)
    fr = W.rope_freqs_cis(4096, D)
    pos = rng.integers(0, 4096, T).astype(np.int32)
    fwd = oracle.rope_apply(x, fr, pos)
    back = oracle.rope_apply(fwd, fr, pos, inverse=True)
    # R^T R = (c^2 + s^2) I, and the f32 table has c^2 + s^2 within a few ulps of 1; each of
    # the two roundings per step errs by at most one ulp of the pair's magnitude |a| + |b|
    m = np.repeat(np.abs(x[..., 0::2]) + np.abs(x[..., 1::2]), 2, axis=-1).astype(np.float64)
    assert np.all(np.abs(back.astype(np.float64) - x) <= 8 * 2.0 ** -24 * m)
    assert not np.array_equal(fwd, x)


def test_position_outside_the_table_is_rejected():
    fr = W.rope_freqs_cis(16, 8)
    x = W.normal_values((2, 1, 8), "f32", 14, 1)
    with pytest.raises(ValueError):
        oracle.rope_apply(x, fr, np.array([3, 16], np.int32), inverse=True)
