"""Pins of the CPU oracle against facts the pages and the mathematics fix (no GPU needed).

Each test checks the oracle against something other than itself: the mask the AstrAI
internals page prints, numpy complex multiplication, closed forms and invariants of RoPE,
fp64 torch scaled_dot_product_attention, and identities of the method (decode = last row of
causal prefill, split-K merge = unsplit, paged = contiguous, resumed prefill = suffix rows).
"""
import math
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_apply_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_mask(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([float(tok) for tok in line.split()])
    return np.array(rows)


# ------------------------------------------------------------------------------------------
# mask (AstrAI internals, "Autoregression & Causal Masking")
# ------------------------------------------------------------------------------------------


def test_mask_matches_printed_5x5():
    golden = _read_mask(os.path.join(GOLDEN, "causal_mask_5x5.txt"))
    assert golden.shape == (5, 5)
    got = oracle.causal_mask(5)
    assert np.array_equal(np.isinf(got), np.isinf(golden))
    assert np.array_equal(got[np.isfinite(got)], golden[np.isfinite(golden)])
    assert np.all(got[np.isinf(got)] < 0)


# ------------------------------------------------------------------------------------------
# RoPE (AstrAI internals, "Rotary Position Embedding"; inference guide "Rotary Embedding Backend")
# ------------------------------------------------------------------------------------------


def _f64_table(max_len, dim, base=10000.0):
    theta = base ** (-2.0 * np.arange(dim // 2) / dim)
    ang = np.arange(max_len)[:, None] * theta[None, :]
    return np.stack([np.cos(ang), np.sin(ang)], axis=-1)


def test_rope_is_complex_multiplication_of_adjacent_pairs():
    rng = np.random.default_rng(1)
    T, nh, D = 5, 3, 16
    x = rng.standard_normal((T, nh, D))
    fr = _f64_table(40, D)
    pos = rng.integers(0, 40, T).astype(np.int32)
    got = oracle.rope_f64(x, fr, pos)
    z = x[..., 0::2] + 1j * x[..., 1::2]                      # view_as_complex pairing
    rot = fr[pos][:, None, :, 0] + 1j * fr[pos][:, None, :, 1]
    ref = z * rot
    assert np.allclose(got[..., 0::2], ref.real, rtol=0, atol=1e-15)
    assert np.allclose(got[..., 1::2], ref.imag, rtol=0, atol=1e-15)


def test_rope_d2_matches_cmath_rotation():
    # head_dim 2: one pair rotated by angle p * theta_0 = p
    for p in [0, 1, 5, 17]:
        fr = np.array([[[math.cos(q), math.sin(q)]] for q in range(20)])
        x = np.array([[[0.3, -1.7]]])
        got = oracle.rope_f64(x, fr, np.array([p], np.int32))[0, 0]
        ref = complex(0.3, -1.7) * complex(math.cos(p), math.sin(p))
        assert abs(got[0] - ref.real) < 1e-15 and abs(got[1] - ref.imag) < 1e-15


def test_rope_only_mixes_its_own_pair():
    D = 8
    fr = _f64_table(10, D)
    base = np.zeros((1, 1, D))
    for e in range(D):
        x = base.copy()
        x[0, 0, e] = 1.0
        y = oracle.rope_f64(x, fr, np.array([7], np.int32))[0, 0]
        pair = {e - e % 2, e - e % 2 + 1}
        assert all(abs(y[i]) < 1e-300 for i in range(D) if i not in pair)


def test_rope_identity_at_position_zero_and_norm_preserved():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 2, 32))
    fr = _f64_table(100, 32)
    y0 = oracle.rope_f64(x, fr, np.zeros(4, np.int32))
    assert np.array_equal(y0, x)
    pos = np.array([3, 50, 99, 1], np.int32)
    y = oracle.rope_f64(x, fr, pos)
    n_in = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    n_out = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    assert np.allclose(n_in, n_out, rtol=1e-14, atol=0)


def test_rope_relative_position_property():
    # q_i^T k_j depends only on i - j (fp64 table: exact up to rounding)
    rng = np.random.default_rng(3)
    D = 64
    fr = _f64_table(400, D)
    q = rng.standard_normal((1, 1, D))
    k = rng.standard_normal((1, 1, D))
    for (i, j, c) in [(5, 2, 100), (0, 9, 31), (77, 77, 200), (3, 150, 7)]:
        a = (oracle.rope_f64(q, fr, np.array([i], np.int32)) *
             oracle.rope_f64(k, fr, np.array([j], np.int32))).sum()
        b = (oracle.rope_f64(q, fr, np.array([i + c], np.int32)) *
             oracle.rope_f64(k, fr, np.array([j + c], np.int32))).sum()
        assert abs(a - b) < 1e-12 * (1 + abs(a))


def test_rope_composition_closed_form():
    # R_a R_b = R_{a+b}: rotating by b then by a equals rotating by a + b
    rng = np.random.default_rng(4)
    D = 16
    fr = _f64_table(64, D)
    x = rng.standard_normal((3, 2, D))
    a = np.array([4, 10, 0], np.int32)
    b = np.array([9, 30, 13], np.int32)
    two = oracle.rope_f64(oracle.rope_f64(x, fr, b), fr, a)
    one = oracle.rope_f64(x, fr, a + b)
    assert np.allclose(two, one, rtol=0, atol=1e-13)


def _ulp_bound_f32(a, b, c, s):
    u = 2.0 ** -24
    ac, bs, as_, bc = a * c, b * s, a * s, b * c
    re, im = ac - bs, as_ + bc
    return (u * (abs(ac) + abs(bs) + abs(re)) * 1.001 + 1e-45,
            u * (abs(as_) + abs(bc) + abs(im)) * 1.001 + 1e-45)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rope_rounding_spec_within_bound_of_exact(dtype):
    rng = np.random.default_rng(5)
    T, H, Hk, D = 33, 4, 2, 64
    q = W.normal_values((T, H, D), dtype, 7, 1)
    k = W.normal_values((T, Hk, D), dtype, 7, 2)
    v = W.normal_values((T, Hk, D), dtype, 7, 3)
    fr = W.rope_freqs_cis(256, D)
    pos = rng.integers(0, 256, T).astype(np.int32)
    loc = rng.permutation(100)[:T].astype(np.int32)
    et = np.uint16 if dtype == "bf16" else np.float32
    kl = np.zeros((100, Hk, D), et)
    vl = np.zeros((100, Hk, D), et)
    q_out = oracle.rope_kv_write(q, k, v, fr, pos, loc, kl, vl)
    wid = (lambda a: W.f32_from_bf16_bits(a).astype(np.float64)) if dtype == "bf16" else \
        (lambda a: a.astype(np.float64))
    exact = oracle.rope_f64(wid(q), fr.astype(np.float64), pos)
    got = wid(q_out)
    xin = wid(q)
    a, b = xin[..., 0::2], xin[..., 1::2]
    c = fr[pos][:, None, :, 0].astype(np.float64)
    s = fr[pos][:, None, :, 1].astype(np.float64)
    br, bi = _ulp_bound_f32(a, b, c, s)
    if dtype == "bf16":  # the final rounding to bf16 adds half an ulp of bf16
        br = br + 2.0 ** -8 * np.abs(exact[..., 0::2]) * 1.01
        bi = bi + 2.0 ** -8 * np.abs(exact[..., 1::2]) * 1.01
    assert np.all(np.abs(got[..., 0::2] - exact[..., 0::2]) <= br)
    assert np.all(np.abs(got[..., 1::2] - exact[..., 1::2]) <= bi)


def test_rope_f32_spec_is_separately_rounded_products():
    # the R5 specification evaluated with numpy float32 scalars (IEEE, never fused)
    rng = np.random.default_rng(6)
    T, H, Hk, D = 9, 2, 1, 32
    q = W.normal_values((T, H, D), "f32", 8, 1) * np.float32(3.0)
    k = W.normal_values((T, Hk, D), "f32", 8, 2)
    v = W.normal_values((T, Hk, D), "f32", 8, 3)
    fr = W.rope_freqs_cis(64, D)
    pos = rng.integers(0, 64, T).astype(np.int32)
    loc = np.arange(T, dtype=np.int32)
    kl = np.zeros((T, Hk, D), np.float32)
    vl = np.zeros((T, Hk, D), np.float32)
    q_out = oracle.rope_kv_write(q, k, v, fr, pos, loc, kl, vl)
    a, b = q[..., 0::2], q[..., 1::2]
    c = fr[pos][:, None, :, 0]
    s = fr[pos][:, None, :, 1]
    re = (a * c).astype(np.float32) - (b * s).astype(np.float32)
    im = (a * s).astype(np.float32) + (b * c).astype(np.float32)
    assert np.array_equal(q_out[..., 0::2], re) and np.array_equal(q_out[..., 1::2], im)


def test_kv_write_scatters_rows_and_leaves_others():
    rng = np.random.default_rng(7)
    T, H, Hk, D, size = 6, 4, 2, 16, 50
    q = W.normal_values((T, H, D), "bf16", 9, 1)
    k = W.normal_values((T, Hk, D), "bf16", 9, 2)
    v = W.normal_values((T, Hk, D), "bf16", 9, 3)
    fr = W.rope_freqs_cis(32, D)
    pos = rng.integers(0, 32, T).astype(np.int32)
    loc = rng.permutation(size)[:T].astype(np.int32)
    kl = np.full((size, Hk, D), 0xABCD, np.uint16)
    vl = np.full((size, Hk, D), 0x1234, np.uint16)
    oracle.rope_kv_write(q, k, v, fr, pos, loc, kl, vl)
    others = np.setdiff1d(np.arange(size), loc)
    assert np.all(kl[others] == 0xABCD) and np.all(vl[others] == 0x1234)
    assert np.array_equal(vl[loc], v)
    # cached K equals the rotation of k at the token's position (rotation before write)
    exact = oracle.rope_f64(W.f32_from_bf16_bits(k).astype(np.float64), fr.astype(np.float64), pos)
    assert np.max(np.abs(W.f32_from_bf16_bits(kl[loc]) - exact)) < 2e-2
    kq = np.zeros((T, H, D), np.uint16)
    kq[:, :Hk] = k  # the same rows rotated through the q path give the same bits
    kl2 = np.zeros((size, Hk, D), np.uint16)
    vl2 = np.zeros((size, Hk, D), np.uint16)
    q2 = oracle.rope_kv_write(kq, k, v, fr, pos, loc, kl2, vl2)
    assert np.array_equal(q2[:, :Hk], kl[loc])


def test_kv_write_rejects_out_of_range():
    T, H, Hk, D = 2, 2, 1, 8
    q = np.zeros((T, H, D), np.float32)
    k = np.zeros((T, Hk, D), np.float32)
    fr = W.rope_freqs_cis(4, D)
    kl = np.zeros((4, Hk, D), np.float32)
    vl = np.zeros((4, Hk, D), np.float32)
    with pytest.raises(ValueError):
        oracle.rope_kv_write(q, k, k, fr, np.array([0, 4], np.int32), np.array([0, 1], np.int32), kl, vl)
    with pytest.raises(ValueError):
        oracle.rope_kv_write(q, k, k, fr, np.array([0, 1], np.int32), np.array([0, 9], np.int32), kl, vl)


def test_freqs_table_closed_forms():
    D, n = 128, 300
    fr = W.rope_freqs_cis(n, D).astype(np.float64)
    assert fr.shape == (n, D // 2, 2) and W.rope_freqs_cis(n, D).dtype == np.float32
    assert np.all(fr[0, :, 0] == 1.0) and np.all(fr[0, :, 1] == 0.0)
    assert np.allclose(fr[..., 0] ** 2 + fr[..., 1] ** 2, 1.0, atol=2e-7)
    p = np.arange(n)
    assert np.allclose(fr[:, 0, 0], [math.cos(x) for x in p], atol=1e-7)  # theta_0 = 1
    assert np.allclose(fr[:, 0, 1], [math.sin(x) for x in p], atol=1e-7)
    last = 10000.0 ** (-(D - 2) / D)
    assert np.allclose(fr[:, -1, 1], np.sin(p * last), atol=1e-7)
    za = fr[37, :, 0] + 1j * fr[37, :, 1]
    zb = fr[101, :, 0] + 1j * fr[101, :, 1]
    zc = fr[138, :, 0] + 1j * fr[138, :, 1]
    assert np.allclose(za * zb, zc, atol=1e-6)


# ------------------------------------------------------------------------------------------
# attention (AstrAI internals "KV Cache Mathematics" / "Attention Backend"; inference guide)
# ------------------------------------------------------------------------------------------


def _contig(seed, B, H, Hk, D, lens, dtype="f32", msl=None):
    msl = msl or int(max(lens))
    size = B * msl
    kl = W.normal_values((size, Hk, D), dtype, seed, 1)
    vl = W.normal_values((size, Hk, D), dtype, seed, 2)
    r2t = (np.arange(B)[:, None] * msl + np.arange(msl)[None, :]).astype(np.int32)
    return kl, vl, r2t, msl


def _wid(a):
    return W.f32_from_bf16_bits(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


def _sdpa(q, k, v, causal):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    return F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                          torch.from_numpy(v), is_causal=causal).numpy()


@pytest.mark.parametrize("dtype,G", [("f32", 1), ("f32", 2), ("bf16", 4)])
def test_prefill_matches_torch_sdpa_contiguous(dtype, G):
    B, Hk, D, L = 3, 2, 32, 19
    H = Hk * G
    lens = [L] * B
    kl, vl, r2t, msl = _contig(11, B, H, Hk, D, lens, dtype)
    q = W.normal_values((B * L, H, D), dtype, 11, 3)
    ind = W.prefix_sum(lens)
    got = oracle.prefill(q, kl, vl, r2t, np.arange(B, dtype=np.int32), ind, ind)
    qq = _wid(q).reshape(B, L, H, D).transpose(0, 2, 1, 3)
    kk = _wid(kl).reshape(B, msl, Hk, D).transpose(0, 2, 1, 3).repeat(G, axis=1)
    vv = _wid(vl).reshape(B, msl, Hk, D).transpose(0, 2, 1, 3).repeat(G, axis=1)
    ref = _sdpa(qq, kk, vv, True).transpose(0, 2, 1, 3).reshape(B * L, H, D)
    assert np.max(np.abs(got - ref)) < 1e-12


@pytest.mark.parametrize("G", [1, 4])
def test_decode_matches_torch_sdpa(G):
    B, Hk, D = 4, 2, 64
    H = Hk * G
    lens = np.array([1, 5, 33, 64], np.int32)
    kl, vl, r2t, msl = _contig(12, B, H, Hk, D, lens, "bf16")
    q = W.normal_values((B, H, D), "bf16", 12, 3)
    got = oracle.decode(q, kl, vl, r2t, np.arange(B, dtype=np.int32), lens)
    for b in range(B):
        L = int(lens[b])
        qq = _wid(q[b])[None, :, None, :]
        kk = _wid(kl[b * msl: b * msl + L]).transpose(1, 0, 2)[None].repeat(G, axis=1)
        vv = _wid(vl[b * msl: b * msl + L]).transpose(1, 0, 2)[None].repeat(G, axis=1)
        ref = _sdpa(qq, kk, vv, False)[0, :, 0, :]
        assert np.max(np.abs(got[b] - ref)) < 1e-12


def test_brute_force_tiny():
    # d = 4, up to 5 keys: the matrix softmax written out explicitly
    rng = np.random.default_rng(13)
    D, H, Hk = 4, 2, 1
    lens = [5, 3]
    kl = rng.standard_normal((10, Hk, D)).astype(np.float32)
    vl = rng.standard_normal((10, Hk, D)).astype(np.float32)
    r2t = np.array([[0, 1, 2, 3, 4], [5, 6, 7, 8, 9]], np.int32)
    q = rng.standard_normal((8, H, D)).astype(np.float32)
    ind = W.prefix_sum(lens)
    got = oracle.prefill(q, kl, vl, r2t, np.array([0, 1], np.int32), ind, ind)
    for b, (L, off) in enumerate(zip(lens, [0, 5])):
        Kb = kl[off: off + L, 0].astype(np.float64)
        Vb = vl[off: off + L, 0].astype(np.float64)
        for h in range(H):
            Q = q[ind[b]: ind[b + 1], h].astype(np.float64)
            S = Q @ Kb.T / 2.0
            S[np.triu_indices(L, 1)] = -np.inf
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            assert np.max(np.abs(got[ind[b]: ind[b + 1], h] - P @ Vb)) < 1e-14


def test_softmax_weights_sum_to_one_and_uniform_v():
    B, H, Hk, D = 2, 2, 1, 32
    lens = np.array([20, 32], np.int32)
    kl, _, r2t, msl = _contig(14, B, H, Hk, D, lens, "f32")
    q = W.normal_values((B, H, D), "f32", 14, 3) * np.float32(2.0)
    # one-hot values: output e = weight of key e
    vl = np.zeros_like(kl)
    for b in range(B):
        for j in range(msl):
            vl[b * msl + j, 0, j] = 1.0
    out = oracle.decode(q, kl, vl, r2t, np.arange(B, dtype=np.int32), lens)
    for b in range(B):
        w = out[b, :, : lens[b]]
        assert np.all(w > 0) and np.allclose(w.sum(-1), 1.0, atol=1e-12)
        assert np.all(out[b, :, lens[b]:] == 0)
    vl[:] = 0.625
    out = oracle.decode(q, kl, vl, r2t, np.arange(B, dtype=np.int32), lens)
    assert np.allclose(out, 0.625, atol=1e-14)


def test_decode_equals_last_row_of_causal_prefill():
    B, H, Hk, D = 3, 8, 2, 64
    lens = np.array([1, 17, 40], np.int32)
    kl, vl, r2t, msl = _contig(15, B, H, Hk, D, lens, "bf16")
    qp = W.normal_values((int(lens.sum()), H, D), "bf16", 15, 3)
    ind = W.prefix_sum(lens)
    pre = oracle.prefill(qp, kl, vl, r2t, np.arange(B, dtype=np.int32), ind, ind)
    last = ind[1:] - 1
    dec = oracle.decode(np.ascontiguousarray(qp[last]), kl, vl, r2t, np.arange(B, dtype=np.int32), lens)
    assert np.array_equal(dec, pre[last])


def test_split_merge_equals_unsplit():
    B, H, Hk, D = 3, 4, 2, 32
    lens = np.array([1, 9, 30], np.int32)
    kl, vl, r2t, msl = _contig(16, B, H, Hk, D, lens, "bf16")
    q = W.normal_values((B, H, D), "bf16", 16, 3)
    rpi = np.arange(B, dtype=np.int32)
    ref = oracle.decode(q, kl, vl, r2t, rpi, lens)
    for chunk in [1, 4, 7, 30, 64]:
        S = (30 + chunk - 1) // chunk
        o_p, m_p, l_p, out = oracle.decode_split(q, kl, vl, r2t, rpi, lens, chunk, S)
        assert np.max(np.abs(out - ref)) < 1e-12
        for b in range(B):
            n = (lens[b] + chunk - 1) // chunk
            assert np.all(np.isfinite(m_p[b, :, :n])) and np.all(np.isnan(m_p[b, :, n:]))
            assert np.all(l_p[b, :, :n] >= 1.0)  # the max term contributes exp(0) = 1
        if chunk >= 30:
            assert np.max(np.abs(o_p[:, :, 0] - ref)) < 1e-13


def test_paged_equals_contiguous_bitwise():
    B, H, Hk, D = 3, 4, 2, 32
    lens = np.array([13, 40, 64], np.int32)
    kl, vl, r2t, msl = _contig(17, B, H, Hk, D, lens, "bf16")
    rng = np.random.default_rng(17)
    pool = 5 * B * msl
    perm = rng.permutation(pool)[: B * msl].astype(np.int32)
    kp = np.zeros((pool, Hk, D), np.uint16)
    vp = np.zeros((pool, Hk, D), np.uint16)
    kp[perm] = kl
    vp[perm] = vl
    r2t_p = perm[r2t]
    q = W.normal_values((B, H, D), "bf16", 17, 3)
    rpi = np.arange(B, dtype=np.int32)
    assert np.array_equal(oracle.decode(q, kl, vl, r2t, rpi, lens),
                          oracle.decode(q, kp, vp, r2t_p, rpi, lens))
    qp = W.normal_values((int(lens.sum()), H, D), "bf16", 17, 4)
    ind = W.prefix_sum(lens)
    assert np.array_equal(oracle.prefill(qp, kl, vl, r2t, rpi, ind, ind),
                          oracle.prefill(qp, kp, vp, r2t_p, rpi, ind, ind))


def test_resumed_prefill_equals_suffix_of_full_prefill():
    # the request resumes right after its cached prefix: its rows are the tail rows of the
    # prefill that would have covered the whole sequence (AstrAI inference guide, RadixCache)
    B, H, Hk, D = 2, 4, 1, 32
    kv = np.array([48, 37], np.int32)
    prefix = np.array([16, 32], np.int32)
    kl, vl, r2t, msl = _contig(18, B, H, Hk, D, kv, "bf16")
    rpi = np.arange(B, dtype=np.int32)
    qfull = W.normal_values((int(kv.sum()), H, D), "bf16", 18, 3)
    ind = W.prefix_sum(kv)
    full = oracle.prefill(qfull, kl, vl, r2t, rpi, ind, ind)
    keep = np.concatenate([np.arange(ind[b] + prefix[b], ind[b + 1]) for b in range(B)])
    qo = W.prefix_sum(kv - prefix)
    res = oracle.prefill(np.ascontiguousarray(qfull[keep]), kl, vl, r2t, rpi, qo, ind)
    assert np.array_equal(res, full[keep])
    sub = oracle.prefill(np.ascontiguousarray(qfull[keep]), kl, vl, r2t, rpi, qo, ind,
                         rows=np.array([0, 5, 36], np.int32))
    assert np.array_equal(sub, res[[0, 5, 36]])


def test_tiny_chain_decode_equals_prefill_row():
    # the tiny configuration: prefill {7, 13}, then a decode step at positions 7 and 13
    wl = W.tiny_chain()
    pool = wl.pool
    kl, vl = pool.k_buffer[0], pool.v_buffer[0]
    r = wl.rope
    q1 = oracle.rope_kv_write(r.q, r.k, r.v, r.freqs_cis, r.position_ids, r.out_cache_loc, kl, vl)
    r2 = wl.rope2
    q2 = oracle.rope_kv_write(r2.q, r2.k, r2.v, r2.freqs_cis, r2.position_ids, r2.out_cache_loc, kl, vl)
    d = wl.decode2
    dec = oracle.decode(q2, kl, vl, pool.req_to_token, d.req_pool_indices, d.seq_lens)
    # prefill over {8, 14} tokens whose last rows are the decode queries
    qa = np.concatenate([q1[0:7], q2[0:1], q1[7:20], q2[1:2]])
    ind = W.prefix_sum(d.seq_lens)
    pre = oracle.prefill(qa, kl, vl, pool.req_to_token, d.req_pool_indices, ind, ind)
    assert np.array_equal(dec, pre[ind[1:] - 1])
    o_p, m_p, l_p, merged = oracle.decode_split(q2, kl, vl, pool.req_to_token,
                                                d.req_pool_indices, d.seq_lens, 4, 4)
    assert np.max(np.abs(merged - dec)) < 1e-12


def test_oracle_thread_count_does_not_change_results():
    B, H, Hk, D = 4, 8, 2, 32
    lens = np.array([10, 64, 33, 2], np.int32)
    kl, vl, r2t, msl = _contig(19, B, H, Hk, D, lens, "bf16")
    q = W.normal_values((B, H, D), "bf16", 19, 3)
    rpi = np.arange(B, dtype=np.int32)
    n0 = oracle.num_threads()
    try:
        oracle.set_num_threads(1)
        a = oracle.decode(q, kl, vl, r2t, rpi, lens)
        oracle.set_num_threads(max(2, n0))
        b = oracle.decode(q, kl, vl, r2t, rpi, lens)
    finally:
        oracle.set_num_threads(n0)
    assert np.array_equal(a, b)
