"""Training-path RoPE on the GPU (astr_rope_apply / astr_rope_backward) against the oracle.

Rotation is index-exact arithmetic under the rounding specification, so the comparison is
bit for bit, for the forward and for the backward (the rotation by -theta).
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_apply_gb300 as A
from paged_kv_cache_apply_gb300 import build as B
from paged_kv_cache_apply_gb300 import device as DV
from paged_kv_cache_apply_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()
    oracle.build()
    import torch
    torch.cuda.init()


def _dev(a, dt):
    return DV.to_torch(a, dt, "cuda")


@pytest.mark.parametrize("dtype,T,H,Hk,D,fmax", [
    ("bf16", 2304, 16, 4, 128, 8192),
    ("f32", 37, 4, 2, 64, 100),
    ("bf16", 129, 8, 0, 64, 300),     # q only
    ("f32", 5, 0, 3, 128, 16),        # k only
])
@pytest.mark.parametrize("inverse", [False, True])
@pytest.mark.parametrize("in_place", [False, True])
def test_bit_exact_against_oracle(dtype, T, H, Hk, D, fmax, inverse, in_place):
    import torch
    seed = W.SEED_BASE + 1000 + T + H + Hk
    rng = np.random.default_rng(seed)
    qh = W.normal_values((T, max(H, 1), D), dtype, seed, 1)[:, :H]
    kh = W.normal_values((T, max(Hk, 1), D), dtype, seed, 2)[:, :Hk]
    fr = W.rope_freqs_cis(fmax, D)
    pos = rng.integers(0, fmax, T).astype(np.int32)
    q, k = _dev(np.ascontiguousarray(qh), dtype), _dev(np.ascontiguousarray(kh), dtype)
    qo = q if in_place else torch.empty_like(q)
    ko = k if in_place else torch.empty_like(k)
    f, p = _dev(fr, "f32"), _dev(pos, "i32")
    call = A.astr_rope_backward if inverse else A.astr_rope_apply
    call(q, qo, k if Hk else None, ko if Hk else None, f, p)
    torch.cuda.synchronize()
    if H:
        assert np.array_equal(DV.to_host(qo), oracle.rope_apply(qh, fr, pos, inverse=inverse))
    if Hk:
        assert np.array_equal(DV.to_host(ko), oracle.rope_apply(kh, fr, pos, inverse=inverse))
    assert A.astr_device_error() == 0


def test_forward_reproduces_rope_kv_write_q_out():
    # the training forward and the inference write rotate q with the same arithmetic
    import torch
    wl = W.mixed_b256_p4x512(n_decode=16, lmax=600, n_prefill=1, chunk_len=200)
    dw = DV.DeviceWorkload.upload(wl)
    dw.run_rope()
    r = dw.rope
    q_out = torch.empty_like(r["q"])
    A.astr_rope_apply(r["q"], q_out, None, None, r["freqs"], r["pos"])
    torch.cuda.synchronize()
    assert torch.equal(q_out.view(torch.int16), r["q_out"].view(torch.int16))


@pytest.mark.parametrize("dt,D", [("bf16", 128), ("f32", 64)])
def test_autograd_function_runs_both_passes_in_the_library(dt, D):
    import torch
    from paged_kv_cache_apply_gb300.rotary import apply_rotary_emb
    Bn, L, H, Hk = 2, 50, 8, 2
    seed = W.SEED_BASE + 1100 + D
    qh = W.normal_values((Bn * L, H, D), dt, seed, 1)
    kh = W.normal_values((Bn * L, Hk, D), dt, seed, 2)
    gqh = W.normal_values((Bn * L, H, D), dt, seed, 3)
    gkh = W.normal_values((Bn * L, Hk, D), dt, seed, 4)
    fr = W.rope_freqs_cis(256, D)
    pos = np.tile(np.arange(L, dtype=np.int32), Bn)
    q = _dev(qh, dt).view(Bn, L, H, D).detach().requires_grad_(True)
    k = _dev(kh, dt).view(Bn, L, Hk, D).detach().requires_grad_(True)
    qr, kr = apply_rotary_emb(q, k, _dev(fr, "f32"), _dev(pos, "i32").view(Bn, L))
    torch.autograd.backward([qr, kr], [_dev(gqh, dt).view(Bn, L, H, D),
                                       _dev(gkh, dt).view(Bn, L, Hk, D)])
    torch.cuda.synchronize()
    assert np.array_equal(DV.to_host(qr.detach().reshape(-1, H, D)), oracle.rope_apply(qh, fr, pos))
    assert np.array_equal(DV.to_host(kr.detach().reshape(-1, Hk, D)), oracle.rope_apply(kh, fr, pos))
    assert np.array_equal(DV.to_host(q.grad.reshape(-1, H, D)), oracle.rope_apply(gqh, fr, pos, inverse=True))
    assert np.array_equal(DV.to_host(k.grad.reshape(-1, Hk, D)), oracle.rope_apply(gkh, fr, pos, inverse=True))


def test_bad_position_is_skipped_and_flagged():
    import torch
    D = 64
    fr = W.rope_freqs_cis(32, D)
    qh = W.normal_values((3, 2, D), "f32", 5, 1)
    pos = np.array([1, 32, -1], np.int32)
    q = _dev(qh, "f32")
    out = torch.full_like(q, 7.0)
    A.astr_rope_backward(q, out, None, None, _dev(fr, "f32"), _dev(pos, "i32"))
    torch.cuda.synchronize()
    got = DV.to_host(out)
    assert np.array_equal(got[0], oracle.rope_apply(qh[:1], fr, pos[:1], inverse=True)[0])
    assert np.all(got[1:] == 7.0)
    assert A.astr_device_error() == 0x2  # ASTR_DEVERR_POS


def test_argument_errors():
    import torch
    q = torch.zeros((4, 2, 96), dtype=torch.float32, device="cuda")
    f = torch.zeros((8, 48, 2), dtype=torch.float32, device="cuda")
    p = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(A.AstrError) as e:
        A.astr_rope_apply(q, q, None, None, f, p)
    assert e.value.status == 2  # head_dim 96 is not served
    f = torch.zeros((8, 32, 2), dtype=torch.float32, device="cuda")
    flat = torch.zeros(4 * 2 * 64 + 1, dtype=torch.float32, device="cuda")
    q = flat[1:].view(4, 2, 64)  # 4 bytes past a 16-byte boundary
    with pytest.raises(A.AstrError) as e:
        A.astr_rope_apply(q, q, None, None, f, p)
    assert e.value.status == 1
    with pytest.raises(TypeError):
        A.astr_rope_apply(q, q, None, None, f, p.long())
