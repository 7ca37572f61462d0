"""Decode with RoPE and the new token's cache write folded in (astr_decode_attention_rope).

It must leave exactly the cache bytes and produce exactly the decode output of the two separate
calls (astr_rope_kv_write, then astr_decode_attention), and match the oracle's rotate + write
followed by its decode.
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


def _f64(a):
    return W.f32_from_bf16_bits(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


def _fused(dw):
    r, d = dw.rope, dw.decode
    d["kv"].out_cache_loc = r["loc"]
    dw.refresh()
    A.astr_decode_attention_rope(dw._c(d), d["layer"], r["q"], r["k"], r["v"], dw.n_heads,
                                 r["freqs"], r["freqs"].shape[0], r["pos"])


@pytest.mark.parametrize("H,Hk,page,lens", [
    (16, 4, 16, [1, 20, 333, 5000]),    # G = 4, a split request, a one-token request
    (16, 16, 16, [700, 129]),           # G = 1
    (32, 4, 1, [64, 1000, 2]),          # G = 8, page size 1 (no page runs)
    (64, 4, 16, [4097, 17]),            # G = 16
])
def test_fused_equals_separate_calls_and_oracle(H, Hk, page, lens):
    import torch
    seed = W.SEED_BASE + 800 + sum(lens) + H
    mk = lambda: W.make_case("bf16", H, Hk, 128, page, lens, None, with_rope=True, split_chunk=0,
                             max_splits=64, seed=seed)
    wl = mk()
    two, one = DV.DeviceWorkload.upload(wl), DV.DeviceWorkload.upload(mk())
    two.run_rope()
    two.run_decode()
    _fused(one)
    torch.cuda.synchronize()
    assert A.astr_device_error() == 0
    for lyr in range(wl.pool.n_layers):
        assert np.array_equal(DV.to_host(one.k_buffer[lyr]), DV.to_host(two.k_buffer[lyr]))
        assert np.array_equal(DV.to_host(one.v_buffer[lyr]), DV.to_host(two.v_buffer[lyr]))
    assert np.array_equal(DV.to_host(one.decode["out"]), DV.to_host(two.decode["out"]))
    # the oracle: rotate + write on the host layer, then decode with the rotated query
    r, d = wl.rope, wl.decode
    kl = np.ascontiguousarray(wl.pool.k_buffer[1]).copy()
    vl = np.ascontiguousarray(wl.pool.v_buffer[1]).copy()
    q_ref = oracle.rope_kv_write(r.q, r.k, r.v, r.freqs_cis, r.position_ids, r.out_cache_loc, kl, vl)
    assert np.array_equal(DV.to_host(one.k_buffer[1]), kl)
    assert np.array_equal(DV.to_host(one.v_buffer[1]), vl)
    ref = oracle.decode(q_ref, kl, vl, wl.pool.req_to_token, d.req_pool_indices, d.seq_lens)
    assert np.max(np.abs(_f64(DV.to_host(one.decode["out"])) - ref)) <= 2e-2


def test_fused_rejects_shapes_it_does_not_serve():
    wl = W.make_case("f32", 8, 4, 64, 16, [10, 30], None, with_rope=True)
    dw = DV.DeviceWorkload.upload(wl)
    with pytest.raises(A.AstrError) as e:
        _fused(dw)
    assert e.value.status == 2  # ASTR_ERR_UNSUPPORTED


def test_fused_unsplit_plan_at_a_full_batch():
    """Enough requests (batch x n_kv_heads >= 6 per SM) that the plan leaves every request
    unsplit and launches no merge, the path of the mixed-batch step that bench.py times; lengths
    cover one-token requests, page edges and several 128-token tiles."""
    import torch
    rng = np.random.default_rng(W.SEED_BASE + 870)
    lens = rng.integers(1, 700, size=256)
    lens[:6] = [1, 2, 15, 16, 17, 129]
    seed = W.SEED_BASE + 871
    mk = lambda: W.make_case("bf16", 16, 4, 128, 16, lens, None, with_rope=True, split_chunk=0,
                             max_splits=16, seed=seed)
    wl = mk()
    two, one = DV.DeviceWorkload.upload(wl), DV.DeviceWorkload.upload(mk())
    assert A.astr_decode_plan(one.decode["kv"], 16)[1] == 1
    two.run_rope()
    two.run_decode()
    _fused(one)
    torch.cuda.synchronize()
    assert A.astr_device_error() == 0
    assert np.array_equal(DV.to_host(one.k_buffer[1]), DV.to_host(two.k_buffer[1]))
    assert np.array_equal(DV.to_host(one.v_buffer[1]), DV.to_host(two.v_buffer[1]))
    assert np.array_equal(DV.to_host(one.decode["out"]), DV.to_host(two.decode["out"]))
    r, d = wl.rope, wl.decode
    kl = np.ascontiguousarray(wl.pool.k_buffer[1]).copy()
    vl = np.ascontiguousarray(wl.pool.v_buffer[1]).copy()
    q_ref = oracle.rope_kv_write(r.q, r.k, r.v, r.freqs_cis, r.position_ids, r.out_cache_loc, kl, vl)
    assert np.array_equal(DV.to_host(one.k_buffer[1]), kl)
    assert np.array_equal(DV.to_host(one.v_buffer[1]), vl)
    ref = oracle.decode(q_ref, kl, vl, wl.pool.req_to_token, d.req_pool_indices, d.seq_lens)
    assert np.max(np.abs(_f64(DV.to_host(one.decode["out"])) - ref)) <= 2e-2
