"""Per-step metadata on the device (astr_bind_tasks) and prefill on its padded tile maps.

The device planner must give exactly the host builder's prefix sums and tile order (index
work: bit-exact), with the empty (-1) entries first; the prefill must skip those entries, so
that padded maps give the same bytes as exact ones; and a CUDA graph of bind_tasks followed
by the prefill of every layer must follow new lengths written between replays.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import paged_kv_cache_apply_gb300 as A
from paged_kv_cache_apply_gb300 import build as B
from paged_kv_cache_apply_gb300 import device as DV
from paged_kv_cache_apply_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()
    oracle.build()
    import torch
    torch.cuda.init()
    A.astr_set_checked(False)
    yield
    A.astr_set_checked(False)


def _i32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _plan(q, k, max_tiles, rows=128, decode=False):
    import torch
    B_ = len(k)
    qo, kv = torch.full((B_ + 1,), 7, dtype=torch.int32, device="cuda"), \
        torch.full((B_ + 1,), 7, dtype=torch.int32, device="cuda")
    tb = torch.full((max_tiles,), 5, dtype=torch.int32, device="cuda")
    ti = torch.full((max_tiles,), 5, dtype=torch.int32, device="cuda")
    A.astr_bind_tasks(None if decode else _i32(q), _i32(k), None if decode else qo, kv,
                      tb if max_tiles else None, ti if max_tiles else None, rows)
    torch.cuda.synchronize()
    return [DV.to_host(t) for t in (qo, kv, tb, ti)]


def _expect(q, k, max_tiles, rows=128):
    tb, ti = W.q_tiles(q, k, rows)
    pad = max_tiles - len(tb)
    return (W.prefix_sum(q), W.prefix_sum(k), np.concatenate([np.full(pad, -1), tb]).astype(np.int32),
            np.concatenate([np.full(pad, -1), ti]).astype(np.int32))


@pytest.mark.parametrize("seed,rows", [(0, 128), (1, 128), (2, 128), (3, 64), (4, 1), (5, 200)])
def test_matches_the_host_builder(seed, rows):
    rng = np.random.default_rng([seed, 21])
    Bn = int(rng.integers(1, 40))
    q = rng.integers(0, 1500 if rows > 1 else 60, size=Bn)
    q[rng.random(Bn) < 0.2] = 0
    k = q + rng.integers(0, 3000, size=Bn)
    n = len(W.q_tiles(q, k, rows)[0])
    for max_tiles in (n, n + 37):
        got = _plan(q, k, max_tiles, rows)
        for g, e in zip(got, _expect(q, k, max_tiles, rows)):
            assert np.array_equal(g, e)
    assert A.astr_device_error() == 0


def test_largest_batch_many_blocks():
    # 16383 requests (the most the planner holds): 64 per scan segment, a grid of many blocks
    rng = np.random.default_rng(77)
    q = rng.integers(0, 300, size=16383)
    k = q + rng.integers(0, 2000, size=16383)
    n = len(W.q_tiles(q, k)[0])
    got = _plan(q, k, n + 300)
    for g, e in zip(got, _expect(q, k, n + 300)):
        assert np.array_equal(g, e)
    assert A.astr_device_error() == 0


def test_decode_batch_and_empty_batch():
    lens = np.array([5, 1, 4096, 77], np.int32)
    _, kv, _, _ = _plan(None, lens, 0, decode=True)
    assert np.array_equal(kv, W.prefix_sum(lens))
    qo, kv, tb, ti = _plan(np.zeros(0, np.int32), np.zeros(0, np.int32), 9)
    assert qo.tolist() == [0] and kv.tolist() == [0]
    assert np.all(tb == -1) and np.all(ti == -1)
    assert A.astr_device_error() == 0


def test_device_errors_empty_every_entry():
    q, k = np.array([300, 20]), np.array([300, 10])  # kv_len < q_len
    _, _, tb, ti = _plan(q, k, 8)
    assert np.all(tb == -1) and np.all(ti == -1)
    assert A.astr_device_error() == 0x8  # ASTR_DEVERR_LEN
    q, k = np.array([300, 129]), np.array([300, 129])  # 5 tiles, room for 4
    _, _, tb, ti = _plan(q, k, 4)
    assert np.all(tb == -1) and np.all(ti == -1)
    assert A.astr_device_error() == 0x20  # ASTR_DEVERR_META


def test_host_errors():
    import torch
    z = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(A.AstrError) as e:
        A.astr_bind_tasks(z[:3], z[:3], z, None, z, z)
    assert e.value.status == 1
    big = torch.zeros(16384, dtype=torch.int32, device="cuda")
    ind = torch.zeros(16385, dtype=torch.int32, device="cuda")
    with pytest.raises(A.AstrError) as e:
        A.astr_bind_tasks(big, big, ind, ind, z, z)
    assert e.value.status == 2


def _padded(dw, extra):
    """A prefill KVCache whose tile maps come from astr_bind_tasks with `extra` empty entries."""
    import torch
    p = dw.prefill["kv"]
    q = np.diff(DV.to_host(p.qo_indptr))
    k = np.diff(DV.to_host(p.kv_indptr))
    n = int(p.q_tile_to_batch.shape[0])
    qo, kv = torch.empty_like(p.qo_indptr), torch.empty_like(p.kv_indptr)
    tb = torch.empty(n + extra, dtype=torch.int32, device="cuda")
    ti = torch.empty_like(tb)
    A.astr_bind_tasks(_i32(q), _i32(k), qo, kv, tb, ti, p.q_tile_rows)
    return dataclasses.replace(p, qo_indptr=qo, kv_indptr=kv, q_tile_to_batch=tb, q_tile_to_index=ti)


@pytest.mark.parametrize("dtype,H,Hk,D,page,kv_lens,q_lens", [
    ("bf16", 16, 4, 128, 16, [1, 128, 300, 700], [1, 128, 129, 300]),
    ("bf16", 16, 4, 128, 16, [50, 500, 20], [0, 300, 20]),
    ("f32", 4, 2, 64, 16, [13, 160, 48], [13, 128, 16]),
])
@pytest.mark.parametrize("checked", [False, True])
def test_prefill_on_padded_maps_equals_exact_maps(dtype, H, Hk, D, page, kv_lens, q_lens, checked):
    import torch
    wl = W.make_case(dtype, H, Hk, D, page, kv_lens, q_lens, seed=W.SEED_BASE + 950 + sum(kv_lens))
    dw = DV.DeviceWorkload.upload(wl)
    dw.run_prefill()
    exact = dw.prefill["out"].clone()
    out = torch.zeros_like(exact)
    A.astr_set_checked(checked)
    try:
        A.astr_prefill_attention(_padded(dw, 13), dw.prefill["layer"], dw.prefill["q"], out, dw.n_heads)
    finally:
        A.astr_set_checked(False)
    torch.cuda.synchronize()
    bits = (lambda t: t.view(torch.int16)) if dtype == "bf16" else (lambda t: t)
    assert torch.equal(bits(out), bits(exact))
    assert A.astr_device_error() == 0


def test_two_layer_prefill_graph_follows_device_lengths():
    # one graph: bind_tasks from device q_lens / kv_lens, then the prefill of both layers on the
    # padded maps; between replays the host writes only new lengths
    import torch
    kv_cap = np.array([900, 300, 1500, 64], np.int32)
    q_cap = np.array([900, 100, 700, 64], np.int32)
    wl = W.make_case("bf16", 16, 4, 128, 16, kv_cap, q_cap, n_layers=2, seed=W.SEED_BASE + 960)
    dw = DV.DeviceWorkload.upload(wl)
    p = dw.prefill["kv"]
    rows_cap = int(q_cap.sum())
    max_tiles = 24
    ql_d, kl_d = _i32(q_cap), _i32(kv_cap)
    qo, kv = torch.empty(5, dtype=torch.int32, device="cuda"), torch.empty(5, dtype=torch.int32, device="cuda")
    tb = torch.empty(max_tiles, dtype=torch.int32, device="cuda")
    ti = torch.empty_like(tb)
    kvc = dataclasses.replace(p, qo_indptr=qo, kv_indptr=kv, q_tile_to_batch=tb, q_tile_to_index=ti,
                              n_tokens=rows_cap)
    q = dw.prefill["q"]
    outs = [torch.zeros_like(dw.prefill["out"]) for _ in range(2)]

    def step():
        A.astr_bind_tasks(ql_d, kl_d, qo, kv, tb, ti)
        for lyr in (0, 1):
            A.astr_prefill_attention(kvc, lyr, q, outs[lyr], dw.n_heads)

    step()  # eager first calls
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        step()
    for qn, kn in [(q_cap, kv_cap),
                   (np.array([128, 0, 129, 1], np.int32), np.array([500, 300, 1500, 1], np.int32)),
                   (np.array([0, 0, 0, 0], np.int32), np.array([9, 0, 1, 64], np.int32)),
                   (np.array([1, 100, 700, 63], np.int32), np.array([1, 100, 1000, 64], np.int32))]:
        ql_d.copy_(torch.from_numpy(qn))
        kl_d.copy_(torch.from_numpy(kn))
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        total = int(qn.sum())
        qo_ref, kv_ref = W.prefix_sum(qn), W.prefix_sum(kn)
        assert np.array_equal(DV.to_host(qo), qo_ref) and np.array_equal(DV.to_host(kv), kv_ref)
        for lyr in (0, 1):
            kl = np.ascontiguousarray(wl.pool.k_buffer[lyr])
            vl = np.ascontiguousarray(wl.pool.v_buffer[lyr])
            ref = oracle.prefill(wl.prefill.q[:total], kl, vl, wl.pool.req_to_token,
                                 wl.prefill.req_pool_indices, qo_ref, kv_ref)
            got = W.f32_from_bf16_bits(DV.to_host(outs[lyr])[:total]).astype(np.float64)
            assert got.shape == ref.shape
            if total:
                assert np.max(np.abs(got - ref)) <= TOL["bf16"]
            assert not torch.any(outs[lyr][total:].view(torch.int16) != 0)  # rows past the batch untouched
    assert A.astr_device_error() == 0
