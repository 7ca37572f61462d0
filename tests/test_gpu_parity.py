"""GPU <-> oracle parity through the C ABI, on the same seeded inputs.

Bars: cache slot writes, gathers and the rotated q/k bytes are bit-exact (the rotation's f32
rounding is specified, so the oracle reproduces it); attention outputs are within max-abs
1e-5 for f32 and 2e-2 for bf16 (bf16 storage, f32 accumulation) of the fp64 oracle.
"""
import math

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
    import torch
    torch.cuda.init()
    A.astr_set_checked(False)
    A.astr_set_wait_timeout_ns(1_000_000_000)
    yield
    A.astr_set_checked(False)


def _sync():
    import torch
    torch.cuda.synchronize()


def wid(a):
    return W.f32_from_bf16_bits(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


def maxerr(got, ref):
    return float(np.max(np.abs(wid(got) - ref))) if got.size else 0.0


def host_layer(wl, layer):
    return (np.ascontiguousarray(wl.pool.k_buffer[layer]).copy(),
            np.ascontiguousarray(wl.pool.v_buffer[layer]).copy())


def check_rope(dw, which, kl, vl):
    """Run the oracle's rotate + write on the host layer; compare q_out and the cache bits."""
    r = getattr(dw.wl, which)
    q_ref = oracle.rope_kv_write(r.q, r.k, r.v, r.freqs_cis, r.position_ids, r.out_cache_loc, kl, vl)
    d = getattr(dw, which)
    assert np.array_equal(DV.to_host(d["q_out"]), q_ref), "q_out bits differ"
    return q_ref


def check_cache_equal(dw, layer, kl, vl):
    assert np.array_equal(DV.to_host(dw.k_buffer[layer]), kl), "k cache bits differ"
    assert np.array_equal(DV.to_host(dw.v_buffer[layer]), vl), "v cache bits differ"


# ------------------------------------------------------------------------------------------
# the tiny chain: prefill {7, 13}, then a decode step (f32, head_dim 64, G = 2)
# ------------------------------------------------------------------------------------------


def test_tiny_chain():
    wl = W.tiny_chain()
    dw = DV.DeviceWorkload.upload(wl)
    kl, vl = host_layer(wl, 0)
    dw.run_rope()
    dw.run_prefill()
    _sync()
    q1 = check_rope(dw, "rope", kl, vl)
    check_cache_equal(dw, 0, kl, vl)
    p = wl.prefill
    ref = oracle.prefill(q1, kl, vl, wl.pool.req_to_token, p.req_pool_indices, p.qo_indptr,
                         p.kv_indptr)
    assert maxerr(DV.to_host(dw.prefill["out"]), ref) <= TOL["f32"]
    # decode step at positions 7 and 13, split into chunks of 4
    dw.run_rope("rope2")
    dw.run_decode("decode2")
    _sync()
    q2 = check_rope(dw, "rope2", kl, vl)
    check_cache_equal(dw, 0, kl, vl)
    d = wl.decode2
    ref_d = oracle.decode(q2, kl, vl, wl.pool.req_to_token, d.req_pool_indices, d.seq_lens)
    assert maxerr(DV.to_host(dw.decode2["out"]), ref_d) <= TOL["f32"]
    o_p, m_p, l_p, _ = oracle.decode_split(q2, kl, vl, wl.pool.req_to_token, d.req_pool_indices,
                                           d.seq_lens, 4, 4)
    go = DV.to_host(dw.decode2["o_part"])
    gml = DV.to_host(dw.decode2["ml_part"])
    for b in range(2):
        n = (d.seq_lens[b] + 3) // 4
        assert np.max(np.abs(go[b, :, :n] - o_p[b, :, :n])) <= TOL["f32"]
        lse_gpu = gml[b, :, :n, 0].astype(np.float64) + np.log(gml[b, :, :n, 1].astype(np.float64))
        lse_ref = m_p[b, :, :n] + np.log(l_p[b, :, :n])
        assert np.max(np.abs(lse_gpu - lse_ref)) <= 1e-5


# ------------------------------------------------------------------------------------------
# parametrised small cases
# ------------------------------------------------------------------------------------------

DECODE_CASES = [
    # dtype, H, Hk, D, page, lens, split_chunk
    ("bf16", 16, 4, 128, 16, [1, 16, 17, 300, 1000], 0),
    ("bf16", 16, 4, 128, 1, [1, 2, 31, 32, 33, 700], 64),
    ("bf16", 8, 8, 128, 16, [5, 129, 500], 128),
    ("bf16", 16, 8, 64, 1, [3, 64, 65, 257], 0),
    ("bf16", 32, 4, 128, 16, [40, 333, 2049], 256),
    ("f32", 8, 4, 64, 16, [1, 33, 250], 32),
    ("f32", 4, 4, 128, 1, [7, 100, 129], 0),
    ("f32", 16, 2, 128, 16, [2, 90, 400], 96),
    ("bf16", 2, 2, 64, 1, [1, 8, 4000], 512),
    ("bf16", 64, 4, 128, 16, [1, 129, 1000], 0),      # G = 16 on the tensor cores
]


@pytest.mark.parametrize("dtype,H,Hk,D,page,lens,chunk", DECODE_CASES)
def test_decode_cases(dtype, H, Hk, D, page, lens, chunk):
    wl = W.make_case(dtype, H, Hk, D, page, lens, None, split_chunk=chunk, max_splits=64,
                     seed=W.SEED_BASE + 200 + sum(lens) + H)
    dw = DV.DeviceWorkload.upload(wl)
    dw.run_decode()
    _sync()
    kl, vl = host_layer(wl, 1)
    d = wl.decode
    ref = oracle.decode(d.q, kl, vl, wl.pool.req_to_token, d.req_pool_indices, d.seq_lens)
    assert maxerr(DV.to_host(dw.decode["out"]), ref) <= TOL[dtype]
    # the cache is read-only for decode
    assert np.array_equal(DV.to_host(dw.k_buffer), wl.pool.k_buffer)


PREFILL_CASES = [
    # dtype, H, Hk, D, page, kv_lens, q_lens
    ("bf16", 16, 4, 128, 16, [1, 128, 300, 700], [1, 128, 129, 300]),
    ("bf16", 8, 2, 64, 1, [200, 17, 256], [72, 17, 255]),
    ("f32", 4, 2, 64, 16, [13, 160, 48], [13, 128, 16]),
    ("f32", 8, 1, 128, 1, [100, 37], [99, 5]),
    ("bf16", 16, 16, 128, 16, [1040, 130], [16, 130]),
    ("bf16", 12, 4, 128, 16, [300, 77], [300, 40]),        # G = 3: one query head per block
    ("bf16", 32, 4, 128, 16, [600, 129], [256, 129]),      # G = 8: four head pairs per group
    ("bf16", 16, 4, 128, 1, [400, 129, 64], [400, 1, 64]),  # page 1: no page runs, all cp.async
    ("bf16", 16, 4, 128, 16, [50, 500, 20], [0, 300, 20]),  # a request with no new rows
    # 400 head-pair items for at most 152 blocks: every block of the persistent kernel runs
    # several items in turn (whole tiles, tiles cut by the request's end, resumed prefixes)
    ("bf16", 4, 2, 128, 16, [129 + 37 * (b % 5) for b in range(100)], [129 - (b % 3) * 60 for b in range(100)]),
    # 232 items with G = 4 on one-token pages: every K/V row comes by cp.async, with prefixes
    ("bf16", 16, 4, 128, 1, [129, 300, 256, 400, 140, 260, 535, 129, 257, 190, 300, 480],
     [129, 200, 256, 300, 140, 260, 135, 129, 257, 190, 300, 280]),
    # G = 8 with more items than SMs: four head pairs per KV group in the persistent kernel
    ("bf16", 32, 4, 128, 16, [300, 256, 400, 512, 256, 384], [256, 256, 256, 300, 256, 384]),
]


@pytest.mark.parametrize("dtype,H,Hk,D,page,kv_lens,q_lens", PREFILL_CASES)
def test_prefill_cases(dtype, H, Hk, D, page, kv_lens, q_lens):
    wl = W.make_case(dtype, H, Hk, D, page, kv_lens, q_lens, seed=W.SEED_BASE + 300 + sum(kv_lens))
    dw = DV.DeviceWorkload.upload(wl)
    dw.run_prefill()
    _sync()
    kl, vl = host_layer(wl, 1)
    p = wl.prefill
    ref = oracle.prefill(p.q, kl, vl, wl.pool.req_to_token, p.req_pool_indices, p.qo_indptr,
                         p.kv_indptr)
    assert maxerr(DV.to_host(dw.prefill["out"]), ref) <= TOL[dtype]
    assert A.astr_device_error() == 0  # no bounded wait ran out, no index was rejected


@pytest.mark.parametrize("dtype,D,G,page", [("bf16", 128, 4, 16), ("f32", 64, 2, 1),
                                            ("bf16", 64, 8, 1), ("f32", 128, 1, 16)])
def test_rope_then_decode_and_prefill(dtype, D, G, page):
    Hk = 2
    H = G * Hk
    # decode: new token at L-1 written by the fused step, then attended
    wl = W.make_case(dtype, H, Hk, D, page, [1, 20, 333], None, with_rope=True,
                     seed=W.SEED_BASE + 400 + D + G)
    dw = DV.DeviceWorkload.upload(wl)
    dw.run_rope()
    dw.run_decode()
    _sync()
    kl, vl = host_layer(wl, 1)
    q_ref = check_rope(dw, "rope", kl, vl)
    check_cache_equal(dw, 1, kl, vl)
    assert np.array_equal(DV.to_host(dw.k_buffer[0]), wl.pool.k_buffer[0])  # other layer intact
    d = wl.decode
    ref = oracle.decode(q_ref, kl, vl, wl.pool.req_to_token, d.req_pool_indices, d.seq_lens)
    assert maxerr(DV.to_host(dw.decode["out"]), ref) <= TOL[dtype]
    # prefill with a page-aligned cached prefix
    wl = W.make_case(dtype, H, Hk, D, page, [150, 48, 16], [134, 48, 1], with_rope=True,
                     seed=W.SEED_BASE + 500 + D + G)
    dw = DV.DeviceWorkload.upload(wl)
    dw.run_rope()
    dw.run_prefill()
    _sync()
    kl, vl = host_layer(wl, 1)
    q_ref = check_rope(dw, "rope", kl, vl)
    check_cache_equal(dw, 1, kl, vl)
    p = wl.prefill
    ref = oracle.prefill(q_ref, kl, vl, wl.pool.req_to_token, p.req_pool_indices, p.qo_indptr,
                         p.kv_indptr)
    assert maxerr(DV.to_host(dw.prefill["out"]), ref) <= TOL[dtype]


def test_rope_in_place_matches_out_of_place():
    import torch
    wl = W.make_case("bf16", 16, 4, 128, 16, [10, 300], [10, 300], with_rope=True)
    dw = DV.DeviceWorkload.upload(wl)
    r = dw.rope
    q_inplace = r["q"].clone()
    A.astr_rope_kv_write(r["kv"], r["layer"], q_inplace, q_inplace, r["k"], r["v"], 16,
                         r["freqs"], r["freqs"].shape[0], r["pos"])
    dw.run_rope()
    _sync()
    assert torch.equal(q_inplace.view(torch.int16), r["q_out"].view(torch.int16))


# ------------------------------------------------------------------------------------------
# guard regions: nothing outside the named outputs is written
# ------------------------------------------------------------------------------------------


def test_outputs_do_not_spill_into_guard_regions():
    import torch
    wl = W.make_case("bf16", 16, 4, 128, 16, [100, 4097, 33], None, split_chunk=512,
                     max_splits=9)
    dw = DV.DeviceWorkload.upload(wl)
    d = dw.decode
    G = 4096
    big = torch.full((2 * G + d["out"].numel(),), 12345, dtype=torch.int16, device="cuda")
    out = big[G: G + d["out"].numel()].view(torch.bfloat16).view(d["out"].shape)
    d["kv"].decode_out = out
    dw.refresh()
    dw.run_decode()
    _sync()
    assert torch.all(big[:G] == 12345) and torch.all(big[G + d["out"].numel():] == 12345)
    kl, vl = host_layer(wl, 1)
    ref = oracle.decode(wl.decode.q, kl, vl, wl.pool.req_to_token, wl.decode.req_pool_indices,
                        wl.decode.seq_lens)
    assert maxerr(DV.to_host(out), ref) <= TOL["bf16"]


# ------------------------------------------------------------------------------------------
# error paths: bad indices and timeouts raise flags instead of faulting
# ------------------------------------------------------------------------------------------


def test_bad_slot_sets_flag_not_fault():
    import torch
    wl = W.make_case("bf16", 8, 2, 128, 1, [50, 60], None)
    dw = DV.DeviceWorkload.upload(wl)
    A.astr_device_error()  # clear
    r = int(wl.decode.req_pool_indices[1])
    dw.req_to_token[r, 7] = -5
    dw.req_to_token[r, 8] = wl.pool.size + 3
    dw.run_decode()
    assert A.astr_device_error() & A.DEVERR_SLOT
    A.astr_set_checked(True)
    try:
        with pytest.raises(A.AstrError) as ei:
            dw.run_decode()
        assert ei.value.status == 4
    finally:
        A.astr_set_checked(False)
    # the context is still usable: request 0 is untouched and correct
    dw.req_to_token[r, 7] = int(wl.pool.req_to_token[r, 7])
    dw.req_to_token[r, 8] = int(wl.pool.req_to_token[r, 8])
    dw.run_decode()
    _sync()
    assert A.astr_device_error() == 0
    kl, vl = host_layer(wl, 1)
    ref = oracle.decode(wl.decode.q, kl, vl, wl.pool.req_to_token, wl.decode.req_pool_indices,
                        wl.decode.seq_lens)
    assert maxerr(DV.to_host(dw.decode["out"]), ref) <= TOL["bf16"]
    del torch


def test_rope_bad_position_and_slot_skip_token():
    wl = W.make_case("f32", 4, 2, 64, 1, [5, 9], None, with_rope=True, freqs_max_len=9)
    dw = DV.DeviceWorkload.upload(wl)
    A.astr_device_error()
    dw.rope["pos"][1] = 9            # past the table
    dw.rope["loc"][0] = wl.pool.size  # past the pool
    dw.run_rope()
    flags = A.astr_device_error()
    assert flags & A.DEVERR_POS and flags & A.DEVERR_SLOT
    # both tokens skipped entirely: the cache is unchanged
    assert np.array_equal(DV.to_host(dw.k_buffer), wl.pool.k_buffer)


def test_checked_mode_catches_inconsistent_indptr():
    wl = W.make_case("bf16", 8, 2, 64, 16, [20, 40], None)
    dw = DV.DeviceWorkload.upload(wl)
    dw.decode["kv"].kv_indptr[2] = 59
    A.astr_set_checked(True)
    try:
        with pytest.raises(A.AstrError) as ei:
            dw.run_decode()
        assert ei.value.status == 4 and "0x20" in str(ei.value)
    finally:
        A.astr_set_checked(False)


def test_bounded_wait_runs_out_and_context_survives():
    assert A.astr_selftest_wait_timeout(2_000_000) == 5
    assert A.astr_device_error() == 0
    # a real decode afterwards is still correct
    wl = W.make_case("bf16", 16, 4, 128, 16, [77, 500], None)
    dw = DV.DeviceWorkload.upload(wl)
    dw.run_decode()
    _sync()
    kl, vl = host_layer(wl, 1)
    ref = oracle.decode(wl.decode.q, kl, vl, wl.pool.req_to_token, wl.decode.req_pool_indices,
                        wl.decode.seq_lens)
    assert maxerr(DV.to_host(dw.decode["out"]), ref) <= TOL["bf16"]


def test_tiny_wait_limit_never_faults():
    wl = W.make_case("bf16", 16, 4, 128, 1, [3000, 2000], None, split_chunk=0)
    dw = DV.DeviceWorkload.upload(wl)
    A.astr_set_wait_timeout_ns(1)
    try:
        for _ in range(3):
            dw.run_decode()
        _sync()
    finally:
        A.astr_set_wait_timeout_ns(1_000_000_000)
    A.astr_device_error()  # timeouts may or may not have fired; clear either way
    dw.run_decode()
    _sync()
    assert A.astr_device_error() == 0
    kl, vl = host_layer(wl, 1)
    ref = oracle.decode(wl.decode.q, kl, vl, wl.pool.req_to_token, wl.decode.req_pool_indices,
                        wl.decode.seq_lens)
    assert maxerr(DV.to_host(dw.decode["out"]), ref) <= TOL["bf16"]


def test_concurrent_decodes_on_two_streams():
    # the persistent decode takes its work items from a per-call counter: calls in flight at the
    # same time on different streams must not take each other's items
    import torch
    cases = []
    for k, lens in enumerate([[900, 3000, 17, 5000], [4096, 1, 2500, 700, 128]]):
        wl = W.make_case("bf16", 16, 4, 128, 16, lens, None, split_chunk=0, max_splits=64,
                         seed=W.SEED_BASE + 700 + k)
        cases.append((wl, DV.DeviceWorkload.upload(wl)))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    _sync()
    for rep in range(3):
        for (wl, dw), s in zip(cases, streams):
            dw.run_decode(stream=s.cuda_stream)
    _sync()
    for wl, dw in cases:
        kl, vl = host_layer(wl, 1)
        d = wl.decode
        ref = oracle.decode(d.q, kl, vl, wl.pool.req_to_token, d.req_pool_indices, d.seq_lens)
        assert maxerr(DV.to_host(dw.decode["out"]), ref) <= TOL["bf16"]
    assert A.astr_device_error() == 0


def test_empty_batches_are_no_ops():
    import torch
    wl = W.make_case("bf16", 8, 2, 64, 16, [20], None)
    dw = DV.DeviceWorkload.upload(wl)
    kv = dw.decode["kv"]
    kv.batch = 0
    dw.refresh()
    before = dw.decode["out"].clone()
    dw.run_decode()
    kv2 = dw.decode["kv"]
    _sync()
    assert torch.equal(before.view(torch.int16), dw.decode["out"].view(torch.int16))
    del kv2


@pytest.mark.parametrize("B,lens_kind", [(1100, "varied"), (1024, "ties")])
def test_decode_large_batches_rank_or_not(B, lens_kind):
    # up to 1024 requests the persistent decode ranks them by length (ties by index) and may
    # leave them unsplit; beyond that it claims them in index order. Both must cover every
    # request exactly once.
    rng = np.random.default_rng(B)
    if lens_kind == "ties":
        lens = rng.choice([100, 128, 129, 256, 700], B).astype(np.int32)  # many equal tile counts
    else:
        lens = rng.integers(1, 600, B).astype(np.int32)
    wl = W.make_case("bf16", 16, 4, 128, 16, lens, None, n_layers=1, layer_id=0, split_chunk=0,
                     max_splits=16, seed=W.SEED_BASE + 1300 + B)
    dw = DV.DeviceWorkload.upload(wl)
    dw.decode["out"].zero_()
    dw.run_decode()
    _sync()
    d = wl.decode
    sel = np.sort(rng.choice(B, 96, replace=False)).astype(np.int32)
    ref = oracle.decode(d.q, wl.pool.k_buffer[0], wl.pool.v_buffer[0], wl.pool.req_to_token,
                        d.req_pool_indices, d.seq_lens, sel=sel)
    got = DV.to_host(dw.decode["out"])
    assert maxerr(got[sel], ref[sel]) <= TOL["bf16"]
    # and no request was skipped: every output row was written (zeroed before the call)
    assert np.all(np.any(got.reshape(B, -1) != 0, axis=1))
    assert A.astr_device_error() == 0


@pytest.mark.parametrize("dtype,H,Hk,D", [
    ("bf16", 24, 4, 128),   # 32 head rows x 16 chunks = 512 chunks: four per thread of a 128-thread block
    ("bf16", 32, 4, 128),   # 640 chunks: more than four per thread, the one-thread-per-chunk kernel
    ("f32", 40, 8, 128),    # 896 chunks of 32 bytes
    ("bf16", 2, 1, 64),     # 32 chunks: one per thread, most threads idle
])
def test_rope_write_chunks_per_thread(dtype, H, Hk, D):
    """The rotate + write over every chunk-per-thread count the block-per-token launch takes,
    bit for bit against the oracle (q_out, and the whole layer of both caches)."""
    wl = W.make_case(dtype, H, Hk, D, 16, [5, 130, 257], [5, 130, 257], with_rope=True,
                     seed=W.SEED_BASE + 700 + H + Hk + D)
    dw = DV.DeviceWorkload.upload(wl)
    kl, vl = host_layer(wl, 1)
    dw.run_rope()
    _sync()
    check_rope(dw, "rope", kl, vl)
    check_cache_equal(dw, 1, kl, vl)
    assert A.astr_device_error() == 0
