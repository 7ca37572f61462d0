"""The seeded workload builders produce the tables the pages describe (host only)."""
import numpy as np
import pytest

from paged_kv_cache_apply_gb300 import workloads as W


def test_normal_values_deterministic_and_chunk_independent():
    a = W.normal_values((3, 1000), "f32", 5, 1)
    b = W.normal_values((3, 1000), "f32", 5, 1)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, W.normal_values((3, 1000), "f32", 5, 2))
    h = W.normal_values((5000,), "bf16", 5, 1)
    assert h.dtype == np.uint16
    assert np.array_equal(h, W.bf16_bits_from_f32(W.normal_values((5000,), "f32", 5, 1)))


def test_bf16_rounding_ties_to_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9], np.float32)
    got = W.f32_from_bf16_bits(W.bf16_bits_from_f32(x))
    assert np.array_equal(got, np.array([1.0, 1.0, 1.0 + 2 ** -6, -2.5, 1.0], np.float32))


def test_tiny_config_tables():
    wl = W.tiny_chain()
    assert list(wl.rope.out_cache_loc[:7]) == list(range(7))
    assert list(wl.rope.out_cache_loc[7:]) == list(range(64, 77))
    assert list(wl.rope2.out_cache_loc) == [7, 77]
    assert list(wl.rope2.position_ids) == [7, 13]
    assert list(wl.decode2.seq_lens) == [8, 14] and wl.decode2.max_len == 14
    assert list(wl.prefill.qo_indptr) == [0, 7, 20]
    assert list(wl.prefill.q_tile_to_batch) == [0, 1] and list(wl.prefill.q_tile_to_index) == [0, 0]


def _check_paged(pool, rpi, lens, page):
    slots = []
    for b, r in enumerate(rpi):
        s = pool.req_to_token[r, : lens[b]]
        assert np.all((s >= 0) & (s < pool.size))
        if page > 1:
            n = (lens[b] // page) * page
            blk = s[:n].reshape(-1, page)
            assert np.all(blk[:, 0] % page == 0) and np.all(np.diff(blk, axis=1) == 1)
        slots.append(s)
    allslots = np.concatenate(slots)
    assert np.unique(allslots).size == allslots.size


def test_decode_config_small():
    wl = W.decode_b64_page1(batch=6, lmin=5, lmax=40, pool_slots=500)
    d = wl.decode
    assert np.array_equal(d.kv_indptr, W.prefix_sum(d.seq_lens))
    assert d.max_len == d.seq_lens.max()
    _check_paged(wl.pool, d.req_pool_indices, d.seq_lens, 1)
    assert np.unique(d.req_pool_indices).size == d.batch


def test_prefill_config_small():
    wl = W.prefill_b8_varlen(batch=6, qmin=10, qmax=300, pmax=64)
    p = wl.prefill
    q = np.diff(p.qo_indptr)
    k = np.diff(p.kv_indptr)
    pre = k - q
    assert np.all(pre >= 0) and np.all(pre % 16 == 0) and np.sum(pre > 0) <= 3
    _check_paged(wl.pool, p.req_pool_indices, k, 16)
    tiles = sorted(zip(p.q_tile_to_batch, p.q_tile_to_index))
    assert tiles == sorted((b, t) for b in range(6) for t in range((q[b] + 127) // 128))


def test_long_decode_config_small():
    wl = W.long_decode_b4(batch=3, lmin=100, lmax=400, pool_pages=100, chunk=64)
    d = wl.decode
    assert d.split_chunk == 64 and d.max_splits == (400 + 63) // 64
    _check_paged(wl.pool, d.req_pool_indices, d.seq_lens, 16)


def test_mixed_config_small():
    wl = W.mixed_b256_p4x512(n_decode=5, lmin=3, lmax=50, n_prefill=2, chunk_len=20, freqs_max_len=64)
    r, d, p = wl.rope, wl.decode, wl.prefill
    assert r.n_tokens == 5 + 40
    assert np.array_equal(r.position_ids[:5], d.seq_lens - 1)
    assert list(r.position_ids[5:25]) == list(range(20))
    # the new decode token goes to the slot of its position in the request's page table
    for b in range(5):
        assert r.out_cache_loc[b] == wl.pool.req_to_token[d.req_pool_indices[b], d.seq_lens[b] - 1]
    assert np.unique(r.out_cache_loc).size == r.n_tokens
    assert p.q_token_offset == 5 and list(p.qo_indptr) == [0, 20, 40]
    # cached prefix rows hold data, the new-token slots start empty
    k = wl.pool.k_buffer[0]
    assert np.all(k[r.out_cache_loc] == 0)
    assert np.any(k[wl.pool.req_to_token[d.req_pool_indices[0], 0]] != 0) or d.seq_lens[0] == 1


@pytest.mark.parametrize("name", ["tiny_chain"])
def test_freqs_table_shape(name):
    wl = W.make(name)
    assert wl.rope.freqs_cis.shape == (64, 32, 2)
