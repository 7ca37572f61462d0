"""The radix cache drives resumed prefill: a later request reuses an earlier one's complete
pages and prefills only its new rows.

AstrAI inference guide, "KVCache System": a later request resumes prefill immediately after
its longest complete-page hit; the prefill kernel then reads the shared prefix straight from
the cached pages. K and V are made a function of (token, position), as a model's are, so the
cached prefix of request A is exactly what request B would have computed, and B's resumed
prefill must equal the oracle's prefill of B from scratch.
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


def test_radix_hit_drives_a_resumed_prefill():
    import torch
    ps, H, Hk, D, V, P = 16, 16, 4, 128, 8, 1024
    seed = W.SEED_BASE + 1200
    Kt = W.normal_values((V, P, Hk, D), "bf16", seed, 1)  # K and V of token v at position p
    Vt = W.normal_values((V, P, Hk, D), "bf16", seed, 2)
    rng = np.random.default_rng(seed)
    n_pages = 160
    pool = A.PagePool(n_pages, ps)
    kb = np.zeros((1, n_pages * ps, Hk, D), np.uint16)
    vb = np.zeros_like(kb)

    def write(toks, slots, lo, hi):  # what a prefill of positions lo..hi-1 leaves in the cache
        j = np.arange(lo, hi)
        kb[0, slots[lo:hi]] = Kt[toks[lo:hi], j]
        vb[0, slots[lo:hi]] = Vt[toks[lo:hi], j]

    # request A: 700 prompt tokens prefilled, one token sampled (not yet in KV), then done
    tA = rng.integers(0, V, 700)
    pA = pool.alloc((700 + ps - 1) // ps)
    sA = pool.slots(pA, 700)
    write(tA, sA, 0, 700)
    pool.record(np.concatenate([tA, [3]]), 700, pA)
    pool.release(pA)
    assert pool.stats()[1] == 700 // ps  # complete pages only

    # B shares A's first 500 tokens; C shares nothing
    tB = np.concatenate([tA[:500], rng.integers(0, V, 300)])
    tC = rng.integers(0, V, 300)
    tC[0] = (tA[0] + 1) % V
    reqs = []
    for toks in (tB, tC):
        L = len(toks)
        hit = pool.match(toks[:L - 1])  # keep at least one row to compute
        pages = np.concatenate([hit, pool.alloc((L + ps - 1) // ps - len(hit))]).astype(np.int32)
        slots = pool.slots(pages, L)
        Pb = len(hit) * ps
        if Pb:  # the hit pages hold exactly this request's prefix
            j = np.arange(Pb)
            assert np.array_equal(kb[0, slots[:Pb]], Kt[toks[:Pb], j])
            assert np.array_equal(vb[0, slots[:Pb]], Vt[toks[:Pb], j])
        write(toks, slots, Pb, L)
        reqs.append((toks, pages, slots, Pb))
    assert reqs[0][3] == (500 // ps) * ps and reqs[1][3] == 0

    # one ragged, resumed prefill over both, reading the pool through req_to_token
    q_lens = np.array([len(t) - Pb for t, _, _, Pb in reqs], np.int32)
    kv_lens = np.array([len(t) for t, _, _, _ in reqs], np.int32)
    r2t = np.zeros((4, 1024), np.int32)
    for b, (toks, _, slots, _) in enumerate(reqs):
        r2t[b + 1, :len(toks)] = slots
    rpi = np.array([1, 2], np.int32)
    qo, kv, tb, ti = A.astr_prefill_tiles(q_lens, kv_lens)
    q = W.normal_values((int(q_lens.sum()), H, D), "bf16", seed, 3)
    dev = lambda a, dt: DV.to_torch(a, dt, "cuda")
    kbd, vbd = dev(kb, "bf16"), dev(vb, "bf16")
    kvc = A.KVCache(kbd, vbd, req_to_token=dev(r2t, "i32"), req_pool_indices=dev(rpi, "i32"),
                    qo_indptr=dev(qo, "i32"), kv_indptr=dev(kv, "i32"),
                    q_tile_to_batch=dev(tb, "i32"), q_tile_to_index=dev(ti, "i32"),
                    q_tile_rows=128, n_tokens=int(q_lens.sum()))
    qd = dev(q, "bf16")
    out = torch.empty_like(qd)
    A.astr_prefill_attention(kvc, 0, qd, out, H)
    torch.cuda.synchronize()
    assert A.astr_device_error() == 0
    got = DV.to_host(out)

    # the oracle: each request from scratch over contiguous K/V of its own tokens
    for b, (toks, _, _, Pb) in enumerate(reqs):
        L = len(toks)
        j = np.arange(L)
        kl, vl = np.ascontiguousarray(Kt[toks, j]), np.ascontiguousarray(Vt[toks, j])
        ref = oracle.prefill(q[qo[b]:qo[b + 1]], kl, vl, j[None, :].astype(np.int32),
                             np.zeros(1, np.int32), np.array([0, L - Pb], np.int32),
                             np.array([0, L], np.int32))
        err = np.max(np.abs(W.f32_from_bf16_bits(got[qo[b]:qo[b + 1]]).astype(np.float64) - ref))
        assert err <= 2e-2, (b, err)

    # completion of B records its new complete pages under A's prefix; C's stand alone
    cached_before = pool.stats()[1]
    for toks, pages, _, _ in reqs:
        pool.record(toks, len(toks), pages)
        pool.release(pages)
    assert pool.stats()[1] == cached_before + (800 - 496) // ps + 300 // ps
