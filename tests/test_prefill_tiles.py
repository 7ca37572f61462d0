"""Host-side prefill metadata (astr_prefill_tiles): indptrs and cost-ordered Q-tile maps."""
import ctypes as C

import numpy as np
import pytest

import paged_kv_cache_apply_gb300 as A
from paged_kv_cache_apply_gb300 import build as B
from paged_kv_cache_apply_gb300 import workloads as W


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()


def _cost(q, k, b, t, rows=128):
    return (k[b] - q[b] + min(q[b], (t + 1) * rows) + 127) // 128


@pytest.mark.parametrize("seed", range(6))
def test_matches_the_input_builder_and_covers_every_row_once(seed):
    rng = np.random.default_rng([seed, 11])
    B_ = int(rng.integers(1, 12))
    q = rng.integers(0, 2000, size=B_).astype(np.int32)
    k = (q + rng.integers(0, 1500, size=B_)).astype(np.int32)
    qo, kv, tb, ti = A.astr_prefill_tiles(q, k)
    assert np.array_equal(qo, W.prefix_sum(q)) and np.array_equal(kv, W.prefix_sum(k))
    tb2, ti2 = W.q_tiles(q, k)
    assert np.array_equal(tb, tb2) and np.array_equal(ti, ti2)
    # every row of every request exactly once
    covered = np.zeros(int(q.sum()), dtype=np.int32)
    for b, t in zip(tb, ti):
        lo, hi = qo[b] + 128 * t, min(qo[b] + 128 * (t + 1), qo[b + 1])
        assert lo < hi
        covered[lo:hi] += 1
    assert np.all(covered == 1)
    # cheapest first; equal costs in request order
    c = [_cost(q, k, b, t) for b, t in zip(tb, ti)]
    assert all(x <= y for x, y in zip(c, c[1:]))
    for i in range(len(c) - 1):
        if c[i] == c[i + 1]:
            assert (tb[i], ti[i]) < (tb[i + 1], ti[i + 1])


def test_errors_and_empty_batch():
    L = A.lib()
    P = C.POINTER(C.c_int32)
    p = lambda a: a.ctypes.data_as(P)
    n = C.c_int32(-1)
    qo, kv = np.full(3, 7, np.int32), np.full(3, 7, np.int32)
    assert L.astr_prefill_tiles(None, None, 0, 128, p(qo), p(kv), None, None, 0, C.byref(n)) == 0
    assert n.value == 0 and qo[0] == 0 and kv[0] == 0
    assert L.astr_prefill_tiles(None, None, 0, 128, None, p(kv), None, None, 0, C.byref(n)) == 1
    q = np.array([10, 300], np.int32)
    k = np.array([5, 300], np.int32)  # kv_len < q_len
    tb, ti = np.zeros(8, np.int32), np.zeros(8, np.int32)
    assert L.astr_prefill_tiles(p(q), p(k), 2, 128, p(qo), p(kv), p(tb), p(ti), 8, C.byref(n)) == 1
    k = np.array([10, 300], np.int32)
    assert L.astr_prefill_tiles(p(q), p(k), 2, 128, p(qo), p(kv), p(tb), p(ti), 3, C.byref(n)) == 1
    assert n.value == 4 and b"max_tiles" in L.astr_last_error()
    assert L.astr_prefill_tiles(p(q), p(k), 2, 128, p(qo), p(kv), p(tb), p(ti), 4, C.byref(n)) == 0
