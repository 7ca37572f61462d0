"""The library's host page pool (astr_pool_*) against the plain model, operation by operation.

Index work: every returned page list, count and error must be identical.
"""
import numpy as np
import pytest

import paged_kv_cache_apply_gb300 as A
from oracle.page_pool_model import Invalid, NoSpace, PagePoolModel
from paged_kv_cache_apply_gb300 import build as B


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()


def _both(fn_lib, fn_model):
    """Run one operation on both; errors must agree (AstrError status vs model exception)."""
    try:
        got = fn_lib()
        lib_err = None
    except A.AstrError as e:
        got, lib_err = None, e.status
    try:
        want = fn_model()
        model_err = None
    except NoSpace:
        want, model_err = None, 6
    except Invalid:
        want, model_err = None, 1
    assert lib_err == model_err
    return got, want


@pytest.mark.parametrize("seed,ps,n_pages,vocab", [(0, 4, 48, 2), (1, 16, 64, 3), (2, 2, 20, 2),
                                                   (3, 1, 30, 2), (4, 8, 300, 4)])
def test_random_operation_sequences_agree(seed, ps, n_pages, vocab):
    rng = np.random.default_rng([seed, 77])
    pool, model = A.PagePool(n_pages, ps), PagePoolModel(n_pages, ps)
    base = [int(x) for x in rng.integers(0, vocab, 8 * ps)]
    live = []
    for step in range(600):
        op = int(rng.integers(0, 6))
        if op <= 1 or not live:  # a new request: match, then allocate the rest
            cut = int(rng.integers(0, 8 * ps))
            toks = base[:cut] + [int(x) for x in rng.integers(0, vocab, int(rng.integers(1, 4 * ps)))]
            cap = None if rng.random() < 0.7 else int(rng.integers(0, 4))
            got, want = _both(lambda: list(pool.match(toks, cap)), lambda: model.match(toks, cap))
            assert got == want
            need = (len(toks) + ps - 1) // ps - len(got)
            g2, w2 = _both(lambda: list(pool.alloc(need)), lambda: model.alloc(need))
            assert g2 == w2
            if g2 is None:
                pool.release(got)
                model.release(want)
                continue
            live.append((toks, got + g2))
        elif op == 2:  # completion: record the materialised tokens, then release
            toks, pages = live.pop(int(rng.integers(0, len(live))))
            n_mat = int(rng.integers(0, len(toks) + 1))
            _both(lambda: pool.record(toks, n_mat, pages), lambda: model.record(toks, n_mat, pages))
            _both(lambda: pool.release(pages), lambda: model.release(pages))
        elif op == 3:  # abandoned: release only
            toks, pages = live.pop(int(rng.integers(0, len(live))))
            _both(lambda: pool.release(pages), lambda: model.release(pages))
        elif op == 4 and live:  # rejected calls: a release not held, a record with a repeat
            toks, pages = live[int(rng.integers(0, len(live)))]
            bad = list(pages) + list(pages)
            _both(lambda: pool.release(bad), lambda: model.release(bad))
            if len(pages) >= 2:
                rep = [pages[0]] * len(pages)
                _both(lambda: pool.record(toks, len(toks), rep), lambda: model.record(toks, len(toks), rep))
        else:  # a big allocation that may need evictions
            n = int(rng.integers(0, n_pages // 2))
            g2, w2 = _both(lambda: list(pool.alloc(n)), lambda: model.alloc(n))
            assert g2 == w2
            if g2:
                _both(lambda: pool.release(g2), lambda: model.release(w2))
        assert pool.stats() == model.stats()
        for p in range(n_pages):
            r, c, h = pool.page_info(p)
            assert r == model.ref[p] and c == model.cached(p)
            assert (h != 0) == c
    for toks, pages in live:
        pool.release(pages)
        model.release(pages)
    assert pool.stats() == model.stats()


def test_entry_hash_depends_on_the_parent_path():
    ps = 4
    pool = A.PagePool(16, ps)
    X, Y, Z = [1] * ps, [2] * ps, [3] * ps
    a, b = pool.alloc(2), pool.alloc(2)
    pool.record(X + Y, 2 * ps, a)
    pool.record(Z + Y, 2 * ps, b)
    assert pool.page_info(int(a[1]))[2] != pool.page_info(int(b[1]))[2]
    pool.release(a)
    pool.release(b)


def test_argument_errors():
    with pytest.raises(A.AstrError):
        A.PagePool(0, 4)
    pool = A.PagePool(4, 4)
    with pytest.raises(A.AstrError) as e:
        pool.alloc(5)
    assert e.value.status == 6
    with pytest.raises(A.AstrError):
        pool.page_info(4)
    assert list(pool.slots([3, 1], 6)) == [12, 13, 14, 15, 4, 5]
    assert list(pool.slots([2], 0)) == []
    with pytest.raises(A.AstrError):
        pool.slots([3, 1], 9)  # two pages of 4 hold 8 tokens
    with pytest.raises(A.AstrError):
        pool.slots([3, 4], 6)  # page 4 is outside a 4-page pool


def test_concurrent_threads_keep_the_pool_consistent():
    # every call takes the pool's mutex: four threads running request lifecycles at once must
    # leave every page accounted for
    import threading
    ps, n_pages = 4, 256
    pool = A.PagePool(n_pages, ps)
    base = [7] * (8 * ps)
    errors = []

    def worker(seed):
        rng = np.random.default_rng(seed)
        try:
            for _ in range(300):
                toks = base[:int(rng.integers(0, 8 * ps))] + [int(x) for x in rng.integers(0, 3, 6)]
                hit = list(pool.match(toks[:-1]))
                try:
                    new = list(pool.alloc((len(toks) + ps - 1) // ps - len(hit)))
                except A.AstrError as e:
                    assert e.status == 6
                    pool.release(hit)
                    continue
                pages = hit + new
                pool.record(toks, len(toks) - 1, pages)
                pool.release(pages)
        except Exception as e:  # surfaced below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(s,)) for s in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[:3]
    free, cached, evictable = pool.stats()
    held = sum(pool.page_info(p)[0] > 0 for p in range(n_pages))
    assert held == 0 and free + cached == n_pages and evictable <= cached
