"""Pins of the paged-pool model (oracle.page_pool_model) against what the pages fix.

AstrAI inference guide, "KVCache System", and internals, "Cache Architecture": complete pages
only, matched along exact parent paths, ref-counted, evicted least recently used; partial
pages private; the final sampled token is not recorded.
"""
import itertools

import numpy as np
import pytest

from oracle.page_pool_model import Invalid, NoSpace, PagePoolModel


def _seq(rng, n, vocab=5):
    return [int(x) for x in rng.integers(0, vocab, n)]


def _brute_force_hit(recorded, query, ps):
    """Longest k such that some recorded sequence's first k complete pages equal the query's,
    and for each position the page that the earliest such sequence recorded."""
    best = []
    for k in range(1, len(query) // ps + 1):
        page_at = None
        for toks, n_mat, pages in recorded:
            if n_mat // ps >= k and list(toks[:k * ps]) == list(query[:k * ps]):
                page_at = pages[k - 1]
                break
        if page_at is None:
            break
        best.append(page_at)
    return best


@pytest.mark.parametrize("ps", [2, 4, 16])
def test_match_equals_brute_force_longest_complete_page_hit(ps):
    rng = np.random.default_rng(ps)
    m = PagePoolModel(4096, ps)
    recorded = []
    base = _seq(rng, 6 * ps, vocab=3)
    for r in range(25):
        # prefixes of one another with random divergence, so paths share and branch
        cut = int(rng.integers(0, 5 * ps))
        toks = base[:cut] + _seq(rng, int(rng.integers(1, 4 * ps)), vocab=3)
        hit = m.match(toks)
        new = m.alloc((len(toks) + ps - 1) // ps - len(hit))
        pages = hit + new
        n_mat = int(rng.integers(0, len(toks) + 1))
        m.record(toks, n_mat, pages)
        recorded.append((toks, n_mat, pages))
        m.release(pages)
    for q in range(40):
        cut = int(rng.integers(0, 6 * ps))
        query = base[:cut] + _seq(rng, int(rng.integers(0, 3 * ps)), vocab=3)
        got = m.match(query)
        assert got == _brute_force_hit(recorded, query, ps)
        m.release(got)


def test_identical_page_is_not_shared_under_another_parent():
    ps = 4
    m = PagePoolModel(64, ps)
    X, Y, Z = [1] * ps, [2] * ps, [3] * ps
    a = m.alloc(2)
    m.record(X + Y, 2 * ps, a)
    m.release(a)
    assert m.match(Z + Y) == []            # Y exists, but under X
    b = m.alloc(2)
    m.record(Z + Y, 2 * ps, b)
    m.release(b)
    got = m.match(Z + Y)
    assert got == list(b) and got[1] != a[1]
    m.release(got)


def test_partial_page_and_final_sampled_token_are_not_recorded():
    ps = 4
    m = PagePoolModel(16, ps)
    toks = list(range(2 * ps + 1))
    pages = m.alloc(3)
    m.record(toks, len(toks) - 1, pages)   # 2 * ps materialised: two complete pages
    assert m.stats()[1] == 2 and not m.cached(pages[2])
    m.release(pages)
    assert pages[2] in m.free
    m2 = PagePoolModel(16, ps)
    toks = list(range(2 * ps))
    pages = m2.alloc(2)
    m2.record(toks, len(toks) - 1, pages)  # the last token not decoded into KV: one page
    assert m2.stats()[1] == 1 and m2.cached(pages[0]) and not m2.cached(pages[1])


def test_lru_evicts_least_recently_used_leaf_first_and_leaves_before_parents():
    ps = 2
    m = PagePoolModel(5, ps)
    pa, pb, pc = m.alloc(1), m.alloc(1), m.alloc(1)
    m.record([1, 1], 2, pa)
    m.record([2, 2], 2, pb)
    m.record([3, 3], 2, pc)
    for p in (pa, pb, pc):
        m.release(p)
    m.release(m.match([1, 1]))             # A used most recently now
    chain = m.alloc(2)                     # the two free pages
    m.record([4, 4, 5, 5], 4, chain)
    m.release(chain)                       # chain: parent (4,4) with leaf (5,5)
    order = []
    for _ in range(5):
        before = {e.page for e in m._live()}
        got = m.alloc(1)
        after = {e.page for e in m._live()}
        order.append((before - after).pop())
        assert got == [order[-1]]
    # B, C (oldest uses), A, then the chain's leaf, then its parent
    assert order == [pb[0], pc[0], pa[0], chain[1], chain[0]]


def test_referenced_pages_are_never_evicted():
    ps = 2
    m = PagePoolModel(3, ps)
    p = m.alloc(3)
    m.record([1, 1, 2, 2, 3, 3], 6, p)
    m.release(p)
    held = m.match([1, 1, 2, 2])
    assert held == p[:2]
    assert m.alloc(1) == [p[2]]            # only the unheld leaf can go
    with pytest.raises(NoSpace):
        m.alloc(1)
    assert m.cached(p[0]) and m.cached(p[1])


def test_rejected_calls_change_nothing():
    ps = 2
    m = PagePoolModel(8, ps)
    p = m.alloc(2)
    snap = (set(m.free), list(m.ref), m.stats())
    with pytest.raises(Invalid):
        m.release([p[0], p[0]])            # one reference held, two released
    with pytest.raises(Invalid):
        m.record([1, 1, 2, 2], 4, [p[0], p[0]])
    with pytest.raises(Invalid):
        m.record([1, 1], 2, [7])           # not held
    assert (set(m.free), list(m.ref), m.stats()) == snap


def test_page_size_one_shares_nothing():
    m = PagePoolModel(8, 1)
    p = m.alloc(3)
    m.record([5, 6, 7], 3, p)
    m.release(p)
    assert m.match([5, 6, 7]) == [] and m.stats() == (8, 0, 0)


def test_conservation_over_random_operations():
    rng = np.random.default_rng(9)
    ps, n_pages = 3, 40
    m = PagePoolModel(n_pages, ps)
    live = []
    for step in range(400):
        op = rng.integers(0, 3)
        if op == 0 or not live:
            toks = _seq(rng, int(rng.integers(1, 5 * ps)), vocab=2)
            hit = m.match(toks)
            try:
                new = m.alloc((len(toks) + ps - 1) // ps - len(hit))
            except NoSpace:
                m.release(hit)
                continue
            live.append((toks, hit + new))
        elif op == 1:
            toks, pages = live.pop(int(rng.integers(0, len(live))))
            m.record(toks, int(rng.integers(0, len(toks) + 1)), pages)
            m.release(pages)
        else:
            toks, pages = live.pop(int(rng.integers(0, len(live))))
            m.release(pages)
        cached = {e.page for e in m._live()}
        assert len(cached) == len(m._live())           # a page holds at most one entry
        assert not (cached & m.free)
        held = {p for p in range(n_pages) if m.ref[p] > 0}
        assert not (held & m.free)
        assert len(m.free | cached | held) == n_pages  # every page is accounted for
        assert all(r >= 0 for r in m.ref)
