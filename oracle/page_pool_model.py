"""Plain model of the paged pool's bookkeeping -- TEST INFRASTRUCTURE ONLY.

AstrAI inference guide, "KVCache System": PagePool over a bitmask page allocator with
ref-counts and LRU eviction, and RadixCache, which indexes complete token pages as
parent-linked edges and compares each page's exact token tuple while walking from the root
(an identical page is reused only under the same parent prefix); only fully materialised pages
enter it, a partial final page stays private to its request, and a later request resumes
prefill right after the longest complete-page hit. AstrAI internals, "Cache Architecture":
prefix sharing exists only when page_size > 1.

This model is written for checking by eye, not for speed: the cache is a flat list of entries
(parent entry, token tuple, page, last use), every lookup scans it, and there is no hashing.
The readings it takes where the pages are silent (the same ones the library takes):
  * a use (match or record through an entry) advances a logical clock by one per entry;
  * eviction removes the unreferenced leaf entry with the smallest (last use, page) first;
    a parent whose last child went becomes a leaf in its turn;
  * allocation hands out the lowest free page numbers, after evicting only as many entries as
    it needs; if even evicting everything evictable is not enough it fails, and the evictions
    made on the way stand;
  * recording a tuple that already has an edge under the same parent keeps the cached page;
  * rejected calls (a page not held, a page already cached elsewhere or given twice, a release
    of a reference not held) change nothing.
Only tests/ may import it; the library never does.
"""
from __future__ import annotations


class NoSpace(Exception):
    """alloc could not find enough free or evictable pages."""


class Invalid(Exception):
    """A call the pool rejects without changing anything."""


class _Entry:
    def __init__(self, parent, toks, page, last):
        self.parent = parent  # another _Entry, or None for the root's children
        self.toks = toks      # tuple of page_size token ids
        self.page = page
        self.last = last
        self.alive = True


class PagePoolModel:
    def __init__(self, n_pages: int, page_size: int):
        self.n_pages, self.ps = n_pages, page_size
        self.free = set(range(n_pages))
        self.ref = [0] * n_pages
        self.entries = []
        self.clock = 0

    # -- queries -------------------------------------------------------------------------
    def _live(self):
        return [e for e in self.entries if e.alive]

    def _find(self, parent, toks):
        for e in self._live():
            if e.parent is parent and e.toks == toks:
                return e
        return None

    def _has_child(self, e):
        return any(c.parent is e for c in self._live())

    def _evictable(self):
        return [e for e in self._live() if self.ref[e.page] == 0 and not self._has_child(e)]

    def cached(self, page):
        return any(e.page == page for e in self._live())

    def stats(self):
        return len(self.free), len(self._live()), len(self._evictable())

    # -- operations ----------------------------------------------------------------------
    def match(self, tokens, max_pages=None):
        if self.ps == 1:
            return []
        whole = len(tokens) // self.ps
        if max_pages is not None:
            whole = min(whole, max_pages)
        out, parent = [], None
        for i in range(whole):
            e = self._find(parent, tuple(tokens[i * self.ps:(i + 1) * self.ps]))
            if e is None:
                break
            self.ref[e.page] += 1
            self.clock += 1
            e.last = self.clock
            out.append(e.page)
            parent = e
        return out

    def alloc(self, n):
        while len(self.free) < n:
            cands = self._evictable()
            if not cands:
                break
            victim = min(cands, key=lambda e: (e.last, e.page))
            victim.alive = False
            self.free.add(victim.page)
        if len(self.free) < n:
            raise NoSpace()
        pages = sorted(self.free)[:n]
        for p in pages:
            self.free.remove(p)
            self.ref[p] = 1
        return pages

    def record(self, tokens, n_materialized, pages):
        if self.ps == 1:
            return
        whole = n_materialized // self.ps
        if whole > len(pages):
            raise Invalid("fewer pages than complete pages")
        for p in pages[:whole]:
            if not (0 <= p < self.n_pages) or self.ref[p] < 1:
                raise Invalid("a page the caller does not hold")
        # the part of the path that would be new must not reuse a cached page or repeat one
        parent = None
        for i in range(whole):
            e = self._find(parent, tuple(tokens[i * self.ps:(i + 1) * self.ps]))
            if e is None:
                rest = list(pages[i:whole])
                if any(self.cached(p) for p in rest) or len(set(rest)) != len(rest):
                    raise Invalid("a page cached elsewhere, or given twice")
                break
            parent = e
        parent = None
        for i in range(whole):
            toks = tuple(tokens[i * self.ps:(i + 1) * self.ps])
            e = self._find(parent, toks)
            if e is None:
                e = _Entry(parent, toks, pages[i], 0)
                self.entries.append(e)
            self.clock += 1
            e.last = self.clock
            parent = e

    def release(self, pages):
        want = {}
        for p in pages:
            if not (0 <= p < self.n_pages):
                raise Invalid("page out of range")
            want[p] = want.get(p, 0) + 1
            if want[p] > self.ref[p]:
                raise Invalid("a reference not held")
        for p in pages:
            self.ref[p] -= 1
            if self.ref[p] == 0 and not self.cached(p):
                self.free.add(p)
