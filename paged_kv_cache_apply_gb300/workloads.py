"""Seeded synthetic workloads for the paged KV-cache attention path.

This module is shared by the tests, ``bench.py`` and ``__graft_entry__.smoke()``. It holds only
random draws, index tables and memory layouts: no rotation, no attention and no softmax
arithmetic. Both the CUDA path and the CPU oracle consume what it builds.

Layouts follow the pages' ``KVCache`` dataclass (AstrAI inference guide, "KVCache System"):

* ``k_buffer`` / ``v_buffer``: ``[n_layers, size, n_kv_heads, head_dim]``, flat token-level slots.
* ``req_to_token``: ``[num_reqs, max_ctx_len]`` int32, request row and position -> physical slot.
* ``req_pool_indices``, ``seq_lens``: ``[batch]`` int32.
* ``kv_indptr`` / ``qo_indptr``: ``[batch + 1]`` int32 prefix sums of kv / q lengths.
* ``q_tile_to_batch`` / ``q_tile_to_index``: ``[num_q_tiles]`` int32, 128-row Q tiles.
* ``out_cache_loc``: ``[n_tokens]`` int32 write slots of this forward.

The ``freqs_cis`` table (AstrAI internals, "Rotary Position Embedding": ``[max_len, dim/2, 2]``
f32 ``[cos, sin]`` pairs) is precomputed here, outside the path, from the RoFormer frequencies
theta_i = base^(-2i/dim) cited by the AstrAI paper's model section (RoPE theta 10000).

bf16 values are stored as their raw uint16 bit patterns.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

SEED_BASE = 20260
Q_TILE_ROWS = 128

# ---------------------------------------------------------------------------------------------
# value draws
# ---------------------------------------------------------------------------------------------


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return uint16 bits.

    This is the input recipe's "N(0,1) cast to bf16". The draws contain no NaN.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def f32_from_bf16_bits(h: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_CHUNK = 1 << 21


def _fill_chunk(out: np.ndarray, seed: int, stream: int, ci: int, bf16: bool) -> None:
    lo = ci * _CHUNK
    hi = min(out.size, lo + _CHUNK)
    rng = np.random.default_rng([seed, stream, ci])
    x = rng.standard_normal(hi - lo, dtype=np.float32)
    out[lo:hi] = bf16_bits_from_f32(x) if bf16 else x


def normal_values(shape, dtype: str, seed: int, stream: int) -> np.ndarray:
    """N(0,1) draws of ``shape`` as float32 (``dtype='f32'``) or bf16 bits (``'bf16'``).

    Values depend only on (seed, stream, element index): chunk ``ci`` of 2^21 elements is
    drawn from PCG64 seeded with ``[seed, stream, ci]``, so the thread count never matters.
    """
    bf16 = dtype == "bf16"
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16 if bf16 else np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK
    if nchunks <= 1:
        if n:
            _fill_chunk(out, seed, stream, 0, bf16)
    else:
        workers = max(1, min(16, os.cpu_count() or 1, nchunks))
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(lambda ci: _fill_chunk(out, seed, stream, ci, bf16), range(nchunks)))
    return out.reshape(shape)


def rope_freqs_cis(max_len: int, dim: int, base: float = 10000.0) -> np.ndarray:
    """The precomputed RoPE table ``[max_len, dim/2, 2]`` f32 of ``[cos, sin]`` pairs.

    Entry ``[p, i]`` is (cos(p*theta_i), sin(p*theta_i)) with theta_i = base^(-2i/dim),
    evaluated in float64 and rounded to float32 once.
    """
    i = np.arange(dim // 2, dtype=np.float64)
    theta = base ** (-2.0 * i / dim)
    ang = np.arange(max_len, dtype=np.float64)[:, None] * theta[None, :]
    return np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)


# ---------------------------------------------------------------------------------------------
# host-side tables (what bind_tasks() would hand to the attention layers)
# ---------------------------------------------------------------------------------------------


def prefix_sum(lengths) -> np.ndarray:
    out = np.zeros(len(lengths) + 1, dtype=np.int64)
    out[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return out.astype(np.int32)


def q_tiles(q_lens, kv_lens=None, tile_rows: int = Q_TILE_ROWS):
    """``q_tile_to_batch`` / ``q_tile_to_index`` for ``tile_rows``-row Q tiles per request.

    Without ``kv_lens`` the tiles are listed request by request. With them, the tiles are
    listed by the number of 128-key KV tiles each one visits under the causal mask, cheapest
    first (ties in request order). The tensor-core prefill starts its blocks from the end of
    the list, so the costliest tiles are scheduled first and the SMs finish together. Any
    order gives the same result.
    """
    tb, ti, cost = [], [], []
    for b, ql in enumerate(q_lens):
        ql = int(ql)
        prefix = 0 if kv_lens is None else int(kv_lens[b]) - ql
        for t in range((ql + tile_rows - 1) // tile_rows):
            tb.append(b)
            ti.append(t)
            last_row = min(ql, (t + 1) * tile_rows)
            cost.append((prefix + last_row + 127) // 128)
    order = np.argsort(np.asarray(cost), kind="stable") if kv_lens is not None else np.arange(len(tb))
    return (np.asarray(tb, dtype=np.int32)[order], np.asarray(ti, dtype=np.int32)[order])


@dataclass
class PagedPool:
    """Host copy of KVStorage + ReqToTokenPool."""

    dtype: str  # 'f32' | 'bf16'
    n_layers: int
    size: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    k_buffer: np.ndarray  # [n_layers, size, Hk, D] float32 or uint16
    v_buffer: np.ndarray
    req_to_token: np.ndarray  # [num_reqs, max_ctx_len] int32

    @property
    def num_reqs(self) -> int:
        return int(self.req_to_token.shape[0])

    @property
    def max_ctx_len(self) -> int:
        return int(self.req_to_token.shape[1])


@dataclass
class RopeStep:
    """Inputs of one fused rotate + cache-write call over ``n_tokens`` packed tokens."""

    q: np.ndarray  # [T, H, D]
    k: np.ndarray  # [T, Hk, D]
    v: np.ndarray  # [T, Hk, D]
    position_ids: np.ndarray  # [T] int32
    out_cache_loc: np.ndarray  # [T] int32
    freqs_cis: np.ndarray  # [max_len, D/2, 2] f32
    layer_id: int = 0

    @property
    def n_tokens(self) -> int:
        return int(self.position_ids.shape[0])


@dataclass
class DecodeBatch:
    req_pool_indices: np.ndarray  # [B]
    seq_lens: np.ndarray  # [B]
    kv_indptr: np.ndarray  # [B+1]
    max_len: int
    q: Optional[np.ndarray]  # [B, H, D] or None when it is the rope step's q_out
    q_token_offset: int = 0  # first row of the rope step's q_out when q is None
    split_chunk: int = 0  # 0: the library picks the chunk
    max_splits: int = 16
    layer_id: int = 0

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])


@dataclass
class PrefillBatch:
    req_pool_indices: np.ndarray  # [B]
    qo_indptr: np.ndarray  # [B+1]
    kv_indptr: np.ndarray  # [B+1]
    q_tile_to_batch: np.ndarray
    q_tile_to_index: np.ndarray
    q: Optional[np.ndarray]  # [sum q, H, D] or None
    q_token_offset: int = 0
    q_tile_rows: int = Q_TILE_ROWS
    layer_id: int = 0

    @property
    def batch(self) -> int:
        return int(self.qo_indptr.shape[0] - 1)

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr[-1])


@dataclass
class Workload:
    name: str
    description: str
    n_heads: int
    pool: PagedPool
    rope: Optional[RopeStep] = None
    prefill: Optional[PrefillBatch] = None
    decode: Optional[DecodeBatch] = None
    # second phase (the tiny chain: prefill first, then one decode step per request)
    rope2: Optional[RopeStep] = None
    decode2: Optional[DecodeBatch] = None
    meta: dict = field(default_factory=dict)


# ---------------------------------------------------------------------------------------------
# slot placement
# ---------------------------------------------------------------------------------------------


def _paged_slots(rng, page_counts, page_size: int, n_pages_pool: int):
    """Place each request's pages at random, distinct pages of the pool (a shuffled free list).

    Returns one slot array per request covering ``page_counts[b] * page_size`` positions.
    """
    need = int(sum(page_counts))
    assert need <= n_pages_pool
    free = rng.permutation(n_pages_pool)[:need]
    out, at = [], 0
    for pc in page_counts:
        pages = free[at:at + pc].astype(np.int64)
        at += pc
        slots = (pages[:, None] * page_size + np.arange(page_size)[None, :]).reshape(-1)
        out.append(slots.astype(np.int32))
    return out


def _fill_rows(pool: PagedPool, slots: np.ndarray, seed: int, stream: int, layer: int = 0):
    """Write N(0,1) K and V rows into ``slots`` of one layer (the cached prefix)."""
    slots = np.sort(np.asarray(slots, dtype=np.int64))
    shape = (slots.size, pool.n_kv_heads, pool.head_dim)
    pool.k_buffer[layer, slots] = normal_values(shape, pool.dtype, seed, stream)
    pool.v_buffer[layer, slots] = normal_values(shape, pool.dtype, seed, stream + 1)


def _empty_pool(dtype, n_layers, size, hk, d, page_size, num_reqs, max_ctx) -> PagedPool:
    et = np.uint16 if dtype == "bf16" else np.float32
    return PagedPool(
        dtype=dtype, n_layers=n_layers, size=size, n_kv_heads=hk, head_dim=d,
        page_size=page_size,
        k_buffer=np.zeros((n_layers, size, hk, d), dtype=et),
        v_buffer=np.zeros((n_layers, size, hk, d), dtype=et),
        req_to_token=np.zeros((num_reqs, max_ctx), dtype=np.int32),
    )


# ---------------------------------------------------------------------------------------------
# the five configurations
# ---------------------------------------------------------------------------------------------


def tiny_chain(seed: int = SEED_BASE + 1) -> Workload:
    """Tiny chain, f32: prefill of {7, 13} tokens, then one decode step per request.

    1 layer, batch 2, 4 q heads, 2 KV heads, head_dim 64, contiguous pool with
    max_seq_len 64 (slot = req_idx * 64 + pos), freqs base 10000 and max_len 64.
    """
    H, Hk, D, msl = 4, 2, 64, 64
    lens = np.array([7, 13], dtype=np.int32)
    pool = _empty_pool("f32", 1, 2 * msl, Hk, D, 1, 2, msl)
    pool.req_to_token[:] = (np.arange(2)[:, None] * msl + np.arange(msl)[None, :]).astype(np.int32)
    freqs = rope_freqs_cis(64, D)
    T = int(lens.sum())
    pos = np.concatenate([np.arange(n) for n in lens]).astype(np.int32)
    req = np.concatenate([np.full(n, b) for b, n in enumerate(lens)])
    loc = pool.req_to_token[req, pos].astype(np.int32)
    rope = RopeStep(
        q=normal_values((T, H, D), "f32", seed, 1), k=normal_values((T, Hk, D), "f32", seed, 2),
        v=normal_values((T, Hk, D), "f32", seed, 3), position_ids=pos, out_cache_loc=loc,
        freqs_cis=freqs)
    tb, ti = q_tiles(lens)
    rpi = np.array([0, 1], dtype=np.int32)
    prefill = PrefillBatch(req_pool_indices=rpi, qo_indptr=prefix_sum(lens),
                           kv_indptr=prefix_sum(lens), q_tile_to_batch=tb, q_tile_to_index=ti,
                           q=None, q_token_offset=0)
    # decode step: the next token of each request sits at position len (seq_lens len + 1)
    pos2 = lens.copy()
    loc2 = pool.req_to_token[np.arange(2), pos2].astype(np.int32)
    rope2 = RopeStep(
        q=normal_values((2, H, D), "f32", seed, 4), k=normal_values((2, Hk, D), "f32", seed, 5),
        v=normal_values((2, Hk, D), "f32", seed, 6), position_ids=pos2, out_cache_loc=loc2,
        freqs_cis=freqs)
    sl2 = lens + 1
    decode2 = DecodeBatch(req_pool_indices=rpi, seq_lens=sl2, kv_indptr=prefix_sum(sl2),
                          max_len=int(sl2.max()), q=None, q_token_offset=0, split_chunk=4,
                          max_splits=4)
    return Workload("tiny_chain", "1 layer, B=2, H=4, Hk=2, D=64, f32, prefill {7,13} then decode",
                    H, pool, rope=rope, prefill=prefill, rope2=rope2, decode2=decode2,
                    meta={"seed": seed})


def decode_b64_page1(seed: int = SEED_BASE + 2, batch: int = 64, lmin: int = 512, lmax: int = 4096,
            pool_slots: int = 400_000) -> Workload:
    """Decode, bf16, H=16, Hk=4, D=128, page_size 1 over a 400k-slot pool."""
    H, Hk, D = 16, 4, 128
    rng = np.random.default_rng([seed, 0])
    lens = rng.integers(lmin, lmax + 1, size=batch).astype(np.int32)
    num_reqs = 2 * batch
    pool = _empty_pool("bf16", 1, pool_slots, Hk, D, 1, num_reqs, lmax)
    rpi = rng.permutation(num_reqs)[:batch].astype(np.int32)
    perm = rng.permutation(pool_slots)[: int(lens.sum())].astype(np.int32)
    at = 0
    for b in range(batch):
        pool.req_to_token[rpi[b], : lens[b]] = perm[at: at + lens[b]]
        at += lens[b]
    _fill_rows(pool, perm, seed, 10)
    dec = DecodeBatch(req_pool_indices=rpi, seq_lens=lens, kv_indptr=prefix_sum(lens),
                      max_len=int(lens.max()), q=normal_values((batch, H, D), "bf16", seed, 20),
                      split_chunk=0, max_splits=16)
    return Workload("decode_b64_page1", f"decode bf16 B={batch} L~U[{lmin},{lmax}] page 1", H, pool,
                    decode=dec, meta={"seed": seed})


def prefill_b8_varlen(seed: int = SEED_BASE + 3, batch: int = 8, qmin: int = 256, qmax: int = 2048,
            pmax: int = 1024, page: int = 16) -> Workload:
    """Varlen causal prefill, bf16, half the requests resumed after a page-aligned prefix."""
    H, Hk, D = 16, 4, 128
    rng = np.random.default_rng([seed, 0])
    qlens = rng.integers(qmin, qmax + 1, size=batch).astype(np.int32)
    prefix = np.zeros(batch, dtype=np.int32)
    resumed = rng.permutation(batch)[: batch // 2]
    prefix[resumed] = (rng.integers(0, pmax + 1, size=resumed.size) // page) * page
    kvl = prefix + qlens
    pages = [(int(k) + page - 1) // page for k in kvl]
    n_pages = int(np.ceil(1.5 * sum(pages)))
    max_ctx = int(((kvl.max() + page - 1) // page) * page)
    num_reqs = 2 * batch
    pool = _empty_pool("bf16", 1, n_pages * page, Hk, D, page, num_reqs, max_ctx)
    rpi = rng.permutation(num_reqs)[:batch].astype(np.int32)
    slots = _paged_slots(rng, pages, page, n_pages)
    used = []
    for b in range(batch):
        pool.req_to_token[rpi[b], : slots[b].size] = slots[b]
        used.append(slots[b][: kvl[b]])
    _fill_rows(pool, np.concatenate(used), seed, 10)
    tb, ti = q_tiles(qlens, kvl)
    pre = PrefillBatch(req_pool_indices=rpi, qo_indptr=prefix_sum(qlens),
                       kv_indptr=prefix_sum(kvl), q_tile_to_batch=tb, q_tile_to_index=ti,
                       q=normal_values((int(qlens.sum()), H, D), "bf16", seed, 20))
    return Workload("prefill_b8_varlen", f"prefill bf16 B={batch} Q~U[{qmin},{qmax}] resumed half",
                    H, pool, prefill=pre, meta={"seed": seed, "prefix": prefix.tolist()})


def long_decode_b4(seed: int = SEED_BASE + 4, batch: int = 4, lmin: int = 32768, lmax: int = 131072,
            pool_pages: int = 65536, page: int = 16, chunk: int = 4096) -> Workload:
    """Long-context split-K decode, fixed 4096-token chunks, page_size 16."""
    H, Hk, D = 16, 4, 128
    rng = np.random.default_rng([seed, 0])
    lens = rng.integers(lmin, lmax + 1, size=batch).astype(np.int32)
    pages = [(int(n) + page - 1) // page for n in lens]
    num_reqs = 2 * batch
    max_ctx = int(((lmax + page - 1) // page) * page)
    pool = _empty_pool("bf16", 1, pool_pages * page, Hk, D, page, num_reqs, max_ctx)
    rpi = rng.permutation(num_reqs)[:batch].astype(np.int32)
    slots = _paged_slots(rng, pages, page, pool_pages)
    used = []
    for b in range(batch):
        pool.req_to_token[rpi[b], : slots[b].size] = slots[b]
        used.append(slots[b][: lens[b]])
    _fill_rows(pool, np.concatenate(used), seed, 10)
    max_splits = (lmax + chunk - 1) // chunk
    dec = DecodeBatch(req_pool_indices=rpi, seq_lens=lens, kv_indptr=prefix_sum(lens),
                      max_len=int(lens.max()), q=normal_values((batch, H, D), "bf16", seed, 20),
                      split_chunk=chunk, max_splits=max_splits)
    return Workload("long_decode_b4", f"split-K decode bf16 B={batch} L~U[{lmin},{lmax}]", H,
                    pool, decode=dec, meta={"seed": seed})


def mixed_b256_p4x512(seed: int = SEED_BASE + 5, n_decode: int = 256, lmin: int = 128, lmax: int = 8192,
            n_prefill: int = 4, chunk_len: int = 512, page: int = 16,
            freqs_max_len: int = 8192) -> Workload:
    """Mixed continuous batch: 256 decode requests + 4 prefill chunks of 512 new tokens.

    One fused rotate + write over all new tokens (decode tokens first, then the prefill
    chunks), then prefill attention over the chunks, then decode attention. Each decode
    request has positions 0..L-2 already cached; its new token sits at position L-1.
    """
    H, Hk, D = 16, 4, 128
    rng = np.random.default_rng([seed, 0])
    dl = rng.integers(lmin, lmax + 1, size=n_decode).astype(np.int32)
    pl = np.full(n_prefill, chunk_len, dtype=np.int32)
    all_len = np.concatenate([dl, pl])
    pages = [(int(n) + page - 1) // page for n in all_len]
    n_pages = int(np.ceil(1.5 * sum(pages)))
    num_reqs = 2 * (n_decode + n_prefill)
    max_ctx = int(((max(lmax, chunk_len) + page - 1) // page) * page)
    pool = _empty_pool("bf16", 1, n_pages * page, Hk, D, page, num_reqs, max_ctx)
    rows = rng.permutation(num_reqs)[: n_decode + n_prefill].astype(np.int32)
    slots = _paged_slots(rng, pages, page, n_pages)
    cached = []
    for r in range(n_decode + n_prefill):
        pool.req_to_token[rows[r], : slots[r].size] = slots[r]
        if r < n_decode:
            cached.append(slots[r][: dl[r] - 1])
    _fill_rows(pool, np.concatenate(cached), seed, 10)
    T = n_decode + int(pl.sum())
    pos = np.concatenate([dl - 1] + [np.arange(n) for n in pl]).astype(np.int32)
    reqs = np.concatenate([np.arange(n_decode)] +
                          [np.full(n, n_decode + j) for j, n in enumerate(pl)])
    loc = pool.req_to_token[rows[reqs], pos].astype(np.int32)
    rope = RopeStep(q=normal_values((T, H, D), "bf16", seed, 20),
                    k=normal_values((T, Hk, D), "bf16", seed, 21),
                    v=normal_values((T, Hk, D), "bf16", seed, 22),
                    position_ids=pos, out_cache_loc=loc,
                    freqs_cis=rope_freqs_cis(freqs_max_len, D))
    dec = DecodeBatch(req_pool_indices=rows[:n_decode], seq_lens=dl, kv_indptr=prefix_sum(dl),
                      max_len=int(dl.max()), q=None, q_token_offset=0, split_chunk=0,
                      max_splits=16)
    tb, ti = q_tiles(pl, pl)
    pre = PrefillBatch(req_pool_indices=rows[n_decode:], qo_indptr=prefix_sum(pl),
                       kv_indptr=prefix_sum(pl), q_tile_to_batch=tb, q_tile_to_index=ti,
                       q=None, q_token_offset=n_decode)
    return Workload("mixed_b256_p4x512",
                    f"mixed bf16: {n_decode} decode L~U[{lmin},{lmax}] + {n_prefill}x{chunk_len} "
                    "prefill, fused rope+write", H, pool, rope=rope, prefill=pre, decode=dec,
                    meta={"seed": seed})


WORKLOADS = {f.__name__: f for f in (tiny_chain, decode_b64_page1, prefill_b8_varlen,
                                    long_decode_b4, mixed_b256_p4x512)}


def make(name: str, **kw) -> Workload:
    """The named workload (a key of WORKLOADS)."""
    return WORKLOADS[name](**kw)


def make_case(dtype: str, n_heads: int, n_kv_heads: int, head_dim: int, page: int, kv_lens,
              q_lens=None, n_layers: int = 2, layer_id: int = 1, seed: int = SEED_BASE + 100,
              split_chunk: int = 0, max_splits: int = 16, with_rope: bool = False,
              freqs_max_len: int = 0) -> Workload:
    """A small paged case for parametrised tests.

    ``q_lens is None`` builds a decode batch (one query per request at position L-1);
    otherwise a prefill batch with prefix P_b = kv_lens[b] - q_lens[b]. With ``with_rope`` the
    newest token of every request (decode) or the request's q_lens new tokens (prefill) are
    left empty in the cache and produced by a fused rotate + write step, whose q_out feeds the
    attention call. Every layer of the pool is filled, so a wrong layer offset is visible.
    """
    rng = np.random.default_rng([seed, 0])
    kv_lens = np.asarray(kv_lens, dtype=np.int32)
    B = kv_lens.size
    pages = [max(1, (int(n) + page - 1) // page) for n in kv_lens]
    n_pages = int(np.ceil(1.5 * sum(pages))) + 1
    max_ctx = int(max(pages) * page)
    num_reqs = 2 * B + 1
    pool = _empty_pool(dtype, n_layers, n_pages * page, n_kv_heads, head_dim, page, num_reqs,
                       max_ctx)
    rows = rng.permutation(num_reqs)[:B].astype(np.int32)
    slots = _paged_slots(rng, pages, page, n_pages)
    decode = q_lens is None
    qn = np.ones(B, np.int32) if decode else np.asarray(q_lens, dtype=np.int32)
    cached = []
    for b in range(B):
        pool.req_to_token[rows[b], : slots[b].size] = slots[b]
        upto = int(kv_lens[b] - qn[b]) if with_rope else int(kv_lens[b])
        cached.append(slots[b][:upto])
    for lyr in range(n_layers):
        _fill_rows(pool, np.concatenate(cached), seed, 10 + 2 * lyr, layer=lyr)
    H, D = n_heads, head_dim
    rope = None
    q_total = int(qn.sum())
    if with_rope:
        pos = np.concatenate([np.arange(kv_lens[b] - qn[b], kv_lens[b]) for b in range(B)])
        reqs = np.concatenate([np.full(qn[b], b) for b in range(B)])
        loc = pool.req_to_token[rows[reqs], pos].astype(np.int32)
        fm = freqs_max_len or int(kv_lens.max())
        rope = RopeStep(q=normal_values((q_total, H, D), dtype, seed, 30),
                        k=normal_values((q_total, n_kv_heads, D), dtype, seed, 31),
                        v=normal_values((q_total, n_kv_heads, D), dtype, seed, 32),
                        position_ids=pos.astype(np.int32), out_cache_loc=loc,
                        freqs_cis=rope_freqs_cis(fm, D), layer_id=layer_id)
    q = None if with_rope else normal_values((q_total, H, D), dtype, seed, 20)
    if decode:
        dec = DecodeBatch(req_pool_indices=rows, seq_lens=kv_lens, kv_indptr=prefix_sum(kv_lens),
                          max_len=int(kv_lens.max()), q=q, split_chunk=split_chunk,
                          max_splits=max_splits, layer_id=layer_id)
        return Workload("case_decode", "parametrised decode case", H, pool, rope=rope, decode=dec,
                        meta={"seed": seed})
    tb, ti = q_tiles(qn)
    pre = PrefillBatch(req_pool_indices=rows, qo_indptr=prefix_sum(qn), kv_indptr=prefix_sum(kv_lens),
                       q_tile_to_batch=tb, q_tile_to_index=ti, q=q, layer_id=layer_id)
    return Workload("case_prefill", "parametrised prefill case", H, pool, rope=rope, prefill=pre,
                    meta={"seed": seed})
