"""Python binding of libastr.so: the GB300 paged KV-cache attention path.

Argument marshalling only: every step of the path runs in the library's CUDA kernels. The
names and arguments are those of include/astr.h; torch tensors are passed by data_ptr() after
device, dtype and contiguity checks, and the stream defaults to torch's current stream. A
missing library raises at import of the first call -- there is no other implementation.
"""
from __future__ import annotations

import ctypes as C
import os
import threading
from dataclasses import dataclass
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libastr.so")

ASTR_F32, ASTR_BF16 = 0, 1
STATUS = {0: "ASTR_OK", 1: "ASTR_ERR_INVALID", 2: "ASTR_ERR_UNSUPPORTED", 3: "ASTR_ERR_CUDA",
          4: "ASTR_ERR_INDEX", 5: "ASTR_ERR_TIMEOUT", 6: "ASTR_ERR_NO_SPACE"}
DEVERR_SLOT, DEVERR_POS, DEVERR_ROW, DEVERR_LEN, DEVERR_TIMEOUT, DEVERR_META = 1, 2, 4, 8, 16, 32


class AstrError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class astr_kv_cache(C.Structure):
    """ctypes mirror of ``astr_kv_cache`` (field order and types as in include/astr.h)."""

    _fields_ = [
        ("k_buffer", C.c_void_p), ("v_buffer", C.c_void_p),
        ("n_layers", C.c_int32), ("n_kv_heads", C.c_int32), ("size", C.c_int64),
        ("head_dim", C.c_int32), ("dtype", C.c_int32),
        ("req_to_token", C.c_void_p), ("num_reqs", C.c_int32), ("max_ctx_len", C.c_int32),
        ("req_pool_indices", C.c_void_p), ("seq_lens", C.c_void_p),
        ("batch", C.c_int32), ("max_len", C.c_int32),
        ("out_cache_loc", C.c_void_p), ("n_tokens", C.c_int64),
        ("kv_indptr", C.c_void_p), ("qo_indptr", C.c_void_p),
        ("q_tile_to_batch", C.c_void_p), ("q_tile_to_index", C.c_void_p),
        ("num_q_tiles", C.c_int32), ("q_tile_rows", C.c_int32),
        ("decode_o_part", C.c_void_p), ("decode_ml_part", C.c_void_p),
        ("max_splits", C.c_int32), ("split_chunk", C.c_int32),
        ("decode_out", C.c_void_p),
    ]


_lock = threading.Lock()
_lib = None


def lib():
    """Load libastr.so (built by ``paged_kv_cache_apply_gb300.build``); raise if it is absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m paged_kv_cache_apply_gb300.build` (nvcc, sm_103a)")
            L = C.CDLL(LIB_PATH)
            P, I32, I64 = C.c_void_p, C.c_int32, C.c_int64
            KV = C.POINTER(astr_kv_cache)
            L.astr_rope_kv_write.argtypes = [KV, I32, P, P, P, P, I32, P, I32, P, P]
            L.astr_decode_attention.argtypes = [KV, I32, P, I32, P]
            L.astr_decode_attention_noalloc.argtypes = [KV, I32, P, I32, P]
            L.astr_decode_attention_rope.argtypes = [KV, I32, P, P, P, I32, P, I32, P, P]
            PI = C.POINTER(I32)
            L.astr_prefill_tiles.argtypes = [PI, PI, I32, I32, PI, PI, PI, PI, I32, PI]
            L.astr_bind_tasks.argtypes = [P, P, I32, I32, P, P, P, P, I32, P]
            PP = C.c_void_p
            L.astr_pool_create.argtypes = [I32, I32, C.POINTER(PP)]
            L.astr_pool_destroy.argtypes = [PP]
            L.astr_pool_match.argtypes = [PP, PI, C.c_int64, I32, PI, PI]
            L.astr_pool_alloc.argtypes = [PP, I32, PI]
            L.astr_pool_record.argtypes = [PP, PI, C.c_int64, PI, I32]
            L.astr_pool_release.argtypes = [PP, PI, I32]
            L.astr_pool_stats.argtypes = [PP, PI, PI, PI]
            L.astr_pool_page_info.argtypes = [PP, I32, PI, PI, C.POINTER(C.c_uint64)]
            L.astr_pool_slots.argtypes = [PP, PI, I32, C.c_int64, PI]
            L.astr_rope_apply.argtypes = [P, P, P, P, C.c_int64, I32, I32, I32, I32, P, I32, P, P]
            L.astr_rope_backward.argtypes = [P, P, P, P, C.c_int64, I32, I32, I32, I32, P, I32, P, P]
            L.astr_decode_plan.argtypes = [KV, I32, C.POINTER(I32), C.POINTER(I32)]
            L.astr_prefill_attention.argtypes = [KV, I32, P, P, I32, P]
            L.astr_last_error.restype = C.c_char_p
            L.astr_set_checked.argtypes = [I32]
            L.astr_set_wait_timeout_ns.argtypes = [I64]
            L.astr_device_error.argtypes = [P, C.POINTER(C.c_uint32)]
            L.astr_selftest_wait_timeout.argtypes = [P, I64]
            L.astr_version.restype = I32
            L.astr_kv_cache_bytes.restype = I32
            for name in ["astr_rope_kv_write", "astr_decode_attention", "astr_decode_plan",
                         "astr_decode_attention_noalloc", "astr_decode_attention_rope",
                         "astr_prefill_tiles", "astr_bind_tasks", "astr_rope_apply",
                         "astr_rope_backward", "astr_pool_create", "astr_pool_destroy",
                         "astr_pool_match", "astr_pool_alloc", "astr_pool_record",
                         "astr_pool_release", "astr_pool_stats", "astr_pool_page_info", "astr_pool_slots",
                         "astr_prefill_attention", "astr_set_checked", "astr_set_wait_timeout_ns",
                         "astr_device_error", "astr_selftest_wait_timeout"]:
                getattr(L, name).restype = I32
            _lib = L
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise AstrError(status, lib().astr_last_error().decode())


def _ptr(t) -> Optional[int]:
    """Device pointer of a torch tensor (contiguous), an int, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors passed to libastr must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return ASTR_F32
    if t.dtype == torch.bfloat16:
        return ASTR_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: libastr takes float32 or bfloat16")


@dataclass
class KVCache:
    """The pages' ``KVCache`` dataclass over torch device tensors (a plain data record without methods).

    ``k_buffer``/``v_buffer``: [n_layers, size, n_kv_heads, head_dim]; every index tensor is
    int32. ``max_len`` is a host int. Unused fields stay None.
    """

    k_buffer: object
    v_buffer: object
    req_to_token: object = None
    req_pool_indices: object = None
    seq_lens: object = None
    max_len: int = 0
    out_cache_loc: object = None
    kv_indptr: object = None
    qo_indptr: object = None
    q_tile_to_batch: object = None
    q_tile_to_index: object = None
    q_tile_rows: int = 128
    decode_o_part: object = None
    decode_ml_part: object = None
    split_chunk: int = 0
    decode_out: object = None
    batch: Optional[int] = None
    n_tokens: Optional[int] = None

    def as_c(self) -> astr_kv_cache:
        import torch
        kb = self.k_buffer
        if kb.dim() != 4 or self.v_buffer.shape != kb.shape or self.v_buffer.dtype != kb.dtype:
            raise ValueError("k_buffer / v_buffer must both be [n_layers, size, n_kv_heads, head_dim]")
        for name in ["req_to_token", "req_pool_indices", "seq_lens", "out_cache_loc", "kv_indptr",
                     "qo_indptr", "q_tile_to_batch", "q_tile_to_index"]:
            t = getattr(self, name)
            if t is not None and t.dtype != torch.int32:
                raise TypeError(f"{name} must be int32")
        c = astr_kv_cache()
        c.k_buffer, c.v_buffer = _ptr(kb), _ptr(self.v_buffer)
        c.n_layers, c.size, c.n_kv_heads, c.head_dim = kb.shape[0], kb.shape[1], kb.shape[2], kb.shape[3]
        c.dtype = _dtype_code(kb)
        if self.req_to_token is not None:
            c.req_to_token = _ptr(self.req_to_token)
            c.num_reqs, c.max_ctx_len = self.req_to_token.shape
        c.req_pool_indices = _ptr(self.req_pool_indices)
        c.seq_lens = _ptr(self.seq_lens)
        if self.batch is not None:
            c.batch = self.batch
        elif self.req_pool_indices is not None:
            c.batch = self.req_pool_indices.shape[0]
        c.max_len = int(self.max_len)
        c.out_cache_loc = _ptr(self.out_cache_loc)
        if self.n_tokens is not None:
            c.n_tokens = int(self.n_tokens)
        elif self.out_cache_loc is not None:
            c.n_tokens = self.out_cache_loc.shape[0]
        c.kv_indptr = _ptr(self.kv_indptr)
        c.qo_indptr = _ptr(self.qo_indptr)
        c.q_tile_to_batch = _ptr(self.q_tile_to_batch)
        c.q_tile_to_index = _ptr(self.q_tile_to_index)
        if self.q_tile_to_batch is not None:
            c.num_q_tiles = self.q_tile_to_batch.shape[0]
        c.q_tile_rows = int(self.q_tile_rows)
        c.decode_o_part = _ptr(self.decode_o_part)
        c.decode_ml_part = _ptr(self.decode_ml_part)
        if self.decode_o_part is not None:
            c.max_splits = self.decode_o_part.shape[2]
        c.split_chunk = int(self.split_chunk)
        c.decode_out = _ptr(self.decode_out)
        return c


def _kv(kv):
    return kv if isinstance(kv, astr_kv_cache) else kv.as_c()


def astr_rope_kv_write(kv, layer_id, q, q_out, k, v, n_heads, freqs_cis, freqs_max_len,
                       position_ids, stream=None) -> None:
    c = _kv(kv)
    _check(lib().astr_rope_kv_write(C.byref(c), int(layer_id), _ptr(q), _ptr(q_out), _ptr(k),
                                    _ptr(v), int(n_heads), _ptr(freqs_cis), int(freqs_max_len),
                                    _ptr(position_ids), _stream(stream)))


def astr_decode_attention(kv, layer_id, q, n_heads, stream=None) -> None:
    c = _kv(kv)
    _check(lib().astr_decode_attention(C.byref(c), int(layer_id), _ptr(q), int(n_heads),
                                       _stream(stream)))


def astr_decode_attention_rope(kv, layer_id: int, q, k_new, v_new, n_heads: int, freqs_cis,
                               freqs_max_len: int, position_ids, stream=None) -> None:
    """Decode with RoPE and the new token's K/V write folded in (q, k_new not rotated yet)."""
    c = _kv(kv)
    _check(lib().astr_decode_attention_rope(C.byref(c), int(layer_id), _ptr(q), _ptr(k_new),
                                            _ptr(v_new), int(n_heads), _ptr(freqs_cis),
                                            int(freqs_max_len), _ptr(position_ids),
                                            _stream(stream)))


def _rope_apply_args(q, q_out, k, k_out, freqs_cis, position_ids):
    import torch
    if q.dim() != 3 or q_out.shape != q.shape or q_out.dtype != q.dtype:
        raise ValueError("q / q_out must both be [n_tokens, n_heads, head_dim] of one dtype")
    T, H, D = q.shape
    Hk = 0
    if k is not None:
        if k.dim() != 3 or k.shape[0] != T or k.shape[2] != D or k_out is None or \
                k_out.shape != k.shape or k.dtype != q.dtype or k_out.dtype != q.dtype:
            raise ValueError("k / k_out must both be [n_tokens, n_kv_heads, head_dim] like q")
        Hk = k.shape[1]
    if freqs_cis.dtype != torch.float32 or position_ids.dtype != torch.int32:
        raise TypeError("freqs_cis must be float32 and position_ids int32")
    return (_ptr(q), _ptr(q_out), _ptr(k), _ptr(k_out), int(T), int(H), int(Hk), int(D),
            _dtype_code(q), _ptr(freqs_cis), int(freqs_cis.shape[0]), _ptr(position_ids))


def astr_rope_apply(q, q_out, k, k_out, freqs_cis, position_ids, stream=None) -> None:
    """Training-path RoPE, no cache write: q_out = R q, k_out = R k (k may be None)."""
    _check(lib().astr_rope_apply(*_rope_apply_args(q, q_out, k, k_out, freqs_cis, position_ids),
                                 _stream(stream)))


def astr_rope_backward(grad_q_out, grad_q, grad_k_out, grad_k, freqs_cis, position_ids,
                       stream=None) -> None:
    """The backward of astr_rope_apply: grad_q = R^T grad_q_out, grad_k = R^T grad_k_out."""
    _check(lib().astr_rope_backward(*_rope_apply_args(grad_q_out, grad_q, grad_k_out, grad_k,
                                                      freqs_cis, position_ids), _stream(stream)))


def astr_decode_attention_noalloc(kv, layer_id, q, n_heads, stream=None) -> None:
    """Decode without caller scratch: for callers that cannot allocate device memory."""
    c = _kv(kv)
    _check(lib().astr_decode_attention_noalloc(C.byref(c), int(layer_id), _ptr(q), int(n_heads),
                                               _stream(stream)))


def astr_prefill_tiles(q_lens, kv_lens, q_tile_rows: int = 128):
    """Host-side prefill metadata: (qo_indptr, kv_indptr, q_tile_to_batch, q_tile_to_index) as
    int32 numpy arrays, the tiles cheapest first."""
    import numpy as np
    ql = np.ascontiguousarray(q_lens, dtype=np.int32)
    kl = np.ascontiguousarray(kv_lens, dtype=np.int32)
    B = int(ql.size)
    P = C.POINTER(C.c_int32)
    ptr = lambda a: a.ctypes.data_as(P)
    n = C.c_int32(0)
    qo, kv = np.zeros(B + 1, np.int32), np.zeros(B + 1, np.int32)
    st = lib().astr_prefill_tiles(ptr(ql), ptr(kl), B, int(q_tile_rows), ptr(qo), ptr(kv), None, None,
                                  0, C.byref(n))
    tb, ti = np.zeros(max(n.value, 1), np.int32), np.zeros(max(n.value, 1), np.int32)
    if st != 0 and n.value == 0:
        _check(st)
    _check(lib().astr_prefill_tiles(ptr(ql), ptr(kl), B, int(q_tile_rows), ptr(qo), ptr(kv), ptr(tb),
                                    ptr(ti), n.value, C.byref(n)))
    return qo, kv, tb[:n.value], ti[:n.value]


def astr_bind_tasks(q_lens, kv_lens, qo_indptr, kv_indptr, q_tile_to_batch=None,
                    q_tile_to_index=None, q_tile_rows: int = 128, stream=None) -> None:
    """Device-side per-step metadata: fills qo_indptr / kv_indptr and the tile maps (their
    length is the capacity; unused entries become -1). q_lens None: a decode batch."""
    import torch
    for t in (q_lens, kv_lens, qo_indptr, kv_indptr, q_tile_to_batch, q_tile_to_index):
        if t is not None and t.dtype != torch.int32:
            raise TypeError("astr_bind_tasks takes int32 tensors")
    B = int(kv_lens.shape[0])
    max_tiles = 0 if q_tile_to_batch is None else int(q_tile_to_batch.shape[0])
    if q_tile_to_index is not None and int(q_tile_to_index.shape[0]) != max_tiles:
        raise ValueError("q_tile_to_batch and q_tile_to_index differ in length")
    _check(lib().astr_bind_tasks(_ptr(q_lens), _ptr(kv_lens), B, int(q_tile_rows), _ptr(qo_indptr),
                                 _ptr(kv_indptr), _ptr(q_tile_to_batch), _ptr(q_tile_to_index),
                                 max_tiles, _stream(stream)))


class PagePool:
    """The host page pool of libastr: a bitmask page allocator with reference counts and LRU
    eviction, and a radix cache of complete token pages (astr_pool_* in include/astr.h).
    Arguments and results are int32 numpy arrays / Python ints; page p owns the slots
    [p * page_size, (p + 1) * page_size)."""

    def __init__(self, n_pages: int, page_size: int):
        self.page_size = int(page_size)
        h = C.c_void_p()
        _check(lib().astr_pool_create(int(n_pages), self.page_size, C.byref(h)))
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            lib().astr_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _i32(a):
        import numpy as np
        return np.ascontiguousarray(a, dtype=np.int32)

    @staticmethod
    def _p(a):
        return a.ctypes.data_as(C.POINTER(C.c_int32))

    def match(self, tokens, max_pages=None):
        """Pages of the longest cached complete-page prefix of tokens (each now referenced)."""
        import numpy as np
        t = self._i32(tokens)
        mp = t.size // self.page_size if max_pages is None else int(max_pages)
        out = np.zeros(max(mp, 1), np.int32)
        n = C.c_int32(0)
        _check(lib().astr_pool_match(self._h, self._p(t), t.size, mp, self._p(out), C.byref(n)))
        return out[:n.value].copy()

    def alloc(self, n: int):
        import numpy as np
        out = np.zeros(max(int(n), 1), np.int32)
        _check(lib().astr_pool_alloc(self._h, int(n), self._p(out)))
        return out[:int(n)].copy()

    def record(self, tokens, n_materialized: int, pages):
        t, p = self._i32(tokens), self._i32(pages)
        _check(lib().astr_pool_record(self._h, self._p(t), int(n_materialized), self._p(p), p.size))

    def release(self, pages):
        p = self._i32(pages)
        _check(lib().astr_pool_release(self._h, self._p(p), p.size))

    def stats(self):
        """(free pages, cached pages, evictable pages)."""
        a, b, c = C.c_int32(), C.c_int32(), C.c_int32()
        _check(lib().astr_pool_stats(self._h, C.byref(a), C.byref(b), C.byref(c)))
        return a.value, b.value, c.value

    def page_info(self, page: int):
        """(references, cached, entry hash) of one page."""
        r, c, h = C.c_int32(), C.c_int32(), C.c_uint64()
        _check(lib().astr_pool_page_info(self._h, int(page), C.byref(r), C.byref(c), C.byref(h)))
        return r.value, bool(c.value), h.value

    def slots(self, pages, n_tokens: int):
        """The req_to_token row entries of positions 0..n_tokens-1 held in `pages`."""
        import numpy as np
        p = self._i32(pages)
        out = np.zeros(max(int(n_tokens), 1), np.int32)
        _check(lib().astr_pool_slots(self._h, self._p(p), p.size, int(n_tokens), self._p(out)))
        return out[:int(n_tokens)].copy()


def astr_decode_plan(kv, n_heads):
    c = _kv(kv)
    chunk, n = C.c_int32(0), C.c_int32(0)
    _check(lib().astr_decode_plan(C.byref(c), int(n_heads), C.byref(chunk), C.byref(n)))
    return chunk.value, n.value


def astr_prefill_attention(kv, layer_id, q, out, n_heads, stream=None) -> None:
    c = _kv(kv)
    _check(lib().astr_prefill_attention(C.byref(c), int(layer_id), _ptr(q), _ptr(out),
                                        int(n_heads), _stream(stream)))


def astr_set_checked(on: bool) -> None:
    _check(lib().astr_set_checked(1 if on else 0))


def astr_set_wait_timeout_ns(ns: int) -> None:
    _check(lib().astr_set_wait_timeout_ns(int(ns)))


def astr_device_error(stream=None) -> int:
    flags = C.c_uint32(0)
    _check(lib().astr_device_error(_stream(stream), C.byref(flags)))
    return flags.value


def astr_selftest_wait_timeout(ns: int, stream=None) -> int:
    """Run the bounded-wait self-test; returns the raw status (ASTR_ERR_TIMEOUT = 5 expected)."""
    return lib().astr_selftest_wait_timeout(_stream(stream), int(ns))


def astr_version() -> int:
    return lib().astr_version()
