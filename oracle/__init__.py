"""CPU oracle for the paged KV-cache attention path -- TEST INFRASTRUCTURE ONLY.

Wraps ``astr_oracle.c`` (plain fp64 C, see its header for the cited definitions and the
readings R1-R5). Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package; the CUDA library never does.

Arrays are numpy: bf16 data is passed as uint16 bit patterns, f32 as float32, indices int32.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "astr_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp contraction off, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_LIB)
            P, I, I64 = C.c_void_p, C.c_int, C.c_int64
            L.oracle_causal_mask.argtypes = [I, P]
            L.oracle_rope_f64.argtypes = [I64, I, I, P, P, I, P, P]
            L.oracle_rope_f64.restype = I
            L.oracle_rope_kv_write.argtypes = [I, I64, I, I, I, P, P, P, P, I, P, P, I64, P, P, P]
            L.oracle_rope_kv_write.restype = I
            L.oracle_rope_apply.argtypes = [I, I64, I, I, P, P, I, P, I, P]
            L.oracle_rope_apply.restype = I
            L.oracle_decode.argtypes = [I, I, I, I, I, P, P, P, I64, P, I, I, P, P, I, P, P]
            L.oracle_decode.restype = I
            L.oracle_decode_split.argtypes = [I, I, I, I, I, P, P, P, I64, P, I, I, P, P, I, I,
                                              P, P, P, P]
            L.oracle_decode_split.restype = I
            L.oracle_prefill.argtypes = [I, I, I, I, I, P, P, P, I64, P, I, I, P, P, P, I64, P, P]
            L.oracle_prefill.restype = I
            L.oracle_num_threads.restype = I
            L.oracle_set_num_threads.argtypes = [I]
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def _dt(arr) -> int:
    if arr.dtype == np.uint16:
        return BF16
    if arr.dtype == np.float32:
        return F32
    raise TypeError(f"unsupported element type {arr.dtype}")


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


def causal_mask(n: int) -> np.ndarray:
    out = np.empty((n, n), dtype=np.float64)
    lib().oracle_causal_mask(n, _p(out))
    return out


def rope_f64(x: np.ndarray, freqs: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """Exact rotation of x [T, nh, D] (any float dtype) by an fp64 table [max_len, D/2, 2]."""
    x = _c(x, np.float64)
    fr = _c(freqs, np.float64)
    pos = _c(pos, np.int32)
    T, nh, D = x.shape
    out = np.zeros_like(x)
    bad = lib().oracle_rope_f64(T, nh, D, _p(x), _p(fr), fr.shape[0], _p(pos), _p(out))
    if bad:
        raise ValueError(f"{bad} positions outside the table")
    return out


def rope_kv_write(q, k, v, freqs, pos, loc, k_layer, v_layer):
    """Rotate q/k under the f32 rounding specification, write k/v rows at ``loc``.

    ``k_layer``/``v_layer`` are one layer's [size, Hk, D] arrays, modified in place.
    Returns q_out (same dtype as q).
    """
    dt = _dt(q)
    et = q.dtype
    q = _c(q, et); k = _c(k, et); v = _c(v, et)
    fr = _c(freqs, np.float32)
    pos = _c(pos, np.int32); loc = _c(loc, np.int32)
    assert k_layer.flags.c_contiguous and v_layer.flags.c_contiguous
    assert k_layer.dtype == et and v_layer.dtype == et
    T, H, D = q.shape
    Hk = k.shape[1]
    q_out = np.zeros_like(q)
    bad = lib().oracle_rope_kv_write(dt, T, H, Hk, D, _p(q), _p(k), _p(v), _p(fr), fr.shape[0],
                                     _p(pos), _p(loc), k_layer.shape[0], _p(q_out),
                                     _p(k_layer), _p(v_layer))
    if bad:
        raise ValueError(f"{bad} tokens with a position or slot out of range")
    return q_out


def rope_apply(x, freqs, pos, inverse=False):
    """RoPE with no cache write, under the f32 rounding specification: the rotation by theta
    (inverse False, the training forward) or by -theta (inverse True: R^T, which maps the
    gradient of the rotated tensor to the gradient of its input). x: [T, nh, D]."""
    dt = _dt(x)
    et = x.dtype
    x = _c(x, et)
    fr = _c(freqs, np.float32)
    pos = _c(pos, np.int32)
    T, nh, D = x.shape
    out = np.zeros_like(x)
    bad = lib().oracle_rope_apply(dt, T, nh, D, _p(x), _p(fr), fr.shape[0], _p(pos),
                                  1 if inverse else 0, _p(out))
    if bad:
        raise ValueError(f"{bad} tokens with a position out of range")
    return out


def _check_layer(k_layer, v_layer, et):
    assert k_layer.flags.c_contiguous and v_layer.flags.c_contiguous
    assert k_layer.dtype == et and v_layer.dtype == et


def decode(q, k_layer, v_layer, req_to_token, req_pool_indices, seq_lens, sel=None):
    """fp64 decode output [B, H, D] (rows of unselected requests stay zero)."""
    et = q.dtype
    dt = _dt(q)
    q = _c(q, et)
    _check_layer(k_layer, v_layer, et)
    r2t = _c(req_to_token, np.int32)
    rpi = _c(req_pool_indices, np.int32)
    sl = _c(seq_lens, np.int32)
    B, H, D = q.shape
    Hk = k_layer.shape[1]
    out = np.zeros((B, H, D), dtype=np.float64)
    sel_a = None if sel is None else _c(sel, np.int32)
    fails = lib().oracle_decode(dt, B, H, Hk, D, _p(q), _p(k_layer), _p(v_layer),
                                k_layer.shape[0], _p(r2t), r2t.shape[0], r2t.shape[1], _p(rpi),
                                _p(sl), 0 if sel_a is None else sel_a.size, _p(sel_a), _p(out))
    if fails:
        raise ValueError(f"{fails} decode units failed validation")
    return out


def decode_split(q, k_layer, v_layer, req_to_token, req_pool_indices, seq_lens, chunk,
                 max_splits):
    """fp64 split-K partials and their log-sum-exp merge.

    Returns (o_part [B,H,S,D], m_part [B,H,S], l_part [B,H,S], out [B,H,D]); partial entries
    past ceil(L/chunk) are NaN.
    """
    et = q.dtype
    dt = _dt(q)
    q = _c(q, et)
    _check_layer(k_layer, v_layer, et)
    r2t = _c(req_to_token, np.int32)
    rpi = _c(req_pool_indices, np.int32)
    sl = _c(seq_lens, np.int32)
    B, H, D = q.shape
    Hk = k_layer.shape[1]
    S = int(max_splits)
    o_part = np.full((B, H, S, D), np.nan)
    m_part = np.full((B, H, S), np.nan)
    l_part = np.full((B, H, S), np.nan)
    out = np.zeros((B, H, D))
    fails = lib().oracle_decode_split(dt, B, H, Hk, D, _p(q), _p(k_layer), _p(v_layer),
                                      k_layer.shape[0], _p(r2t), r2t.shape[0], r2t.shape[1],
                                      _p(rpi), _p(sl), int(chunk), S, _p(o_part), _p(m_part),
                                      _p(l_part), _p(out))
    if fails:
        raise ValueError(f"{fails} split decode units failed validation")
    return o_part, m_part, l_part, out


def prefill(q, k_layer, v_layer, req_to_token, req_pool_indices, qo_indptr, kv_indptr,
            rows=None):
    """fp64 prefill output for the packed rows ``rows`` (all rows when None): [n, H, D]."""
    et = q.dtype
    dt = _dt(q)
    q = _c(q, et)
    _check_layer(k_layer, v_layer, et)
    r2t = _c(req_to_token, np.int32)
    rpi = _c(req_pool_indices, np.int32)
    qo = _c(qo_indptr, np.int32)
    kv = _c(kv_indptr, np.int32)
    T, H, D = q.shape
    Hk = k_layer.shape[1]
    B = qo.size - 1
    rows_a = None if rows is None else _c(rows, np.int32)
    n = T if rows_a is None else rows_a.size
    out = np.zeros((n, H, D), dtype=np.float64)
    fails = lib().oracle_prefill(dt, B, H, Hk, D, _p(q), _p(k_layer), _p(v_layer),
                                 k_layer.shape[0], _p(r2t), r2t.shape[0], r2t.shape[1], _p(rpi),
                                 _p(qo), _p(kv), n, _p(rows_a), _p(out))
    if fails:
        raise ValueError(f"{fails} prefill units failed validation")
    return out
