"""The C-ABI library loads, exports every symbol include/astr.h declares, and validates
arguments on the host (no GPU: only calls that fail validation before any CUDA work)."""
import ctypes as C
import os
import re

import pytest

import paged_kv_cache_apply_gb300 as A
from paged_kv_cache_apply_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "astr.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    return A.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(astr_\w+)\s*\(", text)))


def test_header_declares_the_three_path_calls():
    names = declared_functions()
    for n in ["astr_rope_kv_write", "astr_decode_attention", "astr_prefill_attention"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_struct_mirror_matches_library(L):
    assert L.astr_kv_cache_bytes() == C.sizeof(A.astr_kv_cache)
    assert A.astr_version() == 100


def _fake_cache(**kw):
    c = A.astr_kv_cache()
    c.k_buffer = c.v_buffer = 0x10000
    c.n_layers, c.size, c.n_kv_heads, c.head_dim, c.dtype = 1, 100, 2, 64, A.ASTR_BF16
    c.req_to_token = c.req_pool_indices = c.seq_lens = c.decode_out = 0x20000
    c.num_reqs, c.max_ctx_len, c.batch, c.max_len = 4, 64, 2, 64
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _status(L, fn, *args):
    st = getattr(L, fn)(*args)
    return st, L.astr_last_error().decode()


@pytest.mark.parametrize("field,value,expect", [
    ("head_dim", 96, 2), ("dtype", 7, 2), ("n_kv_heads", 0, 1), ("size", 0, 1),
    ("k_buffer", 0, 1), ("k_buffer", 0x10008, 1), ("n_layers", 0, 1),
])
def test_decode_rejects_bad_cache(L, field, value, expect):
    c = _fake_cache(**{field: value})
    st, msg = _status(L, "astr_decode_attention", C.byref(c), 0, 0x30000, 4, None)
    assert st == expect and msg


def test_decode_rejects_bad_heads_and_layer(L):
    c = _fake_cache()
    assert _status(L, "astr_decode_attention", C.byref(c), 0, 0x30000, 3, None)[0] == 1
    assert _status(L, "astr_decode_attention", C.byref(c), 1, 0x30000, 4, None)[0] == 1
    assert _status(L, "astr_decode_attention", None, 0, 0x30000, 4, None)[0] == 1
    # group size 32 / 2 = 16 is not served
    assert _status(L, "astr_decode_attention", C.byref(c), 0, 0x30000, 32, None)[0] == 2
    # max_len beyond the table width
    c2 = _fake_cache(max_len=65)
    assert _status(L, "astr_decode_attention", C.byref(c2), 0, 0x30000, 4, None)[0] == 1
    # several splits needed but no scratch
    c3 = _fake_cache(split_chunk=16)
    st, msg = _status(L, "astr_decode_attention", C.byref(c3), 0, 0x30000, 4, None)
    assert st == 1 and "splits" in msg
    # scratch too small for the splits
    c4 = _fake_cache(split_chunk=16, decode_o_part=0x40000, decode_ml_part=0x50000, max_splits=3)
    st, msg = _status(L, "astr_decode_attention", C.byref(c4), 0, 0x30000, 4, None)
    assert st == 1 and "max_splits" in msg


def test_decode_plan_host_only(L):
    c = _fake_cache(split_chunk=16, max_len=50)
    chunk, n = C.c_int32(), C.c_int32()
    assert L.astr_decode_plan(C.byref(c), 4, C.byref(chunk), C.byref(n)) == 0
    assert (chunk.value, n.value) == (16, 4)
    c = _fake_cache(max_len=50)  # no scratch: one chunk covers max_len
    assert L.astr_decode_plan(C.byref(c), 4, C.byref(chunk), C.byref(n)) == 0
    assert (chunk.value, n.value) == (50, 1)


def _sms():
    # the planner asks the current device for its SM count and assumes 148 without one
    try:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.get_device_properties(0).multi_processor_count
    except Exception:
        pass
    return 148


def _plan_rule(batch, Hk, max_len, max_splits):
    """The library's automatic split plan for the tensor-core decode kernel (decode_chunk in
    csrc/astr_api.cu), restated.

    Whole requests (no split) when the kernel ranks the batch (<= 1024 requests) and
    batch x n_kv_heads >= 6 x SMs. Otherwise about four items per SM from a mean length of
    max_len / 2, within [512, 4096] tokens, no more splits than max_splits, rounded up to whole
    128-token tiles, and at most max_len."""
    sms = _sms()
    if batch <= 1024 and batch * Hk >= 6 * sms:
        return max_len, 1
    c = (batch * max_len // 2) * Hk // (sms * 4)
    c = min(max(c, 512), 4096)
    c = max(c, -(-max_len // max_splits))
    c = min(-(-c // 128) * 128, max_len)
    return c, -(-max_len // c)


@pytest.mark.parametrize("batch,Hk,max_len,max_splits", [
    (256, 4, 8192, 16), (64, 4, 4096, 16), (4, 4, 131072, 32), (1, 4, 600, 8), (2000, 4, 8192, 8),
    (300, 1, 1 << 20, 512),
])
def test_decode_plan_follows_the_stated_rule(L, batch, Hk, max_len, max_splits):
    c = _fake_cache(head_dim=128, n_kv_heads=Hk, batch=batch, max_len=max_len, max_ctx_len=max_len,
                    decode_o_part=0x40000, decode_ml_part=0x50000, max_splits=max_splits)
    chunk, n = C.c_int32(), C.c_int32()
    assert L.astr_decode_plan(C.byref(c), 4 * Hk, C.byref(chunk), C.byref(n)) == 0
    assert (chunk.value, n.value) == _plan_rule(batch, Hk, max_len, max_splits)
    assert n.value <= max_splits and chunk.value * n.value >= max_len


def test_prefill_and_rope_reject_bad_arguments(L):
    c = _fake_cache(qo_indptr=0x1000, kv_indptr=0x1000, q_tile_to_batch=0x1000,
                    q_tile_to_index=0x1000, num_q_tiles=2, q_tile_rows=64)
    st, msg = _status(L, "astr_prefill_attention", C.byref(c), 0, 0x30000, 0x30000, 4, None)
    assert st == 2 and "q_tile_rows" in msg
    c.q_tile_rows = 128
    assert _status(L, "astr_prefill_attention", C.byref(c), 0, None, 0x30000, 4, None)[0] == 1
    r = _fake_cache(out_cache_loc=0x1000, n_tokens=3)
    assert _status(L, "astr_rope_kv_write", C.byref(r), 0, 0x30000, 0x30000, 0x30000, 0x30000,
                   4, None, 64, 0x1000, None)[0] == 1
    assert _status(L, "astr_rope_kv_write", C.byref(r), 0, 0x30000, 0x30000, 0x30000, 0x30000,
                   4, 0x30000, 0, 0x1000, None)[0] == 1
    r0 = _fake_cache(n_tokens=0)  # nothing to do
    assert _status(L, "astr_rope_kv_write", C.byref(r0), 0, None, None, None, None, 4, None, 0,
                   None, None)[0] == 0


def test_python_errors_carry_the_message(L):
    c = _fake_cache(head_dim=32)
    with pytest.raises(A.AstrError) as ei:
        A.astr_decode_attention(c, 0, 0x30000, 4, stream=0)
    assert ei.value.status == 2 and "head_dim" in str(ei.value)
