"""The allocation-free decode entry point against the oracle and the regular one, through the
C ABI.

Callers that cannot allocate device memory (plugin hosts that receive only a call's
tensors, runtimes that reserve all device memory at start-up) call
astr_decode_attention_noalloc, which keeps the split-K partials in a fixed 8 MiB array
inside the library instead of caller-provided decode_o_part / decode_ml_part. On the same
inputs it runs the same plan and kernels as astr_decode_attention, so its output must be
byte-identical to that call's and within the float tolerance of the oracle's decode, call
after call, since every call reuses the same array. The file sorts last so that a stop at its
first failure has run every other test; it also passes on its own in a fresh process.
"""
import ctypes as C

import numpy as np
import pytest

import oracle
import paged_kv_cache_apply_gb300 as A
from paged_kv_cache_apply_gb300 import build as B
from paged_kv_cache_apply_gb300 import device as DV
from paged_kv_cache_apply_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()
    oracle.build()
    import torch
    torch.cuda.init()


def _f64(t):
    a = DV.to_host(t)
    return W.f32_from_bf16_bits(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


@pytest.mark.parametrize("dtype,H,Hk,D,page,lens,chunk", [
    ("bf16", 16, 4, 128, 16, [100, 3000, 4097, 1], 0),   # tensor-core decode, library-chosen splits
    ("bf16", 16, 4, 128, 1, [700, 2500, 31], 512),       # explicit chunk, page size 1
    ("f32", 8, 2, 64, 16, [33, 900, 129], 128),          # CUDA-core decode
])
def test_noalloc_matches_oracle_and_regular_decode_on_consecutive_calls(dtype, H, Hk, D, page, lens, chunk):
    import torch
    wl = W.make_case(dtype, H, Hk, D, page, lens, None, split_chunk=chunk, max_splits=64,
                     seed=W.SEED_BASE + 900 + sum(lens))
    dw = DV.DeviceWorkload.upload(wl)
    d = dw.decode
    c = dw._c(d)
    assert A.astr_decode_plan(c, H)[1] > 1  # the regular call really splits
    # the plan the no-alloc call derives: its split limit is what the built-in scratch holds
    cn = A.astr_kv_cache.from_buffer_copy(c)
    cn.max_splits = (8 << 20) // (4 * len(lens) * H * (D + 2))
    assert A.astr_decode_plan(cn, H) == A.astr_decode_plan(c, H)  # so it splits as well
    dw.run_decode()
    torch.cuda.synchronize()
    regular = DV.to_host(d["out"])
    dd = wl.decode
    ref = oracle.decode(dd.q, wl.pool.k_buffer[dd.layer_id], wl.pool.v_buffer[dd.layer_id],
                        wl.pool.req_to_token, dd.req_pool_indices, dd.seq_lens)
    assert np.max(np.abs(_f64(d["out"]) - ref)) <= TOL[dtype]
    for _ in range(2):
        d["out"].zero_()
        A.astr_decode_attention_noalloc(c, d["layer"], d["q"], H)
        torch.cuda.synchronize()
        assert np.array_equal(DV.to_host(d["out"]), regular)
        assert np.max(np.abs(_f64(d["out"]) - ref)) <= TOL[dtype]
    assert A.astr_device_error() == 0


def test_noalloc_rejects_a_split_plan_beyond_its_scratch():
    wl = W.make_case("bf16", 16, 4, 128, 16, [4096] * 64, None, split_chunk=128, max_splits=64)
    dw = DV.DeviceWorkload.upload(wl)
    d = dw.decode
    c = dw._c(d)
    # 64 requests x 16 heads x (128 + 2) floats per split: 32 splits need 17 MB > 8 MiB
    st = A.lib().astr_decode_attention_noalloc(C.byref(c), d["layer"], A._ptr(d["q"]), 16,
                                               A._stream(None))
    assert st == 1
    assert "scratch" in A.lib().astr_last_error().decode()
