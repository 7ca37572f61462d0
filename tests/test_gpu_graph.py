"""CUDA graphs: a captured step replays exactly what the same calls compute eagerly.

Serving loops capture a decode step once and replay it, changing only the contents of the
device-side metadata between replays. Every entry point passes its plan (grid, split count,
tensor maps) by value at the call, so a capture bakes in the plan for the host fields it was
given (batch, max_len, n_tokens); replays may change the device arrays within those bounds.
"""
import dataclasses

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


def _bits(t):
    import torch
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def _same(a, b):
    import torch
    return torch.equal(_bits(a), _bits(b))


def _capture(fn):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        fn()
    return g


def test_mixed_step_graph_replays_match_eager():
    # rotate + write, ragged prefill and the persistent decode in one graph
    import torch
    wl = W.mixed_b256_p4x512(n_decode=40, lmax=3000, n_prefill=2, chunk_len=300)
    dw = DV.DeviceWorkload.upload(wl)
    k0, v0 = dw.k_buffer.clone(), dw.v_buffer.clone()
    outs = [dw.rope["q_out"], dw.prefill["out"], dw.decode["out"]]
    dw.run_step()  # eager: also the first call of each entry point (before any capture)
    torch.cuda.synchronize()
    ref = [t.clone() for t in outs] + [dw.k_buffer.clone(), dw.v_buffer.clone()]
    dw.k_buffer.copy_(k0)
    dw.v_buffer.copy_(v0)
    for t in outs:
        t.zero_()
    torch.cuda.synchronize()
    g = _capture(dw.run_step)
    torch.cuda.synchronize()
    assert all(not torch.any(_bits(t) != 0) for t in outs)  # capturing ran nothing
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    got = outs + [dw.k_buffer, dw.v_buffer]
    for a, b in zip(got, ref):
        assert _same(a, b)
    assert A.astr_device_error() == 0


def test_two_layer_decode_graph_follows_device_lengths():
    # one graph decodes two layers; between replays only the device seq_lens / kv_indptr change
    # (max_len, a host field, stays the captured upper bound)
    import torch
    lens = np.array([700, 2500, 33, 4000, 1], np.int32)
    wl = W.make_case("bf16", 16, 4, 128, 16, lens, None, n_layers=2, split_chunk=0,
                     max_splits=64, seed=W.SEED_BASE + 900)
    dw = DV.DeviceWorkload.upload(wl)
    d = dw.decode
    kvs = [dataclasses.replace(d["kv"], decode_out=torch.zeros_like(d["out"])) for _ in range(2)]

    def step():
        for lyr in (0, 1):
            A.astr_decode_attention(kvs[lyr], lyr, d["q"], dw.n_heads)

    step()
    torch.cuda.synchronize()
    g = _capture(step)
    seq_lens, kv_indptr = kvs[0].seq_lens, kvs[0].kv_indptr
    for new in (lens, np.array([700, 1200, 33, 3999, 1], np.int32),
                np.array([1, 1, 1, 1, 1], np.int32), lens):
        seq_lens.copy_(torch.from_numpy(new))
        kv_indptr.copy_(torch.from_numpy(W.prefix_sum(new)))
        for kv in kvs:
            kv.decode_out.zero_()
        g.replay()
        torch.cuda.synchronize()
        replayed = [kv.decode_out.clone() for kv in kvs]
        step()  # the same calls, eagerly, on the same device metadata
        torch.cuda.synchronize()
        for lyr in (0, 1):
            assert _same(replayed[lyr], kvs[lyr].decode_out)
            kl = np.ascontiguousarray(wl.pool.k_buffer[lyr])
            vl = np.ascontiguousarray(wl.pool.v_buffer[lyr])
            ref = oracle.decode(wl.decode.q, kl, vl, wl.pool.req_to_token,
                                wl.decode.req_pool_indices, new)
            got = DV.to_host(replayed[lyr])
            got = W.f32_from_bf16_bits(got).astype(np.float64)
            assert np.max(np.abs(got - ref)) <= 2e-2
    assert A.astr_device_error() == 0


def test_fused_rope_decode_graph_matches_eager():
    import torch
    mk = lambda: W.make_case("bf16", 16, 4, 128, 16, [1, 20, 333, 5000], None, with_rope=True,
                             split_chunk=0, max_splits=64, seed=W.SEED_BASE + 910)
    eager, graphed = DV.DeviceWorkload.upload(mk()), DV.DeviceWorkload.upload(mk())
    k0, v0 = graphed.k_buffer.clone(), graphed.v_buffer.clone()

    def fused(dw):
        r, d = dw.rope, dw.decode
        d["kv"].out_cache_loc = r["loc"]
        dw.refresh()
        A.astr_decode_attention_rope(dw._c(d), d["layer"], r["q"], r["k"], r["v"], dw.n_heads,
                                     r["freqs"], r["freqs"].shape[0], r["pos"])

    fused(eager)
    fused(graphed)  # first call before the capture
    torch.cuda.synchronize()
    graphed.k_buffer.copy_(k0)
    graphed.v_buffer.copy_(v0)
    graphed.decode["out"].zero_()
    torch.cuda.synchronize()
    g = _capture(lambda: fused(graphed))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert _same(graphed.decode["out"], eager.decode["out"])
    assert _same(graphed.k_buffer, eager.k_buffer) and _same(graphed.v_buffer, eager.v_buffer)
    assert A.astr_device_error() == 0
