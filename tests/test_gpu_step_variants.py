"""The ways DeviceWorkload.run_step can run a step leave exactly the same bytes.

Serial (rotate + write, prefill, decode on one stream), overlapped (the prefill on a second
stream, concurrent with the decode) and fused (the decode rotating and writing its own new
tokens while the second stream rotates and writes the prefill tokens and runs the prefill).
"""
import pytest

from paged_kv_cache_apply_gb300 import build as B
from paged_kv_cache_apply_gb300 import device as DV
from paged_kv_cache_apply_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()
    import torch
    torch.cuda.init()


def _run(mode):
    import torch
    wl = W.mixed_b256_p4x512(n_decode=48, lmax=3000, n_prefill=3, chunk_len=260)
    dw = DV.DeviceWorkload.upload(wl)
    side = torch.cuda.Stream()
    assert dw.fusable()
    for _ in range(2):  # twice: the second step rewrites the same bytes
        if mode == "serial":
            dw.run_step()
        else:
            dw.run_step(side_stream=side, fused=mode == "fused")
    torch.cuda.synchronize()
    return [t.view(torch.int16).clone() for t in (dw.prefill["out"], dw.decode["out"], dw.k_buffer,
                                                  dw.v_buffer)]


def test_overlapped_and_fused_steps_equal_the_serial_step():
    import torch
    ref = _run("serial")
    for mode in ("overlapped", "fused"):
        got = _run(mode)
        for a, b in zip(got, ref):
            assert torch.equal(a, b), mode


def test_fused_step_follows_rebound_tensors():
    # pack() moves the step's inputs into one buffer; the fused step must use the new views
    import torch
    wl = W.mixed_b256_p4x512(n_decode=16, lmax=900, n_prefill=1, chunk_len=200)
    dw = DV.DeviceWorkload.upload(wl)
    side = torch.cuda.Stream()
    dw.run_step(side_stream=side, fused=True)
    torch.cuda.synchronize()
    ref = dw.decode["out"].clone()
    arena = dw.pack(dw.step_inputs())
    dw.rope["q"].zero_()  # the packed copy of the decode and prefill queries' source
    dw.run_step(side_stream=side, fused=True)
    torch.cuda.synchronize()
    assert not torch.equal(dw.decode["out"].view(torch.int16), ref.view(torch.int16))
    del arena
