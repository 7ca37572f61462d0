"""The five configurations at full size, in the launch configuration bench.py times.

Every attention output the oracle can afford is compared (all decode outputs, all prefill rows
of the mixed batch, a stratified sample of the varlen prefill rows); every written cache row
and every rotated q row is compared bit for bit, and every other cache row is checked
unchanged. The mixed batch runs both as bench.py's timed step (two streams, the decode with
its tokens' rotate + write folded in, unsplit) and as three serial calls.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_apply_gb300 as A
from paged_kv_cache_apply_gb300 import build as B
from paged_kv_cache_apply_gb300 import device as DV
from paged_kv_cache_apply_gb300 import workloads as W

pytestmark = pytest.mark.gpu
TOL_BF16 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()


def _sync():
    import torch
    torch.cuda.synchronize()


def wid(a):
    return W.f32_from_bf16_bits(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


def test_decode_b64_page1():
    wl = W.decode_b64_page1()
    dw = DV.DeviceWorkload.upload(wl)
    dw.run_decode()
    _sync()
    d = wl.decode
    ref = oracle.decode(d.q, wl.pool.k_buffer[0], wl.pool.v_buffer[0], wl.pool.req_to_token,
                        d.req_pool_indices, d.seq_lens)
    err = np.max(np.abs(wid(DV.to_host(dw.decode["out"])) - ref))
    assert err <= TOL_BF16, err


def test_prefill_b8_varlen_resumed():
    wl = W.prefill_b8_varlen()
    dw = DV.DeviceWorkload.upload(wl)
    A.astr_device_error()  # clear
    dw.prefill["out"].fill_(float("nan"))  # a row the kernel never writes stays NaN
    dw.run_prefill()
    _sync()
    assert A.astr_device_error() == 0
    import torch
    assert not bool(torch.isnan(dw.prefill["out"]).any()), "prefill rows left unwritten"
    p = wl.prefill
    rng = np.random.default_rng(3)
    rows = set()
    for b in range(p.batch):
        q0, q1 = int(p.qo_indptr[b]), int(p.qo_indptr[b + 1])
        for i in [0, 1, 126, 127, 128, 129, q1 - q0 - 2, q1 - q0 - 1]:
            if 0 <= i < q1 - q0:
                rows.add(q0 + i)
        rows.update(rng.integers(q0, q1, 24).tolist())
    rows = np.array(sorted(rows), dtype=np.int32)
    ref = oracle.prefill(p.q, wl.pool.k_buffer[0], wl.pool.v_buffer[0], wl.pool.req_to_token,
                         p.req_pool_indices, p.qo_indptr, p.kv_indptr, rows=rows)
    got = wid(DV.to_host(dw.prefill["out"])[rows])
    err = np.max(np.abs(got - ref))
    assert err <= TOL_BF16, err


def test_long_decode_b4_split():
    wl = W.long_decode_b4()
    dw = DV.DeviceWorkload.upload(wl)
    dw.run_decode()
    _sync()
    d = wl.decode
    kl, vl = wl.pool.k_buffer[0], wl.pool.v_buffer[0]
    ref = oracle.decode(d.q, kl, vl, wl.pool.req_to_token, d.req_pool_indices, d.seq_lens)
    err = np.max(np.abs(wid(DV.to_host(dw.decode["out"])) - ref))
    assert err <= TOL_BF16, err
    # the fixed 4096-token partials of request 0 against the oracle's
    one = np.ascontiguousarray(d.q[:1])
    o_p, m_p, l_p, _ = oracle.decode_split(one, kl, vl, wl.pool.req_to_token,
                                           d.req_pool_indices[:1], d.seq_lens[:1], 4096,
                                           d.max_splits)
    n = (int(d.seq_lens[0]) + 4095) // 4096
    go = DV.to_host(dw.decode["o_part"])[0, :, :n]
    gml = DV.to_host(dw.decode["ml_part"])[0, :, :n].astype(np.float64)
    assert np.max(np.abs(go - o_p[0, :, :n])) <= 1e-3
    lse = gml[..., 0] + np.log(gml[..., 1])
    assert np.max(np.abs(lse - (m_p[0, :, :n] + np.log(l_p[0, :, :n])))) <= 1e-3


def _mixed_reference(wl):
    """The oracle's rotate + write over all 2304 new tokens, then its prefill of every chunk row
    and its decode of every request, on a host copy of the layer."""
    kl = np.ascontiguousarray(wl.pool.k_buffer[0]).copy()
    vl = np.ascontiguousarray(wl.pool.v_buffer[0]).copy()
    r = wl.rope
    q_ref = oracle.rope_kv_write(r.q, r.k, r.v, r.freqs_cis, r.position_ids, r.out_cache_loc, kl, vl)
    p = wl.prefill
    q_pre = q_ref[p.q_token_offset: p.q_token_offset + p.total_q]
    ref_p = oracle.prefill(q_pre, kl, vl, wl.pool.req_to_token, p.req_pool_indices, p.qo_indptr,
                           p.kv_indptr)
    d = wl.decode
    q_dec = np.ascontiguousarray(q_ref[: d.batch])
    ref_d = oracle.decode(q_dec, kl, vl, wl.pool.req_to_token, d.req_pool_indices, d.seq_lens)
    return kl, vl, q_ref, ref_p, ref_d


def _check_mixed(wl, dw, k_before, v_before, q_rows):
    """Every written cache row bit-exact, every other row unchanged, the rotated q of `q_rows`
    bit-exact, and every prefill row and decode output within the bf16 tolerance."""
    import torch
    kl, vl, q_ref, ref_p, ref_d = _mixed_reference(wl)
    r = wl.rope
    got_q = DV.to_host(dw.rope["q_out"])
    assert np.array_equal(got_q[q_rows], q_ref[q_rows])
    loc = torch.from_numpy(r.out_cache_loc.astype(np.int64)).cuda()
    assert np.array_equal(DV.to_host(dw.k_buffer[0, loc]), kl[r.out_cache_loc])
    assert np.array_equal(DV.to_host(dw.v_buffer[0, loc]), vl[r.out_cache_loc])
    for buf, before in ((dw.k_buffer, k_before), (dw.v_buffer, v_before)):
        changed = (buf != before).flatten(2).any(dim=2)[0].nonzero().flatten().cpu().numpy()
        assert set(changed.tolist()) <= set(r.out_cache_loc.tolist())
    err_p = np.max(np.abs(wid(DV.to_host(dw.prefill["out"])) - ref_p))
    assert err_p <= TOL_BF16, err_p
    err_d = np.max(np.abs(wid(DV.to_host(dw.decode["out"])) - ref_d))
    assert err_d <= TOL_BF16, err_d


def test_mixed_b256_p4x512_timed_step():
    """Exactly the step bench.py times: the prefill tokens' rotate + write and the prefill on a
    second stream, and, concurrently on the main stream, the decode of all 256 requests with
    their own rotate + write folded in (astr_decode_attention_rope), left unsplit by the plan."""
    import torch
    import paged_kv_cache_apply_gb300 as A
    wl = W.mixed_b256_p4x512()
    dw = DV.DeviceWorkload.upload(wl)
    assert dw.fusable()
    assert A.astr_decode_plan(dw.decode["kv"], wl.n_heads)[1] == 1  # the unsplit plan
    k_before, v_before = dw.k_buffer.clone(), dw.v_buffer.clone()
    dw.rope["q_out"].view(torch.int16).fill_(0x7FC0)  # the decode tokens' q_out stays unwritten
    dw.run_step(side_stream=torch.cuda.Stream(), fused=True)
    _sync()
    assert A.astr_device_error() == 0
    n = wl.decode.batch
    assert np.all(DV.to_host(dw.rope["q_out"][:n]) == 0x7FC0)
    _check_mixed(wl, dw, k_before, v_before, np.arange(n, wl.rope.n_tokens))


def test_mixed_b256_p4x512_serial_step():
    """The same batch with the three calls one after another on one stream (rotate + write of
    all tokens, prefill, decode)."""
    wl = W.mixed_b256_p4x512()
    dw = DV.DeviceWorkload.upload(wl)
    k_before, v_before = dw.k_buffer.clone(), dw.v_buffer.clone()
    dw.run_step()
    _sync()
    _check_mixed(wl, dw, k_before, v_before, np.arange(wl.rope.n_tokens))
