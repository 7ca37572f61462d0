"""Device plumbing: upload a seeded workload with torch, build the KVCache views, run steps.

Data movement and argument marshalling only; every step runs in libastr's kernels through
the binding in this package.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

from . import (KVCache, astr_decode_attention, astr_decode_attention_rope,
               astr_prefill_attention, astr_rope_kv_write)
from .workloads import Workload


def to_torch(arr: np.ndarray, dtype: str, device="cuda", pin: bool = False):
    """Host array -> torch tensor. bf16 data arrives as uint16 bit patterns."""
    import torch
    a = np.ascontiguousarray(arr)
    if dtype == "bf16":
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    elif dtype == "f32":
        t = torch.from_numpy(a.astype(np.float32, copy=False))
    elif dtype == "i32":
        t = torch.from_numpy(a.astype(np.int32, copy=False))
    else:
        raise ValueError(dtype)
    if device == "cpu":
        return t.pin_memory() if pin else t
    return t.to(device)


def to_host(t) -> np.ndarray:
    """torch tensor -> numpy (bf16 -> uint16 bits)."""
    import torch
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


@dataclass
class DeviceWorkload:
    wl: Workload
    k_buffer: object
    v_buffer: object
    req_to_token: object
    n_heads: int
    rope: Optional[dict] = None
    rope2: Optional[dict] = None
    prefill: Optional[dict] = None
    decode: Optional[dict] = None
    decode2: Optional[dict] = None

    # ------------------------------------------------------------------
    @classmethod
    def upload(cls, wl: Workload, device="cuda") -> "DeviceWorkload":
        import torch
        dt = wl.pool.dtype
        dw = cls(wl=wl, k_buffer=to_torch(wl.pool.k_buffer, dt, device),
                 v_buffer=to_torch(wl.pool.v_buffer, dt, device),
                 req_to_token=to_torch(wl.pool.req_to_token, "i32", device), n_heads=wl.n_heads)
        tdt = torch.bfloat16 if dt == "bf16" else torch.float32

        def rope_dict(r):
            if r is None:
                return None
            d = dict(q=to_torch(r.q, dt, device), k=to_torch(r.k, dt, device),
                     v=to_torch(r.v, dt, device), pos=to_torch(r.position_ids, "i32", device),
                     loc=to_torch(r.out_cache_loc, "i32", device),
                     freqs=to_torch(r.freqs_cis, "f32", device), layer=r.layer_id)
            d["q_out"] = torch.empty_like(d["q"])
            d["kv"] = KVCache(dw.k_buffer, dw.v_buffer, out_cache_loc=d["loc"])
            return d

        dw.rope = rope_dict(wl.rope)
        dw.rope2 = rope_dict(wl.rope2)

        def q_of(batch, rope, rows):
            if batch.q is not None:
                return to_torch(batch.q, dt, device)
            return rope["q_out"][batch.q_token_offset: batch.q_token_offset + rows]

        if wl.prefill is not None:
            p = wl.prefill
            q = q_of(p, dw.rope, p.total_q)
            d = dict(q=q, out=torch.empty((p.total_q, wl.n_heads, wl.pool.head_dim), dtype=tdt,
                                          device=device), layer=p.layer_id)
            d["kv"] = KVCache(dw.k_buffer, dw.v_buffer, req_to_token=dw.req_to_token,
                              req_pool_indices=to_torch(p.req_pool_indices, "i32", device),
                              qo_indptr=to_torch(p.qo_indptr, "i32", device),
                              kv_indptr=to_torch(p.kv_indptr, "i32", device),
                              q_tile_to_batch=to_torch(p.q_tile_to_batch, "i32", device),
                              q_tile_to_index=to_torch(p.q_tile_to_index, "i32", device),
                              q_tile_rows=p.q_tile_rows, n_tokens=p.total_q)
            dw.prefill = d

        def decode_dict(dec, rope):
            if dec is None:
                return None
            q = q_of(dec, rope, dec.batch)
            H, D = wl.n_heads, wl.pool.head_dim
            d = dict(q=q, layer=dec.layer_id,
                     out=torch.empty((dec.batch, H, D), dtype=tdt, device=device),
                     o_part=torch.empty((dec.batch, H, dec.max_splits, D), dtype=torch.float32,
                                        device=device),
                     ml_part=torch.empty((dec.batch, H, dec.max_splits, 2), dtype=torch.float32,
                                         device=device))
            d["kv"] = KVCache(dw.k_buffer, dw.v_buffer, req_to_token=dw.req_to_token,
                              req_pool_indices=to_torch(dec.req_pool_indices, "i32", device),
                              seq_lens=to_torch(dec.seq_lens, "i32", device), max_len=dec.max_len,
                              kv_indptr=to_torch(dec.kv_indptr, "i32", device),
                              decode_o_part=d["o_part"], decode_ml_part=d["ml_part"],
                              split_chunk=dec.split_chunk, decode_out=d["out"])
            return d

        dw.decode = decode_dict(wl.decode, dw.rope)
        dw.decode2 = decode_dict(wl.decode2, dw.rope2)
        return dw

    # ------------------------------------------------------------------
    @staticmethod
    def _c(d):
        """The C struct of a step's KVCache, built once (call refresh() after editing fields)."""
        if "c" not in d:
            d["c"] = d["kv"].as_c()
        return d["c"]

    def step_inputs(self):
        """What a step takes from the host: the new tokens' q, k, v, positions and slots, and the
        batch metadata. The cache and the page table stay resident."""
        out = []
        if self.rope is not None:
            r = self.rope
            out += [r["q"], r["k"], r["v"], r["pos"], r["loc"]]
        if self.prefill is not None:
            kv = self.prefill["kv"]
            out += [kv.req_pool_indices, kv.qo_indptr, kv.kv_indptr, kv.q_tile_to_batch,
                    kv.q_tile_to_index]
        if self.decode is not None:
            kv = self.decode["kv"]
            out += [kv.req_pool_indices, kv.seq_lens, kv.kv_indptr]
        return out

    def step_outputs(self):
        """What a step hands back: the prefill and decode attention outputs."""
        return [d["out"] for d in (self.prefill, self.decode) if d is not None]

    def pack(self, tensors, align: int = 256):
        """Moves `tensors` into one contiguous device buffer (each slot `align`-byte aligned) and
        points every reference of the workload at the new copies, so that one copy moves them
        all between host and device. Returns the uint8 buffer."""
        import torch
        sizes = [t.numel() * t.element_size() for t in tensors]
        offs, at = [], 0
        for n in sizes:
            offs.append(at)
            at += (n + align - 1) // align * align
        arena = torch.zeros(at, dtype=torch.uint8, device=tensors[0].device)  # padding stays 0
        for t, o, n in zip(tensors, offs, sizes):
            view = arena[o:o + n].view(t.dtype).view(t.shape)
            view.copy_(t)
            self._rebind(t, view)
        self.refresh()
        return arena

    def _rebind(self, old, new):
        for d in [self.rope, self.rope2, self.prefill, self.decode, self.decode2]:
            if d is None:
                continue
            for k, v in list(d.items()):
                if v is old:
                    d[k] = new
            kv = d.get("kv")
            if kv is not None:
                for name, v in list(vars(kv).items()):
                    if v is old:
                        setattr(kv, name, new)

    def refresh(self):
        self.__dict__.pop("_fused_cache", None)  # holds slices and structs of the old tensors
        for d in [self.rope, self.rope2, self.prefill, self.decode, self.decode2]:
            if d is not None:
                d.pop("c", None)

    def run_rope(self, which="rope", stream=None):
        self.run_rope_dict(getattr(self, which), stream)

    def run_rope_dict(self, r, stream=None):
        astr_rope_kv_write(self._c(r), r["layer"], r["q"], r["q_out"], r["k"], r["v"],
                           self.n_heads, r["freqs"], r["freqs"].shape[0], r["pos"], stream)

    def run_prefill(self, stream=None):
        p = self.prefill
        astr_prefill_attention(self._c(p), p["layer"], p["q"], p["out"], self.n_heads, stream)

    def run_decode(self, which="decode", stream=None):
        d = getattr(self, which)
        astr_decode_attention(self._c(d), d["layer"], d["q"], self.n_heads, stream)

    def _fused_parts(self):
        """For a step whose decode tokens lead the rope batch: the rope of the prefill tokens
        alone, and the decode call with the decode tokens' rotation and cache write folded in."""
        import dataclasses
        key = (id(self.rope), id(self.prefill), id(self.decode))
        cache = self.__dict__.setdefault("_fused_cache", {})
        if key not in cache:
            r, d, n = self.rope, self.decode, self.wl.decode.batch
            rp = {k: (v[n:] if k in ("q", "q_out", "k", "v", "pos", "loc") else v)
                  for k, v in r.items() if k not in ("kv", "c")}
            rp["kv"] = KVCache(self.k_buffer, self.v_buffer, out_cache_loc=rp["loc"])
            dk = dataclasses.replace(d["kv"], out_cache_loc=r["loc"][:n])
            cache[key] = (rp, dk.as_c(), (r["q"][:n], r["k"][:n], r["v"][:n], r["pos"][:n]))
        return cache[key]

    def fusable(self):
        """Whether run_step(fused=True) applies: decode tokens first in the rope batch, the
        prefill's rows right after them, and both queries taken from the rotated q."""
        w = self.wl
        return (self.rope is not None and self.prefill is not None and self.decode is not None and
                w.decode.q is None and w.decode.q_token_offset == 0 and w.prefill.q is None and
                w.prefill.q_token_offset == w.decode.batch)

    def run_step(self, stream=None, side_stream=None, fused=False):
        """One pass of the path over the batch: rotate + write, then prefill, then decode.

        With `side_stream` (a torch.cuda.Stream) the prefill runs there, concurrently with the
        decode on the main stream (`stream`, a torch.cuda.Stream, else the current one): both
        only read what the rotate + write produced and write disjoint outputs. The main stream
        waits for the prefill before the step ends. With `fused` as well (see fusable()), the
        decode rotates and writes its own new tokens (astr_decode_attention_rope) and the side
        stream rotates and writes only the prefill tokens before the prefill, so neither waits
        for the other; the results are the same bytes."""
        if fused and side_stream is not None and self.fusable():
            import torch
            main = stream if stream is not None else torch.cuda.current_stream()
            if not hasattr(self, "_step_events"):
                self._step_events = (torch.cuda.Event(), torch.cuda.Event())
            begun, prefilled = self._step_events
            rp, dec_c, (q, k_new, v_new, pos) = self._fused_parts()
            begun.record(main)  # the side stream starts after whatever preceded the step
            side_stream.wait_event(begun)
            self.run_rope_dict(rp, side_stream.cuda_stream)
            self.run_prefill(side_stream.cuda_stream)
            d = self.decode
            astr_decode_attention_rope(dec_c, d["layer"], q, k_new, v_new, self.n_heads, rp["freqs"],
                                       rp["freqs"].shape[0], pos, main.cuda_stream)
            prefilled.record(side_stream)
            main.wait_event(prefilled)
            return
        if side_stream is None or self.prefill is None or self.decode is None:
            if self.rope is not None:
                self.run_rope("rope", stream)
            if self.prefill is not None:
                self.run_prefill(stream)
            if self.decode is not None:
                self.run_decode("decode", stream)
            return
        import torch
        main = stream if stream is not None else torch.cuda.current_stream()
        if not hasattr(self, "_step_events"):
            self._step_events = (torch.cuda.Event(), torch.cuda.Event())
        written, prefilled = self._step_events
        if self.rope is not None:
            self.run_rope("rope", main.cuda_stream)
        written.record(main)
        side_stream.wait_event(written)
        self.run_prefill(side_stream.cuda_stream)
        self.run_decode("decode", main.cuda_stream)
        prefilled.record(side_stream)
        main.wait_event(prefilled)
