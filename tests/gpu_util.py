"""Helpers for the GPU parity tests: device inputs for a workload, runs through the C ABI."""
from __future__ import annotations

import numpy as np
import torch

from workloads import torch_gen

TOL_ABS = 1e-3
TOL_REL = 1e-2


def dev():
    return torch.device("cuda:0")


def to_dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev()).view(torch.bfloat16)
    t = torch.from_numpy(a).to(dev())
    return t if dtype is None else t.to(dtype)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy bits."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = "") -> float:
    """|got - ref| <= 1e-3 + 1e-2 |ref| elementwise (the decode-attention tolerance)."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bad = ~(err <= TOL_ABS + TOL_REL * np.abs(ref))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first {idx.tolist()} "
                             f"got {got[tuple(idx[0])]} ref {ref[tuple(idx[0])]}")
    return float(err.max()) if err.size else 0.0


class DeviceDecode:
    """Device state of a ``DecodeWorkload``: pool, tables, lengths, queries, workspace, status."""

    def __init__(self, wl, fill_nan: bool = True, generate_on_device: bool = False):
        import paged_kv_cache_180_gb300 as pkv
        self.pkv = pkv
        self.wl = wl
        self.pool = pkv.KVPool(wl.num_pages, device=dev())
        if fill_nan:
            self.pool.buffer.view(torch.int16).fill_(-1)  # 0xFFFF: a NaN pattern in every untouched slot
        self.status = torch.zeros(1, dtype=torch.int32, device=dev())
        self.bt = to_dev(np.ascontiguousarray(wl.block_tables))            # [S, L, B]
        self.lens = to_dev(wl.context_lens)
        self.ws = pkv.decode_workspace(wl.num_seqs, device=dev())
        self.out = torch.empty(wl.num_seqs, wl.num_q_heads, wl.head_dim, dtype=torch.float32, device=dev())
        self.generate_on_device = generate_on_device

    def append_all(self, layer: int = 0, seqs=None):
        if self.generate_on_device:
            k, v, slots = torch_gen.workload_kv(self.wl, layer, dev(), seqs=seqs)
        else:
            if seqs is None:
                kn, vn, sn = self.wl.kv_all(layer)
            else:
                parts = [self.wl.kv_tokens(s, layer) for s in seqs]
                kn = np.concatenate([p[0] for p in parts])
                vn = np.concatenate([p[1] for p in parts])
                sn = np.concatenate([self.wl.slot_mapping(s, layer, 0, int(self.wl.context_lens[s])) for s in seqs])
            k, v, slots = to_dev(kn), to_dev(vn), to_dev(sn)
        if slots.numel():
            self.pkv.kv_append(self.pool, k, v, slots, self.status)

    def q(self, layer: int = 0) -> torch.Tensor:
        if self.generate_on_device:
            return torch_gen.workload_q(self.wl, layer, dev())
        return to_dev(self.wl.q(layer))

    def attend(self, layer: int = 0, num_ctas: int = 0, q: torch.Tensor | None = None, lens: torch.Tensor | None = None,
               max_context: int | None = None) -> torch.Tensor:
        wl = self.wl
        blocks = wl.max_blocks
        bt_layer = self.bt.view(-1)[layer * blocks:]
        self.pkv.paged_decode_attention(self.pool, self.out, self.q(layer) if q is None else q, bt_layer,
                                        wl.num_layers * blocks, self.lens if lens is None else lens,
                                        wl.max_context if max_context is None else max_context, wl.scale,
                                        self.ws, self.status, num_ctas=num_ctas)
        return self.out

    def status_value(self) -> int:
        torch.cuda.synchronize()
        return int(self.status.item())


def oracle_decode_threaded(wl, layer: int = 0, seqs=None):
    """The oracle's decode attention for every (or the chosen) sequence of ``wl``, one sequence
    per host thread: each thread draws its sequence's K/V, appends them into one shared oracle
    pool (sequences own disjoint pages) and attends.  Returns (out [num_seqs, H, D] float64,
    OR of the error bits).  The C calls release the GIL, so a 256 x 2048 batch takes seconds."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    chosen = range(wl.num_seqs) if seqs is None else seqs
    pool = oracle.Pool(wl.num_pages, wl.page_tokens, wl.num_kv_heads, wl.head_dim)
    q = wl.q(layer)
    bt = np.ascontiguousarray(wl.block_tables[:, layer, :])
    lens = np.ascontiguousarray(wl.context_lens)
    out = np.zeros((wl.num_seqs, wl.num_q_heads, wl.head_dim), dtype=np.float64)

    def one(s):
        c = int(lens[s])
        if c > 0 and wl.has_pages(s):
            k, v = wl.kv_tokens(s, layer)
            assert oracle.kv_append(pool, k, v, wl.slot_mapping(s, layer, 0, c)) == 0
        o, err = oracle.paged_decode_attention(pool, q[s:s + 1], bt[s:s + 1], lens[s:s + 1], wl.scale,
                                               wl.max_context)
        out[s] = o[0]
        return err

    with ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        errs = list(ex.map(one, chosen))
    bits = 0
    for e in errs:
        bits |= e
    return out, bits
