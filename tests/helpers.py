"""Shared helpers of the GPU tests: upload a seeded workload and run library calls on it."""
from __future__ import annotations

import numpy as np
import torch

import gen
import sparse_paged_kv_score_gb300 as spkv

DEV = torch.device("cuda:0")


def bf(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(DEV)


def f32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(DEV)


def u32_as_i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint32).view(np.int32)).to(DEV)


class Dev:
    """A sparse workload on the device with its library handle."""

    def __init__(self, w: dict, page_cnt=None, max_units: int = 0, summary_bf16: bool = False):
        self.w = w
        self.B, self.Hq, self.Hk, self.npm = w["B"], w["Hq"], w["Hk"], w["np_max"]
        self.k_pool, self.v_pool = bf(w["k_pool"]), bf(w["v_pool"])
        self.ksum = torch.zeros(self.Hk, w["n_phys"], 4, 128, device=DEV,
                                dtype=torch.bfloat16 if summary_bf16 else torch.float32)
        cnt = gen.page_counts(w) if page_cnt is None else page_cnt
        self.cnt = i32(cnt)
        self.cache = spkv.paged_kv_create(self.k_pool, self.v_pool, self.ksum, self.cnt,
                                          max_units=max_units)
        self.pt = i32(w["page_table"])
        self.L = i32(w["seq_len"])
        self.q = bf(w["q"])

    def scores(self, q=None) -> torch.Tensor:
        s = torch.empty(self.B, self.Hk, self.npm, dtype=torch.float32, device=DEV)
        spkv.score_blocks(self.cache, self.q if q is None else q, self.pt, self.L, s)
        return s

    def new_alive(self) -> torch.Tensor:
        return torch.full((self.B, self.Hk, (self.npm + 31) // 32), -1, dtype=torch.int32, device=DEV)

    def select(self, scores, evict, alive, k_q, k_e):
        stride = k_q + k_e + 1
        sel = torch.empty(self.B, self.Hk, stride, dtype=torch.int32, device=DEV)
        n_sel = torch.empty(self.B, self.Hk, dtype=torch.int32, device=DEV)
        spkv.select_topk(self.cache, scores, evict, alive, self.L, k_q, k_e, sel, n_sel)
        return sel, n_sel

    def attn(self, sel, n_sel, q=None):
        out = torch.empty(self.B, self.Hq, 128, dtype=torch.float32, device=DEV)
        lse = torch.empty(self.B, self.Hq, dtype=torch.float32, device=DEV)
        spkv.sparse_decode_attn(self.cache, self.q if q is None else q, self.pt, sel, n_sel, self.L,
                                out, lse)
        return out, lse

    def errors(self):
        return spkv.get_device_error(self.cache)

    def close(self):
        self.cache.close()


def host_bits(x):
    """bf16 device tensor -> its uint16 bit patterns on the host."""
    return x.view(torch.int16).cpu().numpy().view(np.uint16)


def pinned_bf16(a: np.ndarray) -> torch.Tensor:
    t = torch.empty(a.shape, dtype=torch.int16, pin_memory=True)
    t.numpy()[...] = a.view(np.int16)
    return t.view(torch.bfloat16)


class Offload:
    """Host pool (pinned), device slot pool with its handle, and the residency tables."""

    def __init__(self, d: Dev, n_slots: int):
        w = d.w
        self.d, self.n_slots = d, n_slots
        self.B, self.Hk = w["B"], w["Hk"]
        self.U = self.B * self.Hk
        self.k_host, self.v_host = pinned_bf16(w["k_pool"]), pinned_bf16(w["v_pool"])
        shp = (self.Hk, self.B * n_slots, 64, 128)
        self.k_slots = torch.zeros(shp, dtype=torch.bfloat16, device=DEV)
        self.v_slots = torch.zeros(shp, dtype=torch.bfloat16, device=DEV)
        self.slots = spkv.paged_kv_create(self.k_slots, self.v_slots, None, None, max_units=self.U)
        self.resident = i32(np.full((self.U, n_slots), -1, np.int32))
        self.ts = i32(np.full((self.U, n_slots), np.iinfo(np.int32).min, np.int32))

    def step(self, sel, n_sel, t, q):
        U, stride = self.U, sel.shape[-1]
        miss = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        nm = torch.empty(U, dtype=torch.int32, device=DEV)
        slot = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        spkv.resident_setdiff(self.d.cache, self.resident, sel, n_sel, miss, nm, slot)
        vic = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        hist = torch.empty(U, 64, dtype=torch.int32, device=DEV)
        spkv.lru_bucket_update(self.d.cache, self.resident, self.ts, slot, n_sel.view(U), miss, nm, t, 1, vic,
                               hist)
        slot_before = slot.clone()
        spkv.retrieve_pages(self.slots, self.k_host, self.v_host, self.d.pt, miss, nm, vic, slot, n_sel,
                            self.n_slots)
        B, Hq = q.shape[0], q.shape[1]
        out = torch.empty(B, Hq, 128, dtype=torch.float32, device=DEV)
        lse = torch.empty(B, Hq, dtype=torch.float32, device=DEV)
        spkv.sparse_decode_attn_slots(self.slots, q, sel, slot.view(sel.shape), n_sel, self.n_slots, self.d.L,
                                      out, lse)
        return dict(miss=miss, nm=nm, slot_before=slot_before, vic=vic, slot=slot, out=out, lse=lse)

    def close(self):
        self.slots.close()


def alive_bits_to_bytes(words: np.ndarray, np_max: int) -> np.ndarray:
    w = words.astype(np.uint32)
    bits = (w[..., :, None] >> np.arange(32, dtype=np.uint32)) & 1
    return bits.reshape(*w.shape[:-1], -1)[..., :np_max].astype(np.uint8)


def alive_bytes_to_bits(b: np.ndarray) -> np.ndarray:
    npm = b.shape[-1]
    nw = (npm + 31) // 32
    pad = np.zeros((*b.shape[:-1], nw * 32), np.uint32)
    pad[..., :npm] = b
    pad = pad.reshape(*b.shape[:-1], nw, 32)
    return (pad << np.arange(32, dtype=np.uint32)).sum(-1).astype(np.uint32)


def attn_errors(out: np.ndarray, ref: np.ndarray):
    e = np.abs(out.astype(np.float64) - ref)
    return float(e.max()), float(e.mean())
