"""GPU parity of the two-level page directory ([Spin] 2C, hierarchical metadata management).

The *_dir calls resolve every logical page through the directory (device-tier segments, host-tier
segments read in place from pinned memory, unmapped ranges) instead of a flat page table.  Given
the same table contents they must return bit for bit what the flat-table calls return; those are
checked against the fp64 oracle elsewhere, and the oracle's own translation (dir_to_table) is
pinned on the CPU.  The directories here are built by the library's manager (spkv_pagemap_*), so
its allocation on demand, promotion and eviction are exercised as well.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import sparse_paged_kv_score_gb300 as spkv
from helpers import DEV, Dev, Offload, bf, f32, i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_paged_kv_score_gb300 import build
    build.build()
    spkv.load()


def _pagemap(table, seg_shift, n_dev, promote_every=0):
    """A manager holding `table` ([B][np_max] host int32); every promote_every-th mapped segment is
    promoted to the device tier (0: none)."""
    B, npm = table.shape
    pm = spkv.PageMap(B, npm, seg_shift=seg_shift, n_dev_segs=n_dev)
    seg = 1 << seg_shift
    k = 0
    for b in range(B):
        pm.map(b, 0, table[b])
        for s in range(0, npm, seg):
            if (table[b, s:s + seg] >= 0).any():
                if promote_every and k % promote_every == 0:
                    pm.promote(b, s)
                k += 1
    pm.sync()
    return pm


@pytest.mark.parametrize("tiers", ["host", "device", "mixed", "few_slots"])
def test_dir_calls_equal_flat_calls_262k(tiers):
    """The 262k-context workload (batch 8, 40 q / 8 kv heads, 4096 pages per request): block scores
    and sparse attention through the directory equal the flat-table calls bit for bit, with every
    segment on the host tier, every one on the device tier, half of them, or 16 device slots
    recycled by promotion (the last promotions evict the earlier ones)."""
    w = gen.long262k(seed=0)
    B, Hk, npm = w["B"], w["Hk"], w["np_max"]
    U = B * Hk
    d = Dev(w, max_units=U)
    q = bf(gen.walk_queries(w, 1)[0])
    s_flat = d.scores(q)
    sel, n_sel = d.select(s_flat, f32(w["evict"]), d.new_alive(), w["k_q"], w["k_e"])
    out_f, lse_f = d.attn(sel, n_sel, q=q)
    shift = 8
    n_segs = B * npm // (1 << shift)
    n_dev, every = {"host": (0, 0), "device": (n_segs, 1), "mixed": (n_segs, 2), "few_slots": (16, 1)}[tiers]
    pm = _pagemap(w["page_table"], shift, n_dev, every)
    s_dir = torch.full_like(s_flat, float("nan"))
    spkv.score_blocks_dir(d.cache, q, pm, d.L, s_dir)
    out_d = torch.full_like(out_f, float("nan"))
    lse_d = torch.full_like(lse_f, float("nan"))
    spkv.sparse_decode_attn_dir(d.cache, q, pm, sel, n_sel, d.L, out_d, lse_d)
    torch.cuda.synchronize()
    assert torch.equal(s_dir, s_flat)
    assert torch.equal(out_d, out_f) and torch.equal(lse_d, lse_f)
    assert d.errors() == (0, 0)
    dev_bytes, host_bytes = pm.nbytes()
    flat_bytes = B * npm * 4
    if tiers == "host":      # only the directory and the chunk table stay on the device
        assert dev_bytes < flat_bytes / 100
    pm.close()
    d.close()


def test_retrieve_through_the_directory_equals_flat():
    """Swap-in from the host pool with the host-page table in a directory (mixed tiers): the slot
    pools and slot lists equal the flat-table retrieve's, bit for bit, over a few steps."""
    w = gen.sparse_workload(4, 16, 4, 64 * 300 + 20, 24, 8, seed=17)
    d = Dev(w, max_units=16)
    offs = [Offload(d, 64), Offload(d, 64)]
    pm = _pagemap(w["page_table"], 5, 12, 3)
    alive = d.new_alive()
    ev = f32(w["evict"])
    U, stride = 16, 33
    for t in range(4):
        q = bf(gen.rows_bf16(17, 50 + t, 4 * 16).reshape(4, 16, 128))
        sel, n_sel = d.select(d.scores(q), ev, alive, 24, 8)
        outs = []
        for k, off in enumerate(offs):
            miss = torch.empty(U, stride, dtype=torch.int32, device=DEV)
            nm = torch.empty(U, dtype=torch.int32, device=DEV)
            slot = torch.empty(U, stride, dtype=torch.int32, device=DEV)
            spkv.resident_setdiff(d.cache, off.resident, sel, n_sel, miss, nm, slot)
            vic = torch.empty(U, stride, dtype=torch.int32, device=DEV)
            hist = torch.empty(U, 64, dtype=torch.int32, device=DEV)
            spkv.lru_bucket_update(d.cache, off.resident, off.ts, slot, n_sel.view(U), miss, nm, t, 1, vic, hist)
            if k == 0:
                spkv.retrieve_pages(off.slots, off.k_host, off.v_host, d.pt, miss, nm, vic, slot, n_sel, 64)
            else:
                spkv.retrieve_pages_dir(off.slots, off.k_host, off.v_host, pm, miss, nm, vic, slot, n_sel, 64)
            outs.append(slot)
        torch.cuda.synchronize()
        assert torch.equal(outs[0], outs[1])
        assert torch.equal(offs[0].k_slots, offs[1].k_slots) and torch.equal(offs[0].v_slots, offs[1].v_slots)
    for off in offs:
        assert spkv.get_device_error(off.slots) == (0, 0)
        off.close()
    pm.close()
    d.close()


def test_unmapped_pages_are_flagged_not_faulted():
    """A page whose segment was never mapped reads as -1: scoring flags SPKV_DEVERR_PHYS and scores
    it -inf; the same for a page unmapped inside a mapped segment; the rest equals the flat call."""
    w = gen.sparse_workload(2, 8, 2, 64 * 100 + 3, 8, 8, seed=5)
    d = Dev(w)
    table = w["page_table"].copy()
    table[0, 32:48] = -1          # a whole 16-page segment (shift 4) never mapped
    table[1, 7] = -1              # one page unmapped inside a mapped segment
    pm = _pagemap(table, 4, 4, 5)
    s_flat = d.scores()
    s_dir = torch.empty_like(s_flat)
    spkv.score_blocks_dir(d.cache, d.q, pm, d.L, s_dir)
    torch.cuda.synchronize()
    st, bits = d.errors()
    assert bits == spkv.DEVERR["PHYS"]
    sd, sf = s_dir.cpu().numpy(), s_flat.cpu().numpy()
    assert np.isneginf(sd[0, :, 32:48]).all() and np.isneginf(sd[1, :, 7]).all()
    keep = np.ones(sd.shape, bool)
    keep[0, :, 32:48] = False
    keep[1, :, 7] = False
    assert np.array_equal(sd[keep], sf[keep])
    pm.close()
    d.close()


def test_manager_metadata_follows_the_pages_in_use():
    """A 1M-page logical space per request with 4096 pages in use each: host segments are allocated
    only for the ranges in use (16, 17 and 17 segments of 256 ids: the last two ranges are not
    aligned), in one chunk of 64 segments; the device holds the directory, the device slots and the
    chunk table, far less than a flat table of the logical space."""
    B, npm, shift = 3, 1 << 20, 8
    starts = (0, 5000, 900_000)
    pm = spkv.PageMap(B, npm, seg_shift=shift, n_dev_segs=8)
    for b, start in enumerate(starts):
        pm.map(b, start, np.arange(4096, dtype=np.int32) + 4096 * b)
        pm.promote(b, start)
    pm.sync()
    dev_bytes, host_bytes = pm.nbytes()
    v = pm.view()
    assert v.n_host_segs == 16 + 17 + 17 and v.n_dir == npm >> shift
    assert host_bytes == 64 * (1 << shift) * 4
    flat = B * npm * 4
    assert dev_bytes == B * v.n_dir * 4 + 8 * (1 << shift) * 4 + ((B * v.n_dir + 63) // 64) * 8
    assert dev_bytes < flat / 30
    with pytest.raises(spkv.SpkvError):      # a segment with no mapped page cannot be promoted
        pm.promote(0, 500_000)
    pm.close()
