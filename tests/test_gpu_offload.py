"""GPU parity of the offload path: the full pool in pinned host memory, a slot pool on the device.

Each decode step runs score -> select -> set-difference -> LRU -> retrieve_pages (host-to-device
swap-in of the missing pages into their victim slots) -> sparse_decode_attn_slots, and compares
with the fp64 oracle: the slot list and the whole slot pool bit for bit, attention within the
attention tolerance.  Attention over the slots must also equal, bit for bit, attention over the
device-resident pool with the same selection: same kernel, same pages in the same order.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import sparse_paged_kv_score_gb300 as spkv
from sparse_paged_kv_score_gb300 import _abi
from helpers import DEV, Dev, Offload, attn_errors, bf, f32, host_bits, i32

pytestmark = pytest.mark.gpu

ATTN_MAX, ATTN_MEAN, LSE_TOL = 1e-2, 1e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_paged_kv_score_gb300 import build
    build.build()
    spkv.load()


def host(x):
    return x.cpu().numpy()


def _run(w, n_slots, steps, seed):
    B, Hk, Hq = w["B"], w["Hk"], w["Hq"]
    U = B * Hk
    k_q, k_e = w["k_q"], w["k_e"]
    stride = k_q + k_e + 1
    d = Dev(w, max_units=U)
    off = Offload(d, n_slots)
    alive = d.new_alive()
    ev = f32(w["evict"])
    # a fresh query every step, so the query-aware half of the selection changes and slots recycle
    qs = [gen.rows_bf16(seed, 950 + t, B * Hq).reshape(B, Hq, 128) for t in range(steps)]
    k_slots_h = np.zeros((Hk, B * n_slots, 64, 128), np.uint16)
    v_slots_h = np.zeros_like(k_slots_h)
    n_missing_total = 0
    for t in range(steps):
        q = bf(qs[t])
        sel, n_sel = d.select(d.scores(q), ev, alive, k_q, k_e)
        r = off.step(sel, n_sel, t, q)
        ref_out, ref_lse = d.attn(sel, n_sel, q=q)
        torch.cuda.synchronize()
        sel_h, n_h = host(sel).reshape(U, stride), host(n_sel).reshape(U)
        full = oracle.retrieve_batch(w["k_pool"], w["v_pool"], w["page_table"], host(r["miss"]), host(r["nm"]),
                                     host(r["vic"]), host(r["slot_before"]), n_h, k_slots_h, v_slots_h, n_slots)
        assert np.array_equal(host(r["slot"]), full)
        assert np.array_equal(host_bits(off.k_slots), k_slots_h)
        assert np.array_equal(host_bits(off.v_slots), v_slots_h)
        # same kernel, same pages, same order: bitwise equal to attention over the device pool
        assert torch.equal(r["out"], ref_out) and torch.equal(r["lse"], ref_lse)
        ro, rl = oracle.slot_attn_batch(qs[t], k_slots_h, v_slots_h, sel_h.reshape(B, Hk, stride),
                                        full.reshape(B, Hk, stride), n_h.reshape(B, Hk), w["seq_len"], n_slots)
        mx, mean = attn_errors(host(r["out"]), ro)
        assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (mx, mean)
        assert np.abs(host(r["lse"]) - rl).max() <= LSE_TOL
        n_missing_total += int(host(r["nm"]).sum())
    assert d.errors() == (0, 0)
    assert spkv.get_device_error(off.slots) == (0, 0)
    off.close()
    d.close()
    return n_missing_total


@pytest.mark.parametrize("seed", [0, 1])
def test_offload_trajectory_bitexact(seed):
    # 40 pages per request, 16 slots per unit: the budget of 10 + local page fits, most of the
    # context does not, so slots are recycled and pages come back after eviction
    w = gen.sparse_workload(3, 8, 2, 64 * 40 - 17, 6, 4, seed=seed)
    n = _run(w, n_slots=16, steps=12, seed=seed)
    assert n > 3 * 2 * 11   # more than the first step's misses


def test_offload_ragged_and_groups():
    # short contexts (fewer candidates than the budget: ragged selections), G = 5
    w = gen.sparse_workload(4, 10, 2, 64 * 5 - 3, 8, 4, seed=3)
    _run(w, n_slots=13, steps=5, seed=3)


def test_offload_slots_equal_to_budget():
    # exactly stride slots: every untouched slot is a victim at every step
    w = gen.sparse_workload(2, 8, 2, 64 * 30, 3, 3, seed=4)
    _run(w, n_slots=7, steps=6, seed=4)


def test_retrieve_bad_victims_flag_without_fault():
    w = gen.sparse_workload(1, 8, 2, 64 * 8, 2, 2, seed=5)
    d = Dev(w, max_units=2)
    off = Offload(d, 6)
    U, stride = 2, 5
    miss = i32(np.array([[1, 2, -1, -1, -1], [0, -1, -1, -1, -1]], np.int32))
    nm = i32(np.array([2, 1], np.int32))
    vic = i32(np.array([[0, 99, -1, -1, -1], [-7, -1, -1, -1, -1]], np.int32))   # out of range
    slot = i32(np.array([[-1, -1, 3, -1, -1], [-1, 4, -1, -1, -1]], np.int32))
    n_sel = i32(np.array([3, 2], np.int32))
    spkv.retrieve_pages(off.slots, off.k_host, off.v_host, d.pt, miss, nm, vic, slot, n_sel, 6)
    st, bits = spkv.get_device_error(off.slots)
    assert st == _abi.SPKV_EDEVICE and bits == spkv.DEVERR["SLOT"]
    # the one valid copy happened; the rest were skipped
    got = host_bits(off.k_slots)
    assert np.array_equal(got[0, 0], w["k_pool"][0, w["page_table"][0, 1]])
    assert host(slot)[0].tolist() == [0, -1, 3, -1, -1]
    off.close()
    d.close()
