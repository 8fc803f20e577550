"""The allocation-free form of sparse decode attention.

Some callers cannot allocate device memory at all: an inference engine that owns every byte of
device memory through its own allocator and forbids cudaMalloc once serving starts, or code
that may not create a library handle (creating one allocates the handle's split-K workspace).
sparse_decode_attn_noalloc serves them: it takes the pool directly, allocates nothing, and keeps
its split-K scratch in a fixed device array inside the library.  These tests call it through the
C ABI and check its output element by element against the fp64 oracle, on calls in a row that
reuse the scratch the previous call left behind: at the scratch's unit limit (512 units), with
the largest group (16 query heads per kv head, whose kernel keeps 16 heads per scratch record),
and with selections long enough that every unit is split over many chunks of the page sequence.
They also check that the handle-based sparse_decode_attn returns the same values, that a batch
larger than the scratch is refused, and that a call without an error word is refused (errors in
the device data are reported only there).  The file name makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import sparse_paged_kv_score_gb300 as spkv
from helpers import DEV, Dev, attn_errors, bf, f32, i32

pytestmark = pytest.mark.gpu

ATTN_MAX, ATTN_MEAN, LSE_TOL = 1e-2, 1e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_paged_kv_score_gb300 import build
    build.build()
    spkv.load()


def _noalloc_vs_oracle(d: Dev, sel, n_sel, q_np, err):
    """One no-alloc call on q_np; its output against the oracle, fed the same selection."""
    w = d.w
    q = bf(q_np)
    out = torch.full((d.B, d.Hq, 128), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((d.B, d.Hq), float("nan"), dtype=torch.float32, device=DEV)
    spkv.sparse_decode_attn_noalloc(d.k_pool, d.v_pool, q, d.pt, sel, n_sel, d.L, out, lse, err)
    torch.cuda.synchronize()
    ro, rl = oracle.sparse_attn_batch(q_np, w["k_pool"], w["v_pool"], w["page_table"], sel.cpu().numpy(),
                                      n_sel.cpu().numpy(), w["seq_len"])
    mx, mean = attn_errors(out.cpu().numpy(), ro)
    assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (mx, mean)
    assert np.abs(lse.cpu().numpy() - rl).max() <= LSE_TOL
    return out, lse, q


@pytest.mark.parametrize("case", [
    # (B, Hq, Hk, context, k_q, k_e): 512 units (the limit), G = 4
    (64, 32, 8, 64 * 40 + 11, 16, 16),
    # G = 16: one kv head per 16 query heads, 256 units
    (128, 32, 2, 64 * 30 + 5, 12, 12),
    # 16 units of 601 selected pages: each unit spans many static ranges and dynamic chunks
    (2, 32, 8, 64 * 640 + 33, 300, 300),
])
def test_noalloc_matches_oracle_on_calls_in_a_row(case):
    B, Hq, Hk, L, k_q, k_e = case
    w = gen.sparse_workload(B, Hq, Hk, L, k_q, k_e, seed=31 + B, outlier_p=0.01)
    d = Dev(w, max_units=B * Hk)
    sel, n_sel = d.select(d.scores(), f32(w["evict"]), d.new_alive(), k_q, k_e)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for call in range(2):
        q_np = w["q"] if call == 0 else gen.rows_bf16(77 + call, 1, B * Hq).reshape(B, Hq, 128)
        out, lse, q = _noalloc_vs_oracle(d, sel, n_sel, q_np, err)
        # and the handle-based entry point on the same inputs returns the same values
        ref_out, ref_lse = d.attn(sel, n_sel, q=q)
        torch.cuda.synchronize()
        assert np.abs(out.cpu().numpy() - ref_out.cpu().numpy()).max() <= 1e-5
        assert np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy()).max() <= 1e-5
    assert int(err.item()) == 0
    assert d.errors() == (0, 0)
    d.close()


def test_noalloc_smaller_call_after_a_larger_one():
    """512 units, then 24 units, then 512 again: the records the larger call left in the scratch
    (for units the smaller call does not have) must not leak into the smaller call's results."""
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    big = gen.sparse_workload(64, 32, 8, 64 * 36 + 7, 16, 16, seed=5, outlier_p=0.01)
    small = gen.sparse_workload(3, 32, 8, 64 * 90 + 40, 40, 20, seed=6)
    devs = [Dev(big, max_units=512), Dev(small, max_units=24)]
    sels = [d.select(d.scores(), f32(d.w["evict"]), d.new_alive(), d.w["k_q"], d.w["k_e"]) for d in devs]
    for i in (0, 1, 0):
        d, (sel, n_sel) = devs[i], sels[i]
        _noalloc_vs_oracle(d, sel, n_sel, d.w["q"], err)
    assert int(err.item()) == 0
    for d in devs:
        d.close()


def test_noalloc_reports_bad_pages_in_the_callers_error_word():
    """A selected page past the request's context is skipped and flagged in dev_err; the rest
    of the unit is still attended (checked against the oracle on the pages that remain)."""
    w = gen.sparse_workload(2, 8, 2, 64 * 20 + 3, 6, 6, seed=9)
    d = Dev(w, max_units=4)
    sel, n_sel = d.select(d.scores(), f32(w["evict"]), d.new_alive(), 6, 6)
    bad = sel.clone()
    bad[0, 1, 0] = 10_000                              # logical page id out of range
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty(2, 8, 128, dtype=torch.float32, device=DEV)
    lse = torch.empty(2, 8, dtype=torch.float32, device=DEV)
    spkv.sparse_decode_attn_noalloc(d.k_pool, d.v_pool, d.q, d.pt, bad, n_sel, d.L, out, lse, err)
    torch.cuda.synchronize()
    assert int(err.item()) & spkv.DEVERR["PAGE_ID"]
    # the oracle on the unit without its bad first page
    keep = sel.cpu().numpy().copy()
    nk = n_sel.cpu().numpy().copy()
    keep[0, 1, :-1] = keep[0, 1, 1:]
    keep[0, 1, -1] = -1
    nk[0, 1] -= 1
    ro, rl = oracle.sparse_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["page_table"], keep, nk, w["seq_len"])
    mx, mean = attn_errors(out.cpu().numpy(), ro)
    assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (mx, mean)
    d.close()


def _tiny_args(B, Hk=8):
    k = torch.zeros(Hk, 1, 64, 128, dtype=torch.bfloat16, device=DEV)
    q = torch.zeros(B, Hk * 4, 128, dtype=torch.bfloat16, device=DEV)
    pt = torch.zeros(B, 1, dtype=torch.int32, device=DEV)
    sel = torch.zeros(B, Hk, 1, dtype=torch.int32, device=DEV)
    n_sel = torch.ones(B, Hk, dtype=torch.int32, device=DEV)
    L = torch.ones(B, dtype=torch.int32, device=DEV)
    out = torch.zeros(B, Hk * 4, 128, dtype=torch.float32, device=DEV)
    lse = torch.zeros(B, Hk * 4, dtype=torch.float32, device=DEV)
    return k, q, pt, sel, n_sel, L, out, lse


def test_noalloc_refuses_batches_beyond_its_scratch():
    k, q, pt, sel, n_sel, L, out, lse = _tiny_args(65)      # 520 units > 512
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(spkv.SpkvError) as e:
        spkv.sparse_decode_attn_noalloc(k, k, q, pt, sel, n_sel, L, out, lse, err)
    assert e.value.status == -6


def test_noalloc_refuses_a_call_without_an_error_word():
    k, q, pt, sel, n_sel, L, out, lse = _tiny_args(2)
    with pytest.raises(ValueError):
        spkv.sparse_decode_attn_noalloc(k, k, q, pt, sel, n_sel, L, out, lse, None)
    # through the C ABI directly: a NULL error word is an argument error, nothing is launched
    lib = spkv.load()
    st = lib.sparse_decode_attn_noalloc(k.data_ptr(), k.data_ptr(), 8, 1, q.data_ptr(), 2, 32, pt.data_ptr(), 1,
                                        sel.data_ptr(), n_sel.data_ptr(), 1, L.data_ptr(), out.data_ptr(),
                                        lse.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert st == -1


def test_noalloc_refuses_host_memory():
    k, q, pt, sel, n_sel, L, out, lse = _tiny_args(2)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    host_out = torch.zeros(2, 32, 128, dtype=torch.float32).pin_memory()
    lib = spkv.load()
    st = lib.sparse_decode_attn_noalloc(k.data_ptr(), k.data_ptr(), 8, 1, q.data_ptr(), 2, 32, pt.data_ptr(), 1,
                                        sel.data_ptr(), n_sel.data_ptr(), 1, L.data_ptr(), host_out.data_ptr(),
                                        lse.data_ptr(), err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == -1
