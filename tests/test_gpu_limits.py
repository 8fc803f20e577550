"""The decode path at the largest sizes one call accepts, and the host-side rejection just past
them (no kernel runs for a rejected call).

Units: one call serves at most 4096 (request, kv head) units (the attention kernel's prefix table
and the handle's workspace are sized for it); 512 requests x 8 kv heads fill it exactly, on short
ragged contexts so the pools stay small."""
import numpy as np
import pytest
import torch

import gen
import oracle
import sparse_paged_kv_score_gb300 as spkv
from helpers import DEV, Dev, attn_errors, bf, f32, i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_paged_kv_score_gb300 import build
    build.build()
    spkv.load()


def test_4096_units_full_step_and_rejection_past_it():
    B, Hq, Hk = 512, 16, 8
    w = gen.sparse_workload(B, Hq, Hk, 64 * 3 + 5, 1, 1, seed=21)
    w["seq_len"] = (64 + 1 + (np.arange(B) * 37) % (64 * 3 + 5 - 64)).astype(np.int32)   # ragged: 2..4 pages
    U = B * Hk
    d = Dev(w, max_units=U)
    s = d.scores()
    k_q, k_e = w["k_q"], w["k_e"]
    stride = k_q + k_e + 1
    # the fused selection + residency kernel on every unit
    alive = d.new_alive()
    sel = torch.empty(B, Hk, stride, dtype=torch.int32, device=DEV)
    n_sel = torch.empty(B, Hk, dtype=torch.int32, device=DEV)
    resident = torch.full((U, 16), -1, dtype=torch.int32, device=DEV)
    ts = torch.full((U, 16), np.iinfo(np.int32).min, dtype=torch.int32, device=DEV)
    missing, slot, victims = (torch.empty(U, stride, dtype=torch.int32, device=DEV) for _ in range(3))
    n_missing = torch.empty(U, dtype=torch.int32, device=DEV)
    hist = torch.empty(U, 64, dtype=torch.int32, device=DEV)
    spkv.select_resident_update(d.cache, s, f32(w["evict"]), alive, d.L, k_q, k_e, sel, n_sel, resident, ts, 0, 1,
                                missing, n_missing, slot, victims, hist)
    out, lse = d.attn(sel, n_sel)
    torch.cuda.synchronize()
    assert d.errors() == (0, 0)
    s_h, sel_h, n_h = s.cpu().numpy(), sel.cpu().numpy(), n_sel.cpu().numpy()
    # selection: bit-exact with the oracle on the GPU's own scores, every unit
    o_sel, o_n, _ = oracle.select_batch(s_h.astype(np.float64), w["evict"].astype(np.float64),
                                        np.ones((B, Hk, w["np_max"]), np.uint8), w["seq_len"], k_q, k_e)
    assert np.array_equal(sel_h, o_sel) and np.array_equal(n_h, o_n)
    assert np.array_equal(n_missing.cpu().numpy(), n_h.reshape(U))   # all slots started empty
    # attention on sampled units, including the first and the last
    units = np.unique(np.concatenate([[0, U - 1], np.random.default_rng(21).choice(U, 62, replace=False)]))
    ro, rl = oracle.sparse_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["page_table"], sel_h, n_h, w["seq_len"],
                                      units=units.astype(np.int32))
    G = Hq // Hk
    rows = np.concatenate([(u // Hk) * Hq + (u % Hk) * G + np.arange(G) for u in units])
    o, r = out.cpu().numpy().reshape(-1, 128)[rows], ro.reshape(-1, 128)[rows]
    mx, mean = attn_errors(o, r)
    assert mx <= 1e-2 and mean <= 1e-3, (mx, mean)
    assert np.abs(lse.cpu().numpy().reshape(-1)[rows] - rl.reshape(-1)[rows]).max() <= 1e-3
    # one unit more than the handle holds is refused before any launch
    q1 = torch.zeros(B + 1, Hq, 128, dtype=torch.bfloat16, device=DEV)
    pt1 = torch.zeros(B + 1, w["np_max"], dtype=torch.int32, device=DEV)
    sel1 = torch.zeros(B + 1, Hk, stride, dtype=torch.int32, device=DEV)
    n1 = torch.ones(B + 1, Hk, dtype=torch.int32, device=DEV)
    L1 = torch.full((B + 1,), 65, dtype=torch.int32, device=DEV)
    o1 = torch.empty(B + 1, Hq, 128, dtype=torch.float32, device=DEV)
    l1 = torch.empty(B + 1, Hq, dtype=torch.float32, device=DEV)
    with pytest.raises(spkv.SpkvError, match="EINVAL"):
        spkv.sparse_decode_attn(d.cache, q1, pt1, sel1, n1, L1, o1, l1)
    d.close()
    # and a handle cannot be made for more than 4096 units
    with pytest.raises(spkv.SpkvError, match="EINVAL"):
        spkv.paged_kv_create(d.k_pool, d.v_pool, d.ksum, d.cnt, max_units=U + 1)


def test_selection_at_32768_pages_and_4096_entries():
    """The CTA form of the selection at its largest context (32768 pages, 2M tokens) and largest
    list (k_q + k_e + 1 = 4096), bit-exact with the oracle on the same scores; one page or one
    list entry more is refused.  Selection reads only scores, so the pool is a tiny one."""
    from helpers import alive_bits_to_bytes, alive_bytes_to_bits, u32_as_i32
    small = gen.sparse_workload(2, 4, 2, 64 * 4, 1, 1, seed=5)
    d = Dev(small)
    B, Hk, npm = 2, 2, 32768
    rng = np.random.default_rng(32768)
    seq = np.array([64 * npm, 64 * npm - 1000], np.int32)
    for k_q, k_e in [(64, 64), (2000, 2095)]:
        s = (np.round(rng.standard_normal((B, Hk, npm)) * 8) / 8).astype(np.float32)   # many exact ties
        e = (np.round(rng.standard_normal((B, Hk, npm)) * 4) / 4).astype(np.float32)
        alive = rng.random((B, Hk, npm)) < 0.5
        alive_dev = u32_as_i32(alive_bytes_to_bits(alive.astype(np.uint8)))
        stride = k_q + k_e + 1
        sel = torch.empty(B, Hk, stride, dtype=torch.int32, device=DEV)
        n_sel = torch.empty(B, Hk, dtype=torch.int32, device=DEV)
        spkv.select_topk(d.cache, f32(s), f32(e), alive_dev, i32(seq), k_q, k_e, sel, n_sel)
        o_sel, o_n, o_alive = oracle.select_batch(s.astype(np.float64), e.astype(np.float64), alive.astype(np.uint8),
                                                  seq, k_q, k_e)
        assert np.array_equal(sel.cpu().numpy(), o_sel) and np.array_equal(n_sel.cpu().numpy(), o_n)
        assert np.array_equal(alive_bits_to_bytes(alive_dev.cpu().numpy().view(np.uint32), npm), o_alive)
    assert d.errors() == (0, 0)
    # past either limit: refused before any launch
    s1 = torch.zeros(B, Hk, npm + 1, dtype=torch.float32, device=DEV)
    a1 = torch.zeros(B, Hk, (npm + 1 + 31) // 32, dtype=torch.int32, device=DEV)
    sel1 = torch.empty(B, Hk, 3, dtype=torch.int32, device=DEV)
    n1 = torch.empty(B, Hk, dtype=torch.int32, device=DEV)
    with pytest.raises(spkv.SpkvError, match="EINVAL"):
        spkv.select_topk(d.cache, s1, s1, a1, i32(seq), 1, 1, sel1, n1)
    s2 = torch.zeros(B, Hk, 8192, dtype=torch.float32, device=DEV)
    a2 = torch.zeros(B, Hk, 8192 // 32, dtype=torch.int32, device=DEV)
    sel2 = torch.empty(B, Hk, 4097, dtype=torch.int32, device=DEV)
    with pytest.raises(spkv.SpkvError, match="EINVAL"):
        spkv.select_topk(d.cache, s2, s2, a2, i32(seq), 2000, 2096, sel2, n1)
    d.close()


@pytest.mark.parametrize("np_max", [1025, 1536, 2047, 2048, 2049, 4095, 4096, 5000, 8192, 8193, 16384, 16385, 20000])
def test_selection_cta_form_across_sizes(np_max):
    """The CTA form of the selection (more than 1024 pages: 512 threads of 4, 8, 16 or 32 pages,
    then 1024 threads of 32) at the edges of each page-per-thread size, bit-exact with the oracle on
    the same scores: coarse scores with many exact ties and -0.0, random alive masks, ragged
    contexts, budgets from 0 to more than the candidates.  Sizes that are not a multiple of 4, and
    score rows that start off a 16-byte boundary, take the per-element loads."""
    from helpers import alive_bits_to_bytes, alive_bytes_to_bits, u32_as_i32
    small = gen.sparse_workload(3, 4, 2, 64 * 4, 1, 1, seed=6)
    d = Dev(small)
    B, Hk = 3, 2
    rng = np.random.default_rng(np_max)
    seq = np.array([64 * np_max, max(1, 64 * np_max - 70), int(rng.integers(1, 64 * np_max + 1))], np.int32)
    for k_q, k_e, offset in [(64, 64, 0), (0, 7, 0), (9, 0, 1), (min(np_max + 3, 4093), 2, 0), (300, 200, 1)]:
        s = (np.round(rng.standard_normal((B, Hk, np_max)) * 2) / 2).astype(np.float32)
        s[rng.random(s.shape) < 0.1] = -0.0
        e = (np.round(rng.standard_normal((B, Hk, np_max)) * 3) / 3).astype(np.float32)
        alive = rng.random((B, Hk, np_max)) < 0.7
        alive_dev = u32_as_i32(alive_bytes_to_bits(alive.astype(np.uint8)))
        # offset 1: both score rows start one float past a 16-byte boundary
        sb = torch.zeros(B * Hk * np_max + 4, dtype=torch.float32, device=DEV)
        eb = torch.zeros_like(sb)
        s_dev = sb[offset:offset + B * Hk * np_max].view(B, Hk, np_max)
        e_dev = eb[offset:offset + B * Hk * np_max].view(B, Hk, np_max)
        s_dev.copy_(f32(s))
        e_dev.copy_(f32(e))
        stride = k_q + k_e + 1
        sel = torch.empty(B, Hk, stride, dtype=torch.int32, device=DEV)
        n_sel = torch.empty(B, Hk, dtype=torch.int32, device=DEV)
        spkv.select_topk(d.cache, s_dev, e_dev, alive_dev, i32(seq), k_q, k_e, sel, n_sel)
        o_sel, o_n, o_alive = oracle.select_batch(s.astype(np.float64), e.astype(np.float64), alive.astype(np.uint8),
                                                  seq, k_q, k_e)
        assert np.array_equal(sel.cpu().numpy(), o_sel) and np.array_equal(n_sel.cpu().numpy(), o_n)
        assert np.array_equal(alive_bits_to_bytes(alive_dev.cpu().numpy().view(np.uint32), np_max), o_alive)
    assert d.errors() == (0, 0)
    d.close()
