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
