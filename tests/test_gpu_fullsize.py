"""Full-size GPU parity on the five decode workloads, in the launch configuration bench.py times
(one persistent CTA per SM for attention, one CTA per unit for the bookkeeping kernels).

Where the fp64 oracle is cheap it checks every output (attention, selection, set-difference,
LRU); where it is not (block scores over 0.5 GB of summaries, the materialised lazy oracle over
~20k rotated keys per unit), it checks a seeded sample of units.  Trajectory workloads also
check the NOSA invariants on the GPU's own selections: gamma(t) >= k_e / k and no evicted page
re-entering the eviction-head set.
"""
import math

import numpy as np
import pytest
import torch

import gen
import oracle
import sparse_paged_kv_score_gb300 as spkv
from helpers import DEV, Dev, Offload, alive_bits_to_bytes, attn_errors, bf, f32, host_bits, i32, u32_as_i32

pytestmark = pytest.mark.gpu

ATTN_MAX, ATTN_MEAN, LSE_TOL = 1e-2, 1e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_paged_kv_score_gb300 import build
    build.build()
    spkv.load()


def f64(bits):
    return gen.bf16_to_f32(bits).astype(np.float64)


def check_scores_sampled(w, s_gpu, units):
    """GPU block scores vs fp64 oracle scores on sampled units, within the fp32 bound."""
    ref = oracle.score_batch(w["q"], w["k_pool"], w["page_table"], w["seq_len"], units=units)
    q = f64(w["q"])
    G = w["G"]
    for u in units:
        b, h = divmod(int(u), w["Hk"])
        s, r = s_gpu[b, h].astype(np.float64), ref[b, h]
        assert np.array_equal(np.isinf(s), np.isinf(r))
        fin = np.isfinite(r)
        qs = np.abs(q[b, h * G:(h + 1) * G].sum(0))
        pages = w["page_table"][b][fin]
        keys = f64(w["k_pool"][h, pages]).reshape(len(pages), 4, 16, 128).mean(2)
        bound = 2e-5 * (np.abs(keys) @ qs).max(1) / math.sqrt(128) + 1e-7
        assert (np.abs(s[fin] - r[fin]) <= bound).all(), (u, np.abs(s[fin] - r[fin]).max())
    return ref


def check_select_same_scores(w, s_gpu, evict, alive_before, k_q, k_e, sel, n_sel, alive_after):
    o_sel, o_n, o_alive = oracle.select_batch(s_gpu.astype(np.float64), evict.astype(np.float64),
                                              alive_before, w["seq_len"], k_q, k_e)
    assert np.array_equal(sel, o_sel)
    assert np.array_equal(n_sel, o_n)
    assert np.array_equal(alive_after, o_alive)


def check_attn(w, out, lse, sel, n_sel, units=None):
    ro, rl = oracle.sparse_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["page_table"], sel, n_sel,
                                      w["seq_len"], units=units)
    if units is not None:
        rows = np.concatenate([np.arange(u % w["Hk"] * w["G"], (u % w["Hk"] + 1) * w["G"]) +
                               (u // w["Hk"]) * w["Hq"] for u in units])
        o, r = out.reshape(-1, 128)[rows], ro.reshape(-1, 128)[rows]
        l, rl = lse.reshape(-1)[rows], rl.reshape(-1)[rows]
    else:
        o, r, l = out, ro, lse
    mx, mean = attn_errors(o, r)
    assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (mx, mean)
    assert np.abs(l - rl).max() <= LSE_TOL
    return mx, mean


def host(x):
    return x.cpu().numpy()


# ------------------------------------------------------------------ Llama-3-8B layer (bench workload)

def test_llama8b_full_step():
    w = gen.llama8b(seed=0)
    B, Hk, Hq, npm = w["B"], w["Hk"], w["Hq"], w["np_max"]
    k_q, k_e = w["k_q"], w["k_e"]
    U = B * Hk
    L = int(w["seq_len"][0])
    d = Dev(w, max_units=U)
    # the step's own token is written at position L-1, as the bench does
    phys = w["page_table"][:, (L - 1) // 64].astype(np.int32)
    tok = np.full(B, (L - 1) % 64, np.int32)
    kn = gen.rows_bf16(3, 31, U).reshape(B, Hk, 128)
    vn = gen.rows_bf16(3, 32, U).reshape(B, Hk, 128)
    spkv.paged_kv_append(d.cache, i32(phys), i32(tok), bf(kn), bf(vn))
    for b in range(B):
        w["k_pool"][:, phys[b], tok[b]] = kn[b]
        w["v_pool"][:, phys[b], tok[b]] = vn[b]
    s = d.scores()
    alive = d.new_alive()
    sel, n_sel = d.select(s, f32(w["evict"]), alive, k_q, k_e)
    out, lse = d.attn(sel, n_sel)
    torch.cuda.synchronize()
    s_h, sel_h, n_h = host(s), host(sel), host(n_sel)
    rng = np.random.default_rng(0)
    sample = np.sort(rng.choice(U, U // 2, replace=False))     # half of the 256 units
    s_or = check_scores_sampled(w, s_h, sample)
    check_select_same_scores(w, s_h, w["evict"], np.ones((B, Hk, npm), np.uint8), k_q, k_e, sel_h, n_h,
                             alive_bits_to_bytes(host(alive).view(np.uint32), npm))
    # against the oracle's own fp64 scores: differences only among near-ties at the k-th score
    o_sel, o_n, o_alive = oracle.select_batch(s_or, w["evict"], np.ones((B, Hk, npm), np.uint8),
                                              w["seq_len"], k_q, k_e, units=sample)
    local = (L - 1) // 64
    for u in sample:
        b, h = divmod(int(u), Hk)
        E = {p for p in range(local) if o_alive[b, h, p]}
        cand = sorted((p for p in range(local) if p not in E), key=lambda p: -s_or[b, h, p])
        kth = s_or[b, h, cand[k_q - 1]]
        for p in set(sel_h[b, h, :n_h[b, h]].tolist()) ^ set(o_sel[b, h, :o_n[b, h]].tolist()):
            assert abs(s_or[b, h, p] - kth) <= 1e-5 * abs(kth)
    mx, mean = check_attn(w, host(out), host(lse), sel_h, n_h)
    # residency bookkeeping for two consecutive steps
    resident = np.full((U, 2048), -1, np.int32)
    ts = np.full((U, 2048), np.iinfo(np.int32).min, np.int32)
    r_dev, t_dev = i32(resident), i32(ts)
    stride = k_q + k_e + 1
    for t in range(2):
        miss = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        nm = torch.empty(U, dtype=torch.int32, device=DEV)
        slot = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        spkv.resident_setdiff(d.cache, r_dev, sel, n_sel, miss, nm, slot)
        vic = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        hist = torch.empty(U, 64, dtype=torch.int32, device=DEV)
        spkv.lru_bucket_update(d.cache, r_dev, t_dev, slot, n_sel.view(U), miss, nm, t, 1, vic, hist)
        o_miss, o_nm, o_slot = oracle.setdiff_batch(resident, sel_h.reshape(U, stride), n_h.reshape(U))
        assert np.array_equal(host(miss), o_miss) and np.array_equal(host(nm), o_nm)
        assert np.array_equal(host(slot), o_slot)
        resident, ts, o_vic, o_hist = oracle.lru_batch(resident, ts, o_slot, n_h.reshape(U), o_miss, o_nm, t, 1)
        assert np.array_equal(host(vic), o_vic) and np.array_equal(host(hist), o_hist)
        assert np.array_equal(host(r_dev), resident) and np.array_equal(host(t_dev), ts)
    # lazy-RoPE form on the same selected pages, presented as 8 documents x 4096 tokens
    stride = k_q + k_e + 1
    pg = np.maximum(sel_h, 0)
    phys_l = np.take_along_axis(np.broadcast_to(w["page_table"][:, None, :], (B, Hk, npm)), pg, 2)
    valid_l = np.minimum(64, L - 64 * pg).astype(np.int32)
    slot_l = (pg // 64).astype(np.int32)
    words = spkv.pack_page_words(phys_l, valid_l, slot_l)
    doc_pos = np.tile(np.arange(8, dtype=np.int32) * 4096, (B, 1))
    qpos = np.full(B, L - 1, np.int32)
    n_pages = np.full(B, stride, np.int32)
    lout = torch.empty_like(out)
    llse = torch.empty_like(lse)
    spkv.lazy_rope_decode_attn(d.cache, d.q, i32(qpos), u32_as_i32(words), i32(n_pages), i32(doc_pos),
                               500000.0, lout, llse)
    lu = np.sort(rng.choice(U, U // 2, replace=False))
    ro, rl = oracle.lazy_attn_batch(w["q"], w["k_pool"], w["v_pool"], phys_l, valid_l, slot_l, n_pages,
                                    qpos, doc_pos, 500000.0, materialise=True, units=lu)
    rows = np.concatenate([np.arange((u % Hk) * 4, (u % Hk + 1) * 4) + (u // Hk) * Hq for u in lu])
    mx2, mean2 = attn_errors(host(lout).reshape(-1, 128)[rows], ro.reshape(-1, 128)[rows])
    assert mx2 <= ATTN_MAX and mean2 <= ATTN_MEAN, (mx2, mean2)
    assert np.abs(host(llse).reshape(-1)[rows] - rl.reshape(-1)[rows]).max() <= LSE_TOL
    assert d.errors() == (0, 0)
    d.close()


# ------------------------------------------------------------------ lazy-RoPE RAG decode

def test_lazy_rag_full_size_sampled():
    w = gen.lazy_rag(seed=0)
    B, Hq, Hk = w["B"], w["Hq"], w["Hk"]
    k_pool, v_pool = bf(w["k_pool"]), bf(w["v_pool"])
    ksum = torch.zeros(Hk, w["n_phys"], 4, 128, dtype=torch.float32, device=DEV)
    cache = spkv.paged_kv_create(k_pool, v_pool, ksum, i32(w["page_cnt"]), max_units=B * Hk)
    ok = w["phys"] >= 0
    words = np.zeros(w["phys"].shape, np.uint32)
    words[ok] = spkv.pack_page_words(w["phys"][ok], w["valid"][ok], w["slot"][ok])
    out = torch.empty(B, Hq, 128, dtype=torch.float32, device=DEV)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=DEV)
    spkv.lazy_rope_decode_attn(cache, bf(w["q"]), i32(w["qpos"]), u32_as_i32(words), i32(w["n_pages"]),
                               i32(w["doc_pos"]), w["theta"], out, lse)
    torch.cuda.synchronize()
    units = np.sort(np.random.default_rng(1).choice(B * Hk, B * Hk // 2, replace=False))   # half of 512
    ro, rl = oracle.lazy_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"],
                                    w["n_pages"], w["qpos"], w["doc_pos"], w["theta"], materialise=True,
                                    units=units)
    G = w["G"]
    rows = np.concatenate([np.arange((u % Hk) * G, (u % Hk + 1) * G) + (u // Hk) * Hq for u in units])
    mx, mean = attn_errors(host(out).reshape(-1, 128)[rows], ro.reshape(-1, 128)[rows])
    assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (mx, mean)
    assert np.abs(host(lse).reshape(-1)[rows] - rl.reshape(-1)[rows]).max() <= LSE_TOL
    assert np.isfinite(host(out)).all()
    assert spkv.get_device_error(cache) == (0, 0)
    cache.close()


# ------------------------------------------------------------------ 262k context with residency

def test_long262k_residency_trajectory():
    steps = 32
    w = gen.long262k(seed=0)
    B, Hk, npm = w["B"], w["Hk"], w["np_max"]
    U = B * Hk
    k_q, k_e = w["k_q"], w["k_e"]
    stride = k_q + k_e + 1
    n_slots = w["n_slots"]
    qs = gen.walk_queries(w, steps)
    d = Dev(w, max_units=U)
    alive = d.new_alive()
    alive_h = np.ones((B, Hk, npm), np.uint8)
    resident = np.full((U, n_slots), -1, np.int32)
    ts = np.full((U, n_slots), np.iinfo(np.int32).min, np.int32)
    r_dev, t_dev = i32(resident), i32(ts)
    ev = f32(w["evict"])
    hits = []
    for t in range(steps):
        q = bf(qs[t])
        s = d.scores(q)
        sel, n_sel = d.select(s, ev, alive, k_q, k_e)
        miss = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        nm = torch.empty(U, dtype=torch.int32, device=DEV)
        slot = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        spkv.resident_setdiff(d.cache, r_dev, sel, n_sel, miss, nm, slot)
        vic = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        hist = torch.empty(U, 64, dtype=torch.int32, device=DEV)
        spkv.lru_bucket_update(d.cache, r_dev, t_dev, slot, n_sel.view(U), miss, nm, t, 1, vic, hist)
        out, lse = d.attn(sel, n_sel, q=q)
        torch.cuda.synchronize()
        s_h, sel_h, n_h = host(s), host(sel), host(n_sel)
        after = alive_bits_to_bytes(host(alive).view(np.uint32), npm)
        check_select_same_scores(w, s_h, w["evict"], alive_h, k_q, k_e, sel_h, n_h, after)
        alive_h = after
        o_miss, o_nm, o_slot = oracle.setdiff_batch(resident, sel_h.reshape(U, stride), n_h.reshape(U))
        assert np.array_equal(host(miss), o_miss) and np.array_equal(host(nm), o_nm)
        assert np.array_equal(host(slot), o_slot)
        resident, ts, o_vic, o_hist = oracle.lru_batch(resident, ts, o_slot, n_h.reshape(U), o_miss, o_nm, t, 1)
        assert np.array_equal(host(vic), o_vic) and np.array_equal(host(hist), o_hist)
        assert np.array_equal(host(r_dev), resident) and np.array_equal(host(t_dev), ts)
        hits.append(1.0 - o_nm.sum() / n_h.sum())
        if t % 4 == 0 or t == steps - 1:
            wq = dict(w)
            wq["q"] = qs[t]
            # scores over 4096 pages per unit: half of the units at the ends, a few in between
            su = np.arange(0, U, 2) if t in (0, steps - 1) else np.array([0, 13, 37, 63])
            check_scores_sampled(wq, s_h, su)
            check_attn(wq, host(out), host(lse), sel_h, n_h)
    # the query walks slowly, so most selected pages stay resident from step to step
    assert hits[0] == 0.0 and np.mean(hits[1:]) > 0.5
    assert d.errors() == (0, 0)
    d.close()


def test_long262k_offload_trajectory():
    """The same workload with the pool offloaded: pages come from pinned host memory into each
    unit's 2048 slots (retrieve_pages) and attention reads them there."""
    steps = 8
    w = gen.long262k(seed=0)
    B, Hk = w["B"], w["Hk"]
    U = B * Hk
    k_q, k_e = w["k_q"], w["k_e"]
    stride = k_q + k_e + 1
    n_slots = w["n_slots"]
    qs = gen.walk_queries(w, steps)
    d = Dev(w, max_units=U)
    off = Offload(d, n_slots)
    alive = d.new_alive()
    ev = f32(w["evict"])
    for t in range(steps):
        q = bf(qs[t])
        sel, n_sel = d.select(d.scores(q), ev, alive, k_q, k_e)
        r = off.step(sel, n_sel, t, q)
        out, lse = d.attn(sel, n_sel, q=q)
        torch.cuda.synchronize()
        assert torch.equal(r["out"], out) and torch.equal(r["lse"], lse)
        sel_h, n_h = host(sel).reshape(U, stride), host(n_sel).reshape(U)
        sl, res = host(r["slot"]), host(off.resident)
        if t == 0:
            assert np.array_equal(host(r["nm"]), n_h)   # empty buffers: everything is missing
        for u in range(U):
            n = n_h[u]
            assert ((sl[u, :n] >= 0) & (sl[u, :n] < n_slots)).all() and len(set(sl[u, :n].tolist())) == n
            assert np.array_equal(res[u, sl[u, :n]], sel_h[u, :n])
        for u in (0, 29, 63):
            b, h = divmod(u, Hk)
            n = n_h[u]
            rows = torch.from_numpy(b * n_slots + sl[u, :n].astype(np.int64)).to(DEV)
            got_k = host_bits(off.k_slots[h].index_select(0, rows))
            got_v = host_bits(off.v_slots[h].index_select(0, rows))
            src = w["page_table"][b, sel_h[u, :n]]
            assert np.array_equal(got_k, w["k_pool"][h, src]) and np.array_equal(got_v, w["v_pool"][h, src])
        if t == steps - 1:
            wq = dict(w)
            wq["q"] = qs[t]
            check_attn(wq, host(r["out"]), host(r["lse"]), host(sel), host(n_sel), units=np.array([0, 29, 63]))
    assert d.errors() == (0, 0)
    assert spkv.get_device_error(off.slots) == (0, 0)
    off.close()
    d.close()


# ------------------------------------------------------------------ NOSA trajectory

def _trajectory(w, steps, check_attn_steps, score_units=None, score_steps=()):
    B, Hk, npm = w["B"], w["Hk"], w["np_max"]
    k_q, k_e = w["k_q"], w["k_e"]
    k = k_q + k_e
    d = Dev(w, max_units=B * Hk)
    alive = d.new_alive()
    alive_h = np.ones((B, Hk, npm), np.uint8)
    L = w["seq_len"].copy()
    prev_S, dead = None, np.zeros((B, Hk, npm), bool)
    gammas = []
    e_walk = None
    for t in range(steps):
        inp = gen.traj_step_inputs(w, t, e_walk)
        e_walk = inp["evict"]
        inp["evict"] = e_walk.astype(np.float32)
        phys = np.array([w["page_table"][b, L[b] // 64] for b in range(B)], np.int32)
        tok = (L % 64).astype(np.int32)
        spkv.paged_kv_append(d.cache, i32(phys), i32(tok), bf(inp["k_new"]), bf(inp["v_new"]))
        for b in range(B):
            w["k_pool"][:, phys[b], tok[b]] = inp["k_new"][b]
            w["v_pool"][:, phys[b], tok[b]] = inp["v_new"][b]
        L += 1
        w["seq_len"] = L.copy()
        d.L.copy_(i32(L))
        q = bf(inp["q"])
        s = d.scores(q)
        sel, n_sel = d.select(s, f32(inp["evict"]), alive, k_q, k_e)
        out, lse = d.attn(sel, n_sel, q=q)
        torch.cuda.synchronize()
        s_h, sel_h, n_h = host(s), host(sel), host(n_sel)
        after = alive_bits_to_bytes(host(alive).view(np.uint32), npm)
        check_select_same_scores(w, s_h, inp["evict"], alive_h, k_q, k_e, sel_h, n_h, after)
        local = (L - 1) // 64
        for b in range(B):
            for h in range(Hk):
                E = {p for p in range(local[b]) if after[b, h, p]}
                assert not any(dead[b, h, p] for p in E), "evicted page re-entered E"
                for p in range(local[b]):
                    if alive_h[b, h, p] and not after[b, h, p]:
                        dead[b, h, p] = True
        S = [[set(sel_h[b, h, :n_h[b, h]].tolist()) for h in range(Hk)] for b in range(B)]
        if prev_S is not None:
            for b in range(B):
                for h in range(Hk):
                    R = S[b][h] - {int(local[b])}
                    if local[b] >= k:
                        g = len(R & prev_S[b][h]) / k
                        gammas.append(g)
                        assert g >= k_e / k - 1e-12
        prev_S = S
        alive_h = after
        if t in check_attn_steps:
            wq = dict(w)
            wq["q"] = inp["q"]
            check_attn(wq, host(out), host(lse), sel_h, n_h)
            su = score_units if t in score_steps else np.array([0, 5, B * Hk - 1])
            check_scores_sampled(wq, s_h, su)
    assert d.errors() == (0, 0)
    d.close()
    return gammas


def test_nosa_trajectory_64_steps():
    w = gen.nosa_traj(seed=0)
    g = _trajectory(w, 64, check_attn_steps=tuple(range(0, 64, 4)) + (63,),
                    score_units=np.arange(0, w["B"] * w["Hk"], 2), score_steps=(0, 31, 63))
    assert min(g) >= 0.75


def test_small_trajectory_crossing_page_boundaries():
    w = gen.sparse_workload(3, 16, 4, 64 * 24 - 10, 4, 6, seed=9, extra_tokens=200)
    g = _trajectory(w, 150, check_attn_steps=(0, 9, 10, 74, 149))
    assert min(g) >= 0.6 - 1e-12
