"""Pins for the fp64 oracle, against things other than the oracle itself.

Each pin is chosen so that a plausible slip in the oracle fails at least one of them:

* page word      -- exhaustive per-field round trip, fixed known words, range rejection.
* sub-block mean -- closed form on integer-valued keys; numpy mean; partial / empty sub-blocks.
* block score    -- pooling linearity (the mean of the token scores of a sub-block equals the
                    score of its mean key), brute force in numpy over all pages; a constructed
                    page whose best sub-block is known; -inf at and after the local page.
* selection      -- the defining property of a top-k under (score desc, page asc), tie cases,
                    alive-bit updates, padding; the NOSA locality bound gamma(t) >= k_e/k and
                    "an evicted page never re-enters" over random trajectories that cross page
                    boundaries; sparse == dense when the budget covers every page.
* attention      -- scipy logsumexp/softmax; identical keys give the mean of V; a single token;
                    page-order invariance; the split/merge identity of the LSE statistics.
* RoPE / lazy    -- R(0) = I, R(a)R(b) = R(a+b), norm preservation, the theta_0 = 1 pair,
                    dependence on n - m only, lazy == materialised, P = 0 reduces to plain
                    attention.
* set-difference -- Python sets.
* bucketed LRU   -- bucket-by-bucket brute force, plus invariants (victims distinct, untouched,
                    all selected pages resident afterwards, histogram sums to the slot count).
"""
import itertools
import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import gen
import oracle

D, PAGE = 128, 64


def bf(x):
    return gen.f32_to_bf16(np.asarray(x, np.float32))


def f(x):
    return gen.bf16_to_f32(x).astype(np.float64)


# ------------------------------------------------------------------------------ page word

def test_meta_known_words():
    assert oracle.meta_pack(0, 1, 0) == 0
    assert oracle.meta_pack(1, 64, 0) == 0x00FC0001
    assert oracle.meta_pack(0x3FFFF, 64, 255) == 0xFFFFFFFF
    assert oracle.meta_pack(5, 2, 3) == (5 | (1 << 18) | (3 << 24))


@pytest.mark.parametrize("field", ["phys", "valid", "slot"])
def test_meta_roundtrip_each_field_exhaustive(field):
    rng = np.random.default_rng(1)
    ranges = {"phys": range(1 << 18), "valid": range(1, 65), "slot": range(256)}
    others = {k: int(rng.integers(r.start, r.stop)) for k, r in ranges.items()}
    for v in ranges[field]:
        args = dict(others)
        args[field] = v
        w = oracle.meta_pack(args["phys"], args["valid"], args["slot"])
        assert oracle.meta_unpack(w) == (args["phys"], args["valid"], args["slot"])


def test_meta_roundtrip_random_and_rejects():
    rng = np.random.default_rng(2)
    for _ in range(3000):
        p, v, s = int(rng.integers(0, 1 << 18)), int(rng.integers(1, 65)), int(rng.integers(0, 256))
        assert oracle.meta_unpack(oracle.meta_pack(p, v, s)) == (p, v, s)
    for bad in [(-1, 1, 0), (1 << 18, 1, 0), (0, 0, 0), (0, 65, 0), (0, 1, 256), (0, 1, -1)]:
        with pytest.raises(ValueError):
            oracle.meta_pack(*bad)


# ------------------------------------------------------------------------------ pooling

def test_page_means_closed_form():
    t = np.arange(PAGE)[:, None]
    page = bf(np.broadcast_to((t % 16) - 7.0, (PAGE, D)))     # each sub-block holds -7..8
    mean, cnt = oracle.page_means(page, 64)
    assert cnt.tolist() == [16, 16, 16, 16]
    assert np.all(mean == 0.5)
    mean, cnt = oracle.page_means(page, 40)                    # rows 32..39 hold -7..0
    assert cnt.tolist() == [16, 16, 8, 0]
    assert np.all(mean[:2] == 0.5) and np.all(mean[2] == -3.5) and np.all(mean[3] == 0.0)


def test_page_means_numpy():
    page = gen.rows_bf16(3, 1, PAGE)
    mean, _ = oracle.page_means(page, 64)
    ref = f(page).reshape(4, 16, D).mean(axis=1)
    assert np.allclose(mean, ref, rtol=0, atol=1e-12)


def _scores_bruteforce(q, kplane, pt_row, L, np_out):
    """Pooled token scores: for each sub-block, the mean over its 16 tokens of
    sum_g q_g . k_t / sqrt(d); then the max over the 4 sub-blocks."""
    local = (L - 1) // PAGE
    out = np.full(np_out, -np.inf)
    qf = f(q)
    for p in range(min(local, np_out)):
        keys = f(kplane[pt_row[p]])                  # 64 x 128
        tok = (keys @ qf.T).sum(axis=1) / math.sqrt(D)    # per-token group score
        out[p] = tok.reshape(4, 16).mean(axis=1).max()
    return out


def test_score_unit_pooling_linearity_bruteforce():
    w = gen.sparse_workload(1, 8, 2, 1000, 4, 4, seed=11, outlier_p=0.05)
    for h in range(2):
        q = w["q"][0, h * 4:(h + 1) * 4]
        s = oracle.score_unit(q, w["k_pool"][h], w["page_table"][0], 1000, w["np_max"])
        ref = _scores_bruteforce(q, w["k_pool"][h], w["page_table"][0], 1000, w["np_max"])
        assert np.array_equal(np.isinf(s), np.isinf(ref))
        fin = np.isfinite(ref)
        assert np.allclose(s[fin], ref[fin], rtol=1e-12, atol=1e-12)
    # local page = (1000-1)//64 = 15; pages 15.. are not candidates
    assert np.isinf(s[15:]).all() and np.isfinite(s[:15]).all()


def test_score_unit_picks_best_subblock_and_sums_group():
    # one page; sub-block 2 has mean +1 on dim 0, the others -1; q_g = e_0 for both heads
    page = np.full((PAGE, D), 0.0, np.float32)
    page[:, 0] = -1.0
    page[32:48, 0] = 1.0
    kplane = bf(page)[None]                         # n_phys = 1
    q = bf(np.eye(1, D, 0).repeat(2, 0))            # G = 2, both e_0
    s = oracle.score_unit(q, kplane, np.array([0, 0], np.int32), 2 * PAGE, 2)
    assert s[0] == pytest.approx(2.0 / math.sqrt(D), abs=1e-15)   # (1 + 1) / sqrt(128)
    assert s[1] == -np.inf


# ------------------------------------------------------------------------------ selection

def _assert_topk(chosen, pool, sc, k):
    chosen, pool = set(chosen), set(pool)
    assert chosen <= pool and len(chosen) == min(k, len(pool))
    for a in chosen:
        for b in pool - chosen:
            assert (sc[a] > sc[b]) or (sc[a] == sc[b] and a < b)


@pytest.mark.parametrize("seed", range(12))
def test_select_topk_definition_with_ties(seed):
    rng = np.random.default_rng(seed)
    npg = int(rng.integers(3, 40))
    L = int(rng.integers(1, npg * PAGE + 1))
    local = (L - 1) // PAGE
    s = rng.integers(-3, 4, npg).astype(np.float64)      # many ties
    e = rng.integers(-3, 4, npg).astype(np.float64)
    alive = (rng.random(npg) < 0.7).astype(np.uint8)
    k_q, k_e = int(rng.integers(0, 6)), int(rng.integers(0, 6))
    sel, n, alive2 = oracle.select_unit(s, e, alive, L, k_q, k_e)
    cand = list(range(min(local, npg)))
    A = [p for p in cand if alive[p]]
    E = [p for p in A if alive2[p]]
    _assert_topk(E, A, e, k_e)
    # unselected alive candidates die; non-candidates keep their bit
    assert all(alive2[p] == 0 for p in set(A) - set(E))
    assert np.array_equal(alive2[min(local, npg):], alive[min(local, npg):])
    R = [int(x) for x in sel[:n - 1]]
    Q = sorted(set(R) - set(E))
    _assert_topk(Q, [p for p in cand if p not in E], s, k_q)
    assert R == sorted(R) and sel[n - 1] == local and (sel[n:] == -1).all()
    assert len(R) == len(set(R)) == len(E) + len(Q)


def _run_traj(seed, L0, steps, k_e, k_q, npg):
    rng = np.random.default_rng(seed)
    e = rng.normal(size=npg)
    alive = np.ones(npg, np.uint8)
    prev_S, dead = None, set()
    k = k_e + k_q
    gammas = []
    for t in range(steps):
        L = L0 + t + 1
        e = e + 0.1 * rng.normal(size=npg)
        s = rng.normal(size=npg)
        before = alive.copy()
        sel, n, alive = oracle.select_unit(s, e, alive, L, k_q, k_e)
        local = (L - 1) // PAGE
        E = {p for p in range(local) if alive[p]}
        assert not (E & dead), "an evicted page re-entered the eviction-head set"
        assert all(before[p] for p in E)
        dead |= {p for p in range(local) if before[p] and not alive[p]}
        R = set(int(x) for x in sel[:n - 1])
        S = R | {local}
        if prev_S is not None and local >= k:
            gamma = len(R & prev_S) / k
            gammas.append(gamma)
            assert gamma >= k_e / k - 1e-12
        prev_S = S
    return gammas


@pytest.mark.parametrize("seed", range(4))
def test_locality_and_monotone_eviction_across_page_boundaries(seed):
    # 150 steps starting 20 tokens before a page boundary: crosses 3 boundaries
    g = _run_traj(seed, L0=40 * PAGE - 20, steps=150, k_e=12, k_q=4, npg=45)
    assert len(g) == 149 and min(g) >= 0.75


def test_locality_small_budgets():
    _run_traj(9, L0=10 * PAGE - 3, steps=200, k_e=3, k_q=5, npg=15)


# ------------------------------------------------------------------------------ attention

def _dense_ref(q, kplane, vplane, phys, valid):
    keys = np.concatenate([f(kplane[p, :v]) for p, v in zip(phys, valid)])
    vals = np.concatenate([f(vplane[p, :v]) for p, v in zip(phys, valid)])
    z = f(q) @ keys.T / math.sqrt(D)
    return softmax(z, axis=1) @ vals, logsumexp(z, axis=1)


def test_attn_scipy_bruteforce():
    w = gen.sparse_workload(1, 8, 2, 700, 4, 4, seed=5, outlier_p=0.05)
    phys = w["page_table"][0, [0, 3, 5, 10]]
    valid = np.array([64, 64, 64, 700 - 640], np.int32)
    q = w["q"][0, :4]
    out, lse = oracle.attn_unit(q, w["k_pool"][0], w["v_pool"][0], phys, valid)
    ro, rl = _dense_ref(q, w["k_pool"][0], w["v_pool"][0], phys, valid)
    assert np.allclose(out, ro, atol=1e-12) and np.allclose(lse, rl, atol=1e-12)


def test_attn_identical_keys_and_single_token():
    kplane = bf(np.tile(gen.normal_f32(0, 1, D), (2, PAGE, 1)))     # all keys the same
    vplane = gen.rows_bf16(0, 2, 2 * PAGE).reshape(2, PAGE, D)
    q = gen.rows_bf16(0, 3, 3)
    out, lse = oracle.attn_unit(q, kplane, vplane, [0, 1], [64, 30])
    vals = np.concatenate([f(vplane[0]), f(vplane[1, :30])])
    assert np.allclose(out, vals.mean(0)[None], atol=1e-12)
    z = f(q) @ f(kplane[0, 0]) / math.sqrt(D)
    assert np.allclose(lse, z + math.log(94), atol=1e-12)
    out1, lse1 = oracle.attn_unit(q, kplane, vplane, [1], [1])
    assert np.allclose(out1, f(vplane[1, 0])[None], atol=0) and np.allclose(lse1, z, atol=1e-13)
    out0, lse0 = oracle.attn_unit(q, kplane, vplane, [], [])
    assert (out0 == 0).all() and (lse0 == -np.inf).all()


def test_attn_page_order_invariance_and_lse_merge():
    w = gen.sparse_workload(1, 4, 1, 64 * 9, 2, 2, seed=8)
    K, V, q = w["k_pool"][0], w["v_pool"][0], w["q"][0]
    phys = w["page_table"][0]
    valid = np.full(9, 64, np.int32)
    o, l = oracle.attn_unit(q, K, V, phys, valid)
    perm = np.random.default_rng(0).permutation(9)
    o2, l2 = oracle.attn_unit(q, K, V, phys[perm], valid[perm])
    assert np.allclose(o, o2, atol=1e-13) and np.allclose(l, l2, atol=1e-13)
    oa, la = oracle.attn_unit(q, K, V, phys[:4], valid[:4])
    ob, lb = oracle.attn_unit(q, K, V, phys[4:], valid[4:])
    lm = np.logaddexp(la, lb)
    om = oa * np.exp(la - lm)[:, None] + ob * np.exp(lb - lm)[:, None]
    assert np.allclose(om, o, atol=1e-12) and np.allclose(lm, l, atol=1e-12)


def test_sparse_equals_dense_when_budget_covers_everything():
    w = gen.sparse_workload(1, 8, 2, 64 * 6 + 10, 8, 8, seed=4)
    s = oracle.score_batch(w["q"], w["k_pool"], w["page_table"], w["seq_len"])
    sel, n_sel, _ = oracle.select_batch(s, w["evict"], np.ones_like(w["evict"], np.uint8),
                                        w["seq_len"], 8, 8)
    assert (n_sel == 7).all() and (sel[..., :7] == np.arange(7)).all()
    out, lse = oracle.sparse_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["page_table"], sel,
                                        n_sel, w["seq_len"])
    for h in range(2):
        ro, rl = _dense_ref(w["q"][0, 4 * h:4 * h + 4], w["k_pool"][h], w["v_pool"][h],
                            w["page_table"][0, :7], [64] * 6 + [10])
        assert np.allclose(out[0, 4 * h:4 * h + 4], ro, atol=1e-12)
        assert np.allclose(lse[0, 4 * h:4 * h + 4], rl, atol=1e-12)


# ------------------------------------------------------------------------------ RoPE / lazy

def test_rope_identities():
    x = gen.normal_f64(1, 1, D)
    th = 500000.0
    assert np.allclose(oracle.rope(x, 0, th), x, atol=0)
    a, b = 1234.0, -567.0
    assert np.allclose(oracle.rope(oracle.rope(x, a, th), b, th), oracle.rope(x, a + b, th), atol=1e-10)
    assert abs(np.linalg.norm(oracle.rope(x, 98765.0, th)) - np.linalg.norm(x)) < 1e-11
    # dimension pair 0 has frequency theta^0 = 1: e_0 -> (cos p) e_0 + (sin p) e_64
    e0 = np.eye(1, D, 0)[0]
    y = oracle.rope(e0, 2.0, th)
    assert y[0] == pytest.approx(math.cos(2.0), abs=1e-15)
    assert y[64] == pytest.approx(math.sin(2.0), abs=1e-15)
    assert np.count_nonzero(y) == 2
    # the last pair turns slowest: theta^(-126/128)
    e63 = np.eye(1, D, 63)[0]
    y = oracle.rope(e63, 1e5, th)
    ang = 1e5 * th ** (-126 / 128)
    assert y[63] == pytest.approx(math.cos(ang), abs=1e-12)
    assert y[127] == pytest.approx(math.sin(ang), abs=1e-12)


def test_rope_scores_depend_on_offset_only():
    q, k = gen.normal_f64(2, 1, D), gen.normal_f64(2, 2, D)
    th = 500000.0
    base = oracle.rope(q, 40000, th) @ oracle.rope(k, 1000, th)
    for n, m in [(39000, 0), (45000, 6000), (100000, 61000)]:
        assert oracle.rope(q, n, th) @ oracle.rope(k, m, th) == pytest.approx(base, abs=1e-9)


def _lazy_case(seed):
    w = gen.lazy_rag(seed=seed, B=2, Hq=4, Hk=2, n_docs=6, docs_per_req=3, min_len=70, max_len=200,
                     theta=500000.0)
    return w


def test_lazy_equals_materialised():
    w = _lazy_case(3)
    om, lm = oracle.lazy_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["phys"], w["valid"],
                                    w["slot"], w["n_pages"], w["qpos"], w["doc_pos"], w["theta"],
                                    materialise=True)
    ol, ll = oracle.lazy_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["phys"], w["valid"],
                                    w["slot"], w["n_pages"], w["qpos"], w["doc_pos"], w["theta"],
                                    materialise=False)
    assert np.abs(om - ol).max() <= 1e-12 and np.abs(lm - ll).max() <= 1e-12


def test_lazy_single_doc_at_query_reduces_to_plain_attention():
    # one document placed at offset P with the query at n = P: relative offset 0, R(0) = I
    w = _lazy_case(4)
    b, n = 0, int(w["n_pages"][0])
    first = w["slot"][b, :n] == 0
    phys, valid = w["phys"][b, :n][first], w["valid"][b, :n][first]
    slot = np.zeros(len(phys), np.int32)
    for P in (0, 777):
        out, lse = oracle.attn_lazy_unit(w["q"][b, :2], w["k_pool"][0], w["v_pool"][0], phys, valid,
                                         slot, P, [P], w["theta"])
        ro, rl = oracle.attn_unit(w["q"][b, :2], w["k_pool"][0], w["v_pool"][0], phys, valid)
        assert np.allclose(out, ro, atol=1e-13) and np.allclose(lse, rl, atol=1e-13)


def test_lazy_differs_from_unrotated_when_offsets_nonzero():
    # guards against a rotation that silently does nothing
    w = _lazy_case(5)
    b, n = 1, int(w["n_pages"][1])
    out, _ = oracle.attn_lazy_unit(w["q"][b, :2], w["k_pool"][0], w["v_pool"][0], w["phys"][b, :n],
                                   w["valid"][b, :n], w["slot"][b, :n], w["qpos"][b],
                                   w["doc_pos"][b], w["theta"])
    ro, _ = oracle.attn_unit(w["q"][b, :2], w["k_pool"][0], w["v_pool"][0], w["phys"][b, :n],
                             w["valid"][b, :n])
    assert np.abs(out - ro).max() > 1e-3


# ------------------------------------------------------------------------------ set-difference

@pytest.mark.parametrize("seed", range(6))
def test_setdiff_python_sets(seed):
    rng = np.random.default_rng(seed)
    n_slots, stride = 40, 12
    resident = np.full(n_slots, -1, np.int32)
    ids = rng.choice(100, size=int(rng.integers(0, n_slots)), replace=False)
    pos = rng.choice(n_slots, size=len(ids), replace=False)
    resident[pos] = ids
    n_sel = int(rng.integers(0, stride + 1))
    sel = np.full(stride, -1, np.int32)
    sel[:n_sel] = np.sort(rng.choice(100, size=n_sel, replace=False))
    missing, nm, slot = oracle.setdiff_unit(resident, sel, n_sel, stride)
    want = sorted(set(sel[:n_sel].tolist()) - set(resident.tolist()))
    assert missing[:nm].tolist() == want and (missing[nm:] == -1).all()
    for i in range(n_sel):
        if sel[i] in set(resident.tolist()):
            assert resident[slot[i]] == sel[i]
        else:
            assert slot[i] == -1
    assert (slot[n_sel:] == -1).all()


# ------------------------------------------------------------------------------ bucketed LRU

def _lru_bucket(res, stamp, t, W):
    """Bucket of one slot, written out case by case: an empty slot is the oldest there is; a
    slot stamped at or after t (a clock that stepped back, or a wrapped counter) is as recent
    as a slot can be; otherwise whole bucket widths elapsed since the stamp, capped at 63."""
    if res < 0:
        return 63
    if int(stamp) >= int(t):
        return 0
    return min(63, (int(t) - int(stamp)) // W)


def _lru_bruteforce(resident, ts, slot, n_sel, missing, n_missing, t, W):
    resident, ts = resident.copy(), ts.copy()
    hits = {int(s) for s in slot[:n_sel] if s >= 0}
    for s in hits:
        ts[s] = t
    bucket = [_lru_bucket(resident[s], ts[s], t, W) for s in range(len(ts))]
    order = []
    for b in range(63, -1, -1):                 # oldest bucket first, slots ascending inside
        order += [s for s in range(len(ts)) if bucket[s] == b and s not in hits]
    victims = order[:n_missing]
    for i, s in enumerate(victims):
        resident[s] = missing[i]
        ts[s] = t
    hist = np.bincount(bucket, minlength=64)
    return resident, ts, victims, hist


@pytest.mark.parametrize("W", [1, 3])
def test_lru_bruteforce_trajectory(W):
    rng = np.random.default_rng(W)
    n_slots, stride = 24, 7
    resident = np.full(n_slots, -1, np.int32)
    ts = np.full(n_slots, np.iinfo(np.int32).min, np.int32)
    for t in range(60):
        n_sel = int(rng.integers(1, stride + 1))
        sel = np.full(stride, -1, np.int32)
        sel[:n_sel] = np.sort(rng.choice(40, size=n_sel, replace=False))
        missing, nm, slot = oracle.setdiff_unit(resident, sel, n_sel, stride)
        r2, t2, vic, hist = oracle.lru_unit(resident, ts, slot, n_sel, missing, nm, t, W, stride)
        br, bt, bv, bh = _lru_bruteforce(resident, ts, slot, n_sel, missing, nm, t, W)
        assert np.array_equal(r2, br) and np.array_equal(t2, bt)
        assert vic[:nm].tolist() == bv and (vic[nm:] == -1).all()
        assert np.array_equal(hist, bh) and hist.sum() == n_slots
        assert len(set(vic[:nm].tolist())) == nm
        assert set(sel[:n_sel].tolist()) <= set(r2.tolist())
        assert all(t2[s] == t for s in range(n_slots) if r2[s] in set(sel[:n_sel].tolist()))
        resident, ts = r2, t2


@pytest.mark.parametrize("W", [1, 3])
def test_lru_bruteforce_trajectory_with_clock_stepping_back(W):
    """Times that jump back (and forward again) leave timestamps later than t; such a slot must
    count as age 0 (bucket 0), not as a negative age."""
    rng = np.random.default_rng(10 + W)
    n_slots, stride = 20, 6
    resident = np.full(n_slots, -1, np.int32)
    ts = np.full(n_slots, np.iinfo(np.int32).min, np.int32)
    times = [0, 1, 2, 40, 41, 3, 4, 90, 5, 6, 7, 200, 8, 9, 300, 10, 11, 12]
    saw_future = False
    for t in times:
        n_sel = int(rng.integers(1, stride + 1))
        sel = np.full(stride, -1, np.int32)
        sel[:n_sel] = np.sort(rng.choice(35, size=n_sel, replace=False))
        missing, nm, slot = oracle.setdiff_unit(resident, sel, n_sel, stride)
        saw_future |= bool(((resident >= 0) & (ts > t)).any())
        r2, t2, vic, hist = oracle.lru_unit(resident, ts, slot, n_sel, missing, nm, t, W, stride)
        br, bt, bv, bh = _lru_bruteforce(resident, ts, slot, n_sel, missing, nm, t, W)
        assert np.array_equal(r2, br) and np.array_equal(t2, bt)
        assert vic[:nm].tolist() == bv and (vic[nm:] == -1).all()
        assert np.array_equal(hist, bh) and hist.sum() == n_slots
        resident, ts = r2, t2
    assert saw_future


def test_lru_future_timestamp_is_bucket_zero():
    """Hand-checked: at t = 5 a slot stamped 10 is the newest (bucket 0), so it is evicted last."""
    resident = np.array([1, 2, 3], np.int32)
    ts = np.array([10, 3, 0], np.int32)
    r, t2, vic, hist = oracle.lru_unit(resident, ts, [-1], 1, [7, 8, 9], 3, 5, 1, 3)
    # ages: slot 0 in the future -> 0, slot 1 -> 2, slot 2 -> 5: oldest first is 2, 1, 0
    assert vic.tolist() == [2, 1, 0]
    assert hist[0] == 1 and hist[2] == 1 and hist[5] == 1 and hist.sum() == 3
    r, t2, vic, hist = oracle.lru_unit(resident, ts, [-1], 1, [7], 1, 5, 3, 3)
    # W = 3: ages 0, 2, 5 -> buckets 0, 0, 1; the bucket-1 slot goes first
    assert vic.tolist() == [2, -1, -1] and hist[0] == 2 and hist[1] == 1


def test_lru_empty_slots_are_oldest():
    resident = np.array([5, -1, 7, -1], np.int32)
    ts = np.array([0, np.iinfo(np.int32).min, 1, np.iinfo(np.int32).min], np.int32)
    r, t, vic, hist = oracle.lru_unit(resident, ts, [-1, -1], 2, [8, 9], 2, 2, 1, 2)
    assert vic.tolist() == [1, 3] and r.tolist() == [5, 8, 7, 9] and hist[63] == 2
    r, t, vic, hist = oracle.lru_unit(r, t, [-1, -1, -1], 3, [10, 11, 12], 3, 3, 1, 3)
    # ages now: slot0 3, slot1 1, slot2 2, slot3 1 -> order 0, 2, 1
    assert vic.tolist() == [0, 2, 1] and hist[3] == 1 and hist[2] == 1 and hist[1] == 2


# ------------------------------------------------------------------------------ retrieve (swap-in)

def _offload_case(seed, B=2, Hk=2, G=2, npg=14, n_slots=6, stride=5):
    """A small host pool, an empty slot pool and a page table with scattered host pages."""
    rng = np.random.default_rng(seed)
    n_host = B * npg + 3
    k_host = gen.rows_bf16(seed, 901, Hk * n_host * 64).reshape(Hk, n_host, 64, 128)
    v_host = gen.rows_bf16(seed, 902, Hk * n_host * 64).reshape(Hk, n_host, 64, 128)
    pt = rng.permutation(n_host)[:B * npg].reshape(B, npg).astype(np.int32)
    L = np.array([npg * 64 - int(rng.integers(0, 64)) for _ in range(B)], np.int32)
    q = gen.rows_bf16(seed, 903, B * Hk * G).reshape(B, Hk * G, 128)
    return rng, k_host, v_host, pt, L, q, n_slots, stride


@pytest.mark.parametrize("seed", range(3))
def test_retrieve_trajectory_invariants(seed):
    """Over a trajectory of selections: every selected page ends up in its slot byte for byte,
    only victim slots of the unit's own range change, the resident table names the slot's page,
    and attention over the slots equals attention over the host pool exactly."""
    rng, k_host, v_host, pt, L, q, n_slots, stride = _offload_case(seed)
    B, npg = pt.shape
    Hk = k_host.shape[0]
    U = B * Hk
    k_slots = np.zeros((Hk, B * n_slots, 64, 128), np.uint16)
    v_slots = np.zeros_like(k_slots)
    resident = np.full((U, n_slots), -1, np.int32)
    ts = np.full((U, n_slots), np.iinfo(np.int32).min, np.int32)
    for t in range(25):
        sel = np.full((U, stride), -1, np.int32)
        n_sel = rng.integers(1, stride + 1, U).astype(np.int32)
        for u in range(U):
            sel[u, :n_sel[u]] = np.sort(rng.choice(npg, size=n_sel[u], replace=False))
        missing, nm, slot = oracle.setdiff_batch(resident, sel, n_sel)
        resident, ts, victims, _ = oracle.lru_batch(resident, ts, slot, n_sel, missing, nm, t, 2)
        k_before, v_before = k_slots.copy(), v_slots.copy()
        full = oracle.retrieve_batch(k_host, v_host, pt, missing, nm, victims, slot, n_sel, k_slots,
                                     v_slots, n_slots)
        changed = set()
        for h in range(Hk):
            for p in range(B * n_slots):
                if not (np.array_equal(k_slots[h, p], k_before[h, p])
                        and np.array_equal(v_slots[h, p], v_before[h, p])):
                    changed.add((h, p))
        for u in range(U):
            b, h = divmod(u, Hk)
            n = n_sel[u]
            assert (full[u, :n] >= 0).all() and (full[u, :n] < n_slots).all()
            assert len(set(full[u, :n].tolist())) == n
            hits = [i for i in range(n) if slot[u, i] >= 0]
            assert all(full[u, i] == slot[u, i] for i in hits)
            for i in range(n):
                s = int(full[u, i])
                assert resident[u, s] == sel[u, i]
                hp = pt[b, sel[u, i]]
                assert np.array_equal(k_slots[h, b * n_slots + s], k_host[h, hp])
                assert np.array_equal(v_slots[h, b * n_slots + s], v_host[h, hp])
        # the only pages written are the victims of each unit (content may coincide otherwise)
        vict = {(u % Hk, (u // Hk) * n_slots + int(victims[u, j])) for u in range(U) for j in range(nm[u])}
        assert changed <= vict
        out_s, lse_s = oracle.slot_attn_batch(q, k_slots, v_slots, sel.reshape(B, Hk, stride),
                                              full.reshape(B, Hk, stride), n_sel.reshape(B, Hk), L, n_slots)
        out_h, lse_h = oracle.sparse_attn_batch(q, k_host, v_host, pt, sel.reshape(B, Hk, stride),
                                                n_sel.reshape(B, Hk), L)
        assert np.array_equal(out_s, out_h) and np.array_equal(lse_s, lse_h)


def test_retrieve_hand_example():
    """One unit, four slots, a hand-checked swap-in: selection [1, 4, 6], page 4 resident in
    slot 2, victims 0 and 3 for pages 1 and 6."""
    k_host = np.arange(1 * 8 * 64 * 128, dtype=np.uint16).reshape(1, 8, 64, 128)
    v_host = (k_host + 7).astype(np.uint16)
    pt = np.array([[7, 6, 5, 4, 3, 2, 1, 0]], np.int32)
    k_slots = np.zeros((1, 4, 64, 128), np.uint16)
    v_slots = np.zeros_like(k_slots)
    slot = np.array([[-1, 2, -1, -1]], np.int32)
    full = oracle.retrieve_batch(k_host, v_host, pt, [[1, 6, -1, -1]], [2], [[0, 3, -1, -1]], slot, [3],
                                 k_slots, v_slots, 4)
    assert full.tolist() == [[0, 2, 3, -1]]
    assert np.array_equal(k_slots[0, 0], k_host[0, 6]) and np.array_equal(v_slots[0, 3], v_host[0, 1])
    assert not k_slots[0, 1].any() and not k_slots[0, 2].any()


# ------------------------------------------------------------------------------ lazy prefill

def _prefill_case(seed, T=5, theta=10000.0):
    w = gen.lazy_rag(seed=seed, B=2, Hq=4, Hk=2, n_docs=6, docs_per_req=3, min_len=70, max_len=200,
                     theta=theta)
    q = gen.rows_bf16(seed, 990, 2 * T * 4).reshape(2, T, 4, 128)
    return w, q


def _complex_rope_prefill(w, q, theta):
    """Independent brute force: RoPE as multiplication of the complex numbers x_i + i x_(i+64) by
    exp(i pos theta^(-i/64)); keys placed at their absolute positions; dense scipy softmax."""
    B, T, Hq, _ = q.shape
    Hk = w["Hk"]
    G = Hq // Hk
    freq = theta ** (-np.arange(64) / 64.0)
    cplx = lambda x: x[..., :64] + 1j * x[..., 64:]
    out = np.zeros((B, T, Hq, 128))
    lse = np.zeros((B, T, Hq))
    for b in range(B):
        n = w["n_pages"][b]
        for h in range(Hk):
            ks, vs, kpos = [], [], []
            for i in range(n):
                rows = slice(0, w["valid"][b, i])
                ks.append(f(w["k_pool"][h, w["phys"][b, i], rows]))
                vs.append(f(w["v_pool"][h, w["phys"][b, i], rows]))
                kpos += [w["doc_pos"][b, w["slot"][b, i]]] * w["valid"][b, i]
            K, V, kpos = np.concatenate(ks), np.concatenate(vs), np.array(kpos, np.float64)
            Kc = cplx(K) * np.exp(1j * kpos[:, None] * freq[None, :])   # keys carry doc-local rotation
            for t in range(T):
                pos = w["qpos"][b] + t
                for g in range(G):
                    qc = cplx(f(q[b, t, h * G + g])) * np.exp(1j * pos * freq)
                    z = (qc.real @ Kc.real.T + qc.imag @ Kc.imag.T) / math.sqrt(128)
                    out[b, t, h * G + g] = softmax(z) @ V
                    lse[b, t, h * G + g] = logsumexp(z)
    return out, lse


@pytest.mark.parametrize("materialise", [True, False])
def test_prefill_complex_rope_bruteforce(materialise):
    w, q = _prefill_case(5)
    out, lse = oracle.lazy_prefill_batch(q, w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"],
                                         w["n_pages"], w["qpos"], w["doc_pos"], 10000.0, materialise=materialise)
    ro, rl = _complex_rope_prefill(w, q, 10000.0)
    assert np.abs(out - ro).max() < 1e-10 and np.abs(lse - rl).max() < 1e-10


def test_prefill_depends_on_relative_positions_only():
    """Moving the query rows and every document by the same offset changes nothing; moving one
    document does."""
    w, q = _prefill_case(6, T=3)
    args = (w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"], w["n_pages"])
    o1, l1 = oracle.lazy_prefill_batch(q, *args, w["qpos"], w["doc_pos"], 500000.0)
    o2, l2 = oracle.lazy_prefill_batch(q, *args, w["qpos"] + 12345, w["doc_pos"] + 12345, 500000.0)
    assert np.abs(o1 - o2).max() < 1e-9 and np.abs(l1 - l2).max() < 1e-9
    dp = w["doc_pos"].copy()
    dp[:, 1] += 7
    o3, _ = oracle.lazy_prefill_batch(q, *args, w["qpos"], dp, 500000.0)
    assert np.abs(o1 - o3).max() > 1e-4


def test_prefill_rows_are_decode_queries():
    """Row t of a prefill equals lazy decode attention with the query at qpos + t."""
    w, q = _prefill_case(7, T=4)
    out, lse = oracle.lazy_prefill_batch(q, w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"],
                                         w["n_pages"], w["qpos"], w["doc_pos"], 500000.0, materialise=False)
    for t in range(4):
        od, ld = oracle.lazy_attn_batch(q[:, t], w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"],
                                        w["n_pages"], w["qpos"] + t, w["doc_pos"], 500000.0, materialise=False)
        assert np.array_equal(out[:, t], od) and np.array_equal(lse[:, t], ld)


# ------------------------------------------------------------------------------ prefill step (causal)

def _step_bruteforce(w, theta, slopes=None):
    """Independent brute force of the whole prefill step: every listed key gets its absolute
    position m = doc_pos[slot] + page_start + row; a row at position n attends to the keys with
    m <= n.  RoPE: complex rotation (keys by doc_pos, since they carry their document-local
    rotation; the query by n).  ALiBi (slopes given): no rotation, bias -slope (n - m).  scipy
    softmax / logsumexp over the visible keys."""
    q = w["q"]
    B, T, Hq, _ = q.shape
    Hk = w["Hk"]
    G = Hq // Hk
    freq = theta ** (-np.arange(64) / 64.0)
    cplx = lambda x: x[..., :64] + 1j * x[..., 64:]
    out, lse = np.zeros((B, T, Hq, 128)), np.zeros((B, T, Hq))
    for b in range(B):
        n_p = w["n_pages"][b]
        for h in range(Hk):
            ks, vs, mpos, dpos = [], [], [], []
            for i in range(n_p):
                v = w["valid"][b, i]
                ks.append(f(w["k_pool"][h, w["phys"][b, i], :v]))
                vs.append(f(w["v_pool"][h, w["phys"][b, i], :v]))
                d = w["doc_pos"][b, w["slot"][b, i]]
                mpos += [d + w["page_start"][b, i] + r for r in range(v)]
                dpos += [d] * v
            K, V = np.concatenate(ks), np.concatenate(vs)
            mpos, dpos = np.array(mpos, np.float64), np.array(dpos, np.float64)
            Kc = cplx(K) * np.exp(1j * dpos[:, None] * freq[None, :])
            for t in range(T):
                n = w["qpos0"][b] + t
                vis = mpos <= n
                for g in range(G):
                    hq = h * G + g
                    if slopes is None:
                        qc = cplx(f(q[b, t, hq])) * np.exp(1j * n * freq)
                        z = (qc.real @ Kc.real.T + qc.imag @ Kc.imag.T) / math.sqrt(128)
                    else:
                        z = K @ f(q[b, t, hq]) / math.sqrt(128) - float(slopes[hq]) * (n - mpos)
                    out[b, t, hq] = softmax(z[vis]) @ V[vis]
                    lse[b, t, hq] = logsumexp(z[vis])
    return out, lse


def _step_args(w):
    return (w["q"], w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"], w["page_start"], w["n_pages"],
            w["qpos0"], w["doc_pos"])


@pytest.mark.parametrize("mode", ["materialised", "lazy"])
def test_prefill_step_scipy_bruteforce(mode):
    """Cached documents plus the rows' own keys (T = 70 spans two self pages): the causal mask by
    absolute position, against the independent brute force."""
    w = gen.prefill_step(seed=21, B=2, T=70, Hq=4, Hk=2, n_docs=4, docs_per_req=2, min_len=64, max_len=200,
                         theta=10000.0)
    out, lse = oracle.prefill_step_batch(*_step_args(w), 10000.0, mode=mode)
    ro, rl = _step_bruteforce(w, 10000.0)
    assert np.abs(out - ro).max() < 1e-10 and np.abs(lse - rl).max() < 1e-10


def test_prefill_step_without_cached_documents_closed_forms():
    """Only the rows' own keys: row 0 sees key 0 alone, so its output is V of key 0 and its LSE
    the single score; a key after row t never changes row t."""
    w = gen.prefill_step(seed=22, B=2, T=20, Hq=2, Hk=1, theta=500000.0, cached=False)
    out, lse = oracle.prefill_step_batch(*_step_args(w), 500000.0)
    for b in range(2):
        v0 = f(w["v_pool"][0, w["phys"][b, 0], 0])
        for hq in range(2):
            assert np.abs(out[b, 0, hq] - v0).max() < 1e-12
            k0 = f(w["k_pool"][0, w["phys"][b, 0], 0])
            # row 0 and key 0 both sit at position 0 of the prompt: R(0) on both
            assert abs(lse[b, 0, hq] - float(f(w["q"][b, 0, hq]) @ k0) / math.sqrt(128)) < 1e-12
    w2 = dict(w)
    kp, vp = w["k_pool"].copy(), w["v_pool"].copy()
    kp[0, w["phys"][0, 0], 11:] = gen.rows_bf16(5, 77, 64 - 11)
    vp[0, w["phys"][0, 0], 11:] = gen.rows_bf16(5, 78, 64 - 11)
    w2["k_pool"], w2["v_pool"] = kp, vp
    out2, lse2 = oracle.prefill_step_batch(*_step_args(w2), 500000.0)
    assert np.array_equal(out2[0, :11], out[0, :11]) and np.array_equal(lse2[0, :11], lse[0, :11])
    assert np.abs(out2[0, 11:] - out[0, 11:]).max() > 1e-3


def test_prefill_step_equals_cached_prefill_when_nothing_follows_the_rows():
    """Without the rows' own pages every key precedes every row: the step is the cached-document
    prefill."""
    w = gen.prefill_step(seed=23, B=2, T=6, Hq=4, Hk=2, n_docs=5, docs_per_req=2, min_len=64, max_len=300)
    n_cached = w["n_pages"] - 1
    args = (w["q"], w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"])
    o1, l1 = oracle.prefill_step_batch(*args, w["page_start"], n_cached, w["qpos0"], w["doc_pos"], w["theta"])
    o2, l2 = oracle.lazy_prefill_batch(*args, n_cached, w["qpos0"], w["doc_pos"], w["theta"], materialise=True)
    assert np.abs(o1 - o2).max() < 1e-12 and np.abs(l1 - l2).max() < 1e-12


def _np_bf16(x):
    """Nearest bf16 (ties to even) of fp64 values, by scaling the significand to 8 bits."""
    m, e = np.frexp(np.asarray(x, np.float64))
    return np.ldexp(np.rint(m * 256.0), e - 8)


def test_prefill_step_bf16_rotated_query_mode():
    """Mode lazy_bf16q rounds each document's rotated query to bf16: against a numpy brute force
    that does the same (numpy RoPE, numpy rounding), and different from the exact lazy form."""
    w = gen.prefill_step(seed=24, B=1, T=3, Hq=2, Hk=1, n_docs=3, docs_per_req=2, min_len=64, max_len=150,
                         theta=10000.0)
    out, lse = oracle.prefill_step_batch(*_step_args(w), 10000.0, mode="lazy_bf16q")
    exact, _ = oracle.prefill_step_batch(*_step_args(w), 10000.0, mode="lazy")
    freq = 10000.0 ** (-np.arange(64) / 64.0)
    n_p = w["n_pages"][0]
    for t in range(3):
        n = w["qpos0"][0] + t
        for hq in range(2):
            zs, vs = [], []
            for i in range(n_p):
                d = w["doc_pos"][0, w["slot"][0, i]]
                a = (n - d) * freq
                x = f(w["q"][0, t, hq])
                qr = np.concatenate([x[:64] * np.cos(a) - x[64:] * np.sin(a), x[64:] * np.cos(a) + x[:64] * np.sin(a)])
                qr = _np_bf16(qr)
                for r in range(w["valid"][0, i]):
                    if d + w["page_start"][0, i] + r > n:
                        continue
                    zs.append(qr @ f(w["k_pool"][0, w["phys"][0, i], r]) / math.sqrt(128))
                    vs.append(f(w["v_pool"][0, w["phys"][0, i], r]))
            zs = np.array(zs)
            assert np.abs(out[0, t, hq] - softmax(zs) @ np.array(vs)).max() < 1e-10
            assert abs(lse[0, t, hq] - logsumexp(zs)) < 1e-10
    assert np.abs(out - exact).max() > 1e-6          # the rounding is real


def test_alibi_step_scipy_bruteforce():
    """The ALiBi prefill with the rows' own keys listed: causal by position, brute force."""
    w = gen.prefill_step(seed=25, B=2, T=70, Hq=4, Hk=2, n_docs=4, docs_per_req=2, min_len=64, max_len=200)
    slopes = np.array([0.01, 0.05, 0.2, 0.0], np.float32)
    out, lse = oracle.alibi_prefill_batch(w["q"], w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"],
                                          w["page_start"], w["n_pages"], w["qpos0"], w["doc_pos"], slopes)
    ro, rl = _step_bruteforce(w, 10000.0, slopes=slopes)
    assert np.abs(out - ro).max() < 1e-10 and np.abs(lse - rl).max() < 1e-10


# ------------------------------------------------------------------------------ ALiBi prefill

def _alibi_args(w):
    return (w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"], w["page_start"], w["n_pages"])


def _plain_prefill(w, q):
    """Dense softmax attention over every listed key (no position term), scipy."""
    B, T, Hq, _ = q.shape
    G = Hq // w["Hk"]
    out, lse = np.zeros((B, T, Hq, 128)), np.zeros((B, T, Hq))
    for b in range(B):
        n = w["n_pages"][b]
        for h in range(w["Hk"]):
            K = np.concatenate([f(w["k_pool"][h, w["phys"][b, i], :w["valid"][b, i]]) for i in range(n)])
            V = np.concatenate([f(w["v_pool"][h, w["phys"][b, i], :w["valid"][b, i]]) for i in range(n)])
            for t in range(T):
                for g in range(G):
                    z = K @ f(q[b, t, h * G + g]) / math.sqrt(128)
                    out[b, t, h * G + g] = softmax(z) @ V
                    lse[b, t, h * G + g] = logsumexp(z)
    return out, lse


def test_alibi_zero_slope_is_plain_attention_and_nonzero_slopes_are_not():
    w, q = _prefill_case(8, T=3)
    slopes = np.array([0.0, 0.05, 0.0, 0.25], np.float32)
    out, lse = oracle.alibi_prefill_batch(q, *_alibi_args(w), w["qpos"], w["doc_pos"], slopes)
    ro, rl = _plain_prefill(w, q)
    for hq in (0, 2):
        assert np.abs(out[:, :, hq] - ro[:, :, hq]).max() < 1e-10
        assert np.abs(lse[:, :, hq] - rl[:, :, hq]).max() < 1e-10
    for hq in (1, 3):
        assert np.abs(out[:, :, hq] - ro[:, :, hq]).max() > 1e-3


def test_alibi_two_equal_keys_closed_form():
    """Two keys with the same K row at positions m0 < m1 and a query at n: their weights are in the
    ratio exp(-s (n - m0)) : exp(-s (n - m1)), so out = (v0 + e^{s (m1 - m0)} v1) / (1 + e^{s (m1 - m0)})
    and lse = q.k / sqrt(128) - s (n - m1) + log(1 + e^{-s (m1 - m0)})."""
    k = gen.rows_bf16(9, 1, 1)[0]
    v = gen.rows_bf16(9, 2, 2)
    k_pool = np.zeros((1, 2, 64, 128), np.uint16)
    v_pool = np.zeros((1, 2, 64, 128), np.uint16)
    k_pool[0, 1, 0] = k_pool[0, 1, 1] = k                      # page 1 holds the two tokens
    v_pool[0, 1, 0], v_pool[0, 1, 1] = v[0], v[1]
    q = gen.rows_bf16(9, 3, 1).reshape(1, 1, 1, 128)
    phys, valid, slot = np.array([[1]]), np.array([[2]]), np.array([[0]])
    page_start, doc_pos, qpos = np.array([[10]]), np.array([[100]]), np.array([500])
    s = 0.0625                                                 # exact in fp32
    out, lse = oracle.alibi_prefill_batch(q, k_pool, v_pool, phys, valid, slot, page_start, np.array([1]), qpos,
                                          doc_pos, np.array([s], np.float32))
    m0, m1, n = 110.0, 111.0, 500.0
    r = math.exp(s * (m1 - m0))
    want = (f(v[0]) + r * f(v[1])) / (1 + r)
    qk = float(f(q[0, 0, 0]) @ f(k)) / math.sqrt(128)
    assert np.abs(out[0, 0, 0] - want).max() < 1e-12
    assert abs(lse[0, 0, 0] - (qk - s * (n - m1) + math.log1p(math.exp(-s * (m1 - m0))))) < 1e-10


def test_alibi_positions_not_list_order():
    """Shifting the rows and every document by the same offset changes nothing (distance only);
    listing the pages in another order changes nothing (positions come from doc_pos and
    page_start); moving one page's start does."""
    w, q = _prefill_case(10, T=2)
    slopes = np.array([0.01, 0.03, 0.1, 0.5], np.float32)
    o1, l1 = oracle.alibi_prefill_batch(q, *_alibi_args(w), w["qpos"], w["doc_pos"], slopes)
    o2, l2 = oracle.alibi_prefill_batch(q, *_alibi_args(w), w["qpos"] + 777, w["doc_pos"] + 777, slopes)
    assert np.abs(o1 - o2).max() < 1e-9 and np.abs(l1 - l2).max() < 1e-9
    perm_w = dict(w)
    for key in ("phys", "valid", "slot", "page_start"):
        a = w[key].copy()
        for b in range(w["B"]):
            n = w["n_pages"][b]
            a[b, :n] = w[key][b, gen.permutation(10, 40 + b, n)]
        perm_w[key] = a
    o3, l3 = oracle.alibi_prefill_batch(q, *_alibi_args(perm_w), w["qpos"], w["doc_pos"], slopes)
    assert np.abs(o1 - o3).max() < 1e-12 and np.abs(l1 - l3).max() < 1e-12
    ps = w["page_start"].copy()
    ps[0, 1] += 5
    moved = dict(w, page_start=ps)
    o4, _ = oracle.alibi_prefill_batch(q, *_alibi_args(moved), w["qpos"], w["doc_pos"], slopes)
    assert np.abs(o1 - o4).max() > 1e-6


# ------------------------------------------------------------------------------ bf16 summaries

def test_round_bf16_matches_the_generator_rounding():
    """fp64 -> bf16 round-to-nearest-even (frexp / rint) against the generator's fp32 bit
    arithmetic, on fp32-exact values including exact ties."""
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(20000) * 10.0 ** rng.integers(-3, 4, 20000)).astype(np.float32)
    ties = (np.float32(1.0) + np.arange(1, 64, 2, dtype=np.float32) * np.float32(2.0 ** -8)).astype(np.float32)
    x = np.concatenate([x, ties, -ties])
    want = gen.bf16_to_f32(gen.f32_to_bf16(x)).astype(np.float64)
    got = np.array([oracle.round_bf16(float(v)) for v in x])
    assert np.array_equal(got, want)


def test_scores_from_bf16_summaries_bruteforce():
    """Keys with few significant bits (every fp32 sum exact): scores from bf16-rounded sums by
    numpy against the oracle, then the distance to the fp32-summary scores stays within half a
    bf16 ulp of each sum."""
    rng = np.random.default_rng(3)
    Hk, n_phys, G = 1, 6, 3
    keys = (rng.integers(-40, 41, (Hk, n_phys, 64, 128)) / 8.0).astype(np.float32)
    k_pool = gen.f32_to_bf16(keys)
    q = gen.rows_bf16(3, 77, G).reshape(1, G, 128)
    pt = np.arange(n_phys, dtype=np.int32).reshape(1, n_phys)
    L = np.array([n_phys * 64], np.int32)
    s16 = oracle.score_batch(q, k_pool, pt, L, summary_bf16=True)[0, 0]
    s32 = oracle.score_batch(q, k_pool, pt, L)[0, 0]
    sums = f(k_pool[0]).reshape(n_phys, 4, 16, 128).sum(2)                  # exact in fp32 here
    means16 = gen.bf16_to_f32(gen.f32_to_bf16(sums.astype(np.float32))).astype(np.float64) / 16.0
    qs = f(q[0]).sum(0)
    want = (means16 @ qs).max(1) / math.sqrt(128)
    want[n_phys - 1:] = -np.inf                                             # the local page and after
    assert np.allclose(s16[:n_phys - 1], want[:n_phys - 1], rtol=0, atol=1e-12)
    assert np.isneginf(s16[n_phys - 1])
    bound = (np.abs(sums) * 2.0 ** -9 / 16.0) @ np.abs(qs) / math.sqrt(128)
    diff = np.abs(s16[:n_phys - 1] - s32[:n_phys - 1])
    assert (diff <= bound.max(1)[:n_phys - 1] + 1e-12).all()
    assert diff.max() > 0                                                   # the rounding is real


# ------------------------------------------------------------------------------ column score S

def _colscore_case(seed, B=2, Hq=4, Hk=2, n=200, alpha=9):
    w = gen.sparse_workload(B, Hq, Hk, n, 4, 4, seed=seed)
    q = gen.rows_bf16(seed, 555, B * alpha * Hq).reshape(B, alpha, Hq, 128)
    return w, q


def test_column_scores_scipy_bruteforce():
    w, q = _colscore_case(1)
    n, alpha = int(w["seq_len"][0]), q.shape[1]
    S = oracle.column_scores_batch(q, w["k_pool"], w["page_table"], w["seq_len"], w["np_max"] * 64)
    G = w["Hq"] // w["Hk"]
    for b in range(w["B"]):
        for hq in range(w["Hq"]):
            h = hq // G
            K = np.concatenate([f(w["k_pool"][h, w["page_table"][b, p]]) for p in range(w["np_max"])])[:n]
            Q = f(q[b, :, hq])
            Z = Q @ K.T / math.sqrt(128)
            want = np.zeros(w["np_max"] * 64)
            for j in range(alpha):
                pos = n - alpha + j
                want[:pos + 1] += softmax(Z[j, :pos + 1])
            assert np.allclose(S[b, hq], want, rtol=1e-10, atol=1e-13)


def test_column_scores_given_lse_scipy_bruteforce():
    """The given-LSE form against numpy: with each row's exact log-sum-exp (scipy) it is the
    softmax column sum; adding c to a row's LSE scales that row's contribution by exp(-c)."""
    w, q = _colscore_case(4, n=64 * 2 + 45, alpha=13)
    n, alpha = int(w["seq_len"][0]), q.shape[1]
    G = w["Hq"] // w["Hk"]
    lse = np.zeros((w["B"], alpha, w["Hq"]))
    want = np.zeros((w["B"], w["Hq"], w["np_max"] * 64))
    shift = np.linspace(-0.7, 1.3, alpha)                 # a different shift per row
    want_shift = np.zeros_like(want)
    for b in range(w["B"]):
        for hq in range(w["Hq"]):
            h = hq // G
            K = np.concatenate([f(w["k_pool"][h, w["page_table"][b, p]]) for p in range(w["np_max"])])[:n]
            Z = f(q[b, :, hq]) @ K.T / math.sqrt(128)
            for j in range(alpha):
                pos = n - alpha + j
                lse[b, j, hq] = logsumexp(Z[j, :pos + 1])
                p = softmax(Z[j, :pos + 1])
                want[b, hq, :pos + 1] += p
                want_shift[b, hq, :pos + 1] += p * math.exp(-shift[j])
    S = oracle.column_scores_given_lse_batch(q, lse, w["k_pool"], w["page_table"], w["seq_len"], w["np_max"] * 64)
    assert np.allclose(S, want, rtol=1e-10, atol=1e-13)
    assert np.allclose(S, oracle.column_scores_batch(q, w["k_pool"], w["page_table"], w["seq_len"],
                                                     w["np_max"] * 64), rtol=1e-10, atol=1e-13)
    S2 = oracle.column_scores_given_lse_batch(q, lse + shift[None, :, None], w["k_pool"], w["page_table"],
                                              w["seq_len"], w["np_max"] * 64)
    assert np.allclose(S2, want_shift, rtol=1e-10, atol=1e-13)


def test_column_scores_invariants():
    """Each row's probabilities sum to one, so S sums to alpha; keys after row j's position get
    nothing from it, so the last key collects only the last row; S >= 0; nothing past n."""
    w, q = _colscore_case(2, n=64 * 3 + 17, alpha=20)
    n, alpha = int(w["seq_len"][0]), q.shape[1]
    S = oracle.column_scores_batch(q, w["k_pool"], w["page_table"], w["seq_len"], w["np_max"] * 64)
    assert np.allclose(S.sum(-1), alpha, rtol=0, atol=1e-9)
    assert (S >= 0).all() and (S[..., n:] == 0).all()
    # the newest key is seen by the last row only: S[n-1] = A[alpha-1][n-1] < 1
    assert (S[..., n - 1] < 1).all() and (S[..., n - 1] > 0).all()
    # a window covering the whole prompt: every row sums to one over its own prefix
    w2, q2 = _colscore_case(3, n=30, alpha=30)
    S2 = oracle.column_scores_batch(q2, w2["k_pool"], w2["page_table"], w2["seq_len"], 64)
    assert np.allclose(S2.sum(-1), 30, rtol=0, atol=1e-9)
    assert (S2[..., 0] >= 1 - 1e-12).all()      # row 0 sits at position 0 and sees key 0 alone


# ------------------------------------------------------------------------------ two-level page directory

def _split_table(table, shift, rng, dev_frac):
    """A directory for a flat table, built independently: each segment that holds a mapped page gets
    a host copy; a random share of them also a device copy (the directory then names the device)."""
    B, npm = table.shape
    seg = 1 << shift
    n_dir = (npm + seg - 1) // seg
    dir_ = np.full((B, n_dir), -1, np.int32)
    host, dev = [], []
    for b in range(B):
        for s_ in range(n_dir):
            chunk = np.full(seg, -1, np.int32)
            part = table[b, s_ * seg:(s_ + 1) * seg]
            chunk[:len(part)] = part
            if (chunk < 0).all():
                continue
            if rng.random() < dev_frac:
                dir_[b, s_] = len(dev)
                dev.append(chunk)
            else:
                dir_[b, s_] = -2 - len(host)
                host.append(chunk)
    z = np.zeros((1, seg), np.int32)
    return dir_, (np.array(dev) if dev else z), (np.array(host) if host else z)


@pytest.mark.parametrize("shift,dev_frac", [(4, 0.0), (8, 0.5), (6, 1.0)])
def test_dir_lookup_equals_flat_table(shift, dev_frac):
    rng = np.random.default_rng(shift)
    B, npm = 5, 1000
    table = rng.integers(0, 50000, (B, npm)).astype(np.int32)
    table[1, 300:700] = -1                 # an unmapped stretch spanning whole segments
    table[3, 950:] = -1
    d, dev, host = _split_table(table, shift, rng, dev_frac)
    assert np.array_equal(oracle.dir_to_table(d, shift, dev, host, npm), table)
    # entries naming segments that do not exist read as unmapped
    bad = d.copy()
    bad[0, 0] = 10 ** 6
    bad[2, 1] = -2 - 10 ** 6
    t2 = oracle.dir_to_table(bad, shift, dev, host, npm)
    seg = 1 << shift
    assert (t2[0, :seg] == -1).all() and (t2[2, seg:2 * seg] == -1).all()
    assert np.array_equal(t2[4], table[4])


def test_dir_metadata_follows_the_pages_in_use():
    """Only segments with a mapped page exist: a 1M-page logical space with 3 x 4096 pages in use
    needs about 3 x 16 segments of 256 ids, whatever the logical size."""
    shift, npm = 8, 1 << 20
    table = np.full((3, npm), -1, np.int32)
    for b, start in enumerate((0, 5000, 900_000)):
        table[b, start:start + 4096] = np.arange(4096) + 4096 * b
    d, dev, host = _split_table(table, shift, np.random.default_rng(0), 0.0)
    n_segs = int((d != -1).sum())
    # 4096 pages fill 16 aligned segments; the ranges starting at 5000 and 900000 are not aligned
    # to 256 and touch 17 each
    assert n_segs == 16 + 17 + 17
    assert host.shape[0] * (1 << shift) * 4 < table.nbytes / 200    # 50 KiB of segments for 12 MiB of flat table
    assert np.array_equal(oracle.dir_to_table(d, shift, dev, host, npm), table)
