"""GPU parity: every kernel, called through the C ABI, against the fp64 oracle on seeded inputs.

Acceptance (attention): max |dO| <= 1e-2 and mean |dO| <= 1e-3 against the fp64 oracle on the
same bf16 inputs, LSE within 1e-3.  Selection, set-difference and LRU: bit-exact when both
sides rank the same fp32 scores; against fp64 oracle scores, differences are allowed only among
pages within 1e-5 relative of the k-th score.  Block scores: within an fp32 summation bound
derived from the operand magnitudes (2e-5 x sum |q_sum| |mean|, about twice the worst-case
rounding of the 16 + 128 + G term sums).
"""
import math

import numpy as np
import pytest
import torch

import gen
import oracle
import sparse_paged_kv_score_gb300 as spkv
from helpers import DEV, Dev, alive_bits_to_bytes, alive_bytes_to_bits, attn_errors, bf, f32, i32, u32_as_i32

pytestmark = pytest.mark.gpu

ATTN_MAX, ATTN_MEAN, LSE_TOL = 1e-2, 1e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_paged_kv_score_gb300 import build
    build.build()
    spkv.load()


def f64(bits):
    return gen.bf16_to_f32(bits).astype(np.float64)


# ------------------------------------------------------------------ summaries / append

def test_summaries_match_oracle_means():
    w = gen.sparse_workload(2, 8, 2, 64 * 5 + 37, 4, 4, seed=3)   # last page holds 37 tokens
    d = Dev(w)
    ks = d.ksum.cpu().numpy()
    cnt = gen.page_counts(w)
    for h in range(2):
        for p in range(w["n_phys"]):
            mean, c = oracle.page_means(w["k_pool"][h, p], cnt[p])
            assert np.allclose(ks[h, p], mean * c[:, None], rtol=0, atol=2e-5)
    assert d.errors() == (0, 0)
    d.close()


@pytest.mark.parametrize("summary_bf16", [False, True])
def test_append_equals_rebuild(summary_bf16):
    B, Hk = 3, 2
    w = gen.sparse_workload(B, 8, Hk, 64 * 3 - 2, 4, 4, seed=5, extra_tokens=70)
    d = Dev(w, summary_bf16=summary_bf16)
    L = w["seq_len"].copy()
    for step in range(4):      # crosses the page boundary at 192
        phys = np.array([w["page_table"][b, L[b] // 64] for b in range(B)], np.int32)
        tok = (L % 64).astype(np.int32)
        kn = gen.rows_bf16(9, 100 + step, B * Hk).reshape(B, Hk, 128)
        vn = gen.rows_bf16(9, 200 + step, B * Hk).reshape(B, Hk, 128)
        spkv.paged_kv_append(d.cache, i32(phys), i32(tok), bf(kn), bf(vn))
        for b in range(B):
            w["k_pool"][:, phys[b], tok[b]] = kn[b]
            w["v_pool"][:, phys[b], tok[b]] = vn[b]
        L += 1
    torch.cuda.synchronize()
    w["seq_len"] = L
    assert np.array_equal(d.k_pool.view(torch.int16).cpu().numpy().view(np.uint16), w["k_pool"])
    assert np.array_equal(d.v_pool.view(torch.int16).cpu().numpy().view(np.uint16), w["v_pool"])
    assert np.array_equal(d.cnt.cpu().numpy(), gen.page_counts(w))
    fresh = Dev(w, summary_bf16=summary_bf16)      # summary build from scratch on the updated pool
    assert torch.equal(d.ksum, fresh.ksum), "append and create must give bitwise equal sums"
    assert d.errors() == (0, 0)
    d.close()
    fresh.close()


@pytest.mark.parametrize("summary_bf16", [False, True])
def test_decode_append_score_equals_append_then_score(summary_bf16):
    """The fused decode call gives bitwise the pools, page counts, summaries and scores of
    paged_kv_append at position seq_len - 1 followed by score_blocks, over steps that cross a page
    boundary (a token landing in row 0 of a fresh page)."""
    B, Hk, Hq = 3, 2, 8
    w = gen.sparse_workload(B, Hq, Hk, 64 * 3 - 2, 4, 4, seed=6, extra_tokens=70)
    two, one = Dev(w, summary_bf16=summary_bf16), Dev(w, summary_bf16=summary_bf16)
    L = w["seq_len"].copy()
    for step in range(4):
        L1 = L + 1                               # seq_len counts the new token
        phys = np.array([w["page_table"][b, L[b] // 64] for b in range(B)], np.int32)
        kn = bf(gen.rows_bf16(10, 100 + step, B * Hk).reshape(B, Hk, 128))
        vn = bf(gen.rows_bf16(10, 200 + step, B * Hk).reshape(B, Hk, 128))
        q = bf(gen.rows_bf16(10, 300 + step, B * Hq).reshape(B, Hq, 128))
        s_two = torch.empty(B, Hk, w["np_max"], dtype=torch.float32, device=DEV)
        s_one = torch.empty_like(s_two)
        spkv.paged_kv_append(two.cache, i32(phys), i32((L % 64).astype(np.int32)), kn, vn)
        spkv.score_blocks(two.cache, q, two.pt, i32(L1), s_two)
        spkv.decode_append_score(one.cache, kn, vn, q, one.pt, i32(L1), s_one)
        assert torch.equal(s_two, s_one)
        L = L1
    torch.cuda.synchronize()
    assert torch.equal(two.k_pool.view(torch.int16), one.k_pool.view(torch.int16))
    assert torch.equal(two.v_pool.view(torch.int16), one.v_pool.view(torch.int16))
    assert torch.equal(two.cnt, one.cnt)
    assert torch.equal(two.ksum, one.ksum)
    assert two.errors() == (0, 0) and one.errors() == (0, 0)
    two.close()
    one.close()


def test_decode_append_score_bad_local_page_flags_and_skips():
    B, Hk, Hq = 3, 2, 8
    w = gen.sparse_workload(B, Hq, Hk, 64 * 2 + 9, 4, 4, seed=8)
    d = Dev(w)
    before = d.k_pool.clone()
    pt = w["page_table"].copy()
    local = (w["seq_len"] - 1) // 64
    pt[1, local[1]] = w["n_phys"]                # request 1's local page is out of range
    kn = bf(gen.rows_bf16(11, 1, B * Hk).reshape(B, Hk, 128))
    vn = bf(gen.rows_bf16(11, 2, B * Hk).reshape(B, Hk, 128))
    s = torch.empty(B, Hk, w["np_max"], dtype=torch.float32, device=DEV)
    spkv.decode_append_score(d.cache, kn, vn, d.q, i32(pt), d.L, s)
    st, bits = d.errors()
    assert bits == spkv.DEVERR["PHYS"]
    changed = (d.k_pool.view(torch.int16) != before.view(torch.int16)).any(-1).nonzero().cpu().numpy()
    # only the rows at position seq_len - 1 of requests 0 and 2 changed (every kv head)
    want = sorted((h, int(w["page_table"][b, local[b]]), int((w["seq_len"][b] - 1) % 64))
                  for b in (0, 2) for h in range(Hk))
    assert sorted(map(tuple, changed.tolist())) == want
    assert torch.equal(s, d.scores())            # scores are unaffected by the append
    d.close()


# ------------------------------------------------------------------ block scores

def _score_bound(w):
    q = f64(w["q"])
    B, Hk, G = w["B"], w["Hk"], w["G"]
    bound = np.zeros((B, Hk, w["np_max"]))
    for b in range(B):
        for h in range(Hk):
            qs = np.abs(q[b, h * G:(h + 1) * G].sum(0))
            for p in range(w["np_max"]):
                keys = f64(w["k_pool"][h, w["page_table"][b, p]])
                m = np.abs(keys.reshape(4, 16, 128).mean(1))
                bound[b, h, p] = 2e-5 * (m @ qs).max() / math.sqrt(128) + 1e-7
    return bound


@pytest.mark.parametrize("which", ["tiny", "mid"])
def test_score_blocks_vs_oracle(which):
    w = gen.tiny() if which == "tiny" else gen.sparse_workload(3, 32, 8, 64 * 40 + 5, 8, 8, seed=7,
                                                                outlier_p=0.01)
    d = Dev(w)
    s = d.scores().cpu().numpy().astype(np.float64)
    ref = oracle.score_batch(w["q"], w["k_pool"], w["page_table"], w["seq_len"])
    assert np.array_equal(np.isinf(s), np.isinf(ref))
    fin = np.isfinite(ref)
    bound = _score_bound(w)
    diff = np.abs(s[fin] - ref[fin])
    assert (diff <= bound[fin]).all(), diff.max()
    assert d.errors() == (0, 0)
    d.close()


@pytest.mark.parametrize("which", ["tiny", "mid"])
def test_score_blocks_bf16_summaries_vs_oracle(which):
    """bf16 summaries: the GPU rounds its fixed-order fp32 sum, the oracle the exact sum, so a
    summary element may differ by one bf16 ulp (at most 2^-7 relative) on top of the fp32 bound."""
    w = gen.tiny() if which == "tiny" else gen.sparse_workload(3, 32, 8, 64 * 40 + 5, 8, 8, seed=7,
                                                                outlier_p=0.01)
    d = Dev(w, summary_bf16=True)
    assert d.ksum.dtype == torch.bfloat16
    s = d.scores().cpu().numpy().astype(np.float64)
    ref = oracle.score_batch(w["q"], w["k_pool"], w["page_table"], w["seq_len"], summary_bf16=True)
    assert np.array_equal(np.isinf(s), np.isinf(ref))
    fin = np.isfinite(ref)
    q = f64(w["q"])
    G = w["G"]
    ulp = np.zeros_like(ref)
    for b in range(w["B"]):
        for h in range(w["Hk"]):
            qs = np.abs(q[b, h * G:(h + 1) * G].sum(0))
            m = np.abs(f64(w["k_pool"][h, w["page_table"][b]]).reshape(-1, 4, 16, 128).mean(2))
            ulp[b, h] = 2.0 ** -7 * (m @ qs).max(1) / math.sqrt(128)
    diff = np.abs(s[fin] - ref[fin])
    assert (diff <= _score_bound(w)[fin] + ulp[fin]).all(), diff.max()
    # and the bf16 scores stay close to the fp32-summary ones
    s32 = oracle.score_batch(w["q"], w["k_pool"], w["page_table"], w["seq_len"])
    assert np.abs(s[fin] - s32[fin]).max() <= (ulp[fin] + _score_bound(w)[fin]).max()
    assert d.errors() == (0, 0)
    d.close()


# ------------------------------------------------------------------ selection

def _check_select_bitexact(d, s_dev, e_np, alive_dev, k_q, k_e):
    alive_before = alive_bits_to_bytes(alive_dev.cpu().numpy().view(np.uint32), d.npm)
    sel, n_sel = d.select(s_dev, f32(e_np), alive_dev, k_q, k_e)
    o_sel, o_n, o_alive = oracle.select_batch(s_dev.cpu().numpy().astype(np.float64),
                                              e_np.astype(np.float64), alive_before, d.w["seq_len"],
                                              k_q, k_e)
    assert np.array_equal(sel.cpu().numpy(), o_sel)
    assert np.array_equal(n_sel.cpu().numpy(), o_n)
    got_alive = alive_bits_to_bytes(alive_dev.cpu().numpy().view(np.uint32), d.npm)
    assert np.array_equal(got_alive, o_alive)       # bits past np_max are padding
    return sel, n_sel


@pytest.mark.parametrize("which", ["tiny", "mid", "ties", "fewcand"])
def test_select_bitexact_on_same_scores(which):
    if which == "fewcand":     # fewer candidates than the budgets
        w = gen.sparse_workload(2, 8, 2, 64 * 5 + 3, 8, 8, seed=2)
    elif which == "tiny":
        w = gen.tiny()
    else:
        w = gen.sparse_workload(4, 32, 8, 64 * 300 + 17, 24, 40, seed=11, outlier_p=0.01)
    d = Dev(w)
    s = d.scores()
    e = w["evict"].copy()
    if which == "ties":
        s = torch.round(s * 2) / 2
        e = np.round(e * 2) / 2
        e[..., ::7] = -0.0
        e[..., 3::7] = 0.0
    alive = d.new_alive()
    for step in range(3):
        _check_select_bitexact(d, s, e, alive, w["k_q"], w["k_e"])
        e = e + 0.3 * gen.normal_f32(1, 50 + step, e.size).reshape(e.shape)
        if which == "ties":
            e = np.round(e * 2) / 2
    assert d.errors() == (0, 0)
    d.close()


@pytest.mark.parametrize("np_max", [1, 32, 33, 128, 129, 256, 257, 512, 513, 1000, 1024, 1025])
def test_select_bitexact_across_context_sizes(np_max):
    """Both selection forms (one warp per unit up to 1024 pages, one CTA per unit above) on
    coarse scores with many exact ties, random alive masks, ragged contexts and budgets from 0
    to more than the candidates."""
    rng = np.random.default_rng(np_max)
    w = gen.sparse_workload(3, 4, 2, 64 * np_max, 8, 8, seed=np_max)
    w["seq_len"] = np.array([64 * np_max, max(1, 64 * np_max - 70), int(rng.integers(1, 64 * np_max + 1))],
                            np.int32)
    d = Dev(w)
    shape = (w["B"], w["Hk"], np_max)
    for k_q, k_e in [(8, 8), (0, 5), (5, 0), (np_max + 3, 2), (1, np_max)]:
        s = np.round(rng.standard_normal(shape) * 2) / 2
        s[rng.random(shape) < 0.1] = -0.0
        alive = rng.random(shape) < 0.7
        alive_dev = u32_as_i32(alive_bytes_to_bits(alive.astype(np.uint8)))
        for step in range(2):
            e = (np.round(rng.standard_normal(shape) * 3) / 3).astype(np.float32)
            _check_select_bitexact(d, f32(s), e, alive_dev, k_q, k_e)
    assert d.errors() == (0, 0)
    d.close()


@pytest.mark.parametrize("np_max, n_slots, times", [(96, 40, None), (512, 2048, None), (1000, 300, None),
                                                    (1500, 700, None), (96, 40, (0, 1, 9, 2, 3, 30, 4, 5)),
                                                    (1500, 700, (0, 1, 9, 2, 3, 30, 4, 5))])
def test_select_resident_update_equals_three_calls(np_max, n_slots, times):
    """The fused call (one kernel up to 1024 pages, three launches above) against select_topk +
    resident_setdiff + lru_bucket_update on copies of the same state, and both against the oracle,
    bit for bit, over a trajectory whose residency buffer fills and recycles.  With `times`, the
    clock steps back twice, so some slots carry timestamps later than t (age 0, bucket 0)."""
    w = gen.sparse_workload(3, 8, 2, 64 * np_max - 5, 10, 6, seed=np_max)
    d = Dev(w)
    B, Hk = w["B"], w["Hk"]
    U, k_q, k_e = B * Hk, w["k_q"], w["k_e"]
    stride = k_q + k_e + 1
    rng = np.random.default_rng(np_max)
    shape = (B, Hk, np_max)

    def state():
        return dict(alive=d.new_alive(), resident=i32(np.full((U, n_slots), -1, np.int32)),
                    ts=i32(np.full((U, n_slots), np.iinfo(np.int32).min, np.int32)))

    def outputs():
        z = lambda *sh: torch.empty(*sh, dtype=torch.int32, device=DEV)
        return dict(sel=z(B, Hk, stride), n_sel=z(B, Hk), missing=z(U, stride), n_missing=z(U), slot=z(U, stride),
                    victims=z(U, stride), hist=z(U, 64))

    a, b = state(), state()
    h_alive = np.ones(shape, np.uint8)
    h_res = np.full((U, n_slots), -1, np.int32)
    h_ts = np.full((U, n_slots), np.iinfo(np.int32).min, np.int32)
    saw_future = False
    for t in (range(8) if times is None else times):
        saw_future |= bool(((h_res >= 0) & (h_ts > t)).any())
        s = (np.round(rng.standard_normal(shape) * 4) / 4).astype(np.float32)
        e = (np.round(rng.standard_normal(shape) * 4) / 4).astype(np.float32)
        s_d, e_d = f32(s), f32(e)
        fa, fb = outputs(), outputs()
        spkv.select_resident_update(d.cache, s_d, e_d, a["alive"], d.L, k_q, k_e, fa["sel"], fa["n_sel"],
                                    a["resident"], a["ts"], t, 2, fa["missing"], fa["n_missing"], fa["slot"],
                                    fa["victims"], fa["hist"])
        spkv.select_topk(d.cache, s_d, e_d, b["alive"], d.L, k_q, k_e, fb["sel"], fb["n_sel"])
        spkv.resident_setdiff(d.cache, b["resident"], fb["sel"], fb["n_sel"], fb["missing"], fb["n_missing"],
                              fb["slot"])
        spkv.lru_bucket_update(d.cache, b["resident"], b["ts"], fb["slot"], fb["n_sel"].view(U), fb["missing"],
                               fb["n_missing"], t, 2, fb["victims"], fb["hist"])
        torch.cuda.synchronize()
        for k in fa:
            assert torch.equal(fa[k], fb[k]), k
        for k in a:
            assert torch.equal(a[k], b[k]), k
        o_sel, o_n, h_alive = oracle.select_batch(s.astype(np.float64), e.astype(np.float64), h_alive,
                                                  w["seq_len"], k_q, k_e)
        o_miss, o_nm, o_slot = oracle.setdiff_batch(h_res, o_sel.reshape(U, stride), o_n.reshape(U))
        h_res, h_ts, o_vic, o_hist = oracle.lru_batch(h_res, h_ts, o_slot, o_n.reshape(U), o_miss, o_nm, t, 2)
        assert np.array_equal(fa["sel"].cpu().numpy(), o_sel) and np.array_equal(fa["n_sel"].cpu().numpy(), o_n)
        assert np.array_equal(fa["missing"].cpu().numpy(), o_miss)
        assert np.array_equal(fa["n_missing"].cpu().numpy(), o_nm)
        assert np.array_equal(fa["slot"].cpu().numpy(), o_slot)
        assert np.array_equal(fa["victims"].cpu().numpy(), o_vic)
        assert np.array_equal(fa["hist"].cpu().numpy(), o_hist)
        assert np.array_equal(a["resident"].cpu().numpy(), h_res) and np.array_equal(a["ts"].cpu().numpy(), h_ts)
        assert np.array_equal(alive_bits_to_bytes(a["alive"].cpu().numpy().view(np.uint32), np_max), h_alive)
    assert saw_future == (times is not None)
    assert d.errors() == (0, 0)
    d.close()


def test_select_vs_oracle_scores_with_near_tie_rule():
    w = gen.sparse_workload(4, 32, 8, 64 * 200 + 9, 16, 16, seed=13, outlier_p=0.01)
    d = Dev(w)
    sel, n_sel = d.select(d.scores(), f32(w["evict"]), d.new_alive(), w["k_q"], w["k_e"])
    sel, n_sel = sel.cpu().numpy(), n_sel.cpu().numpy()
    s_or = oracle.score_batch(w["q"], w["k_pool"], w["page_table"], w["seq_len"])
    o_sel, o_n, o_alive = oracle.select_batch(s_or, w["evict"], np.ones(s_or.shape, np.uint8),
                                              w["seq_len"], w["k_q"], w["k_e"])
    local = (w["seq_len"] - 1) // 64
    for b in range(w["B"]):
        for h in range(w["Hk"]):
            E = {p for p in range(local[b]) if o_alive[b, h, p]}
            g = set(sel[b, h, :n_sel[b, h] - 1].tolist())
            o = set(o_sel[b, h, :o_n[b, h] - 1].tolist())
            assert E <= g, "eviction-head set ranks identical fp32 scores and must match"
            cand = sorted((p for p in range(local[b]) if p not in E), key=lambda p: -s_or[b, h, p])
            kth = s_or[b, h, cand[w["k_q"] - 1]]
            for p in g ^ o:
                assert abs(s_or[b, h, p] - kth) <= 1e-5 * abs(kth), (b, h, p)
    d.close()


# ------------------------------------------------------------------ sparse attention

def _random_lists(w, rng, stride, lens=None):
    B, Hk = w["B"], w["Hk"]
    sel = np.full((B, Hk, stride), -1, np.int32)
    n_sel = np.zeros((B, Hk), np.int32)
    for b in range(B):
        npg = (int(w["seq_len"][b]) + 63) // 64
        for h in range(Hk):
            n = int(rng.integers(0, min(stride, npg) + 1)) if lens is None else min(lens, npg)
            pages = np.sort(rng.choice(npg, size=n, replace=False))
            sel[b, h, :n] = pages
            n_sel[b, h] = n
    return sel, n_sel


@pytest.mark.parametrize("B,Hq,Hk", [(1, 8, 2), (5, 16, 4), (3, 40, 8), (2, 16, 1), (4, 8, 8),
                                     (2, 40, 4), (3, 6, 2), (2, 6, 3)])
def test_sparse_attn_random_lists(B, Hq, Hk):
    rng = np.random.default_rng(B * 100 + Hq + Hk)
    w = gen.sparse_workload(B, Hq, Hk, 64 * 48, 8, 8, seed=B + Hq, outlier_p=0.01)
    w["seq_len"] = rng.integers(1, 64 * 48 + 1, B).astype(np.int32)
    w["seq_len"][0] = 64 * 48
    d = Dev(w)
    sel, n_sel = _random_lists(w, rng, stride=20)
    out, lse = d.attn(i32(sel), i32(n_sel))
    ro, rl = oracle.sparse_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["page_table"], sel, n_sel,
                                      w["seq_len"])
    mx, mean = attn_errors(out.cpu().numpy(), ro)
    assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (mx, mean)
    l = lse.cpu().numpy()
    assert np.array_equal(np.isinf(l), np.isinf(rl))
    fin = np.isfinite(rl)
    assert np.abs(l[fin] - rl[fin]).max() <= LSE_TOL
    assert d.errors() == (0, 0)
    d.close()


@pytest.mark.parametrize("B,n_pages", [(16, 65), (125, 2), (40, 33)])
def test_sparse_attn_split_k_paths(B, n_pages):
    """Units split over several CTAs (partial merge) and CTAs that cover many whole units."""
    rng = np.random.default_rng(B)
    w = gen.sparse_workload(B, 32, 8, 64 * 70 + 11, 8, 8, seed=B)
    d = Dev(w, max_units=B * 8)
    sel, n_sel = _random_lists(w, rng, stride=n_pages, lens=n_pages)
    out, lse = d.attn(i32(sel), i32(n_sel))
    ro, rl = oracle.sparse_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["page_table"], sel, n_sel,
                                      w["seq_len"])
    mx, mean = attn_errors(out.cpu().numpy(), ro)
    assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (mx, mean)
    assert np.abs(lse.cpu().numpy() - rl).max() <= LSE_TOL
    # a second call reuses the arrival counters: must give the same bits
    out2, lse2 = d.attn(i32(sel), i32(n_sel))
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    assert d.errors() == (0, 0)
    d.close()


def test_attn_never_reads_rows_past_valid():
    w = gen.sparse_workload(2, 8, 2, 64 * 10 - 20, 4, 4, seed=21)
    local_phys = w["page_table"][:, 9]
    w_nan = dict(w)
    w_nan["k_pool"] = w["k_pool"].copy()
    w_nan["v_pool"] = w["v_pool"].copy()
    for b in range(2):
        w_nan["k_pool"][:, local_phys[b], 44:] = 0x7FC0     # bf16 NaN
        w_nan["v_pool"][:, local_phys[b], 44:] = 0x7FC0
    d = Dev(w_nan)
    sel = np.tile(np.arange(10, dtype=np.int32), (2, 2, 1))
    n_sel = np.full((2, 2), 10, np.int32)
    out, lse = d.attn(i32(sel), i32(n_sel))
    o = out.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(lse.cpu().numpy()).all()
    ro, rl = oracle.sparse_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["page_table"], sel, n_sel,
                                      w["seq_len"])
    assert attn_errors(o, ro)[0] <= ATTN_MAX
    d.close()


def test_bad_device_ids_set_error_bits_without_fault():
    w = gen.sparse_workload(2, 8, 2, 64 * 10, 4, 4, seed=22)
    d = Dev(w)
    sel = np.tile(np.arange(10, dtype=np.int32), (2, 2, 1))
    sel[0, 1, 3] = 10 ** 6
    sel[1, 0, 0] = -5
    n_sel = np.full((2, 2), 10, np.int32)
    out, lse = d.attn(i32(sel), i32(n_sel))
    st, bits = d.errors()
    assert st == -4 and bits & spkv.DEVERR["PAGE_ID"]
    ro, rl = oracle.sparse_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["page_table"], sel, n_sel,
                                      w["seq_len"], units=np.array([0, 3]))
    o = out.cpu().numpy()
    assert attn_errors(o[0, :4], ro[0, :4])[0] <= ATTN_MAX      # unit 0 untouched by the bad ids
    assert attn_errors(o[1, 4:], ro[1, 4:])[0] <= ATTN_MAX      # unit 3
    assert d.errors() == (0, 0)                                  # the word was cleared
    d.close()


# ------------------------------------------------------------------ lazy RoPE attention

def _lazy_dev(w):
    k_pool, v_pool = bf(w["k_pool"]), bf(w["v_pool"])
    ksum = torch.zeros(w["Hk"], w["n_phys"], 4, 128, dtype=torch.float32, device=DEV)
    cache = spkv.paged_kv_create(k_pool, v_pool, ksum, i32(w["page_cnt"]))
    return cache, (k_pool, v_pool, ksum)


def _words(phys, valid, slot):
    ok = phys >= 0
    words = np.zeros(phys.shape, np.uint32)
    words[ok] = spkv.pack_page_words(phys[ok], valid[ok], slot[ok])
    return words


@pytest.mark.parametrize("seed,Hq,Hk", [(1, 16, 4), (2, 32, 8), (3, 8, 1), (4, 12, 4), (5, 4, 4)])
def test_lazy_rope_vs_materialised_oracle(seed, Hq, Hk):
    w = gen.lazy_rag(seed=seed, B=6, Hq=Hq, Hk=Hk, n_docs=20, docs_per_req=4, min_len=100, max_len=2000)
    cache, keep = _lazy_dev(w)
    words = _words(w["phys"], w["valid"], w["slot"])
    B = w["B"]
    out = torch.empty(B, Hq, 128, dtype=torch.float32, device=DEV)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=DEV)
    spkv.lazy_rope_decode_attn(cache, bf(w["q"]), i32(w["qpos"]), u32_as_i32(words), i32(w["n_pages"]),
                               i32(w["doc_pos"]), w["theta"], out, lse)
    ro, rl = oracle.lazy_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"],
                                    w["n_pages"], w["qpos"], w["doc_pos"], w["theta"], materialise=True)
    mx, mean = attn_errors(out.cpu().numpy(), ro)
    assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (mx, mean)
    assert np.abs(lse.cpu().numpy() - rl).max() <= LSE_TOL
    assert spkv.get_device_error(cache) == (0, 0)
    cache.close()


def test_lazy_rope_per_head_page_lists():
    w = gen.lazy_rag(seed=4, B=3, Hq=16, Hk=4, n_docs=10, docs_per_req=3, min_len=64, max_len=1500)
    rng = np.random.default_rng(0)
    B, Hk, npm = w["B"], w["Hk"], w["np_max"]
    phys = np.full((B, Hk, npm), -1, np.int32)
    valid = np.zeros((B, Hk, npm), np.int32)
    slot = np.zeros((B, Hk, npm), np.int32)
    n_pages = np.zeros(B, np.int32)
    for b in range(B):
        n = int(w["n_pages"][b])
        keep = n // 2
        n_pages[b] = keep
        for h in range(Hk):
            idx = np.sort(rng.choice(n, size=keep, replace=False))
            phys[b, h, :keep] = w["phys"][b, idx]
            valid[b, h, :keep] = w["valid"][b, idx]
            slot[b, h, :keep] = w["slot"][b, idx]
    cache, keep_alive = _lazy_dev(w)
    words = _words(phys, valid, slot)
    out = torch.empty(B, w["Hq"], 128, dtype=torch.float32, device=DEV)
    lse = torch.empty(B, w["Hq"], dtype=torch.float32, device=DEV)
    spkv.lazy_rope_decode_attn(cache, bf(w["q"]), i32(w["qpos"]), u32_as_i32(words), i32(n_pages),
                               i32(w["doc_pos"]), w["theta"], out, lse)
    ro, rl = oracle.lazy_attn_batch(w["q"], w["k_pool"], w["v_pool"], phys, valid, slot, n_pages,
                                    w["qpos"], w["doc_pos"], w["theta"], materialise=True)
    mx, mean = attn_errors(out.cpu().numpy(), ro)
    assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (mx, mean)
    cache.close()


# ------------------------------------------------------------------ residency bookkeeping

@pytest.mark.parametrize("W", [1, 2])
def test_setdiff_and_lru_trajectory_bitexact(W):
    rng = np.random.default_rng(W)
    U, n_slots, stride = 6, 64, 9
    w = gen.tiny()
    d = Dev(w)
    resident = np.full((U, n_slots), -1, np.int32)
    ts = np.full((U, n_slots), np.iinfo(np.int32).min, np.int32)
    r_dev, t_dev = i32(resident), i32(ts)
    for t in range(40):
        sel = np.full((U, stride), -1, np.int32)
        n_sel = np.zeros(U, np.int32)
        for u in range(U):
            n = int(rng.integers(0, stride + 1))
            sel[u, :n] = np.sort(rng.choice(150, size=n, replace=False))
            n_sel[u] = n
        miss = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        nm = torch.empty(U, dtype=torch.int32, device=DEV)
        slot = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        spkv.resident_setdiff(d.cache, r_dev, i32(sel), i32(n_sel), miss, nm, slot)
        o_miss, o_nm, o_slot = oracle.setdiff_batch(resident, sel, n_sel)
        assert np.array_equal(miss.cpu().numpy(), o_miss)
        assert np.array_equal(nm.cpu().numpy(), o_nm)
        assert np.array_equal(slot.cpu().numpy(), o_slot)
        vic = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        hist = torch.empty(U, 64, dtype=torch.int32, device=DEV)
        spkv.lru_bucket_update(d.cache, r_dev, t_dev, slot, i32(n_sel), miss, nm, t, W, vic, hist)
        resident, ts, o_vic, o_hist = oracle.lru_batch(resident, ts, o_slot, n_sel, o_miss, o_nm, t, W)
        assert np.array_equal(vic.cpu().numpy(), o_vic)
        assert np.array_equal(hist.cpu().numpy(), o_hist)
        assert np.array_equal(r_dev.cpu().numpy(), resident)
        assert np.array_equal(t_dev.cpu().numpy(), ts)
    assert d.errors() == (0, 0)
    d.close()


# ------------------------------------------------------------------ more shapes and edge cases

@pytest.mark.parametrize("Hq,Hk", [(32, 2), (24, 2), (12, 1)])
def test_lazy_rope_large_groups(Hq, Hk):
    """Group sizes 9..16 take the two-n-tile path of the kernel (16 query heads per tile)."""
    w = gen.lazy_rag(seed=7, B=3, Hq=Hq, Hk=Hk, n_docs=8, docs_per_req=3, min_len=64, max_len=1200)
    cache, keep = _lazy_dev(w)
    words = _words(w["phys"], w["valid"], w["slot"])
    B = w["B"]
    out = torch.empty(B, Hq, 128, dtype=torch.float32, device=DEV)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=DEV)
    spkv.lazy_rope_decode_attn(cache, bf(w["q"]), i32(w["qpos"]), u32_as_i32(words), i32(w["n_pages"]),
                               i32(w["doc_pos"]), w["theta"], out, lse)
    ro, rl = oracle.lazy_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"],
                                    w["n_pages"], w["qpos"], w["doc_pos"], w["theta"], materialise=True)
    mx, mean = attn_errors(out.cpu().numpy(), ro)
    assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (mx, mean)
    assert np.abs(lse.cpu().numpy() - rl).max() <= LSE_TOL
    cache.close()


def test_all_units_empty():
    w = gen.sparse_workload(3, 8, 2, 64 * 4, 2, 2, seed=1)
    d = Dev(w)
    sel = np.full((3, 2, 5), -1, np.int32)
    n_sel = np.zeros((3, 2), np.int32)
    out, lse = d.attn(i32(sel), i32(n_sel))
    assert (out.cpu().numpy() == 0).all() and np.isneginf(lse.cpu().numpy()).all()
    out2, lse2 = d.attn(i32(sel), i32(n_sel))     # the chunk counter must be intact
    assert torch.equal(out, out2)
    assert d.errors() == (0, 0)
    d.close()


def test_large_budgets_and_long_context_selection():
    """k = 600 pages of 2047 candidates: several radix passes with many ties at the threshold."""
    w = gen.sparse_workload(2, 8, 2, 64 * 2048, 300, 300, seed=17, extra_tokens=0)
    d = Dev(w)
    s = d.scores()
    s = torch.round(s * 8) / 8                      # coarse scores: many exact ties
    e = np.round(w["evict"] * 4) / 4
    alive = d.new_alive()
    sel, n_sel = _check_select_bitexact(d, s, e, alive, w["k_q"], w["k_e"])
    out, lse = d.attn(sel, n_sel)
    ro, rl = oracle.sparse_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["page_table"], sel.cpu().numpy(),
                                      n_sel.cpu().numpy(), w["seq_len"])
    mx, mean = attn_errors(out.cpu().numpy(), ro)
    assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (mx, mean)
    assert d.errors() == (0, 0)
    d.close()


def test_one_unit_many_pages_split_across_all_ctas():
    """A single (request, kv head) unit of 2000 pages: the split-K merge of hundreds of parts."""
    w = gen.sparse_workload(1, 4, 1, 64 * 2000 + 5, 8, 8, seed=23)
    d = Dev(w)
    n = 2001
    sel = np.arange(n, dtype=np.int32).reshape(1, 1, n)
    n_sel = np.full((1, 1), n, np.int32)
    out, lse = d.attn(i32(sel), i32(n_sel))
    ro, rl = oracle.sparse_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["page_table"], sel, n_sel, w["seq_len"])
    mx, mean = attn_errors(out.cpu().numpy(), ro)
    assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (mx, mean)
    assert np.abs(lse.cpu().numpy() - rl).max() <= LSE_TOL
    assert d.errors() == (0, 0)
    d.close()
