"""GPU parity of the LazyAttention prefill kernel (tcgen05) against the fp64 oracle.

The oracle materialises keys rotated to their absolute positions; the kernel rotates each query
row once per document and runs QK^T and PV on the tensor cores with bf16 operands and fp32
accumulation, so the rotated query enters them rounded once to bf16 (reading R20).  Acceptance:

* against the exact oracle, the attention output within the decode tolerance (max 1e-2, mean
  1e-3) at the pages' input scale, and every row's LSE within the bound that rounding implies:
  each score moves by at most 2^-8 sum_i |q'_i| |k_i| / sqrt(128), at most 2^-8 sum over the
  64 rotation pairs of |q pair| |k pair| / sqrt(128) (a rotation keeps each pair's norm), and a
  log-sum-exp moves by at most the largest move among its terms;
* against the oracle's bf16-rounded-query form (the same rounding, exact elsewhere), output and
  LSE within (1e-2, 1e-3, 1e-3);
* inputs scaled by c (stress cases) move every score, and every error above, c times as much:
  those tolerances are multiplied by c.
Each case also checks the relative L2 error of the whole output, so that small outputs (long,
flat softmaxes) still test something.  The ALiBi form does not rotate the query (it enters the
tensor cores exactly), so it is held to (1e-2, 1e-3, 1e-3) against the exact oracle directly.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import sparse_paged_kv_score_gb300 as spkv
from helpers import DEV, attn_errors, bf, i32, u32_as_i32

pytestmark = pytest.mark.gpu

ATTN_MAX, ATTN_MEAN, LSE_TOL, REL_L2 = 1e-2, 1e-3, 1e-3, 2e-2
U_BF16 = 2.0 ** -8          # unit roundoff of bf16 (8 significant bits, nearest)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_paged_kv_score_gb300 import build
    build.build()
    spkv.load()


def _cache(w):
    k_pool, v_pool = bf(w["k_pool"]), bf(w["v_pool"])
    ksum = torch.zeros(w["Hk"], w["n_phys"], 4, 128, dtype=torch.float32, device=DEV)
    cache = spkv.paged_kv_create(k_pool, v_pool, ksum, i32(w["page_cnt"]))
    return cache, (k_pool, v_pool, ksum)


def _words(phys, valid, slot):
    ok = phys >= 0
    words = np.zeros(phys.shape, np.uint32)
    words[ok] = spkv.pack_page_words(phys[ok], valid[ok], slot[ok])
    return words


def _queries(seed, B, T, Hq, scale):
    q = gen.rows_bf16(seed, 4242, B * T * Hq).reshape(B, T, Hq, 128)
    if scale != 1.0:
        q = gen.f32_to_bf16(gen.bf16_to_f32(q) * np.float32(scale))
    return q


def _run(w, q, phys, valid, slot, n_pages, qpos0, doc_pos):
    B, T, Hq = q.shape[0], q.shape[1], q.shape[2]
    cache, keep = _cache(w)
    words = _words(phys, valid, slot)
    out = torch.full((B, T, Hq, 128), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((B, T, Hq), float("nan"), dtype=torch.float32, device=DEV)
    spkv.lazy_rope_prefill_attn(cache, bf(q), i32(qpos0), u32_as_i32(words), i32(n_pages), i32(doc_pos),
                                w["theta"], out, lse)
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert spkv.get_device_error(cache) == (0, 0)
    cache.close()
    return o, l


def _check(o, l, ro, rl, scale=1.0, lse_bound=None):
    mx, mean = attn_errors(o, ro)
    assert mx <= ATTN_MAX * scale and mean <= ATTN_MEAN * scale, (mx, mean)
    rel = np.linalg.norm((o - ro).ravel()) / max(np.linalg.norm(ro.ravel()), 1e-30)
    assert rel <= REL_L2, rel
    assert np.array_equal(np.isinf(l), np.isinf(rl))
    fin = np.isfinite(rl)
    tol = LSE_TOL * scale if lse_bound is None else lse_bound[fin]
    assert (np.abs(l[fin] - rl[fin]) <= tol).all(), np.abs(l[fin] - rl[fin]).max()
    return mx, mean, rel


def _pair_norms(x):
    x = gen.bf16_to_f32(x).astype(np.float64)
    return np.hypot(x[..., :64], x[..., 64:])


def _lse_bound(w, q, phys, valid, slot, page_start, n_pages, qpos0, doc_pos, causal=False):
    """Per (request, row, query head): 2^-8 max over the row's visible keys of
    sum over rotation pairs |q pair| |k pair| / sqrt(128), plus 1e-5 for the fp32 arithmetic."""
    B, T, Hq, _ = q.shape
    Hk = w["Hk"]
    G = Hq // Hk
    if phys.ndim == 2:
        phys, valid, slot, page_start = (a[:, None, :] for a in (phys, valid, slot, page_start))
    out = np.zeros((B, T, Hq))
    for b in range(B):
        n = n_pages[b]
        for h in range(Hk):
            mh = 0 if phys.shape[1] == 1 else h
            rows, pos = [], []
            for i in range(n):
                v = valid[b, mh, i]
                rows.append(_pair_norms(w["k_pool"][h, phys[b, mh, i], :v]))
                pos.append(doc_pos[b, slot[b, mh, i]] + page_start[b, mh, i] + np.arange(v))
            if not rows:
                continue
            rk, pos = np.concatenate(rows), np.concatenate(pos)
            rq = _pair_norms(q[b, :, h * G:(h + 1) * G])            # [T][G][64]
            m = rq @ rk.T                                           # [T][G][keys]
            if causal:
                m = np.where(pos[None, None, :] <= (qpos0[b] + np.arange(T))[:, None, None], m, 0.0)
            out[b, :, h * G:(h + 1) * G] = U_BF16 * m.max(-1) / np.sqrt(128.0)
    return out + 1e-5


def _check_rope(w, q, o, l, phys, valid, slot, page_start, n_pages, qpos0, doc_pos, scale=1.0, causal=False,
                items=None):
    """Both acceptance checks of a RoPE prefill result (module docstring)."""
    args = (q, w["k_pool"], w["v_pool"], phys, valid, slot, page_start, n_pages, qpos0, doc_pos, w["theta"])
    ex, exl = oracle.prefill_step_batch(*args, mode="materialised", items=items)
    rq, rql = oracle.prefill_step_batch(*args, mode="lazy_bf16q", items=items)
    bound = _lse_bound(w, q, phys, valid, slot, page_start, n_pages, qpos0, doc_pos, causal)   # scales by itself
    sel = _item_rows(items, q.shape, w["Hk"])
    _check(sel(o), sel(l), sel(ex), sel(exl), scale=scale, lse_bound=sel(bound))
    _check(sel(o), sel(l), sel(rq), sel(rql), scale=scale)


def _item_rows(items, shape, Hk):
    """Selects the (b, t, kv head) work items' rows of [B][T][Hq](...) arrays (all when None)."""
    if items is None:
        return lambda a: a
    B, T, Hq = shape[:3]
    G = Hq // Hk
    idx = [(it // Hk // T, it // Hk % T, it % Hk) for it in items]
    return lambda a: np.array([a[b, t, h * G:(h + 1) * G] for b, t, h in idx])


@pytest.mark.parametrize("seed,Hq,Hk,T", [(1, 8, 2, 5), (2, 16, 4, 128), (3, 8, 8, 200), (4, 32, 2, 33),
                                          (5, 4, 1, 129)])
def test_prefill_vs_materialised_oracle(seed, Hq, Hk, T):
    """Tiles of 128 rows with ragged tails, group sizes 1..16, partial last pages of documents."""
    w = gen.lazy_rag(seed=seed, B=3, Hq=Hq, Hk=Hk, n_docs=12, docs_per_req=4, min_len=70, max_len=900)
    q = _queries(seed, w["B"], T, Hq, 1.0)
    o, l = _run(w, q, w["phys"], w["valid"], w["slot"], w["n_pages"], w["qpos"], w["doc_pos"])
    _check_rope(w, q, o, l, w["phys"], w["valid"], w["slot"], w["page_start"], w["n_pages"], w["qpos"], w["doc_pos"])


@pytest.mark.parametrize("seed,Hq,Hk,T", [(1, 8, 2, 5), (2, 16, 4, 128), (4, 32, 2, 33)])
def test_prefill_queries_scaled_three_times(seed, Hq, Hk, T):
    """Queries three times the unit scale: every score, hence every rounding error, moves three times
    as much, and the tolerances scale with it."""
    w = gen.lazy_rag(seed=seed, B=3, Hq=Hq, Hk=Hk, n_docs=12, docs_per_req=4, min_len=70, max_len=900)
    q = _queries(seed, w["B"], T, Hq, 3.0)
    o, l = _run(w, q, w["phys"], w["valid"], w["slot"], w["n_pages"], w["qpos"], w["doc_pos"])
    _check_rope(w, q, o, l, w["phys"], w["valid"], w["slot"], w["page_start"], w["n_pages"], w["qpos"], w["doc_pos"],
                scale=3.0)


def test_prefill_long_documents_rescale_path():
    """Hundreds of pages per request, the keys of each request's last document scaled x3: the
    running row maximum jumps by far more than 2^8 when that document is reached, so the O
    rescale in tensor memory runs."""
    w = gen.lazy_rag(seed=9, B=2, Hq=8, Hk=2, n_docs=8, docs_per_req=8, min_len=2000, max_len=4096)
    last = np.unique(w["phys"][w["slot"] == 7])
    last = last[last >= 0]
    w["k_pool"][:, last] = gen.f32_to_bf16(gen.bf16_to_f32(w["k_pool"][:, last]) * np.float32(3.0))
    q = _queries(9, w["B"], 130, 8, 1.0)
    o, l = _run(w, q, w["phys"], w["valid"], w["slot"], w["n_pages"], w["qpos"], w["doc_pos"])
    items = np.array([i for i in range(w["B"] * 130 * w["Hk"]) if i % 37 == 0], np.int32)
    # the x3 keys dominate every row: scale 3 (the LSE bound follows the keys by itself)
    _check_rope(w, q, o, l, w["phys"], w["valid"], w["slot"], w["page_start"], w["n_pages"], w["qpos"], w["doc_pos"],
                scale=3.0, items=items)


def test_prefill_row_maximum_growing_inside_a_page_group():
    """A row's maximum jumping by more than 2^8 inside a group of two pages: keys set to zero
    before, and keys scaled x3 in, the last 32 tokens of (A) a request's first page (the first
    group's second 32-key block) and (B) the fourth page of another request's first document
    (the second group's fourth block: O is rescaled there).  The keys that dominate are three times
    the unit scale: scale 3."""
    w = gen.lazy_rag(seed=13, B=3, Hq=8, Hk=2, n_docs=6, docs_per_req=3, min_len=300, max_len=900)
    B = w["B"]
    kp = gen.bf16_to_f32(w["k_pool"])

    def first_doc(b):
        n = int(w["n_pages"][b])
        sl = w["slot"][b, :n]
        end = next((i for i in range(1, n) if sl[i] != sl[0]), n)
        return w["phys"][b, :end], w["valid"][b, :end]

    pa, va = first_doc(0)
    assert va[0] == 64
    kp[:, pa[0], 0:32] = 0.0
    kp[:, pa[0], 32:64] *= np.float32(3.0)
    case_b = False
    for b in range(1, B):
        pb, vb = first_doc(b)
        if len(pb) >= 4 and (vb[:4] == 64).all() and not set(pb[:4].tolist()) & set(pa.tolist()):
            kp[:, pb[:3]] = 0.0
            kp[:, pb[3], 0:32] = 0.0
            kp[:, pb[3], 32:64] *= np.float32(3.0)
            case_b = True
            break
    assert case_b
    w["k_pool"] = gen.f32_to_bf16(kp)
    q = _queries(13, B, 70, 8, 1.0)
    o, l = _run(w, q, w["phys"], w["valid"], w["slot"], w["n_pages"], w["qpos"], w["doc_pos"])
    assert np.isfinite(l).all()
    _check_rope(w, q, o, l, w["phys"], w["valid"], w["slot"], w["page_start"], w["n_pages"], w["qpos"], w["doc_pos"],
                scale=3.0)


def test_prefill_per_head_page_lists_and_empty_request():
    """Per-kv-head page lists in a different order per head, and a request without pages."""
    w = gen.lazy_rag(seed=6, B=3, Hq=8, Hk=2, n_docs=10, docs_per_req=3, min_len=64, max_len=700)
    rng = np.random.default_rng(6)
    B, Hk, npm = w["B"], w["Hk"], w["np_max"]
    phys = np.full((B, Hk, npm), -1, np.int32)
    valid = np.zeros((B, Hk, npm), np.int32)
    slot = np.zeros((B, Hk, npm), np.int32)
    pstart = np.zeros((B, Hk, npm), np.int32)
    n_pages = w["n_pages"].copy()
    n_pages[1] = 0
    for b in range(B):
        n = n_pages[b]
        for h in range(Hk):
            perm = rng.permutation(n) if h % 2 else np.arange(n)   # pages of a head in any order
            phys[b, h, :n] = w["phys"][b, perm]
            valid[b, h, :n] = w["valid"][b, perm]
            slot[b, h, :n] = w["slot"][b, perm]
            pstart[b, h, :n] = w["page_start"][b, perm]
    q = _queries(6, B, 70, 8, 1.0)
    o, l = _run(w, q, phys, valid, slot, n_pages, w["qpos"], w["doc_pos"])
    assert (o[1] == 0).all() and np.isneginf(l[1]).all()
    _check_rope(w, q, o, l, phys, valid, slot, pstart, n_pages, w["qpos"], w["doc_pos"])


def test_prefill_bad_page_words_flag_without_fault():
    w = gen.lazy_rag(seed=7, B=2, Hq=4, Hk=1, n_docs=4, docs_per_req=2, min_len=64, max_len=300)
    words = _words(w["phys"], w["valid"], w["slot"])
    words[0, 0] = (words[0, 0] & ~np.uint32(0x3FFFF)) | np.uint32((1 << 18) - 1)   # physical page out of range
    words[1, 1] = (words[1, 1] & np.uint32(0x00FFFFFF)) | np.uint32(200 << 24)       # document slot out of range
    cache, keep = _cache(w)
    out = torch.empty(2, 3, 4, 128, dtype=torch.float32, device=DEV)
    lse = torch.empty(2, 3, 4, dtype=torch.float32, device=DEV)
    q = _queries(7, 2, 3, 4, 1.0)
    spkv.lazy_rope_prefill_attn(cache, bf(q), i32(w["qpos"]), u32_as_i32(words), i32(w["n_pages"]),
                                i32(w["doc_pos"]), w["theta"], out, lse)
    st, bits = spkv.get_device_error(cache)
    assert bits == (spkv.DEVERR["PHYS"] | spkv.DEVERR["SLOT"])
    assert torch.isfinite(out).all()
    cache.close()


# ------------------------------------------------------------------ ALiBi form

def _slopes(Hq):
    """A geometric set of slopes, one per query head (the values do not matter to parity)."""
    return (2.0 ** (-8.0 * (np.arange(Hq) + 1) / Hq)).astype(np.float32)


def _run_alibi(w, q, phys, valid, slot, page_start, n_pages, qpos0, doc_pos, slopes):
    B, T, Hq = q.shape[0], q.shape[1], q.shape[2]
    cache, keep = _cache(w)
    words = _words(phys, valid, slot)
    out = torch.full((B, T, Hq, 128), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((B, T, Hq), float("nan"), dtype=torch.float32, device=DEV)
    spkv.lazy_alibi_prefill_attn(cache, bf(q), i32(qpos0), u32_as_i32(words), i32(n_pages), i32(page_start),
                                 i32(doc_pos), torch.from_numpy(slopes).to(DEV), out, lse)
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert spkv.get_device_error(cache) == (0, 0)
    cache.close()
    return o, l


@pytest.mark.parametrize("seed,Hq,Hk,T", [(11, 8, 2, 5), (12, 16, 4, 128), (13, 8, 8, 200), (14, 32, 2, 33)])
def test_alibi_prefill_vs_oracle(seed, Hq, Hk, T):
    """Tiles of 128 rows with ragged tails, group sizes 1..16, documents at unaligned offsets:
    the bias spans hundreds of nats across a request, so the running maximum moves and O is
    rescaled as nearer documents arrive."""
    w = gen.lazy_rag(seed=seed, B=3, Hq=Hq, Hk=Hk, n_docs=12, docs_per_req=4, min_len=70, max_len=900)
    q = _queries(seed, w["B"], T, Hq, 1.0)
    sl = _slopes(Hq)
    o, l = _run_alibi(w, q, w["phys"], w["valid"], w["slot"], w["page_start"], w["n_pages"], w["qpos"],
                      w["doc_pos"], sl)
    ro, rl = oracle.alibi_prefill_batch(q, w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"],
                                        w["page_start"], w["n_pages"], w["qpos"], w["doc_pos"], sl)
    _check(o, l, ro, rl)


def test_alibi_prefill_per_head_page_order_and_empty_request():
    """Positions come from doc_pos and page_start, not from the list order: per-kv-head page lists
    in different orders give the oracle's result; a request without pages gives 0 and -inf."""
    w = gen.lazy_rag(seed=15, B=3, Hq=8, Hk=2, n_docs=10, docs_per_req=3, min_len=64, max_len=700)
    rng = np.random.default_rng(15)
    B, Hk, npm = w["B"], w["Hk"], w["np_max"]
    arrs = {k: np.zeros((B, Hk, npm), np.int32) for k in ("phys", "valid", "slot", "page_start")}
    arrs["phys"][:] = -1
    n_pages = w["n_pages"].copy()
    n_pages[1] = 0
    for b in range(B):
        n = n_pages[b]
        for h in range(Hk):
            perm = rng.permutation(n) if h % 2 else np.arange(n)
            for k in arrs:
                arrs[k][b, h, :n] = w[k][b, perm]
    q = _queries(15, B, 70, 8, 1.0)
    sl = _slopes(8)
    o, l = _run_alibi(w, q, arrs["phys"], arrs["valid"], arrs["slot"], arrs["page_start"], n_pages, w["qpos"],
                      w["doc_pos"], sl)
    ro, rl = oracle.alibi_prefill_batch(q, w["k_pool"], w["v_pool"], arrs["phys"], arrs["valid"], arrs["slot"],
                                        arrs["page_start"], n_pages, w["qpos"], w["doc_pos"], sl)
    assert (o[1] == 0).all() and np.isneginf(l[1]).all()
    _check(o, l, ro, rl)


# ------------------------------------------------------------------ the whole prefill step

def _run_step(w, slopes=None):
    B, T, Hq = w["q"].shape[:3]
    cache, keep = _cache(w)
    words = _words(w["phys"], w["valid"], w["slot"])
    out = torch.full((B, T, Hq, 128), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((B, T, Hq), float("nan"), dtype=torch.float32, device=DEV)
    args = (cache, bf(w["q"]), i32(w["qpos0"]), u32_as_i32(words), i32(w["n_pages"]), i32(w["page_start"]),
            i32(w["doc_pos"]))
    if slopes is None:
        spkv.lazy_rope_prefill_step(*args, w["theta"], out, lse)
    else:
        spkv.lazy_alibi_prefill_attn(*args, torch.from_numpy(slopes).to(DEV), out, lse)
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert spkv.get_device_error(cache) == (0, 0)
    cache.close()
    return o, l


@pytest.mark.parametrize("seed,T,Hq,Hk,cached", [(31, 5, 8, 2, True), (32, 128, 8, 2, True), (33, 200, 16, 4, True),
                                                (34, 300, 8, 2, False), (35, 64, 4, 1, True)])
def test_prefill_step_vs_oracle(seed, T, Hq, Hk, cached):
    """The whole step: cached documents plus the rows' own keys, listed as a document at qpos0 and
    attended causally; several 128-row tiles, tiles that see only part of the rows' own pages, a
    prompt with no cached document at all."""
    w = gen.prefill_step(seed=seed, B=3, T=T, Hq=Hq, Hk=Hk, cached=cached)
    o, l = _run_step(w)
    _check_rope(w, w["q"], o, l, w["phys"], w["valid"], w["slot"], w["page_start"], w["n_pages"], w["qpos0"],
                w["doc_pos"], causal=True)


@pytest.mark.parametrize("seed,T,cached", [(41, 70, True), (42, 200, False)])
def test_alibi_prefill_step_vs_oracle(seed, T, cached):
    """The ALiBi prefill with the rows' own keys listed: causal by position."""
    w = gen.prefill_step(seed=seed, B=3, T=T, Hq=8, Hk=2, cached=cached)
    sl = _slopes(8)
    o, l = _run_step(w, slopes=sl)
    ro, rl = oracle.alibi_prefill_batch(w["q"], w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"],
                                        w["page_start"], w["n_pages"], w["qpos0"], w["doc_pos"], sl)
    _check(o, l, ro, rl)


def test_prefill_step_equals_cached_prefill_without_own_pages():
    """With only cached documents listed nothing is masked: the step equals lazy_rope_prefill_attn bit
    for bit."""
    w = gen.prefill_step(seed=43, B=2, T=40, Hq=8, Hk=2)
    n_cached = (w["n_pages"] - 1).astype(np.int32)
    w2 = dict(w, n_pages=n_cached)
    o1, l1 = _run_step(w2)
    o2, l2 = _run(w2, w["q"], w["phys"], w["valid"], w["slot"], n_cached, w["qpos0"], w["doc_pos"])
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
