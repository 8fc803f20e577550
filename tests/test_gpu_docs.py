"""GPU parity of the document-major lazy-RoPE decode (lazy_rope_decode_attn_docs).

Requests that share cached documents are served job by job: one document, one kv head, the query
rows of up to 16 / G requests holding it.  The result must be exactly lazy_rope_decode_attn's for
the request's concatenated page list, so each case is checked against the fp64 materialised oracle
on those lists (attention tolerance, LSE 1e-3) and against lazy_rope_decode_attn itself.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import sparse_paged_kv_score_gb300 as spkv
from helpers import DEV, attn_errors, bf, i32, u32_as_i32

pytestmark = pytest.mark.gpu

ATTN_MAX, ATTN_MEAN, LSE_TOL = 1e-2, 1e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_paged_kv_score_gb300 import build
    build.build()
    spkv.load()


def _lists(w, req_docs, doc_pages_len=None):
    """Each request's concatenated page list (phys, valid, slot) from its documents, for the oracle and
    for lazy_rope_decode_attn."""
    B, D = req_docs.shape
    first = w["doc_first"]
    rows = []
    for b in range(B):
        ph, va, sl = [], [], []
        for i in range(D):
            d = req_docs[b, i]
            if d < 0:
                continue
            ph += w["doc_phys"][first[d]:first[d + 1]].tolist()
            va += w["doc_valid"][first[d]:first[d + 1]].tolist()
            sl += [i] * int(first[d + 1] - first[d])
        rows.append((ph, va, sl))
    npm = max(1, max(len(r[0]) for r in rows))
    phys = np.full((B, npm), -1, np.int32)
    valid = np.ones((B, npm), np.int32)
    slot = np.zeros((B, npm), np.int32)
    n_pages = np.zeros(B, np.int32)
    for b, (ph, va, sl) in enumerate(rows):
        n = len(ph)
        phys[b, :n], valid[b, :n], slot[b, :n], n_pages[b] = ph, va, sl, n
    return phys, valid, slot, n_pages


def _run_both(w, req_docs, doc_pos, qpos, q, steps=1):
    """The document-major call (steps calls in a row, qpos advancing by one each) and, for the last,
    lazy_rope_decode_attn on the concatenated lists.  Returns host arrays and the lists."""
    B, Hq, Hk = q.shape[0], q.shape[1], w["Hk"]
    k_pool, v_pool = bf(w["k_pool"]), bf(w["v_pool"])
    ksum = torch.zeros(Hk, w["n_phys"], 4, 128, dtype=torch.float32, device=DEV)
    cache = spkv.paged_kv_create(k_pool, v_pool, ksum, i32(w["page_cnt"]), max_units=B * Hk)
    words = spkv.pack_page_words(w["doc_phys"], w["doc_valid"], np.zeros_like(w["doc_phys"]))
    plan = spkv.DocPlan(cache, Hq, req_docs, w["doc_first"])
    dq = bf(q)
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=DEV)
    for t in range(steps):
        qp = i32(qpos + t)
        spkv.lazy_rope_decode_attn_docs(cache, plan, dq, qp, u32_as_i32(words), i32(w["doc_first"]), i32(doc_pos),
                                        w["theta"], out, lse)
    phys, valid, slot, n_pages = _lists(w, req_docs)
    ok = phys >= 0
    mw = np.zeros(phys.shape, np.uint32)
    mw[ok] = spkv.pack_page_words(phys[ok], valid[ok], slot[ok])
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    qlast = qpos + steps - 1
    spkv.lazy_rope_decode_attn(cache, dq, i32(qlast), u32_as_i32(mw), i32(n_pages), i32(doc_pos), w["theta"], out2,
                               lse2)
    torch.cuda.synchronize()
    err = spkv.get_device_error(cache)
    n_jobs = plan.n_jobs
    plan.close()
    cache.close()
    return out.cpu().numpy(), lse.cpu().numpy(), out2.cpu().numpy(), lse2.cpu().numpy(), \
        (phys, valid, slot, n_pages, qlast), err, n_jobs


def _check(w, q, doc_pos, res, units=None):
    o, l, o2, l2, (phys, valid, slot, n_pages, qlast), err, _ = res
    assert err == (0, 0)
    ro, rl = oracle.lazy_attn_batch(q, w["k_pool"], w["v_pool"], phys, valid, slot, n_pages, qlast, doc_pos,
                                    w["theta"], materialise=True, units=units)
    if units is not None:
        G, Hk, Hq = q.shape[1] // w["Hk"], w["Hk"], q.shape[1]
        rows = np.concatenate([np.arange((u % Hk) * G, (u % Hk + 1) * G) + (u // Hk) * Hq for u in units])
        sel = lambda a: a.reshape(-1, *a.shape[2:])[rows]   # noqa: E731
    else:
        sel = lambda a: a                                     # noqa: E731
    mx, mean = attn_errors(sel(o), sel(ro))
    assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (mx, mean)
    fin = np.isfinite(sel(rl))
    assert np.array_equal(np.isfinite(sel(l)), fin)
    assert np.abs(sel(l)[fin] - sel(rl)[fin]).max() <= LSE_TOL
    # the per-request form on the same lists agrees (two fp32 paths, same bf16 hi/lo splits)
    assert np.abs(o - o2).max() <= 1e-4 and np.abs(l[np.isfinite(l)] - l2[np.isfinite(l2)]).max() <= 1e-4


@pytest.mark.parametrize("seed,Hq,Hk", [(1, 8, 2), (2, 8, 8), (3, 32, 2), (4, 16, 8)])
def test_docs_vs_oracle(seed, Hq, Hk):
    """Zipf-drawn documents shared by many requests; groups of 4, 1, 16 and 2 query heads (16, 16, 1
    and 8 requests per job)."""
    w = gen.lazy_rag(seed=seed, B=12, Hq=Hq, Hk=Hk, n_docs=9, docs_per_req=4, min_len=70, max_len=900)
    res = _run_both(w, w["picks"], w["doc_pos"], w["qpos"], w["q"])
    _check(w, w["q"], w["doc_pos"], res)
    # shared documents: fewer jobs than (request, kv head, slot)s once a job holds several requests
    opj = max(1, 16 // (Hq // Hk))
    assert res[-1] <= w["B"] * w["Hk"] * 4 and (opj == 1 or res[-1] < w["B"] * w["Hk"] * 4)


def test_docs_empty_slots_duplicates_and_empty_documents():
    """Slots without a document, a request without any, the same document twice in one request (two
    offsets), and a document with no pages."""
    w = gen.lazy_rag(seed=5, B=5, Hq=8, Hk=2, n_docs=6, docs_per_req=4, min_len=64, max_len=500)
    first = w["doc_first"].copy()
    # document 6: no pages (appended at the end of the layout)
    w["doc_first"] = np.concatenate([first, [first[-1]]]).astype(np.int32)
    req = np.array([[0, -1, 2, 0], [-1, -1, -1, -1], [6, 1, 6, 3], [5, 5, -1, 4], [2, 3, 1, 0]], np.int32)
    lens = np.diff(w["doc_first"]) * 64
    doc_pos = np.zeros((5, 4), np.int32)
    qpos = np.zeros(5, np.int32)
    for b in range(5):
        pos = 0
        for i in range(4):
            doc_pos[b, i] = pos
            if req[b, i] >= 0:
                pos += int(lens[req[b, i]]) - 17 * i       # arbitrary, not page aligned
        qpos[b] = pos + 3
    q = gen.rows_bf16(5, 77, 5 * 8).reshape(5, 8, 128)
    res = _run_both(w, req, doc_pos, qpos, q)
    o, l = res[0], res[1]
    assert (o[1] == 0).all() and np.isneginf(l[1]).all()
    _check(w, q, doc_pos, res)


def test_docs_calls_in_a_row():
    """Three decode steps in a row (the query position advancing): the job counter and partials are
    reused; the last step's result is checked."""
    w = gen.lazy_rag(seed=7, B=8, Hq=8, Hk=2, n_docs=7, docs_per_req=3, min_len=100, max_len=700)
    res = _run_both(w, w["picks"], w["doc_pos"], w["qpos"], w["q"], steps=3)
    _check(w, w["q"], w["doc_pos"], res)


def test_docs_bad_page_word_flags_without_fault():
    w = gen.lazy_rag(seed=8, B=3, Hq=4, Hk=1, n_docs=4, docs_per_req=2, min_len=64, max_len=300)
    k_pool, v_pool = bf(w["k_pool"]), bf(w["v_pool"])
    ksum = torch.zeros(1, w["n_phys"], 4, 128, dtype=torch.float32, device=DEV)
    cache = spkv.paged_kv_create(k_pool, v_pool, ksum, i32(w["page_cnt"]))
    words = spkv.pack_page_words(w["doc_phys"], w["doc_valid"], np.zeros_like(w["doc_phys"]))
    words[1] = (words[1] & ~np.uint32(0x3FFFF)) | np.uint32((1 << 18) - 1)    # physical page out of range
    plan = spkv.DocPlan(cache, 4, w["picks"], w["doc_first"])
    out = torch.empty(3, 4, 128, dtype=torch.float32, device=DEV)
    lse = torch.empty(3, 4, dtype=torch.float32, device=DEV)
    spkv.lazy_rope_decode_attn_docs(cache, plan, bf(w["q"]), i32(w["qpos"]), u32_as_i32(words), i32(w["doc_first"]),
                                    i32(w["doc_pos"]), w["theta"], out, lse)
    st, bits = spkv.get_device_error(cache)
    assert bits == spkv.DEVERR["PHYS"] and torch.isfinite(out).all()
    plan.close()
    cache.close()


def test_docs_plan_rejects_bad_document_ids():
    w = gen.lazy_rag(seed=9, B=2, Hq=4, Hk=1, n_docs=3, docs_per_req=2, min_len=64, max_len=200)
    k_pool = bf(w["k_pool"])
    cache = spkv.paged_kv_create(k_pool, k_pool, None, None)
    with pytest.raises(spkv.SpkvError):
        spkv.DocPlan(cache, 4, np.array([[0, 3], [1, 2]], np.int32), w["doc_first"])     # document 3 of 3
    cache.close()
