"""GPU parity of the LazyAttention prefill kernel (tcgen05) against the fp64 oracle.

The oracle materialises keys rotated to their absolute positions; the kernel rotates each query
row once per document and runs QK^T and PV on the tensor cores with bf16 operands and fp32
accumulation.  Besides the attention tolerance, each case checks the relative L2 error of the
whole output, so that small outputs (long, flat softmaxes) still test something.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import sparse_paged_kv_score_gb300 as spkv
from helpers import DEV, attn_errors, bf, i32, u32_as_i32

pytestmark = pytest.mark.gpu

ATTN_MAX, ATTN_MEAN, LSE_TOL, REL_L2 = 1e-2, 1e-3, 1e-2, 2e-2


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


def _check(o, l, ro, rl):
    mx, mean = attn_errors(o, ro)
    assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (mx, mean)
    rel = np.linalg.norm((o - ro).ravel()) / max(np.linalg.norm(ro.ravel()), 1e-30)
    assert rel <= REL_L2, rel
    assert np.array_equal(np.isinf(l), np.isinf(rl))
    fin = np.isfinite(rl)
    assert np.abs(l[fin] - rl[fin]).max() <= LSE_TOL
    return mx, mean, rel


@pytest.mark.parametrize("seed,Hq,Hk,T", [(1, 8, 2, 5), (2, 16, 4, 128), (3, 8, 8, 200), (4, 32, 2, 33),
                                          (5, 4, 1, 129)])
def test_prefill_vs_materialised_oracle(seed, Hq, Hk, T):
    """Tiles of 128 rows with ragged tails, group sizes 1..16, partial last pages of documents."""
    w = gen.lazy_rag(seed=seed, B=3, Hq=Hq, Hk=Hk, n_docs=12, docs_per_req=4, min_len=70, max_len=900)
    q = _queries(seed, w["B"], T, Hq, 1.0)
    o, l = _run(w, q, w["phys"], w["valid"], w["slot"], w["n_pages"], w["qpos"], w["doc_pos"])
    ro, rl = oracle.lazy_prefill_batch(q, w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"],
                                       w["n_pages"], w["qpos"], w["doc_pos"], w["theta"], materialise=True)
    _check(o, l, ro, rl)


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
    ro, rl = oracle.lazy_prefill_batch(q, w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"],
                                       w["n_pages"], w["qpos"], w["doc_pos"], w["theta"], items=items)
    # compare the sampled (b, t, kv head) rows only
    G = 8 // w["Hk"]
    sel_o, sel_r, sel_l, sel_rl = [], [], [], []
    for it in items:
        h, bt = it % w["Hk"], it // w["Hk"]
        t, b = bt % 130, bt // 130
        sel_o.append(o[b, t, h * G:(h + 1) * G])
        sel_r.append(ro[b, t, h * G:(h + 1) * G])
        sel_l.append(l[b, t, h * G:(h + 1) * G])
        sel_rl.append(rl[b, t, h * G:(h + 1) * G])
    _check(np.array(sel_o), np.array(sel_l), np.array(sel_r), np.array(sel_rl))


def test_prefill_row_maximum_growing_inside_a_page_group():
    """A row's maximum jumping by more than 2^8 inside a group of two pages: keys set to zero
    before, and keys scaled x3 in, the last 32 tokens of (A) a request's first page (the first
    group's second 32-key block) and (B) the fourth page of another request's first document
    (the second group's fourth block: O is rescaled there).  With keys three times the unit
    scale, the bf16 rounding of the rotated query moves their scores three times as much, so
    this case allows three times the attention and LSE tolerances."""
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
    ro, rl = oracle.lazy_prefill_batch(q, w["k_pool"], w["v_pool"], w["phys"], w["valid"], w["slot"],
                                       w["n_pages"], w["qpos"], w["doc_pos"], w["theta"], materialise=True)
    mx, mean = attn_errors(o, ro)
    assert mx <= 3 * ATTN_MAX and mean <= 3 * ATTN_MEAN, (mx, mean)
    rel = np.linalg.norm((o - ro).ravel()) / np.linalg.norm(ro.ravel())
    assert rel <= REL_L2, rel
    assert np.isfinite(l).all()
    assert np.abs(l - rl).max() <= 3 * LSE_TOL


def test_prefill_per_head_page_lists_and_empty_request():
    """Per-kv-head page lists in a different order per head, and a request without pages."""
    w = gen.lazy_rag(seed=6, B=3, Hq=8, Hk=2, n_docs=10, docs_per_req=3, min_len=64, max_len=700)
    rng = np.random.default_rng(6)
    B, Hk, npm = w["B"], w["Hk"], w["np_max"]
    phys = np.full((B, Hk, npm), -1, np.int32)
    valid = np.zeros((B, Hk, npm), np.int32)
    slot = np.zeros((B, Hk, npm), np.int32)
    n_pages = w["n_pages"].copy()
    n_pages[1] = 0
    for b in range(B):
        n = n_pages[b]
        for h in range(Hk):
            perm = rng.permutation(n) if h % 2 else np.arange(n)   # pages of a head in any order
            phys[b, h, :n] = w["phys"][b, perm]
            valid[b, h, :n] = w["valid"][b, perm]
            slot[b, h, :n] = w["slot"][b, perm]
    q = _queries(6, B, 70, 8, 1.0)
    o, l = _run(w, q, phys, valid, slot, n_pages, w["qpos"], w["doc_pos"])
    ro, rl = oracle.lazy_prefill_batch(q, w["k_pool"], w["v_pool"], phys, valid, slot, n_pages, w["qpos"],
                                       w["doc_pos"], w["theta"], materialise=True)
    assert (o[1] == 0).all() and np.isneginf(l[1]).all()
    _check(o, l, ro, rl)


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
