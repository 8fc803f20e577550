"""The decode step captured as CUDA graphs (how bench.py and a serving loop run it) gives bitwise
the results of the same calls launched one by one, step after step, including the residency
state the steps carry forward."""
import numpy as np
import pytest
import torch

import gen
import sparse_paged_kv_score_gb300 as spkv
from helpers import DEV, bf, i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_paged_kv_score_gb300 import build
    build.build()
    spkv.load()


class _Step:
    """One handle and its per-step state on the Llama-3-8B-layer shapes at batch 4."""

    def __init__(self, w):
        B, Hk, npm = w["B"], w["Hk"], w["np_max"]
        self.k_pool, self.v_pool = bf(w["k_pool"]), bf(w["v_pool"])
        self.ksum = torch.zeros(Hk, w["n_phys"], 4, 128, dtype=torch.float32, device=DEV)
        self.cnt = i32(gen.page_counts(w))
        U = B * Hk
        self.cache = spkv.paged_kv_create(self.k_pool, self.v_pool, self.ksum, self.cnt, max_units=U)
        self.pt, self.seq = i32(w["page_table"]), i32(w["seq_len"])
        self.k_q, self.k_e = w["k_q"], w["k_e"]
        stride = self.k_q + self.k_e + 1
        self.scores = torch.empty(B, Hk, npm, dtype=torch.float32, device=DEV)
        self.alive = torch.full((B, Hk, (npm + 31) // 32), -1, dtype=torch.int32, device=DEV)
        self.sel = torch.empty(B, Hk, stride, dtype=torch.int32, device=DEV)
        self.n_sel = torch.empty(B, Hk, dtype=torch.int32, device=DEV)
        self.resident = torch.full((U, 256), -1, dtype=torch.int32, device=DEV)
        self.ts = torch.full((U, 256), np.iinfo(np.int32).min, dtype=torch.int32, device=DEV)
        self.missing = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        self.n_missing = torch.empty(U, dtype=torch.int32, device=DEV)
        self.slot = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        self.victims = torch.empty(U, stride, dtype=torch.int32, device=DEV)
        self.hist = torch.empty(U, 64, dtype=torch.int32, device=DEV)
        self.out = torch.empty(B, w["Hq"], 128, dtype=torch.float32, device=DEV)
        self.lse = torch.empty(B, w["Hq"], dtype=torch.float32, device=DEV)

    def run(self, q, ev, kn, vn, t):
        spkv.decode_append_score(self.cache, kn, vn, q, self.pt, self.seq, self.scores)
        spkv.select_resident_update(self.cache, self.scores, ev, self.alive, self.seq, self.k_q, self.k_e, self.sel,
                                    self.n_sel, self.resident, self.ts, t, 1, self.missing, self.n_missing,
                                    self.slot, self.victims, self.hist)
        spkv.sparse_decode_attn(self.cache, q, self.pt, self.sel, self.n_sel, self.seq, self.out, self.lse)

    def state(self):
        return [x.clone() for x in (self.out, self.lse, self.sel, self.n_sel, self.alive, self.resident, self.ts,
                                    self.missing, self.victims, self.hist, self.ksum, self.k_pool, self.v_pool)]


def test_graph_replayed_steps_equal_eager_steps():
    w = gen.llama8b(seed=3, B=4)
    B, Hq, Hk = w["B"], w["Hq"], w["Hk"]
    n = 6
    qs = [bf(gen.rows_bf16(3, 100 + i, B * Hq).reshape(B, Hq, 128)) for i in range(n)]
    evs = [torch.from_numpy(gen.normal_f64(3, 200 + i, B * Hk * w["np_max"]).astype(np.float32)
                            .reshape(B, Hk, w["np_max"])).to(DEV) for i in range(n)]
    kn = [bf(gen.rows_bf16(3, 300 + i, B * Hk).reshape(B, Hk, 128)) for i in range(n)]
    vn = [bf(gen.rows_bf16(3, 400 + i, B * Hk).reshape(B, Hk, 128)) for i in range(n)]
    eager, graphed = _Step(w), _Step(w)
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graphs = []
    for i in range(n):                       # capture every step first (nothing runs while capturing)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            graphed.run(qs[i], evs[i], kn[i], vn[i], i)
        graphs.append(g)
    torch.cuda.synchronize()
    for i in range(n):
        eager.run(qs[i], evs[i], kn[i], vn[i], i)
        graphs[i].replay()
        torch.cuda.synchronize()
        for a, b in zip(eager.state(), graphed.state()):
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b), f"step {i}"
    assert spkv.get_device_error(eager.cache) == (0, 0)
    assert spkv.get_device_error(graphed.cache) == (0, 0)
    eager.cache.close()
    graphed.cache.close()


def test_bookkeeping_beside_attention_equals_fused_schedule():
    """The bench's default step runs the selection, then the set-difference and LRU update on a
    second stream while the attention streams its pages (it does not read their results), joining
    before the next step.  Over six steps, eagerly and replayed from CUDA graphs, every output and
    the residency state equal the fused schedule's bit for bit."""
    w = gen.llama8b(seed=4, B=4)
    B, Hq, Hk = w["B"], w["Hq"], w["Hk"]
    n = 6
    qs = [bf(gen.rows_bf16(4, 100 + i, B * Hq).reshape(B, Hq, 128)) for i in range(n)]
    evs = [torch.from_numpy(gen.normal_f64(4, 200 + i, B * Hk * w["np_max"]).astype(np.float32)
                            .reshape(B, Hk, w["np_max"])).to(DEV) for i in range(n)]
    kn = [bf(gen.rows_bf16(4, 300 + i, B * Hk).reshape(B, Hk, 128)) for i in range(n)]
    vn = [bf(gen.rows_bf16(4, 400 + i, B * Hk).reshape(B, Hk, 128)) for i in range(n)]
    side = torch.cuda.Stream()

    def overlap(st, i):
        spkv.decode_append_score(st.cache, kn[i], vn[i], qs[i], st.pt, st.seq, st.scores)
        spkv.select_topk(st.cache, st.scores, evs[i], st.alive, st.seq, st.k_q, st.k_e, st.sel, st.n_sel)
        main = torch.cuda.current_stream()
        side.wait_stream(main)
        with torch.cuda.stream(side):
            spkv.resident_setdiff(st.cache, st.resident, st.sel, st.n_sel, st.missing, st.n_missing, st.slot)
            spkv.lru_bucket_update(st.cache, st.resident, st.ts, st.slot, st.n_sel, st.missing, st.n_missing, i, 1,
                                   st.victims, st.hist)
        spkv.sparse_decode_attn(st.cache, qs[i], st.pt, st.sel, st.n_sel, st.seq, st.out, st.lse)
        main.wait_stream(side)

    fused, eager, graphed = _Step(w), _Step(w), _Step(w)
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graphs = []
    for i in range(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            overlap(graphed, i)
        graphs.append(g)
    torch.cuda.synchronize()
    for i in range(n):
        fused.run(qs[i], evs[i], kn[i], vn[i], i)
        overlap(eager, i)
        graphs[i].replay()
        torch.cuda.synchronize()
        ref = fused.state() + [fused.missing.clone(), fused.n_missing.clone(), fused.slot.clone()]
        for st in (eager, graphed):
            got = st.state() + [st.missing.clone(), st.n_missing.clone(), st.slot.clone()]
            for a, b in zip(ref, got):
                assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                                   b.view(torch.int16) if b.dtype == torch.bfloat16 else b), f"step {i}"
    for st in (fused, eager, graphed):
        assert spkv.get_device_error(st.cache) == (0, 0)
        st.cache.close()


def test_document_major_decode_and_column_scores_in_graphs():
    """The document-major lazy decode (whose plan carries a job counter from call to call) and both
    column-score forms (whose calls build a tensor map of the window rows on the host) captured as
    CUDA graphs and replayed several times give bitwise what the eager calls give."""
    from helpers import u32_as_i32
    w = gen.lazy_rag(seed=21, B=10, Hq=8, Hk=2, n_docs=8, docs_per_req=3, min_len=100, max_len=700)
    B, Hq, Hk = w["B"], w["Hq"], w["Hk"]
    k_pool, v_pool = bf(w["k_pool"]), bf(w["v_pool"])
    cache = spkv.paged_kv_create(k_pool, v_pool, None, None, max_units=B * Hk)
    plan = spkv.DocPlan(cache, Hq, w["picks"], w["doc_first"])
    words = u32_as_i32(spkv.pack_page_words(w["doc_phys"], w["doc_valid"], np.zeros_like(w["doc_phys"])))
    q, qpos, df, dp = bf(w["q"]), i32(w["qpos"]), i32(w["doc_first"]), i32(w["doc_pos"])
    out = torch.empty(B, Hq, 128, dtype=torch.float32, device=DEV)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=DEV)
    # column scores over request 0's first document's pages as a prompt (window 40 rows)
    sw = gen.sparse_workload(3, Hq, Hk, 64 * 7 + 9, 4, 4, seed=22)
    ck = bf(sw["k_pool"])
    ccache = spkv.paged_kv_create(ck, ck, None, None)
    alpha = 40
    cq = bf(gen.rows_bf16(22, 329, 3 * alpha * Hq).reshape(3, alpha, Hq, 128))
    cpt, cseq = i32(sw["page_table"]), i32(sw["seq_len"])
    clse = torch.from_numpy(np.random.default_rng(3).normal(6.0, 1.0, (3, alpha, Hq)).astype(np.float32)).to(DEV)
    s1 = torch.empty(3, Hq, sw["np_max"] * 64, dtype=torch.float32, device=DEV)
    s2 = torch.empty_like(s1)

    def calls():
        spkv.lazy_rope_decode_attn_docs(cache, plan, q, qpos, words, df, dp, w["theta"], out, lse)
        spkv.attn_column_scores(ccache, cq, cpt, cseq, s1)
        spkv.attn_column_scores_lse(ccache, cq, clse, cpt, cseq, s2)

    calls()
    torch.cuda.synchronize()
    eager = [x.clone() for x in (out, lse, s1, s2)]
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side):
        calls()
    torch.cuda.synchronize()
    for _ in range(3):
        for x in (out, lse, s1, s2):
            x.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(eager, (out, lse, s1, s2)):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert spkv.get_device_error(cache) == (0, 0) and spkv.get_device_error(ccache) == (0, 0)
    plan.close()
    cache.close()
    ccache.close()
