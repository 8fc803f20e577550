"""Block-sparse decode attention over a paged, head-major KV cache, for NVIDIA GB300 (sm_103a).

A thin Python binding over the C ABI of ``libspkv.so`` (``include/spkv.h``).  Each function
has the name of the C entry point it calls and only marshals arguments: it checks dtypes,
devices and shapes of the torch tensors, then passes raw pointers, sizes and the current CUDA
stream.  Every step of the decode path runs in the library's own CUDA kernels; nothing here
computes.  Outputs are caller-allocated tensors, filled in place.

    cache = paged_kv_create(k_pool, v_pool, ksum, page_cnt)
    score_blocks(cache, q, page_table, seq_len, scores)
    select_topk(cache, scores, evict, alive, seq_len, k_q, k_e, sel, n_sel)
    resident_setdiff(cache, resident, sel, n_sel, missing, n_missing, slot)
    lru_bucket_update(cache, resident, ts, slot, n_sel, missing, n_missing, t, 1, victims, hist)
    sparse_decode_attn(cache, q, page_table, sel, n_sel, seq_len, out, lse)
    lazy_rope_decode_attn(cache, q, qpos, meta, n_pages, doc_pos, theta, out, lse)

With the full pool offloaded to pinned host memory and a slot pool on the device:

    slots = paged_kv_create(k_slots, v_slots, None, None)
    retrieve_pages(slots, k_host, v_host, page_table, missing, n_missing, victims, slot, n_sel, n_slots)
    sparse_decode_attn_slots(slots, q, sel, slot, n_sel, n_slots, seq_len, out, lse)
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from ._abi import DEVERR, SpkvDesc, SpkvError, SpkvPageDir, check, load

__all__ = ["PagedKVCache", "paged_kv_create", "paged_kv_append", "score_blocks", "decode_append_score",
           "select_topk",
           "sparse_decode_attn", "lazy_rope_decode_attn", "resident_setdiff", "lru_bucket_update",
           "select_resident_update", "retrieve_pages", "sparse_decode_attn_slots", "lazy_rope_prefill_attn",
           "lazy_rope_prefill_step",
           "attn_column_scores", "attn_column_scores_lse", "lazy_alibi_prefill_attn",
           "sparse_decode_attn_noalloc", "pack_page_words", "get_device_error", "SpkvError", "DEVERR",
           "PageMap", "score_blocks_dir", "sparse_decode_attn_dir", "retrieve_pages_dir", "DocPlan",
           "lazy_rope_decode_attn_docs",
           "load"]

HEAD_DIM, PAGE, SUBBLOCK = 128, 64, 16


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _t(x: torch.Tensor, dtype, name: str, shape=None) -> int:
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if x.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {x.dtype}")
    if not x.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None and tuple(x.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(x.shape)}")
    return x.data_ptr()


def _host(x: torch.Tensor, dtype, name: str, shape=None) -> int:
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if x.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {x.dtype}")
    if x.is_cuda or not x.is_pinned():
        raise ValueError(f"{name}: must be a pinned host tensor")
    if not x.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None and tuple(x.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(x.shape)}")
    return x.data_ptr()


class PagedKVCache:
    """Owns one library handle (``spkv_cache_t``) for a caller-owned pool.

    ``ksum`` is fp32, or bf16 for summaries rounded once to bf16 (half the bytes that
    ``score_blocks`` reads).  ``ksum`` and ``page_cnt`` may both be None: a handle without summaries, for a pool of
    resident slots that is only attended (``retrieve_pages``, ``sparse_decode_attn_slots``)."""

    def __init__(self, k_pool, v_pool, ksum, page_cnt, max_units: int = 0, stream=None):
        Hk, n_phys = k_pool.shape[0], k_pool.shape[1]
        shp = (Hk, n_phys, PAGE, HEAD_DIM)
        if (ksum is None) != (page_cnt is None):
            raise ValueError("ksum and page_cnt are given together or not at all")
        ksum_bf16 = ksum is not None and ksum.dtype == torch.bfloat16   # bf16 summaries: half the scoring bytes
        self.desc = SpkvDesc(Hk, HEAD_DIM, PAGE, SUBBLOCK, n_phys,
                             _t(k_pool, torch.bfloat16, "k_pool", shp),
                             _t(v_pool, torch.bfloat16, "v_pool", shp),
                             None if ksum is None else _t(ksum, torch.bfloat16 if ksum_bf16 else torch.float32, "ksum",
                                                          (Hk, n_phys, 4, HEAD_DIM)),
                             None if page_cnt is None else _t(page_cnt, torch.int32, "page_cnt", (n_phys,)),
                             int(max_units), int(ksum_bf16))
        self.n_kv_heads, self.n_phys = Hk, n_phys
        self.tensors = (k_pool, v_pool, ksum, page_cnt)   # keep the buffers alive
        h = ctypes.c_void_p()
        check("paged_kv_create", load().paged_kv_create(ctypes.byref(self.desc), _stream(stream),
                                                        ctypes.byref(h)))
        self.handle = h

    @property
    def sm_count(self) -> int:
        return load().spkv_sm_count(self.handle)

    def set_wait_limit(self, ns: int) -> None:
        """Limit (nanoseconds) of the attention kernels' bounded hand-off waits; 1 s by default."""
        check("spkv_set_wait_limit", load().spkv_set_wait_limit(self.handle, int(ns)))

    def close(self):
        if self.handle:
            torch.cuda.synchronize()
            check("paged_kv_destroy", load().paged_kv_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            if self.handle:
                load().paged_kv_destroy(self.handle)
                self.handle = None
        except Exception:
            pass


def paged_kv_create(k_pool, v_pool, ksum, page_cnt, max_units: int = 0, stream=None) -> PagedKVCache:
    return PagedKVCache(k_pool, v_pool, ksum, page_cnt, max_units, stream)


def paged_kv_append(cache: PagedKVCache, phys_page, tok_in_page, k_new, v_new, stream=None):
    n = phys_page.shape[0]
    shp = (n, cache.n_kv_heads, HEAD_DIM)
    check("paged_kv_append", load().paged_kv_append(
        cache.handle, _t(phys_page, torch.int32, "phys_page", (n,)),
        _t(tok_in_page, torch.int32, "tok_in_page", (n,)), _t(k_new, torch.bfloat16, "k_new", shp),
        _t(v_new, torch.bfloat16, "v_new", shp), n, _stream(stream)))


def score_blocks(cache: PagedKVCache, q, page_table, seq_len, scores, stream=None):
    B, Hq = q.shape[0], q.shape[1]
    np_max = page_table.shape[1]
    check("score_blocks", load().score_blocks(
        cache.handle, _t(q, torch.bfloat16, "q", (B, Hq, HEAD_DIM)), B, Hq,
        _t(page_table, torch.int32, "page_table", (B, np_max)), np_max,
        _t(seq_len, torch.int32, "seq_len", (B,)),
        _t(scores, torch.float32, "scores", (B, cache.n_kv_heads, np_max)), _stream(stream)))


def decode_append_score(cache: PagedKVCache, k_new, v_new, q, page_table, seq_len, scores, stream=None):
    """paged_kv_append of each request's new row at position seq_len[b] - 1 (its local page) and
    score_blocks, in one launch.  k_new, v_new: bf16 [B][Hk][128]."""
    B, Hq = q.shape[0], q.shape[1]
    np_max = page_table.shape[1]
    shp = (B, cache.n_kv_heads, HEAD_DIM)
    check("decode_append_score", load().decode_append_score(
        cache.handle, _t(k_new, torch.bfloat16, "k_new", shp), _t(v_new, torch.bfloat16, "v_new", shp),
        _t(q, torch.bfloat16, "q", (B, Hq, HEAD_DIM)), B, Hq,
        _t(page_table, torch.int32, "page_table", (B, np_max)), np_max,
        _t(seq_len, torch.int32, "seq_len", (B,)),
        _t(scores, torch.float32, "scores", (B, cache.n_kv_heads, np_max)), _stream(stream)))


def select_topk(cache: PagedKVCache, q_scores, evict_scores, alive, seq_len, k_q: int, k_e: int, sel,
                n_sel, stream=None):
    B, Hk, np_max = q_scores.shape
    stride = k_q + k_e + 1
    check("select_topk", load().select_topk(
        cache.handle, _t(q_scores, torch.float32, "q_scores", (B, Hk, np_max)),
        _t(evict_scores, torch.float32, "evict_scores", (B, Hk, np_max)),
        _t(alive, torch.int32, "alive", (B, Hk, (np_max + 31) // 32)), B, np_max,
        _t(seq_len, torch.int32, "seq_len", (B,)), int(k_q), int(k_e),
        _t(sel, torch.int32, "sel", (B, Hk, stride)), _t(n_sel, torch.int32, "n_sel", (B, Hk)),
        _stream(stream)))


def sparse_decode_attn(cache: PagedKVCache, q, page_table, sel, n_sel, seq_len, out, lse, stream=None):
    B, Hq = q.shape[0], q.shape[1]
    np_max = page_table.shape[1]
    stride = sel.shape[2]
    check("sparse_decode_attn", load().sparse_decode_attn(
        cache.handle, _t(q, torch.bfloat16, "q", (B, Hq, HEAD_DIM)), B, Hq,
        _t(page_table, torch.int32, "page_table", (B, np_max)), np_max,
        _t(sel, torch.int32, "sel", (B, cache.n_kv_heads, stride)),
        _t(n_sel, torch.int32, "n_sel", (B, cache.n_kv_heads)), stride,
        _t(seq_len, torch.int32, "seq_len", (B,)), _t(out, torch.float32, "out", (B, Hq, HEAD_DIM)),
        _t(lse, torch.float32, "lse", (B, Hq)), _stream(stream)))


def sparse_decode_attn_slots(cache: PagedKVCache, q, sel, slot, n_sel, n_slots: int, seq_len, out, lse,
                             stream=None):
    """sparse_decode_attn reading page sel[b][h][i] from slot page b * n_slots + slot[b][h][i]
    of the handle's pools (the slot pool that ``retrieve_pages`` fills)."""
    B, Hq = q.shape[0], q.shape[1]
    stride = sel.shape[2]
    check("sparse_decode_attn_slots", load().sparse_decode_attn_slots(
        cache.handle, _t(q, torch.bfloat16, "q", (B, Hq, HEAD_DIM)), B, Hq,
        _t(sel, torch.int32, "sel", (B, cache.n_kv_heads, stride)),
        _t(slot, torch.int32, "slot", (B, cache.n_kv_heads, stride)),
        _t(n_sel, torch.int32, "n_sel", (B, cache.n_kv_heads)), stride, int(n_slots),
        _t(seq_len, torch.int32, "seq_len", (B,)), _t(out, torch.float32, "out", (B, Hq, HEAD_DIM)),
        _t(lse, torch.float32, "lse", (B, Hq)), _stream(stream)))


def retrieve_pages(cache: PagedKVCache, k_host, v_host, page_table, missing, n_missing, victims, slot, n_sel,
                   n_slots: int, stream=None):
    """Copies each unit's missing pages from the pinned host pool (k_host, v_host:
    bf16 [Hk][n_host_pages][64][128]) into its victim slots of the handle's slot pool, and
    fills the -1 entries of ``slot`` (in place) with those victims."""
    Hk = cache.n_kv_heads
    n_host = k_host.shape[1]
    hshp = (Hk, n_host, PAGE, HEAD_DIM)
    B, np_max = page_table.shape
    stride = slot.shape[-1]
    for name, x, want in (("missing", missing, B * Hk * stride), ("victims", victims, B * Hk * stride),
                          ("slot", slot, B * Hk * stride), ("n_missing", n_missing, B * Hk),
                          ("n_sel", n_sel, B * Hk)):
        if x.numel() != want:
            raise ValueError(f"{name}: expected {want} elements")
    check("retrieve_pages", load().retrieve_pages(
        cache.handle, _host(k_host, torch.bfloat16, "k_host", hshp),
        _host(v_host, torch.bfloat16, "v_host", hshp), n_host,
        _t(page_table, torch.int32, "page_table", (B, np_max)), np_max, B,
        _t(missing, torch.int32, "missing"), _t(n_missing, torch.int32, "n_missing"),
        _t(victims, torch.int32, "victims"), _t(slot, torch.int32, "slot"),
        _t(n_sel, torch.int32, "n_sel"), stride, int(n_slots), _stream(stream)))


def sparse_decode_attn_noalloc(k_pool, v_pool, q, page_table, sel, n_sel, seq_len, out, lse, dev_err,
                               stream=None):
    """sparse_decode_attn for callers that cannot allocate device memory.

    No handle and no allocation: the pool is passed directly and the split-K scratch is a
    fixed device array inside the library (SPKV_NOALLOC_SCRATCH_BYTES per GPU, held until the
    process exits).  At most 512 (request, kv head) units per call.  Calls on one device share
    that scratch, so they must not overlap on the GPU.  ``dev_err`` (required) is an int32
    device tensor of one element that receives the device error bits.  The call runs on the
    device that holds ``k_pool`` (every tensor must be on it), on that device's current stream
    unless ``stream`` is given.
    """
    Hk, n_phys = k_pool.shape[0], k_pool.shape[1]
    shp = (Hk, n_phys, PAGE, HEAD_DIM)
    B, Hq = q.shape[0], q.shape[1]
    np_max = page_table.shape[1]
    stride = sel.shape[2]
    if dev_err is None:
        raise ValueError("dev_err: an int32 device tensor of one element is required")
    tensors = (k_pool, v_pool, q, page_table, sel, n_sel, seq_len, out, lse, dev_err)
    if not all(isinstance(x, torch.Tensor) and x.device == k_pool.device for x in tensors):
        raise ValueError("sparse_decode_attn_noalloc: every tensor must be on the device of k_pool")
    with torch.cuda.device(k_pool.device):
        check("sparse_decode_attn_noalloc", load().sparse_decode_attn_noalloc(
            _t(k_pool, torch.bfloat16, "k_pool", shp), _t(v_pool, torch.bfloat16, "v_pool", shp), Hk, n_phys,
            _t(q, torch.bfloat16, "q", (B, Hq, HEAD_DIM)), B, Hq,
            _t(page_table, torch.int32, "page_table", (B, np_max)), np_max,
            _t(sel, torch.int32, "sel", (B, Hk, stride)), _t(n_sel, torch.int32, "n_sel", (B, Hk)), stride,
            _t(seq_len, torch.int32, "seq_len", (B,)), _t(out, torch.float32, "out", (B, Hq, HEAD_DIM)),
            _t(lse, torch.float32, "lse", (B, Hq)), _t(dev_err, torch.int32, "dev_err", (1,)),
            _stream(stream)))


def lazy_rope_decode_attn(cache: PagedKVCache, q, qpos, meta, n_pages, doc_pos, theta: float, out, lse,
                          stream=None):
    """meta: int32 tensor holding the uint32 page words, [B][meta_heads][np_max] or [B][np_max]."""
    B, Hq = q.shape[0], q.shape[1]
    if meta.dim() == 2:
        meta = meta.unsqueeze(1)
    meta_heads, np_max = meta.shape[1], meta.shape[2]
    max_docs = doc_pos.shape[1]
    check("lazy_rope_decode_attn", load().lazy_rope_decode_attn(
        cache.handle, _t(q, torch.bfloat16, "q", (B, Hq, HEAD_DIM)), B, Hq,
        _t(qpos, torch.int32, "qpos", (B,)), _t(meta, torch.int32, "meta", (B, meta_heads, np_max)),
        meta_heads, _t(n_pages, torch.int32, "n_pages", (B,)), np_max,
        _t(doc_pos, torch.int32, "doc_pos", (B, max_docs)), max_docs, float(theta),
        _t(out, torch.float32, "out", (B, Hq, HEAD_DIM)), _t(lse, torch.float32, "lse", (B, Hq)),
        _stream(stream)))


class DocPlan:
    """Document-major schedule of lazy-RoPE decode over shared cached documents (built on the host
    from req_docs: host int32 [B][max_docs], -1 for an empty slot; doc_first: host int32
    [n_docs + 1]).  Reused by every lazy_rope_decode_attn_docs call of that batch composition."""

    def __init__(self, cache: PagedKVCache, Hq: int, req_docs, doc_first):
        req_docs = np.ascontiguousarray(req_docs, np.int32)
        doc_first = np.ascontiguousarray(doc_first, np.int32)
        B, max_docs = req_docs.shape
        h = ctypes.c_void_p()
        check("lazy_docs_plan_create", load().lazy_docs_plan_create(
            cache.handle, B, int(Hq), req_docs.ctypes.data, max_docs, doc_first.size - 1, doc_first.ctypes.data,
            ctypes.byref(h)))
        self.handle, self.B, self.Hq, self.max_docs = h, B, int(Hq), max_docs

    @property
    def n_jobs(self) -> int:
        return load().lazy_docs_plan_jobs(self.handle)

    def close(self):
        if self.handle:
            torch.cuda.synchronize()
            check("lazy_docs_plan_destroy", load().lazy_docs_plan_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            if self.handle:
                load().lazy_docs_plan_destroy(self.handle)
                self.handle = None
        except Exception:
            pass


def lazy_rope_decode_attn_docs(cache: PagedKVCache, plan: DocPlan, q, qpos, doc_pages, doc_first, doc_pos,
                               theta: float, out, lse, stream=None):
    """lazy_rope_decode_attn over shared documents, grouped by document.  doc_pages: int32 tensor of the
    uint32 page words of every document; doc_first: int32 [n_docs + 1]; doc_pos: int32 [B][max_docs]."""
    B, Hq = plan.B, plan.Hq
    check("lazy_rope_decode_attn_docs", load().lazy_rope_decode_attn_docs(
        cache.handle, plan.handle, _t(q, torch.bfloat16, "q", (B, Hq, HEAD_DIM)), _t(qpos, torch.int32, "qpos", (B,)),
        _t(doc_pages, torch.int32, "doc_pages"), _t(doc_first, torch.int32, "doc_first"),
        _t(doc_pos, torch.int32, "doc_pos", (B, plan.max_docs)), float(theta),
        _t(out, torch.float32, "out", (B, Hq, HEAD_DIM)), _t(lse, torch.float32, "lse", (B, Hq)), _stream(stream)))


def lazy_rope_prefill_attn(cache: PagedKVCache, q, qpos0, meta, n_pages, doc_pos, theta: float, out, lse,
                           stream=None):
    """LazyAttention prefill: q bf16 [B][T][Hq][128] rows at positions qpos0[b] + t over the cached
    document pages; meta: int32 tensor of page words, [B][meta_heads][np_max] or [B][np_max]."""
    B, T, Hq = q.shape[0], q.shape[1], q.shape[2]
    if meta.dim() == 2:
        meta = meta.unsqueeze(1)
    meta_heads, np_max = meta.shape[1], meta.shape[2]
    max_docs = doc_pos.shape[1]
    check("lazy_rope_prefill_attn", load().lazy_rope_prefill_attn(
        cache.handle, _t(q, torch.bfloat16, "q", (B, T, Hq, HEAD_DIM)), B, T, Hq,
        _t(qpos0, torch.int32, "qpos0", (B,)), _t(meta, torch.int32, "meta", (B, meta_heads, np_max)),
        meta_heads, _t(n_pages, torch.int32, "n_pages", (B,)), np_max,
        _t(doc_pos, torch.int32, "doc_pos", (B, max_docs)), max_docs, float(theta),
        _t(out, torch.float32, "out", (B, T, Hq, HEAD_DIM)), _t(lse, torch.float32, "lse", (B, T, Hq)),
        _stream(stream)))


def lazy_rope_prefill_step(cache: PagedKVCache, q, qpos0, meta, n_pages, page_start, doc_pos, theta: float, out,
                           lse, stream=None):
    """The whole RoPE prefill step: lazy_rope_prefill_attn over every listed key at a position
    doc_pos[slot] + page_start + row <= the query row's position (the new rows' own pages listed as a
    document placed at qpos0 give their causal attention); page_start int32 with the shape of meta."""
    B, T, Hq = q.shape[0], q.shape[1], q.shape[2]
    if meta.dim() == 2:
        meta = meta.unsqueeze(1)
    if page_start.dim() == 2:
        page_start = page_start.unsqueeze(1)
    meta_heads, np_max = meta.shape[1], meta.shape[2]
    max_docs = doc_pos.shape[1]
    check("lazy_rope_prefill_step", load().lazy_rope_prefill_step(
        cache.handle, _t(q, torch.bfloat16, "q", (B, T, Hq, HEAD_DIM)), B, T, Hq,
        _t(qpos0, torch.int32, "qpos0", (B,)), _t(meta, torch.int32, "meta", (B, meta_heads, np_max)),
        meta_heads, _t(n_pages, torch.int32, "n_pages", (B,)), np_max,
        _t(page_start, torch.int32, "page_start", (B, meta_heads, np_max)),
        _t(doc_pos, torch.int32, "doc_pos", (B, max_docs)), max_docs, float(theta),
        _t(out, torch.float32, "out", (B, T, Hq, HEAD_DIM)), _t(lse, torch.float32, "lse", (B, T, Hq)),
        _stream(stream)))


def lazy_alibi_prefill_attn(cache: PagedKVCache, q, qpos0, meta, n_pages, page_start, doc_pos, slopes, out, lse,
                            stream=None):
    """The prefill for ALiBi models: keys unrotated, bias -slopes[hq] * (n - m) with m = doc_pos[slot] +
    page_start + row; page_start int32 with the shape of meta, slopes fp32 [Hq]."""
    B, T, Hq = q.shape[0], q.shape[1], q.shape[2]
    if meta.dim() == 2:
        meta = meta.unsqueeze(1)
    if page_start.dim() == 2:
        page_start = page_start.unsqueeze(1)
    meta_heads, np_max = meta.shape[1], meta.shape[2]
    max_docs = doc_pos.shape[1]
    check("lazy_alibi_prefill_attn", load().lazy_alibi_prefill_attn(
        cache.handle, _t(q, torch.bfloat16, "q", (B, T, Hq, HEAD_DIM)), B, T, Hq,
        _t(qpos0, torch.int32, "qpos0", (B,)), _t(meta, torch.int32, "meta", (B, meta_heads, np_max)),
        meta_heads, _t(n_pages, torch.int32, "n_pages", (B,)), np_max,
        _t(page_start, torch.int32, "page_start", (B, meta_heads, np_max)),
        _t(doc_pos, torch.int32, "doc_pos", (B, max_docs)), max_docs, _t(slopes, torch.float32, "slopes", (Hq,)),
        _t(out, torch.float32, "out", (B, T, Hq, HEAD_DIM)), _t(lse, torch.float32, "lse", (B, T, Hq)),
        _stream(stream)))


def attn_column_scores(cache: PagedKVCache, q, page_table, seq_len, scores, stream=None):
    """PyramidKV-style key scores: q bf16 [B][alpha][Hq][128] (the prompt's last alpha rows);
    scores fp32 [B][Hq][64 np_max] (output)."""
    B, alpha, Hq = q.shape[0], q.shape[1], q.shape[2]
    np_max = page_table.shape[1]
    check("attn_column_scores", load().attn_column_scores(
        cache.handle, _t(q, torch.bfloat16, "q", (B, alpha, Hq, HEAD_DIM)), B, alpha, Hq,
        _t(page_table, torch.int32, "page_table", (B, np_max)), np_max,
        _t(seq_len, torch.int32, "seq_len", (B,)), _t(scores, torch.float32, "scores", (B, Hq, np_max * PAGE)),
        _stream(stream)))


def attn_column_scores_lse(cache: PagedKVCache, q, lse, page_table, seq_len, scores, stream=None):
    """attn_column_scores from the window rows' log-sum-exp lse fp32 [B][alpha][Hq] (natural log),
    as the attention over the same keys returns it; only the probability pass runs."""
    B, alpha, Hq = q.shape[0], q.shape[1], q.shape[2]
    np_max = page_table.shape[1]
    check("attn_column_scores_lse", load().attn_column_scores_lse(
        cache.handle, _t(q, torch.bfloat16, "q", (B, alpha, Hq, HEAD_DIM)),
        _t(lse, torch.float32, "lse", (B, alpha, Hq)), B, alpha, Hq,
        _t(page_table, torch.int32, "page_table", (B, np_max)), np_max,
        _t(seq_len, torch.int32, "seq_len", (B,)), _t(scores, torch.float32, "scores", (B, Hq, np_max * PAGE)),
        _stream(stream)))


def resident_setdiff(cache: PagedKVCache, resident, sel, n_sel, missing, n_missing, slot, stream=None):
    n_units, n_slots = resident.shape
    stride = sel.shape[-1]
    for name, x, want in (("sel", sel, n_units * stride), ("n_sel", n_sel, n_units),
                          ("missing", missing, n_units * stride), ("n_missing", n_missing, n_units),
                          ("slot", slot, n_units * stride)):
        if x.numel() != want:
            raise ValueError(f"{name}: expected {want} elements")
    check("resident_setdiff", load().resident_setdiff(
        cache.handle, _t(resident, torch.int32, "resident"), n_slots,
        _t(sel, torch.int32, "sel"), _t(n_sel, torch.int32, "n_sel"), stride, n_units,
        _t(missing, torch.int32, "missing"), _t(n_missing, torch.int32, "n_missing"),
        _t(slot, torch.int32, "slot"), _stream(stream)))


def lru_bucket_update(cache: PagedKVCache, resident, ts, slot, n_sel, missing, n_missing, t_now: int,
                      bucket_width: int, victims, hist, stream=None):
    n_units, n_slots = resident.shape
    stride = slot.shape[-1]
    for name, x, want in (("ts", ts, n_units * n_slots), ("slot", slot, n_units * stride),
                          ("n_sel", n_sel, n_units), ("missing", missing, n_units * stride),
                          ("n_missing", n_missing, n_units), ("victims", victims, n_units * stride),
                          ("hist", hist, n_units * 64)):
        if x.numel() != want:
            raise ValueError(f"{name}: expected {want} elements")
    check("lru_bucket_update", load().lru_bucket_update(
        cache.handle, _t(resident, torch.int32, "resident"), _t(ts, torch.int32, "ts"), n_slots,
        _t(slot, torch.int32, "slot"), _t(n_sel, torch.int32, "n_sel"),
        _t(missing, torch.int32, "missing"), _t(n_missing, torch.int32, "n_missing"), stride, n_units,
        int(t_now), int(bucket_width), _t(victims, torch.int32, "victims"),
        _t(hist, torch.int32, "hist"), _stream(stream)))


def select_resident_update(cache: PagedKVCache, q_scores, evict_scores, alive, seq_len, k_q: int, k_e: int, sel,
                           n_sel, resident, ts, t_now: int, bucket_width: int, missing, n_missing, slot, victims,
                           hist, stream=None):
    """select_topk, resident_setdiff and lru_bucket_update in one call (identical results)."""
    B, Hk, np_max = q_scores.shape
    stride = k_q + k_e + 1
    U = B * Hk
    n_units, n_slots = resident.shape
    if n_units != U:
        raise ValueError(f"resident: expected {U} rows")
    for name, x, want in (("ts", ts, U * n_slots), ("missing", missing, U * stride), ("n_missing", n_missing, U),
                          ("slot", slot, U * stride), ("victims", victims, U * stride), ("hist", hist, U * 64)):
        if x.numel() != want:
            raise ValueError(f"{name}: expected {want} elements")
    check("select_resident_update", load().select_resident_update(
        cache.handle, _t(q_scores, torch.float32, "q_scores", (B, Hk, np_max)),
        _t(evict_scores, torch.float32, "evict_scores", (B, Hk, np_max)),
        _t(alive, torch.int32, "alive", (B, Hk, (np_max + 31) // 32)), B, np_max,
        _t(seq_len, torch.int32, "seq_len", (B,)), int(k_q), int(k_e),
        _t(sel, torch.int32, "sel", (B, Hk, stride)), _t(n_sel, torch.int32, "n_sel", (B, Hk)),
        _t(resident, torch.int32, "resident"), _t(ts, torch.int32, "ts"), n_slots, int(t_now),
        int(bucket_width), _t(missing, torch.int32, "missing"), _t(n_missing, torch.int32, "n_missing"),
        _t(slot, torch.int32, "slot"), _t(victims, torch.int32, "victims"), _t(hist, torch.int32, "hist"),
        _stream(stream)))


class PageMap:
    """A two-level page directory ([Spin] 2C) managed by the library: a GPU directory of segments of
    2^seg_shift page ids, host segments allocated on demand in pinned memory, and n_dev_segs device
    slots for hot segments.  ``map`` and ``promote`` change the host state; ``sync`` brings the device
    up to date (and waits for the stream).  Pass the PageMap to the *_dir calls."""

    def __init__(self, B: int, np_max: int, seg_shift: int = 8, n_dev_segs: int = 0):
        h = ctypes.c_void_p()
        check("spkv_pagemap_create", load().spkv_pagemap_create(int(B), int(np_max), int(seg_shift),
                                                                int(n_dev_segs), ctypes.byref(h)))
        self.handle, self.B, self.np_max, self.seg_shift = h, B, np_max, seg_shift

    def map(self, b: int, first_page: int, phys) -> None:
        """Logical pages first_page .. of request b get the ids in phys (host int32; -1 unmaps)."""
        phys = np.ascontiguousarray(phys, np.int32)
        check("spkv_pagemap_map", load().spkv_pagemap_map(self.handle, int(b), int(first_page), phys.size,
                                                          phys.ctypes.data))

    def promote(self, b: int, page: int) -> None:
        check("spkv_pagemap_promote", load().spkv_pagemap_promote(self.handle, int(b), int(page)))

    def sync(self, stream=None) -> None:
        check("spkv_pagemap_sync", load().spkv_pagemap_sync(self.handle, _stream(stream)))

    def view(self) -> SpkvPageDir:
        v = SpkvPageDir()
        check("spkv_pagemap_view", load().spkv_pagemap_view(self.handle, ctypes.byref(v)))
        return v

    def nbytes(self):
        """(device bytes, host bytes) of the directory's metadata."""
        d, h = ctypes.c_int64(), ctypes.c_int64()
        check("spkv_pagemap_bytes", load().spkv_pagemap_bytes(self.handle, ctypes.byref(d), ctypes.byref(h)))
        return int(d.value), int(h.value)

    def close(self):
        if self.handle:
            torch.cuda.synchronize()
            check("spkv_pagemap_destroy", load().spkv_pagemap_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            if self.handle:
                load().spkv_pagemap_destroy(self.handle)
                self.handle = None
        except Exception:
            pass


def score_blocks_dir(cache: PagedKVCache, q, pagemap: PageMap, seq_len, scores, stream=None):
    """score_blocks with the page table given by a PageMap."""
    B, Hq = q.shape[0], q.shape[1]
    v = pagemap.view()
    np_max = pagemap.np_max
    check("score_blocks_dir", load().score_blocks_dir(
        cache.handle, _t(q, torch.bfloat16, "q", (B, Hq, HEAD_DIM)), B, Hq, ctypes.byref(v), np_max,
        _t(seq_len, torch.int32, "seq_len", (B,)),
        _t(scores, torch.float32, "scores", (B, cache.n_kv_heads, np_max)), _stream(stream)))


def sparse_decode_attn_dir(cache: PagedKVCache, q, pagemap: PageMap, sel, n_sel, seq_len, out, lse, stream=None):
    """sparse_decode_attn with the page table given by a PageMap."""
    B, Hq = q.shape[0], q.shape[1]
    stride = sel.shape[2]
    v = pagemap.view()
    check("sparse_decode_attn_dir", load().sparse_decode_attn_dir(
        cache.handle, _t(q, torch.bfloat16, "q", (B, Hq, HEAD_DIM)), B, Hq, ctypes.byref(v), pagemap.np_max,
        _t(sel, torch.int32, "sel", (B, cache.n_kv_heads, stride)),
        _t(n_sel, torch.int32, "n_sel", (B, cache.n_kv_heads)), stride,
        _t(seq_len, torch.int32, "seq_len", (B,)), _t(out, torch.float32, "out", (B, Hq, HEAD_DIM)),
        _t(lse, torch.float32, "lse", (B, Hq)), _stream(stream)))


def retrieve_pages_dir(cache: PagedKVCache, k_host, v_host, pagemap: PageMap, missing, n_missing, victims, slot,
                       n_sel, n_slots: int, stream=None):
    """retrieve_pages with the host-page table given by a PageMap."""
    Hk = cache.n_kv_heads
    n_host = k_host.shape[1]
    hshp = (Hk, n_host, PAGE, HEAD_DIM)
    B = pagemap.B
    stride = slot.shape[-1]
    v = pagemap.view()
    check("retrieve_pages_dir", load().retrieve_pages_dir(
        cache.handle, _host(k_host, torch.bfloat16, "k_host", hshp),
        _host(v_host, torch.bfloat16, "v_host", hshp), n_host, ctypes.byref(v), pagemap.np_max, B,
        _t(missing, torch.int32, "missing"), _t(n_missing, torch.int32, "n_missing"),
        _t(victims, torch.int32, "victims"), _t(slot, torch.int32, "slot"),
        _t(n_sel, torch.int32, "n_sel"), stride, int(n_slots), _stream(stream)))


def pack_page_words(phys, valid, doc_slot) -> np.ndarray:
    """Host helper: packs page words (uint32) for lazy_rope_decode_attn via the C ABI."""
    phys = np.ascontiguousarray(phys, np.int32)
    valid = np.ascontiguousarray(valid, np.int32)
    doc_slot = np.ascontiguousarray(doc_slot, np.int32)
    if not (phys.shape == valid.shape == doc_slot.shape):
        raise ValueError("phys, valid and doc_slot must have the same shape")
    out = np.empty(phys.shape, np.uint32)
    check("spkv_pack_page_words", load().spkv_pack_page_words(
        phys.ctypes.data, valid.ctypes.data, doc_slot.ctypes.data, phys.size, out.ctypes.data))
    return out


def get_device_error(cache: PagedKVCache, stream=None):
    """Waits for the stream; returns (status, bits) of the device error word and clears it."""
    bits = ctypes.c_uint32(0)
    st = load().spkv_get_device_error(cache.handle, _stream(stream), ctypes.byref(bits))
    return st, int(bits.value)
