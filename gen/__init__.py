"""Seeded synthetic inputs for the sparse paged-KV decode path.

This module is shared by the fp64 oracle tests, the GPU parity tests and ``bench.py``.
It contains no scoring, selection or attention arithmetic: only random numbers
(SplitMix64 + Box-Muller, see ``spkv_gen.cpp``) and the *structure* of each workload
(page tables, sequence lengths, document layouts, Zipf document draws).

Workloads (sizes from the five decode configurations this library is measured on):

* ``tiny``        batch 1, 8 q / 2 kv heads, context 4096, k = 16 (k_q 8, k_e 8).
* ``llama8b``     batch 32, 32 q / 8 kv heads, context 32768, k = 64 (32/32); each key row
                  is scaled x20 with probability 0.01 (stand-in for massive activations).
* ``lazy_rag``    batch 64, 32 q / 8 kv heads; a pool of 256 documents of 1024..4096 tokens;
                  each request concatenates 8 documents drawn Zipf(s = 1.1).
* ``long262k``    batch 8, 40 q / 8 kv heads, context 262144, k = 128, 2048 resident slots.
* ``nosa_traj``   batch 16, 32 q / 8 kv heads, context 65536, k = 64 (k_e 48, k_q 16),
                  64 decode steps appending one token each.

Arrays holding bf16 values are ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HEAD_DIM = 128
PAGE = 64
SUBBLOCK = 16

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spkv_gen.cpp")
_SO = os.path.join(_HERE, "libspkvgen.so")
_lib = None

# Stream tags: one independent random stream per tensor kind.
TAG_K, TAG_V, TAG_Q, TAG_E, TAG_PERM = 1, 2, 3, 4, 5
TAG_DOC_LEN, TAG_DOC_PICK, TAG_DOC_PERM = 6, 7, 8
TAG_SELF_K, TAG_SELF_V, TAG_ROWS_Q = 9, 10, 11
TAG_STEP_E, TAG_STEP_Q, TAG_STEP_K, TAG_STEP_V = 1000, 2000, 3000, 4000


def build(force: bool = False) -> str:
    """Compiles ``libspkvgen.so`` with g++ if it is missing or older than its source."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp])
        os.replace(tmp, _SO)
    return _SO


def _l():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        u64, i64, i32, f64, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                                  ctypes.c_void_p)
        lib.gen_uniform_f64.argtypes = [u64, u64, i64, i64, vp, i32]
        lib.gen_normal_f32.argtypes = [u64, u64, i64, i64, f64, vp, i32]
        lib.gen_normal_f64.argtypes = [u64, u64, i64, i64, vp, i32]
        lib.gen_rows_bf16.argtypes = [u64, u64, i64, i64, i32, f64, f64, vp, i32]
        lib.gen_f32_to_bf16.argtypes = [vp, i64, vp]
        for f in (lib.gen_uniform_f64, lib.gen_normal_f32, lib.gen_normal_f64, lib.gen_rows_bf16,
                  lib.gen_f32_to_bf16):
            f.restype = None
        _lib = lib
    return _lib


def _nthreads() -> int:
    return int(os.environ.get("SPKV_GEN_THREADS", "0"))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# ----------------------------------------------------------------------------- primitives

def uniform(seed: int, tag: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, np.float64)
    _l().gen_uniform_f64(seed, tag, offset, n, _ptr(out), _nthreads())
    return out


def normal_f32(seed: int, tag: int, n: int, scale: float = 1.0, offset: int = 0) -> np.ndarray:
    out = np.empty(n, np.float32)
    _l().gen_normal_f32(seed, tag, offset, n, scale, _ptr(out), _nthreads())
    return out


def normal_f64(seed: int, tag: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, np.float64)
    _l().gen_normal_f64(seed, tag, offset, n, _ptr(out), _nthreads())
    return out


def rows_bf16(seed: int, tag: int, n_rows: int, row_len: int = HEAD_DIM, row_offset: int = 0,
              outlier_p: float = 0.0, outlier_scale: float = 20.0) -> np.ndarray:
    out = np.empty((n_rows, row_len), np.uint16)
    _l().gen_rows_bf16(seed, tag, row_offset, n_rows, row_len, outlier_p, outlier_scale, _ptr(out),
                       _nthreads())
    return out


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    _l().gen_f32_to_bf16(_ptr(x), x.size, _ptr(out))
    return out


def bf16_to_f32(x: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 (for inspecting inputs)."""
    return (x.astype(np.uint32) << 16).view(np.float32)


def permutation(seed: int, tag: int, n: int) -> np.ndarray:
    """A seeded permutation of 0..n-1 (stable argsort of n uniforms)."""
    return np.argsort(uniform(seed, tag, n), kind="stable").astype(np.int32)


# ----------------------------------------------------------------------------- workloads

def sparse_workload(B: int, Hq: int, Hk: int, L: int, k_q: int, k_e: int, seed: int = 0,
                    outlier_p: float = 0.0, extra_tokens: int = 0, name: str = "") -> dict:
    """A batch of B requests with context L tokens each, over a head-major paged pool.

    ``extra_tokens`` reserves page-table room (and physical pages) for later appends.
    Physical pages are a seeded permutation, so consecutive logical pages are scattered.
    The K rows carry the outlier scaling (if any); V rows and q are plain N(0,1).
    Eviction scores ``evict`` are fp32 N(0,1), one per (request, kv head, logical page).
    """
    np_max = (L + extra_tokens + PAGE - 1) // PAGE
    n_phys = B * np_max
    perm = permutation(seed, TAG_PERM, n_phys)
    page_table = perm.reshape(B, np_max).astype(np.int32)
    rows = Hk * n_phys * PAGE
    k_pool = rows_bf16(seed, TAG_K, rows, outlier_p=outlier_p).reshape(Hk, n_phys, PAGE, HEAD_DIM)
    v_pool = rows_bf16(seed, TAG_V, rows).reshape(Hk, n_phys, PAGE, HEAD_DIM)
    q = rows_bf16(seed, TAG_Q, B * Hq).reshape(B, Hq, HEAD_DIM)
    evict = normal_f32(seed, TAG_E, B * Hk * np_max).reshape(B, Hk, np_max)
    seq_len = np.full(B, L, np.int32)
    return dict(name=name, B=B, Hq=Hq, Hk=Hk, G=Hq // Hk, D=HEAD_DIM, T=PAGE, np_max=np_max,
                n_phys=n_phys, page_table=page_table, k_pool=k_pool, v_pool=v_pool, q=q,
                evict=evict, seq_len=seq_len, k_q=k_q, k_e=k_e, seed=seed)


def page_counts(w: dict) -> np.ndarray:
    """Valid tokens held by every physical page of a sparse workload (0 for unused pages)."""
    cnt = np.zeros(w["n_phys"], np.int32)
    for b in range(w["B"]):
        L = int(w["seq_len"][b])
        n = (L + PAGE - 1) // PAGE
        for p in range(n):
            cnt[w["page_table"][b, p]] = min(PAGE, L - PAGE * p)
    return cnt


def tiny(seed: int = 0) -> dict:
    return sparse_workload(1, 8, 2, 4096, 8, 8, seed, name="tiny sparse decode B1 Hq8/Hk2 L4096 k16")


def llama8b(seed: int = 0, B: int = 32) -> dict:
    return sparse_workload(B, 32, 8, 32768, 32, 32, seed, outlier_p=0.01,
                           name=f"Llama-3-8B-layer sparse decode B{B} Hq32/Hk8 L32768 k64")


def long262k(seed: int = 0, B: int = 8) -> dict:
    w = sparse_workload(B, 40, 8, 262144, 128, 0, seed,
                        name=f"262k sparse decode + residency B{B} Hq40/Hk8 k128")
    w["n_slots"] = 2048
    return w


def nosa_traj(seed: int = 0, B: int = 16, steps: int = 64) -> dict:
    w = sparse_workload(B, 32, 8, 65536, 16, 48, seed, extra_tokens=steps,
                        name=f"NOSA trajectory B{B} Hq32/Hk8 L65536 k64 (k_e48,k_q16) {steps} steps")
    w["steps"] = steps
    return w


def traj_step_inputs(w: dict, t: int, prev_evict=None) -> dict:
    """Inputs that step t of a decode trajectory consumes.

    The eviction scores follow a random walk (step std 0.1) starting from ``w['evict']``: pass the
    previous step's scores as ``prev_evict`` (None at t = 0 or to replay the walk from the start).
    The query is fresh N(0,1); one new K and V row per (request, kv head) is appended.
    """
    B, Hk, Hq, npm = w["B"], w["Hk"], w["Hq"], w["np_max"]
    seed = w["seed"]
    if prev_evict is None:
        e = w["evict"].astype(np.float64).copy()
        first = 0
    else:
        e = np.asarray(prev_evict, np.float64).copy()
        first = t
    for s in range(first, t + 1):
        e += normal_f64(seed, TAG_STEP_E + s, B * Hk * npm).reshape(B, Hk, npm) * 0.1
    return dict(
        evict=e,
        q=rows_bf16(seed, TAG_STEP_Q + t, B * Hq).reshape(B, Hq, HEAD_DIM),
        k_new=rows_bf16(seed, TAG_STEP_K + t, B * Hk).reshape(B, Hk, HEAD_DIM),
        v_new=rows_bf16(seed, TAG_STEP_V + t, B * Hk).reshape(B, Hk, HEAD_DIM),
    )


def walk_queries(w: dict, steps: int) -> list:
    """Query random walk: fp32 master q0 ~ N(0,1), plus N(0, 0.1^2) per step, rounded to bf16."""
    B, Hq = w["B"], w["Hq"]
    seed = w["seed"]
    master = normal_f32(seed, TAG_Q, B * Hq * HEAD_DIM).astype(np.float32)
    out = []
    for t in range(steps):
        if t > 0:
            master = master + normal_f32(seed, TAG_STEP_Q + t, master.size, 0.1)
        out.append(f32_to_bf16(master).reshape(B, Hq, HEAD_DIM))
    return out


def zipf_draws(seed: int, tag: int, n: int, n_ranks: int, s: float) -> np.ndarray:
    """n i.i.d. draws of rank-1 (0-based document ids) from Zipf(s) over ranks 1..n_ranks."""
    w = 1.0 / np.arange(1, n_ranks + 1, dtype=np.float64) ** s
    cdf = np.cumsum(w / w.sum())
    u = uniform(seed, tag, n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), n_ranks - 1).astype(np.int32)


def lazy_rag(seed: int = 0, B: int = 64, Hq: int = 32, Hk: int = 8, n_docs: int = 256,
             docs_per_req: int = 8, min_len: int = 1024, max_len: int = 4096,
             zipf_s: float = 1.1, theta: float = 500000.0) -> dict:
    """Position-agnostic document reuse: requests concatenate shared cached documents.

    Document d has ``doc_len[d]`` tokens drawn uniformly from [min_len, max_len]; its
    ceil(len/64) pages are scattered over the pool and its last page is partially filled.
    Request b places its 8 documents contiguously: document slot i starts at token
    ``doc_pos[b, i]`` (the sum of the earlier lengths, so offsets are not page aligned) and
    the query sits at ``qpos[b]`` = total length.  Stored keys are N(0,1) bf16 (they stand for
    keys that carry only their document-local rotation).
    """
    u = uniform(seed, TAG_DOC_LEN, n_docs)
    doc_len = (min_len + np.floor(u * (max_len - min_len + 1))).astype(np.int64)
    doc_len = np.minimum(doc_len, max_len)
    doc_pages = (doc_len + PAGE - 1) // PAGE
    n_phys = int(doc_pages.sum())
    perm = permutation(seed, TAG_DOC_PERM, n_phys)
    first = np.concatenate([[0], np.cumsum(doc_pages)[:-1]])
    doc_phys = [perm[first[d]:first[d] + doc_pages[d]].astype(np.int32) for d in range(n_docs)]
    picks = zipf_draws(seed, TAG_DOC_PICK, B * docs_per_req, n_docs, zipf_s).reshape(B, docs_per_req)
    n_pages = np.array([int(doc_pages[picks[b]].sum()) for b in range(B)], np.int32)
    np_max = int(n_pages.max())
    phys = np.full((B, np_max), -1, np.int32)
    valid = np.zeros((B, np_max), np.int32)
    slot = np.zeros((B, np_max), np.int32)
    page_start = np.zeros((B, np_max), np.int32)   # document-local position of each page's first token
    doc_pos = np.zeros((B, docs_per_req), np.int32)
    qpos = np.zeros(B, np.int32)
    for b in range(B):
        j, pos = 0, 0
        for i, d in enumerate(picks[b]):
            doc_pos[b, i] = pos
            L = int(doc_len[d])
            for p in range(int(doc_pages[d])):
                phys[b, j] = doc_phys[d][p]
                valid[b, j] = min(PAGE, L - PAGE * p)
                slot[b, j] = i
                page_start[b, j] = PAGE * p
                j += 1
            pos += L
        qpos[b] = pos
    rows = Hk * n_phys * PAGE
    k_pool = rows_bf16(seed, TAG_K, rows).reshape(Hk, n_phys, PAGE, HEAD_DIM)
    v_pool = rows_bf16(seed, TAG_V, rows).reshape(Hk, n_phys, PAGE, HEAD_DIM)
    q = rows_bf16(seed, TAG_Q, B * Hq).reshape(B, Hq, HEAD_DIM)
    cnt = np.zeros(n_phys, np.int32)
    for d in range(n_docs):
        for p in range(int(doc_pages[d])):
            cnt[doc_phys[d][p]] = min(PAGE, int(doc_len[d]) - PAGE * p)
    doc_first = np.concatenate([[0], np.cumsum(doc_pages)]).astype(np.int32)
    doc_phys = np.concatenate(doc_phys).astype(np.int32)
    doc_valid = np.concatenate([np.minimum(PAGE, int(doc_len[d]) - PAGE * np.arange(int(doc_pages[d])))
                                for d in range(n_docs)]).astype(np.int32)
    return dict(name=f"lazy-RoPE RAG decode B{B} Hq{Hq}/Hk{Hk} {n_docs} docs x{docs_per_req} Zipf({zipf_s})",
                doc_first=doc_first, doc_phys=doc_phys, doc_valid=doc_valid,
                B=B, Hq=Hq, Hk=Hk, G=Hq // Hk, D=HEAD_DIM, T=PAGE, n_phys=n_phys, np_max=np_max,
                k_pool=k_pool, v_pool=v_pool, q=q, phys=phys, valid=valid, slot=slot, page_start=page_start,
                n_pages=n_pages, doc_pos=doc_pos, qpos=qpos, theta=theta, picks=picks,
                doc_len=doc_len, page_cnt=cnt, max_docs=docs_per_req, seed=seed)


def prefill_step(seed: int = 0, B: int = 3, T: int = 128, Hq: int = 8, Hk: int = 2, n_docs: int = 12,
                 docs_per_req: int = 4, min_len: int = 70, max_len: int = 900, theta: float = 500000.0,
                 cached: bool = True) -> dict:
    """A prompt's prefill step: each request's cached documents (the ``lazy_rag`` layout, none when
    ``cached`` is False) followed by its T new rows' own K/V in ceil(T/64) fresh pages, listed last as
    one more document placed at the first new row's position ``qpos0`` (the cached length); its pages
    have document-local starts 0, 64, ...  ``q`` holds the new rows' queries [B][T][Hq][128].  The new
    keys stand for keys that carry the rotation of their position inside the prompt."""
    if cached:
        w = lazy_rag(seed, B, Hq, Hk, n_docs, docs_per_req, min_len, max_len, theta=theta)
    else:
        w = dict(name="", B=B, Hq=Hq, Hk=Hk, G=Hq // Hk, D=HEAD_DIM, T=PAGE, n_phys=0, np_max=0,
                 k_pool=np.zeros((Hk, 0, PAGE, HEAD_DIM), np.uint16), v_pool=np.zeros((Hk, 0, PAGE, HEAD_DIM), np.uint16),
                 phys=np.zeros((B, 0), np.int32), valid=np.zeros((B, 0), np.int32), slot=np.zeros((B, 0), np.int32),
                 page_start=np.zeros((B, 0), np.int32), n_pages=np.zeros(B, np.int32),
                 doc_pos=np.zeros((B, 0), np.int32), qpos=np.zeros(B, np.int32), theta=theta,
                 page_cnt=np.zeros(0, np.int32), max_docs=0, seed=seed)
    n_self = (T + PAGE - 1) // PAGE
    n_old = w["n_phys"]
    n_phys = n_old + B * n_self
    rows = Hk * B * n_self * PAGE
    k_new = rows_bf16(seed, TAG_SELF_K, rows).reshape(Hk, B * n_self, PAGE, HEAD_DIM)
    v_new = rows_bf16(seed, TAG_SELF_V, rows).reshape(Hk, B * n_self, PAGE, HEAD_DIM)
    k_pool = np.concatenate([w["k_pool"], k_new], axis=1)
    v_pool = np.concatenate([w["v_pool"], v_new], axis=1)
    np_max = int((w["n_pages"] + n_self).max())
    slot_self = w["max_docs"]
    arrs = {}
    for key, fill in (("phys", -1), ("valid", 0), ("slot", 0), ("page_start", 0)):
        a = np.full((B, np_max), fill, np.int32)
        a[:, :w[key].shape[1]] = w[key]
        arrs[key] = a
    cnt = np.concatenate([w["page_cnt"], np.zeros(B * n_self, np.int32)])
    for b in range(B):
        j0 = int(w["n_pages"][b])
        for p in range(n_self):
            ph = n_old + b * n_self + p
            arrs["phys"][b, j0 + p] = ph
            arrs["valid"][b, j0 + p] = min(PAGE, T - PAGE * p)
            arrs["slot"][b, j0 + p] = slot_self
            arrs["page_start"][b, j0 + p] = PAGE * p
            cnt[ph] = min(PAGE, T - PAGE * p)
    doc_pos = np.concatenate([w["doc_pos"], w["qpos"][:, None]], axis=1).astype(np.int32)
    q = rows_bf16(seed, TAG_ROWS_Q, B * T * Hq).reshape(B, T, Hq, HEAD_DIM)
    return dict(name=f"prefill step B{B} T{T} Hq{Hq}/Hk{Hk}", B=B, T=T, Hq=Hq, Hk=Hk, G=Hq // Hk, n_phys=n_phys,
                np_max=np_max, k_pool=k_pool, v_pool=v_pool, q=q, n_pages=(w["n_pages"] + n_self).astype(np.int32),
                doc_pos=doc_pos, qpos0=w["qpos"].astype(np.int32), theta=theta, page_cnt=cnt,
                max_docs=slot_self + 1, seed=seed, **arrs)
