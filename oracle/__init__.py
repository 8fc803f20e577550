"""fp64 CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference
legs may import this package.  The library under ``sparse_paged_kv_score_gb300`` never does.

The arithmetic lives in ``oracle.cpp`` (plain C++17, double precision, one function per step
of the decode path, each citing the page passage it follows).  This module only compiles it
with g++ and marshals numpy arrays.  bf16 tensors are passed as ``numpy.uint16`` bit patterns.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py`` against brute
force, closed forms, invariants or library routines (see that file's docstring).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

D, PAGE, NSUB = 128, 64, 4


def build(force: bool = False) -> str:
    """Compiles ``liboracle.so`` with g++ if it is missing or older than its source."""
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
        vp, i32, i64, f64, u32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double,
                                  ctypes.c_uint32)
        sig = {
            "orc_meta_pack": ([i32, i32, i32, vp], i32),
            "orc_meta_unpack": ([u32, vp, vp, vp], None),
            "orc_page_means": ([vp, i32, vp, vp], None),
            "orc_score_unit": ([vp, i32, vp, vp, i32, i32, vp], None),
            "orc_select_unit": ([vp, vp, vp, i32, i32, i32, i32, vp, vp], None),
            "orc_attn_unit": ([vp, i32, vp, vp, vp, vp, i32, vp, vp], None),
            "orc_rope": ([vp, f64, f64, vp], None),
            "orc_attn_materialised_unit": ([vp, i32, vp, vp, vp, vp, vp, i32, i32, vp, f64, vp, vp],
                                           None),
            "orc_attn_lazy_unit": ([vp, i32, vp, vp, vp, vp, vp, i32, i32, vp, f64, vp, vp], None),
            "orc_setdiff_unit": ([vp, i32, vp, i32, i32, vp, vp, vp], None),
            "orc_lru_unit": ([vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, vp, vp], None),
            "orc_score_batch": ([i32, i32, i32, vp, vp, i64, vp, i32, vp, vp, i32, vp, i32], None),
            "orc_score_batch_ex": ([i32, i32, i32, vp, vp, i64, vp, i32, vp, vp, i32, i32, vp, i32], None),
            "orc_round_bf16": ([f64], f64),
            "orc_select_batch": ([i32, vp, vp, vp, i32, vp, i32, i32, vp, vp, vp, i32, i32], None),
            "orc_sparse_attn_batch": ([i32, i32, i32, vp, vp, vp, i64, vp, i32, vp, vp, i32, vp, vp,
                                       i32, vp, vp, i32], None),
            "orc_lazy_attn_batch": ([i32, i32, i32, vp, vp, vp, i64, vp, vp, vp, i32, vp, i32, vp, vp,
                                     i32, f64, i32, vp, i32, vp, vp, i32], None),
            "orc_setdiff_batch": ([vp, i32, vp, vp, i32, i32, vp, vp, vp, i32], None),
            "orc_lru_batch": ([vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, i32], None),
            "orc_lazy_prefill_batch": ([i32, i32, i32, i32, vp, vp, vp, i64, vp, vp, vp, i32, vp, i32, vp, vp,
                                        i32, f64, i32, vp, i32, vp, vp, i32], None),
            "orc_alibi_prefill_batch": ([i32, i32, i32, i32, vp, vp, vp, i64, vp, vp, vp, vp, i32, vp, i32, vp,
                                         vp, i32, vp, vp, i32, vp, vp, i32], None),
            "orc_column_scores_batch": ([i32, i32, i32, i32, vp, vp, i64, vp, i32, vp, i32, vp, i32, vp, i32],
                                        None),
            "orc_dir_to_table": ([i32, i32, vp, i32, i32, vp, i32, vp, i64, vp], None),
            "orc_prefill_step_batch": ([i32, i32, i32, i32, vp, vp, vp, i64, vp, vp, vp, vp, i32, vp, i32, vp, vp,
                                        i32, f64, i32, vp, i32, vp, vp, i32], None),
            "orc_column_scores_given_lse_batch": ([i32, i32, i32, i32, vp, vp, vp, i64, vp, i32, vp, i32, vp, i32,
                                                   vp, i32], None),
            "orc_retrieve_unit": ([vp, vp, vp, vp, i32, vp, vp, i32, vp, vp], None),
            "orc_retrieve_batch": ([i32, i32, vp, vp, i64, vp, i32, vp, vp, vp, vp, vp, i32, vp, vp, i64,
                                    i32, i32], None),
            "orc_slot_attn_batch": ([i32, i32, i32, vp, vp, vp, i64, vp, vp, vp, i32, i32, vp, vp, i32,
                                     vp, vp, i32], None),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
    return _lib


def _c(a, dtype):
    """Contiguous array of the given dtype (copy only when needed)."""
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


# ------------------------------------------------------------------ single-unit functions

def meta_pack(phys: int, valid: int, slot: int) -> int:
    w = np.zeros(1, np.uint32)
    if _l().orc_meta_pack(int(phys), int(valid), int(slot), _p(w)) != 0:
        raise ValueError("page word field out of range")
    return int(w[0])


def meta_unpack(word: int):
    a = np.zeros(3, np.int32)
    _l().orc_meta_unpack(int(word) & 0xFFFFFFFF, _p(a[0:]), _p(a[1:]), _p(a[2:]))
    return int(a[0]), int(a[1]), int(a[2])


def page_means(page: np.ndarray, valid: int):
    page = _c(page, np.uint16)
    mean = np.zeros((NSUB, D), np.float64)
    cnt = np.zeros(NSUB, np.int32)
    _l().orc_page_means(_p(page), int(valid), _p(mean), _p(cnt))
    return mean, cnt


def score_unit(q: np.ndarray, kplane: np.ndarray, pt_row: np.ndarray, seq_len: int, np_out: int):
    q, kplane, pt_row = _c(q, np.uint16), _c(kplane, np.uint16), _c(pt_row, np.int32)
    s = np.zeros(np_out, np.float64)
    _l().orc_score_unit(_p(q), q.shape[0], _p(kplane), _p(pt_row), int(seq_len), int(np_out), _p(s))
    return s


def select_unit(s, e, alive, seq_len: int, k_q: int, k_e: int):
    """Returns (sel[k_e+k_q+1], n_sel, alive_after) for one unit."""
    s, e = _c(s, np.float64), _c(e, np.float64)
    alive = _c(alive, np.uint8).copy()
    sel = np.zeros(k_e + k_q + 1, np.int32)
    n = np.zeros(1, np.int32)
    _l().orc_select_unit(_p(s), _p(e), _p(alive), s.shape[0], int(seq_len), int(k_q), int(k_e),
                         _p(sel), _p(n))
    return sel, int(n[0]), alive


def attn_unit(q, kplane, vplane, phys, valid):
    q, kplane, vplane = _c(q, np.uint16), _c(kplane, np.uint16), _c(vplane, np.uint16)
    phys, valid = _c(phys, np.int32), _c(valid, np.int32)
    G = q.shape[0]
    out = np.zeros((G, D), np.float64)
    lse = np.zeros(G, np.float64)
    _l().orc_attn_unit(_p(q), G, _p(kplane), _p(vplane), _p(phys), _p(valid), phys.shape[0], _p(out),
                       _p(lse))
    return out, lse


def rope(x, pos: float, theta: float):
    x = _c(x, np.float64)
    y = np.zeros(D, np.float64)
    _l().orc_rope(_p(x), float(pos), float(theta), _p(y))
    return y


def _lazy_unit(fn, q, kplane, vplane, phys, valid, slot, qpos, doc_pos, theta):
    q, kplane, vplane = _c(q, np.uint16), _c(kplane, np.uint16), _c(vplane, np.uint16)
    phys, valid, slot, doc_pos = (_c(phys, np.int32), _c(valid, np.int32), _c(slot, np.int32),
                                  _c(doc_pos, np.int32))
    G = q.shape[0]
    out = np.zeros((G, D), np.float64)
    lse = np.zeros(G, np.float64)
    fn(_p(q), G, _p(kplane), _p(vplane), _p(phys), _p(valid), _p(slot), phys.shape[0], int(qpos),
       _p(doc_pos), float(theta), _p(out), _p(lse))
    return out, lse


def attn_materialised_unit(q, kplane, vplane, phys, valid, slot, qpos, doc_pos, theta):
    return _lazy_unit(_l().orc_attn_materialised_unit, q, kplane, vplane, phys, valid, slot, qpos,
                      doc_pos, theta)


def attn_lazy_unit(q, kplane, vplane, phys, valid, slot, qpos, doc_pos, theta):
    return _lazy_unit(_l().orc_attn_lazy_unit, q, kplane, vplane, phys, valid, slot, qpos, doc_pos,
                      theta)


def setdiff_unit(resident, sel, n_sel: int, stride: int):
    resident, sel = _c(resident, np.int32), _c(sel, np.int32)
    missing = np.zeros(stride, np.int32)
    slot = np.zeros(stride, np.int32)
    nm = np.zeros(1, np.int32)
    _l().orc_setdiff_unit(_p(resident), resident.shape[0], _p(sel), int(n_sel), int(stride),
                          _p(missing), _p(nm), _p(slot))
    return missing, int(nm[0]), slot


def lru_unit(resident, ts, slot, n_sel: int, missing, n_missing: int, t: int, W: int, stride: int):
    """Returns (resident_after, ts_after, victims, hist)."""
    resident, ts = _c(resident, np.int32).copy(), _c(ts, np.int32).copy()
    slot, missing = _c(slot, np.int32), _c(missing, np.int32)
    victims = np.zeros(stride, np.int32)
    hist = np.zeros(64, np.int32)
    _l().orc_lru_unit(_p(resident), _p(ts), resident.shape[0], _p(slot), int(n_sel), _p(missing),
                      int(n_missing), int(t), int(W), int(stride), _p(victims), _p(hist))
    return resident, ts, victims, hist


# ------------------------------------------------------------------ batch drivers

def _units(units, n):
    return _c(np.arange(n) if units is None else units, np.int32)


def round_bf16(x: float) -> float:
    return _l().orc_round_bf16(float(x))


def score_batch(q, k_pool, page_table, seq_len, units=None, nthreads: int = 0, summary_bf16: bool = False):
    """Block scores [B][Hk][np_max] (fp64) for the listed units (others left 0); with
    summary_bf16 the sub-block sums are rounded to bf16 before the means are taken."""
    q, k_pool = _c(q, np.uint16), _c(k_pool, np.uint16)
    page_table, seq_len = _c(page_table, np.int32), _c(seq_len, np.int32)
    B, Hq, _ = q.shape
    Hk, n_phys = k_pool.shape[0], k_pool.shape[1]
    np_max = page_table.shape[1]
    u = _units(units, B * Hk)
    s = np.zeros((B, Hk, np_max), np.float64)
    _l().orc_score_batch_ex(B, Hq, Hk, _p(q), _p(k_pool), n_phys, _p(page_table), np_max, _p(seq_len),
                            _p(u), u.shape[0], int(bool(summary_bf16)), _p(s), nthreads)
    return s


def select_batch(s, e, alive, seq_len, k_q: int, k_e: int, units=None, nthreads: int = 0):
    """Returns (sel[B][Hk][k+1], n_sel[B][Hk], alive_after[B][Hk][np_max] as uint8)."""
    s, e = _c(s, np.float64), _c(e, np.float64)
    alive = _c(alive, np.uint8).copy()
    seq_len = _c(seq_len, np.int32)
    B, Hk, np_max = s.shape
    stride = k_e + k_q + 1
    sel = np.full((B, Hk, stride), -1, np.int32)
    n_sel = np.zeros((B, Hk), np.int32)
    u = _units(units, B * Hk)
    _l().orc_select_batch(Hk, _p(s), _p(e), _p(alive), np_max, _p(seq_len), int(k_q), int(k_e),
                          _p(sel), _p(n_sel), _p(u), u.shape[0], nthreads)
    return sel, n_sel, alive


def sparse_attn_batch(q, k_pool, v_pool, page_table, sel, n_sel, seq_len, units=None,
                      nthreads: int = 0):
    """Returns (out[B][Hq][128], lse[B][Hq]) in fp64 for the listed units."""
    q, k_pool, v_pool = _c(q, np.uint16), _c(k_pool, np.uint16), _c(v_pool, np.uint16)
    page_table, sel, n_sel, seq_len = (_c(page_table, np.int32), _c(sel, np.int32),
                                       _c(n_sel, np.int32), _c(seq_len, np.int32))
    B, Hq, _ = q.shape
    Hk, n_phys = k_pool.shape[0], k_pool.shape[1]
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    u = _units(units, B * Hk)
    _l().orc_sparse_attn_batch(B, Hq, Hk, _p(q), _p(k_pool), _p(v_pool), n_phys, _p(page_table),
                               page_table.shape[1], _p(sel), _p(n_sel), sel.shape[-1], _p(seq_len),
                               _p(u), u.shape[0], _p(out), _p(lse), nthreads)
    return out, lse


def lazy_attn_batch(q, k_pool, v_pool, phys, valid, slot, n_pages, qpos, doc_pos, theta: float,
                    materialise: bool = True, units=None, nthreads: int = 0):
    """Lazy-RoPE attention; phys/valid/slot are [B][meta_heads][np_max] or [B][np_max]."""
    q, k_pool, v_pool = _c(q, np.uint16), _c(k_pool, np.uint16), _c(v_pool, np.uint16)
    if phys.ndim == 2:
        phys, valid, slot = phys[:, None, :], valid[:, None, :], slot[:, None, :]
    phys, valid, slot = _c(phys, np.int32), _c(valid, np.int32), _c(slot, np.int32)
    n_pages, qpos, doc_pos = _c(n_pages, np.int32), _c(qpos, np.int32), _c(doc_pos, np.int32)
    B, Hq, _ = q.shape
    Hk, n_phys = k_pool.shape[0], k_pool.shape[1]
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    u = _units(units, B * Hk)
    _l().orc_lazy_attn_batch(B, Hq, Hk, _p(q), _p(k_pool), _p(v_pool), n_phys, _p(phys), _p(valid),
                             _p(slot), phys.shape[1], _p(n_pages), phys.shape[2], _p(qpos),
                             _p(doc_pos), doc_pos.shape[1], float(theta), int(bool(materialise)),
                             _p(u), u.shape[0], _p(out), _p(lse), nthreads)
    return out, lse


def setdiff_batch(resident, sel, n_sel, nthreads: int = 0):
    """resident [U][n_slots], sel [U][stride] -> (missing [U][stride], n_missing [U], slot [U][stride])."""
    resident, sel, n_sel = _c(resident, np.int32), _c(sel, np.int32), _c(n_sel, np.int32)
    U, n_slots = resident.shape
    stride = sel.shape[1]
    missing = np.zeros((U, stride), np.int32)
    slot = np.zeros((U, stride), np.int32)
    nm = np.zeros(U, np.int32)
    _l().orc_setdiff_batch(_p(resident), n_slots, _p(sel), _p(n_sel), stride, U, _p(missing), _p(nm),
                           _p(slot), nthreads)
    return missing, nm, slot


def lru_batch(resident, ts, slot, n_sel, missing, n_missing, t: int, W: int, nthreads: int = 0):
    """Returns (resident_after, ts_after, victims [U][stride], hist [U][64])."""
    resident, ts = _c(resident, np.int32).copy(), _c(ts, np.int32).copy()
    slot, n_sel, missing, n_missing = (_c(slot, np.int32), _c(n_sel, np.int32), _c(missing, np.int32),
                                       _c(n_missing, np.int32))
    U, n_slots = resident.shape
    stride = slot.shape[1]
    victims = np.zeros((U, stride), np.int32)
    hist = np.zeros((U, 64), np.int32)
    _l().orc_lru_batch(_p(resident), _p(ts), n_slots, _p(slot), _p(n_sel), _p(missing), _p(n_missing),
                       stride, U, int(t), int(W), _p(victims), _p(hist), nthreads)
    return resident, ts, victims, hist


def retrieve_batch(k_host, v_host, page_table, missing, n_missing, victims, slot, n_sel, k_slots, v_slots,
                   n_slots: int, nthreads: int = 0):
    """Swap-in: copies missing pages into their victim slots of k_slots / v_slots (uint16
    [Hk][n_slot_pages][64][128], modified in place).  slot is [B][Hk][stride] (or [U][stride]);
    returns the completed slot list (same shape)."""
    k_host, v_host = _c(k_host, np.uint16), _c(v_host, np.uint16)
    if not (k_slots.dtype == np.uint16 and v_slots.dtype == np.uint16 and k_slots.flags.c_contiguous
            and v_slots.flags.c_contiguous):
        raise ValueError("k_slots / v_slots must be C-contiguous uint16 arrays (updated in place)")
    page_table = _c(page_table, np.int32)
    missing, n_missing, victims, n_sel = (_c(missing, np.int32), _c(n_missing, np.int32),
                                          _c(victims, np.int32), _c(n_sel, np.int32))
    out_slot = _c(slot, np.int32).copy()
    Hk, n_host = k_host.shape[0], k_host.shape[1]
    B, np_max = page_table.shape
    stride = out_slot.shape[-1]
    _l().orc_retrieve_batch(B, Hk, _p(k_host), _p(v_host), n_host, _p(page_table), np_max, _p(missing),
                            _p(n_missing), _p(victims), _p(out_slot), _p(n_sel), stride, _p(k_slots),
                            _p(v_slots), k_slots.shape[1], int(n_slots), nthreads)
    return out_slot


def slot_attn_batch(q, k_slots, v_slots, sel, slot, n_sel, seq_len, n_slots: int, units=None,
                    nthreads: int = 0):
    """Attention over the selected pages read from their slots; (out[B][Hq][128], lse[B][Hq])."""
    q, k_slots, v_slots = _c(q, np.uint16), _c(k_slots, np.uint16), _c(v_slots, np.uint16)
    sel, slot, n_sel, seq_len = _c(sel, np.int32), _c(slot, np.int32), _c(n_sel, np.int32), _c(seq_len, np.int32)
    B, Hq, _ = q.shape
    Hk = k_slots.shape[0]
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    u = _units(units, B * Hk)
    _l().orc_slot_attn_batch(B, Hq, Hk, _p(q), _p(k_slots), _p(v_slots), k_slots.shape[1], _p(sel), _p(slot),
                             _p(n_sel), sel.shape[-1], int(n_slots), _p(seq_len), _p(u), u.shape[0], _p(out),
                             _p(lse), nthreads)
    return out, lse


def lazy_prefill_batch(q, k_pool, v_pool, phys, valid, slot, n_pages, qpos0, doc_pos, theta: float,
                       materialise: bool = True, items=None, nthreads: int = 0):
    """LazyAttention prefill: q [B][T][Hq][128] (bf16 bits); phys/valid/slot [B][meta_heads][np_max]
    or [B][np_max].  Returns (out [B][T][Hq][128], lse [B][T][Hq]) in fp64 for the listed work
    items ((b * T + t) * Hk + h; all when None)."""
    q, k_pool, v_pool = _c(q, np.uint16), _c(k_pool, np.uint16), _c(v_pool, np.uint16)
    if phys.ndim == 2:
        phys, valid, slot = phys[:, None, :], valid[:, None, :], slot[:, None, :]
    phys, valid, slot = _c(phys, np.int32), _c(valid, np.int32), _c(slot, np.int32)
    n_pages, qpos0, doc_pos = _c(n_pages, np.int32), _c(qpos0, np.int32), _c(doc_pos, np.int32)
    B, T, Hq, _ = q.shape
    Hk, n_phys = k_pool.shape[0], k_pool.shape[1]
    out = np.zeros((B, T, Hq, D), np.float64)
    lse = np.zeros((B, T, Hq), np.float64)
    it = _units(items, B * T * Hk)
    _l().orc_lazy_prefill_batch(B, T, Hq, Hk, _p(q), _p(k_pool), _p(v_pool), n_phys, _p(phys), _p(valid),
                                _p(slot), phys.shape[1], _p(n_pages), phys.shape[2], _p(qpos0), _p(doc_pos),
                                doc_pos.shape[1], float(theta), int(bool(materialise)), _p(it), it.shape[0],
                                _p(out), _p(lse), nthreads)
    return out, lse


def prefill_step_batch(q, k_pool, v_pool, phys, valid, slot, page_start, n_pages, qpos0, doc_pos, theta: float,
                       mode: str = "materialised", items=None, nthreads: int = 0):
    """The whole RoPE prefill step: rows at positions qpos0[b] + t over every listed key at a position
    m = doc_pos[slot] + page_start + row <= the row's position (the rows' own keys listed as a document
    placed at qpos0).  mode: "materialised" (keys rotated to their positions), "lazy" (query rotated
    per document) or "lazy_bf16q" (the lazy form with the rotated query rounded to bf16).
    Arrays as lazy_prefill_batch, page_start with the shape of phys.  Returns (out, lse)."""
    modes = {"materialised": 0, "lazy": 1, "lazy_bf16q": 2}
    q, k_pool, v_pool = _c(q, np.uint16), _c(k_pool, np.uint16), _c(v_pool, np.uint16)
    if phys.ndim == 2:
        phys, valid, slot, page_start = phys[:, None, :], valid[:, None, :], slot[:, None, :], page_start[:, None, :]
    phys, valid, slot, page_start = (_c(phys, np.int32), _c(valid, np.int32), _c(slot, np.int32),
                                     _c(page_start, np.int32))
    n_pages, qpos0, doc_pos = _c(n_pages, np.int32), _c(qpos0, np.int32), _c(doc_pos, np.int32)
    B, T, Hq, _ = q.shape
    Hk, n_phys = k_pool.shape[0], k_pool.shape[1]
    out = np.zeros((B, T, Hq, D), np.float64)
    lse = np.zeros((B, T, Hq), np.float64)
    it = _units(items, B * T * Hk)
    _l().orc_prefill_step_batch(B, T, Hq, Hk, _p(q), _p(k_pool), _p(v_pool), n_phys, _p(phys), _p(valid), _p(slot),
                                _p(page_start), phys.shape[1], _p(n_pages), phys.shape[2], _p(qpos0), _p(doc_pos),
                                doc_pos.shape[1], float(theta), modes[mode], _p(it), it.shape[0], _p(out), _p(lse),
                                nthreads)
    return out, lse


def alibi_prefill_batch(q, k_pool, v_pool, phys, valid, slot, page_start, n_pages, qpos0, doc_pos, slopes,
                        items=None, nthreads: int = 0):
    """ALiBi prefill over cached documents: like lazy_prefill_batch with the linear position bias
    -slopes[hq] * (n - m) instead of the rotation; page_start (document-local position of each
    listed page's first token) has the shape of phys; slopes [Hq] (fp32).  Returns (out, lse)."""
    q, k_pool, v_pool = _c(q, np.uint16), _c(k_pool, np.uint16), _c(v_pool, np.uint16)
    if phys.ndim == 2:
        phys, valid, slot, page_start = phys[:, None, :], valid[:, None, :], slot[:, None, :], page_start[:, None, :]
    phys, valid, slot, page_start = (_c(phys, np.int32), _c(valid, np.int32), _c(slot, np.int32),
                                     _c(page_start, np.int32))
    n_pages, qpos0, doc_pos = _c(n_pages, np.int32), _c(qpos0, np.int32), _c(doc_pos, np.int32)
    slopes = _c(slopes, np.float32)
    B, T, Hq, _ = q.shape
    Hk, n_phys = k_pool.shape[0], k_pool.shape[1]
    out = np.zeros((B, T, Hq, D), np.float64)
    lse = np.zeros((B, T, Hq), np.float64)
    it = _units(items, B * T * Hk)
    _l().orc_alibi_prefill_batch(B, T, Hq, Hk, _p(q), _p(k_pool), _p(v_pool), n_phys, _p(phys), _p(valid),
                                 _p(slot), _p(page_start), phys.shape[1], _p(n_pages), phys.shape[2], _p(qpos0),
                                 _p(doc_pos), doc_pos.shape[1], _p(slopes), _p(it), it.shape[0], _p(out), _p(lse),
                                 nthreads)
    return out, lse


def column_scores_batch(q, k_pool, page_table, seq_len, n_out: int, items=None, nthreads: int = 0):
    """PyramidKV-style score S per (request, query head): q [B][alpha][Hq][128] (bf16 bits) are the
    prompt's last alpha rows; returns S [B][Hq][n_out] (fp64) for the listed items (b * Hq + hq)."""
    q, k_pool = _c(q, np.uint16), _c(k_pool, np.uint16)
    page_table, seq_len = _c(page_table, np.int32), _c(seq_len, np.int32)
    B, alpha, Hq, _ = q.shape
    Hk, n_phys = k_pool.shape[0], k_pool.shape[1]
    S = np.zeros((B, Hq, n_out), np.float64)
    it = _units(items, B * Hq)
    _l().orc_column_scores_batch(B, Hq, Hk, alpha, _p(q), _p(k_pool), n_phys, _p(page_table), page_table.shape[1],
                                 _p(seq_len), int(n_out), _p(it), it.shape[0], _p(S), nthreads)
    return S


def column_scores_given_lse_batch(q, lse, k_pool, page_table, seq_len, n_out: int, items=None, nthreads: int = 0):
    """The column score with each window row's log-sum-exp given: lse [B][alpha][Hq] (natural log);
    S[b][hq][i] = sum over the rows j that see key i of exp(q_j . k_i / sqrt(128) - lse[b][j][hq])."""
    q, k_pool = _c(q, np.uint16), _c(k_pool, np.uint16)
    lse = _c(lse, np.float64)
    page_table, seq_len = _c(page_table, np.int32), _c(seq_len, np.int32)
    B, alpha, Hq, _ = q.shape
    if lse.shape != (B, alpha, Hq):
        raise ValueError("lse must be [B][alpha][Hq]")
    Hk, n_phys = k_pool.shape[0], k_pool.shape[1]
    S = np.zeros((B, Hq, n_out), np.float64)
    it = _units(items, B * Hq)
    _l().orc_column_scores_given_lse_batch(B, Hq, Hk, alpha, _p(q), _p(lse), _p(k_pool), n_phys, _p(page_table),
                                           page_table.shape[1], _p(seq_len), int(n_out), _p(it), it.shape[0],
                                           _p(S), nthreads)
    return S


def dir_to_table(dir_, shift: int, dev_segs, host_segs, np_max: int):
    """The flat page table [B][np_max] a two-level directory describes: dir_ [B][n_dir] (entries
    >= 0 device segment, <= -2 host segment -2 - e, -1 unmapped), dev_segs [n_dev][2^shift],
    host_segs [n_host][2^shift]."""
    dir_ = _c(dir_, np.int32)
    seg = 1 << shift
    dev_segs = _c(np.asarray(dev_segs).reshape(-1, seg), np.int32)
    host_segs = _c(np.asarray(host_segs).reshape(-1, seg), np.int32)
    B, n_dir = dir_.shape
    out = np.zeros((B, np_max), np.int32)
    _l().orc_dir_to_table(B, int(np_max), _p(dir_), n_dir, int(shift), _p(dev_segs), dev_segs.shape[0],
                          _p(host_segs), host_segs.shape[0], _p(out))
    return out
