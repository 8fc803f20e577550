"""ctypes view of ``libspkv.so`` (the C ABI in ``include/spkv.h``).

Loading fails loudly: there is no fallback path.  If the library has not been built, calling
any operation raises ``RuntimeError`` telling how to build it.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
SO_PATH = os.path.join(_HERE, "libspkv.so")

SPKV_OK, SPKV_EINVAL, SPKV_ENOMEM, SPKV_ECUDA, SPKV_EDEVICE, SPKV_ETIMEOUT, SPKV_EUNSUPPORTED = \
    0, -1, -2, -3, -4, -5, -6
DEVERR = {"PAGE_ID": 1, "PHYS": 2, "SLOT": 4, "ORDER": 8, "CAPACITY": 16, "TIMEOUT": 32}

# Every entry point declared in include/spkv.h, with its ctypes signature.
_vp, _i32, _i64, _u32, _f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint32, ctypes.c_float


class SpkvDesc(ctypes.Structure):
    _fields_ = [("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_tokens", ctypes.c_int32), ("subblock", ctypes.c_int32),
                ("n_phys_pages", ctypes.c_int64), ("k_pool", _vp), ("v_pool", _vp),
                ("ksum", _vp), ("page_cnt", _vp), ("max_units", ctypes.c_int32), ("ksum_bf16", ctypes.c_int32)]


class SpkvPageDir(ctypes.Structure):
    _fields_ = [("dir", _vp), ("dev_segs", _vp), ("host_chunks", _vp), ("n_dir", ctypes.c_int32),
                ("seg_shift", ctypes.c_int32), ("n_dev_segs", ctypes.c_int32), ("chunk_shift", ctypes.c_int32),
                ("n_host_segs", ctypes.c_int64)]


_pd = ctypes.POINTER(SpkvPageDir)

SIGNATURES = {
    "paged_kv_create": ([ctypes.POINTER(SpkvDesc), _vp, ctypes.POINTER(_vp)], _i32),
    "paged_kv_append": ([_vp, _vp, _vp, _vp, _vp, _i32, _vp], _i32),
    "score_blocks": ([_vp, _vp, _i32, _i32, _vp, _i32, _vp, _vp, _vp], _i32),
    "decode_append_score": ([_vp, _vp, _vp, _vp, _i32, _i32, _vp, _i32, _vp, _vp, _vp], _i32),
    "select_topk": ([_vp, _vp, _vp, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _vp, _vp], _i32),
    "sparse_decode_attn": ([_vp, _vp, _i32, _i32, _vp, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _vp], _i32),
    "lazy_rope_decode_attn": ([_vp, _vp, _i32, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _i32, _f32, _vp, _vp,
                               _vp], _i32),
    "lazy_rope_prefill_attn": ([_vp, _vp, _i32, _i32, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _i32, _f32, _vp,
                                _vp, _vp], _i32),
    "lazy_rope_prefill_step": ([_vp, _vp, _i32, _i32, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _vp, _i32, _f32, _vp,
                                _vp, _vp], _i32),
    "lazy_alibi_prefill_attn": ([_vp, _vp, _i32, _i32, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _vp, _i32, _vp,
                                 _vp, _vp, _vp], _i32),
    "attn_column_scores": ([_vp, _vp, _i32, _i32, _i32, _vp, _i32, _vp, _vp, _vp], _i32),
    "attn_column_scores_lse": ([_vp, _vp, _vp, _i32, _i32, _i32, _vp, _i32, _vp, _vp, _vp], _i32),
    "resident_setdiff": ([_vp, _vp, _i32, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp], _i32),
    "lru_bucket_update": ([_vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp],
                          _i32),
    "select_resident_update": ([_vp, _vp, _vp, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _i32,
                                _i32, _vp, _vp, _vp, _vp, _vp, _vp], _i32),
    "retrieve_pages": ([_vp, _vp, _vp, _i64, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp], _i32),
    "sparse_decode_attn_slots": ([_vp, _vp, _i32, _i32, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp], _i32),
    "sparse_decode_attn_noalloc": ([_vp, _vp, _i32, _i64, _vp, _i32, _i32, _vp, _i32, _vp, _vp, _i32,
                                    _vp, _vp, _vp, _vp, _vp], _i32),
    "spkv_pack_page_words": ([_vp, _vp, _vp, _i64, _vp], _i32),
    "lazy_docs_plan_create": ([_vp, _i32, _i32, _vp, _i32, _i32, _vp, ctypes.POINTER(_vp)], _i32),
    "lazy_docs_plan_jobs": ([_vp], _i32),
    "lazy_docs_plan_destroy": ([_vp], _i32),
    "lazy_rope_decode_attn_docs": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _vp, _vp], _i32),
    "score_blocks_dir": ([_vp, _vp, _i32, _i32, _pd, _i32, _vp, _vp, _vp], _i32),
    "sparse_decode_attn_dir": ([_vp, _vp, _i32, _i32, _pd, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _vp], _i32),
    "retrieve_pages_dir": ([_vp, _vp, _vp, _i64, _pd, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp], _i32),
    "spkv_pagemap_create": ([_i32, _i32, _i32, _i32, ctypes.POINTER(_vp)], _i32),
    "spkv_pagemap_map": ([_vp, _i32, _i32, _i32, _vp], _i32),
    "spkv_pagemap_promote": ([_vp, _i32, _i32], _i32),
    "spkv_pagemap_sync": ([_vp, _vp], _i32),
    "spkv_pagemap_view": ([_vp, _pd], _i32),
    "spkv_pagemap_bytes": ([_vp, ctypes.POINTER(_i64), ctypes.POINTER(_i64)], _i32),
    "spkv_pagemap_destroy": ([_vp], _i32),
    "spkv_get_device_error": ([_vp, _vp, ctypes.POINTER(_u32)], _i32),
    "paged_kv_destroy": ([_vp], _i32),
    "spkv_sm_count": ([_vp], _i32),
    "spkv_set_wait_limit": ([_vp, ctypes.c_uint64], _i32),
    "spkv_status_string": ([_i32], ctypes.c_char_p),
}

_lib = None


def load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(SO_PATH):
            raise RuntimeError(
                f"{SO_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()'). There is no fallback path.")
        lib = ctypes.CDLL(SO_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


class SpkvError(RuntimeError):
    def __init__(self, fn: str, status: int, bits: int = 0):
        msg = load().spkv_status_string(status).decode()
        if bits:
            msg += " (device error bits " + ", ".join(k for k, v in DEVERR.items() if bits & v) + ")"
        super().__init__(f"{fn}: {msg}")
        self.status = status
        self.bits = bits


def check(fn: str, status: int) -> None:
    if status != SPKV_OK:
        raise SpkvError(fn, status)
