"""The C-ABI library loads and exports every entry point that include/spkv.h declares.

CPU-only: only host-side paths run (symbol lookup, the host packing helper, argument
rejection that happens before any CUDA call)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spkv.h")


@pytest.fixture(scope="module")
def lib():
    from sparse_paged_kv_score_gb300 import build
    build.build()
    from sparse_paged_kv_score_gb300 import _abi
    return _abi.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, re.M)))


def test_header_declares_the_decode_path():
    names = declared_functions()
    for f in ["paged_kv_create", "paged_kv_append", "score_blocks", "decode_append_score", "select_topk", "sparse_decode_attn",
              "lazy_rope_decode_attn", "resident_setdiff", "lru_bucket_update", "spkv_get_device_error",
              "paged_kv_destroy", "spkv_status_string", "spkv_pack_page_words", "spkv_sm_count",
              "retrieve_pages", "sparse_decode_attn_slots", "select_resident_update",
              "lazy_rope_prefill_attn", "lazy_alibi_prefill_attn", "attn_column_scores"]:
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    from sparse_paged_kv_score_gb300 import _abi
    for name in declared_functions():
        assert hasattr(lib, name), f"libspkv.so does not export {name}"
        assert name in _abi.SIGNATURES, f"binding has no signature for {name}"


def test_status_strings(lib):
    assert lib.spkv_status_string(0) == b"SPKV_OK"
    assert b"EINVAL" in lib.spkv_status_string(-1)
    assert lib.spkv_status_string(12345) == b"unknown status"


def test_host_argument_rejection_without_gpu(lib):
    from sparse_paged_kv_score_gb300 import _abi
    out = ctypes.c_void_p()
    assert lib.paged_kv_create(None, None, ctypes.byref(out)) == _abi.SPKV_EINVAL
    d = _abi.SpkvDesc(8, 64, 64, 16, 16, None, None, None, None, 0, 0)
    assert lib.paged_kv_create(ctypes.byref(d), None, ctypes.byref(out)) == _abi.SPKV_EUNSUPPORTED
    d = _abi.SpkvDesc(8, 128, 64, 16, 16, None, None, None, None, 0, 0)
    assert lib.paged_kv_create(ctypes.byref(d), None, ctypes.byref(out)) == _abi.SPKV_EINVAL
    assert lib.sparse_decode_attn(None, None, 1, 8, None, 1, None, None, 1, None, None, None, None) \
        == _abi.SPKV_EINVAL
    assert lib.paged_kv_destroy(None) == _abi.SPKV_EINVAL
    assert lib.retrieve_pages(None, None, None, 1, None, 1, 1, None, None, None, None, None, 1, 1, None) \
        == _abi.SPKV_EINVAL
    assert lib.sparse_decode_attn_slots(None, None, 1, 8, None, None, None, 1, 1, None, None, None, None) \
        == _abi.SPKV_EINVAL
    # summaries are given together or not at all
    d = _abi.SpkvDesc(8, 128, 64, 16, 16, 16, 16, 16, None, 0, 0)
    assert lib.paged_kv_create(ctypes.byref(d), None, ctypes.byref(out)) == _abi.SPKV_EINVAL
    d = _abi.SpkvDesc(8, 128, 64, 16, 16, 16, 16, 16, 16, 0, 2)   # summary type flag out of range
    assert lib.paged_kv_create(ctypes.byref(d), None, ctypes.byref(out)) == _abi.SPKV_EINVAL


def test_pack_page_words_matches_oracle_packing(lib):
    import sparse_paged_kv_score_gb300 as spkv
    rng = np.random.default_rng(0)
    phys = rng.integers(0, 1 << 18, 5000).astype(np.int32)
    valid = rng.integers(1, 65, 5000).astype(np.int32)
    slot = rng.integers(0, 256, 5000).astype(np.int32)
    words = spkv.pack_page_words(phys, valid, slot)
    want = [oracle.meta_pack(p, v, s) for p, v, s in zip(phys, valid, slot)]
    assert words.tolist() == want
    with pytest.raises(spkv.SpkvError):
        spkv.pack_page_words([1], [65], [0])
    with pytest.raises(spkv.SpkvError):
        spkv.pack_page_words([1 << 18], [1], [0])
