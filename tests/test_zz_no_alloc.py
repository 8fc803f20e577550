"""The allocation-free form of sparse decode attention.

Some callers cannot allocate device memory at all: an inference engine that owns every byte of
device memory through its own allocator and forbids cudaMalloc once serving starts, or code
that may not create a library handle (creating one allocates the handle's split-K workspace).
sparse_decode_attn_noalloc serves them: it takes the pool directly, allocates nothing, and keeps
its split-K scratch in a fixed device array inside the library.  These tests call it through the
C ABI and check that it returns what the handle-based sparse_decode_attn returns, on two calls
in a row (the second call reuses the scratch the first one left behind), and that it refuses a
batch larger than its scratch.  The file name makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

import gen
import sparse_paged_kv_score_gb300 as spkv
from helpers import DEV, Dev, attn_errors, bf, f32

pytestmark = pytest.mark.gpu

ATTN_MAX, ATTN_MEAN = 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_paged_kv_score_gb300 import build
    build.build()
    spkv.load()


def test_noalloc_matches_handle_entry_point_on_two_calls():
    w = gen.sparse_workload(16, 32, 8, 64 * 70 + 11, 32, 32, seed=31, outlier_p=0.01)
    d = Dev(w, max_units=128)
    sel, n_sel = d.select(d.scores(), f32(w["evict"]), d.new_alive(), w["k_q"], w["k_e"])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for call in range(2):
        q = d.q if call == 0 else bf(gen.rows_bf16(77, 1, w["B"] * w["Hq"]).reshape(w["B"], w["Hq"], 128))
        ref_out, ref_lse = d.attn(sel, n_sel, q=q)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        spkv.sparse_decode_attn_noalloc(d.k_pool, d.v_pool, q, d.pt, sel, n_sel, d.L, out, lse, dev_err=err)
        torch.cuda.synchronize()
        mx, mean = attn_errors(out.cpu().numpy(), ref_out.cpu().numpy().astype(np.float64))
        assert mx <= ATTN_MAX and mean <= ATTN_MEAN, (call, mx, mean)
        assert np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy()).max() <= 1e-3
    assert int(err.item()) == 0
    assert d.errors() == (0, 0)
    d.close()


def test_noalloc_refuses_batches_beyond_its_scratch():
    B, Hk = 65, 8                      # 520 units > 512
    k = torch.zeros(Hk, 1, 64, 128, dtype=torch.bfloat16, device=DEV)
    q = torch.zeros(B, Hk * 4, 128, dtype=torch.bfloat16, device=DEV)
    pt = torch.zeros(B, 1, dtype=torch.int32, device=DEV)
    sel = torch.zeros(B, Hk, 1, dtype=torch.int32, device=DEV)
    n_sel = torch.ones(B, Hk, dtype=torch.int32, device=DEV)
    L = torch.ones(B, dtype=torch.int32, device=DEV)
    out = torch.zeros(B, Hk * 4, 128, dtype=torch.float32, device=DEV)
    lse = torch.zeros(B, Hk * 4, dtype=torch.float32, device=DEV)
    with pytest.raises(spkv.SpkvError) as e:
        spkv.sparse_decode_attn_noalloc(k, k, q, pt, sel, n_sel, L, out, lse)
    assert e.value.status == -6
