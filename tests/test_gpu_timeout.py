"""The bounded waits inside the attention kernel end as an error status, not as a hung GPU.

Every hand-off between the warps of an attention CTA (pages from the producer to the consumers,
stages back, partial results to the epilogue warp) waits on an mbarrier for a limited time.  With
the handle's limit at 0, a wait gives up as soon as its phase is not already complete: the
consumers' first wait always comes before the producer's first page has arrived, and the epilogue's
first wait before any consumer has handed anything over, so the call must report SPKV_ETIMEOUT.
Nothing faults and nothing hangs: each CTA waits (with the full limit) for its own copies in
flight and returns.  The next call with the default limit must then be correct again.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import sparse_paged_kv_score_gb300 as spkv
from helpers import DEV, Dev, attn_errors, f32

pytestmark = pytest.mark.gpu


def test_wait_limit_zero_reports_timeout_then_the_handle_recovers():
    w = gen.sparse_workload(8, 32, 8, 64 * 200 + 17, 32, 32, seed=41)
    d = Dev(w)
    sel, n_sel = d.select(d.scores(), f32(w["evict"]), d.new_alive(), w["k_q"], w["k_e"])
    torch.cuda.synchronize()
    assert d.errors() == (0, 0)
    d.cache.set_wait_limit(0)
    d.attn(sel, n_sel)
    st, bits = d.errors()
    assert st == -5 and bits & spkv.DEVERR["TIMEOUT"], (st, bits)
    d.cache.set_wait_limit(1_000_000_000)
    for _ in range(2):
        out, lse = d.attn(sel, n_sel)
        torch.cuda.synchronize()
        assert d.errors() == (0, 0)
        ro, rl = oracle.sparse_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["page_table"], sel.cpu().numpy(),
                                          n_sel.cpu().numpy(), w["seq_len"])
        mx, mean = attn_errors(out.cpu().numpy(), ro)
        assert mx <= 1e-2 and mean <= 1e-3, (mx, mean)
        assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-3
    d.close()


def test_wait_limit_is_checked_on_the_host():
    w = gen.tiny(seed=0)
    d = Dev(w)
    with pytest.raises(spkv.SpkvError):
        d.cache.set_wait_limit(20_000_000_000)
    d.close()
