"""GPU parity of the PyramidKV-style column score S (tcgen05) against the fp64 oracle.

Both sides take every score from each row's log-sum-exp (two passes), the GPU in fp32 with
bf16 operands that are exact inputs: each probability carries a relative error of a few 1e-6, so
S matches to 1e-4 relative (plus 1e-6 absolute), and every row's probabilities still sum to one.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import sparse_paged_kv_score_gb300 as spkv
from helpers import DEV, Dev, bf, i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_paged_kv_score_gb300 import build
    build.build()
    spkv.load()


def _run(w, q, seq_len=None):
    d = Dev(w)
    B, alpha, Hq = q.shape[0], q.shape[1], q.shape[2]
    L = i32(w["seq_len"] if seq_len is None else seq_len)
    out = torch.full((B, Hq, w["np_max"] * 64), float("nan"), dtype=torch.float32, device=DEV)
    spkv.attn_column_scores(d.cache, bf(q), d.pt, L, out)
    res = out.cpu().numpy()
    err = d.errors()
    d.close()
    return res, err


def _check(S, ref, alpha, n):
    assert np.isfinite(S).all()
    assert (np.abs(S - ref) <= 1e-4 * np.abs(ref) + 1e-6).all(), np.abs(S - ref).max()
    assert np.allclose(S.sum(-1), np.minimum(alpha, n), rtol=1e-4, atol=0)


@pytest.mark.parametrize("n,alpha,Hq,Hk", [(200, 9, 8, 2), (64 * 5, 64, 8, 2), (64 * 7 + 13, 128, 16, 4),
                                           (130, 1, 4, 1), (64 * 3, 128, 40, 8), (64 * 9 + 1, 100, 8, 8),
                                           (128, 128, 8, 2), (200, 200, 8, 2)])
def test_column_scores_vs_oracle(n, alpha, Hq, Hk):
    w = gen.sparse_workload(2, Hq, Hk, n, 4, 4, seed=n + alpha)
    q = gen.rows_bf16(n, 321, 2 * alpha * Hq).reshape(2, alpha, Hq, 128)
    S, err = _run(w, q)
    ref = oracle.column_scores_batch(q, w["k_pool"], w["page_table"], w["seq_len"], w["np_max"] * 64)
    assert err == (0, 0)
    _check(S, ref, alpha, n)


@pytest.mark.parametrize("n,alpha", [(5000, 256), (64 * 4 + 7, 129), (64 * 6, 300)])
def test_column_scores_windows_over_one_tile(n, alpha):
    """Windows of more than 128 rows run as 128-row chunks whose column sums add; 5000 / 256 is
    the prompt and window of the page's worked example."""
    w = gen.sparse_workload(1, 8, 2, n, 4, 4, seed=n + alpha)
    q = gen.rows_bf16(n, 324, alpha * 8).reshape(1, alpha, 8, 128)
    S, err = _run(w, q)
    items = np.array([0, 5], np.int32) if n > 1000 else None
    ref = oracle.column_scores_batch(q, w["k_pool"], w["page_table"], w["seq_len"], w["np_max"] * 64, items=items)
    assert err == (0, 0)
    for it in (items if items is not None else range(8)):
        _check(S[0, it], ref[0, it], alpha, n)


def test_column_scores_two_chunk_grid_is_reproducible():
    """A window of 129..256 rows runs both 128-row chunks in one grid, adding onto a zeroed row; two
    addends onto zero round the same in either order, so repeated calls agree bit for bit."""
    w = gen.sparse_workload(2, 8, 2, 64 * 9 + 3, 4, 4, seed=33)
    q = gen.rows_bf16(33, 325, 2 * 200 * 8).reshape(2, 200, 8, 128)
    d = Dev(w)
    outs = []
    for _ in range(3):
        out = torch.full((2, 8, w["np_max"] * 64), float("nan"), dtype=torch.float32, device=DEV)
        spkv.attn_column_scores(d.cache, bf(q), d.pt, i32(w["seq_len"]), out)
        outs.append(out.cpu().numpy())
    assert d.errors() == (0, 0)
    d.close()
    assert all(np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)) for o in outs[1:])
    ref = oracle.column_scores_batch(q, w["k_pool"], w["page_table"], w["seq_len"], w["np_max"] * 64)
    for b in range(2):
        _check(outs[0][b], ref[b], 200, int(w["seq_len"][b]))


def test_column_scores_window_limit():
    w = gen.sparse_workload(1, 8, 2, 2048, 4, 4, seed=3)
    d = Dev(w)
    q = torch.zeros(1, 1025, 8, 128, dtype=torch.bfloat16, device=DEV)
    out = torch.zeros(1, 8, w["np_max"] * 64, dtype=torch.float32, device=DEV)
    with pytest.raises(spkv.SpkvError, match="UNSUPPORTED"):
        spkv.attn_column_scores(d.cache, q, d.pt, i32(w["seq_len"]), out)
    d.close()


def test_column_scores_ragged_prompts_and_rejected_request():
    """Prompts of different lengths in one call; a prompt shorter than the window is rejected
    (error bit, zero row) without disturbing the others."""
    w = gen.sparse_workload(3, 8, 2, 64 * 6, 4, 4, seed=11)
    alpha = 40
    seq = np.array([64 * 6, 64 * 2 + 5, 20], np.int32)   # the last is shorter than alpha
    q = gen.rows_bf16(11, 322, 3 * alpha * 8).reshape(3, alpha, 8, 128)
    S, err = _run(w, q, seq)
    assert err[1] == spkv.DEVERR["PAGE_ID"]
    assert (S[2] == 0).all()
    ref = oracle.column_scores_batch(q[:2], w["k_pool"], w["page_table"][:2], seq[:2], w["np_max"] * 64)
    for b in range(2):
        _check(S[b], ref[b], alpha, seq[b])


def test_column_scores_full_context_sampled_heads():
    """A 32768-token prompt (512 pages) with a 128-row window, sampled query heads."""
    w = gen.sparse_workload(1, 32, 8, 32768, 4, 4, seed=12, outlier_p=0.01)
    alpha = 128
    q = gen.rows_bf16(12, 323, alpha * 32).reshape(1, alpha, 32, 128)
    S, err = _run(w, q)
    assert err == (0, 0)
    items = np.array([0, 13, 31], np.int32)
    ref = oracle.column_scores_batch(q, w["k_pool"], w["page_table"], w["seq_len"], w["np_max"] * 64, items=items)
    for it in items:
        _check(S[0, it], ref[0, it], alpha, 32768)


def _window_lse(w, q):
    """Each window row's log-sum-exp over its visible keys, in numpy fp64 from the bf16 inputs,
    rounded to fp32 as an attention call returns it: [B][alpha][Hq]."""
    B, alpha, Hq = q.shape[0], q.shape[1], q.shape[2]
    G = Hq // w["Hk"]
    out = np.zeros((B, alpha, Hq), np.float32)
    for b in range(B):
        n = int(w["seq_len"][b])
        for hq in range(Hq):
            K = gen.bf16_to_f32(w["k_pool"][hq // G, w["page_table"][b]]).reshape(-1, 128)[:n].astype(np.float64)
            Z = gen.bf16_to_f32(q[b, :, hq]).astype(np.float64) @ K.T / np.sqrt(128.0)
            for j in range(alpha):
                z = Z[j, :n - alpha + j + 1]
                m = z.max()
                out[b, j, hq] = m + np.log(np.exp(z - m).sum())
    return out


@pytest.mark.parametrize("n,alpha,Hq,Hk", [(200, 9, 8, 2), (64 * 7 + 13, 128, 16, 4), (64 * 4 + 7, 129, 8, 2),
                                           (64 * 6, 300, 8, 2), (5000, 256, 8, 2), (256, 256, 8, 2),
                                           (64 * 5 + 3, 64 * 5 + 3, 16, 4)])
def test_column_scores_from_given_lse_vs_oracle(n, alpha, Hq, Hk):
    """The probability pass alone, from each row's LSE as an attention call would return it (fp32):
    against the oracle's given-LSE form on the same fp32 LSE, and against the two-pass GPU form."""
    w = gen.sparse_workload(2, Hq, Hk, n, 4, 4, seed=n + 7 * alpha)
    q = gen.rows_bf16(n, 326, 2 * alpha * Hq).reshape(2, alpha, Hq, 128)
    lse = _window_lse(w, q)
    d = Dev(w)
    out = torch.full((2, Hq, w["np_max"] * 64), float("nan"), dtype=torch.float32, device=DEV)
    spkv.attn_column_scores_lse(d.cache, bf(q), torch.from_numpy(lse).to(DEV), d.pt, i32(w["seq_len"]), out)
    two = torch.full_like(out, float("nan"))
    spkv.attn_column_scores(d.cache, bf(q), d.pt, i32(w["seq_len"]), two)
    S, S2 = out.cpu().numpy(), two.cpu().numpy()
    assert d.errors() == (0, 0)
    d.close()
    items = np.array([0, Hq + 3], np.int32) if n > 1000 else None
    ref = oracle.column_scores_given_lse_batch(q, lse.astype(np.float64), w["k_pool"], w["page_table"],
                                               w["seq_len"], w["np_max"] * 64, items=items)
    for it in (items if items is not None else range(2 * Hq)):
        b, hq = divmod(int(it), Hq)
        _check(S[b, hq], ref[b, hq], alpha, n)
    assert np.allclose(S, S2, rtol=1e-4, atol=1e-6)


def test_column_scores_lse_argument_checks():
    w = gen.sparse_workload(1, 8, 2, 256, 4, 4, seed=3)
    d = Dev(w)
    q = torch.zeros(1, 8, 8, 128, dtype=torch.bfloat16, device=DEV)
    out = torch.zeros(1, 8, w["np_max"] * 64, dtype=torch.float32, device=DEV)
    lib = spkv.load()
    st = lib.attn_column_scores_lse(d.cache.handle, q.data_ptr(), None, 1, 8, 8, d.pt.data_ptr(), w["np_max"],
                                    i32(w["seq_len"]).data_ptr(), out.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    assert st == -1
    d.close()


def test_column_scores_lse_ragged_rejected_and_reproducible():
    """The keys-as-M form over a ragged batch: prompts of different lengths (tile counts), one shorter
    than the window (rejected: error bit, zero row), persistent CTAs whose tile ranges cut through
    (request, head) pairs; repeated calls agree bit for bit, and every valid row matches the oracle."""
    w = gen.sparse_workload(5, 8, 2, 64 * 11, 4, 4, seed=41)
    alpha = 40
    seq = np.array([64 * 6, 64 * 2 + 5, 20, 64 * 11, 64 * 3], np.int32)
    q = gen.rows_bf16(41, 327, 5 * alpha * 8).reshape(5, alpha, 8, 128)
    wl = dict(w, seq_len=np.where(seq >= alpha, seq, alpha).astype(np.int32))
    lse = _window_lse(wl, q)
    lse[2] = 0.0
    d = Dev(w)
    outs = []
    for _ in range(2):
        out = torch.full((5, 8, w["np_max"] * 64), float("nan"), dtype=torch.float32, device=DEV)
        spkv.attn_column_scores_lse(d.cache, bf(q), torch.from_numpy(lse).to(DEV), d.pt, i32(seq), out)
        outs.append(out.cpu().numpy())
    st, bits = d.errors()
    d.close()
    assert bits == spkv.DEVERR["PAGE_ID"]
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    S = outs[0]
    assert (S[2] == 0).all()
    keep = np.array([0, 1, 3, 4])
    ref = oracle.column_scores_given_lse_batch(q[keep], lse[keep].astype(np.float64), w["k_pool"],
                                               w["page_table"][keep], seq[keep], w["np_max"] * 64)
    for i, b in enumerate(keep):
        for hq in range(8):
            _check(S[b, hq], ref[i, hq], alpha, int(seq[b]))


def test_column_scores_lse_beyond_the_tile_table():
    """More requests than the keys-as-M form's tile table holds (4096): both forms run the row-major
    kernel instead (the given-LSE form its probability pass, the other both passes in one launch),
    with the same results."""
    B, alpha = 4100, 4
    w = gen.sparse_workload(B, 4, 1, 64 + 9, 2, 2, seed=43)
    q = gen.rows_bf16(43, 328, B * alpha * 4).reshape(B, alpha, 4, 128)
    items = np.array([0, 4 * 4095 + 1, 4 * 4099 + 3], np.int32)
    lse = np.zeros((B, alpha, 4), np.float32)
    sub = np.array([0, 4095, 4099])
    wl = dict(w, seq_len=w["seq_len"][sub], page_table=w["page_table"][sub])
    lse[sub] = _window_lse(wl, q[sub])
    d = Dev(w)
    out = torch.full((B, 4, w["np_max"] * 64), float("nan"), dtype=torch.float32, device=DEV)
    spkv.attn_column_scores_lse(d.cache, bf(q), torch.from_numpy(lse).to(DEV), d.pt, i32(w["seq_len"]), out)
    two = torch.full_like(out, float("nan"))
    spkv.attn_column_scores(d.cache, bf(q), d.pt, i32(w["seq_len"]), two)
    S, S2 = out.cpu().numpy(), two.cpu().numpy()
    assert d.errors() == (0, 0)
    d.close()
    ref = oracle.column_scores_given_lse_batch(q, lse.astype(np.float64), w["k_pool"], w["page_table"],
                                               w["seq_len"], w["np_max"] * 64, items=items)
    ref2 = oracle.column_scores_batch(q, w["k_pool"], w["page_table"], w["seq_len"], w["np_max"] * 64, items=items)
    for it in items:
        b, hq = divmod(int(it), 4)
        _check(S[b, hq], ref[b, hq], alpha, int(w["seq_len"][b]))
        _check(S2[b, hq], ref2[b, hq], alpha, int(w["seq_len"][b]))
