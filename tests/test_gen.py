"""The seeded input generator: determinism, counter-based slicing, distributions, bf16 rounding."""
import numpy as np

import gen


def test_counter_based_slices_match_whole():
    a = gen.normal_f64(7, 3, 1000)
    b = gen.normal_f64(7, 3, 400, offset=600)
    assert np.array_equal(a[600:], b)
    r = gen.rows_bf16(1, 2, 50, outlier_p=0.3)
    r2 = gen.rows_bf16(1, 2, 20, row_offset=30, outlier_p=0.3)
    assert np.array_equal(r[30:], r2)


def test_streams_and_seeds_differ():
    assert not np.array_equal(gen.uniform(0, 1, 64), gen.uniform(0, 2, 64))
    assert not np.array_equal(gen.uniform(0, 1, 64), gen.uniform(1, 1, 64))


def test_normal_moments():
    x = gen.normal_f64(0, 9, 400_000)
    assert abs(x.mean()) < 0.01
    assert abs(x.var() - 1.0) < 0.01
    u = gen.uniform(0, 9, 200_000)
    assert 0.0 < u.min() and u.max() < 1.0 and abs(u.mean() - 0.5) < 0.005


def test_bf16_round_to_nearest_even():
    # 1.0, the tie 1 + 2^-8 (rounds to even = 1.0), the tie 1 + 3*2^-8 (rounds up to 1 + 2^-6),
    # -2.5 (exact), and a value just above the tie.
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -8 + 2 ** -20],
                 np.float32)
    got = gen.f32_to_bf16(x)
    assert got.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F81]
    assert np.array_equal(gen.bf16_to_f32(got)[[0, 3]], np.array([1.0, -2.5], np.float32))


def test_outlier_rows_fraction_and_scale():
    rows = gen.rows_bf16(0, 1, 20000, outlier_p=0.01, outlier_scale=20.0)
    base = gen.rows_bf16(0, 1, 20000)
    f = gen.bf16_to_f32(rows).astype(np.float64)
    g = gen.bf16_to_f32(base).astype(np.float64)
    ratio = np.abs(f).sum(1) / np.abs(g).sum(1)
    scaled = ratio > 10
    assert 0.005 < scaled.mean() < 0.015
    assert np.allclose(ratio[scaled], 20.0, rtol=0.02)
    assert np.allclose(ratio[~scaled], 1.0)


def test_tiny_workload_structure():
    w = gen.tiny()
    assert w["k_pool"].shape == (2, 64, 64, 128)
    assert sorted(w["page_table"].ravel().tolist()) == list(range(64))
    assert w["q"].shape == (1, 8, 128) and w["evict"].shape == (1, 2, 64)


def test_lazy_workload_structure():
    w = gen.lazy_rag(B=4, n_docs=16, docs_per_req=3, min_len=100, max_len=300)
    for b in range(4):
        n = w["n_pages"][b]
        assert (w["phys"][b, :n] >= 0).all() and (w["phys"][b, n:] == -1).all()
        assert w["valid"][b, :n].sum() == w["qpos"][b]
        # documents are contiguous: slot i starts at the sum of the previous lengths
        lens = w["doc_len"][w["picks"][b]]
        assert np.array_equal(w["doc_pos"][b], np.concatenate([[0], np.cumsum(lens)[:-1]]))


def test_zipf_draws_top_rank_probability():
    d = gen.zipf_draws(0, 77, 200_000, 256, 1.1)
    h = 1.0 / np.arange(1, 257) ** 1.1
    assert abs((d == 0).mean() - h[0] / h.sum()) < 0.005
    assert d.min() >= 0 and d.max() <= 255
