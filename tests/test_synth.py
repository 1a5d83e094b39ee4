"""Checks of the seeded input generator (inputs only; no pipeline arithmetic)."""
import numpy as np

import synth


def test_graph_is_clean_csr():
    g = synth.chung_lu(5000, 10.0, 2.1, 300.0, 0)
    assert g.indptr[0] == 0 and g.indptr[-1] == g.m == len(g.indices)
    assert np.all(np.diff(g.indptr) >= 0)
    assert g.indices.min() >= 0 and g.indices.max() < g.n
    for u in range(0, g.n, 7):
        row = g.indices[g.indptr[u]:g.indptr[u + 1]]
        assert np.all(np.diff(row) > 0)          # sorted, no repeats
        assert not np.any(row == u)              # no self-loops


def test_graph_deterministic_and_seeded():
    a = synth.chung_lu(3000, 8.0, 2.0, 200.0, 7)
    b = synth.chung_lu(3000, 8.0, 2.0, 200.0, 7)
    c = synth.chung_lu(3000, 8.0, 2.0, 200.0, 8)
    assert np.array_equal(a.indptr, b.indptr) and np.array_equal(a.indices, b.indices)
    assert not np.array_equal(a.indices[: min(a.m, c.m)], c.indices[: min(a.m, c.m)])


def test_chung_lu_weights_hit_target_mean_and_max():
    n, mean, gamma, wmax = 100000, 20.0, 2.1, 3000.0
    w = np.array([synth._load().synth_chung_lu_weight(n, mean, gamma, wmax, i) for i in (0, 1, 10, n - 1)])
    assert w[0] <= wmax and w[0] > 0.5 * wmax
    assert np.all(np.diff(w) < 0)
    g = synth.chung_lu(n, mean, gamma, wmax, 0)
    d = g.degrees()
    assert 0.8 * mean < d.mean() <= mean        # dedup only removes edges
    assert d.max() <= 1.2 * wmax
    # heavy tail: the top 1% of nodes hold a large share of the edges
    top = np.sort(d)[::-1][: n // 100].sum()
    assert top > 0.1 * d.sum()


def test_degree_is_not_encoded_in_id():
    g = synth.chung_lu(20000, 10.0, 2.1, 500.0, 0)
    d = g.degrees().astype(float)
    ids = np.arange(g.n, dtype=float)
    assert abs(np.corrcoef(ids, d)[0, 1]) < 0.05


def test_features_normal_and_deterministic():
    f = synth.features(4000, 50, "f32", 0)
    assert abs(f.mean()) < 0.02 and abs(f.std() - 1) < 0.02
    assert np.array_equal(f[100:110], synth.features(10, 50, "f32", 0, row0=100))
    b = synth.features(100, 50, "bf16", 0)
    fb = (b.astype(np.uint32) << 16).view(np.float32)
    assert np.allclose(fb, f[:100], rtol=2 ** -8, atol=0)


def test_batch_seeds_distinct_masked_and_disjoint():
    n = 50000
    b0 = synth.batch_seeds(n, 0.08, 0, 512)
    b1 = synth.batch_seeds(n, 0.08, 1, 512)
    assert len(b0) == len(b1) == 512
    assert len(set(b0.tolist()) | set(b1.tolist())) == 1024
    assert 0.07 * n < synth.mask_count(n, 0.08) < 0.09 * n
    allb = synth.batch_seeds(1000, 1.0, 0, 1000)
    assert sorted(allb.tolist()) == list(range(1000))
    assert len(synth.batch_seeds(1000, 1.0, 1, 1000)) == 0
