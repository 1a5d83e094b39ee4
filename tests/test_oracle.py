"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: published
known-answer vectors, a worked example derived from them by hand, closed forms,
library routines (numpy, scipy), invariants and brute force on tiny inputs.
"""
import itertools
import os

import numpy as np
import pytest
import scipy.sparse as sp
from scipy import stats

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------ Philox
def test_philox_known_answers():
    rows = _read_rows("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for r in rows:
        words = [int(x, 16) for x in r]
        ctr, key, want = words[:4], words[4:6], words[6:10]
        assert [int(x) for x in oracle.philox4x32_10(ctr, key)] == want


def test_sample_key_uses_word_j_mod_4():
    # keys of positions 0..3 of (v=0, hop=0, seed=0) are the first KAT vector
    want = [int(x, 16) for x in _read_rows("philox4x32_10_kat.txt")[0][6:10]]
    assert [oracle.sample_key(0, 0, 0, j) for j in range(4)] == want


def test_sample_worked_example():
    indptr = np.array([0, 4], np.int64)
    for row in _read_rows("sample_worked_example.txt"):
        f, want = int(row[0]), [int(x) for x in row[1:]]
        assert oracle.sample_positions(indptr, 0, f, 0, 0).tolist() == want


# ---------------------------------------------------------------- sampling
def _random_graph(rng, n, max_deg):
    deg = rng.integers(0, max_deg + 1, size=n)
    indptr = np.concatenate([[0], np.cumsum(deg)]).astype(np.int64)
    indices = rng.integers(0, n, size=int(indptr[-1])).astype(np.int32)
    return indptr, indices


def test_sample_size_and_full_rows_brute_force():
    rng = np.random.default_rng(1)
    indptr, _ = _random_graph(rng, 60, 40)
    for v in range(60):
        deg = int(indptr[v + 1] - indptr[v])
        for f in (1, 3, 5, 10, 25):
            for hop in (1, 2):
                p = oracle.sample_positions(indptr, v, f, hop, 12345)
                assert len(p) == min(deg, f)
                assert len(set(p.tolist())) == len(p)
                assert np.all(np.diff(p) > 0) and (len(p) == 0 or (p[0] >= 0 and p[-1] < deg))
                if deg <= f:
                    assert p.tolist() == list(range(deg))


def _inclusion_stat(counts, R, f, deg):
    # inclusion counts of a uniform f-subset: covariance R*p(1-p)*d/(d-1)*(I - 11^T/d)
    p = f / deg
    expect = R * p
    scale = R * p * (1 - p) * deg / (deg - 1)
    t = float(((counts - expect) ** 2).sum() / scale)
    return stats.chi2.sf(t, deg - 1)


@pytest.mark.parametrize("deg,f", [(20, 5), (50, 10), (7, 6)])
def test_inclusion_uniform_chi_square(deg, f):
    # GARDEN page, Section IV-C: the sampler must not alter sampling
    # probabilities: every position is kept with probability f/deg
    indptr = np.array([0, deg], np.int64)
    R = 20000
    counts = np.zeros(deg)
    for s in range(R):
        counts[oracle.sample_positions(indptr, 0, f, 1, 0x1234_0000_0000 + s)] += 1
    assert counts.sum() == R * f
    assert _inclusion_stat(counts, R, f, deg) > 1e-3


def test_subsets_equiprobable_chi_square():
    # uniform without replacement: all C(5,2) = 10 subsets equally likely
    indptr = np.array([0, 5], np.int64)
    R = 20000
    subsets = {c: 0 for c in itertools.combinations(range(5), 2)}
    for s in range(R):
        subsets[tuple(oracle.sample_positions(indptr, 0, 2, 2, 977 * s + 3).tolist())] += 1
    obs = np.array(list(subsets.values()), float)
    assert stats.chisquare(obs).pvalue > 1e-3


def test_hub_row_spanning_many_counter_blocks():
    # a star hub with 1000 leaves: positions cover 250 Philox counter blocks
    deg, f, R = 1000, 15, 4000
    indptr = np.array([0, deg], np.int64)
    counts = np.zeros(deg)
    for s in range(R):
        counts[oracle.sample_positions(indptr, 0, f, 3, s)] += 1
    assert _inclusion_stat(counts, R, f, deg) > 1e-3
    # the four words of one counter block are all used
    by_word = counts.reshape(-1, 4).sum(axis=0)
    assert stats.chisquare(by_word).pvalue > 1e-3


def test_sample_depends_on_hop_node_and_seed():
    indptr = np.array([0, 100, 200], np.int64)
    a = oracle.sample_positions(indptr, 0, 5, 1, 7).tolist()
    assert a != oracle.sample_positions(indptr, 0, 5, 2, 7).tolist()
    assert a != oracle.sample_positions(indptr, 1, 5, 1, 7).tolist()
    assert a != oracle.sample_positions(indptr, 0, 5, 1, 8).tolist()
    assert a == oracle.sample_positions(indptr, 0, 5, 1, 7).tolist()


# ------------------------------------------------------- multi-hop + relabel
def _first_occurrence(prefix, ids):
    seen = set(int(x) for x in prefix)
    out = []
    for x in ids:
        x = int(x)
        if x not in seen:
            seen.add(x)
            out.append(x)
    return out


def _check_blocks(indptr, indices, seeds, fanouts, seed, b):
    B = len(seeds)
    assert b.unique[:B].tolist() == list(seeds)                   # seeds first
    assert len(set(b.unique.tolist())) == len(b.unique)          # bijection
    for h in range(1, len(fanouts) + 1):
        f = fanouts[h - 1]
        n_prev, n_cur = b.hop_off[h - 1], b.hop_off[h]
        assert n_prev <= n_cur                                   # V_{h-1} is a prefix of V_h
        bp, idx, nbr, pos = b.indptr[h - 1], b.idx[h - 1], b.nbr[h - 1], b.pos[h - 1]
        assert len(bp) == n_prev + 1 and bp[0] == 0 and bp[-1] == len(idx)
        assert np.all(idx >= 0) and np.all(idx < n_cur)
        assert np.array_equal(b.unique[idx], nbr)                 # round trip
        for d in range(n_prev):
            v = int(b.unique[d])
            deg = int(indptr[v + 1] - indptr[v])
            lo, hi = int(bp[d]), int(bp[d + 1])
            assert hi - lo == min(deg, f)
            assert np.array_equal(nbr[lo:hi], indices[indptr[v] + pos[lo:hi]])
            assert np.array_equal(pos[lo:hi], oracle.sample_positions(indptr, v, f, h, seed))
        # the new nodes of the hop, in order of first occurrence
        assert b.unique[n_prev:n_cur].tolist() == _first_occurrence(b.unique[:n_prev], nbr)


def test_sampler_run_invariants_tiny():
    w = synth.workload("tiny")
    g = synth.chung_lu(2000, w.mean_deg, w.gamma, 200.0, 0)
    seeds = synth.batch_seeds(g.n, 1.0, 0, 64)
    b = oracle.sampler_run(g.indptr, g.indices, seeds, [10, 5], 99)
    _check_blocks(g.indptr, g.indices, seeds.tolist(), [10, 5], 99, b)
    assert b.hop_off[2] > b.hop_off[1] > b.hop_off[0] == 64


def test_sampler_run_hand_graph():
    # path 0->1->2->3 plus node 0 -> {1,2,3}: seeds [0]; fanout 5 keeps all
    indptr = np.array([0, 3, 4, 5, 5], np.int64)
    indices = np.array([1, 2, 3, 2, 3], np.int32)
    b = oracle.sampler_run(indptr, indices, [0], [5, 5], 1)
    assert b.unique.tolist() == [0, 1, 2, 3]
    assert b.hop_off == [1, 4, 4]
    assert b.indptr[0].tolist() == [0, 3] and b.idx[0].tolist() == [1, 2, 3]
    # hop 2 samples every node of V_1 = {0,1,2,3}
    assert b.indptr[1].tolist() == [0, 3, 4, 5, 5]
    assert b.idx[1].tolist() == [1, 2, 3, 2, 3]


def test_sampler_run_deterministic_over_threads():
    g = synth.chung_lu(5000, 12.0, 2.0, 300.0, 3)
    seeds = synth.batch_seeds(g.n, 1.0, 2, 100)
    n0 = oracle.num_threads()
    try:
        oracle.set_threads(1)
        a = oracle.sampler_run(g.indptr, g.indices, seeds, [8, 4, 2], 5)
        oracle.set_threads(max(2, n0))
        b = oracle.sampler_run(g.indptr, g.indices, seeds, [8, 4, 2], 5)
    finally:
        oracle.set_threads(n0)
    assert np.array_equal(a.unique, b.unique)
    for h in range(3):
        assert np.array_equal(a.idx[h], b.idx[h]) and np.array_equal(a.indptr[h], b.indptr[h])


def test_super_batch_layout():
    g = synth.chung_lu(3000, 10.0, 2.1, 200.0, 1)
    seed_lists = [synth.batch_seeds(g.n, 1.0, k, 32) for k in range(4)]
    sb = oracle.super_batch_run(g.indptr, g.indices, seed_lists, [6, 3], 11)
    tot = sb.totals()
    assert len(sb.unique) == tot[-1]
    for h in range(1, 3):
        bp, idx = sb.indptr[h - 1], sb.idx[h - 1]
        assert len(bp) == tot[h - 1] + 1 and bp[-1] == len(idx) == sb.edge_counts[:, h - 1].sum()
        # each concatenated row maps back to its sub-batch's own block
        row = 0
        s_off = 0
        for k, r in enumerate(sb.runs):
            for d in range(r.hop_off[h - 1]):
                lo, hi = bp[row], bp[row + 1]
                rl, rh = r.indptr[h - 1][d], r.indptr[h - 1][d + 1]
                assert np.array_equal(idx[lo:hi] - s_off, r.idx[h - 1][rl:rh])
                row += 1
            s_off += r.hop_off[h]


def test_relabel_standalone():
    rng = np.random.default_rng(4)
    prefix = rng.permutation(1000)[:50].astype(np.int32)
    ids = rng.integers(0, 1000, size=3000).astype(np.int32)
    unique, local = oracle.relabel(ids, prefix)
    assert unique[:50].tolist() == prefix.tolist()
    assert len(set(unique.tolist())) == len(unique)
    assert np.array_equal(unique[local], ids)
    assert unique[50:].tolist() == _first_occurrence(prefix, ids)
    with pytest.raises(ValueError):
        oracle.relabel(ids, np.array([1, 1], np.int32))


# ------------------------------------------------------------------ gather
def test_gather_matches_take():
    rng = np.random.default_rng(5)
    feat = synth.features(500, 24, "f32", 1)
    ids = rng.integers(0, 500, size=2000).astype(np.int32)
    assert np.array_equal(oracle.gather(feat, ids).view(np.uint32), np.take(feat, ids, axis=0).view(np.uint32))
    fb = synth.features(500, 64, "bf16", 1)
    assert np.array_equal(oracle.gather(fb, ids), np.take(fb, ids, axis=0))


# --------------------------------------------------------------- aggregate
def test_aggregate_star_closed_form():
    # hub 0 aggregates leaves 1..n with x_v[c] = v + c: mean = (n+1)/2 + c
    n, dim = 40, 6
    indptr = np.array([0, n], np.int64)
    idx = np.arange(1, n + 1, dtype=np.int32)
    h = (np.arange(n + 1)[:, None] + np.arange(dim)[None, :]).astype(np.float32)
    out, _ = oracle.aggregate_fwd(indptr, idx, h)
    assert np.array_equal(out[0], (n + 1) / 2 + np.arange(dim))


def test_aggregate_complete_graph_closed_form():
    # K_n without self-loops, x_v[c] = v + c: mean over the others = (S - x_v)/(n-1)
    n, dim = 9, 5
    indptr = np.arange(0, n * (n - 1) + 1, n - 1, dtype=np.int64)
    idx = np.array([u for v in range(n) for u in range(n) if u != v], np.int32)
    x = (np.arange(n)[:, None] + np.arange(dim)[None, :]).astype(np.float32)
    out, _ = oracle.aggregate_fwd(indptr, idx, x)
    want = (x.astype(np.float64).sum(axis=0)[None, :] - x) / (n - 1)
    assert np.array_equal(out, want)
    # backward of all-ones: every node is named by n-1 rows of weight 1/(n-1)
    g, _ = oracle.aggregate_bwd(indptr, idx, n, np.ones((n, dim), np.float32))
    assert np.allclose(g, 1.0, rtol=0, atol=1e-15)


def test_aggregate_empty_rows_are_zero():
    indptr = np.array([0, 0, 2, 2], np.int64)
    idx = np.array([0, 1], np.int32)
    h = np.array([[1.0, 2.0], [3.0, 4.0]], np.float32)
    out, _ = oracle.aggregate_fwd(indptr, idx, h)
    assert out.tolist() == [[0, 0], [2, 3], [0, 0]]


def _random_block(rng, n_dst, n_src, f):
    c = rng.integers(0, f + 1, size=n_dst)
    indptr = np.concatenate([[0], np.cumsum(c)]).astype(np.int64)
    idx = rng.integers(0, n_src, size=int(indptr[-1])).astype(np.int32)
    return indptr, idx


def test_aggregate_matches_scipy_sparse():
    rng = np.random.default_rng(6)
    indptr, idx = _random_block(rng, 300, 900, 12)
    c = np.diff(indptr)
    A = sp.csr_matrix((np.ones(len(idx)), idx, indptr), shape=(300, 900))
    x = rng.standard_normal((900, 16)).astype(np.float32)
    out, am = oracle.aggregate_fwd(indptr, idx, x)
    want = (A @ x.astype(np.float64)) / np.maximum(c, 1)[:, None]
    assert np.allclose(out, want, rtol=1e-13, atol=1e-13)
    assert np.allclose(am, (A @ np.abs(x.astype(np.float64))) / np.maximum(c, 1)[:, None])
    g = rng.standard_normal((300, 16)).astype(np.float32)
    gs, _ = oracle.aggregate_bwd(indptr, idx, 900, g)
    wantb = A.T @ (g.astype(np.float64) / np.maximum(c, 1)[:, None])
    assert np.allclose(gs, wantb, rtol=1e-13, atol=1e-13)


def test_aggregate_adjoint_identity():
    rng = np.random.default_rng(7)
    indptr, idx = _random_block(rng, 200, 500, 9)
    x = rng.standard_normal((500, 8)).astype(np.float32)
    y = rng.standard_normal((200, 8)).astype(np.float32)
    ax, _ = oracle.aggregate_fwd(indptr, idx, x)
    aty, _ = oracle.aggregate_bwd(indptr, idx, 500, y)
    lhs = float((ax * y.astype(np.float64)).sum())
    rhs = float((x.astype(np.float64) * aty).sum())
    assert abs(lhs - rhs) <= 1e-10 * (1 + abs(lhs))


def test_aggregate_bf16_input():
    rng = np.random.default_rng(8)
    indptr, idx = _random_block(rng, 50, 80, 6)
    xb = synth.features(80, 32, "bf16", 2)
    out, _ = oracle.aggregate_fwd(indptr, idx, xb)
    out32, _ = oracle.aggregate_fwd(indptr, idx, oracle.bf16_to_f32(xb).reshape(80, 32))
    assert np.array_equal(out, out32)


def test_bf16_decode_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x8000, 0x7F80], np.uint16)
    assert oracle.bf16_to_f32(bits).tolist()[:5] == [1.0, -1.0, 3.140625, 0.0, -0.0]
    assert np.isinf(oracle.bf16_to_f32(bits)[5])


# ------------------------------------------------------------- key ties
def _key_ties():
    rows = _read_rows("key_ties.txt")
    with open(os.path.join(GOLDEN, "key_ties.txt")) as fh:
        seed = int(fh.read().split("Seed ")[1].split(",")[0], 16)
    return seed, [[int(r[0]), int(r[1]), int(r[2]), int(r[3]), int(r[4]), int(r[5], 16), int(r[6])] for r in rows]


def test_key_tie_rows_pin_the_position_tie_break():
    # Rows whose two positions share a Philox key (found by make_key_ties.py):
    # the oracle's own key function gives them the same key, with `rank`
    # smaller keys in the row, and the sample of fanout rank + 1 keeps the
    # lower position only (reading: ties in the key go to the lower position).
    seed, rows = _key_ties()
    assert len(rows) >= 3
    for v, deg, f, j_lo, j_hi, key, rank in rows:
        assert j_lo < j_hi
        keys = np.array([oracle.sample_key(seed, 1, v, j) for j in range(deg)], np.uint64)
        assert keys[j_lo] == key and keys[j_hi] == key
        assert int((keys < key).sum()) == rank and f == rank + 1
        indptr = np.zeros(v + 2, np.int64)
        indptr[v + 1] = deg
        got = oracle.sample_positions(indptr, v, f, 1, seed)
        want = np.sort(np.concatenate([np.nonzero(keys < key)[0], [j_lo]]))
        assert np.array_equal(got, want)


# ------------------------------------------------------- SAGE UPDATE (NEXT-1)
def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 values exactly representable in bf16 -> their bf16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    assert not (b & 0xFFFF).any()
    return (b >> 16).astype(np.uint16)


@pytest.mark.parametrize("bf16", [False, True])
def test_sage_fwd_reduces_to_sums_for_identity_blocks(bf16):
    # W = [I | I]: y = h + m; W = [0 | I]: out = ReLU(m); W = [I | 0]: ReLU(h).
    # Small integers are exact in bf16 and in every sum.
    rng = np.random.default_rng(40)
    n, d = 7, 5
    h = rng.integers(-4, 5, size=(n, d)).astype(np.float32)
    m = rng.integers(-4, 5, size=(n, d)).astype(np.float32)
    eye, zero = np.eye(d, dtype=np.float32), np.zeros((d, d), np.float32)
    conv = _to_bf16_bits if bf16 else (lambda a: a)
    for W, want_y in ((np.hstack([eye, eye]), h + m), (np.hstack([zero, eye]), m), (np.hstack([eye, zero]), h)):
        y, out, am = oracle.sage_fwd(conv(h), conv(m), conv(W))
        assert np.array_equal(y, want_y)
        assert np.array_equal(out, np.maximum(want_y, 0))
        assert np.all(am >= np.abs(y))


def _sage_case(rng, n, d, d_out, margin=0.05):
    """Random float32 inputs whose pre-activations all stay at least `margin`
    away from 0 (so small perturbations cross no ReLU kink)."""
    while True:
        h = rng.standard_normal((n, d)).astype(np.float32)
        m = rng.standard_normal((n, d)).astype(np.float32)
        W = rng.standard_normal((d_out, 2 * d)).astype(np.float32)
        y, _, _ = oracle.sage_fwd(h, m, W)
        if np.abs(y).min() > margin and (y > 0).any() and (y < 0).any():
            return h, m, W


def test_sage_bwd_matches_central_differences():
    # The loss L = sum g * ReLU(y) is linear in each input away from ReLU kinks,
    # so a central difference with a power-of-two step is exact up to fp64
    # rounding: it pins dW, dh and dm without retyping the formulas.
    rng = np.random.default_rng(41)
    n, d, d_out = 4, 3, 5
    h, m, W = _sage_case(rng, n, d, d_out)
    g = rng.standard_normal((n, d_out)).astype(np.float32)
    y, _, _ = oracle.sage_fwd(h, m, W)
    dW, _, dh, dm, _ = oracle.sage_bwd(h, m, W, y, g)
    step = np.float32(2.0 ** -12)

    def loss(hh, mm, ww):
        return float((oracle.sage_fwd(hh, mm, ww)[1] * g.astype(np.float64)).sum())

    for name, arr, grad in (("W", W, dW), ("h", h, dh), ("m", m, dm)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(arr.shape):
            hi, lo = arr.copy(), arr.copy()
            hi[idx] += step
            lo[idx] -= step
            args = {"h": (h, m, W), "m": (h, m, W), "W": (h, m, W)}[name]
            a_hi = [hi if x is arr else x for x in args]
            a_lo = [lo if x is arr else x for x in args]
            num[idx] = (loss(*a_hi) - loss(*a_lo)) / (2 * float(step))
        assert np.allclose(num, grad, rtol=1e-9, atol=1e-9), name


def test_sage_adjoint_identity_where_relu_is_active():
    # With every pre-activation positive the layer is the linear map
    # z -> z W^T, so <y, g> = <z, dz> = <W, dW> (z = [h | m]).
    rng = np.random.default_rng(42)
    n, d, d_out = 6, 4, 3
    h = rng.random((n, d)).astype(np.float32) + 0.1
    m = rng.random((n, d)).astype(np.float32) + 0.1
    W = rng.random((d_out, 2 * d)).astype(np.float32) + 0.1
    g = rng.standard_normal((n, d_out)).astype(np.float32)
    y, out, _ = oracle.sage_fwd(h, m, W)
    assert (y > 0).all() and np.array_equal(y, out)
    dW, _, dh, dm, _ = oracle.sage_bwd(h, m, W, y, g)
    z = np.hstack([h, m]).astype(np.float64)
    a = float((y * g).sum())
    assert np.isclose(a, float((z * np.hstack([dh, dm])).sum()), rtol=1e-12)
    assert np.isclose(a, float((W.astype(np.float64) * dW).sum()), rtol=1e-12)


def test_sage_bwd_zero_where_relu_is_off():
    # y <= 0 (including y exactly 0: h = -m with W = [I | I]) passes no gradient.
    d = 3
    h = np.array([[1, -2, 3], [0, 0, 0]], np.float32)
    m = np.array([[-1, 1, 1], [0, 0, 0]], np.float32)
    W = np.hstack([np.eye(d), np.eye(d)]).astype(np.float32)
    y, out, _ = oracle.sage_fwd(h, m, W)
    assert y.tolist() == [[0, -1, 4], [0, 0, 0]]
    g = np.ones((2, d), np.float32)
    dW, _, dh, dm, _ = oracle.sage_bwd(h, m, W, y, g)
    assert dh.tolist() == [[0, 0, 1], [0, 0, 0]] and dm.tolist() == dh.tolist()
    # only (row 0, output 2) is active, with dy = 1: dW's row 2 is z's row 0
    assert dW.tolist() == [[0] * 6, [0] * 6, [1, -2, 3, -1, 1, 1]]


# ----------------------------------------------- full-link statistics, recoding
def _golden_access_stats():
    rows = {}
    scores = {}
    for line in open(os.path.join(GOLDEN, "access_stats_example.txt")):
        if line.startswith("#") or not line.strip():
            continue
        k, *v = line.split()
        if k == "score":
            scores[int(v[0])] = int(v[1])
        else:
            rows[k] = [int(x) for x in v]
    return rows, scores


def test_access_stats_worked_example():
    rows, scores = _golden_access_stats()
    b = oracle.Blocks(np.array(rows["unique"], np.int32), rows["hop_off"], [None] * 2, [None] * 2, [], [])
    score = np.zeros(10, np.uint32)
    oracle.access_stats(b, rows["omega"], rows["w_in"][0], score)
    for v in range(10):
        assert score[v] == scores.get(v, 0), v


def _sampled_batches(n_batches=6):
    g = synth.chung_lu(3000, 8.0, 2.1, 200.0, 5)
    out = []
    for k in range(n_batches):
        seeds = synth.batch_seeds(g.n, 1.0, k, 50, 5)
        out.append(oracle.sampler_run(g.indptr, g.indices, seeds, [6, 4, 3], 77 + k))
    return g, out


def test_access_stats_plain_count_and_closed_form_total():
    g, runs = _sampled_batches()
    # w_in = 1, omega = 0: the conventional count of gathered appearances
    plain = np.zeros(g.n, np.uint32)
    for r in runs:
        oracle.access_stats(r, [0, 0, 0], 1, plain)
    assert np.array_equal(plain, np.bincount(np.concatenate([r.unique for r in runs]), minlength=g.n))
    # the total over nodes: w_in |V_L| + sum_l omega_l (|V_l| + |V_{l-1}|), per batch
    om, w_in = [2, 7, 3], 4
    score = np.zeros(g.n, np.uint32)
    want = 0
    for r in runs:
        oracle.access_stats(r, om, w_in, score)
        off = r.hop_off
        want += w_in * off[3] + sum(om[l - 1] * (off[l] + off[l - 1]) for l in (1, 2, 3))
    assert int(score.astype(np.int64).sum()) == want
    # linear in the weights
    a = np.zeros(g.n, np.uint32)
    b = np.zeros(g.n, np.uint32)
    for r in runs:
        oracle.access_stats(r, [1, 0, 2], 0, a)
        oracle.access_stats(r, [1, 7, 1], 4, b)
    assert np.array_equal(a + b, score)


def test_rank_by_score_matches_lexsort():
    rng = np.random.default_rng(3)
    score = rng.integers(0, 6, size=5000).astype(np.uint32)  # many ties
    order, rank_of = oracle.rank_by_score(score)
    want = np.lexsort((np.arange(5000), -score.astype(np.int64)))
    assert np.array_equal(order, want)
    assert np.array_equal(rank_of[order], np.arange(5000))


def test_graph_renumber_is_the_permuted_matrix():
    import scipy.sparse as sp
    g = synth.chung_lu(2000, 9.0, 2.1, 150.0, 2)
    rng = np.random.default_rng(4)
    order = rng.permutation(g.n).astype(np.int32)
    rank_of = np.empty_like(order)
    rank_of[order] = np.arange(g.n, dtype=np.int32)
    ip, ix = oracle.graph_renumber(g.indptr, g.indices, order, rank_of)
    A = sp.csr_matrix((np.ones(g.m), g.indices, g.indptr), shape=(g.n, g.n))
    B = sp.csr_matrix((np.ones(len(ix)), ix, ip), shape=(g.n, g.n))
    assert (A[order][:, order] != B).nnz == 0  # new (r, c) = old (order[r], order[c])
    assert np.array_equal(np.diff(ip), np.diff(g.indptr)[order])
    # renumbering back with the inverse permutation gives the graph back,
    # position for position
    ip2, ix2 = oracle.graph_renumber(ip, ix, rank_of, order)
    assert np.array_equal(ip2, g.indptr) and np.array_equal(ix2, g.indices)
    ip3, ix3 = oracle.graph_renumber(g.indptr, g.indices, np.arange(g.n, dtype=np.int32),
                                     np.arange(g.n, dtype=np.int32))
    assert np.array_equal(ip3, g.indptr) and np.array_equal(ix3, g.indices)


# ------------------------------------------- dynamic cache, match and reorder
def test_dyn_cache_without_decay_counts_residual_appearances():
    # gamma = 1 (g = 2^16): no decay, every batch weighs 2^8, so the window's
    # score is 256 x the number of batches a node appeared in, static misses only
    rng = np.random.default_rng(0)
    n = 500
    cached = np.zeros(n, np.uint8)
    cached[:100] = 1
    dc = oracle.DynCache(n, 1 << 16, 4, 50, cached)
    lists = [rng.choice(n, 120, replace=False).astype(np.int32) for _ in range(4)]
    for u in lists:
        dc.batch(u)
    dyn = dc.update()
    cnt = np.bincount(np.concatenate(lists), minlength=n) * (1 - cached.astype(np.int64))
    assert np.array_equal(dc.S.astype(np.int64), 256 * cnt)
    assert not dc.A.any()
    want = np.lexsort((np.arange(n), -cnt))[:50]
    want = want[cnt[want] > 0]
    assert np.array_equal(dyn, want)
    assert not cached[dyn].any()


def test_dyn_cache_half_decay_worked_example():
    # gamma = 1/2, T = 3: W = (64, 128, 256), gamma^3 = 2^13 / 2^16.  Node 7
    # appears in batches 0 and 2 of the first window and batch 1 of the
    # second.  Eq. (5) in reals, in units of one occurrence: 1, 0.5, 1.25,
    # then 0.625, 1.3125, 0.65625; in Q8 that is 320 and then 168.
    dc = oracle.DynCache(10, 1 << 15, 3, 2, np.zeros(10, np.uint8))
    assert list(dc.W) == [64, 128, 256] and dc.G == 1 << 13
    for u in ([7, 1], [2], [7]):
        dc.batch(np.array(u, np.int32))
    dyn = dc.update()
    assert dc.S[7] == 320 and dc.S[1] == 64 and dc.S[2] == 128
    assert list(dyn) == [7, 2]
    for u in ([3], [7], [3]):
        dc.batch(np.array(u, np.int32))
    dc.update()
    assert dc.S[7] == 168


def test_dyn_cache_tracks_the_real_valued_recursion():
    # any gamma: the fixed-point window scores stay within rounding of Eq. (5)
    # run batch by batch in double precision
    rng = np.random.default_rng(2)
    n, T = 300, 5
    g = 52000
    gamma = g / 65536.0
    dc = oracle.DynCache(n, g, T, 10, np.zeros(n, np.uint8))
    real = np.zeros(n)
    for w in range(4):
        for j in range(T):
            u = rng.choice(n, 80, replace=False).astype(np.int32)
            dc.batch(u)
            real *= gamma
            real[u] += 1.0
        dc.update()
        # each rounding down loses at most one unit of 2^-8 per batch, and
        # earlier losses only shrink under the decay
        err = real * 256 - dc.S
        assert np.all(err >= -1e-9) and np.all(err <= T * (w + 1) + 1e-9)


def test_match_positions():
    rng = np.random.default_rng(3)
    prev = rng.choice(10000, 3000, replace=False).astype(np.int32)
    cur = rng.choice(10000, 4000, replace=False).astype(np.int32)
    pos = oracle.match(prev, cur, 10000)
    where = {int(v): i for i, v in enumerate(prev)}
    assert list(pos) == [where.get(int(v), -1) for v in cur]


def test_overlap_and_greedy_order():
    rng = np.random.default_rng(4)
    lists = [rng.choice(2000, int(rng.integers(100, 900)), replace=False).astype(np.int32) for _ in range(7)]
    O = oracle.overlap(lists, 2000)
    for a in range(7):
        for b in range(7):
            assert O[a, b] == len(np.intersect1d(lists[a], lists[b]))
    order = oracle.greedy_order(O, 2)
    assert sorted(order) == list(range(7)) and order[0] == 2
    for k in range(1, 7):  # each step takes the untaken batch overlapping most with the last
        rest = [b for b in range(7) if b not in order[:k]]
        best = max(rest, key=lambda b: (O[order[k - 1], b], -b))
        assert order[k] == best
    # a worked example: from batch 0, 0-2 overlap most, then 2-1 (1 beats 3 on the tie)
    O2 = np.array([[9, 1, 5, 0], [1, 9, 4, 2], [5, 4, 9, 4], [0, 2, 4, 9]])
    assert list(oracle.greedy_order(O2, 0)) == [0, 2, 1, 3]


def test_in_degree_and_ranking_with_a_tie_key():
    g = synth.chung_lu(3000, 8.0, 2.1, 200.0, 9)
    deg = oracle.in_degree(g.indices, g.n)
    assert np.array_equal(deg, np.bincount(g.indices, minlength=g.n))
    rng = np.random.default_rng(6)
    score = rng.integers(0, 3, size=g.n).astype(np.uint32)  # mostly ties
    order, rank_of = oracle.rank_by_score(score, deg)
    want = np.lexsort((np.arange(g.n), -deg.astype(np.int64), -score.astype(np.int64)))
    assert np.array_equal(order, want)
    assert np.array_equal(rank_of[order], np.arange(g.n))
