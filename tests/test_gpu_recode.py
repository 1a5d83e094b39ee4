"""Parity of the cache presampling and node recoding calls with the oracle
(GARDEN page, Section IV-A: hot nodes recoded to compact IDs, ID-range hit
test; Section IV-B, Eq. (4): full-link access statistics), all bit-exact:
  - sg_access_stats against oracle.access_stats, one mini-batch and a
    super-batch, several layer weights;
  - sg_rank_by_score against oracle.rank_by_score (ties, ragged sizes);
  - sg_graph_renumber against oracle.graph_renumber (int32 and int64
    offsets) and its permutation check;
  - the ID-range cache (no slot map) against the oracle's gather;
  - the whole recoded pipeline (presample, rank, recode, ID-range cache,
    sample, gather, forward, backward) against the oracle on the recoded
    graph.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import as_f64, assert_close, dev_i32, torch_to_np
from sampling_gnn_mini_gb300 import binding as sg
from sampling_gnn_mini_gb300.pipeline import MiniBatchPipeline

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()


def _u32(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("omega,w_in", [([0, 0], 1), ([3, 5], 1), ([1, 2], 0)])
def test_access_stats_one_batch(omega, w_in):
    g = synth.chung_lu(10000, 10.0, 2.1, 500.0, 0)
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    fan = [10, 5]
    score = torch.zeros(g.n, dtype=torch.int32, device="cuda")
    want = np.zeros(g.n, np.uint32)
    bounds = sg.sg_sampler_bounds(G, 256, fan)
    buf = sg.SampleBuffers(bounds, graph=G, n_seeds=256, fanouts=fan)
    for b in range(5):
        seeds = synth.batch_seeds(g.n, 1.0, b, 256)
        sg.sg_sampler_run(G, dev_i32(seeds), fan, 1000 + b, buf)
        sg.sg_access_stats(buf, omega, w_in, score)
        oracle.access_stats(oracle.sampler_run(g.indptr, g.indices, seeds, fan, 1000 + b), omega, w_in, want)
    sg.sg_stream_check()
    assert np.array_equal(_u32(score), want)


def test_access_stats_super_batch():
    g = synth.chung_lu(20000, 12.0, 2.0, 800.0, 3)
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    fan = [8, 4, 3]
    lists = [synth.batch_seeds(g.n, 1.0, k, 100 + 37 * k, 3) for k in range(5)]
    bptr = np.concatenate([[0], np.cumsum([len(x) for x in lists])]).tolist()
    bounds = sg.sg_sampler_bounds(G, bptr[-1], fan, bptr)
    buf = sg.SampleBuffers(bounds, graph=G, n_seeds=bptr[-1], fanouts=fan, batch_ptr=bptr)
    sg.sg_sampler_run(G, dev_i32(np.concatenate(lists)), fan, 99, buf, bptr)
    score = torch.zeros(g.n, dtype=torch.int32, device="cuda")
    sg.sg_access_stats(buf, [2, 1, 4], 3, score, n_sub=len(lists))
    sg.sg_stream_check()
    want = np.zeros(g.n, np.uint32)
    for s in lists:
        oracle.access_stats(oracle.sampler_run(g.indptr, g.indices, s, fan, 99), [2, 1, 4], 3, want)
    assert np.array_equal(_u32(score), want)


@pytest.mark.parametrize("n,hi", [(1, 5), (4095, 3), (4097, 1 << 20), (100_000, 7), (1_000_003, 1 << 31)])
@pytest.mark.parametrize("with_tie", [False, True])
def test_rank_by_score_matches_oracle(n, hi, with_tie):
    rng = np.random.default_rng(n)
    score = rng.integers(0, hi, size=n, dtype=np.uint64).astype(np.uint32)
    score[: n // 7] = score[0]  # a long run of ties
    tie = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32) if with_tie else None
    if with_tie:
        tie[n // 3: n // 2] = 5  # ties of both keys, decided by ID
    order, rank_of = sg.sg_rank_by_score(torch.from_numpy(score.view(np.int32)).cuda(),
                                         None if tie is None else torch.from_numpy(tie.view(np.int32)).cuda())
    sg.sg_stream_check()
    w_order, w_rank = oracle.rank_by_score(score, tie)
    assert np.array_equal(order.cpu().numpy(), w_order)
    assert np.array_equal(rank_of.cpu().numpy(), w_rank)


@pytest.mark.parametrize("offset_bits", [32, 64])
def test_in_degree_matches_oracle(offset_bits):
    g = synth.chung_lu(40000, 12.0, 2.0, 3000.0, 12)
    G = sg.sg_graph_load(g.indptr if offset_bits == 64 else g.indptr.astype(np.int32), g.indices, offset_bits)
    deg = sg.sg_graph_in_degree(G)
    sg.sg_stream_check()
    assert np.array_equal(deg.cpu().numpy().view(np.uint32), oracle.in_degree(g.indices, g.n))


@pytest.mark.parametrize("offset_bits", [32, 64])
def test_graph_renumber_matches_oracle(offset_bits):
    g = synth.chung_lu(30000, 11.0, 2.1, 2000.0, 4)
    ip = g.indptr if offset_bits == 64 else g.indptr.astype(np.int32)
    G = sg.sg_graph_load(ip, g.indices, offset_bits)
    rng = np.random.default_rng(5)
    score = rng.integers(0, 9, size=g.n).astype(np.uint32)
    order, rank_of = oracle.rank_by_score(score)
    G2 = sg.sg_graph_renumber(G, dev_i32(order), dev_i32(rank_of))
    assert (G2.n_nodes, G2.n_edges, G2.offset_bits, G2.max_degree) == (G.n_nodes, G.n_edges, offset_bits,
                                                                      G.max_degree)
    w_ip, w_ix = oracle.graph_renumber(g.indptr, g.indices, order, rank_of)
    ip2, ix2 = sg.sg_graph_copy_out(G2)
    assert np.array_equal(ip2.astype(np.int64), w_ip)
    assert np.array_equal(ix2, w_ix)


def test_graph_renumber_reads_back_exactly():
    # a second recoding with the inverse permutation gives the first graph back
    g = synth.chung_lu(5000, 9.0, 2.1, 300.0, 6)
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    rng = np.random.default_rng(7)
    order = rng.permutation(g.n).astype(np.int32)
    rank_of = np.empty_like(order)
    rank_of[order] = np.arange(g.n, dtype=np.int32)
    G2 = sg.sg_graph_renumber(G, dev_i32(order), dev_i32(rank_of))
    G3 = sg.sg_graph_renumber(G2, dev_i32(rank_of), dev_i32(order))
    ip3, ix3 = sg.sg_graph_copy_out(G3)
    assert np.array_equal(ip3, g.indptr.astype(np.int32)) and np.array_equal(ix3, g.indices)


def test_graph_renumber_rejects_a_non_permutation():
    g = synth.chung_lu(1000, 5.0, 2.1, 50.0, 8)
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    order = np.arange(g.n, dtype=np.int32)
    rank_of = order.copy()
    order[5] = 6  # node 6 twice, node 5 never
    with pytest.raises(sg.SgError) as e:
        sg.sg_graph_renumber(G, dev_i32(order), dev_i32(rank_of))
    assert e.value.status == sg.SG_ERR_INVALID_ARG


@pytest.mark.parametrize("frac", [0.0, 0.3, 1.0])
def test_id_range_cache_gather(frac):
    n, dim = 50000, 64
    feat = synth.features(n, dim, "f32", 9)
    host = torch.from_numpy(feat).pin_memory()
    c = int(frac * n)
    cache = sg.sg_cache_build(host, None, sg.SG_F32, n, dim, None, c)
    assert cache.n_cache == c and cache.slot_of_ptr() in (None, 0)
    ids = np.random.default_rng(1).integers(0, n, size=70001).astype(np.int32)
    out = torch.zeros((len(ids), dim), device="cuda")
    stats = torch.zeros(2, dtype=torch.int64, device="cuda")
    sg.sg_gather(cache, dev_i32(ids), len(ids), None, out, stats)
    sg.sg_stream_check()
    assert np.array_equal(out.cpu().numpy(), oracle.gather(feat, ids))
    hits, misses = stats.cpu().tolist()
    assert hits == int((ids < c).sum()) and misses == int((ids >= c).sum())


def test_recoded_pipeline_matches_oracle():
    """Mid's shape at a tenth of its nodes: presampled Eq. (4) statistics,
    ranking and recoding on the GPU, features laid out in the new order, an
    ID-range cache of half the rows, then a full step against the oracle on
    the recoded graph."""
    n, fan, B, dim = 240_000, [15, 10, 5], 1024, 100
    g = synth.chung_lu(n, 26.0, 2.0, 6000.0, 0)
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    bounds = sg.sg_sampler_bounds(G, B, fan)
    buf = sg.SampleBuffers(bounds, graph=G, n_seeds=B, fanouts=fan)
    score = torch.zeros(n, dtype=torch.int32, device="cuda")
    for b in range(8):
        sg.sg_sampler_run(G, dev_i32(synth.batch_seeds(n, 1.0, b, B, 0, 1000)), fan, 5000 + b, buf)
        sg.sg_access_stats(buf, [1, 1, 1], 1, score)
    order, rank_of = sg.sg_rank_by_score(score, sg.sg_graph_in_degree(G))
    G2 = sg.sg_graph_renumber(G, order, rank_of)
    sg.sg_stream_check()
    order_h, rank_h = order.cpu().numpy(), rank_of.cpu().numpy()
    want_order, _ = oracle.rank_by_score(score.cpu().numpy().view(np.uint32), oracle.in_degree(g.indices, n))
    assert np.array_equal(order_h, want_order)
    ip2, ix2 = oracle.graph_renumber(g.indptr, g.indices, order_h, rank_h)
    feat = synth.features(n, dim, "f32", 0)[order_h]  # new row r = old row order[r]
    host = torch.from_numpy(np.ascontiguousarray(feat)).pin_memory()
    cache = sg.sg_cache_build(host, None, sg.SG_F32, n, dim, None, n // 2)
    pipe = MiniBatchPipeline(G2, cache, fan, B)
    seeds = rank_h[synth.batch_seeds(n, 1.0, 3, B)]
    pipe.set_batch(dev_i32(seeds), 77)
    pipe.step()
    sg.sg_stream_check()
    ref = oracle.sampler_run(ip2, ix2, seeds, fan, 77)
    c = pipe.buf.counts.cpu().numpy()
    assert [int(x) for x in c[:4]] == list(ref.hop_off)
    nH = ref.hop_off[-1]
    assert np.array_equal(pipe.buf.unique[:nH].cpu().numpy(), ref.unique)
    for h in range(3):
        assert np.array_equal(pipe.buf.indptr[h][: ref.hop_off[h] + 1].cpu().numpy(), ref.indptr[h].astype(np.int32))
        assert np.array_equal(pipe.buf.idx[h][: len(ref.idx[h])].cpu().numpy(), ref.idx[h])
    x = torch_to_np(pipe.x[:nH])
    assert np.array_equal(x, oracle.gather(feat, ref.unique))
    hits, misses = pipe.stats.cpu().tolist()
    assert hits == int((ref.unique < n // 2).sum()) and hits + misses == nH
    hh = x
    for h in range(3, 0, -1):
        want, am = oracle.aggregate_fwd(ref.indptr[h - 1], ref.idx[h - 1], hh)
        got = torch_to_np(pipe.h_feat[h - 1][: ref.hop_off[h - 1]])
        assert_close(as_f64(got), want, am, 1e-5, "forward hop %d" % h)
        hh = got
    gg = torch_to_np(pipe.g_feat[0][:B])
    for h in range(1, 4):
        want, am = oracle.aggregate_bwd(ref.indptr[h - 1], ref.idx[h - 1], ref.hop_off[h], gg)
        got = torch_to_np(pipe.g_feat[h][: ref.hop_off[h]])
        assert_close(as_f64(got), want, am, 1e-5, "backward hop %d" % h)
        gg = got
