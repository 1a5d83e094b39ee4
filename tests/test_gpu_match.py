"""Parity of Match-Reorder (FastGL explainer page) with the oracle, exact:
sg_match against oracle.match, sg_overlap against oracle.overlap,
sg_greedy_order against oracle.greedy_order, and sg_gather_reuse (rows of
the previous batch reused) against the oracle's gather of the batch."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import dev_i32
from sampling_gnn_mini_gb300 import binding as sg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()


def _sampled(n=50_000, batches=6, B=400, fan=(10, 5)):
    g = synth.chung_lu(n, 14.0, 2.0, 3000.0, 21)
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    bounds = sg.sg_sampler_bounds(G, B, list(fan))
    buf = sg.SampleBuffers(bounds, graph=G, n_seeds=B, fanouts=list(fan))
    lists = []
    for b in range(batches):
        sg.sg_sampler_run(G, dev_i32(synth.batch_seeds(n, 1.0, b, B, 21)), list(fan), 900 + b, buf)
        nH = int(buf.counts[len(fan)].item())
        lists.append(buf.unique[:nH].clone())
    sg.sg_stream_check()
    return n, lists


def test_match_matches_oracle_and_leaves_the_map_idle():
    n, lists = _sampled()
    match_map = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    matched = torch.zeros(1, dtype=torch.int32, device="cuda")
    for a, b in ((0, 1), (1, 2), (4, 4), (5, 0)):
        prev, cur = lists[a], lists[b]
        pos = torch.empty(cur.numel(), dtype=torch.int32, device="cuda")
        matched.zero_()
        # counts through device pointers, one entry short of the capacities
        pn = torch.tensor([prev.numel() - 1], dtype=torch.int32, device="cuda")
        sg.sg_match(prev, prev.numel(), pn, cur, cur.numel(), None, match_map, pos, matched)
        sg.sg_stream_check()
        want = oracle.match(prev.cpu().numpy()[:-1], cur.cpu().numpy(), n)
        assert np.array_equal(pos.cpu().numpy(), want)
        assert int(matched.item()) == int((want >= 0).sum())
        assert bool((match_map == -1).all())


def test_overlap_and_greedy_order_match_oracle():
    n, lists = _sampled(batches=9)
    off = np.concatenate([[0], np.cumsum([x.numel() for x in lists])])
    ids = torch.cat(lists)
    mask = torch.zeros(n, dtype=torch.int32, device="cuda")
    O = sg.sg_overlap(ids, off, mask)
    sg.sg_stream_check()
    want = oracle.overlap([x.cpu().numpy() for x in lists], n)
    assert np.array_equal(O.cpu().numpy(), want)
    assert bool((mask == 0).all())
    for first in (0, 4, 8):
        assert np.array_equal(sg.sg_greedy_order(want, first), oracle.greedy_order(want, first))


@pytest.mark.parametrize("frac", [0.0, 0.4])
def test_gather_reuse_matches_oracle(frac):
    n, lists = _sampled()
    dim = 64
    feat = synth.features(n, dim, "f32", 21)
    host = torch.from_numpy(feat).pin_memory()
    cache = sg.sg_cache_build(host, None, sg.SG_F32, n, dim, None, int(frac * n))
    match_map = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    prev_rows = None
    for b, cur in enumerate(lists):
        m = cur.numel()
        out = torch.full((m, dim), 7.0, device="cuda")
        stats = torch.zeros(2, dtype=torch.int64, device="cuda")
        reused = torch.zeros(1, dtype=torch.int64, device="cuda")
        if prev_rows is None:
            sg.sg_gather(cache, cur, m, None, out, stats)
            want_reused = 0
        else:
            pos = torch.empty(m, dtype=torch.int32, device="cuda")
            sg.sg_match(lists[b - 1], lists[b - 1].numel(), None, cur, m, None, match_map, pos)
            sg.sg_gather_reuse(cache, cur, m, None, pos, prev_rows, out, stats, reused)
            want_reused = int((pos >= 0).sum().item())
        sg.sg_stream_check()
        cur_h = cur.cpu().numpy()
        assert np.array_equal(out.cpu().numpy(), oracle.gather(feat, cur_h))
        hits, misses = stats.cpu().tolist()
        assert int(reused.item()) == want_reused and hits + misses + want_reused == m
        prev_rows = out
