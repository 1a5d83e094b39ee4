"""Parity of the bounded dynamic cache (GARDEN page, Section IV-B, Eq. (5)-(6))
with the oracle, bit-exact: the scores after every window, the dynamic set
(Top-K), and the gather through static + dynamic caches (rows byte-identical
to the table's; hits = static hits + dynamic hits)."""
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


@pytest.mark.parametrize("ranked,g,T,k", [(False, 52000, 4, 3000), (True, 1 << 15, 3, 500), (False, 1 << 16, 1, 20000)])
def test_dynamic_cache_matches_oracle(ranked, g, T, k):
    n, dim, fan, B = 60_000, 32, [10, 5], 300
    gr = synth.chung_lu(n, 12.0, 2.1, 1500.0, 11)
    G = sg.sg_graph_load(gr.indptr.astype(np.int32), gr.indices)
    feat = synth.features(n, dim, "f32", 11)
    host = torch.from_numpy(feat).pin_memory()
    C = n // 10
    if ranked:  # a slot-map static cache of the highest-degree nodes
        rk = np.argsort(-np.diff(gr.indptr), kind="stable")[:C].astype(np.int32)
        cache = sg.sg_cache_build(host, None, sg.SG_F32, n, dim, rk, C)
        cached = np.zeros(n, np.uint8)
        cached[rk] = 1
    else:  # an ID-range static cache
        cache = sg.sg_cache_build(host, None, sg.SG_F32, n, dim, None, C)
        cached = (np.arange(n) < C).astype(np.uint8)
    sg.sg_dyn_cache_create(cache, k, g, T)
    ref = oracle.DynCache(n, g, T, k, cached)
    bounds = sg.sg_sampler_bounds(G, B, fan)
    buf = sg.SampleBuffers(bounds, graph=G, n_seeds=B, fanouts=fan)
    out = torch.zeros((bounds.max_nodes[2], dim), device="cuda")
    stats = torch.zeros(2, dtype=torch.int64, device="cuda")
    dyn_set = np.zeros(0, np.int32)
    for b in range(3 * T + 1):
        seeds = synth.batch_seeds(n, 1.0, b, B, 11)
        sg.sg_sampler_run(G, dev_i32(seeds), fan, 500 + b, buf)
        d_n = buf.counts[2:3]
        # the gather reads the dynamic set of the previous window
        stats.zero_()
        sg.sg_gather(cache, buf.unique, bounds.max_nodes[2], d_n, out, stats)
        sg.sg_stream_check()
        nH = int(d_n.item())
        uq = buf.unique[:nH].cpu().numpy()
        assert np.array_equal(out[:nH].cpu().numpy(), oracle.gather(feat, uq))
        hits, misses = stats.cpu().tolist()
        assert hits == int(cached[uq].sum()) + int(np.isin(uq, dyn_set).sum()) and hits + misses == nH
        sg.sg_dyn_cache_batch(cache, buf.unique, bounds.max_nodes[2], d_n)
        ref.batch(uq)
        if ref.j == T:
            dyn_set = ref.update()
            kk, j, S, nodes = sg.sg_dyn_cache_state(cache)
            assert kk == k and j == 0
            assert np.array_equal(S, ref.S), "scores after window"
            assert np.array_equal(np.sort(nodes[nodes >= 0]), np.sort(dyn_set)), "dynamic set"
            assert not cached[dyn_set].any()
    sg.sg_stream_check()


def test_dynamic_cache_rejects_bad_requests():
    n, dim = 1000, 16
    host = torch.zeros((n, dim)).pin_memory()
    full = sg.sg_cache_build(host, None, sg.SG_F32, n, dim, None, n)
    with pytest.raises(sg.SgError) as e:
        sg.sg_dyn_cache_create(full, 10, 40000, 4)  # nothing left to supplement
    assert e.value.status == sg.SG_ERR_UNSUPPORTED
    part = sg.sg_cache_build(host, None, sg.SG_F32, n, dim, None, 100)
    for k, g, T in ((0, 40000, 4), (901, 40000, 4), (10, 0, 4), (10, 65537, 4), (10, 40000, 0)):
        with pytest.raises(sg.SgError) as e:
            sg.sg_dyn_cache_create(part, k, g, T)
        assert e.value.status == sg.SG_ERR_INVALID_ARG
    sg.sg_dyn_cache_create(part, 10, 40000, 4)
    with pytest.raises(sg.SgError):
        sg.sg_dyn_cache_create(part, 10, 40000, 4)  # one per cache
