"""Parity of the CUDA library (through the C ABI) with the CPU oracle.

Bit-exact for sampled blocks, relabel maps and gathered rows; aggregation
within the fp tolerance |gpu - oracle| <= tol * (mean |term| + 1e-30) per
element, tol = 1e-5 for fp32 and 1e-2 for bf16 inputs (fp32 accumulation).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (GpuSample, as_f64, assert_blocks_equal, assert_close, assert_super_equal, dev_i32,
                     feat_tensor, torch_to_np)
from sampling_gnn_mini_gb300 import binding as sg
from sampling_gnn_mini_gb300.pipeline import MiniBatchPipeline, OverlappedPipeline

pytestmark = pytest.mark.gpu

TOL_F32, TOL_BF16 = 1e-5, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()
    yield
    torch.cuda.synchronize()


# ------------------------------------------------------------------ gather
def _cache(feat, ranked, n_cache, dev_copy=False):
    dtype = sg.SG_F32 if feat.dtype == np.float32 else sg.SG_BF16
    host = feat_tensor(feat, pinned=True)
    d = feat_tensor(feat, device="cuda") if dev_copy else None
    return sg.sg_cache_build(host, d, dtype, feat.shape[0], feat.shape[1], ranked, n_cache), host


@pytest.mark.parametrize("dtype,dim", [("f32", 64), ("f32", 100), ("bf16", 1024), ("bf16", 40), ("f32", 4)])
def test_gather_bit_exact_for_any_cache_set(dtype, dim):
    n = 3001
    feat = synth.features(n, dim, dtype, 3)
    rng = np.random.default_rng(0)
    ids = rng.integers(0, n, size=4099).astype(np.int32)
    want = oracle.gather(feat, ids)
    sets = {
        "none": (np.zeros(0, np.int32), 0),
        "half": (rng.permutation(n)[: n // 2].astype(np.int32), n // 2),
        "all": (None, n),
        "random": (rng.permutation(n)[: 777].astype(np.int32), 777),
    }
    for name, (ranked, c) in sets.items():
        cache, _host = _cache(feat, ranked, c)
        out = torch.empty((len(ids), dim), dtype=torch.float32 if dtype == "f32" else torch.bfloat16, device="cuda")
        stats = torch.zeros(2, dtype=torch.int64, device="cuda")
        sg.sg_gather(cache, dev_i32(ids), len(ids), None, out, stats)
        sg.sg_stream_check()
        got = torch_to_np(out)
        assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), name
        cached = np.zeros(n, bool)
        if ranked is None:
            cached[:] = True
        else:
            cached[ranked] = True
        hits = int(cached[ids].sum())
        assert stats.cpu().tolist() == [hits, len(ids) - hits], name


def test_gather_device_count_and_fill_from_device_copy():
    n, dim = 500, 32
    feat = synth.features(n, dim, "f32", 4)
    cache, _h = _cache(feat, None, n, dev_copy=True)
    ids = np.arange(n - 1, -1, -1, dtype=np.int32)
    out = torch.full((n, dim), -7.0, device="cuda")
    d_n = torch.tensor([123], dtype=torch.int32, device="cuda")
    sg.sg_gather(cache, dev_i32(ids), n, d_n, out)
    sg.sg_stream_check()
    got = out.cpu().numpy()
    assert np.array_equal(got[:123], feat[ids[:123]])
    assert np.all(got[123:] == -7.0)


def test_gather_in_two_parts_with_device_first_row():
    # a list gathered as [0, first) and [first, n): each part writes only its
    # rows, together they equal the whole gather; first is clamped to n
    n, dim = 700, 100
    feat = synth.features(n, dim, "f32", 5)
    cache, _h = _cache(feat, np.arange(0, n, 3, dtype=np.int32), n // 3 + 1)
    ids = np.random.default_rng(6).permutation(n).astype(np.int32)
    for first, count in ((250, 600), (0, 600), (600, 600), (900, 600)):
        out = torch.full((n, dim), -3.0, device="cuda")
        d_first = torch.tensor([first], dtype=torch.int32, device="cuda")
        d_n = torch.tensor([count], dtype=torch.int32, device="cuda")
        sg.sg_gather(cache, dev_i32(ids), n, d_n, out, d_first=d_first)
        sg.sg_stream_check()
        got = out.cpu().numpy()
        lo = min(first, count)
        assert np.all(got[:lo] == -3.0) and np.all(got[count:] == -3.0)
        assert np.array_equal(got[lo:count], feat[ids[lo:count]])
        sg.sg_gather(cache, dev_i32(ids), n, d_first, out)  # the prefix [0, first)
        sg.sg_stream_check()
        got = out.cpu().numpy()
        assert np.array_equal(got[:count], feat[ids[:count]])


def test_gather_rejects_out_of_range_id():
    n, dim = 100, 16
    feat = synth.features(n, dim, "f32", 5)
    cache, _h = _cache(feat, None, n)
    ids = np.array([3, n, 7], np.int32)  # n is out of range: checked before any read
    out = torch.full((3, dim), 5.0, device="cuda")
    sg.sg_gather(cache, dev_i32(ids), 3, None, out)
    with pytest.raises(sg.SgError) as e:
        sg.sg_stream_check()
    assert e.value.status == sg.SG_ERR_INVALID_INDEX
    got = out.cpu().numpy()
    assert np.array_equal(got[0], feat[3]) and np.all(got[1] == 0) and np.array_equal(got[2], feat[7])
    sg.sg_stream_check()  # the error word was cleared


# --------------------------------------------------------------- aggregate
def _block(rng, n_dst, n_src, max_c, long_rows=()):
    c = rng.integers(0, max_c + 1, size=n_dst)
    c[::17] = 0
    for r, L in long_rows:
        c[r] = L
    indptr = np.concatenate([[0], np.cumsum(c)]).astype(np.int32)
    idx = rng.integers(0, n_src, size=int(indptr[-1])).astype(np.int32)
    return indptr, idx


CASES = [("f32", "f32", 64), ("f32", "f32", 100), ("f32", "f32", 128), ("f32", "f32", 256), ("f32", "f32", 8),
         ("f32", "f32", 5), ("bf16", "bf16", 1024), ("bf16", "bf16", 64), ("bf16", "f32", 256), ("bf16", "bf16", 12),
         ("f32", "f32", 1100)]


@pytest.mark.parametrize("tin,tout,dim", CASES)
def test_aggregate_fwd_matches_oracle(tin, tout, dim):
    rng = np.random.default_rng(dim)
    n_dst, n_src = 1500, 4000
    indptr, idx = _block(rng, n_dst, n_src, 25, long_rows=[(5, 300), (900, 1000)])
    x = synth.features(n_src, dim, tin, 7)
    want, am = oracle.aggregate_fwd(indptr, idx, x)
    out = torch.empty((n_dst, dim), dtype=torch.float32 if tout == "f32" else torch.bfloat16, device="cuda")
    sg.sg_aggregate_fwd(dev_i32(indptr), dev_i32(idx), n_dst, n_src, None, feat_tensor(x, "cuda"), out)
    sg.sg_stream_check()
    assert_close(as_f64(torch_to_np(out)), want, am, TOL_F32 if tin == "f32" else TOL_BF16, "fwd")
    assert np.all(as_f64(torch_to_np(out))[np.diff(indptr) == 0] == 0)


@pytest.mark.parametrize("tin,tout,dim", CASES)
def test_aggregate_bwd_matches_oracle_and_is_deterministic(tin, tout, dim):
    rng = np.random.default_rng(100 + dim)
    n_dst, n_src = 1200, 3000
    indptr, idx = _block(rng, n_dst, n_src, 20)
    # long transposed segments: src 0 in 400 rows (warp list), src 1 in 5000 (global sort)
    extra_rows = []
    rows = [list(idx[indptr[v]:indptr[v + 1]]) for v in range(n_dst)]
    for v in range(400):
        rows[v].append(0)
    rows += [[1, int(rng.integers(2, n_src))] for _ in range(5000)]
    n_dst = len(rows)
    indptr = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    idx = np.array([u for r in rows for u in r], np.int32)
    g = synth.features(n_dst, dim, tin, 8)
    want, am = oracle.aggregate_bwd(indptr, idx, n_src, g)
    ws = sg.aligned_workspace(sg.sg_aggregate_bwd_workspace(n_dst, n_src, len(idx)))
    outs = []
    for _ in range(2):
        out = torch.empty((n_src, dim), dtype=torch.float32 if tout == "f32" else torch.bfloat16, device="cuda")
        sg.sg_aggregate_bwd(dev_i32(indptr), dev_i32(idx), n_dst, n_src, len(idx), None, feat_tensor(g, "cuda"), out, ws)
        sg.sg_stream_check()
        outs.append(torch_to_np(out))
    assert np.array_equal(outs[0].view(np.uint8), outs[1].view(np.uint8)), "backward not deterministic"
    assert_close(as_f64(outs[0]), want, am, TOL_F32 if tin == "f32" else TOL_BF16, "bwd")


def _long_row_block(rng, n_dst, n_src):
    """A block where a fifth of the rows are longer than the per-group limit
    (17 to 80 edges) and the rest have 0 to 8."""
    c = rng.integers(0, 9, size=n_dst)
    hub = rng.random(n_dst) < 0.2
    c[hub] = rng.integers(17, 81, size=int(hub.sum()))
    indptr = np.concatenate([[0], np.cumsum(c)]).astype(np.int32)
    idx = rng.integers(0, n_src, size=int(indptr[-1])).astype(np.int32)
    return indptr, idx


@pytest.mark.parametrize("tin,tout,dim", [("f32", "f32", 100), ("f32", "f32", 256), ("f32", "f32", 16),
                                          ("bf16", "bf16", 64), ("bf16", "f32", 128)])
def test_aggregate_long_rows_by_list_and_by_pass_agree(tin, tout, dim):
    # Rows longer than a group's limit are summed by whole warps.  The forward
    # finds them through a shared-memory list when the row capacity is small
    # enough and through a pass over the bounds when it is large (device
    # counts give the rows): the same sums, bit for bit, and the oracle's.
    # The backward (always the pass) must not depend on the capacity either.
    rng = np.random.default_rng(300 + dim)
    n_dst, n_src, big = 20000, 30000, 8_000_000
    indptr, idx = _long_row_block(rng, n_dst, n_src)
    odt = torch.float32 if tout == "f32" else torch.bfloat16
    tol = TOL_F32 if tin == "f32" else TOL_BF16
    x = synth.features(n_src, dim, tin, 11)
    d_ip, d_idx, d_x = dev_i32(indptr), dev_i32(idx), feat_tensor(x, "cuda")
    dims = torch.tensor([n_dst, n_src], dtype=torch.int32, device="cuda")
    want, am = oracle.aggregate_fwd(indptr, idx, x)
    outs = []
    for cap in (n_dst, big):
        out = torch.empty((n_dst, dim), dtype=odt, device="cuda")
        sg.sg_aggregate_fwd(d_ip, d_idx, cap, n_src, dims, d_x, out)
        sg.sg_stream_check()
        outs.append(torch_to_np(out))
    assert np.array_equal(outs[0].view(np.uint8), outs[1].view(np.uint8)), "forward: list and pass differ"
    assert_close(as_f64(outs[0]), want, am, tol, "fwd")
    # backward: the transposed rows of popular sources are long
    g = synth.features(n_dst, dim, tin, 12)
    want, am = oracle.aggregate_bwd(indptr, idx, n_src, g)
    d_g = feat_tensor(g, "cuda")
    outs = []
    for cap in (n_src, big):
        ws = sg.aligned_workspace(sg.sg_aggregate_bwd_workspace(n_dst, cap, len(idx)))
        out = torch.empty((n_src, dim), dtype=odt, device="cuda")
        sg.sg_aggregate_bwd(d_ip, d_idx, n_dst, cap, len(idx), dims, d_g, out, ws)
        sg.sg_stream_check()
        outs.append(torch_to_np(out))
        del ws
    assert np.array_equal(outs[0].view(np.uint8), outs[1].view(np.uint8)), "backward: list and pass differ"
    assert_close(as_f64(outs[0]), want, am, tol, "bwd")


def test_aggregate_uses_device_counts():
    rng = np.random.default_rng(9)
    n_dst, n_src, dim = 300, 800, 64
    indptr, idx = _block(rng, n_dst, n_src, 10)
    x = synth.features(n_src, dim, "f32", 9)
    out = torch.full((n_dst, dim), 3.0, device="cuda")
    dims = torch.tensor([200, n_src], dtype=torch.int32, device="cuda")
    sg.sg_aggregate_fwd(dev_i32(indptr), dev_i32(idx), n_dst, n_src, dims, feat_tensor(x, "cuda"), out)
    sg.sg_stream_check()
    want, am = oracle.aggregate_fwd(indptr[:201], idx[: indptr[200]], x)
    got = out.cpu().numpy().astype(np.float64)
    assert_close(got[:200], want, am, TOL_F32)
    assert np.all(got[200:] == 3.0)


def test_aggregate_rejects_out_of_range_column():
    indptr = np.array([0, 2], np.int32)
    idx = np.array([0, 9], np.int32)  # 9 >= n_src: skipped and reported, never read
    x = torch.ones((4, 16), device="cuda")
    out = torch.empty((1, 16), device="cuda")
    sg.sg_aggregate_fwd(dev_i32(indptr), dev_i32(idx), 1, 4, None, x, out)
    with pytest.raises(sg.SgError) as e:
        sg.sg_stream_check()
    assert e.value.status == sg.SG_ERR_INVALID_INDEX


# ----------------------------------------------------------------- sampling
def _tiny_graph():
    w = synth.workload("tiny")
    return w, synth.chung_lu(w.n_nodes, w.mean_deg, w.gamma, w.wmax, w.rng_seed)


def test_sampler_tiny_config_bit_exact():
    w, g = _tiny_graph()
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    for b in range(3):
        seeds = synth.batch_seeds(g.n, w.p_mask, b, w.batch)
        gpu = GpuSample(G, seeds, w.fanouts, w.sampler_seed(b))
        ref = oracle.sampler_run(g.indptr, g.indices, seeds, w.fanouts, w.sampler_seed(b))
        assert_blocks_equal(gpu, ref)


def test_sampler_int64_offsets_same_result():
    w, g = _tiny_graph()
    G32 = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    G64 = sg.sg_graph_load(g.indptr.astype(np.int64), g.indices)
    assert G64.offset_bits == 64
    seeds = synth.batch_seeds(g.n, 1.0, 7, 300)
    a = GpuSample(G32, seeds, [12, 6, 3], 1234)
    b = GpuSample(G64, seeds, [12, 6, 3], 1234)
    assert np.array_equal(a.unique, b.unique)
    for h in range(3):
        assert np.array_equal(a.idx[h], b.idx[h])
    assert_blocks_equal(b, oracle.sampler_run(g.indptr, g.indices, seeds, [12, 6, 3], 1234))


def _star_plus(n_leaves, extra_rows):
    """Node 0 is a hub with n_leaves neighbours; then rows given explicitly."""
    rows = [list(range(1, n_leaves + 1))] + [[] for _ in range(n_leaves)]
    for v, r in extra_rows.items():
        rows[v] = r
    indptr = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int64)
    indices = np.array([u for r in rows for u in r], np.int32)
    return indptr, indices


@pytest.mark.parametrize("fanout", [1, 5, 25, 128, 256])
def test_sampler_hub_rows_and_fanout_limits(fanout):
    # hub of 20000 leaves (largest degree bin), rows around the fanout, empty rows
    extra = {1: list(range(2, 302)), 2: list(range(3, 3 + fanout)), 3: list(range(4, 4 + fanout + 1)),
             4: list(range(5, 5000))}
    indptr, indices = _star_plus(20000, extra)
    G = sg.sg_graph_load(indptr, indices)
    seeds = [0, 1, 2, 3, 4, 7]
    for seed in (0, 99, 2 ** 40 + 17):
        gpu = GpuSample(G, seeds, [fanout, 2], seed)
        assert_blocks_equal(gpu, oracle.sampler_run(indptr, indices, seeds, [fanout, 2], seed))


def test_sampler_key_ties_take_the_lower_position():
    # rows in which two positions share a Philox key, with the fanout set so
    # that only one of the two is taken (tests/golden/key_ties.txt): the
    # 8-lane group, warp and block paths must all keep the lower position
    path = os.path.join(os.path.dirname(__file__), "golden", "key_ties.txt")
    seed = int(open(path).read().split("Seed ")[1].split(",")[0], 16)
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    for r in rows:
        v, deg, f = int(r[0]), int(r[1]), int(r[2])
        n = max(v + 1, deg + 1)
        indptr = np.zeros(n + 1, np.int64)
        indptr[v + 1:] = deg
        indices = np.array([u if u < v else u + 1 for u in range(deg)], np.int32)  # no self-loop
        G = sg.sg_graph_load(indptr, indices)
        for fanouts in ([f], [f, 3]):
            gpu = GpuSample(G, [v], fanouts, seed)
            assert_blocks_equal(gpu, oracle.sampler_run(indptr, indices, [v], fanouts, seed))


def test_sampler_empty_and_isolated():
    indptr = np.array([0, 0, 0, 2, 2], np.int64)
    indices = np.array([0, 1], np.int32)
    G = sg.sg_graph_load(indptr, indices)
    gpu = GpuSample(G, [0, 1], [3, 3], 5)
    assert gpu.tot_nodes == [2, 2, 2] and gpu.tot_edges == [0, 0]
    gpu = GpuSample(G, [2], [1, 1, 1], 5)
    assert_blocks_equal(gpu, oracle.sampler_run(indptr, indices, [2], [1, 1, 1], 5))


def test_sampler_matches_single_row_definition_statistically():
    # every row of a hop is the oracle's own row sample (positions recovered)
    w, g = _tiny_graph()
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    seeds = synth.batch_seeds(g.n, 1.0, 11, 512)
    gpu = GpuSample(G, seeds, [10, 5], 77)
    for d in range(0, 512, 7):
        v = int(gpu.unique[d])
        lo, hi = gpu.indptr[0][d], gpu.indptr[0][d + 1]
        nbr = gpu.unique[gpu.idx[0][lo:hi]]
        pos = oracle.sample_positions(g.indptr, v, 10, 1, 77)
        assert np.array_equal(nbr, g.indices[g.indptr[v] + pos])


def test_sampler_mid_config_bit_exact():
    w = synth.workload("mid")
    g = synth.chung_lu(w.n_nodes, w.mean_deg, w.gamma, w.wmax, w.rng_seed)
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    for b in (0, 5):
        seeds = synth.batch_seeds(g.n, w.p_mask, b, w.batch)
        gpu = GpuSample(G, seeds, w.fanouts, w.sampler_seed(b))
        assert_blocks_equal(gpu, oracle.sampler_run(g.indptr, g.indices, seeds, w.fanouts, w.sampler_seed(b)))


@pytest.mark.parametrize("gamma", [1.8, 2.6])
def test_super_batch_equals_separate_runs(gamma):
    g = synth.chung_lu(60000, 20.0, gamma, (60000 * 20.0) ** 0.5, 2)
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    K, B = 8, 200
    seed_lists = [synth.batch_seeds(g.n, 1.0, k, B) for k in range(K)]
    seed_lists[3] = seed_lists[3][:50]            # ragged sub-batches
    seed_lists[5] = seed_lists[5][:0]             # an empty one
    bptr = np.concatenate([[0], np.cumsum([len(s) for s in seed_lists])]).tolist()
    seeds = np.concatenate(seed_lists)
    gpu = GpuSample(G, seeds, [20, 10], 4242, batch_ptr=bptr)
    ref = oracle.super_batch_run(g.indptr, g.indices, seed_lists, [20, 10], 4242)
    assert_super_equal(gpu, ref)


def test_relabel_standalone_matches_oracle():
    rng = np.random.default_rng(12)
    prefix = rng.permutation(200000)[:3000].astype(np.int32)
    ids = rng.integers(0, 200000, size=50000).astype(np.int32)
    ids[::3] = prefix[rng.integers(0, 3000, size=len(ids[::3]))]
    unique, local, n = sg.sg_relabel(dev_i32(ids), dev_i32(prefix))
    sg.sg_stream_check()
    want_u, want_l = oracle.relabel(ids, prefix)
    n = int(n.item())
    assert n == len(want_u)
    assert np.array_equal(unique.cpu().numpy()[:n], want_u)
    assert np.array_equal(local.cpu().numpy(), want_l)


def test_sampler_reports_bad_seeds():
    w, g = _tiny_graph()
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    b = sg.sg_sampler_bounds(G, 3, [5])
    buf = sg.SampleBuffers(b, graph=G, n_seeds=3, fanouts=[5])
    sg.sg_sampler_run(G, dev_i32([1, 2, 1]), [5], 0, buf)
    with pytest.raises(sg.SgError) as e:
        sg.sg_stream_check()
    assert e.value.status == sg.SG_ERR_INVALID_ARG
    sg.sg_sampler_run(G, dev_i32([1, g.n + 5, 2]), [5], 0, buf)
    with pytest.raises(sg.SgError) as e:
        sg.sg_stream_check()
    assert e.value.status == sg.SG_ERR_INVALID_INDEX
    with pytest.raises(sg.SgError):
        sg.sg_sampler_bounds(G, 3, [0])
    with pytest.raises(sg.SgError):
        sg.sg_sampler_run(G, dev_i32([1, 2, 3]), [5], 0, buf, batch_ptr=[0, 2])


def test_graph_load_validates():
    with pytest.raises(sg.SgError):
        sg.sg_graph_load(np.array([0, 2, 1], np.int64), np.array([0, 1], np.int32))
    with pytest.raises(sg.SgError):
        sg.sg_graph_load(np.array([0, 1, 2], np.int64), np.array([0, 5], np.int32))
    G = sg.sg_graph_load(np.array([0, 1, 3], np.int32), np.array([1, 0, 1], np.int32))
    assert (G.n_nodes, G.n_edges, G.max_degree) == (2, 3, 2)


# ------------------------------------------------------------------ pipeline
def _tiny_pipeline(backward=True):
    w, g = _tiny_graph()
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    feat = synth.features(g.n, w.dim, w.dtype, 0)
    host = feat_tensor(feat, pinned=True)
    cache = sg.sg_cache_build(host, None, sg.SG_F32, g.n, w.dim, None, g.n)
    return w, g, feat, MiniBatchPipeline(G, cache, w.fanouts, w.batch, backward=backward), host


def _check_pipeline_against_oracle(pipe, w, g, feat, seeds, seed):
    ref = oracle.sampler_run(g.indptr, g.indices, seeds, w.fanouts, seed)
    c = pipe.host_counts()
    assert c["nodes"] == list(ref.hop_off)
    H = pipe.H
    nodes = c["nodes"]
    assert np.array_equal(pipe.buf.unique[: nodes[H]].cpu().numpy(), ref.unique)
    x = torch_to_np(pipe.h_feat[H][: nodes[H]])
    assert np.array_equal(x, oracle.gather(feat, ref.unique))
    # each hop compared on the GPU's own input rows
    for h in range(H, 0, -1):
        hin = torch_to_np(pipe.h_feat[h][: nodes[h]])
        want, am = oracle.aggregate_fwd(ref.indptr[h - 1], ref.idx[h - 1], hin)
        assert_close(as_f64(torch_to_np(pipe.h_feat[h - 1][: nodes[h - 1]])), want, am, TOL_F32, "fwd hop %d" % h)
    for h in range(1, H + 1):
        gin = torch_to_np(pipe.g_feat[h - 1][: nodes[h - 1]])
        want, am = oracle.aggregate_bwd(ref.indptr[h - 1], ref.idx[h - 1], nodes[h], gin)
        assert_close(as_f64(torch_to_np(pipe.g_feat[h][: nodes[h]])), want, am, TOL_F32, "bwd hop %d" % h)


def test_pipeline_step_matches_oracle():
    w, g, feat, pipe, _h = _tiny_pipeline()
    for b in (0, 1):
        seeds = synth.batch_seeds(g.n, w.p_mask, b, w.batch)
        pipe.set_batch(dev_i32(seeds), w.sampler_seed(b))
        pipe.step()
        sg.sg_stream_check()
        _check_pipeline_against_oracle(pipe, w, g, feat, seeds, w.sampler_seed(b))


def test_pipeline_cuda_graph_replay_with_new_batches():
    w, g, feat, pipe, _h = _tiny_pipeline()
    s = torch.cuda.Stream()
    seeds0 = synth.batch_seeds(g.n, w.p_mask, 0, w.batch)
    pipe.set_batch(dev_i32(seeds0), w.sampler_seed(0))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        pipe.step()  # warm-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        pipe.step()
    for b in (3, 4):
        seeds = synth.batch_seeds(g.n, w.p_mask, b, w.batch)
        pipe.set_batch(dev_i32(seeds), w.sampler_seed(b))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        sg.sg_stream_check()
        _check_pipeline_against_oracle(pipe, w, g, feat, seeds, w.sampler_seed(b))


@pytest.mark.parametrize("depth,graphs,n_sub,serial", [(2, True, 1, False), (3, False, 1, False),
                                                      (2, True, 3, False), (1, True, 1, False),
                                                      (2, True, 1, True), (3, False, 1, True)])
def test_overlapped_pipeline_matches_batches_run_alone(depth, graphs, n_sub, serial):
    # Batches (or super-batches of n_sub mini-batches) overlapped on `depth`
    # pipelines (sampling and gather of one batch during the forward and
    # backward of the previous; with serial gathers, one batch sampled during
    # the previous batch's gather, the gathers one after another) give, batch
    # by batch, the same counts, sample, H_0 and input gradient, bit for bit,
    # as the same batches run one at a time.
    w, g, feat, single, host = _tiny_pipeline()
    H = single.H
    n = w.batch * n_sub
    bptr = [w.batch * k for k in range(n_sub + 1)] if n_sub > 1 else None
    if n_sub > 1:
        single = MiniBatchPipeline(single.graph, single.cache, w.fanouts, n, batch_ptr=bptr)
    ov = OverlappedPipeline(single.graph, single.cache, w.fanouts, n, depth=depth, batch_ptr=bptr,
                            serial_gathers=serial)
    batches = list(range(10, 17)) if n_sub == 1 else list(range(7))  # all within one epoch of the mask
    seeds = {b: dev_i32(np.concatenate([synth.batch_seeds(g.n, w.p_mask, b * n_sub + k, w.batch)
                                        for k in range(n_sub)])) for b in batches}
    if graphs:
        for p in ov.pipes:
            p.set_batch(seeds[batches[0]], w.sampler_seed(batches[0]))
        torch.cuda.synchronize()
        ov.capture()
    got = {}

    def inputs(b):
        def f(p, s):
            sd = w.sampler_seed(b)
            p.seeds[:n].copy_(seeds[b], non_blocking=True)
            p.d_seed.fill_(sd if sd < (1 << 63) else sd - (1 << 64))
        return f

    def after(b):
        def f(p, s):
            got[b] = (p.buf.counts.clone(), p.buf.unique.clone(), p.h_feat[0].clone(), p.g_feat[H].clone())
        return f

    for b in batches:
        ov.step(inputs(b), after(b))
    torch.cuda.synchronize()
    for s_ in ov.streams:
        sg.sg_stream_check(s_)
    for b in batches:
        single.set_batch(seeds[b], w.sampler_seed(b))
        single.step()
        torch.cuda.synchronize()
        sg.sg_stream_check()
        counts, unique, h0, gx = got[b]
        assert torch.equal(counts, single.buf.counts), "counts, batch %d" % b
        n = single.host_counts()["nodes"]
        assert torch.equal(unique[: n[H]], single.buf.unique[: n[H]]), "sample, batch %d" % b
        assert torch.equal(h0[: n[0]], single.h_feat[0][: n[0]]), "H_0, batch %d" % b
        assert torch.equal(gx[: n[H]], single.g_feat[H][: n[H]]), "input gradient, batch %d" % b


def test_transpose_blocks_match_stable_sort():
    # the transposed blocks list each src row's edges in edge order, with the
    # dst row and 1 / c_dst; compare with numpy's stable argsort
    w, g = _tiny_graph()
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    seeds = synth.batch_seeds(g.n, 1.0, 5, 256)
    gpu = GpuSample(G, seeds, [10, 5, 3], 31)
    tb = sg.TransposedBuffers(gpu.bounds)
    sg.sg_transpose_blocks(gpu.buf, tb)
    sg.sg_stream_check()
    for h in range(3):
        bp, idx = gpu.indptr[h], gpu.idx[h]
        n_src = gpu.tot_nodes[h + 1]
        order = np.argsort(idx, kind="stable")
        dst = np.repeat(np.arange(len(bp) - 1), np.diff(bp))
        want_ptr = np.concatenate([[0], np.cumsum(np.bincount(idx, minlength=n_src))]).astype(np.int32)
        assert np.array_equal(tb.tptr[h][: n_src + 1].cpu().numpy(), want_ptr)
        assert np.array_equal(tb.tdst[h][: len(idx)].cpu().numpy(), dst[order])
        c = np.diff(bp)[dst[order]].astype(np.float32)
        assert np.array_equal(tb.tw[h][: len(idx)].cpu().numpy(), (1.0 / c).astype(np.float32))


def test_sampler_workspace_reused_across_runs_and_errors():
    # the persistent part of the workspace is left clean by every run, also
    # after a run that reported a repeated seed
    w, g = _tiny_graph()
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    b = sg.sg_sampler_bounds(G, 128, [10, 5])
    buf = sg.SampleBuffers(b, graph=G, n_seeds=128, fanouts=[10, 5])
    for it, bi in enumerate([0, 1, 0, 2]):
        seeds = synth.batch_seeds(g.n, 1.0, bi, 128)
        if it == 2:
            bad = seeds.copy()
            bad[7] = bad[3]
            sg.sg_sampler_run(G, dev_i32(bad), [10, 5], 99, buf)
            with pytest.raises(sg.SgError):
                sg.sg_stream_check()
        sg.sg_sampler_run(G, dev_i32(seeds), [10, 5], 99, buf)
        sg.sg_stream_check()
        ref = oracle.sampler_run(g.indptr, g.indices, seeds, [10, 5], 99)
        assert np.array_equal(buf.unique.cpu().numpy()[: ref.hop_off[-1]], ref.unique)
        assert np.array_equal(buf.idx[1].cpu().numpy()[: len(ref.idx[1])], ref.idx[1])
