"""Parity at the full sizes of the Skew, Billion-edge and Wide workloads, in
the launch configuration the benchmark uses (MiniBatchPipeline: sample,
transpose, gather, forward, backward).

The oracle recomputes: whole mini-batches of the sampler (two sub-batches of
a super-batch), every gathered row, and every aggregation hop forward and
backward (each on the GPU's own input rows) -- whole where the hop's arrays
are small enough for the oracle's fp64 sums, else 20,000 sampled dst rows
(forward) and src rows (backward) through the oracle on a sub-block that
keeps each named dst row whole.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import as_f64, assert_close, dev_i32, torch_to_np
from sampling_gnn_mini_gb300 import binding as sg
from sampling_gnn_mini_gb300.hostmem import pinned_table
from sampling_gnn_mini_gb300.pipeline import MiniBatchPipeline, recode_by_access

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL = {"f32": 1e-5, "bf16": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()
    yield
    torch.cuda.synchronize()


class PinnedTable:
    """The whole feature table in page-locked host memory (as the benchmark
    holds it), with a numpy view for the checks (bf16 as uint16 bits); with
    `order`, row r holds node order[r]'s features (a recoded table)."""

    def __init__(self, n, dim, dtype, seed, order=None):
        self.t = pinned_table(n, dim, torch.float32 if dtype == "f32" else torch.bfloat16)
        if order is None:
            synth.features_into(self.t.data_ptr(), 0, n, dim, dtype, seed)
        else:
            synth.features_rows_into(self.t.data_ptr(), order, dim, dtype, seed)
        self.arr = self.t.numpy() if dtype == "f32" else self.t.view(torch.int16).numpy().view(np.uint16)


def _take(t, rows):
    """Rows of a tensor, as numpy (bf16 as uint16 bits)."""
    return torch_to_np(t[torch.from_numpy(np.asarray(rows, dtype=np.int64)).to(t.device)])


def _sub_blocks(pipe, k):
    """Mini-batch k of a super-batch from the pipeline's concatenated layout."""
    c = pipe.buf.counts.cpu().numpy()
    H, K = pipe.H, len(pipe.batch_ptr) - 1 if pipe.batch_ptr else 1
    per = np.array([[c[(2 * H + 1) * (1 + kk) + h] for h in range(H + 1)] for kk in range(K)], np.int64)
    off = np.concatenate([np.zeros((1, H + 1), np.int64), np.cumsum(per, axis=0)])
    u0 = off[k, H]
    unique = pipe.buf.unique[u0: u0 + per[k, H]].cpu().numpy()
    blocks = []
    for h in range(1, H + 1):
        r0, r1 = off[k, h - 1], off[k, h - 1] + per[k, h - 1]
        ip = pipe.buf.indptr[h - 1][r0: r1 + 1].cpu().numpy().astype(np.int64)
        idx = pipe.buf.idx[h - 1][ip[0]: ip[-1]].cpu().numpy().astype(np.int64) - off[k, h]
        blocks.append((ip - ip[0], idx.astype(np.int32)))
    return per[k].tolist(), unique, blocks


def _check_sampling(pipe, g, seeds_k, k, fanouts, seed):
    ref = oracle.sampler_run(g.indptr, g.indices, seeds_k, fanouts, seed)
    n, unique, blocks = _sub_blocks(pipe, k)
    assert n == list(ref.hop_off)
    assert np.array_equal(unique, ref.unique)
    for h in range(len(fanouts)):
        assert np.array_equal(blocks[h][0], ref.indptr[h]), "indptr, hop %d" % (h + 1)
        assert np.array_equal(blocks[h][1], ref.idx[h]), "idx, hop %d" % (h + 1)


def _check_gather(pipe, feat):
    """Every gathered row, byte for byte, against the oracle's gather of the
    same IDs from the whole table."""
    H = pipe.H
    n = int(pipe.buf.counts[H].item())
    ids = pipe.buf.unique[:n].cpu().numpy()
    got = torch_to_np(pipe.x[:n])
    assert np.array_equal(got, oracle.gather(feat, ids))


# A hop is checked whole when its arrays fit this many elements (fp64 sums and
# |term| sums of the oracle over the whole block); larger hops are checked on
# n_check sampled rows, through the oracle on a sub-block with the same rows.
FULL_ELEMS = 1 << 26


def _row_edges(ip, rows):
    """Edge positions of the given rows of a CSR, row after row."""
    lens = ip[rows + 1] - ip[rows]
    if lens.sum() == 0:
        return np.zeros(0, np.int64)
    first = np.repeat(ip[rows] - np.concatenate([[0], np.cumsum(lens)[:-1]]), lens)
    return first + np.arange(int(lens.sum()))


def _sub_block_fwd(ip, idx, rows):
    """The dst rows `rows` of a block with their whole rows, over the distinct
    srcs they name (returned for the caller to fetch)."""
    sub_ip = np.concatenate([[0], np.cumsum(ip[rows + 1] - ip[rows])])
    uniq, loc = np.unique(idx[_row_edges(ip, rows)], return_inverse=True)
    return sub_ip, loc.astype(np.int32), uniq


def _sub_block_bwd(ip, idx, n_src, srcs):
    """The dst rows that name a src in `srcs`, each with its whole row (so its
    count c_v is unchanged); srcs become columns 0..S-1 and every other src
    the sink column S, whose result is dropped."""
    col = np.full(n_src, len(srcs), np.int64)
    col[srcs] = np.arange(len(srcs))
    dst_of = np.repeat(np.arange(len(ip) - 1), np.diff(ip))
    rows = np.unique(dst_of[col[idx] < len(srcs)])
    sub_ip = np.concatenate([[0], np.cumsum(ip[rows + 1] - ip[rows])])
    return sub_ip, col[idx[_row_edges(ip, rows)]].astype(np.int32), rows


def _check_aggregation(pipe, rng, dtype, n_check=20000):
    """Forward and backward of every hop against the oracle: the whole block
    where it fits FULL_ELEMS, else n_check sampled dst rows (forward) and
    src rows (backward), each on the GPU's own input rows."""
    H = pipe.H
    c = pipe.buf.counts.cpu().numpy()
    dim = pipe.x.shape[1]
    for h in range(1, H + 1):
        n_dst, n_src = int(c[h - 1]), int(c[h])
        ip = pipe.buf.indptr[h - 1][: n_dst + 1].cpu().numpy().astype(np.int64)
        idx = pipe.buf.idx[h - 1][: ip[-1]].cpu().numpy()
        whole = n_src * dim <= FULL_ELEMS
        # forward: out[v] = mean of H_h over row v
        if whole:
            want, am = oracle.aggregate_fwd(ip, idx, torch_to_np(pipe.h_feat[h][:n_src]))
            got = as_f64(torch_to_np(pipe.h_feat[h - 1][:n_dst]))
        else:
            rows = np.sort(rng.choice(n_dst, size=min(n_dst, n_check), replace=False))
            sub_ip, loc, uniq = _sub_block_fwd(ip, idx, rows)
            want, am = oracle.aggregate_fwd(sub_ip, loc, _take(pipe.h_feat[h], uniq))
            got = as_f64(_take(pipe.h_feat[h - 1], rows))
        assert_close(got, want, am, TOL[dtype], "forward hop %d" % h)
        # backward: gsrc[u] = sum over the rows v naming u of gdst[v] / c_v
        if whole:
            want, am = oracle.aggregate_bwd(ip, idx, n_src, torch_to_np(pipe.g_feat[h - 1][:n_dst]))
            got = as_f64(torch_to_np(pipe.g_feat[h][:n_src]))
        else:
            srcs = np.sort(rng.choice(n_src, size=min(n_src, n_check), replace=False))
            sub_ip, sub_idx, rows = _sub_block_bwd(ip, idx, n_src, srcs)
            want, am = oracle.aggregate_bwd(sub_ip, sub_idx, len(srcs) + 1, _take(pipe.g_feat[h - 1], rows))
            want, am = want[: len(srcs)], am[: len(srcs)]
            got = as_f64(_take(pipe.g_feat[h], srcs))
        assert_close(got, want, am, TOL[dtype], "backward hop %d" % h)


# ----------------------------------------------------------------- Skew
SKEW = [("skew_g1.8_b512", (0, 7)), ("skew_g2.0_b512", (0, 7)), ("skew_g2.3_b512", (0, 7)),
        ("skew_g2.6_b512", (0, 7)), ("skew_g1.8_b4096", (0, 5)), ("skew_g2.0_b4096", (0, 3)),
        ("skew_g2.3_b4096", (2, 7)), ("skew_g2.6_b4096", (1, 6))]


@pytest.mark.parametrize("name,check_subs", SKEW)
def test_skew_super_batch_full_size(name, check_subs):
    w = synth.workload(name)
    g = synth.chung_lu(w.n_nodes, w.mean_deg, w.gamma, w.wmax, w.rng_seed)
    G = sg.sg_graph_load(g.indptr.astype(np.int32), g.indices)
    feat = synth.features(w.n_nodes, w.dim, w.dtype, w.rng_seed)
    d_feat = torch.from_numpy(feat).cuda()
    cache = sg.sg_cache_build(None, d_feat, sg.SG_F32, w.n_nodes, w.dim, None, w.n_nodes)  # 100% in HBM
    del d_feat
    bs = synth.BatchStream(w)
    seed_lists = [bs.seeds(k) for k in range(w.n_sub)]
    bptr = np.concatenate([[0], np.cumsum([len(s) for s in seed_lists])]).tolist()
    pipe = MiniBatchPipeline(G, cache, w.fanouts, bptr[-1], batch_ptr=bptr)
    seed = w.sampler_seed(0)
    pipe.set_batch(dev_i32(np.concatenate(seed_lists)), seed)
    pipe.step()
    sg.sg_stream_check()
    for k in check_subs:
        _check_sampling(pipe, g, seed_lists[k], k, w.fanouts, seed)
    rng = np.random.default_rng(1)
    _check_gather(pipe, feat)
    _check_aggregation(pipe, rng, w.dtype)
    del pipe, cache, G, feat
    gc.collect()
    torch.cuda.empty_cache()


# ------------------------------------------------- Billion-edge and Wide
@pytest.mark.parametrize("name", ["billion", "wide"])
def test_host_feature_workloads_full_size(name):
    """The benchmark's launch configuration: presampled full-link statistics,
    ranking and recoding on the GPU, the host table laid out in the new order,
    an ID-range cache of the budget's rows, then one mini-batch through every
    stage, checked against the oracle on the recoded graph."""
    w = synth.workload(name)
    g = synth.chung_lu(w.n_nodes, w.mean_deg, w.gamma, w.wmax, w.rng_seed)
    indptr = g.indptr if w.offset_bits == 64 else g.indptr.astype(np.int32)
    G0 = sg.sg_graph_load(indptr, g.indices, w.offset_bits)
    del g, indptr
    pre = synth.BatchStream(w, epoch0=1000)
    batches = ((dev_i32(pre.seeds(b)), w.presample_seed(b)) for b in range(8))
    G, order, rank_of = recode_by_access(G0, batches, w.fanouts, [1] * w.n_hops)
    del G0
    assert G.offset_bits == w.offset_bits
    ip, ix = sg.sg_graph_copy_out(G)
    order_h, rank_h = order.cpu().numpy(), rank_of.cpu().numpy()
    table = PinnedTable(w.n_nodes, w.dim, w.dtype, w.rng_seed, order=order_h)
    try:
        cache = sg.sg_cache_build(table.t, None, sg.SG_F32 if w.dtype == "f32" else sg.SG_BF16, w.n_nodes, w.dim,
                                  None, w.cache_rows)
        assert cache.slot_of_ptr() in (None, 0)  # the ID-range hit test
        pipe = MiniBatchPipeline(G, cache, w.fanouts, w.batch)
        seeds = rank_h[synth.BatchStream(w).seeds(0)]
        pipe.set_batch(dev_i32(seeds), w.sampler_seed(0))
        pipe.step()
        sg.sg_stream_check()
        hits, misses = pipe.stats.cpu().tolist()
        assert misses > 0 and hits > 0  # both the HBM cache and the host table were read
        n = int(pipe.buf.counts[w.n_hops].item())
        assert hits == int((pipe.buf.unique[:n] < w.cache_rows).sum().item())
        rg = synth.csr_graph(ip.astype(np.int64), ix)
        _check_sampling(pipe, rg, seeds, 0, w.fanouts, w.sampler_seed(0))
        rng = np.random.default_rng(2)
        _check_gather(pipe, table.arr)
        _check_aggregation(pipe, rng, w.dtype)
        del pipe, cache
    finally:
        torch.cuda.synchronize()
    del table, G
    gc.collect()
    torch.cuda.empty_cache()


# ------------------------------------- misses grouped by host-table region
def test_gather_large_host_table_by_region():
    # A 34 GiB host table (over the size from which misses are read grouped by
    # 2 MB region): with the workspace the gather lists the misses region by
    # region and copies them in that order; rows must equal the table's and
    # the plain row-order gather's, bit for bit, in one part and in two.
    dim, n = 128, (34 << 30) // 512
    t = pinned_table(n, dim, torch.float32)
    tv = t.view(torch.int32)
    tv[:, 0] = torch.arange(n, dtype=torch.int32)  # row i starts with i; pages are zero-filled
    tv[:, dim - 1] = -torch.arange(n, dtype=torch.int32)
    rng = np.random.default_rng(5)
    ranked = rng.choice(n, size=n // 3, replace=False).astype(np.int32)
    cache = sg.sg_cache_build(t, None, sg.SG_F32, n, dim, ranked, len(ranked))
    m = 400_000
    ids = rng.integers(0, n, size=m).astype(np.int32)
    d_ids = dev_i32(ids)
    nbytes = sg.sg_gather_workspace(cache, m)
    assert nbytes > 0
    ws = sg.aligned_workspace(nbytes)
    outs = []
    for workspace in (None, ws):
        out = torch.zeros((m, dim), dtype=torch.float32, device="cuda")
        stats = torch.zeros(2, dtype=torch.int64, device="cuda")
        sg.sg_gather(cache, d_ids, m, None, out, stats, workspace=workspace)
        sg.sg_stream_check()
        hits, misses = stats.cpu().tolist()
        assert hits + misses == m and misses > m // 2
        outs.append(out.view(torch.int32).cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
    assert np.array_equal(outs[1][:, 0], ids) and np.array_equal(outs[1][:, dim - 1], -ids)
    assert not outs[1][:, 1: dim - 1].any()
    # two parts: rows [0, first) then [first, m2) (device counts), the rest untouched
    first, m2 = 150_000, 350_000
    out = torch.full((m, dim), 7.0, device="cuda")
    d_first = torch.tensor([first], dtype=torch.int32, device="cuda")
    d_n = torch.tensor([m2], dtype=torch.int32, device="cuda")
    sg.sg_gather(cache, d_ids, m, d_first, out, workspace=ws)  # n = first
    sg.sg_gather(cache, d_ids, m, d_n, out, d_first=d_first, workspace=ws)
    sg.sg_stream_check()
    got = out.view(torch.int32).cpu().numpy()
    assert np.array_equal(got[:m2], outs[0][:m2])
    assert np.all(out[m2:].cpu().numpy() == 7.0)
    del cache, t
    gc.collect()
