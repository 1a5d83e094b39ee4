"""CPU oracle of the mini-batch pipeline (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA library: the
arithmetic lives in ``oracle.c`` (compiled on first use into ``_oracle.so``),
and this module only marshals numpy arrays into it and lays results out.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into _oracle.so (with OpenMP when available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", _SRC, "-o", tmp]
    r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if r.returncode != 0:
        r = subprocess.run(base, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        vp, i64, i32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_set_threads.restype = None
        lib.orc_set_threads.argtypes = [ctypes.c_int]
        lib.orc_philox4x32_10.restype = None
        lib.orc_philox4x32_10.argtypes = [vp, vp, vp]
        lib.orc_sample_key.restype = ctypes.c_uint32
        lib.orc_sample_key.argtypes = [u64, i32, i32, i64]
        lib.orc_sample_positions.restype = i64
        lib.orc_sample_positions.argtypes = [vp, i32, i32, i32, u64, vp]
        lib.orc_sampler_run.restype = ctypes.c_int
        lib.orc_sampler_run.argtypes = [vp, vp, i64, vp, i32, vp, i32, u64,
                                        vp, i64, vp, vp, vp, vp, i64, vp, vp, vp, i64]
        lib.orc_relabel.restype = i64
        lib.orc_relabel.argtypes = [vp, i64, vp, i64, vp, vp]
        lib.orc_gather.restype = None
        lib.orc_gather.argtypes = [vp, i64, vp, i64, vp]
        lib.orc_aggregate_fwd.restype = None
        lib.orc_aggregate_fwd.argtypes = [vp, vp, i64, vp, ctypes.c_int, i32, vp, vp]
        lib.orc_aggregate_bwd.restype = None
        lib.orc_aggregate_bwd.argtypes = [vp, vp, i64, i64, vp, ctypes.c_int, i32, vp, vp]
        lib.orc_sage_fwd.restype = None
        lib.orc_sage_fwd.argtypes = [vp, vp, i32, vp, i32, i64, i32, i32, vp, vp, vp]
        lib.orc_sage_bwd.restype = None
        lib.orc_sage_bwd.argtypes = [vp, vp, i32, vp, i32, vp, vp, i32, i64, i32, i32, vp, vp, vp, vp, vp]
        lib.orc_access_stats.restype = None
        lib.orc_access_stats.argtypes = [vp, vp, i32, vp, ctypes.c_uint32, vp]
        lib.orc_rank_by_score.restype = None
        lib.orc_rank_by_score.argtypes = [vp, i64, vp, vp]
        lib.orc_graph_renumber.restype = None
        lib.orc_graph_renumber.argtypes = [vp, vp, i64, vp, vp, vp, vp]
        lib.orc_in_degree.restype = None
        lib.orc_in_degree.argtypes = [vp, i64, i64, vp]
        lib.orc_rank_by_score_tie.restype = None
        lib.orc_rank_by_score_tie.argtypes = [vp, vp, i64, vp, vp]
        u32 = ctypes.c_uint32
        lib.orc_dyn_weights.restype = u32
        lib.orc_dyn_weights.argtypes = [u32, i32, vp]
        lib.orc_dyn_accumulate.restype = None
        lib.orc_dyn_accumulate.argtypes = [vp, i64, vp, u32, vp]
        lib.orc_dyn_update.restype = i64
        lib.orc_dyn_update.argtypes = [vp, vp, i64, u32, i64, vp]
        lib.orc_match.restype = i64
        lib.orc_match.argtypes = [vp, i64, vp, i64, i64, vp]
        lib.orc_overlap.restype = ctypes.c_int
        lib.orc_overlap.argtypes = [vp, vp, i32, i64, vp]
        lib.orc_greedy_order.restype = None
        lib.orc_greedy_order.argtypes = [vp, i32, i32, vp]
        _lib = lib
        return lib


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_threads(n: int) -> None:
    _load().orc_set_threads(int(n))


def philox4x32_10(ctr, key):
    """One Philox4x32-10 block: counter (4 words), key (2 words) -> 4 words."""
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, np.uint32)
    _load().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def sample_key(seed: int, hop: int, v: int, j: int) -> int:
    return int(_load().orc_sample_key(seed, hop, v, j))


def sample_positions(indptr: np.ndarray, v: int, fanout: int, hop: int, seed: int) -> np.ndarray:
    """Sampled row positions of node v at a hop, ascending."""
    ip = np.ascontiguousarray(indptr, dtype=np.int64)
    deg = int(ip[v + 1] - ip[v])
    out = np.zeros(max(1, min(deg, fanout)), np.int64)
    c = _load().orc_sample_positions(_p(ip), v, fanout, hop, seed, _p(out))
    if c < 0:
        raise MemoryError("oracle sample: allocation failed")
    return out[:c]


def size_bounds(n_nodes: int, n_seeds: int, fanouts):
    """Upper bounds on |V_h| and E_h before dedup (E_h <= |V_{h-1}| f_h)."""
    nb, eb = [n_seeds], []
    for f in fanouts:
        e = nb[-1] * f
        eb.append(e)
        nb.append(min(n_nodes, nb[-1] + e))
    return nb, eb


class Blocks:
    """Result of one mini-batch: V_H (global IDs, seeds first, V_h a prefix),
    and per hop h = 1..H a block CSR over V_{h-1} x V_h."""

    def __init__(self, unique, hop_off, indptrs, idxs, nbrs, poss):
        self.unique = unique          # int32 [|V_H|]
        self.hop_off = hop_off        # list: |V_0| .. |V_H|
        self.indptr = indptrs         # per hop: int64 [|V_{h-1}|+1]
        self.idx = idxs               # per hop: int32 [E_h] local src IDs
        self.nbr = nbrs               # per hop: int32 [E_h] global src IDs
        self.pos = poss               # per hop: int64 [E_h] row positions

    @property
    def n_hops(self):
        return len(self.indptr)

    def edges(self, h):
        return len(self.idx[h - 1])


def sampler_run(indptr, indices, seeds, fanouts, seed: int) -> Blocks:
    """Multi-hop sampling + relabel of one mini-batch (see oracle.c)."""
    ip = np.ascontiguousarray(indptr, dtype=np.int64)
    ix = np.ascontiguousarray(indices, dtype=np.int32)
    sd = np.ascontiguousarray(seeds, dtype=np.int32)
    fo = np.ascontiguousarray(fanouts, dtype=np.int32)
    n_nodes = len(ip) - 1
    H = len(fo)
    nb, eb = size_bounds(n_nodes, len(sd), [int(f) for f in fo])
    cap_u = nb[-1]
    cap_e = max(1, sum(eb))
    cap_ip = sum(nb[:-1]) + H
    unique = np.zeros(max(1, cap_u), np.int32)
    hop_off = np.zeros(H + 1, np.int64)
    edge_off = np.zeros(H + 1, np.int64)
    ip_off = np.zeros(H + 1, np.int64)
    bip = np.zeros(max(1, cap_ip), np.int64)
    bidx = np.zeros(cap_e, np.int32)
    nbr = np.zeros(cap_e, np.int32)
    pos = np.zeros(cap_e, np.int64)
    rc = _load().orc_sampler_run(_p(ip), _p(ix), n_nodes, _p(sd), len(sd), _p(fo), H, seed,
                                 _p(unique), cap_u, _p(hop_off), _p(edge_off), _p(ip_off), _p(bip), cap_ip,
                                 _p(bidx), _p(nbr), _p(pos), cap_e)
    if rc != 0:
        raise ValueError("oracle sampler_run failed (%d)" % rc)
    indptrs, idxs, nbrs, poss = [], [], [], []
    for h in range(1, H + 1):
        a, b = int(edge_off[h - 1]), int(edge_off[h])
        p0 = int(ip_off[h - 1])
        indptrs.append(bip[p0:p0 + int(hop_off[h - 1]) + 1].copy())
        idxs.append(bidx[a:b].copy())
        nbrs.append(nbr[a:b].copy())
        poss.append(pos[a:b].copy())
    return Blocks(unique[:int(hop_off[H])].copy(), [int(x) for x in hop_off], indptrs, idxs, nbrs, poss)


class SuperBlocks:
    """K mini-batches sampled with one hash seed, laid out back to back:
    sub-batch k's V_H occupies unique[U[k]:U[k+1]]; at hop h its dst rows are
    rows D_h[k] + (local dst) and its src rows S_h[k] + (local src), with D_h[k]
    and S_h[k] the sums of |V_{h-1}| and |V_h| over earlier sub-batches."""

    def __init__(self, runs):
        self.runs = runs
        K = len(runs)
        H = runs[0].n_hops
        self.n_sub = K
        self.counts = np.array([[r.hop_off[h] for h in range(H + 1)] for r in runs], np.int64)  # [K, H+1]
        self.edge_counts = np.array([[r.edges(h) for h in range(1, H + 1)] for r in runs], np.int64)
        self.unique = np.concatenate([r.unique for r in runs]) if K else np.zeros(0, np.int32)
        self.indptr, self.idx = [], []
        for h in range(1, H + 1):
            src_off = np.concatenate([[0], np.cumsum(self.counts[:, h])])
            rows, idx, base = [np.zeros(1, np.int64)], [], 0
            for k, r in enumerate(runs):
                rows.append(r.indptr[h - 1][1:] + base)
                idx.append(r.idx[h - 1].astype(np.int64) + src_off[k])
                base += r.edges(h)
            self.indptr.append(np.concatenate(rows))
            self.idx.append(np.concatenate(idx).astype(np.int32) if idx else np.zeros(0, np.int32))

    def totals(self):
        return self.counts.sum(axis=0)


def super_batch_run(indptr, indices, seed_lists, fanouts, seed: int) -> SuperBlocks:
    """A super-batch is, by definition, its K mini-batches sampled one by one
    with the same hash seed."""
    return SuperBlocks([sampler_run(indptr, indices, s, fanouts, seed) for s in seed_lists])


def relabel(ids, prefix):
    """First-occurrence numbering after an already-numbered prefix."""
    a = np.ascontiguousarray(ids, dtype=np.int32)
    p = np.ascontiguousarray(prefix, dtype=np.int32)
    unique = np.zeros(max(1, len(a) + len(p)), np.int32)
    local = np.zeros(max(1, len(a)), np.int32)
    n = _load().orc_relabel(_p(a), len(a), _p(p), len(p), _p(unique), _p(local))
    if n < 0:
        raise ValueError("oracle relabel: bad input")
    return unique[:n].copy(), local[:len(a)].copy()


def gather(feat: np.ndarray, ids) -> np.ndarray:
    """Row gather: out[i] = feat[ids[i]] byte for byte."""
    f = np.ascontiguousarray(feat)
    i = np.ascontiguousarray(ids, dtype=np.int32)
    out = np.empty((len(i),) + f.shape[1:], dtype=f.dtype)
    row_bytes = f.strides[0] if f.ndim > 1 else f.itemsize
    _load().orc_gather(_p(f), row_bytes, _p(i), len(i), _p(out))
    return out


def _dtype_code(h: np.ndarray) -> int:
    if h.dtype == np.float32:
        return F32
    if h.dtype == np.uint16:
        return BF16
    raise TypeError("features must be float32 or uint16 (bf16 bits)")


def aggregate_fwd(indptr, idx, h: np.ndarray):
    """Mean over each dst row's sampled src rows; returns (out, absmean) as
    float64 [n_dst, dim]."""
    ip = np.ascontiguousarray(indptr, dtype=np.int64)
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    hh = np.ascontiguousarray(h)
    n_dst, dim = len(ip) - 1, hh.shape[1]
    out = np.zeros((n_dst, dim), np.float64)
    am = np.zeros((n_dst, dim), np.float64)
    _load().orc_aggregate_fwd(_p(ip), _p(ix), n_dst, _p(hh), _dtype_code(hh), dim, _p(out), _p(am))
    return out, am


def aggregate_bwd(indptr, idx, n_src: int, gdst: np.ndarray):
    """Transpose of the mean map; returns (gsrc, absmean) as float64 [n_src, dim]."""
    ip = np.ascontiguousarray(indptr, dtype=np.int64)
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    g = np.ascontiguousarray(gdst)
    n_dst, dim = len(ip) - 1, g.shape[1]
    out = np.zeros((n_src, dim), np.float64)
    am = np.zeros((n_src, dim), np.float64)
    _load().orc_aggregate_bwd(_p(ip), _p(ix), n_dst, n_src, _p(g), _dtype_code(g), dim, _p(out), _p(am))
    return out, am


def _feat(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    _dtype_code(a)
    return a


def sage_fwd(h: np.ndarray, m: np.ndarray, W: np.ndarray):
    """SAGE UPDATE forward: y = [h | m] W^T, out = ReLU(y).  h, m: [n, d]
    (float32 or bf16 bits, the same type); W: [d_out, 2d] (float32 or bf16
    bits).  Returns (y, out, absum) as float64 [n, d_out]."""
    hh, mm, ww = _feat(h), _feat(m), _feat(W)
    if hh.shape != mm.shape or hh.dtype != mm.dtype:
        raise ValueError("sage_fwd: h and m differ in shape or type")
    n, d = hh.shape
    d_out = ww.shape[0]
    if ww.shape[1] != 2 * d:
        raise ValueError("sage_fwd: W must have 2 * d columns")
    y = np.zeros((n, d_out), np.float64)
    out = np.zeros((n, d_out), np.float64)
    am = np.zeros((n, d_out), np.float64)
    _load().orc_sage_fwd(_p(hh), _p(mm), _dtype_code(hh), _p(ww), _dtype_code(ww), n, d, d_out, _p(y), _p(out), _p(am))
    return y, out, am


def sage_bwd(h: np.ndarray, m: np.ndarray, W: np.ndarray, y: np.ndarray, g: np.ndarray):
    """Backward of sage_fwd for g = dL/dout [n, d_out] (float32 or bf16 bits)
    and the forward's y (float64).  Returns (dW, absum_dW, dh, dm, absum_dz):
    dW [d_out, 2d], dh and dm [n, d], absum_dz [n, 2d], all float64."""
    hh, mm, ww, gg = _feat(h), _feat(m), _feat(W), _feat(g)
    yy = np.ascontiguousarray(y, dtype=np.float64)
    n, d = hh.shape
    d_out = ww.shape[0]
    dW = np.zeros((d_out, 2 * d), np.float64)
    am_w = np.zeros((d_out, 2 * d), np.float64)
    dh = np.zeros((n, d), np.float64)
    dm = np.zeros((n, d), np.float64)
    am_z = np.zeros((n, 2 * d), np.float64)
    _load().orc_sage_bwd(_p(hh), _p(mm), _dtype_code(hh), _p(ww), _dtype_code(ww), _p(yy), _p(gg), _dtype_code(gg),
                         n, d, d_out, _p(dW), _p(am_w), _p(dh), _p(dm), _p(am_z))
    return dW, am_w, dh, dm, am_z


def access_stats(blocks: Blocks, omega, w_in: int, score: np.ndarray) -> None:
    """Adds the full-link access statistics (Eq. (4)) of one mini-batch to
    score (uint32 [n_nodes], updated in place)."""
    assert score.dtype == np.uint32 and score.flags.c_contiguous
    om = np.ascontiguousarray(omega, dtype=np.uint32)
    if len(om) != blocks.n_hops:
        raise ValueError("access_stats: one weight per hop")
    hop = np.ascontiguousarray(blocks.hop_off, dtype=np.int64)
    un = np.ascontiguousarray(blocks.unique, dtype=np.int32)
    _load().orc_access_stats(_p(un), _p(hop), blocks.n_hops, _p(om), int(w_in), _p(score))


def rank_by_score(score: np.ndarray, tie: np.ndarray = None):
    """(order, rank_of): nodes by descending score, then (when given)
    descending tie key, then ascending ID."""
    sc = np.ascontiguousarray(score, dtype=np.uint32)
    n = len(sc)
    order = np.zeros(max(1, n), np.int32)
    rank_of = np.zeros(max(1, n), np.int32)
    if tie is None:
        _load().orc_rank_by_score(_p(sc), n, _p(order), _p(rank_of))
    else:
        tk = np.ascontiguousarray(tie, dtype=np.uint32)
        _load().orc_rank_by_score_tie(_p(sc), _p(tk), n, _p(order), _p(rank_of))
    return order[:n], rank_of[:n]


def in_degree(indices, n_nodes: int) -> np.ndarray:
    """uint32 [n_nodes]: how many CSR positions name each node."""
    ix = np.ascontiguousarray(indices, dtype=np.int32)
    deg = np.zeros(max(1, n_nodes), np.uint32)
    _load().orc_in_degree(_p(ix), len(ix), int(n_nodes), _p(deg))
    return deg[:n_nodes]


def graph_renumber(indptr, indices, order, rank_of):
    """The CSR with node order[r] renamed r; returns (indptr int64, indices int32)."""
    ip = np.ascontiguousarray(indptr, dtype=np.int64)
    ix = np.ascontiguousarray(indices, dtype=np.int32)
    od = np.ascontiguousarray(order, dtype=np.int32)
    rk = np.ascontiguousarray(rank_of, dtype=np.int32)
    n = len(ip) - 1
    new_ip = np.zeros(n + 1, np.int64)
    new_ix = np.zeros(max(1, len(ix)), np.int32)
    _load().orc_graph_renumber(_p(ip), _p(ix), n, _p(od), _p(rk), _p(new_ip), _p(new_ix))
    return new_ip, new_ix[: len(ix)]


class DynCache:
    """The dynamic cache's scores (Eq. (5)-(6), windowed fixed-point reading;
    see oracle.c): gamma = g / 2^16, windows of T batches, k_dyn nodes."""

    def __init__(self, n_nodes: int, g: int, T: int, k_dyn: int, static_cached: np.ndarray):
        self.n, self.T, self.k = int(n_nodes), int(T), int(k_dyn)
        self.W = np.zeros(self.T, np.uint32)
        self.G = int(_load().orc_dyn_weights(int(g), self.T, _p(self.W)))
        self.S = np.zeros(self.n, np.uint32)
        self.A = np.zeros(self.n, np.uint32)
        self.cached = np.ascontiguousarray(static_cached, dtype=np.uint8)
        self.j = 0  # batch within the window

    def batch(self, unique) -> None:
        """Adds one batch's nodes (its V_H); closes the window after T."""
        u = np.ascontiguousarray(unique, dtype=np.int32)
        _load().orc_dyn_accumulate(_p(u), len(u), _p(self.cached), int(self.W[self.j]), _p(self.A))
        self.j += 1

    def update(self) -> np.ndarray:
        """End of a window: the new dynamic set (Eq. (6))."""
        dyn = np.zeros(max(1, self.k), np.int32)
        c = _load().orc_dyn_update(_p(self.S), _p(self.A), self.n, self.G, self.k, _p(dyn))
        if c < 0:
            raise MemoryError("oracle dyn update")
        self.j = 0
        return dyn[:c].copy()


def match(prev, cur, n_nodes: int):
    """Position of each cur ID in prev, or -1 (prev: distinct IDs)."""
    p = np.ascontiguousarray(prev, dtype=np.int32)
    c = np.ascontiguousarray(cur, dtype=np.int32)
    pos = np.zeros(max(1, len(c)), np.int32)
    m = _load().orc_match(_p(p), len(p), _p(c), len(c), int(n_nodes), _p(pos))
    if m < 0:
        raise MemoryError("oracle match")
    return pos[: len(c)]


def overlap(lists, n_nodes: int) -> np.ndarray:
    """G x G matrix of |list a intersect list b| (lists of distinct IDs)."""
    off = np.concatenate([[0], np.cumsum([len(x) for x in lists])]).astype(np.int64)
    ids = np.ascontiguousarray(np.concatenate(lists) if len(lists) else np.zeros(0), dtype=np.int32)
    G = len(lists)
    O = np.zeros((G, G), np.int64)
    if _load().orc_overlap(_p(ids), _p(off), G, int(n_nodes), _p(O)) != 0:
        raise MemoryError("oracle overlap")
    return O


def greedy_order(O: np.ndarray, first: int = 0) -> np.ndarray:
    """Nearest-overlap-first order of G batches from `first` (ties: lowest)."""
    OO = np.ascontiguousarray(O, dtype=np.int64)
    G = OO.shape[0]
    if G > 1024:
        raise ValueError("greedy_order: at most 1024 batches")
    order = np.zeros(G, np.int32)
    _load().orc_greedy_order(_p(OO), G, int(first), _p(order))
    return order


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
