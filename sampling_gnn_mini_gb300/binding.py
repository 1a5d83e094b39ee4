"""ctypes binding of ``libsg.so`` (declared in include/sg.h).

Argument marshalling only: every function here hands raw device pointers,
sizes and the current CUDA stream to the C ABI function of the same name;
all computation runs in the library's kernels.  PyTorch is used for device
and pinned memory and for streams.  If the library is missing or was not
built for this machine, loading fails loudly: there is no other code path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np
import torch

from . import build as _build

SG_OK = 0
SG_ERR_INVALID_ARG = 1
SG_ERR_INVALID_INDEX = 2
SG_ERR_CAPACITY = 3
SG_ERR_OOM = 4
SG_ERR_CUDA = 5
SG_ERR_TIMEOUT = 6
SG_ERR_UNSUPPORTED = 7
SG_F32 = 0
SG_BF16 = 1
SG_MAX_HOPS = 8
SG_MAX_SUB = 64
SG_MAX_FANOUT = 256

_STATUS_NAMES = {0: "SG_OK", 1: "SG_ERR_INVALID_ARG", 2: "SG_ERR_INVALID_INDEX", 3: "SG_ERR_CAPACITY",
                 4: "SG_ERR_OOM", 5: "SG_ERR_CUDA", 6: "SG_ERR_TIMEOUT", 7: "SG_ERR_UNSUPPORTED"}

# every symbol include/sg.h declares
EXPORTS = ["sg_version", "sg_last_error", "sg_stream_check", "sg_graph_load", "sg_graph_destroy", "sg_graph_info",
           "sg_sampler_bounds", "sg_sampler_run", "sg_relabel_workspace", "sg_relabel", "sg_cache_build",
           "sg_cache_destroy", "sg_cache_info", "sg_gather", "sg_aggregate_fwd", "sg_aggregate_bwd_workspace",
           "sg_aggregate_bwd", "sg_read_probe", "sg_hash_probe", "sg_relabel_noalloc", "sg_transpose_workspace",
           "sg_transpose_blocks", "sg_aggregate_bwd_t", "sg_sampler_workspace_init", "sg_gather_workspace",
           "sg_sage_fwd", "sg_sage_bwd", "sg_sage_bwd_workspace", "sg_wait_probe", "sg_wait_probe_workspace",
           "sg_access_stats", "sg_rank_workspace", "sg_rank_by_score", "sg_graph_renumber", "sg_graph_copy_out",
           "sg_dyn_cache_create", "sg_dyn_cache_batch", "sg_dyn_cache_info", "sg_gather_reuse", "sg_match",
           "sg_overlap", "sg_greedy_order", "sg_graph_in_degree"]


class SgError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (_STATUS_NAMES.get(status, str(status)), message))
        self.status = status


class _Bounds(ctypes.Structure):
    _fields_ = [("max_nodes", ctypes.c_int64 * (SG_MAX_HOPS + 1)),
                ("max_edges", ctypes.c_int64 * SG_MAX_HOPS),
                ("counts_len", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_size_t)]


class _Transposed(ctypes.Structure):
    _fields_ = [("tptr", ctypes.c_void_p * SG_MAX_HOPS),
                ("tdst", ctypes.c_void_p * SG_MAX_HOPS),
                ("tw", ctypes.c_void_p * SG_MAX_HOPS)]


class _Blocks(ctypes.Structure):
    _fields_ = [("unique", ctypes.c_void_p),
                ("counts", ctypes.c_void_p),
                ("indptr", ctypes.c_void_p * SG_MAX_HOPS),
                ("idx", ctypes.c_void_p * SG_MAX_HOPS)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Loads libsg.so (building it first if it is missing or stale and nvcc
    is available).  Raises if it cannot be loaded."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError("libsg.so is missing; run sampling_gnn_mini_gb300.build.build()")
        lib = ctypes.CDLL(_build.LIB)
        vp, i32, i64, u64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
        sig = {
            "sg_version": (i32, []),
            "sg_last_error": (i32, [ctypes.c_char_p, sz]),
            "sg_stream_check": (i32, [vp]),
            "sg_graph_load": (i32, [vp, i32, vp, i64, i64, ctypes.POINTER(vp)]),
            "sg_graph_destroy": (i32, [vp]),
            "sg_graph_info": (i32, [vp, vp, vp, vp, vp]),
            "sg_sampler_bounds": (i32, [vp, i32, vp, i32, vp, i32, ctypes.POINTER(_Bounds)]),
            "sg_sampler_run": (i32, [vp, vp, i32, vp, i32, vp, i32, u64, vp, vp, sz, ctypes.POINTER(_Blocks), vp, vp]),
            "sg_relabel_workspace": (sz, [i64, i64]),
            "sg_relabel": (i32, [vp, i64, vp, i64, vp, vp, vp, vp, sz, vp]),
            "sg_cache_build": (i32, [vp, vp, i32, i64, i32, vp, i64, ctypes.POINTER(vp), vp]),
            "sg_cache_destroy": (i32, [vp]),
            "sg_cache_info": (i32, [vp, vp, vp, vp, vp, vp]),
            "sg_gather": (i32, [vp, vp, i64, vp, vp, vp, vp, vp, sz, vp]),
            "sg_gather_workspace": (sz, [vp, i64]),
            "sg_sage_fwd": (i32, [vp, vp, vp, i32, i32, vp, i32, i32, vp, vp, vp]),
            "sg_sage_bwd": (i32, [vp, vp, vp, i32, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]),
            "sg_sage_bwd_workspace": (sz, [i32, i32, i32]),
            "sg_aggregate_fwd": (i32, [vp, vp, i32, i32, vp, vp, i32, i32, vp, i32, vp]),
            "sg_aggregate_bwd_workspace": (sz, [i32, i32, i64]),
            "sg_aggregate_bwd": (i32, [vp, vp, i32, i32, i64, vp, vp, i32, i32, vp, i32, vp, sz, vp]),
            "sg_read_probe": (i32, [vp, i64, vp, vp]),
            "sg_hash_probe": (i32, [i64, u64, vp, vp]),
            "sg_relabel_noalloc": (i32, [vp, i64, vp, i64, vp, vp, vp, vp]),
            "sg_transpose_workspace": (sz, [vp, vp, i32]),
            "sg_transpose_blocks": (i32, [ctypes.POINTER(_Blocks), vp, vp, i32, ctypes.POINTER(_Transposed), vp, sz,
                                          vp]),
            "sg_aggregate_bwd_t": (i32, [vp, vp, vp, i32, i32, vp, vp, i32, i32, vp, i32, vp]),
            "sg_sampler_workspace_init": (i32, [vp, i32, vp, i32, vp, i32, vp, sz, vp]),
            "sg_wait_probe": (i32, [i32, i32, i32, vp, sz, vp, vp]),
            "sg_wait_probe_workspace": (sz, [i32]),
            "sg_access_stats": (i32, [ctypes.POINTER(_Blocks), i64, i32, i32, vp, ctypes.c_uint32, vp, i64, vp]),
            "sg_rank_workspace": (sz, [i64]),
            "sg_rank_by_score": (i32, [vp, vp, i64, vp, vp, vp, sz, vp]),
            "sg_graph_in_degree": (i32, [vp, vp, vp]),
            "sg_graph_renumber": (i32, [vp, vp, vp, ctypes.POINTER(vp), vp]),
            "sg_graph_copy_out": (i32, [vp, vp, vp]),
            "sg_dyn_cache_create": (i32, [vp, i64, ctypes.c_uint32, i32, vp]),
            "sg_dyn_cache_batch": (i32, [vp, vp, i64, vp, vp]),
            "sg_dyn_cache_info": (i32, [vp, vp, vp, vp, vp, vp]),
            "sg_gather_reuse": (i32, [vp, vp, i64, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "sg_match": (i32, [vp, i64, vp, vp, i64, vp, vp, i64, vp, vp, vp]),
            "sg_overlap": (i32, [vp, vp, i32, vp, i64, vp, vp]),
            "sg_greedy_order": (i32, [vp, i32, i32, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


def exported_symbols() -> List[str]:
    lib = load()
    return [n for n in EXPORTS if hasattr(lib, n)]


def sg_last_error() -> str:
    buf = ctypes.create_string_buffer(1024)
    load().sg_last_error(buf, 1024)
    return buf.value.decode(errors="replace")


def _check(st: int) -> None:
    if st != SG_OK:
        raise SgError(st, sg_last_error())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr()
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return int(t)


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def sg_version() -> int:
    return int(load().sg_version())


def sg_stream_check(stream=None) -> None:
    _check(load().sg_stream_check(_stream(stream)))


# ------------------------------------------------------------------- graph
class Graph:
    """Handle of a CSR graph loaded into HBM (freed with the object)."""

    def __init__(self, handle):
        self._h = handle
        n, m, ob, md = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int64()
        _check(load().sg_graph_info(handle, ctypes.byref(n), ctypes.byref(m), ctypes.byref(ob), ctypes.byref(md)))
        self.n_nodes, self.n_edges, self.offset_bits, self.max_degree = n.value, m.value, ob.value, md.value

    @property
    def handle(self):
        return self._h

    def close(self):
        h, self._h = self._h, None
        if h and _lib is not None:
            _lib.sg_graph_destroy(h)

    def __del__(self):
        self.close()


def sg_graph_load(indptr: np.ndarray, indices: np.ndarray, offset_bits: Optional[int] = None) -> Graph:
    """Copies a host CSR (numpy) into HBM.  offset_bits defaults to the
    width of indptr's dtype."""
    indptr = np.ascontiguousarray(indptr)
    if offset_bits is None:
        offset_bits = 64 if indptr.dtype == np.int64 else 32
    indptr = np.ascontiguousarray(indptr, dtype=np.int64 if offset_bits == 64 else np.int32)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    out = ctypes.c_void_p()
    _check(load().sg_graph_load(indptr.ctypes.data, offset_bits, indices.ctypes.data if len(indices) else None,
                                len(indptr) - 1, len(indices), ctypes.byref(out)))
    return Graph(out.value)


def sg_graph_renumber(graph: Graph, order: torch.Tensor, rank_of: torch.Tensor, stream=None) -> Graph:
    """The graph with node order[r] renamed r (device int32 permutations;
    see include/sg.h)."""
    for t in (order, rank_of):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous() or t.numel() != graph.n_nodes:
            raise SgError(SG_ERR_INVALID_ARG, "sg_graph_renumber: order and rank_of must be contiguous int32 "
                                              "device tensors of n_nodes entries")
    out = ctypes.c_void_p()
    _check(load().sg_graph_renumber(graph.handle, order.data_ptr(), rank_of.data_ptr(), ctypes.byref(out),
                                    _stream(stream)))
    return Graph(out.value)


def sg_graph_copy_out(graph: Graph):
    """(indptr, indices) of a loaded graph as host numpy arrays."""
    ip = np.empty(graph.n_nodes + 1, dtype=np.int64 if graph.offset_bits == 64 else np.int32)
    ix = np.empty(max(1, graph.n_edges), dtype=np.int32)
    _check(load().sg_graph_copy_out(graph.handle, ip.ctypes.data, ix.ctypes.data))
    return ip, ix[: graph.n_edges]


# ---------------------------------------------------------------- sampling
@dataclass
class Bounds:
    max_nodes: List[int]
    max_edges: List[int]
    counts_len: int
    workspace_bytes: int


def sg_sampler_bounds(graph: Graph, n_seeds: int, fanouts: Sequence[int], batch_ptr: Optional[Sequence[int]] = None) -> Bounds:
    fo = np.ascontiguousarray(fanouts, dtype=np.int32)
    bp = None if batch_ptr is None else np.ascontiguousarray(batch_ptr, dtype=np.int32)
    b = _Bounds()
    _check(load().sg_sampler_bounds(graph.handle, int(n_seeds), None if bp is None else bp.ctypes.data,
                                    1 if bp is None else len(bp) - 1, fo.ctypes.data, len(fo), ctypes.byref(b)))
    H = len(fo)
    return Bounds([int(b.max_nodes[h]) for h in range(H + 1)], [int(b.max_edges[h]) for h in range(H)],
                  int(b.counts_len), int(b.workspace_bytes))


def _aligned_bytes(nbytes: int, device, align: int = 256) -> torch.Tensor:
    raw = torch.empty(int(nbytes) + align, dtype=torch.uint8, device=device)
    off = (-raw.data_ptr()) % align
    return raw[off:off + int(nbytes)]


class SampleBuffers:
    """Caller-owned device arrays for sg_sampler_run, sized by the bounds.
    With the graph and sampling shape given, the workspace is also prepared
    (sg_sampler_workspace_init); otherwise call init_workspace() before use."""

    def __init__(self, bounds: Bounds, device="cuda", graph=None, n_seeds=None, fanouts=None, batch_ptr=None):
        self.bounds = bounds
        H = len(bounds.max_edges)
        self.n_hops = H
        self.unique = torch.empty(max(1, bounds.max_nodes[H]), dtype=torch.int32, device=device)
        self.counts = torch.zeros(bounds.counts_len, dtype=torch.int32, device=device)
        self.indptr = [torch.empty(bounds.max_nodes[h] + 1, dtype=torch.int32, device=device) for h in range(H)]
        self.idx = [torch.empty(max(1, bounds.max_edges[h]), dtype=torch.int32, device=device) for h in range(H)]
        self.workspace = _aligned_bytes(max(256, bounds.workspace_bytes), device)
        self._blocks = _Blocks()
        self._blocks.unique = self.unique.data_ptr()
        self._blocks.counts = self.counts.data_ptr()
        for h in range(H):
            self._blocks.indptr[h] = self.indptr[h].data_ptr()
            self._blocks.idx[h] = self.idx[h].data_ptr()
        if graph is not None:
            self.init_workspace(graph, n_seeds, fanouts, batch_ptr)

    def init_workspace(self, graph, n_seeds, fanouts, batch_ptr=None, stream=None) -> None:
        fo = np.ascontiguousarray(fanouts, dtype=np.int32)
        bp = None if batch_ptr is None else np.ascontiguousarray(batch_ptr, dtype=np.int32)
        _check(load().sg_sampler_workspace_init(graph.handle, int(n_seeds), None if bp is None else bp.ctypes.data,
                                                1 if bp is None else len(bp) - 1, fo.ctypes.data, len(fo),
                                                self.workspace.data_ptr(), self.workspace.numel(), _stream(stream)))

    def dims(self, h: int) -> torch.Tensor:
        """Device int32[2] = {|V_{h-1}|, |V_h|} totals for the hop-h block."""
        return self.counts[h - 1:h + 1]


def sg_sampler_run(graph: Graph, seeds: torch.Tensor, fanouts: Sequence[int], seed: int, buffers: SampleBuffers,
                   batch_ptr: Optional[Sequence[int]] = None, stream=None, d_seed: Optional[torch.Tensor] = None,
                   hop_events: Optional[Sequence[Optional[torch.cuda.Event]]] = None) -> None:
    """hop_events: one entry per hop (a CUDA event that has been recorded at
    least once, so that it exists, or None); see sg.h."""
    fo = np.ascontiguousarray(fanouts, dtype=np.int32)
    bp = None if batch_ptr is None else np.ascontiguousarray(batch_ptr, dtype=np.int32)
    assert seeds.dtype == torch.int32 and seeds.is_cuda and seeds.is_contiguous()
    evs = None
    if hop_events is not None:
        if len(hop_events) != len(fo):
            raise ValueError("sg_sampler_run: hop_events needs one entry per hop")
        evs = (ctypes.c_void_p * len(fo))(*[None if e is None else e.cuda_event for e in hop_events])
    _check(load().sg_sampler_run(graph.handle, seeds.data_ptr(), int(seeds.numel()),
                                 None if bp is None else bp.ctypes.data, 1 if bp is None else len(bp) - 1,
                                 fo.ctypes.data, len(fo), ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), _ptr(d_seed),
                                 buffers.workspace.data_ptr(), buffers.workspace.numel(),
                                 ctypes.byref(buffers._blocks), evs, _stream(stream)))


def sg_access_stats(buffers: "SampleBuffers", omega: Sequence[int], w_in: int, score: torch.Tensor, n_sub: int = 1,
                    stream=None) -> None:
    """Adds the full-link access statistics (Eq. (4)) of the sampler output in
    buffers to score (device uint32 / int32 [n_nodes]); see include/sg.h."""
    om = np.ascontiguousarray(omega, dtype=np.uint32)
    if len(om) != buffers.n_hops:
        raise SgError(SG_ERR_INVALID_ARG, "sg_access_stats: one weight per hop")
    if score.element_size() != 4 or score.is_floating_point() or not score.is_cuda or not score.is_contiguous():
        raise SgError(SG_ERR_INVALID_ARG, "sg_access_stats: score must be a 32-bit device tensor")
    _check(load().sg_access_stats(ctypes.byref(buffers._blocks), buffers.unique.numel(), buffers.n_hops, int(n_sub),
                                  om.ctypes.data, int(w_in), score.data_ptr(), int(score.numel()), _stream(stream)))


def sg_rank_by_score(score: torch.Tensor, tie: Optional[torch.Tensor] = None, stream=None):
    """(order, rank_of) device int32 tensors: nodes by descending score (the
    32-bit unsigned contents of score), then descending tie key (when
    given), then ascending ID."""
    lib = load()
    n = int(score.numel())
    nbytes = int(lib.sg_rank_workspace(n))
    if nbytes == 0:
        raise SgError(SG_ERR_INVALID_ARG, "sg_rank_by_score: bad size")
    order = torch.empty(n, dtype=torch.int32, device=score.device)
    rank_of = torch.empty(n, dtype=torch.int32, device=score.device)
    ws = _aligned_bytes(nbytes, score.device)
    if tie is not None and (tie.numel() != n or tie.element_size() != 4 or not tie.is_cuda):
        raise SgError(SG_ERR_INVALID_ARG, "sg_rank_by_score: tie must be a 32-bit device tensor like score")
    _check(lib.sg_rank_by_score(score.data_ptr(), _ptr(tie), n, order.data_ptr(), rank_of.data_ptr(), ws.data_ptr(),
                                ws.numel(), _stream(stream)))
    return order, rank_of


def sg_graph_in_degree(graph: Graph, stream=None) -> torch.Tensor:
    """Device int32 [n_nodes] (uint32 contents): the in-degree of each node."""
    deg = torch.empty(graph.n_nodes, dtype=torch.int32, device="cuda")
    _check(load().sg_graph_in_degree(graph.handle, deg.data_ptr(), _stream(stream)))
    return deg


def sg_relabel(ids: torch.Tensor, prefix: torch.Tensor, stream=None):
    """Returns (unique, local, n_unique) device tensors; unique has room for
    len(prefix) + len(ids) entries, of which the first n_unique are used."""
    lib = load()
    n_ids, n_pre = int(ids.numel()), int(prefix.numel())
    dev = ids.device if n_ids else prefix.device
    unique = torch.empty(max(1, n_ids + n_pre), dtype=torch.int32, device=dev)
    local = torch.empty(max(1, n_ids), dtype=torch.int32, device=dev)
    n_unique = torch.zeros(1, dtype=torch.int32, device=dev)
    wsb = lib.sg_relabel_workspace(n_pre, n_ids)
    if wsb == 0:
        raise SgError(SG_ERR_INVALID_ARG, "sg_relabel: sizes out of range")
    ws = _aligned_bytes(wsb, dev)
    _check(lib.sg_relabel(ids.data_ptr() if n_ids else None, n_ids, prefix.data_ptr() if n_pre else None, n_pre,
                          unique.data_ptr(), local.data_ptr(), n_unique.data_ptr(), ws.data_ptr(), ws.numel(),
                          _stream(stream)))
    return unique, local[:n_ids], n_unique


# ------------------------------------------------------------------- cache
class Cache:
    """Handle of the HBM feature cache (freed with the object).  Keeps a
    reference to the host table, which must outlive the cache."""

    def __init__(self, handle, host_ref):
        self._h = handle
        self._host_ref = host_ref
        n, d, dt, c = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
        _check(load().sg_cache_info(handle, ctypes.byref(n), ctypes.byref(d), ctypes.byref(dt), ctypes.byref(c), None))
        self.n_nodes, self.dim, self.dtype, self.n_cache = n.value, d.value, dt.value, c.value

    @property
    def handle(self):
        return self._h

    def slot_of_ptr(self) -> int:
        p = ctypes.c_void_p()
        _check(load().sg_cache_info(self._h, None, None, None, None, ctypes.byref(p)))
        return p.value

    def close(self):
        h, self._h = self._h, None
        if h and _lib is not None:
            _lib.sg_cache_destroy(h)

    def __del__(self):
        self.close()


def sg_cache_build(h_feat: Optional[torch.Tensor], d_feat: Optional[torch.Tensor], dtype: int, n_nodes: int, dim: int,
                   ranked: Optional[np.ndarray], n_cache: int, stream=None) -> Cache:
    rk = None if ranked is None else np.ascontiguousarray(ranked, dtype=np.int32)
    out = ctypes.c_void_p()
    _check(load().sg_cache_build(_ptr(h_feat), _ptr(d_feat), int(dtype), int(n_nodes), int(dim),
                                 None if rk is None else rk.ctypes.data, int(n_cache), ctypes.byref(out),
                                 _stream(stream)))
    return Cache(out.value, h_feat)


def sg_dyn_cache_create(cache: Cache, k_dyn: int, gamma_q16: int, t_update: int, stream=None) -> None:
    """Attaches the bounded dynamic cache (Eq. (5)-(6)) to cache; see sg.h."""
    _check(load().sg_dyn_cache_create(cache.handle, int(k_dyn), int(gamma_q16), int(t_update), _stream(stream)))


def sg_dyn_cache_batch(cache: Cache, ids: torch.Tensor, n_cap: int, d_n: Optional[torch.Tensor] = None,
                       stream=None) -> None:
    """Adds one batch's nodes to the dynamic cache's scores (and updates the
    set at the end of a window)."""
    _check(load().sg_dyn_cache_batch(cache.handle, ids.data_ptr() if n_cap else None, int(n_cap), _ptr(d_n),
                                     _stream(stream)))


def sg_dyn_cache_state(cache: Cache, stream=None):
    """(k_dyn, window position, scores, node per slot), the last two as host
    numpy copies (synchronises the stream)."""
    lib = load()
    k, j = ctypes.c_int64(), ctypes.c_int32()
    _check(lib.sg_dyn_cache_info(cache.handle, ctypes.byref(k), ctypes.byref(j), None, None, _stream(stream)))
    S = np.empty(cache.n_nodes, np.uint32)
    nodes = np.empty(max(1, k.value), np.int32)
    _check(lib.sg_dyn_cache_info(cache.handle, None, None, S.ctypes.data, nodes.ctypes.data, _stream(stream)))
    return k.value, j.value, S, nodes[: k.value]


def sg_gather_workspace(cache: Cache, n_cap: int) -> int:
    return int(load().sg_gather_workspace(cache.handle, int(n_cap)))


def sg_gather(cache: Cache, ids: torch.Tensor, n_cap: int, d_n: Optional[torch.Tensor], out: torch.Tensor,
              stats: Optional[torch.Tensor] = None, stream=None, d_first: Optional[torch.Tensor] = None,
              workspace: Optional[torch.Tensor] = None) -> None:
    _check(load().sg_gather(cache.handle, ids.data_ptr(), int(n_cap), _ptr(d_n), _ptr(d_first), out.data_ptr(),
                            _ptr(stats), _ptr(workspace), 0 if workspace is None else workspace.numel(),
                            _stream(stream)))


def sg_gather_reuse(cache: Cache, ids: torch.Tensor, n_cap: int, d_n: Optional[torch.Tensor], pos: torch.Tensor,
                    prev_rows: torch.Tensor, out: torch.Tensor, stats: Optional[torch.Tensor] = None,
                    reused: Optional[torch.Tensor] = None, stream=None, d_first: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None) -> None:
    """sg_gather that copies matched rows (pos >= 0) from the previous
    batch's rows (see sg.h)."""
    _check(load().sg_gather_reuse(cache.handle, ids.data_ptr(), int(n_cap), _ptr(d_n), _ptr(d_first), pos.data_ptr(),
                                  prev_rows.data_ptr(), out.data_ptr(), _ptr(stats), _ptr(reused), _ptr(workspace),
                                  0 if workspace is None else workspace.numel(), _stream(stream)))


def sg_match(prev: torch.Tensor, prev_cap: int, prev_n: Optional[torch.Tensor], cur: torch.Tensor, cur_cap: int,
             cur_n: Optional[torch.Tensor], match_map: torch.Tensor, pos: torch.Tensor,
             matched: Optional[torch.Tensor] = None, stream=None) -> None:
    """pos[j] = position of cur[j] in prev or -1; match_map: int32 [n_nodes]
    all -1 (left so); see sg.h."""
    _check(load().sg_match(prev.data_ptr() if prev_cap else None, int(prev_cap), _ptr(prev_n),
                           cur.data_ptr() if cur_cap else None, int(cur_cap), _ptr(cur_n), match_map.data_ptr(),
                           int(match_map.numel()), pos.data_ptr() if cur_cap else None, _ptr(matched),
                           _stream(stream)))


def sg_overlap(ids: torch.Tensor, offsets: Sequence[int], mask: torch.Tensor, stream=None) -> torch.Tensor:
    """G x G overlap matrix (device int64) of the lists ids[off[a]:off[a+1]];
    mask: int32/uint32 [n_nodes] all zero (left so)."""
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    G = len(off) - 1
    out = torch.empty((G, G), dtype=torch.int64, device=mask.device)
    _check(load().sg_overlap(ids.data_ptr() if off[-1] else None, off.ctypes.data, G, mask.data_ptr(),
                             int(mask.numel()), out.data_ptr(), _stream(stream)))
    return out


def sg_greedy_order(overlap: np.ndarray, first: int = 0) -> np.ndarray:
    """Nearest-overlap-first order of a group (host)."""
    O = np.ascontiguousarray(overlap, dtype=np.uint64)
    G = O.shape[0]
    order = np.empty(G, np.int32)
    _check(load().sg_greedy_order(O.ctypes.data, G, int(first), order.ctypes.data))
    return order


def sg_sage_fwd(h: torch.Tensor, m: torch.Tensor, W: torch.Tensor, n_cap: int, d_n: Optional[torch.Tensor],
                out: torch.Tensor, y: Optional[torch.Tensor] = None, stream=None) -> None:
    """out = ReLU([h | m] W^T) for the first n rows (see sg.h)."""
    _check(load().sg_sage_fwd(h.data_ptr(), m.data_ptr(), W.data_ptr(), _dtype_code(h), int(n_cap), _ptr(d_n),
                              int(h.shape[1]), int(W.shape[0]), out.data_ptr(), _ptr(y), _stream(stream)))


def sg_sage_bwd_workspace(n_cap: int, dim: int, dtype: int) -> int:
    return int(load().sg_sage_bwd_workspace(int(n_cap), int(dim), int(dtype)))


def sg_sage_bwd(h: torch.Tensor, m: torch.Tensor, W: torch.Tensor, n_cap: int, d_n: Optional[torch.Tensor],
                y: torch.Tensor, g: torch.Tensor, dW: torch.Tensor, dh: torch.Tensor, dm: torch.Tensor,
                workspace: torch.Tensor, stream=None) -> None:
    """Backward of sg_sage_fwd (see sg.h)."""
    _check(load().sg_sage_bwd(h.data_ptr(), m.data_ptr(), W.data_ptr(), _dtype_code(h), int(n_cap), _ptr(d_n),
                              int(h.shape[1]), int(W.shape[0]), y.data_ptr(), g.data_ptr(), dW.data_ptr(),
                              dh.data_ptr(), dm.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream(stream)))


# --------------------------------------------------------------- aggregate
def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SG_F32
    if t.dtype in (torch.bfloat16, torch.uint16, torch.int16):
        return SG_BF16
    raise TypeError("feature tensors must be float32 or bfloat16")


def sg_aggregate_fwd(indptr: torch.Tensor, idx: torch.Tensor, n_dst_cap: int, n_src_cap: int,
                     dims: Optional[torch.Tensor], h: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    dim = h.shape[1]
    _check(load().sg_aggregate_fwd(indptr.data_ptr(), idx.data_ptr(), int(n_dst_cap), int(n_src_cap), _ptr(dims),
                                   h.data_ptr(), _dtype_code(h), int(dim), out.data_ptr(), _dtype_code(out),
                                   _stream(stream)))


def sg_aggregate_bwd_workspace(n_dst_cap: int, n_src_cap: int, n_edge_cap: int) -> int:
    return int(load().sg_aggregate_bwd_workspace(int(n_dst_cap), int(n_src_cap), int(n_edge_cap)))


def sg_aggregate_bwd(indptr: torch.Tensor, idx: torch.Tensor, n_dst_cap: int, n_src_cap: int, n_edge_cap: int,
                     dims: Optional[torch.Tensor], gdst: torch.Tensor, gsrc: torch.Tensor, workspace: torch.Tensor,
                     stream=None) -> None:
    dim = gdst.shape[1]
    _check(load().sg_aggregate_bwd(indptr.data_ptr(), idx.data_ptr(), int(n_dst_cap), int(n_src_cap),
                                   int(n_edge_cap), _ptr(dims), gdst.data_ptr(), _dtype_code(gdst), int(dim),
                                   gsrc.data_ptr(), _dtype_code(gsrc), workspace.data_ptr(), workspace.numel(),
                                   _stream(stream)))


def aligned_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return _aligned_bytes(max(256, nbytes), device)


def sg_read_probe(src_ptr: int, nbytes: int, sink: torch.Tensor, stream=None) -> None:
    _check(load().sg_read_probe(int(src_ptr), int(nbytes), sink.data_ptr(), _stream(stream)))


def sg_wait_probe(n_tiles: int, silent_tile: int, spin_limit: int, out: torch.Tensor, stream=None) -> None:
    """Runs the bounded look-back wait over n_tiles tiles with tile
    silent_tile never publishing (see include/sg.h); out: int32 [n_tiles]."""
    lib = load()
    nbytes = int(lib.sg_wait_probe_workspace(int(n_tiles)))
    ws = _aligned_bytes(max(256, nbytes), out.device)
    _check(lib.sg_wait_probe(int(n_tiles), int(silent_tile), int(spin_limit), ws.data_ptr(), ws.numel(),
                             out.data_ptr(), _stream(stream)))


def sg_hash_probe(n_calls: int, seed: int, sink: torch.Tensor, stream=None) -> None:
    _check(load().sg_hash_probe(int(n_calls), ctypes.c_uint64(seed), sink.data_ptr(), _stream(stream)))


SG_RELABEL_NOALLOC_MAX_IDS = 262144


def sg_relabel_noalloc(ids: torch.Tensor, prefix: torch.Tensor, unique: torch.Tensor, local: torch.Tensor,
                       n_unique: torch.Tensor, stream=None) -> None:
    """Relabel into caller-provided outputs with no allocation by the library
    (its scratch is a static device array; see include/sg.h).  The C entry
    point cannot see the sizes of the output arrays, so they are checked
    here: int32, contiguous, on one CUDA device, unique with room for
    len(prefix) + len(ids) entries, local for len(ids), n_unique for one."""
    n_ids, n_pre = int(ids.numel()), int(prefix.numel())
    arrays = {"ids": ids, "prefix": prefix, "unique": unique, "local": local, "n_unique": n_unique}
    dev = unique.device
    for name, t in arrays.items():
        if not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous() \
                or t.device != dev:
            raise SgError(SG_ERR_INVALID_ARG, "sg_relabel_noalloc: %s must be a contiguous int32 tensor on %s"
                          % (name, dev))
    if unique.numel() < n_pre + n_ids or local.numel() < n_ids or n_unique.numel() < 1:
        raise SgError(SG_ERR_INVALID_ARG, "sg_relabel_noalloc: outputs too small (unique needs %d entries, local %d, "
                      "n_unique 1)" % (n_pre + n_ids, n_ids))
    _check(load().sg_relabel_noalloc(ids.data_ptr() if n_ids else None, n_ids, prefix.data_ptr() if n_pre else None,
                                     n_pre, unique.data_ptr(), local.data_ptr(), n_unique.data_ptr(), _stream(stream)))


class TransposedBuffers:
    """Caller-owned device arrays of the transposed blocks of one
    sampler_run output (sg_transposed), plus the transpose workspace."""

    def __init__(self, bounds: Bounds, device="cuda"):
        H = len(bounds.max_edges)
        self.n_hops = H
        self.bounds = bounds
        self.tptr = [torch.empty(bounds.max_nodes[h] + 2, dtype=torch.int32, device=device) for h in range(1, H + 1)]
        self.tdst = [torch.empty(max(1, bounds.max_edges[h]), dtype=torch.int32, device=device) for h in range(H)]
        self.tw = [torch.empty(max(1, bounds.max_edges[h]), dtype=torch.float32, device=device) for h in range(H)]
        self._mn = np.ascontiguousarray(bounds.max_nodes, dtype=np.int64)
        self._me = np.ascontiguousarray(bounds.max_edges, dtype=np.int64)
        wsb = load().sg_transpose_workspace(self._mn.ctypes.data, self._me.ctypes.data, H)
        if wsb == 0:
            raise SgError(SG_ERR_INVALID_ARG, "sg_transpose_workspace: bad bounds")
        self.workspace = _aligned_bytes(wsb, device)
        self._t = _Transposed()
        for h in range(H):
            self._t.tptr[h] = self.tptr[h].data_ptr()
            self._t.tdst[h] = self.tdst[h].data_ptr()
            self._t.tw[h] = self.tw[h].data_ptr()


def sg_transpose_blocks(buffers: SampleBuffers, tbuf: TransposedBuffers, stream=None) -> None:
    _check(load().sg_transpose_blocks(ctypes.byref(buffers._blocks), tbuf._mn.ctypes.data, tbuf._me.ctypes.data,
                                      tbuf.n_hops, ctypes.byref(tbuf._t), tbuf.workspace.data_ptr(),
                                      tbuf.workspace.numel(), _stream(stream)))


def sg_aggregate_bwd_t(tptr: torch.Tensor, tdst: torch.Tensor, tw: torch.Tensor, n_src_cap: int, n_dst_cap: int,
                       dims: Optional[torch.Tensor], gdst: torch.Tensor, gsrc: torch.Tensor, stream=None) -> None:
    dim = gdst.shape[1]
    _check(load().sg_aggregate_bwd_t(tptr.data_ptr(), tdst.data_ptr(), tw.data_ptr(), int(n_src_cap), int(n_dst_cap),
                                     _ptr(dims), gdst.data_ptr(), _dtype_code(gdst), int(dim), gsrc.data_ptr(),
                                     _dtype_code(gsrc), _stream(stream)))
