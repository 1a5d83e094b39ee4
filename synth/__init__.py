"""Seeded synthetic inputs: Chung-Lu power-law CSR graphs, N(0,1) features and
mini-batch seed nodes.

These are inputs only; this package holds none of the pipeline's arithmetic,
so the CUDA path and the CPU oracle can both consume what it makes.  The C
source (``synth.c``) is compiled on first use into ``_synth.so`` beside it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .configs import CONFIGS, Workload, workload  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "_synth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile synth.c into _synth.so (OpenMP when the compiler has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if r.returncode != 0:
        r = subprocess.run(base, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("synth build failed:\n" + r.stderr)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, u64, dbl, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p
        lib.synth_draw.restype = u64
        lib.synth_draw.argtypes = [u64, u64, u64]
        lib.synth_num_threads.restype = ctypes.c_int
        lib.synth_perm.restype = i64
        lib.synth_perm.argtypes = [u64, i64, i64]
        lib.synth_chung_lu_i0.restype = dbl
        lib.synth_chung_lu_i0.argtypes = [i64, dbl, dbl, dbl]
        lib.synth_chung_lu_weight.restype = dbl
        lib.synth_chung_lu_weight.argtypes = [i64, dbl, dbl, dbl, i64]
        lib.synth_graph_build.restype = vp
        lib.synth_graph_build.argtypes = [i64, dbl, dbl, dbl, u64]
        for name in ("synth_graph_n", "synth_graph_m"):
            getattr(lib, name).restype = i64
            getattr(lib, name).argtypes = [vp]
        lib.synth_graph_indptr.restype = ctypes.POINTER(ctypes.c_int64)
        lib.synth_graph_indptr.argtypes = [vp]
        lib.synth_graph_indices.restype = ctypes.POINTER(ctypes.c_int32)
        lib.synth_graph_indices.argtypes = [vp]
        lib.synth_graph_free.restype = None
        lib.synth_graph_free.argtypes = [vp]
        lib.synth_features.restype = ctypes.c_int
        lib.synth_features.argtypes = [i64, i64, i32, i32, u64, vp]
        lib.synth_features_rows.restype = ctypes.c_int
        lib.synth_features_rows.argtypes = [vp, i64, i32, i32, u64, vp]
        lib.synth_batch_seeds.restype = i32
        lib.synth_batch_seeds.argtypes = [i64, dbl, u64, i64, i64, i32, vp]
        lib.synth_epoch_order.restype = i64
        lib.synth_epoch_order.argtypes = [i64, dbl, u64, i64, vp, i64]
        lib.synth_mask_count.restype = i64
        lib.synth_mask_count.argtypes = [i64, dbl, u64]
        _lib = lib
        return lib


def num_threads() -> int:
    return int(_load().synth_num_threads())


def draw(seed: int, stream: int, i: int) -> int:
    return int(_load().synth_draw(seed, stream, i))


def perm(key: int, n: int, i: int) -> int:
    return int(_load().synth_perm(key, n, i))


class Graph:
    """A CSR graph owned by the C generator.  ``indptr`` (int64, N+1) and
    ``indices`` (int32, M) are zero-copy numpy views that live as long as
    this object."""

    def __init__(self, handle, n, m):
        self._h = handle
        self.n = int(n)
        self.m = int(m)
        lib = _load()
        self.indptr = np.ctypeslib.as_array(lib.synth_graph_indptr(handle), shape=(self.n + 1,))
        if self.m > 0:
            self.indices = np.ctypeslib.as_array(lib.synth_graph_indices(handle), shape=(self.m,))
        else:
            self.indices = np.zeros(0, np.int32)

    def degrees(self) -> np.ndarray:
        return np.diff(self.indptr)

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h and _lib is not None:
            _lib.synth_graph_free(h)


def chung_lu(n: int, mean: float, gamma: float, wmax: float, seed: int = 0) -> Graph:
    """Chung-Lu power-law graph (recipe in synth.c): sorted rows, no
    self-loops, no repeated edges."""
    lib = _load()
    h = lib.synth_graph_build(int(n), float(mean), float(gamma), float(wmax), int(seed))
    if not h:
        raise ValueError("chung_lu: bad parameters or out of host memory")
    return Graph(h, lib.synth_graph_n(h), lib.synth_graph_m(h))


def csr_graph(indptr, indices):
    """A plain in-memory CSR (for hand-made test graphs)."""
    class _G:
        pass
    g = _G()
    g.indptr = np.ascontiguousarray(indptr, dtype=np.int64)
    g.indices = np.ascontiguousarray(indices, dtype=np.int32)
    g.n = len(g.indptr) - 1
    g.m = int(g.indptr[-1])
    g.degrees = lambda: np.diff(g.indptr)
    return g


def features_into(out_ptr: int, row0: int, nrows: int, dim: int, dtype: str, seed: int = 0) -> None:
    """Write rows [row0, row0+nrows) of the N(0,1) feature table to raw memory
    at ``out_ptr`` (fp32 or bf16 as uint16 bits)."""
    code = {"f32": 0, "bf16": 1}[dtype]
    if _load().synth_features(int(row0), int(nrows), int(dim), code, int(seed), ctypes.c_void_p(out_ptr)):
        raise ValueError("features_into: bad arguments")


def features_rows_into(out_ptr: int, ids: np.ndarray, dim: int, dtype: str, seed: int = 0) -> None:
    """Write the feature rows of nodes ids[0], ids[1], ... as consecutive rows
    at ``out_ptr`` (the table laid out for recoded node IDs)."""
    code = {"f32": 0, "bf16": 1}[dtype]
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    if _load().synth_features_rows(ids.ctypes.data, len(ids), int(dim), code, int(seed), ctypes.c_void_p(out_ptr)):
        raise ValueError("features_rows_into: bad arguments")


def features(n: int, dim: int, dtype: str = "f32", seed: int = 0, row0: int = 0) -> np.ndarray:
    """N(0,1) feature rows as numpy: float32, or uint16 bf16 bit patterns."""
    out = np.empty((n, dim), dtype=np.float32 if dtype == "f32" else np.uint16)
    features_into(out.ctypes.data, row0, n, dim, dtype, seed)
    return out


def batch_seeds(n: int, p_mask: float, batch: int, bsize: int, seed: int = 0, epoch: int = 0) -> np.ndarray:
    """Seed nodes of mini-batch ``batch`` of the given epoch (distinct IDs)."""
    out = np.empty(bsize, dtype=np.int32)
    w = _load().synth_batch_seeds(int(n), float(p_mask), int(seed), int(epoch), int(batch), int(bsize),
                                  out.ctypes.data)
    return out[:w].copy()


def epoch_order(n: int, p_mask: float, seed: int, epoch: int, n_train: int) -> np.ndarray:
    """Training nodes in the order of one epoch (batch b = entries [bB, (b+1)B))."""
    out = np.empty(max(1, n_train), dtype=np.int32)
    w = _load().synth_epoch_order(int(n), float(p_mask), int(seed), int(epoch), out.ctypes.data, int(n_train))
    return out[:w]


def mask_count(n: int, p_mask: float, seed: int = 0) -> int:
    return int(_load().synth_mask_count(int(n), float(p_mask), int(seed)))


class BatchStream:
    """Seed batches of a workload, epoch after epoch: batch b is batch
    (b mod n) of epoch epoch0 + b // n, n = batches per epoch (full batches
    of the training mask only)."""

    def __init__(self, w, epoch0: int = 0):
        self.w = w
        self.epoch0 = epoch0
        self.n_train = mask_count(w.n_nodes, w.p_mask, w.rng_seed)
        self.per_epoch = max(1, self.n_train // w.batch)
        self._epoch, self._order = None, None

    def seeds(self, b: int) -> np.ndarray:
        ep, i = divmod(int(b), self.per_epoch)
        if self._epoch != ep:  # the epoch's order in one pass, kept for its batches
            self._order = epoch_order(self.w.n_nodes, self.w.p_mask, self.w.rng_seed, self.epoch0 + ep,
                                      self.n_train)
            self._epoch = ep
        return self._order[i * self.w.batch:(i + 1) * self.w.batch].copy()
