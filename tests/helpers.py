"""Shared helpers of the GPU parity tests (marshalling between numpy, the
oracle and the C ABI)."""
import numpy as np
import torch

import oracle
from sampling_gnn_mini_gb300 import binding as sg


def dev_i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def bf16_to_torch(u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16)


def torch_to_np(t: torch.Tensor) -> np.ndarray:
    """float32 -> float32 array; bfloat16 -> uint16 bit patterns."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return oracle.bf16_to_f32(a).reshape(a.shape).astype(np.float64)
    return a.astype(np.float64)


def feat_tensor(feat: np.ndarray, device=None, pinned=False) -> torch.Tensor:
    t = bf16_to_torch(feat) if feat.dtype == np.uint16 else torch.from_numpy(np.ascontiguousarray(feat))
    if pinned:
        return t.pin_memory()
    return t.to(device) if device else t


def assert_close(got: np.ndarray, want: np.ndarray, absmean: np.ndarray, tol: float, what: str = ""):
    """|got - want| <= tol * (absmean + 1e-30) elementwise: the fp error scale
    of a mean of terms (fp32 accumulation, relative tolerance tol)."""
    err = np.abs(got - want)
    bound = tol * (absmean + 1e-30)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError("%s: %d elements out of tolerance; first at %s: got %r want %r bound %r"
                             % (what, int(bad.sum()), tuple(i), got[tuple(i)], want[tuple(i)], bound[tuple(i)]))


class GpuSample:
    """Runs sg_sampler_run once and copies the result to the host."""

    def __init__(self, graph: sg.Graph, seeds, fanouts, seed, batch_ptr=None):
        seeds = np.ascontiguousarray(seeds, dtype=np.int32)
        self.bounds = sg.sg_sampler_bounds(graph, len(seeds), fanouts, batch_ptr)
        self.buf = sg.SampleBuffers(self.bounds, graph=graph, n_seeds=len(seeds), fanouts=fanouts, batch_ptr=batch_ptr)
        sg.sg_sampler_run(graph, dev_i32(seeds) if len(seeds) else torch.zeros(1, dtype=torch.int32, device="cuda")[:0],
                          fanouts, seed, self.buf, batch_ptr)
        sg.sg_stream_check()
        H = len(fanouts)
        c = self.buf.counts.cpu().numpy()
        self.H = H
        self.counts = c
        self.tot_nodes = [int(x) for x in c[: H + 1]]
        self.tot_edges = [int(x) for x in c[H + 1: 2 * H + 1]]
        self.unique = self.buf.unique.cpu().numpy()[: self.tot_nodes[H]]
        self.indptr = [self.buf.indptr[h].cpu().numpy()[: self.tot_nodes[h] + 1] for h in range(H)]
        self.idx = [self.buf.idx[h].cpu().numpy()[: self.tot_edges[h]] for h in range(H)]

    def sub_counts(self, k):
        H = self.H
        base = (2 * H + 1) * (1 + k)
        return [int(x) for x in self.counts[base: base + H + 1]], [int(x) for x in self.counts[base + H + 1: base + 2 * H + 1]]


def assert_blocks_equal(gpu: GpuSample, ref: "oracle.Blocks"):
    H = gpu.H
    assert gpu.tot_nodes == list(ref.hop_off), (gpu.tot_nodes, ref.hop_off)
    assert np.array_equal(gpu.unique, ref.unique)
    for h in range(H):
        assert gpu.tot_edges[h] == len(ref.idx[h])
        assert np.array_equal(gpu.indptr[h], ref.indptr[h].astype(np.int32)), "indptr of hop %d" % (h + 1)
        assert np.array_equal(gpu.idx[h], ref.idx[h]), "idx of hop %d" % (h + 1)


def assert_super_equal(gpu: GpuSample, ref: "oracle.SuperBlocks"):
    H = gpu.H
    tot = ref.totals()
    assert gpu.tot_nodes == [int(x) for x in tot]
    assert np.array_equal(gpu.unique, ref.unique)
    for k in range(ref.n_sub):
        n, e = gpu.sub_counts(k)
        assert n == [int(x) for x in ref.counts[k]]
        assert e == [int(x) for x in ref.edge_counts[k]]
    for h in range(H):
        assert np.array_equal(gpu.indptr[h], ref.indptr[h].astype(np.int32)), "indptr of hop %d" % (h + 1)
        assert np.array_equal(gpu.idx[h], ref.idx[h]), "idx of hop %d" % (h + 1)
