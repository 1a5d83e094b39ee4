"""One mini-batch of the pipeline, end to end, through the C ABI.

Per step (GARDEN page, Section II-B, Fig. 1: sampling runs outward from the
seeds, aggregation inward from the input nodes):
  1. sg_sampler_run   V_0 .. V_H and the H blocks (sampling + relabel)
  2. sg_gather        X = features of V_H through the HBM cache
  3. sg_aggregate_fwd H_{h-1} = mean over block h of H_h, h = H .. 1 (H_H = X)
  4. sg_aggregate_bwd_t  G_h = transpose of block h applied to G_{h-1}, h = 1 .. H,
                      with G_0 = H_0 (the gradient of 0.5 * ||H_0||^2); the
                      transposed blocks (sg_transpose_blocks) are built on a
                      second stream while 2 and 3 run
Every size that depends on the sample stays on the device (the calls read
the counts the sampler wrote), so a step has no host synchronisation and can
be captured in a CUDA graph and replayed with new seeds (written into the
device seed buffers first).  With one mini-batch the gather runs in two
parts: V_{H-1} is a prefix of V_H and is final once hop H-1 is relabelled
(the sampler records an event there), so its feature rows are gathered on a
second stream while hop H is sampled, and only the rows new at hop H wait for
the sampler.  OverlappedPipeline runs consecutive batches on several such
pipelines, so that one batch's sampling and gather overlap the previous
batch's forward and backward.  This module only allocates buffers and orders
the calls.
"""
from __future__ import annotations

from typing import Iterable, Optional, Sequence, Tuple

import torch

from . import binding as sg


def rank_by_access(graph: sg.Graph, batches: Iterable[Tuple[torch.Tensor, int]], fanouts: Sequence[int],
                   omega: Sequence[int], w_in: int = 1, device="cuda", tie_by_in_degree: bool = True):
    """Presampling statistics and ranking (GARDEN page, Section IV-B): each
    (seeds, hash seed) batch is sampled and its full-link access statistics
    (Eq. (4), weights omega per layer and w_in for input nodes) are added to a
    per-node score on the device; returns (order, rank_of), nodes by
    descending score, equal scores (among them every node the presampled
    batches never reached) by descending in-degree, then by ID.  All sizes of
    a batch must be equal."""
    score = torch.zeros(graph.n_nodes, dtype=torch.int32, device=device)
    buf, n_seeds = None, None
    for seeds, hseed in batches:
        if buf is None:
            n_seeds = int(seeds.numel())
            bounds = sg.sg_sampler_bounds(graph, n_seeds, fanouts)
            buf = sg.SampleBuffers(bounds, device, graph, n_seeds, fanouts)
        elif int(seeds.numel()) != n_seeds:
            raise ValueError("rank_by_access: every presampled batch must have %d seeds" % n_seeds)
        sg.sg_sampler_run(graph, seeds, fanouts, hseed, buf)
        sg.sg_access_stats(buf, omega, w_in, score)
    tie = sg.sg_graph_in_degree(graph) if tie_by_in_degree else None
    return sg.sg_rank_by_score(score, tie)


def recode_by_access(graph: sg.Graph, batches, fanouts, omega, w_in: int = 1, device="cuda",
                     tie_by_in_degree: bool = True):
    """rank_by_access, then the graph recoded so that the node of rank r has
    ID r (Section IV-A): returns (new graph, order, rank_of).  The feature
    table must then be laid out in the new order (new row r = old row
    order[r]) for an ID-range cache, and seeds mapped through rank_of."""
    order, rank_of = rank_by_access(graph, batches, fanouts, omega, w_in, device, tie_by_in_degree)
    return sg.sg_graph_renumber(graph, order, rank_of), order, rank_of


class MiniBatchPipeline:
    def __init__(self, graph: sg.Graph, cache: sg.Cache, fanouts: Sequence[int], n_seeds: int,
                 batch_ptr: Optional[Sequence[int]] = None, backward: bool = True, device="cuda",
                 split_gather: Optional[bool] = None):
        self.graph, self.cache = graph, cache
        self.fanouts = [int(f) for f in fanouts]
        self.H = len(self.fanouts)
        self.n_seeds = int(n_seeds)
        self.batch_ptr = None if batch_ptr is None else [int(x) for x in batch_ptr]
        self.backward = backward
        self.bounds = sg.sg_sampler_bounds(graph, n_seeds, self.fanouts, self.batch_ptr)
        self.buf = sg.SampleBuffers(self.bounds, device, graph, n_seeds, self.fanouts, self.batch_ptr)
        dt = torch.float32 if cache.dtype == sg.SG_F32 else torch.bfloat16
        self.dtype = dt
        d = cache.dim
        nb = self.bounds.max_nodes
        self.seeds = torch.zeros(max(1, n_seeds), dtype=torch.int32, device=device)
        self.d_seed = torch.zeros(1, dtype=torch.int64, device=device)
        # h_feat[h] holds H_h: rows V_h, h = 0..H (h = H is X)
        self.h_feat = [torch.empty(max(1, nb[h]), d, dtype=dt, device=device) for h in range(self.H + 1)]
        self.stats = torch.zeros(2, dtype=torch.int64, device=device)
        # gather scratch for reading misses grouped by host-table region (large
        # host tables only); the two parts of a split gather may overlap, so
        # each has its own
        self.gather_ws = [self._gather_ws(nb[self.H], device), self._gather_ws(nb[self.H - 1], device)]
        if backward:
            self.g_feat = [self.h_feat[0]] + [torch.empty(max(1, nb[h]), d, dtype=dt, device=device)
                                              for h in range(1, self.H + 1)]
            self.tbuf = sg.TransposedBuffers(self.bounds, device)
            self.side = torch.cuda.Stream(device=device)
            self.ev_sampled = torch.cuda.Event()
            self.ev_transposed = torch.cuda.Event()
        # split gather (one mini-batch, two hops or more): the rows of V_{H-1}
        # go first, on their own stream
        can_split = (self.batch_ptr is None or len(self.batch_ptr) == 2) and self.H >= 2
        self.split_gather = can_split if split_gather is None else (bool(split_gather) and can_split)
        if self.split_gather:
            H = self.H
            self.gather_stream = torch.cuda.Stream(device=device)
            self.ev_prefix = torch.cuda.Event()
            self.ev_prefix.record()  # creates the event, whose handle the sampler records
            self.ev_gathered = torch.cuda.Event()
            # |V_{H-1}| of the single mini-batch, final when ev_prefix fires
            at = (2 * H + 1) + (H - 1)
            self.n_prefix = self.buf.counts[at:at + 1]

    def _gather_ws(self, n_cap: int, device) -> Optional[torch.Tensor]:
        nbytes = sg.sg_gather_workspace(self.cache, n_cap)
        return sg.aligned_workspace(nbytes, device) if nbytes > 0 else None

    @property
    def counts(self) -> torch.Tensor:
        return self.buf.counts

    @property
    def x(self) -> torch.Tensor:
        return self.h_feat[self.H]

    def set_batch(self, seeds: torch.Tensor, seed: int) -> None:
        """Copies a new batch's seeds and hash seed into the device buffers."""
        if seeds.numel() != self.n_seeds:
            raise ValueError("set_batch: expected %d seeds, got %d" % (self.n_seeds, seeds.numel()))
        self.seeds[: seeds.numel()].copy_(seeds, non_blocking=True)
        self.d_seed.fill_(seed if seed < (1 << 63) else seed - (1 << 64))

    def sample(self, stream=None, hop_events=None) -> None:
        sg.sg_sampler_run(self.graph, self.seeds[: self.n_seeds], self.fanouts, 0, self.buf, self.batch_ptr,
                          stream=stream, d_seed=self.d_seed, hop_events=hop_events)

    def gather_prefix(self, stream=None) -> None:
        """Rows of V_{H-1} (split gather only)."""
        H = self.H
        sg.sg_gather(self.cache, self.buf.unique, self.bounds.max_nodes[H - 1], self.n_prefix, self.h_feat[H],
                     self.stats, stream=stream, workspace=self.gather_ws[1])

    def gather_rest(self, stream=None) -> None:
        """Rows of V_H from |V_{H-1}| on (split gather only)."""
        H = self.H
        sg.sg_gather(self.cache, self.buf.unique, self.bounds.max_nodes[H], self.buf.counts[H:H + 1],
                     self.h_feat[H], self.stats, stream=stream, d_first=self.n_prefix, workspace=self.gather_ws[0])

    def gather(self, stream=None) -> None:
        H = self.H
        if self.split_gather:
            self.gather_prefix(stream)
            self.gather_rest(stream)
            return
        sg.sg_gather(self.cache, self.buf.unique, self.bounds.max_nodes[H], self.buf.counts[H:H + 1],
                     self.h_feat[H], self.stats, stream=stream, workspace=self.gather_ws[0])

    def forward(self, stream=None) -> None:
        nb = self.bounds.max_nodes
        for h in range(self.H, 0, -1):
            sg.sg_aggregate_fwd(self.buf.indptr[h - 1], self.buf.idx[h - 1], nb[h - 1], nb[h], self.buf.dims(h),
                                self.h_feat[h], self.h_feat[h - 1], stream=stream)

    def transpose(self, stream=None) -> None:
        sg.sg_transpose_blocks(self.buf, self.tbuf, stream=stream)

    def backward_pass(self, stream=None) -> None:
        nb = self.bounds.max_nodes
        t = self.tbuf
        for h in range(1, self.H + 1):
            sg.sg_aggregate_bwd_t(t.tptr[h - 1], t.tdst[h - 1], t.tw[h - 1], nb[h], nb[h - 1], self.buf.dims(h),
                                  self.g_feat[h - 1], self.g_feat[h], stream=stream)

    def load(self, stream=None, join: bool = False) -> None:
        """Sampling, the transposed blocks and the gather of the current batch.
        The transposes fork onto a second stream after sampling; with join
        they are joined back before this returns (as a CUDA graph capture of
        this part alone needs), otherwise train() joins them before the
        backward pass.  With the split gather, V_{H-1}'s rows are gathered on a
        third stream during hop H."""
        main = torch.cuda.current_stream() if stream is None else stream
        self.load_sample(main)
        self.load_gather(main, join)

    def load_sample(self, stream=None) -> None:
        """The first part of load(): sampling (with the split gather's first
        part on its own stream) and the transposes forked to a side stream."""
        main = torch.cuda.current_stream() if stream is None else stream
        if self.split_gather:
            events = [None] * self.H
            events[self.H - 2] = self.ev_prefix
            self.sample(main, hop_events=events)
            self.gather_stream.wait_event(self.ev_prefix)
            self.gather_prefix(self.gather_stream)
            self.ev_gathered.record(self.gather_stream)
        else:
            self.sample(main)
        if self.backward:
            self.ev_sampled.record(main)
            self.side.wait_event(self.ev_sampled)
            self.transpose(self.side)
            self.ev_transposed.record(self.side)

    def load_gather(self, stream=None, join: bool = False) -> None:
        """The second part of load(): the gather (the rest of it, with the
        split gather); with join, the side streams are joined back."""
        main = torch.cuda.current_stream() if stream is None else stream
        if self.split_gather:
            self.gather_rest(main)
            main.wait_event(self.ev_gathered)
        else:
            self.gather(main)
        if self.backward and join:
            main.wait_event(self.ev_transposed)

    def train(self, stream=None, joined: bool = False) -> None:
        """Forward and (if enabled) backward of the batch load() prepared;
        joined: load() joined the transposes already (no wait here, as a CUDA
        graph capture of this part alone needs)."""
        main = torch.cuda.current_stream() if stream is None else stream
        self.forward(main)
        if self.backward:
            if not joined:
                main.wait_event(self.ev_transposed)
            self.backward_pass(main)

    def step(self, stream=None) -> None:
        """Sample, gather, forward and (if enabled) backward of one batch; the
        transposes overlap the gather and the forward."""
        self.load(stream)
        self.train(stream)

    def host_counts(self):
        c = self.buf.counts.cpu().tolist()
        H = self.H
        return {"nodes": c[: H + 1], "edges": c[H + 1: 2 * H + 1]}


class OverlappedPipeline:
    """Consecutive batches overlapped: `depth` MiniBatchPipelines (each with
    its own buffers and streams) take batches in turn, so batch i+1 is
    sampled, transposed and gathered while batch i's forward and backward run
    (the sampler and the zero-copy gather are latency- and link-bound and
    leave most of the GPU's issue slots free).  Batch i+1's forward waits for
    batch i's backward, the order a training loop that updates weights between
    batches needs.  A pipeline is reused `depth` batches later, after its own
    stream has finished with the earlier batch.

    step() enqueues one batch and returns the pipeline that holds it; its
    results (counts, h_feat, g_feat) are valid once that pipeline's stream
    reaches them.  capture() records each pipeline's two parts as CUDA graphs
    (depth 1: the whole step as one graph), which step() then replays.

    With serial_gathers (for host tables large enough that the gather reads
    misses grouped by region), batches still overlap, but their gathers run
    one after another: concurrent gathers of several batches would interleave
    their regions and lose the grouping (measured on the 61 GB Wide table:
    3.6 ms a step with four pipelines gathering at once against 2.8 ms one
    batch at a time).  Each batch's gather is then a single call, after its
    sampling, and batch i+1 is sampled and transposed while batch i gathers.

    suggested_depth() picks the depth (4, or 2 with serial gathers when
    misses are read by region) and suggested_serial_gathers() the mode."""

    @staticmethod
    def suggested_depth(cache: sg.Cache) -> int:
        return 2 if sg.sg_gather_workspace(cache, 1) > 0 else 4

    @staticmethod
    def suggested_serial_gathers(cache: sg.Cache) -> bool:
        return sg.sg_gather_workspace(cache, 1) > 0

    def __init__(self, graph: sg.Graph, cache: sg.Cache, fanouts: Sequence[int], n_seeds: int, depth: int = 2,
                 batch_ptr: Optional[Sequence[int]] = None, backward: bool = True, device="cuda",
                 serial_gathers: bool = False):
        if depth < 1:
            raise ValueError("OverlappedPipeline: depth must be at least 1")
        self.serial_gathers = bool(serial_gathers) and depth > 1
        self.pipes = [MiniBatchPipeline(graph, cache, fanouts, n_seeds, batch_ptr=batch_ptr, backward=backward,
                                        device=device, split_gather=False if self.serial_gathers else None)
                      for _ in range(depth)]
        self.streams = [torch.cuda.Stream(device=device) for _ in range(depth)]
        self.ev_trained = torch.cuda.Event()
        self.ev_trained.record()  # nothing is training yet
        self.ev_gathered = torch.cuda.Event()
        self.ev_gathered.record()  # nothing is gathering yet
        self.graphs = None
        self.i = 0

    @property
    def depth(self) -> int:
        return len(self.pipes)

    def next_slot(self) -> int:
        """Index of the pipeline the next step() uses."""
        return self.i % self.depth

    def capture(self) -> None:
        graphs = []
        if self.depth == 1:  # no overlap: the whole step, transposes beside gather and forward
            p, s = self.pipes[0], self.streams[0]
            with torch.cuda.stream(s):
                p.step(s)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                p.step(s)
            torch.cuda.synchronize()
            self.graphs = [(g, None)]
            return
        for p, s in zip(self.pipes, self.streams):
            with torch.cuda.stream(s):  # warm-up outside the capture
                p.load(s, join=True)
                p.train(s, joined=True)
            s.synchronize()
            gt = torch.cuda.CUDAGraph()
            if self.serial_gathers:  # sampling + transposes, and the gather, as two graphs
                gs, gg = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
                with torch.cuda.graph(gs, stream=s):
                    p.load_sample(s)
                    if p.backward:
                        s.wait_event(p.ev_transposed)
                with torch.cuda.graph(gg, stream=s):
                    p.load_gather(s)
                gl = (gs, gg)
            else:
                gl = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gl, stream=s):
                    p.load(s, join=True)
            with torch.cuda.graph(gt, stream=s):
                p.train(s, joined=True)
            graphs.append((gl, gt))
        torch.cuda.synchronize()
        self.graphs = graphs

    def step(self, set_inputs=None, after=None) -> MiniBatchPipeline:
        """Enqueues one batch.  set_inputs(pipe, stream), if given, is called
        first on the pipeline's stream to write the batch's seeds (for
        instance pipe.set_batch, or copies from pinned memory); after(pipe,
        stream), if given, is called on it once the batch is enqueued (for
        instance to copy results out before the pipeline is reused)."""
        k = self.next_slot()
        p, s = self.pipes[k], self.streams[k]
        with torch.cuda.stream(s):
            if set_inputs is not None:
                set_inputs(p, s)
            if self.depth == 1:
                if self.graphs is None:
                    p.step(s)
                else:
                    self.graphs[0][0].replay()
                if after is not None:
                    after(p, s)
                self.i += 1
                return p
            if self.serial_gathers:
                # this batch samples beside the previous batch's gather; its
                # own gather waits for that one
                if self.graphs is None:
                    p.load_sample(s)
                    if p.backward:
                        s.wait_event(p.ev_transposed)
                else:
                    self.graphs[k][0][0].replay()
                s.wait_event(self.ev_gathered)
                if self.graphs is None:
                    p.load_gather(s)
                else:
                    self.graphs[k][0][1].replay()
                self.ev_gathered.record(s)
            elif self.graphs is None:
                p.load(s, join=True)
            else:
                self.graphs[k][0].replay()
            s.wait_event(self.ev_trained)
            if self.graphs is None:
                p.train(s, joined=True)
            else:
                self.graphs[k][1].replay()
            self.ev_trained.record(s)
            if after is not None:
                after(p, s)
        self.i += 1
        return p

    def wait_all(self, stream=None) -> None:
        """Makes `stream` (default: the current one) wait for every step
        enqueued so far."""
        st = torch.cuda.current_stream() if stream is None else stream
        for s in self.streams:
            ev = torch.cuda.Event()
            ev.record(s)
            st.wait_event(ev)

    def start_after(self, stream=None) -> None:
        """Makes the pipelines' streams wait for `stream` (default: the
        current one), e.g. for inputs written there."""
        st = torch.cuda.current_stream() if stream is None else stream
        ev = torch.cuda.Event()
        ev.record(st)
        for s in self.streams:
            s.wait_event(ev)
