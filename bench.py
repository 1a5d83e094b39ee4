"""Benchmark of the mini-batch pipeline (sample -> relabel -> cached gather ->
mean aggregation forward + backward).  The default workload is the largest
single-GPU one, Billion-edge: a 111M-node Chung-Lu graph (exponent 2.2, mean
degree 14.4, 1.6B edges, int64 offsets), 128-dim fp32 features (57 GB) in
pinned host memory, an HBM cache of 12e9 bytes (21% of the rows) ranked by
presampled access frequency, 3 hops with fanouts [15, 10, 5], 1024 seeds per
batch from a 1% training mask.  --config picks another workload (tiny, mid,
wide, skew_g<gamma>_b<batch>).

One step = one mini-batch through every stage.  Prints one JSON line.
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config billion]
Under torchrun (N > 1) every rank runs its own batches on its own GPU
(replicas, no collective on the data path); the slowest rank's time counts.
--impl reference times the CPU oracle on the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "sampled edges/s, gathered feature GB/s, batch latency; % of memory roofline"


def log(msg: str) -> None:
    """Progress on stderr (the JSON line alone goes to stdout)."""
    sys.stderr.write("[bench %.1fs] %s\n" % (time.time() - _T0, msg))
    sys.stderr.flush()


_T0 = time.time()


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="billion")
    ap.add_argument("--no-recode", action="store_true",
                    help="keep the original node IDs and a slot-map cache of the ranked rows")
    ap.add_argument("--omega", default="", help="layer weights of the access statistics, comma-separated (default 1s)")
    ap.add_argument("--w-in", type=int, default=1, help="input-node weight of the access statistics")
    ap.add_argument("--presample", type=int, default=0,
                    help="presampled batches for the cache ranking (0: the workload's own count, 64)")
    ap.add_argument("--experiment", default="", choices=["", "next"],
                    help="next: measure the dynamic cache and Match-Reorder on the workload instead of the headline")
    ap.add_argument("--dyn-frac", type=float, default=0.1, help="share of the cache budget given to the dynamic cache")
    ap.add_argument("--dyn-gamma", type=float, default=0.9, help="decay per batch of the dynamic cache's scores")
    ap.add_argument("--dyn-window", type=int, default=16, help="batches per dynamic-cache update")
    ap.add_argument("--group", type=int, default=16, help="batches per Match-Reorder group (<= 32)")
    ap.add_argument("--min-seconds", type=float, default=2.0,
                    help="the timed region of --steps steps is repeated (new batches each time) until this long")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="bound on the CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--depth", type=int, default=0,
                    help="pipelines the overlapped batches rotate through (0: OverlappedPipeline.suggested_depth)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_bf16_tflops():
    """The measured dense bf16 GEMM burst rate (TFLOP/s), or None."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            v = json.load(fh).get("bf16_tflops")
        return float(v) if v else None
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# Integer instructions of one Philox4x32-10 call as the library writes it:
# 10 rounds x (2 wide multiplies, 2 three-input XORs, 2 key additions) plus
# the counter setup.
PHILOX_INSTR = 64


def philox_issue_peak(torch, dev) -> float:
    """Philox calls/s at the instruction-issue limit: SMs x 4 schedulers x 32
    lanes x the maximum SM clock / instructions per call."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = None
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            mhz = json.load(fh).get("sm_max_mhz")
    if not mhz:
        mhz = 2070.0
    return sms * 4 * 32 * float(mhz) * 1e6 / PHILOX_INSTR


def sampler_traffic():
    """DRAM bytes per step of the three k_sample launches from the committed
    ncu summary, if the sampler source is the one that was profiled."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", "k_sample_mid.md")
    src = os.path.join(ROOT, "sampling_gnn_mini_gb300", "csrc", "sg_sampler.cu")
    if not (os.path.exists(prof) and os.path.exists(src)):
        return None
    want, traffic = None, None
    for line in open(prof):
        if line.startswith("traffic_bytes_per_step:"):
            traffic = float(line.split(":", 1)[1])
        if line.startswith("sg_sampler.cu sha256:"):
            want = line.split(":", 1)[1].strip()
    have = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return traffic if want == have else None


def gather_traffic(hits: float, misses: float):
    """DRAM bytes of the gather stage for the given hits and misses, scaled by
    units from the committed ncu summary when the gather source is the one
    that was profiled; else None."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", "k_gather_host_misses.md")
    src = os.path.join(ROOT, "sampling_gnn_mini_gb300", "csrc", "sg_gather.cu")
    if not (os.path.exists(prof) and os.path.exists(src)):
        return None
    vals, want = {}, None
    for line in open(prof):
        for key in ("traffic_per_hit_bytes", "traffic_per_miss_bytes"):
            if line.startswith(key + ":"):
                vals[key] = float(line.split(":", 1)[1])
        if line.startswith("sg_gather.cu sha256:"):
            want = line.split(":", 1)[1].strip()
    have = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if want != have or len(vals) != 2:
        return None
    return hits * vals["traffic_per_hit_bytes"] + misses * vals["traffic_per_miss_bytes"]


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workload
class Workload:
    """Graph, features and batches of one config, built once per process.
    With recode=True (the HBM cache holds part of the table) the feature
    table is not filled here: run_ours recodes the graph first (hot nodes to
    the smallest IDs) and fills the table in the new order."""

    def __init__(self, name: str, pinned_features: bool, recode: bool = False):
        import torch
        self.w = synth.workload(name)
        w = self.w
        t0 = time.time()
        self.g = synth.chung_lu(w.n_nodes, w.mean_deg, w.gamma, w.wmax, w.rng_seed)
        self.t_graph = time.time() - t0
        dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        t0 = time.time()
        if pinned_features:
            from sampling_gnn_mini_gb300.hostmem import pinned_table
            self.feat = pinned_table(w.n_nodes, w.dim, dt)
        else:
            self.feat = torch.empty((w.n_nodes, w.dim), dtype=dt)
        self.rank_of = None  # new ID of each node once recoded
        if not recode:
            synth.features_into(self.feat.data_ptr(), 0, w.n_nodes, w.dim, w.dtype, w.rng_seed)
        self.t_feat = time.time() - t0
        self.batches = synth.BatchStream(w, epoch0=0)
        self.presample = synth.BatchStream(w, epoch0=1000)  # a separate series of epochs

    def recoded(self, order: np.ndarray, rank_of: np.ndarray, indptr: np.ndarray, indices: np.ndarray) -> None:
        """Switches to the recoded graph: row r of the feature table becomes
        node order[r]'s row, and seeds are mapped through rank_of."""
        t0 = time.time()
        synth.features_rows_into(self.feat.data_ptr(), order, self.w.dim, self.w.dtype, self.w.rng_seed)
        self.t_feat += time.time() - t0
        self.rank_of = rank_of
        self.g = synth.csr_graph(np.asarray(indptr, dtype=np.int64), indices)

    def seeds(self, batch: int) -> np.ndarray:
        s = self.batches.seeds(batch)
        return s if self.rank_of is None else self.rank_of[s]


def replica_batches(rank: int, world: int, n: int):
    """Batch indices of one rank: rank, rank + world, ...; the ranks' lists
    are disjoint and together are 0 .. n * world - 1."""
    return [rank + world * i for i in range(n)]


def combine_ranks(torch, elapsed_ms: float, counters, device):
    """Whole-job figures of a replica run: the slowest rank's time and the
    sums of the integer counters over ranks (unchanged for one rank)."""
    counters = [int(c) for c in counters]
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return elapsed_ms, counters
    import torch.distributed as dist
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    c = torch.tensor(counters, dtype=torch.int64, device=device)
    dist.all_reduce(c)
    return float(t.item()), [int(x) for x in c.tolist()]


def frontier_ids(counts, unique, H: int, n_sub: int, h: int) -> np.ndarray:
    """Distinct global IDs of V_h over the mini-batches of a step.  unique
    holds each mini-batch's V_H back to back, V_h being a prefix of it; the
    per-mini-batch sizes follow the totals in counts."""
    if n_sub == 1:
        return unique[: counts[h]]
    parts, u0 = [], 0
    for k in range(n_sub):
        base = (2 * H + 1) * (1 + k)
        parts.append(unique[u0: u0 + counts[base + h]])
        u0 += counts[base + H]
    return np.unique(np.concatenate(parts))


def kernels_per_step(H: int, n_sub: int, by_region: bool = False, split: bool = True) -> int:
    """Kernels one step launches: sampler 3 per hop (+1 per hop for a
    super-batch) + 2, transposes 5, gather 1 a call (4 when misses are read
    grouped by host-table region) and 2 calls when one mini-batch of two hops
    or more is gathered in two parts, forward 1 per hop, backward 1 per hop."""
    gathers = (2 if (split and n_sub == 1 and H >= 2) else 1) * (4 if by_region else 1)
    return (2 + 3 * H + (H if n_sub > 1 else 0)) + 5 + gathers + H + H


def setup_workload(args, sg, torch, dev, cache_rows=None):
    """Graph in HBM (recoded by presampled statistics when the cache holds
    part of the table), host feature table and cache, as the headline uses
    them.  Returns (W, G, cache, presample)."""
    from sampling_gnn_mini_gb300.pipeline import rank_by_access
    w0 = synth.workload(args.config)
    recode = w0.cache_rows < w0.n_nodes and not args.no_recode
    W = Workload(args.config, pinned_features=True, recode=recode)
    w, g = W.w, W.g
    H = w.n_hops
    log("workload %s: graph %.1fs, feature table %.1fs" % (w.name, W.t_graph, W.t_feat))

    # graph into HBM; int64 offsets where the config calls for them
    G = sg.sg_graph_load(g.indptr if w.offset_bits == 64 else g.indptr.astype(np.int32), g.indices, w.offset_bits)
    cache_rows = w.cache_rows if cache_rows is None else int(cache_rows)
    omega = [int(x) for x in args.omega.split(",")] if args.omega else [1] * H
    presample = None
    # rank nodes by their full-link access statistics (Eq. (4)) over presampled
    # batches disjoint from the measured ones, all on the GPU; then recode the
    # graph so that the hot nodes hold the smallest IDs (ID-range cache)
    if cache_rows < w.n_nodes:
        t0 = time.time()
        n_pre = args.presample if args.presample > 0 else w.presample_batches
        pre_batches = ((torch.from_numpy(W.presample.seeds(b)).to(dev), w.presample_seed(b)) for b in range(n_pre))
        order, rank_of = rank_by_access(G, pre_batches, w.fanouts, omega, args.w_in, device=dev)
        torch.cuda.synchronize(dev)
        sg.sg_stream_check()
        presample = {"batches": n_pre, "omega": omega, "w_in": args.w_in,
                     "statistics_and_rank_s": time.time() - t0}
        if recode:
            t0 = time.time()
            G2 = sg.sg_graph_renumber(G, order, rank_of)
            del G
            G = G2
            presample["recode_graph_s"] = time.time() - t0
            ip, ix = sg.sg_graph_copy_out(G)  # the recoded CSR, for the host-side bookkeeping and oracle
            W.recoded(order.cpu().numpy(), rank_of.cpu().numpy(), ip, ix)
            del ip, ix
            g = W.g
            ranked = None  # ID-range cache: nodes [0, cache_rows)
        else:
            ranked = order[:cache_rows].cpu().numpy()
        del order, rank_of
        log("presample %s" % presample)
    else:
        ranked = None
    dtype_code = sg.SG_F32 if w.dtype == "f32" else sg.SG_BF16
    cache = sg.sg_cache_build(W.feat if w.host_features else None,
                              None if w.host_features else W.feat.to(dev), dtype_code, w.n_nodes, w.dim,
                              ranked, cache_rows)
    return W, G, cache, presample


def run_ours(args, rank, world, local):
    import torch
    from sampling_gnn_mini_gb300 import binding as sg
    from sampling_gnn_mini_gb300.pipeline import MiniBatchPipeline, OverlappedPipeline

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    sg.load(build_if_missing=True)
    W, G, cache, presample = setup_workload(args, sg, torch, dev)
    w, g = W.w, W.g
    H = w.n_hops
    R = w.row_bytes
    hbm_peak, peak_kind = peaks()
    cache_rows = w.cache_rows
    # a step is one batch, or one super-batch of w.n_sub mini-batches that
    # share the hash seed (mini-batches b * n_sub .. b * n_sub + n_sub - 1)
    n_sub = w.n_sub
    SB = w.batch * n_sub  # seeds a step
    bptr = [w.batch * k for k in range(n_sub + 1)] if n_sub > 1 else None
    pipe = MiniBatchPipeline(G, cache, w.fanouts, SB, batch_ptr=bptr, device=dev)

    # batches of this rank (replicas: disjoint batch indices per rank): the
    # warm-up, then the K steps of the latency and stage regions, then the
    # repeats of the timed region (pool extended once their count is known)
    n_batches = args.warmup + args.steps
    bidx = replica_batches(rank, world, n_batches)

    def make_pool(batch_ids):
        sh = np.stack([np.concatenate([W.seeds(b * n_sub + k) for k in range(n_sub)])
                       for b in batch_ids]).astype(np.int32)
        return sh, torch.from_numpy(sh).to(dev), torch.tensor([w.sampler_seed(b) for b in batch_ids],
                                                              dtype=torch.int64, device=dev)

    seeds_host, seeds_pool, hseed_pool = make_pool(bidx)
    stream = torch.cuda.Stream(device=dev)

    # the whole step as one CUDA graph (the transposes fork onto a second
    # stream inside it), and the same work as per-stage graphs for the
    # per-kernel breakdown
    nb = pipe.bounds.max_nodes
    stages = [("sample", pipe.sample), ("transpose", pipe.transpose), ("gather", pipe.gather)]

    def fwd_hop(h):
        return lambda: sg.sg_aggregate_fwd(pipe.buf.indptr[h - 1], pipe.buf.idx[h - 1], nb[h - 1], nb[h],
                                           pipe.buf.dims(h), pipe.h_feat[h], pipe.h_feat[h - 1])

    def bwd_hop(h):
        t = pipe.tbuf
        return lambda: sg.sg_aggregate_bwd_t(t.tptr[h - 1], t.tdst[h - 1], t.tw[h - 1], nb[h], nb[h - 1],
                                             pipe.buf.dims(h), pipe.g_feat[h - 1], pipe.g_feat[h])

    for h in range(H, 0, -1):
        stages.append(("fwd%d" % h, fwd_hop(h)))
    for h in range(1, H + 1):
        stages.append(("bwd%d" % h, bwd_hop(h)))
    # the SAGE UPDATE (tensor cores) over the largest forward hop's output:
    # ReLU([H_{H-1} own rows | mean] W^T), W of 128 rows (staged region only;
    # the headline step is the four-step path)
    upd = None
    if (w.row_bytes % 16) == 0 and n_sub == 1:
        wdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        upd = {"W": (torch.randn((128, 2 * w.dim), generator=torch.Generator().manual_seed(7)) / (2 * w.dim) ** 0.5)
               .to(wdt).to(dev),
               "out": torch.empty((max(1, nb[H - 1]), 128), dtype=torch.float32, device=dev)}

        def update_hop():
            sg.sg_sage_fwd(pipe.h_feat[H], pipe.h_feat[H - 1], upd["W"], nb[H - 1], pipe.buf.dims(H), upd["out"])

    def load_batch(i):
        pipe.seeds[:SB].copy_(seeds_pool[i], non_blocking=True)
        pipe.d_seed.copy_(hseed_pool[i: i + 1], non_blocking=True)

    with torch.cuda.stream(stream):
        load_batch(0)
        pipe.step(stream)
        for _, fn in stages:
            fn()
    torch.cuda.synchronize(dev)
    sg.sg_stream_check(stream)
    # the optional SAGE UPDATE stage joins the breakdown once it has run
    # cleanly here (an error in it must not cost the rest of the measurement)
    update_note = None
    if upd is not None:
        try:
            with torch.cuda.stream(stream):
                update_hop()
            sg.sg_stream_check(stream)
            stages.append(("update%d" % H, update_hop))
        except sg.SgError as e:
            upd, update_note = None, "SAGE UPDATE stage left out: %s" % e
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph, stream=stream):
        pipe.step(stream)
    graphs = []
    for name, fn in stages:
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=stream):
            fn()
        graphs.append((name, cg))
    torch.cuda.synchronize(dev)
    counts_log = torch.zeros((n_batches, pipe.buf.counts.numel()), dtype=torch.int32, device=dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)] for _ in range(args.steps)]

    def one_step(i):
        load_batch(i)
        step_graph.replay()
        counts_log[i].copy_(pipe.buf.counts, non_blocking=True)

    def one_step_staged(i, events):
        load_batch(i)
        events[0].record(stream)
        for j, (_, cg) in enumerate(graphs):
            cg.replay()
            events[j + 1].record(stream)

    # the headline: consecutive batches overlapped on two pipelines (batch
    # i+1 is sampled and gathered while batch i's forward and backward run;
    # batch i+1's forward still waits for batch i's backward)
    depth = args.depth if args.depth > 0 else OverlappedPipeline.suggested_depth(cache)
    serial = OverlappedPipeline.suggested_serial_gathers(cache)
    ov = OverlappedPipeline(G, cache, w.fanouts, SB, depth=depth, batch_ptr=bptr, device=dev, serial_gathers=serial)
    with torch.cuda.stream(stream):
        load_batch(0)
    for p in ov.pipes:
        p.set_batch(pipe.seeds[:SB].clone(), w.sampler_seed(bidx[0]))
    torch.cuda.synchronize(dev)
    ov.capture()

    def ov_inputs(i):
        def f(p, s):
            p.seeds[:SB].copy_(seeds_pool[i], non_blocking=True)
            p.d_seed.copy_(hseed_pool[i: i + 1], non_blocking=True)
        return f

    def ov_after(i):
        def f(p, s):
            counts_log[i].copy_(p.buf.counts, non_blocking=True)
        return f

    for i in range(args.warmup):
        ov.step(ov_inputs(i), ov_after(i))
    torch.cuda.synchronize(dev)
    for s_ in ov.streams:
        sg.sg_stream_check(s_)

    def timed_region(pool_s, pool_h, first, log):
        """K steps on batches first .. first + K - 1 of the pool, bracketed by
        a barrier and synchronisation; returns the device time in ms."""
        def inputs(i):
            def f(p, s):
                p.seeds[:SB].copy_(pool_s[i], non_blocking=True)
                p.d_seed.copy_(pool_h[i: i + 1], non_blocking=True)
            return f

        def after(i):
            def f(p, s):
                log[i].copy_(p.buf.counts, non_blocking=True)
            return f
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ov.start_after(stream)
        marks = []
        for s_ in range(args.steps):
            k = ov.next_slot()
            ov.step(inputs(first + s_), after(first + s_))
            # an event when each step ends; batches end in order (each step's
            # training waits for the previous one), so the gaps between them
            # are the steps' durations in the steady state
            e = torch.cuda.Event(enable_timing=True)
            e.record(ov.streams[k])
            marks.append(e)
        ov.wait_all(stream)
        b.record(stream)
        torch.cuda.synchronize(dev)
        for s_ in ov.streams:
            sg.sg_stream_check(s_)
        if marks:
            prev = a
            for e in marks:
                step_ms.append(prev.elapsed_time(e))
                prev = e
        return a.elapsed_time(b)

    # a first region on the warm-up pool's last K batches sizes the repeats
    step_ms = []
    calib_ms = timed_region(seeds_pool, hseed_pool, args.warmup, counts_log)
    step_ms.clear()
    repeats = max(1, int(np.ceil(args.min_seconds * 1e3 / max(calib_ms, 1e-3))))
    log("calibration region %.2f ms for %d steps: %d timed regions" % (calib_ms, args.steps, repeats))
    if world > 1:  # every rank runs the same number of regions
        r_t = torch.tensor([repeats], dtype=torch.int64, device=dev)
        torch.distributed.all_reduce(r_t, op=torch.distributed.ReduceOp.MAX)
        repeats = int(r_t.item())
    rep_ids = replica_batches(rank, world, n_batches + repeats * args.steps)[n_batches:]
    _, rep_seeds, rep_hseed = make_pool(rep_ids)
    rep_log = torch.zeros((repeats * args.steps, pipe.buf.counts.numel()), dtype=torch.int32, device=dev)
    clocks = Clocks(local)
    clocks.start()
    torch.cuda.nvtx.range_push("timed")
    region_ms = [timed_region(rep_seeds, rep_hseed, r * args.steps, rep_log) for r in range(repeats)]
    torch.cuda.nvtx.range_pop()
    clk = clocks.stop()
    log("timed regions done: %s ms" % ", ".join("%.2f" % x for x in region_ms[:8]))
    rep_counts = rep_log.cpu().numpy().astype(np.int64)
    region_edges = [int(rep_counts[r * args.steps:(r + 1) * args.steps, H + 1: 2 * H + 1].sum())
                    for r in range(repeats)]
    # the median region by throughput is the headline
    order = sorted(range(repeats), key=lambda r: region_edges[r] / region_ms[r])
    med = order[len(order) // 2]
    elapsed_ms = region_ms[med]
    timed_edges = region_edges[med]
    # batch latency: the same batches one at a time (a step graph each)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            one_step(i)
    torch.cuda.synchronize(dev)
    l_start = torch.cuda.Event(enable_timing=True)
    l_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        l_start.record(stream)
        for s_ in range(args.steps):
            one_step(args.warmup + s_)
        l_end.record(stream)
    torch.cuda.synchronize(dev)
    latency_ms = l_start.elapsed_time(l_end) / args.steps
    sg.sg_stream_check(stream)
    # the same batches stage by stage, for the breakdown (and the cache hits
    # of exactly these batches' gathers)
    pipe.stats.zero_()
    with torch.cuda.stream(stream):
        for s_ in range(args.steps):
            one_step_staged(args.warmup + s_, ev[s_])
    torch.cuda.synchronize(dev)
    sg.sg_stream_check(stream)
    hits, misses = [int(x) for x in pipe.stats.cpu().tolist()]
    stage_runs = {name: [] for name, _ in graphs}
    for s_ in range(args.steps):
        for j, (name, _) in enumerate(graphs):
            stage_runs[name].append(ev[s_][j].elapsed_time(ev[s_][j + 1]))
    # the median over the steps: a zero-copy stall of the host link in one
    # step (seen on this host, independent of the kernels) does not move it
    stage_ms = {name: float(np.median(v)) for name, v in stage_runs.items()}
    stage_mean_ms = {name: float(np.mean(v)) for name, v in stage_runs.items()}
    counts = counts_log[args.warmup:].cpu().numpy()
    counts_all = counts.astype(np.int64)
    nodes = counts[:, : H + 1].astype(np.int64)
    edges = counts[:, H + 1: 2 * H + 1].astype(np.int64)
    elapsed_ms, (total_edges_all, _, _) = combine_ranks(torch, elapsed_ms, [timed_edges, hits, misses], dev)
    value = total_edges_all / (elapsed_ms / 1e3)

    # ---- roofline bookkeeping (outside the timed region) ----
    link = measure_link(sg, torch, dev, stream) if w.host_features else None
    # the link roofline is the faster of the two ways of reading pinned memory
    link_gbs = max(link.values()) if link else None
    hash_rate = measure_hash(sg, torch, dev, stream)
    deg = np.diff(g.indptr)
    # exact algorithmic bytes need the distinct srcs of each block: rerun the
    # measured batches' sampling (deterministic) and count them on the host
    n_book = min(args.steps, 32)  # bookkeeping on the first timed steps
    uniq_src = np.zeros((n_book, H), np.int64)
    hashed = np.zeros((n_book, H), np.int64)
    for s in range(n_book):
        i = args.warmup + s
        with torch.cuda.stream(stream):
            load_batch(i)
            pipe.sample(stream)
        torch.cuda.synchronize(dev)
        uq = pipe.buf.unique[: nodes[s, H]].cpu().numpy()
        for h in range(1, H + 1):
            idx = pipe.buf.idx[h - 1][: edges[s, h - 1]].cpu().numpy()
            uniq_src[s, h - 1] = len(np.unique(idx))
            # every distinct node of the frontier V_{h-1} is sampled once
            d = deg[frontier_ids(counts_all[s], uq, H, n_sub, h - 1)]
            hashed[s, h - 1] = int(d[d > w.fanouts[h - 1]].sum())
    n_H = nodes[:, H].astype(np.float64)
    gather_hbm = (8.0 * n_H).sum() + hits * R + n_H.sum() * R
    gather_host = misses * R
    t_gather = stage_ms["gather"] * args.steps / 1e3
    roof_gather_t = max(gather_hbm / (hbm_peak * 1e9), gather_host / (link_gbs * 1e9) if link_gbs else 0.0)
    # per-launch bytes averaged over the bookkeeping steps, times averaged over all timed steps
    bn, be = nodes[:n_book], edges[:n_book]
    stage_roof = {}
    stage_roof["gather"] = {"bound": "host_link" if link_gbs and gather_host / link_gbs > gather_hbm / hbm_peak else "hbm",
                            "achieved_hbm_gbs": gather_hbm / t_gather / 1e9,
                            "achieved_host_gbs": gather_host / t_gather / 1e9,
                            "frac": roof_gather_t / t_gather}
    for h in range(H, 0, -1):
        byt = float(((bn[:, h - 1] + 1) * 4 + be[:, h - 1] * 4 + uniq_src[:, h - 1] * R + bn[:, h - 1] * R).mean())
        t = stage_ms["fwd%d" % h] / 1e3
        stage_roof["fwd%d" % h] = {"bound": "hbm", "bytes_per_launch": byt,
                                   "achieved_gbs": byt / t / 1e9, "frac": byt / t / 1e9 / hbm_peak,
                                   "per_edge_gbs": float((be[:, h - 1] * R).mean()) / t / 1e9}
    for h in range(1, H + 1):
        # transposed row pointer, dst per edge, weight per edge, gdst rows, gsrc rows
        byt = float(((bn[:, h] + 1) * 4 + be[:, h - 1] * 8 + bn[:, h - 1] * R + bn[:, h] * R).mean())
        t = stage_ms["bwd%d" % h] / 1e3
        stage_roof["bwd%d" % h] = {"bound": "hbm", "bytes_per_launch": byt,
                                   "achieved_gbs": byt / t / 1e9, "frac": byt / t / 1e9 / hbm_peak}
    if upd is not None:
        # A = the dst rows' own states and their means (n_{H-1} x 2d), W, and
        # the fp32 output (n_{H-1} x 128); 2 * n * 2d * 128 flops
        t = stage_ms["update%d" % H] / 1e3
        rows = bn[:, H - 1].astype(np.float64)
        byt = float((rows * 2 * R + 128 * 2 * R + rows * 128 * 4).mean())
        flops = float((2.0 * rows * 2 * w.dim * 128).mean())
        # tensor peak for the arithmetic used: tf32 for fp32 rows (the recipe's
        # nominal tf32 : bf16 ratio, 1.1 : 2.25, times the measured bf16 burst),
        # bf16 measured burst otherwise
        bf16_peak = measured_bf16_tflops()
        tc_peak = bf16_peak * (1.1 / 2.25 if w.dtype == "f32" else 1.0) if bf16_peak else None
        stage_roof["update%d" % H] = {
            "bound": "hbm", "bytes_per_launch": byt, "achieved_gbs": byt / t / 1e9, "frac": byt / t / 1e9 / hbm_peak,
            "flops_per_launch": flops, "achieved_tflops": flops / t / 1e12,
            "tensor_peak_tflops": tc_peak, "tensor_frac": (flops / t / 1e12) / tc_peak if tc_peak else None,
            "arithmetic": "tf32 (tcgen05 kind::tf32)" if w.dtype == "f32" else "bf16 (tcgen05 kind::f16)"}
    t_sample = stage_ms["sample"] / 1e3
    calls = float(hashed.sum(axis=1).mean()) / 4.0
    stage_roof["sample"] = {"bound": "alu", "hash_calls_per_step": calls, "hash_calls_per_s": calls / t_sample,
                            "peak_hash_calls_per_s": hash_rate, "frac": (calls / t_sample) / hash_rate}
    dom = max(stage_ms, key=lambda k: stage_ms[k])
    if dom == "gather":
        ach_bytes = (gather_host if stage_roof["gather"]["bound"] == "host_link" else gather_hbm) / args.steps
        peak = link_gbs if stage_roof["gather"]["bound"] == "host_link" else hbm_peak
        roof = {"kernel": "gather stage (%s a step)" % ("k_gather" if pipe.gather_ws[0] is None else
                                                         "k_gather, k_region_scan, k_region_scatter, k_gather_list"),
                "bound": stage_roof["gather"]["bound"],
                "achieved": ach_bytes / (stage_ms["gather"] / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                "frac": stage_roof["gather"]["frac"],
                "traffic": gather_traffic(hits / args.steps, misses / args.steps),
                "traffic_unit": "DRAM bytes per step of k_gather and k_gather_list, scaled per hit and per miss from "
                                "the ncu capture in profiles/k_gather_host_misses.md",
                "peak_kind": ("measured host link, same run (%s, the faster of zero-copy loads and the copy engine)"
                              % max(link, key=link.get)) if stage_roof["gather"]["bound"] == "host_link"
                else "of " + peak_kind}
    elif dom.startswith("fwd") or dom.startswith("bwd"):
        r = stage_roof[dom]
        roof = {"kernel": dom, "bound": "hbm", "achieved": r["achieved_gbs"], "peak": hbm_peak, "unit": "GB/s",
                "frac": r["frac"], "traffic": None, "peak_kind": "of " + peak_kind}
    else:
        r = stage_roof["sample"]
        issue_peak = philox_issue_peak(torch, dev)
        roof = {"kernel": "sampler (k_sample does the hashing)", "bound": "alu",
                "achieved": r["hash_calls_per_s"] / 1e9, "peak": hash_rate / 1e9, "unit": "G Philox calls/s",
                "frac": r["frac"], "traffic": sampler_traffic(),
                "traffic_unit": "DRAM bytes per step (3 k_sample launches, ncu)",
                "peak_kind": "measured: the same Philox4x32-10 loop alone across the GPU (sg_hash_probe), same run",
                "issue_limit_estimate": issue_peak / 1e9,
                "issue_limit_note": "not measured: SMs x 4 x 32 lanes x max SM clock / %d instructions a call"
                                    % PHILOX_INSTR}

    result = {
        "metric": METRIC, "value": value, "unit": "sampled edges/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "timed_regions": {"repeats": repeats, "median_ms": elapsed_ms, "min_ms": min(region_ms),
                          "max_ms": max(region_ms), "seconds": sum(region_ms) / 1e3,
                          "step_ms_percentiles": None if not step_ms else
                          {q: float(np.percentile(step_ms, q)) for q in (10, 50, 90, 99, 100)},
                          "note": "the timed region of `steps` steps runs `repeats` times on new batches until "
                                  "%.1f s have elapsed; the line reports the median region by throughput"
                                  % args.min_seconds},
        "scaling": "weak", "vs_baseline": None, "dtype": "int32 sampling / " + w.dtype + " features, fp32 accumulation",
        "data": "synthetic Chung-Lu graph and N(0,1) features (seeded); no dataset",
        "config": {"workload": "%s: %d nodes, %d edges, exponent %.1f, mean %.0f, dim %d %s, fanouts %s, batch %s, "
                               "cache %d rows (%.0f%%)" % (w.name, g.n, g.m, w.gamma, w.mean_deg, w.dim, w.dtype,
                                                          w.fanouts, "%d x %d (super-batch)" % (n_sub, w.batch)
                                                          if n_sub > 1 else "%d" % w.batch,
                                                          cache_rows, 100.0 * cache_rows / w.n_nodes),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (CSR %.0f MB, features %.0f MB); a new batch every step"
                         % ((g.indptr.nbytes + g.indices.nbytes) / 1e6, w.n_nodes * R / 1e6)},
        "batch_latency_ms": latency_ms,
        "overlap": (("%d pipelines in turn, gathers one after another (misses come from a host table read by "
                     "region, which concurrent gathers would interleave): batch i+1 is sampled and transposed while "
                     "batch i gathers; batch i+1's forward waits for batch i's backward" % depth) if ov.serial_gathers
                    else ("%d pipelines in turn: batch i+1 is sampled, transposed and gathered while batch i's forward "
                          "and backward run; batch i+1's forward waits for batch i's backward" % depth) if depth > 1
                    else "none: one batch at a time, a step graph each") +
                   ". batch_latency_ms is one batch alone (a step graph per batch, batches back to back)",
        "presample": presample,
        "recoded": W.rank_of is not None,
        "host_table": None if not w.host_features else {
            "bytes": w.n_nodes * R,
            "huge_page_bytes": getattr(getattr(W.feat, "_sg_owner", None), "huge", 0),
            "locked": getattr(getattr(W.feat, "_sg_owner", None), "locked", False),
            "allocation": "huge-page mmap + cudaHostRegister" if hasattr(W.feat, "_sg_owner") else "cudaHostAlloc"},
        "gathered_feature_gbs": n_H.sum() * R / (elapsed_ms / 1e3) / 1e9,
        "gather_kernel_gbs": n_H.sum() * R / t_gather / 1e9,
        "memory_roofline_frac": {k: v["frac"] for k, v in stage_roof.items()},
        "hit_rate": hits / max(1, hits + misses),
        "stage_ms": stage_ms,
        "stage_mean_ms": stage_mean_ms,
        "stage_note": "per-stage times (median over the steps; stage_mean_ms: the means) from a third timed region "
                      "replaying per-stage graphs in sequence, one batch at a time (the headline overlaps batches; "
                      "within a batch the transposes overlap gather and forward)",
        "stages": stage_roof,
        "update_note": update_note,
        "roofline": roof,
        "host_link_gbs": link_gbs,
        "host_link": None if not link else dict(link, roofline=max(link, key=link.get)),
        "per_step": {"nodes": nodes.mean(axis=0).tolist(), "edges": edges.mean(axis=0).tolist()},
        "gpu_launches": kernels_per_step(H, n_sub, pipe.gather_ws[0] is not None, ov.pipes[0].split_gather)
                        * args.steps,
        "clocks": clk,
    }
    if rank == 0 and not args.no_e2e:
        # end-to-end regions on batches none of the earlier regions used
        e2e_first = n_batches + repeats * args.steps

        def e2e_pool(k):
            lo = e2e_first + k * n_batches
            ids = replica_batches(rank, world, lo + n_batches)[lo:]
            sh = np.stack([np.concatenate([W.seeds(b * n_sub + q) for q in range(n_sub)]) for b in ids])
            return sh.astype(np.int32), [w.sampler_seed(b) for b in ids]
        result["e2e"] = measure_e2e(sg, torch, ov, e2e_pool, dev, args, H, w)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return result, W


def measure_link(sg, torch, dev, stream, nbytes=4 << 30):
    """Host-link read rates of a pinned host buffer: zero-copy (sg_read_probe,
    16-byte loads from the device) and the copy engine (cudaMemcpyAsync host
    to device of the same buffer), best of three each, in GB/s."""
    host = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    host.fill_(1)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = {"zero_copy": None, "copy_engine": None}
    with torch.cuda.stream(stream):
        for kind in best:
            for _ in range(3):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                if kind == "zero_copy":
                    sg.sg_read_probe(host.data_ptr(), nbytes, sink, stream)
                else:
                    dst.copy_(host, non_blocking=True)
                b.record(stream)
                b.synchronize()
                gbs = nbytes / (a.elapsed_time(b) / 1e3) / 1e9
                best[kind] = gbs if best[kind] is None else max(best[kind], gbs)
    del host, dst
    return best


def measure_hash(sg, torch, dev, stream, n_calls=1 << 30):
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    best = None
    with torch.cuda.stream(stream):
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            sg.sg_hash_probe(n_calls, 7, sink, stream)
            b.record(stream)
            b.synchronize()
            r = n_calls / (a.elapsed_time(b) / 1e3)
            best = r if best is None else max(best, r)
    return best


def measure_e2e(sg, torch, ov, pool, dev, args, H, w, min_regions=3):
    """Same metric through the public API with host buffers: per step the
    seeds go host -> device from pinned memory and the step's result (the
    seed rows H_0 and the counts) comes back device -> host, with batches
    overlapped as in the headline (OverlappedPipeline, its CUDA graphs).  The
    host reads step j's result after enqueuing step j + depth, so the device
    always has the next step queued (step j's result was copied out on its
    pipeline's stream before that pipeline is reused).  The pinned result
    buffers form a ring of depth + 2 sets.  Like the device-timed headline,
    the region of warmup + steps steps repeats on new batches (pool(k) gives
    region k's seeds and hash seeds) until at least min_regions have run and
    --min-seconds / 2 have elapsed; the median region by throughput is
    reported, every region's figure beside it."""
    B = ov.pipes[0].n_seeds
    lag = ov.depth + 1
    ring = lag + 1
    p0 = ov.pipes[0]
    out_rows = [torch.empty((B, w.dim), dtype=p0.dtype, pin_memory=True) for _ in range(ring)]
    out_counts = [torch.empty(p0.buf.counts.numel(), dtype=torch.int32, pin_memory=True) for _ in range(ring)]
    done = [torch.cuda.Event() for _ in range(ring)]

    def region(seeds_host, hseeds):
        h_seeds = torch.from_numpy(seeds_host).pin_memory()
        h_hseed = torch.tensor(hseeds, dtype=torch.int64).pin_memory()

        def inputs(i):
            def f(p, s):
                p.seeds[:B].copy_(h_seeds[i], non_blocking=True)
                p.d_seed.copy_(h_hseed[i: i + 1], non_blocking=True)
            return f

        def after(i):
            k = i % ring

            def f(p, s):
                out_rows[k].copy_(p.h_feat[0][:B], non_blocking=True)
                out_counts[k].copy_(p.buf.counts, non_blocking=True)
                done[k].record(s)
            return f

        torch.cuda.synchronize(dev)
        n = len(seeds_host)
        edges = 0
        t0 = time.perf_counter()
        for i in range(n + lag):
            if i < n:
                ov.step(inputs(i), after(i))
            j = i - lag + 1  # the oldest step not read yet, once `lag` steps are in flight
            if i >= lag - 1 and j < n:
                done[j % ring].synchronize()
                edges += int(out_counts[j % ring][H + 1: 2 * H + 1].sum())
        dt = time.perf_counter() - t0
        for s in ov.streams:
            sg.sg_stream_check(s)
        return edges / dt, dt / n * 1e3, n

    regions, spent, k = [], 0.0, 0
    while len(regions) < min_regions or spent < args.min_seconds / 2:
        seeds_host, hseeds = pool(k)
        regions.append(region(seeds_host, hseeds))
        spent += regions[-1][1] * regions[-1][2] / 1e3
        k += 1
    med = sorted(regions)[len(regions) // 2]
    return {"value": med[0], "unit": "sampled edges/s", "ms_per_step": med[1], "steps": med[2],
            "regions": len(regions), "region_values": [r[0] for r in regions],
            "h2d_bytes_per_step": B * 4 + 8, "d2h_bytes_per_step": B * w.row_bytes + p0.buf.counts.numel() * 4,
            "note": "per step: seeds copied in from pinned memory, the step's two CUDA graphs (batches overlapped "
                    "on %d pipelines), H_0 and the counts copied out to pinned memory; the host reads step j's result "
                    "after enqueuing step j + %d; the median of %d regions of %d steps on new batches"
                    % (ov.depth, lag - 1, len(regions), med[2])}


# ------------------------------------------------------ NEXT rows measured
def run_next_experiments(args):
    """The dynamic cache (GARDEN Eq. (5)-(6)) and Match-Reorder (FastGL) on
    the workload, against the static cache the headline uses, with the same
    HBM budget: one JSON line with "impl": "experiment" (not the headline).
    Each gather is timed alone with CUDA events (median over the batches)."""
    import torch
    from sampling_gnn_mini_gb300 import binding as sg
    from sampling_gnn_mini_gb300.pipeline import MiniBatchPipeline

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sg.load(build_if_missing=True)
    W, G, cache, presample = setup_workload(args, sg, torch, dev)
    w = W.w
    H = w.n_hops
    if w.n_sub != 1 or w.cache_rows >= w.n_nodes:
        return {"impl": "experiment", "config": w.name, "skipped": "needs one mini-batch a step and a host table"}
    pipe = MiniBatchPipeline(G, cache, w.fanouts, w.batch, backward=False, device=dev, split_gather=False)
    cap = pipe.bounds.max_nodes[H]
    ws = sg.aligned_workspace(sg.sg_gather_workspace(cache, cap)) if sg.sg_gather_workspace(cache, cap) else None
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    outs = [torch.empty((cap, w.dim), dtype=dt, device=dev) for _ in range(2)]

    def timed(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        return a.elapsed_time(b)

    def sample(b):
        pipe.set_batch(torch.from_numpy(W.seeds(b)).to(dev), w.sampler_seed(b))
        pipe.sample()
        n = int(pipe.counts[H].item())
        return pipe.buf.unique[:n].clone()

    # ---- Match-Reorder over groups of batches
    Gn = min(max(args.group, 2), 32)
    groups = max(1, args.steps // Gn)
    match_map = torch.full((w.n_nodes,), -1, dtype=torch.int32, device=dev)
    mask = torch.zeros(w.n_nodes, dtype=torch.int32, device=dev)
    pos = torch.empty(cap, dtype=torch.int32, device=dev)
    stats = torch.zeros(2, dtype=torch.int64, device=dev)
    reused = torch.zeros(1, dtype=torch.int64, device=dev)
    mr = {"natural": {"overlap": [], "ms": [], "reused": 0, "misses": 0, "rows": 0},
          "greedy": {"overlap": [], "ms": [], "reused": 0, "misses": 0, "rows": 0},
          "plain": {"ms": [], "misses": 0, "rows": 0}}
    t_overlap = []
    for gi in range(groups):
        lists = [sample(gi * Gn + k) for k in range(Gn)]
        off = np.concatenate([[0], np.cumsum([x.numel() for x in lists])])
        ids = torch.cat(lists)
        O = None

        def ov():
            nonlocal O
            O = sg.sg_overlap(ids, off, mask)
        t_overlap.append(timed(ov))
        Oh = O.cpu().numpy()
        order = sg.sg_greedy_order(Oh, 0)
        for name, seq in (("natural", list(range(Gn))), ("greedy", list(order))):
            for k in range(1, Gn):
                mr[name]["overlap"].append(Oh[seq[k - 1], seq[k]] / Oh[seq[k], seq[k]])
            prev = None
            for k, b in enumerate(seq):
                cur, out = lists[b], outs[k % 2]
                stats.zero_()
                reused.zero_()
                if prev is None:
                    sg.sg_gather(cache, cur, cur.numel(), None, out, stats, workspace=ws)
                else:
                    def f():
                        sg.sg_match(lists[prev], lists[prev].numel(), None, cur, cur.numel(), None, match_map, pos)
                        sg.sg_gather_reuse(cache, cur, cur.numel(), None, pos, outs[(k - 1) % 2], out, stats, reused,
                                           workspace=ws)
                    mr[name]["ms"].append(timed(f))
                    h, m = stats.cpu().tolist()
                    mr[name]["reused"] += int(reused.item())
                    mr[name]["misses"] += m
                    mr[name]["rows"] += cur.numel()
                prev = b
        for b in range(1, Gn):  # the same batches without reuse
            stats.zero_()
            mr["plain"]["ms"].append(timed(lambda: sg.sg_gather(cache, lists[b], lists[b].numel(), None, outs[0],
                                                               stats, workspace=ws)))
            mr["plain"]["misses"] += int(stats[1].item())
            mr["plain"]["rows"] += lists[b].numel()
        del lists, ids
    sg.sg_stream_check()
    match_reorder = {"group": Gn, "groups": groups, "overlap_ms_median": float(np.median(t_overlap))}
    for name in ("natural", "greedy"):
        d = mr[name]
        match_reorder[name] = {"mean_overlap_with_previous": float(np.mean(d["overlap"])),
                               "reused_row_share": d["reused"] / max(1, d["rows"]),
                               "host_misses_a_batch": d["misses"] / max(1, len(d["ms"])),
                               "match_plus_gather_ms_median": float(np.median(d["ms"]))}
    match_reorder["no_reuse"] = {"host_misses_a_batch": mr["plain"]["misses"] / max(1, len(mr["plain"]["ms"])),
                                 "gather_ms_median": float(np.median(mr["plain"]["ms"]))}

    # ---- dynamic cache: static C - K plus dynamic K against static C
    C = w.cache_rows
    K = max(1, int(args.dyn_frac * C))
    g_q16 = max(1, min(65536, int(round(args.dyn_gamma * 65536))))
    dtype_code = sg.SG_F32 if w.dtype == "f32" else sg.SG_BF16
    cache2 = sg.sg_cache_build(W.feat, None, dtype_code, w.n_nodes, w.dim, None, C - K)
    sg.sg_dyn_cache_create(cache2, K, g_q16, args.dyn_window)
    ws2 = sg.aligned_workspace(sg.sg_gather_workspace(cache2, cap)) if ws is not None else None
    n_b = max(args.dyn_window * 4, args.steps)
    rows_s = {"static": [], "dynamic": []}
    ms_s = {"static": [], "dynamic": []}
    upd_ms = []
    base = 100000  # batches after the Match-Reorder ones
    for b in range(n_b):
        cur = sample(base + b)
        for name, c, wsx in (("static", cache, ws), ("dynamic", cache2, ws2)):
            stats.zero_()
            ms = timed(lambda: sg.sg_gather(c, cur, cur.numel(), None, outs[0], stats, workspace=wsx))
            h, m = stats.cpu().tolist()
            rows_s[name].append((h, m))
            ms_s[name].append(ms)
        t = timed(lambda: sg.sg_dyn_cache_batch(cache2, cur, cur.numel(), None))
        if (b + 1) % args.dyn_window == 0:
            upd_ms.append(t)
    sg.sg_stream_check()
    half = n_b // 2  # after the first windows have filled the dynamic set

    def rate(v):
        h = sum(x[0] for x in v[half:])
        m = sum(x[1] for x in v[half:])
        return h / max(1, h + m)
    dyn = {"budget_rows": C, "dynamic_rows": K, "gamma": g_q16 / 65536.0, "window": args.dyn_window,
           "batches": n_b, "hit_rate_static_only": rate(rows_s["static"]),
           "hit_rate_static_plus_dynamic": rate(rows_s["dynamic"]),
           "gather_ms_median_static_only": float(np.median(ms_s["static"][half:])),
           "gather_ms_median_static_plus_dynamic": float(np.median(ms_s["dynamic"][half:])),
           "window_update_ms_median": float(np.median(upd_ms)) if upd_ms else None,
           "note": "rates and times over the second half of the batches; the window update (Eq. (5) fold, Top-K of "
                   "Eq. (6) by radix selection over the nonzero scores, admission of entering rows from the host "
                   "table) runs once a window"}
    return {"impl": "experiment", "config": w.name, "match_reorder": match_reorder, "dynamic_cache": dyn,
            "presample": presample}


# -------------------------------------------------------------- CPU baseline
def run_oracle_steps(W, batches, budget_s):
    """The oracle's whole step (sample+relabel, gather, forward and backward
    chains in fp64) on the given batches, stopping once budget_s is spent.  A
    step of a super-batch config is its n_sub mini-batches with the shared
    hash seed (a super-batch equals that many separate runs)."""
    import oracle
    w, g = W.w, W.g
    feat = W.feat.numpy() if w.dtype == "f32" else W.feat.view(__import__("torch").int16).numpy().view(np.uint16)
    edges, done, t0 = 0, 0, time.perf_counter()
    for b in batches:
        for k in range(w.n_sub):
            seeds = W.seeds(b * w.n_sub + k)
            r = oracle.sampler_run(g.indptr, g.indices, seeds, w.fanouts, w.sampler_seed(b))
            x = oracle.gather(feat, r.unique)
            hh = x
            for h in range(w.n_hops, 0, -1):
                hh, _ = oracle.aggregate_fwd(r.indptr[h - 1], r.idx[h - 1],
                                             hh.astype(np.float32) if hh.dtype != np.uint16 else hh)
            gg = hh.astype(np.float32)
            for h in range(1, w.n_hops + 1):
                gg, _ = oracle.aggregate_bwd(r.indptr[h - 1], r.idx[h - 1], r.hop_off[h], gg.astype(np.float32))
            edges += sum(len(i) for i in r.idx)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return edges, done, dt


def cpu_baseline(W, budget_s):
    import oracle
    edges, done, dt = run_oracle_steps(W, range(5000, 6000), budget_s)
    return {"value": edges / dt, "unit": "sampled edges/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d %s %s, whole step (sample+relabel, gather, %d-hop forward and backward), %.1f s"
                      % (done, W.w.name, "batches" if W.w.n_sub == 1 else "super-batches of %d" % W.w.n_sub,
                         W.w.n_hops, dt)}


def run_reference(args, rank, world, budget_s: float = 150.0):
    """The oracle, as it stands, on the same workload: at least one warm-up
    batch, then the timed steps one batch (or super-batch) each until
    budget_s of oracle time is spent (at least one step)."""
    if rank != 0:
        return None
    import oracle
    W = Workload(args.config, pinned_features=False)
    w = W.w
    run_oracle_steps(W, range(max(1, min(args.warmup, 3))), 0.0)
    edges, done, dt = 0, 0, 0.0
    for s in range(args.steps):
        e, d, t = run_oracle_steps(W, [args.warmup + s], 0.0)
        edges, done, dt = edges + e, done + d, dt + t
        if dt > budget_s:
            break
    value = edges / dt
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "sampled edges/s", "n_gpus": world,
            "steps": done, "warmup": args.warmup, "ms_per_step": dt / done * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int32 sampling / fp64 sums (CPU oracle)",
            "data": "synthetic Chung-Lu graph and N(0,1) features (seeded); no dataset",
            "config": {"workload": "%s (same graph, features and batches as the GPU arm)" % w.name},
            "cpu_baseline": {"value": value, "unit": "sampled edges/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": "%d %s, one whole step each (at most %.0f s of oracle time)" % (
                                 done, "batches" if w.n_sub == 1 else "super-batches of %d" % w.n_sub, budget_s)},
            "e2e": {"value": value, "unit": "sampled edges/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.experiment == "next":
        if rank == 0:
            print(json.dumps(run_next_experiments(args)), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    res, W = run_ours(args, rank, world, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(W, args.cpu_seconds)
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
