"""Failure detection on the GPU, in the forms that fault, trap or hang no GPU.

- A bounded device wait is made to run out: sg_wait_probe runs the look-back
  of the library's single-pass scans with one tile that never publishes and a
  short spin limit.  The waits behind it give up, the device error word says
  SG_ERR_TIMEOUT, and the stream and the library stay usable.
- An allocation failure is injected on the host (SG_FAULT_INJECT=alloc:N) at
  each allocation of sg_graph_load and sg_cache_build in turn, in a child
  process: the call returns SG_ERR_OOM, frees what it had allocated, and the
  next call succeeds.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from sampling_gnn_mini_gb300 import binding as sg

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()


def _prefixes(n):
    t = np.arange(n, dtype=np.int64)
    return t * (t + 1) // 2


def test_wait_probe_completes_when_every_tile_publishes():
    for n in (1, 33, 1000):
        out = torch.full((n,), -1, dtype=torch.int32, device="cuda")
        sg.sg_wait_probe(n, -1, 1 << 12, out)
        sg.sg_stream_check()
        assert np.array_equal(out.cpu().numpy(), _prefixes(n))


@pytest.mark.parametrize("n,silent", [(64, 5), (300, 0), (300, 298), (2000, 1000)])
def test_bounded_wait_runs_out_and_reports_timeout(n, silent):
    # at least one tile follows the silent one, so some look-back must wait
    out = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    sg.sg_wait_probe(n, silent, 1 << 10, out)
    with pytest.raises(sg.SgError) as e:
        sg.sg_stream_check()
    assert e.value.status == sg.SG_ERR_TIMEOUT
    got = out.cpu().numpy()
    assert np.array_equal(got[:silent], _prefixes(n)[:silent])  # tiles before the silent one are exact
    assert got[silent] == -1
    # the error word was cleared by the check, and the stream is usable
    sg.sg_stream_check()
    out2 = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    sg.sg_wait_probe(n, -1, 1 << 12, out2)
    sg.sg_stream_check()
    assert np.array_equal(out2.cpu().numpy(), _prefixes(n))


def test_wait_probe_rejects_bad_arguments():
    out = torch.zeros(8, dtype=torch.int32, device="cuda")
    for n, lim in ((0, 10), (5000, 10), (8, 0), (8, (1 << 22) + 1)):
        with pytest.raises(sg.SgError) as e:
            sg.sg_wait_probe(n, -1, lim, out)
        assert e.value.status == sg.SG_ERR_INVALID_ARG


CHILD = r"""
import sys
import numpy as np, torch
sys.path.insert(0, %(root)r)
from sampling_gnn_mini_gb300 import binding as sg
sg.load()
torch.cuda.init()
n = 1 << 20
ip = np.arange(n + 1, dtype=np.int32) * 8
ix = (np.arange(n * 8, dtype=np.int64) * 7919 %% n).astype(np.int32)
ranked = np.arange(0, n, 2, dtype=np.int32)
hfeat = torch.zeros((n, 32), dtype=torch.float32).pin_memory()
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
what = sys.argv[1]
try:
    if what == "graph":
        sg.sg_graph_load(ip, ix)
    else:
        sg.sg_cache_build(hfeat, None, sg.SG_F32, n, 32, ranked, len(ranked))
    first = "ok"
except sg.SgError as e:
    first = str(e.status)
torch.cuda.synchronize()
leak = free0 - torch.cuda.mem_get_info()[0]
# the next call (past the injected failure) succeeds
if what == "graph":
    g = sg.sg_graph_load(ip, ix); ok = g.n_edges == n * 8
else:
    c = sg.sg_cache_build(hfeat, None, sg.SG_F32, n, 32, ranked, len(ranked)); ok = c.n_cache == len(ranked)
print(first, leak, ok)
"""


@pytest.mark.parametrize("what,n_allocs", [("graph", 3), ("cache", 4)])
def test_injected_oom_at_every_owned_allocation(what, n_allocs):
    for k in range(1, n_allocs + 1):
        env = dict(os.environ)
        env["SG_FAULT_INJECT"] = "alloc:%d" % k
        r = subprocess.run([sys.executable, "-c", CHILD % {"root": ROOT}, what], env=env, capture_output=True,
                           text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        first, leak, ok = r.stdout.strip().split()[-3:]
        assert first == str(sg.SG_ERR_OOM), (what, k, r.stdout)
        assert int(leak) < (2 << 20), (what, k, leak)  # what was allocated before the failure was freed
        assert ok == "True"
