"""Failure detection without a GPU fault (host side, no GPU needed).

An allocation failure is injected on the host (SG_FAULT_INJECT=alloc:N makes
the library's N-th owned allocation fail before it reaches the CUDA runtime),
in a child process, since the variable is read once per process.  The calls
must return SG_ERR_OOM, hand back no handle and say why.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import ctypes, sys
import numpy as np
sys.path.insert(0, %(root)r)
from sampling_gnn_mini_gb300 import binding as sg
lib = sg.load()
out = ctypes.c_void_p(12345)
ip = np.array([0, 1, 2], np.int32); ix = np.array([1, 0], np.int32)
which = sys.argv[1]
if which == "graph":
    st = lib.sg_graph_load(ip.ctypes.data, 32, ix.ctypes.data, 2, 2, ctypes.byref(out))
else:
    # every node cached from a device copy: no host-table query comes first
    st = lib.sg_cache_build(None, ctypes.c_void_p(1 << 20), sg.SG_F32, 2, 4, None, 2, ctypes.byref(out), None)
print(st, out.value is None, sg.sg_last_error())
"""


def _run(which, inject):
    env = dict(os.environ)
    env["SG_FAULT_INJECT"] = inject
    env["CUDA_VISIBLE_DEVICES"] = ""  # the injected failure must come before any device work
    r = subprocess.run([sys.executable, "-c", CHILD % {"root": ROOT}, which], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    st, no_handle, msg = r.stdout.strip().split(" ", 2)
    return int(st), no_handle == "True", msg


@pytest.mark.parametrize("which", ["graph", "cache"])
def test_injected_allocation_failure_returns_oom(which):
    from sampling_gnn_mini_gb300 import binding as sg
    st, no_handle, msg = _run(which, "alloc:1")
    assert st == sg.SG_ERR_OOM, msg
    assert no_handle
    assert "memory" in msg.lower()


def test_injection_variable_is_validated():
    from sampling_gnn_mini_gb300 import binding as sg
    # a malformed value injects nothing: the call then fails for want of a
    # device (no GPU is visible to the child), not with the injected OOM
    st, no_handle, msg = _run("graph", "alloc:x")
    assert st == sg.SG_ERR_CUDA and no_handle, msg
