"""The C-ABI library builds, loads and exports every symbol that
include/sg.h declares (no GPU needed; no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "sg.h")).read()
    return sorted(set(re.findall(r"^\s*(?:sg_status|int32_t|size_t)\s+(sg_\w+)\s*\(", src, re.M)))


def test_header_declares_the_pipeline_calls():
    names = _declared()
    for call in ("sg_graph_load", "sg_sampler_run", "sg_relabel", "sg_cache_build", "sg_gather",
                 "sg_aggregate_fwd", "sg_aggregate_bwd"):
        assert call in names


def test_library_exports_every_declared_symbol():
    from sampling_gnn_mini_gb300 import binding
    lib = binding.load()
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(binding.EXPORTS) == _declared()


def test_host_only_calls():
    from sampling_gnn_mini_gb300 import binding
    lib = binding.load()
    assert lib.sg_version() >= 100
    assert lib.sg_relabel_workspace(10, 100) > 0
    assert lib.sg_relabel_workspace(-1, 5) == 0
    assert lib.sg_aggregate_bwd_workspace(10, 20, 50) > 0
    # argument errors are reported without touching a device
    b = binding._Bounds()
    fan = (ctypes.c_int32 * 2)(10, 5)
    assert lib.sg_sampler_bounds(None, 4, None, 1, fan, 2, ctypes.byref(b)) == binding.SG_ERR_INVALID_ARG
    assert "NULL graph" in binding.sg_last_error()
    out = ctypes.c_void_p()
    assert lib.sg_graph_load(None, 32, None, 10, 0, ctypes.byref(out)) == binding.SG_ERR_INVALID_ARG
    assert lib.sg_cache_build(None, None, 0, 10, 4, None, 10, ctypes.byref(out), None) == binding.SG_ERR_INVALID_ARG


def test_built_for_sm103a():
    from sampling_gnn_mini_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in build.ARCH
    build.build()
    assert os.path.exists(build.LIB)


def test_product_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "sampling_gnn_mini_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "orc_" not in text, f
