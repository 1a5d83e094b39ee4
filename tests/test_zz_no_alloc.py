"""The relabel entry point that allocates nothing (sg_relabel_noalloc).

It exists for callers that may not allocate device memory themselves or ask
the library to: code running inside another framework's allocator, under a
fixed device-memory budget, or where an allocation would synchronise the
device.  Its scratch is a static device array inside the library, shared by
every call.  This file checks, through the C ABI, that two calls in a row
give exactly what the workspace-taking sg_relabel gives (integer output, so
the tolerance is exact equality), and that requests above its fixed limit
are refused with a clear error.  It is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from sampling_gnn_mini_gb300 import binding as sg

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _case(seed, n_prefix, n_ids, id_range):
    rng = np.random.default_rng(seed)
    prefix = rng.permutation(id_range)[:n_prefix].astype(np.int32)
    ids = rng.integers(0, id_range, size=n_ids).astype(np.int32)
    ids[::4] = prefix[rng.integers(0, max(1, n_prefix), size=len(ids[::4]))] if n_prefix else ids[::4]
    return prefix, ids


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()


def test_noalloc_matches_workspace_relabel_on_two_calls_in_a_row():
    cases = [_case(1, 3000, 120000, 500000), _case(2, 17, 250000, 40000)]
    for prefix, ids in cases:  # two calls in a row share the static scratch
        want_u, want_l, want_n = sg.sg_relabel(_dev(ids), _dev(prefix))
        unique = torch.full((len(ids) + len(prefix),), -1, dtype=torch.int32, device="cuda")
        local = torch.full((len(ids),), -1, dtype=torch.int32, device="cuda")
        n_unique = torch.zeros(1, dtype=torch.int32, device="cuda")
        sg.sg_relabel_noalloc(_dev(ids), _dev(prefix), unique, local, n_unique)
        sg.sg_stream_check()
        n = int(want_n.item())
        assert int(n_unique.item()) == n
        assert torch.equal(unique[:n], want_u[:n])
        assert torch.equal(local, want_l)
        assert torch.equal(unique[: len(prefix)].cpu(), torch.from_numpy(prefix))


def test_noalloc_refuses_requests_above_its_limit():
    n = sg.SG_RELABEL_NOALLOC_MAX_IDS + 1
    ids = torch.zeros(n, dtype=torch.int32, device="cuda")
    prefix = torch.zeros(0, dtype=torch.int32, device="cuda")
    out = torch.zeros(n, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(sg.SgError) as e:
        sg.sg_relabel_noalloc(ids, prefix, out, out, cnt)
    assert e.value.status == sg.SG_ERR_INVALID_ARG
    assert "static scratch limit" in str(e.value)
