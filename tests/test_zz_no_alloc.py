"""The relabel entry point that allocates nothing (sg_relabel_noalloc).

It exists for callers that may not allocate device memory themselves or ask
the library to: code running inside another framework's allocator, under a
fixed device-memory budget, or where an allocation would synchronise the
device.  Its scratch is a static device array inside the library, shared by
every call.  This file checks, through the C ABI, that calls in a row give
exactly what the oracle's first-occurrence relabel gives, and what the
workspace-taking sg_relabel gives (integer output, so the tolerance is exact
equality): a smaller call after a larger one (the scratch keeps the larger
call's contents), a call exactly at the size limit, and calls with no IDs or
no prefix.  Requests above the fixed limit, and outputs too small for the
request, are refused with a clear error.  It is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
from sampling_gnn_mini_gb300 import binding as sg

pytestmark = pytest.mark.gpu

LIMIT = sg.SG_RELABEL_NOALLOC_MAX_IDS


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _case(seed, n_prefix, n_ids, id_range):
    rng = np.random.default_rng(seed)
    prefix = rng.permutation(id_range)[:n_prefix].astype(np.int32)
    ids = rng.integers(0, id_range, size=n_ids).astype(np.int32)
    if n_prefix and n_ids:
        ids[::4] = prefix[rng.integers(0, n_prefix, size=len(ids[::4]))]
    return prefix, ids


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()


def _check(prefix, ids):
    """One sg_relabel_noalloc call against the oracle and sg_relabel."""
    want_u, want_l = oracle.relabel(ids, prefix)
    unique = torch.full((max(1, len(ids) + len(prefix)),), -1, dtype=torch.int32, device="cuda")
    local = torch.full((max(1, len(ids)),), -1, dtype=torch.int32, device="cuda")
    n_unique = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    sg.sg_relabel_noalloc(_dev(ids), _dev(prefix), unique, local, n_unique)
    sg.sg_stream_check()
    n = int(n_unique.item())
    assert n == len(want_u)
    assert np.array_equal(unique[:n].cpu().numpy(), want_u)
    assert np.array_equal(local[: len(ids)].cpu().numpy(), want_l)
    if len(ids) or len(prefix):  # the workspace-taking call agrees
        ref_u, ref_l, ref_n = sg.sg_relabel(_dev(ids), _dev(prefix))
        assert int(ref_n.item()) == n
        assert torch.equal(unique[:n], ref_u[:n])
        assert torch.equal(local[: len(ids)], ref_l[: len(ids)])


def test_noalloc_matches_oracle_on_calls_in_a_row():
    # larger then smaller then larger again: each call clears what it uses of
    # the shared scratch, so the previous call's contents never show
    for prefix, ids in (_case(1, 3000, 120000, 500000), _case(2, 17, 250000, 40000), _case(3, 500, 900, 2000),
                        _case(4, 40, 200000, 1 << 24)):
        _check(prefix, ids)


def test_noalloc_exactly_at_the_limit():
    prefix, ids = _case(5, 4096, LIMIT - 4096, 3 * LIMIT)
    assert len(prefix) + len(ids) == LIMIT
    _check(prefix, ids)
    _check(*_case(6, 10, 1000, 5000))  # and a small call right after it


def test_noalloc_prefix_only_and_ids_only():
    _check(*_case(7, 5000, 0, 100000))   # no IDs: the prefix alone
    _check(*_case(8, 0, 70000, 30000))   # no prefix: first occurrence from 0
    _check(*_case(9, 0, 0, 10))          # nothing at all


def test_noalloc_refuses_requests_above_its_limit():
    n = LIMIT + 1
    ids = torch.zeros(n, dtype=torch.int32, device="cuda")
    prefix = torch.zeros(0, dtype=torch.int32, device="cuda")
    out = torch.zeros(n, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(sg.SgError) as e:
        sg.sg_relabel_noalloc(ids, prefix, out, out, cnt)
    assert e.value.status == sg.SG_ERR_INVALID_ARG
    assert "static scratch limit" in str(e.value)


def test_noalloc_refuses_outputs_too_small_or_of_the_wrong_type():
    ids = _dev(np.arange(100))
    prefix = _dev(np.arange(1000, 1010))
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    good_u = torch.zeros(110, dtype=torch.int32, device="cuda")
    good_l = torch.zeros(100, dtype=torch.int32, device="cuda")
    bad = [(torch.zeros(109, dtype=torch.int32, device="cuda"), good_l, cnt),   # unique one short
           (good_u, torch.zeros(99, dtype=torch.int32, device="cuda"), cnt),    # local one short
           (good_u, good_l, torch.zeros(0, dtype=torch.int32, device="cuda")),  # no count
           (good_u.to(torch.int64), good_l, cnt),                               # wrong type
           (good_u, good_l.cpu(), cnt),                                         # host memory
           (torch.zeros(220, dtype=torch.int32, device="cuda")[::2], good_l, cnt)]  # not contiguous
    for u, l, c in bad:
        with pytest.raises(sg.SgError) as e:
            sg.sg_relabel_noalloc(ids, prefix, u, l, c)
        assert e.value.status == sg.SG_ERR_INVALID_ARG
