"""Parity of the SAGE UPDATE forward (sg_sage_fwd, tcgen05) with the oracle.

Tolerances follow the arithmetic: fp32 inputs go through the tensor cores as
tf32 (10 stored mantissa bits), so each product carries a relative error of at
most about 2^-10 and an output within 2e-3 of the sum of |terms| is right;
bf16 products are exact in fp32 and only the fp32 accumulation rounds
(1e-5 of the sum of |terms|)."""
import numpy as np
import pytest
import torch

import oracle
from sampling_gnn_mini_gb300 import binding as sg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()


def _bf16_bits(a):
    return (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _dev(a, bf16):
    if bf16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


@pytest.mark.parametrize("n,d,bf16", [(300, 100, False), (257, 256, False), (130, 64, True), (1, 8, True)])
def test_sage_fwd_matches_oracle(n, d, bf16):
    # ragged row tiles (n not a multiple of 128) and ragged K tiles (d = 100:
    # columns past d zero-filled by the copy engine)
    rng = np.random.default_rng(n + d)
    h = rng.standard_normal((n, d)).astype(np.float32)
    m = rng.standard_normal((n, d)).astype(np.float32)
    W = (rng.standard_normal((128, 2 * d)) / np.sqrt(2 * d)).astype(np.float32)
    if bf16:
        h, m, W = _bf16_bits(h), _bf16_bits(m), _bf16_bits(W)
    y_ref, out_ref, am = oracle.sage_fwd(h, m, W)
    out = torch.full((n, 128), 7.0, device="cuda")
    y = torch.full((n, 128), 7.0, device="cuda")
    sg.sg_sage_fwd(_dev(h, bf16), _dev(m, bf16), _dev(W, bf16), n, None, out, y)
    sg.sg_stream_check()
    yg = y.cpu().numpy().astype(np.float64)
    og = out.cpu().numpy().astype(np.float64)
    tol = 1e-5 if bf16 else 2e-3
    assert np.all(np.abs(yg - y_ref) <= tol * am + 1e-30)
    assert np.array_equal(og, np.maximum(yg, 0))


def test_sage_fwd_uses_device_count_and_optional_preactivation():
    rng = np.random.default_rng(3)
    n_cap, n, d = 400, 150, 32
    h = rng.standard_normal((n_cap, d)).astype(np.float32)
    m = rng.standard_normal((n_cap, d)).astype(np.float32)
    W = (rng.standard_normal((128, 2 * d)) / 8).astype(np.float32)
    _, out_ref, am = oracle.sage_fwd(h[:n], m[:n], W)
    out = torch.full((n_cap, 128), 7.0, device="cuda")
    d_n = torch.tensor([n], dtype=torch.int32, device="cuda")
    sg.sg_sage_fwd(_dev(h, False), _dev(m, False), _dev(W, False), n_cap, d_n, out)
    sg.sg_stream_check()
    og = out.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(og[:n] - out_ref) <= 2e-3 * am + 1e-30)
    assert np.all(og[n:] == 7.0)


def test_sage_fwd_rejects_unsupported_shapes():
    h = torch.zeros((4, 6), device="cuda")  # 24-byte rows: not a multiple of 16
    W = torch.zeros((128, 12), device="cuda")
    out = torch.zeros((4, 128), device="cuda")
    with pytest.raises(sg.SgError):
        sg.sg_sage_fwd(h, h, W, 4, None, out)
    W64 = torch.zeros((64, 16), device="cuda")  # d_out != 128
    h8 = torch.zeros((4, 8), device="cuda")
    with pytest.raises(sg.SgError):
        sg.sg_sage_fwd(h8, h8, W64, 4, None, out)


# ------------------------------------------------------------ backward
def _bwd_case(n, d, bf16, seed):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((n, d)).astype(np.float32)
    m = rng.standard_normal((n, d)).astype(np.float32)
    W = (rng.standard_normal((128, 2 * d)) / np.sqrt(2 * d)).astype(np.float32)
    g = rng.standard_normal((n, 128)).astype(np.float32)
    if bf16:
        h, m, W = _bf16_bits(h), _bf16_bits(m), _bf16_bits(W)
    return h, m, W, g


def _run_bwd(h, m, W, g, y64, n_cap, n, bf16):
    """sg_sage_bwd on the first n of n_cap rows; returns dW, dh, dm (numpy)."""
    d = h.shape[1]
    dev = lambda a: _dev(np.ascontiguousarray(a), bf16)  # noqa: E731
    y = torch.from_numpy(np.ascontiguousarray(y64.astype(np.float32))).cuda()
    dW = torch.full((128, 2 * d), 7.0, device="cuda")
    dh = torch.full((n_cap, d), 7.0, device="cuda")
    dm = torch.full((n_cap, d), 7.0, device="cuda")
    ws = sg.aligned_workspace(sg.sg_sage_bwd_workspace(n_cap, d, sg.SG_BF16 if bf16 else sg.SG_F32))
    d_n = None if n == n_cap else torch.tensor([n], dtype=torch.int32, device="cuda")
    sg.sg_sage_bwd(dev(h), dev(m), dev(W), n_cap, d_n, y, torch.from_numpy(np.ascontiguousarray(g)).cuda(), dW, dh,
                   dm, ws)
    sg.sg_stream_check()
    return dW.cpu().numpy(), dh.cpu().numpy(), dm.cpu().numpy()


@pytest.mark.parametrize("n,d,bf16", [(300, 100, False), (257, 256, False), (130, 64, True), (1, 8, True),
                                      (1000, 128, True)])
def test_sage_bwd_matches_oracle(n, d, bf16):
    # ragged row tiles and K splits (n not a multiple of 128 or of a K tile),
    # ragged column tiles of dh/dm (2d not a multiple of 128); the oracle's own
    # pre-activation decides the ReLU mask on both sides (ReLU'(0) = 0)
    h, m, W, g = _bwd_case(n, d, bf16, n * 3 + d)
    y_ref, _, _ = oracle.sage_fwd(h, m, W)
    y32 = y_ref.astype(np.float32).astype(np.float64)
    dW_ref, am_w, dh_ref, dm_ref, am_z = oracle.sage_bwd(h, m, W, y32, g)
    dW, dh, dm = _run_bwd(h, m, W, g, y32, n, n, bf16)
    # tf32 rounds both operands (2^-10 each); bf16 rounds dY (2^-9)
    tol = 1e-2 if bf16 else 2e-3
    assert np.all(np.abs(dW - dW_ref) <= tol * am_w + 1e-30)
    dz = np.hstack([dh, dm])
    assert np.all(np.abs(dz - np.hstack([dh_ref, dm_ref])) <= tol * am_z + 1e-30)


def test_sage_bwd_uses_device_count_and_is_deterministic():
    n_cap, n, d = 700, 333, 96
    h, m, W, g = _bwd_case(n_cap, d, False, 11)
    y_ref, _, _ = oracle.sage_fwd(h[:n], m[:n], W)
    y_full = np.zeros((n_cap, 128))
    y_full[:n] = y_ref
    y_full[n:] = 1.0  # rows past the device count must not contribute to dW
    y32 = y_full.astype(np.float32).astype(np.float64)
    dW_ref, am_w, dh_ref, dm_ref, am_z = oracle.sage_bwd(h[:n], m[:n], W, y32[:n], g[:n])
    runs = [_run_bwd(h, m, W, g, y32, n_cap, n, False) for _ in range(2)]
    dW, dh, dm = runs[0]
    assert np.all(np.abs(dW - dW_ref) <= 2e-3 * am_w + 1e-30)
    assert np.all(np.abs(np.hstack([dh[:n], dm[:n]]) - np.hstack([dh_ref, dm_ref])) <= 2e-3 * am_z + 1e-30)
    assert np.all(dh[n:] == 7.0) and np.all(dm[n:] == 7.0)  # rows past the count are not written
    for a, b in zip(runs[0], runs[1]):  # dW's splits are added in a fixed order
        assert np.array_equal(a, b)
