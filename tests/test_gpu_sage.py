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
