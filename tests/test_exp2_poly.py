"""Accuracy of the software 2^x the forward kernel runs on the FMA pipe.

Requirement: maximum relative error <= 2^-9 over [-127, 0]; checked exhaustively
over every fp32 value in that interval (about 1.1e9 values) against 2^x in
fp64 (torch's fp64 exp2 on the device for the sweep, numpy's on the host for the
worst point and for a random sample): the mathematical definition, to far below
fp32 resolution."""
import numpy as np
import pytest
import torch

import exact_attention_blackwell_gb300 as fa

pytestmark = pytest.mark.gpu

LIMIT = 2.0 ** -9


def eval_gpu(x_cpu: torch.Tensor) -> torch.Tensor:
    x = x_cpu.cuda()
    y = torch.empty_like(x)
    assert fa.fa_exp2_poly(x, y, x.numel()) == fa.FA_OK
    torch.cuda.synchronize()
    return y


def test_special_values():
    x = torch.tensor([0.0, -0.0, -1.0, -0.5, 0.5, -126.0, -127.0, -149.0, -150.0, -151.0, -1000.0,
                      float("-inf"), 8.0, 63.0], dtype=torch.float32)
    y = eval_gpu(x).cpu().numpy()
    assert y[0] == 1.0 and y[1] == 1.0
    assert y[2] == pytest.approx(0.5, rel=2e-4) and y[5] == pytest.approx(2.0 ** -126, rel=2e-4)
    assert y[6] == pytest.approx(2.0 ** -127, rel=2e-4)
    assert y[9] == 0.0 and y[10] == 0.0 and y[11] == 0.0
    assert y[12] == pytest.approx(256.0, rel=2e-4) and y[13] == pytest.approx(2.0 ** 63, rel=2e-4)


def test_exhaustive_relative_error():
    # every fp32 in [-127, 0]: the bit patterns 0x80000000 (= -0.0) .. bits(-127.0)
    lo = np.array([-0.0], np.float32).view(np.uint32)[0]
    hi = np.array([-127.0], np.float32).view(np.uint32)[0]
    chunk = 1 << 27
    worst = 0.0
    worst_x = None
    for start in range(int(lo), int(hi) + 1, chunk):
        stop = min(start + chunk, int(hi) + 1)
        bits = torch.arange(start, stop, dtype=torch.int64, device="cuda").to(torch.int32)
        x = bits.view(torch.float32)
        y = torch.empty_like(x)
        assert fa.fa_exp2_poly(x, y, x.numel()) == fa.FA_OK
        ref = torch.exp2(x.double())
        rel = ((y.double() - ref).abs() / ref)
        m, i = rel.max(dim=0)
        if m.item() > worst:
            worst, worst_x = m.item(), x[i].item()
    # spot-check the device fp64 reference against numpy on the worst point
    assert worst <= LIMIT, f"max relative error {worst:.3e} at x={worst_x}"
    yw = eval_gpu(torch.tensor([worst_x], dtype=torch.float32)).double().item()
    assert abs(yw / np.exp2(np.float64(worst_x)) - 1.0) <= LIMIT
    print(f"exp2_poly max relative error over [-127, 0]: {worst:.3e} (2^{np.log2(worst):.2f}) at x={worst_x}")


def test_random_points_against_numpy():
    g = torch.Generator().manual_seed(5)
    x = -127.0 * torch.rand(1 << 22, generator=g, dtype=torch.float64)
    x32 = x.float()
    y = eval_gpu(x32).cpu().numpy().astype(np.float64)
    ref = np.exp2(x32.numpy().astype(np.float64))
    assert (np.abs(y / ref - 1.0) <= LIMIT).all()
