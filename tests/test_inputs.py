"""Pins for the seeded input generator and the e4m3 quantiser it applies.

The e4m3 format (3 mantissa bits, largest finite value 448, smallest subnormal
2^-9) fixes the round-trip error: at most half an ulp, i.e. 2^-4 of |x| for
normal codes and 2^-10 (times the scale) in the subnormal range.
"""

import numpy as np
import torch

import synthetic


def test_seeded_and_deterministic():
    c = synthetic.custom_case(2, 3, 40, 40, 64, False, "bf16", seed=5)
    a, b = synthetic.make_inputs(c), synthetic.make_inputs(c)
    for n in ("q", "k", "v"):
        assert torch.equal(a[n], b[n])
    assert a["q"].dtype == torch.bfloat16 and a["q"].shape == (2, 40, 3, 64)


def test_bf16_is_rounded_randn():
    c = synthetic.custom_case(1, 2, 16, 16, 64, False, "bf16", seed=9)
    x = synthetic.make_inputs(c)
    g = torch.Generator().manual_seed(9)
    q32 = torch.randn((1, 16, 2, 64), generator=g)
    assert torch.equal(x["q"], q32.to(torch.bfloat16))


def test_e4m3_quantiser_bounds():
    c = synthetic.custom_case(2, 4, 1024, 1024, 128, False, "e4m3", seed=31)
    g = torch.Generator().manual_seed(31)
    x = synthetic._draw(g, (2, 1024, 4, 128), outliers=True)
    codes, ds = synthetic.quantize_e4m3_per_head(x)
    assert codes.dtype == torch.float8_e4m3fn and ds.shape == (2, 4)
    cf = codes.to(torch.float64)
    # the per-(b,h) maximum maps to the largest finite code exactly
    assert torch.all(cf.abs().amax(dim=(1, 3)) == 448.0)
    xd = x.to(torch.float64)
    s = ds.to(torch.float64)[:, None, :, None]
    y = xd / s
    err = (y - cf).abs()
    normal = y.abs() >= 2.0 ** -6
    assert torch.all(err[normal] <= 2.0 ** -4 * y.abs()[normal] * (1 + 1e-6))
    assert torch.all(err[~normal] <= 2.0 ** -10 * (1 + 1e-6))
    # outlier rate: 0.1% of entries scaled by 10
    g = torch.Generator().manual_seed(31)
    torch.randn((2, 1024, 4, 128), generator=g)
    u = torch.rand((2, 1024, 4, 128), generator=g)
    rate = (u < synthetic.OUTLIER_RATE).double().mean().item()
    assert 0.0008 < rate < 0.0012
    assert c.outliers


def test_sample_rows_cover_edges():
    c = synthetic.CASES["C3"]
    r = synthetic.sample_rows(c, 256)
    assert r.shape == (256, 3)
    for i in (0, 1, 127, 128, 129, c.N_q - 1):
        assert i in set(r[:, 2].tolist())
    assert r[:, 0].max() < c.B and r[:, 1].max() < c.H and r[:, 2].max() < c.N_q


def test_case_flops():
    assert synthetic.CASES["C4"].flops == 4 * 16 * 16384 * 16384 * 128 / 2
    assert synthetic.CASES["C5"].flops == 4 * 2 * 16 * 8192 * 8192 * 128
