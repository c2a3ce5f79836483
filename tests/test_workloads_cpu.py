"""The seeded input generators: the same (seed, tensor, step) triple gives the same bytes,
and each draw has the distribution the workload recipe states (module docstring of
workloads.py), checked statistically on samples large enough that a wrong parameter
(a std off by a factor, a missing rescale, a wrong outlier count) fails."""
import math

import numpy as np
import torch

import workloads as wl


def test_generator_is_a_pure_function_of_the_triple():
    a = torch.randn(64, generator=wl.generator(4, "x", 0))
    b = torch.randn(64, generator=wl.generator(4, "x", 0))
    assert torch.equal(a, b)
    for other in (wl.generator(4, "x", 1), wl.generator(4, "y", 0), wl.generator(5, "x", 0)):
        assert not torch.equal(a, torch.randn(64, generator=other))


def test_normal_std_and_rounding():
    g = wl.generator(0, "normal-test")
    x = wl.normal((512, 512), 0.02, g)
    assert x.dtype == torch.float32
    assert abs(x.mean().item()) < 0.02 * 5 / 512
    assert abs(x.std().item() / 0.02 - 1) < 0.01
    # bf16 draws are the fp32 draws rounded to nearest even
    xb = wl.normal((512, 512), 0.02, wl.generator(0, "normal-test"), torch.bfloat16)
    assert torch.equal(xb, x.to(torch.bfloat16))


def test_student_t3_has_heavy_tails():
    x = wl.student_t3((1 << 20,), 0.5, wl.generator(2, "t3")).float()
    # t(3): median |t| = 0.7649 (so 0.3825 after x0.5); P(|t| > 5) = 0.01539, ~2.5e-6 for N(0,1)
    med = x.abs().median().item()
    assert abs(med / 0.38245 - 1) < 0.02
    frac = (x.abs() > 2.5).float().mean().item()
    assert abs(frac / 0.01539 - 1) < 0.1


def test_log_uniform_range_and_median():
    v = wl.log_uniform(1 << 16, 1e-3, 1e2, wl.generator(3, "lu"))
    assert v.dtype == torch.float32
    assert v.min().item() >= 1e-3 * (1 - 1e-6) and v.max().item() <= 1e2 * (1 + 1e-6)
    lv = torch.log10(v.double())
    assert abs(lv.median().item() - (-0.5)) < 0.05  # midpoint of log10 range [-3, 2]
    # uniform in log10: each decade holds a fifth of the values
    for d in range(-3, 2):
        f = ((lv >= d) & (lv < d + 1)).double().mean().item()
        assert abs(f - 0.2) < 0.01


def test_outliers_touch_exactly_the_stated_fraction():
    t = torch.ones((100, 1000), dtype=torch.bfloat16)
    o = wl.with_outliers(t, 1e-3, 1000.0, wl.generator(1, "out"))
    assert o.dtype == torch.bfloat16
    assert int((o == 1000.0).sum()) == 100 and int((o == 1.0).sum()) == 100 * 1000 - 100


def test_channel_scaled_normal_column_scales():
    g = wl.generator(3, "csn")
    x = wl.channel_scaled_normal(4096, 64, g).float()
    s = wl.log_uniform(64, 1e-3, 1e2, wl.generator(3, "csn"))  # the same first draw
    ratio = x.std(0) / s
    assert torch.all((ratio - 1).abs() < 0.06), ratio


def test_bf16_bits_round_trip():
    x = torch.tensor([1.0, -2.5, 65504.0, 1e-40], dtype=torch.float32).to(torch.bfloat16)
    b = wl.bf16_bits(x)
    assert b.dtype == np.uint16
    assert b[0] == 0x3F80 and b[1] == 0xC020
    back = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16)
    assert torch.equal(back, x)
    assert math.isclose(wl.host_array(x.float())[1], -2.5)
