"""Seeded input generators: reproducible, distinct per (step, replica), right dtypes and
distributions.  CPU only."""
from fractions import Fraction

import numpy as np
import torch

from bitwise_reproducible_step_gb300 import inputs as I
from tests import exact as X


def test_reproducible_and_distinct():
    wl = I.WORKLOADS["flat1m_r4"]
    a = I.gen_grad(wl, 1, 0, n=10000)
    b = I.gen_grad(wl, 1, 0, n=10000)
    c = I.gen_grad(wl, 1, 1, n=10000)
    d = I.gen_grad(wl, 2, 0, n=10000)
    assert torch.equal(a, b)
    assert not torch.equal(a, c) and not torch.equal(a, d)
    assert abs(a.std().item() - 1e-3) < 1e-4


def test_dtypes_and_distributions():
    n = 200000
    t = I.gen_grad(I.WORKLOADS["flat12m8_r8_student_t"], 1, 0, n=n)
    assert t.dtype == torch.float32
    # Student-t(3) has heavy tails: kurtosis far above the normal's 3
    x = t.double() / 1e-3
    assert (x.abs() > 6).float().mean() > 1e-3
    s = I.gen_grad(I.WORKLOADS["flat1200m_r8_segscale"], 1, 0, n=3 * 4_194_304 + 5)
    scales = I.segment_scales(I.WORKLOADS["flat1200m_r8_segscale"], s.numel(), "cpu")
    assert scales.numel() == 4
    assert torch.all(scales >= 1e-10 * 0.999) and torch.all(scales <= 1e-6 * 1.001)
    b = I.gen_grad(I.WORKLOADS["flat3000m_r8_bf16_spiked_shards"], 1, 0, n=n)
    assert b.dtype == torch.bfloat16
    frac = (b.float().abs() > 1e-4 * 20).float().mean().item()
    assert 0.005 < frac < 0.015


def test_state_and_shards():
    wl = I.WORKLOADS["flat1m_r4"]
    w, m, v = I.gen_state(wl, n=5000)
    assert abs(w.std().item() - 0.02) < 2e-3 and not m.any() and not v.any()
    r = I.shard_ranges(3_000_000_000, 8)
    assert r[0] == (0, 375_000_000) and r[-1][1] == 3_000_000_000
    assert all(r[i][1] == r[i + 1][0] for i in range(7))


def test_hparam_bits_are_nearest_fp32():
    # round the exact decimal (not a double) to fp32
    for name, dec in [("lr", "3e-4"), ("beta1", "0.9"), ("beta2", "0.999"), ("eps", "1e-8"),
                      ("wd", "0.1"), ("clip", "1.0")]:
        assert X.bits(X.f32(Fraction(dec))) == I.HPARAM_BITS[name]


def test_bf16_to_numpy_bits():
    x = torch.tensor([1.0, -2.5, 3e-5], dtype=torch.bfloat16)
    u = I.to_numpy(x)
    assert u.dtype == np.uint16
    assert np.array_equal((u.astype(np.uint32) << 16).view(np.float32), x.float().numpy())
