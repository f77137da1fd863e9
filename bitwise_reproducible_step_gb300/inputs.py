"""Seeded synthetic inputs for the optimizer step.

This module generates data only: replica gradients, initial weights and the
hyperparameter bit patterns.  It holds none of the step's arithmetic, imports neither the
CUDA binding nor the oracle, and is the one module both sides are fed from.

Generator: torch's Philox-based generators (`torch.Generator(device).manual_seed(s)`),
on whatever device the caller names.  The CUDA and CPU generators give different bits for
the same seed; parity never depends on that, because every comparison feeds the SAME bytes
to the CUDA path and to the oracle.

Seed of one buffer: s = (workload_id << 40) | (step << 20) | replica, with replica 0xFFFFF
for the initial weights and 0xFFFFE for per-run segment scales.  Long buffers are drawn in
fixed slices of 2^26 elements; slice j uses seed s | (j << 48).  The slice length is part
of the recipe, so a buffer's bits depend on (workload, step, replica, n) only.

Distributions (N(0, sigma) means standard deviation sigma, as in the Open-1B paper's §3.1,
whose weights are initialised with a standard deviation of 0.02):
  * normal            g = z * sigma
  * student_t3        g = sigma * z0 / sqrt((z1^2 + z2^2 + z3^2) / 3), in fp64, cast to fp32
  * normal_segscale   g = z * (sigma * 10^(-6 + 4U_seg)) with one U_seg ~ U(0,1) per
                      segment of `seg` elements, drawn once per run and shared by replicas
  * normal_spiked_bf16  g = z * sigma, times `spike` where a per-replica per-step
                      Bernoulli(spike_p) mask is set, then rounded to bf16 (RNE)
  weights w ~ N(0, 0.02) (not truncated); m = v = 0.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

SLICE = 1 << 26
W_REPLICA = 0xFFFFF
SEG_REPLICA = 0xFFFFE


def f32_from_bits(b: int) -> float:
    """Python float holding exactly the fp32 value with bit pattern b."""
    return float(np.array([b], dtype=np.uint32).view(np.float32)[0])


# fp32 bit patterns of the step's hyperparameters: the round-to-nearest fp32 values of
# lr 3e-4, beta1 0.9, beta2 0.999 (the checkpoint page's v EMA), eps 1e-8, weight decay
# 0.1 and clip 1.0 (Open-1B §3.2).  Bits, not decimals, so no parser rounds them twice.
HPARAM_BITS = dict(lr=0x399D4952, beta1=0x3F666666, beta2=0x3F7FBE77, eps=0x322BCC77,
                   wd=0x3DCCCCCD, clip=0x3F800000)


def default_hparams() -> dict:
    return {k: f32_from_bits(v) for k, v in HPARAM_BITS.items()}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wid: int              # workload id in the seed
    n: int                # flat fp32 parameters
    R: int                # replica gradient buffers
    grad: str             # distribution name (see module docstring)
    sigma: float
    steps: int
    grad_dtype: str = "f32"   # "f32" or "bf16"
    seg: int = 0
    spike_p: float = 0.0
    spike: float = 1.0
    topologies: tuple = ()    # (nodes, gpus_per_node) pairs, all with product R
    shards: int = 1           # contiguous shard ranges reduced and updated separately


WORKLOADS = {
    w.name: w for w in [
        Workload("flat1m_r4", 1, 1_048_576, 4, "normal", 1e-3, 3),
        Workload("flat12m8_r8_student_t", 2, 12_800_000, 8, "student_t3", 1e-3, 10),
        Workload("flat1200m_r8_segscale", 3, 1_200_000_000, 8, "normal_segscale", 1e-4, 5,
                 seg=4_194_304),
        Workload("flat268m_r32_topologies", 4, 268_435_456, 32, "normal", 1e-3, 3,
                 topologies=((1, 32), (4, 8), (8, 4), (32, 1))),
        Workload("flat3000m_r8_bf16_spiked_shards", 5, 3_000_000_000, 8, "normal_spiked_bf16",
                 1e-4, 3, grad_dtype="bf16", spike_p=0.01, spike=1e3, shards=8),
    ]
}


def seed_of(wid: int, step: int, replica: int) -> int:
    return (wid << 40) | (step << 20) | replica


def _gen(device, s: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def _slices(n: int):
    j = 0
    for lo in range(0, n, SLICE):
        yield j, lo, min(lo + SLICE, n)
        j += 1


def segment_scales(wl: Workload, n: int, device) -> torch.Tensor:
    """Per-segment fp32 multipliers sigma * 10^(-6 + 4U) (normal_segscale only)."""
    nseg = (n + wl.seg - 1) // wl.seg
    u = torch.rand(max(nseg, 1), generator=_gen(device, seed_of(wl.wid, 0, SEG_REPLICA)),
                   device=device, dtype=torch.float64)
    return (wl.sigma * torch.pow(10.0, -6.0 + 4.0 * u)).to(torch.float32)[:nseg]


def gen_grad(wl: Workload, step: int, replica: int, n: int | None = None,
             device="cpu", out: torch.Tensor | None = None) -> torch.Tensor:
    """One replica's gradient for `step` (fp32, or bf16 for bf16 workloads)."""
    n = wl.n if n is None else n
    dt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
    if out is None:
        out = torch.empty(n, dtype=dt, device=device)
    assert out.numel() == n and out.dtype == dt
    s = seed_of(wl.wid, step, replica)
    scales = segment_scales(wl, n, device) if wl.grad == "normal_segscale" else None
    for j, lo, hi in _slices(n):
        gen = _gen(device, s | (j << 48))
        m = hi - lo
        if wl.grad == "normal":
            x = torch.randn(m, generator=gen, device=device, dtype=torch.float32) * wl.sigma
        elif wl.grad == "student_t3":
            z = torch.randn(4, m, generator=gen, device=device, dtype=torch.float64)
            t = z[0] / torch.sqrt((z[1] * z[1] + z[2] * z[2] + z[3] * z[3]) / 3.0)
            x = (wl.sigma * t).to(torch.float32)
        elif wl.grad == "normal_segscale":
            z = torch.randn(m, generator=gen, device=device, dtype=torch.float32)
            idx = torch.arange(lo, hi, device=device) // wl.seg
            x = z * scales[idx]
        elif wl.grad == "normal_spiked_bf16":
            z = torch.randn(m, generator=gen, device=device, dtype=torch.float32) * wl.sigma
            spk = torch.rand(m, generator=gen, device=device) < wl.spike_p
            x = torch.where(spk, z * wl.spike, z)
        else:
            raise ValueError(wl.grad)
        out[lo:hi].copy_(x.to(dt))
    return out


def gen_state(wl: Workload, n: int | None = None, device="cpu"):
    """Initial (w, m, v): w ~ N(0, 0.02), m = v = 0, all fp32."""
    n = wl.n if n is None else n
    w = torch.empty(n, dtype=torch.float32, device=device)
    s = seed_of(wl.wid, 0, W_REPLICA)
    for j, lo, hi in _slices(n):
        w[lo:hi] = torch.randn(hi - lo, generator=_gen(device, s | (j << 48)), device=device,
                               dtype=torch.float32) * 0.02
    m = torch.zeros(n, dtype=torch.float32, device=device)
    v = torch.zeros(n, dtype=torch.float32, device=device)
    return w, m, v


def shard_ranges(n: int, shards: int):
    """Contiguous shard ranges [floor(s n / S), floor((s+1) n / S))."""
    return [(s * n // shards, (s + 1) * n // shards) for s in range(shards)]


def to_numpy(t: torch.Tensor) -> np.ndarray:
    """Host copy as numpy: fp32 stays float32, bf16 becomes its uint16 bit patterns."""
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()
