"""Seeded random configurations of the single-pass step (repstep_step_fused) on the GPU,
every slot against the oracle.

Each case draws, from its own seed, a parameter count (from 1 to about 300K, with sizes at
and around the 4096-element chunk), a replica count (mostly 4, 8 or 16, which the single
pass covers; sometimes another, which takes the two passes), the gradient and
parameter dtypes, the arithmetic mode (IEEE or flush-to-zero), the leaf hash (PF61 or
BLAKE2b), an optional decay mask, whether the root passes run on a second stream, and per step a gradient scale
from the subnormal range up to one that clips.  Four consecutive steps with the two state
buffers alternating and no synchronisation between them; afterwards every step's norm and
root, and the final w, m, v, chunk sums and leaves, are compared with the oracle's own
trajectory (tests/oracle_full.py): 0 differing slots.  The clip pattern over the steps
takes every path of the clip prediction."""
import numpy as np
import pytest
import torch

from bitwise_reproducible_step_gb300 import inputs as I
from bitwise_reproducible_step_gb300 import repstep as rs
from tests import gpu_util as U
from tests import oracle_full as OF

pytestmark = pytest.mark.gpu

CH = 4096
STEPS = 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    U.ensure_built()
    torch.cuda.set_device(0)


def draw(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.choice([1, 17, CH - 1, CH, CH + 1, 2 * CH + 2049, 16 * CH + 33,
                        int(rng.integers(1, 300_000)), int(rng.integers(1, 300_000)),
                        int(rng.integers(1, 300_000))]))
    R = int(rng.choice([4, 8, 4, 8, 16, 32, 3, 12]))
    cfg = dict(n=n, R=R, gbf16=bool(rng.random() < 0.4), wbf16=bool(rng.random() < 0.4),
               ftz=bool(rng.random() < 0.4), audit=bool(rng.random() < 0.25),
               hash_stream=bool(rng.random() < 0.5),
               # per step: small (no clip), subnormal-range, or clipping gradients
               scales=[float(rng.choice([10.0 ** rng.uniform(-6, -3), 10.0 ** rng.uniform(-44, -38),
                                         10.0 ** rng.uniform(1, 3)]))
                       for _ in range(STEPS)])
    if n > 1 and rng.random() < 0.4:
        k = int(rng.integers(1, min(4, n)))
        cuts = sorted(set(int(x) for x in rng.integers(1, n, size=k)))
        cfg["segments"] = [(0, bool(rng.random() < 0.5))] + [(c, bool(rng.random() < 0.5))
                                                             for c in cuts]
    else:
        cfg["segments"] = None
    return cfg


def to_host_w(w):
    if w.dtype == torch.bfloat16:
        return w.view(torch.int16).cpu().numpy().view(np.uint16)
    return w.cpu().numpy()


@pytest.mark.parametrize("seed", range(32))
def test_random_fused_configuration_matches_oracle(seed):
    cfg = draw(5000 + seed)
    n, R = cfg["n"], cfg["R"]
    dev = torch.device("cuda", 0)
    gdt = torch.bfloat16 if cfg["gbf16"] else torch.float32
    ctx = rs.Repstep(n, grad_dtype=gdt, device=dev,
                     param_dtype=torch.bfloat16 if cfg["wbf16"] else torch.float32,
                     subnormals=rs.SUBNORMALS_FTZ if cfg["ftz"] else rs.SUBNORMALS_IEEE,
                     hash_mode=rs.HASH_BLAKE2B if cfg["audit"] else rs.HASH_PF61)
    if cfg["hash_stream"]:
        ctx.set_hash_stream(torch.cuda.Stream(dev))
    if cfg["segments"]:
        ctx.set_decay_mask(rs.decay_mask_from_segments(n, cfg["segments"]).to(dev))
    w32, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    m.copy_(I.gen_grad(U.F32_WL, 9, 0, n=n, device=dev))          # mid-run moments
    v.copy_(I.gen_grad(U.F32_WL, 9, 1, n=n, device=dev).square())
    w = w32.to(torch.bfloat16) if cfg["wbf16"] else w32
    fo = OF.FullOracle(n, R, to_host_w(w), m.cpu().numpy(), v.cpu().numpy(),
                       grad_dtype="bf16" if cfg["gbf16"] else "f32",
                       param_dtype="bf16" if cfg["wbf16"] else "f32",
                       hash_mode=1 if cfg["audit"] else 0, ftz=cfg["ftz"],
                       segments=cfg["segments"], threads=4, slab=4 * CH)
    bufs = [(w, m, v), tuple(torch.empty_like(x) for x in (w, m, v))]
    norms = torch.empty(STEPS, dtype=torch.float32, device=dev)
    roots = torch.empty(STEPS, dtype=torch.int64, device=dev)
    grads = [U.gen_grads(n, R, 300 + 7 * seed + t, gdt, scale=cfg["scales"][t - 1])
             for t in range(1, STEPS + 1)]
    for t in range(1, STEPS + 1):
        ctx.step_fused(grads[t - 1], *bufs[(t - 1) % 2], *bufs[t % 2], U.hp_for(t), step=t,
                       norm_out=norms[t - 1:t], root_out=roots[t - 1:t])
    assert ctx.sync() & ~rs.FLAG_NONFINITE_NORM == 0
    nb = norms.cpu().numpy().view(np.uint32)
    rb = roots.cpu().numpy().view(np.uint64)
    for t in range(1, STEPS + 1):
        last = t == STEPS
        gpu = None
        if last:
            wo, mo, vo = bufs[t % 2]
            gpu = dict(chunk_sums=ctx.chunk_sums_view(), leaves=ctx.leaves_view(), w=wo, m=mo,
                       v=vo, norm=norms[t - 1:t], root=roots[t - 1:t])
        rep = fo.step(grads[t - 1], t, U.HP, gpu)
        what = f"seed {seed} {cfg} step {t}"
        assert rep["norm"]["oracle"] == f"{int(nb[t - 1]):08x}", what
        assert rep["root"]["oracle"] == f"{int(rb[t - 1]):016x}", what
        if last:
            OF.assert_identical(rep, what)
    fo.close()
