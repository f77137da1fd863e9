"""Seeded random configurations of the whole step on the GPU, every slot against the oracle.

Each case draws, from its own seed, a parameter count (from 1 to about 300K, with sizes at
and around the 4096-element chunk), a replica count, the gradient and parameter dtypes,
the arithmetic mode (IEEE or flush-to-zero), the leaf hash (PF61 or BLAKE2b), an optional
decay mask, gradient scales down to the subnormal range, and a split of the parameter
range into 1 to 4 ranges at arbitrary (chunk-cutting) boundaries, reduced and updated
range by range.  Two consecutive steps; after each, g, the chunk sums, w, m, v, every leaf,
the norm and the root are compared with the oracle's own trajectory (tests/oracle_full.py),
0 differing slots.  The options interact here in combinations the other tests take one
at a time."""
import numpy as np
import pytest
import torch

from bitwise_reproducible_step_gb300 import inputs as I
from bitwise_reproducible_step_gb300 import repstep as rs
from tests import gpu_util as U
from tests import oracle_full as OF

pytestmark = pytest.mark.gpu

CH = 4096


@pytest.fixture(scope="module", autouse=True)
def _built():
    U.ensure_built()
    torch.cuda.set_device(0)


def draw(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.choice([1, 17, CH - 1, CH, CH + 1, 3 * CH + 5, 16 * CH + 33,
                        int(rng.integers(1, 300_000)), int(rng.integers(1, 300_000)),
                        int(rng.integers(1, 300_000))]))
    R = int(rng.choice([1, 2, 3, 5, 8, 12, 32]))
    cfg = dict(n=n, R=R, gbf16=bool(rng.random() < 0.4), wbf16=bool(rng.random() < 0.3),
               ftz=bool(rng.random() < 0.3), audit=bool(rng.random() < 0.3),
               scale=float(10.0 ** rng.uniform(-22, 2)))
    if n > 1 and rng.random() < 0.4:
        k = int(rng.integers(1, min(4, n)))
        cuts = sorted(set(int(x) for x in rng.integers(1, n, size=k)))
        cfg["segments"] = [(0, bool(rng.random() < 0.5))] + [(c, bool(rng.random() < 0.5))
                                                             for c in cuts]
    else:
        cfg["segments"] = None
    parts = int(rng.integers(1, 5)) if n > 1 else 1
    cuts = sorted(set(int(x) for x in rng.integers(1, max(n, 2), size=parts - 1))) if n > 1 else []
    bounds = [0] + cuts + [n]
    cfg["ranges"] = [(a, b) for a, b in zip(bounds, bounds[1:]) if b > a] or [(0, n)]
    return cfg


def to_host_w(w):
    if w.dtype == torch.bfloat16:
        return w.view(torch.int16).cpu().numpy().view(np.uint16)
    return w.cpu().numpy()


@pytest.mark.parametrize("seed", range(64))
def test_random_configuration_matches_oracle(seed):
    cfg = draw(1000 + seed)
    n, R = cfg["n"], cfg["R"]
    dev = torch.device("cuda", 0)
    gdt = torch.bfloat16 if cfg["gbf16"] else torch.float32
    ctx = rs.Repstep(n, grad_dtype=gdt, device=dev,
                     param_dtype=torch.bfloat16 if cfg["wbf16"] else torch.float32,
                     subnormals=rs.SUBNORMALS_FTZ if cfg["ftz"] else rs.SUBNORMALS_IEEE,
                     hash_mode=rs.HASH_BLAKE2B if cfg["audit"] else rs.HASH_PF61)
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
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    for t in (1, 2):
        grads = U.gen_grads(n, R, 40 + t + seed, gdt, scale=cfg["scale"] * (1 + 99 * (t == 2)))
        hp = U.hp_for(t)
        for a, b in cfg["ranges"]:
            ctx.reduce(grads, begin=a, count=b - a)
        ctx.clip(hp.clip, norm_out=norm)
        for a, b in cfg["ranges"]:
            ctx.adamw(w, m, v, hp, begin=a, count=b - a)
        ctx.root(t, root_out=root)
        ctx.sync()
        rep = fo.step(grads, t, U.HP, dict(g=ctx.g_view(), chunk_sums=ctx.chunk_sums_view(),
                                           leaves=ctx.leaves_view(), w=w, m=m, v=v, norm=norm,
                                           root=root))
        OF.assert_identical(rep, f"seed {seed} {cfg} step {t}")
    fo.close()
