"""Shared helpers for the GPU parity tests: build once, generate identical inputs for the
CUDA path and the oracle, and compare bit patterns (0 ulp; NaNs compared by class)."""
import numpy as np
import torch

from bitwise_reproducible_step_gb300 import inputs as I
from bitwise_reproducible_step_gb300 import repstep as rs
from oracle import oracle as O

HP = I.default_hparams()
F32_WL = I.WORKLOADS["flat1m_r4"]
BF16_WL = I.WORKLOADS["flat3000m_r8_bf16_spiked_shards"]


def ensure_built():
    from bitwise_reproducible_step_gb300 import build
    build.build()
    rs.lib()


def hp_for(t, clip=None):
    return rs.hparams(lr=HP["lr"], beta1=HP["beta1"], beta2=HP["beta2"], eps=HP["eps"],
                      weight_decay=HP["wd"], clip=HP["clip"] if clip is None else clip, t=t)


def bits32(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous().numpy()
    return np.ascontiguousarray(x).view(np.uint32)


def diff_report(got, want):
    """(differing slots, relFro, max|delta|) between two fp32 arrays -- the statistics of the
    cross-process reproducibility note ("The measurement" section)."""
    g = np.asarray(got, np.float32).astype(np.float64)
    w = np.asarray(want, np.float32).astype(np.float64)
    gb, wb = bits32(np.asarray(got, np.float32)), bits32(np.asarray(want, np.float32))
    both_nan = np.isnan(g) & np.isnan(w)
    differing = int(np.count_nonzero((gb != wb) & ~both_nan))
    fin = np.isfinite(g) & np.isfinite(w)
    with np.errstate(invalid="ignore"):          # inf - inf in the slots fin excludes
        d = np.where(fin, g - w, 0.0)
    den = np.linalg.norm(np.where(fin, w, 0.0))
    rel = float(np.linalg.norm(d) / den) if den > 0 else float(np.linalg.norm(d))
    mx = float(np.max(np.abs(d))) if d.size else 0.0
    return differing, rel, mx


def assert_same_f32(got, want, what=""):
    got = np.asarray(got.detach().cpu() if isinstance(got, torch.Tensor) else got, np.float32)
    want = np.asarray(want, np.float32)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    differing, rel, mx = diff_report(got, want)
    assert differing == 0, f"{what}: {differing} differing slots, relFro {rel:.3e}, max|d| {mx:.3e}"


def gen_grads(n, R, t, dtype=torch.float32, scale=1.0, device="cuda"):
    wl = BF16_WL if dtype == torch.bfloat16 else F32_WL
    out = []
    for r in range(R):
        g = I.gen_grad(wl, t, r, n=n, device=device)
        if scale != 1.0:
            g = (g.float() * scale).to(g.dtype)
        out.append(g.contiguous())
    return out


def oracle_grads(grads):
    return [I.to_numpy(g) for g in grads]


def root_of(t: torch.Tensor) -> int:
    return int(t.cpu().numpy().view(np.uint64)[0])


def oracle_step(grads_np, w, m, v, t, nodes=1, clip=None, hash_mode=0):
    return O.step(grads_np, w, m, v, lr=HP["lr"], beta1=HP["beta1"], beta2=HP["beta2"],
                  eps=HP["eps"], wd=HP["wd"], clip=HP["clip"] if clip is None else clip, t=t,
                  nodes=nodes, hash_mode=hash_mode)


def oracle_step_bf16w(grads_np, w16, m, v, t, clip=None, hash_mode=0):
    """One oracle step with bf16 parameters, composed from the oracle's pieces: reduce,
    norm, clip scale, AdamW on widened bf16 parameters with one rounding back, and the state
    hash over the widened parameters."""
    clip = HP["clip"] if clip is None else clip
    g = O.reduce(grads_np)
    nv = O.norm(g)
    sc = O.clip_scale(nv, clip)
    bc1, bc2 = O.bias_corrections(HP["beta1"], HP["beta2"], t)
    w16, m, v = O.adamw_bf16w(w16, m, v, g, sc, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"],
                              HP["wd"], bc1, bc2)
    wide = O.widen_bf16(w16)
    return dict(w16=w16, m=m, v=v, norm=nv, scale=sc, g=g,
                root=O.state_hash(t, wide, m, v, hash_mode),
                leaves=O.leaves(t, wide, m, v, hash_mode))


def bits16(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    return np.ascontiguousarray(x).view(np.uint16)


def assert_same_bf16(got, want, what=""):
    """bf16 bit patterns equal, NaNs compared by class."""
    gb, wb = bits16(got), bits16(want)
    assert gb.shape == wb.shape, (what, gb.shape, wb.shape)
    nan = lambda b: (b & 0x7FFF) > 0x7F80  # noqa: E731
    bad = (gb != wb) & ~(nan(gb) & nan(wb))
    assert not bad.any(), f"{what}: {int(bad.sum())} differing bf16 slots, first at " \
                          f"{int(np.argmax(bad))}"
