"""Per-segment weight decay ("OPEN-1B: A Fully Auditable Training Run", §3.2 optimizer
paragraph: no decay on embeddings, normalisation gains or RoPE) on the GPU: a device
bitmask built from a segment list, against the oracle's per-segment AdamW, bit for bit."""
import numpy as np
import pytest
import torch

from bitwise_reproducible_step_gb300 import inputs as I
from bitwise_reproducible_step_gb300 import repstep as rs
from oracle import oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    U.ensure_built()
    torch.cuda.set_device(0)


def model_like_segments(n):
    """A flat vector laid out like a small transformer: an embedding, then per block a
    norm gain, attention and MLP matrices; decay only on the matrices.  Boundaries fall on
    odd offsets, inside 4-element groups and inside 32-bit mask words."""
    segs, e, rng = [], 0, np.random.default_rng(9)
    segs.append((0, False))                      # embedding
    e = int(n * 0.11) | 1
    while e < n:
        segs.append((e, False))                  # norm gain
        e += int(rng.integers(3, 700))
        if e >= n:
            break
        segs.append((e, True))                   # matrices
        e += int(rng.integers(1000, max(1001, n // 6)))
    return segs


def oracle_masked(gnp, w, m, v, t, segs, bf16):
    g = O.reduce(gnp)
    nv = O.norm(g)
    sc = O.clip_scale(nv, U.HP["clip"])
    bc1, bc2 = O.bias_corrections(U.HP["beta1"], U.HP["beta2"], t)
    f = O.adamw_bf16w_segments if bf16 else O.adamw_segments
    w, m, v = f(w, m, v, g, sc, U.HP["lr"], U.HP["beta1"], U.HP["beta2"], U.HP["eps"], U.HP["wd"],
                bc1, bc2, segs)
    wide = O.widen_bf16(w) if bf16 else w
    return w, m, v, O.state_hash(t, wide, m, v)


@pytest.mark.parametrize("n,R,bf16", [(5, 2, False), (4097, 4, False), (123_457, 8, False),
                                      (123_457, 8, True), (3 * 4096 + 7, 3, True)])
def test_decay_mask_steps_match_oracle(n, R, bf16):
    segs = model_like_segments(n)
    pdt = torch.bfloat16 if bf16 else torch.float32
    ctx = rs.Repstep(n, device=DEV, param_dtype=pdt)
    ctx.set_decay_mask(rs.decay_mask_from_segments(n, segs).to(DEV))
    w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)
    w = w.to(pdt)
    ow = U.bits16(w) if bf16 else w.cpu().numpy()
    om, ov = m.cpu().numpy(), v.cpu().numpy()
    root = torch.empty(1, dtype=torch.int64, device=DEV)
    for t in (1, 2, 3):
        grads = U.gen_grads(n, R, t, scale=3000.0 if t == 2 else 1.0)
        ctx.step(grads, w, m, v, U.hp_for(t), step=t, root_out=root)
        ctx.sync()
        ow, om, ov, r = oracle_masked(U.oracle_grads(grads), ow, om, ov, t, segs, bf16)
        if bf16:
            U.assert_same_bf16(w, ow, f"w step {t}")
        else:
            U.assert_same_f32(w, ow, f"w step {t}")
        U.assert_same_f32(m, om, f"m step {t}")
        U.assert_same_f32(v, ov, f"v step {t}")
        assert U.root_of(root) == r, f"root step {t}"


def test_decay_mask_with_shard_ranges_and_reset():
    """Ranges cutting mask words and 4-element groups give the unsharded bits; clearing
    the mask restores decay everywhere (the plain step)."""
    n, R = 50_000, 4
    segs = model_like_segments(n)
    mask = rs.decay_mask_from_segments(n, segs).to(DEV)
    grads = U.gen_grads(n, R, 1, scale=2000.0)
    a = rs.Repstep(n, device=DEV)
    b = rs.Repstep(n, device=DEV)
    a.set_decay_mask(mask)
    b.set_decay_mask(mask)
    wa, ma, va = I.gen_state(U.F32_WL, n=n, device=DEV)
    w0 = wa.cpu().numpy()
    wb, mb, vb = wa.clone(), ma.clone(), va.clone()
    hp = U.hp_for(1)
    a.step(grads, wa, ma, va, hp, step=1)
    b.reduce(grads)
    b.clip(hp.clip)
    for lo, hi in [(0, 3), (3, 4101), (4101, 4102), (4102, 33_333), (33_333, 50_000)]:
        b.adamw(wb, mb, vb, hp, begin=lo, count=hi - lo)
    b.root(1)
    a.sync(); b.sync()
    U.assert_same_f32(wb, wa.cpu().numpy(), "w")
    ow, _, _, _ = oracle_masked(U.oracle_grads(grads), w0, np.zeros(n, np.float32),
                                np.zeros(n, np.float32), 1, segs, False)
    U.assert_same_f32(wa, ow, "w vs oracle")
    # mask cleared: the plain step
    c = rs.Repstep(n, device=DEV)
    c.set_decay_mask(mask)
    c.set_decay_mask(None)
    wc, mc, vc = I.gen_state(U.F32_WL, n=n, device=DEV)
    c.step(grads, wc, mc, vc, hp, step=1)
    c.sync()
    ref = U.oracle_step(U.oracle_grads(grads), w0, np.zeros(n, np.float32),
                        np.zeros(n, np.float32), 1)
    U.assert_same_f32(wc, ref["w"], "w without mask")
