"""Software flush-to-zero mode ("OPEN-1B: A Fully Auditable Training Run", §2.1
"Subnormals": FTZ zeroes subnormal results, DAZ subnormal inputs) on the GPU against the
oracle's FTZ functions, bit for bit.  The inputs plant subnormals where every kind of
operation meets them: subnormal gradients (DAZ), gradients whose replica sums and
averages fall below the normal range (FTZ of sums and products), squares below it (the
norm), and subnormal w, m, v (DAZ in AdamW).  Each test also checks that the IEEE oracle
differs on the same inputs, so the flush is really exercised."""
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


def plant_grads(grads):
    """Bands of each replica scaled into and near the subnormal range."""
    out = []
    for r, g in enumerate(grads):
        x = g.float().clone()
        n = x.numel()
        x[n // 8: n // 4] *= 2.0 ** -128            # replica values and sums subnormal
        x[n // 4: 3 * n // 8] *= 2.0 ** -118        # sums normal, averages/products near
        x[n // 2: 5 * n // 8] *= 2.0 ** -62         # squares below the normal range
        x[r::331] = 2.0 ** -140                     # isolated subnormal inputs
        out.append(x.to(g.dtype).contiguous())
    return out


def plant_state(w, m, v):
    n = w.numel()
    w[n // 3::97] = 3.0 * 2.0 ** -140
    m[::53] = -(2.0 ** -130)
    v[::61] = 2.0 ** -135
    m[n // 2: n // 2 + 4096] *= 2.0 ** -125
    return w, m, v


def oracle_ftz_step(gnp, w, m, v, t, segs=None, dp_shard=None, accum=None):
    if dp_shard is None:
        g = O.reduce_ftz(gnp)
    else:
        g = O.reduce_alg1_ftz(gnp, dp_shard, accum or 0)
    nv = O.norm_ftz(g)
    sc = O.clip_scale_ftz(nv, U.HP["clip"])
    bc1, bc2 = O.bias_corrections_ftz(U.HP["beta1"], U.HP["beta2"], t)
    w, m, v = O.adamw_ftz(w, m, v, g, sc, U.HP["lr"], U.HP["beta1"], U.HP["beta2"], U.HP["eps"],
                          U.HP["wd"], bc1, bc2, segments=segs)
    wide = O.widen_bf16(w) if w.dtype == np.uint16 else w
    return dict(g=g, norm=nv, w=w, m=m, v=v, root=O.state_hash(t, wide, m, v))


@pytest.mark.parametrize("n,R,gdt,bf16w", [
    (5, 2, torch.float32, False), (4097, 4, torch.float32, False),
    (3 * 4096 + 1234, 8, torch.bfloat16, False), (50_001, 3, torch.float32, True),
    (123_457, 12, torch.float32, False), (40_000, 33, torch.bfloat16, True),
])
def test_ftz_steps_match_oracle(n, R, gdt, bf16w):
    pdt = torch.bfloat16 if bf16w else torch.float32
    ctx = rs.Repstep(n, grad_dtype=gdt, device=DEV, param_dtype=pdt,
                     subnormals=rs.SUBNORMALS_FTZ)
    w, m, v = plant_state(*I.gen_state(U.F32_WL, n=n, device=DEV))
    w = w.to(pdt)
    ow = U.bits16(w) if bf16w else w.cpu().numpy()
    om, ov = m.cpu().numpy(), v.cpu().numpy()
    norm = torch.empty(1, dtype=torch.float32, device=DEV)
    root = torch.empty(1, dtype=torch.int64, device=DEV)
    differs = False
    for t in (1, 2):
        grads = plant_grads(U.gen_grads(n, R, t, gdt))
        gnp = U.oracle_grads(grads)
        ctx.step(grads, w, m, v, U.hp_for(t), step=t, norm_out=norm, root_out=root)
        ctx.sync()
        ref = oracle_ftz_step(gnp, ow, om, ov, t)
        U.assert_same_f32(ctx.g_view(), ref["g"], f"g step {t}")
        U.assert_same_f32(norm, np.array([ref["norm"]], np.float32), f"norm step {t}")
        if bf16w:
            U.assert_same_bf16(w, ref["w"], f"w step {t}")
        else:
            U.assert_same_f32(w, ref["w"], f"w step {t}")
        U.assert_same_f32(m, ref["m"], f"m step {t}")
        U.assert_same_f32(v, ref["v"], f"v step {t}")
        assert U.root_of(root) == ref["root"], f"root step {t}"
        differs |= not np.array_equal(O.reduce(gnp).view(np.uint32), ref["g"].view(np.uint32))
        ow, om, ov = ref["w"], ref["m"], ref["v"]
    assert differs or n < 64                   # the planted subnormals met a flush


def test_ftz_paper_reduce_with_accumulation_and_ranges():
    n, N, dps, acc = 50_000, 6, 3, 2
    grads = plant_grads(U.gen_grads(n, N * acc, 1))
    gnp = U.oracle_grads(grads)
    a = rs.Repstep(n, device=DEV, subnormals=rs.SUBNORMALS_FTZ)
    b = rs.Repstep(n, device=DEV, subnormals=rs.SUBNORMALS_FTZ)
    a.reduce_paper(grads, dps, accum=acc)
    for lo, hi in [(0, 3), (3, 4100), (4100, 33_333), (33_333, n)]:
        b.reduce_paper(grads, dps, begin=lo, count=hi - lo, accum=acc)
    na, nb = (torch.empty(1, dtype=torch.float32, device=DEV) for _ in range(2))
    a.clip(1.0, norm_out=na)
    b.clip(1.0, norm_out=nb)
    a.sync(); b.sync()
    g = O.reduce_alg1_ftz(gnp, dps, acc)
    U.assert_same_f32(a.g_view(), g, "g")
    U.assert_same_f32(b.g_view(), g, "g in ranges")
    _, chunks = O.norm_ftz(g, with_chunks=True)
    U.assert_same_f32(a.chunk_sums_view(), chunks, "chunk sums")
    U.assert_same_f32(b.chunk_sums_view(), chunks, "chunk sums in ranges")
    assert na.item() == nb.item() == O.norm_ftz(g)
    assert not np.array_equal(O.reduce_alg1_accum(gnp, dps, acc), g)


def test_ftz_with_decay_segments_and_shards():
    n, R = 60_001, 4
    segs = [(0, False), (777, True), (4096 * 3 + 5, False), (20_000, True)]
    grads = plant_grads(U.gen_grads(n, R, 1, scale=2000.0))
    gnp = U.oracle_grads(grads)
    ctx = rs.Repstep(n, device=DEV, subnormals=rs.SUBNORMALS_FTZ)
    ctx.set_decay_mask(rs.decay_mask_from_segments(n, segs).to(DEV))
    w, m, v = plant_state(*I.gen_state(U.F32_WL, n=n, device=DEV))
    ow, om, ov = w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
    hp = U.hp_for(1)
    r = torch.empty(1, dtype=torch.int64, device=DEV)
    ctx.reduce(grads)
    ctx.clip(hp.clip)
    for lo, hi in I.shard_ranges(n, 7):
        ctx.adamw(w, m, v, hp, begin=lo, count=hi - lo)
    ctx.root(1, root_out=r)
    ctx.sync()
    ref = oracle_ftz_step(gnp, ow, om, ov, 1, segs=segs)
    U.assert_same_f32(w, ref["w"], "w")
    U.assert_same_f32(m, ref["m"], "m")
    U.assert_same_f32(v, ref["v"], "v")
    assert U.root_of(r) == ref["root"]


def test_ieee_mode_keeps_subnormals_on_the_same_inputs():
    """The default mode on the planted inputs equals the IEEE oracle (gradual underflow)."""
    n, R = 20_000, 4
    grads = plant_grads(U.gen_grads(n, R, 1))
    gnp = U.oracle_grads(grads)
    ctx = rs.Repstep(n, device=DEV)
    w, m, v = plant_state(*I.gen_state(U.F32_WL, n=n, device=DEV))
    ow, om, ov = w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
    root = torch.empty(1, dtype=torch.int64, device=DEV)
    ctx.step(grads, w, m, v, U.hp_for(1), step=1, root_out=root)
    ctx.sync()
    ref = U.oracle_step(gnp, ow, om, ov, 1)
    U.assert_same_f32(ctx.g_view(), O.reduce(gnp), "g")
    U.assert_same_f32(w, ref["w"], "w")
    U.assert_same_f32(m, ref["m"], "m")
    assert U.root_of(root) == ref["root"]
    g = ctx.g_view().cpu().numpy()
    assert ((g != 0) & (np.abs(g) < np.finfo(np.float32).tiny)).any()   # subnormals survive


@pytest.mark.parametrize("bf16w", [False, True])
def test_ftz_audit_mode(bf16w):
    """FTZ arithmetic with BLAKE2b-64 audit leaves (the AdamW-only kernel variant)."""
    n, R = 3 * 4096 + 77, 4
    pdt = torch.bfloat16 if bf16w else torch.float32
    ctx = rs.Repstep(n, device=DEV, param_dtype=pdt, subnormals=rs.SUBNORMALS_FTZ,
                     hash_mode=rs.HASH_BLAKE2B)
    w, m, v = plant_state(*I.gen_state(U.F32_WL, n=n, device=DEV))
    w = w.to(pdt)
    ow = U.bits16(w) if bf16w else w.cpu().numpy()
    om, ov = m.cpu().numpy(), v.cpu().numpy()
    root = torch.empty(1, dtype=torch.int64, device=DEV)
    grads = plant_grads(U.gen_grads(n, R, 1))
    ctx.step(grads, w, m, v, U.hp_for(1), step=1, root_out=root)
    ctx.sync()
    ref = oracle_ftz_step(U.oracle_grads(grads), ow, om, ov, 1)
    wide = O.widen_bf16(ref["w"]) if bf16w else ref["w"]
    assert U.root_of(root) == O.state_hash(1, wide, ref["m"], ref["v"], hash_mode=1)
    U.assert_same_f32(m, ref["m"], "m")


@pytest.mark.parametrize("nt,grid", [(128, 0), (256, 0), (512, 7), (256, 333)])
def test_ftz_launch_shape_invariance(nt, grid):
    """The FTZ instantiations for every block size give the default shape's bits."""
    n, R = 70_001, 8
    grads = plant_grads(U.gen_grads(n, R, 2))
    out = []
    for kw in ({}, dict(block_threads=nt, grid_blocks=grid)):
        ctx = rs.Repstep(n, device=DEV, subnormals=rs.SUBNORMALS_FTZ, **kw)
        w, m, v = plant_state(*I.gen_state(U.F32_WL, n=n, device=DEV))
        root = torch.empty(1, dtype=torch.int64, device=DEV)
        ctx.step(grads, w, m, v, U.hp_for(2), step=2, root_out=root)
        ctx.sync()
        out.append((w, m, v, U.root_of(root), ctx.g_view().clone()))
    a, b = out
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert a[3] == b[3]
    assert torch.equal(a[4].view(torch.int32), b[4].view(torch.int32))


def _band_case(n, hp_kw, plant):
    """One AdamW step with zero gradients on planted moments and weights, on the GPU in
    the flush-to-zero mode, against the oracle; returns the GPU's (w, m, v)."""
    ctx = rs.Repstep(n, device=DEV, subnormals=rs.SUBNORMALS_FTZ)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)
    plant(w, m, v)
    w0, m0, v0 = w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
    grads = [torch.zeros(n, device=DEV) for _ in range(2)]
    hp = rs.hparams(t=1, **hp_kw)
    ctx.reduce(grads)
    ctx.clip(hp.clip)
    ctx.adamw(w, m, v, hp)
    ctx.sync()
    g0 = np.zeros(n, np.float32)
    bc1, bc2 = O.bias_corrections_ftz(hp_kw["beta1"], hp_kw["beta2"], 1)
    ref = O.adamw_ftz(w0, m0, v0, g0, 1.0, hp_kw["lr"], hp_kw["beta1"], hp_kw["beta2"],
                      hp_kw["eps"], hp_kw["weight_decay"], bc1, bc2)
    for got, want, nm in zip((w, m, v), ref, "wmv"):
        U.assert_same_f32(got, want, nm)
    return w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()


def test_ftz_products_at_the_tininess_boundary():
    """b1*m exactly +-(2^-126 - 2^-150) is tiny (zeroed) although its binary32 rounding
    is 2^-126; b2*v exactly 2^-126 (1 - 2^-46) rounds to 2^-126 with an unbounded
    exponent and is kept."""
    n = 4096 + 5
    tiny = 2.0 ** -126

    def plant(w, m, v):
        m[0::7] = tiny
        m[3::7] = -tiny
        v[1::5] = (1 + 2.0 ** -23) * tiny

    _, m1, v1 = _band_case(n, dict(lr=3e-4, beta1=1 - 2.0 ** -24, beta2=1 - 2.0 ** -23,
                                   eps=1e-8, weight_decay=0.1, clip=1.0), plant)
    # both signs end as +0: the zeroed product is added to (1 - b1) * gc = +0
    assert not m1[0::7].view(np.uint32).any()
    assert not m1[3::7].view(np.uint32).any()
    assert np.all(v1[1::5] == np.float32(tiny))


def test_ftz_quotient_at_the_tininess_boundary():
    """u = mh / (sqrt(vh) + eps) exactly 2^-126 - 2^-150 is zeroed, so w' = w; flushing
    the binary32 quotient instead (2^-126) would give w - 2^-126."""
    n = 4096 + 5

    def plant(w, m, v):
        m[2::9] = (1 - 2.0 ** -24) * 2.0 ** -99    # m' = m/2, mh = m'/(1/2) = m
        v[2::9] = 0.0
        w[2::9] = 2.0 ** -124

    w1, _, _ = _band_case(n, dict(lr=1.0, beta1=0.5, beta2=0.5, eps=2.0 ** 27,
                                  weight_decay=0.0, clip=1.0), plant)
    assert np.all(w1[2::9] == np.float32(2.0 ** -124))
    with np.errstate(under="ignore"):
        ieee_u = np.float32(np.float32((1 - 2.0 ** -24) * 2.0 ** -99) / np.float32(2.0 ** 27))
    assert ieee_u == np.float32(2.0 ** -126)              # the binary32 quotient
