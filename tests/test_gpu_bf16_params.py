"""bf16 parameters ("OPEN-1B: A Fully Auditable Training Run", §3.2 paragraph on
optimizer-state precision): w held in bf16, widened exactly, updated in fp32 against fp32
moments, rounded back to bf16 once to nearest even; the image and the state hash carry w
widened to fp32.  The CUDA path through the C ABI against the oracle, bit for bit."""
import os

import numpy as np
import pytest
import torch

from bitwise_reproducible_step_gb300 import inputs as I
from bitwise_reproducible_step_gb300 import repstep as rs
from oracle import oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    U.ensure_built()
    torch.cuda.set_device(0)


DEV = torch.device("cuda", 0)


def bf16_state(n):
    w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)
    return w.to(torch.bfloat16), m, v


def widened(w16: torch.Tensor) -> np.ndarray:
    return O.widen_bf16(U.bits16(w16))


@pytest.mark.parametrize("n,R,gdtype,hash_mode", [
    (1, 1, torch.float32, 0),
    (7, 3, torch.bfloat16, 0),
    (4095, 4, torch.float32, 0),
    (4096, 8, torch.bfloat16, 0),
    (4097, 5, torch.float32, 1),
    (3 * 4096 + 1234, 8, torch.bfloat16, 0),
    (100003, 16, torch.float32, 0),
    (123457, 12, torch.bfloat16, 1),
    (262144 + 9, 8, torch.bfloat16, 0),
])
def test_bf16_param_steps_match_oracle(n, R, gdtype, hash_mode):
    ctx = rs.Repstep(n, grad_dtype=gdtype, device=DEV, hash_mode=hash_mode,
                     param_dtype=torch.bfloat16)
    w, m, v = bf16_state(n)
    ow, om, ov = U.bits16(w), m.cpu().numpy(), v.cpu().numpy()
    norm = torch.empty(1, dtype=torch.float32, device=DEV)
    root = torch.empty(1, dtype=torch.int64, device=DEV)
    for t, scale in zip((1, 2, 3), (1.0, 3000.0, 1.0)):
        grads = U.gen_grads(n, R, t, gdtype, scale=scale)
        ctx.step(grads, w, m, v, U.hp_for(t), step=t, norm_out=norm, root_out=root)
        ctx.sync()
        ref = U.oracle_step_bf16w(U.oracle_grads(grads), ow, om, ov, t, hash_mode=hash_mode)
        ow, om, ov = ref["w16"], ref["m"], ref["v"]
        U.assert_same_bf16(w, ow, f"w step {t}")
        U.assert_same_f32(m, om, f"m step {t}")
        U.assert_same_f32(v, ov, f"v step {t}")
        U.assert_same_f32(norm, np.array([ref["norm"]], np.float32), f"norm step {t}")
        leaves = ctx.leaves_view().cpu().numpy().view(np.uint64)
        assert np.array_equal(leaves, ref["leaves"]), f"leaves step {t}"
        assert U.root_of(root) == ref["root"], f"root step {t}"
    # the parameters really moved, and stayed bf16 values
    assert not np.array_equal(ow, U.bits16(bf16_state(n)[0]))
    ctx.destroy()


def test_bf16_param_shard_ranges_equal_unsharded():
    """AdamW in ranges whose boundaries are not multiples of 8 elements (the bf16 bulk-copy
    granule), several inside one chunk: the same bits and root as one call."""
    n, R = 50_000, 4
    grads = U.gen_grads(n, R, 1, scale=2000.0)
    a = rs.Repstep(n, device=DEV, param_dtype=torch.bfloat16)
    b = rs.Repstep(n, device=DEV, param_dtype=torch.bfloat16)
    wa, ma, va = bf16_state(n)
    wb, mb, vb = wa.clone(), ma.clone(), va.clone()
    r = torch.empty(2, dtype=torch.int64, device=DEV)
    hp = U.hp_for(1)
    a.step(grads, wa, ma, va, hp, step=1, root_out=r[0:1])
    b.reduce(grads)
    b.clip(hp.clip)
    for lo, hi in [(0, 3), (3, 4100), (4100, 4101), (4101, 12_289), (12_289, 12_290),
                   (12_290, 33_333), (33_333, 50_000)]:
        b.adamw(wb, mb, vb, hp, begin=lo, count=hi - lo)
    b.root(1, root_out=r[1:2])
    a.sync(); b.sync()
    U.assert_same_bf16(wb, U.bits16(wa), "w")
    U.assert_same_f32(mb, ma.cpu().numpy(), "m")
    rr = r.cpu().numpy().view(np.uint64)
    assert rr[0] == rr[1]
    ref = U.oracle_step_bf16w(U.oracle_grads(grads), U.bits16(bf16_state(n)[0]),
                              np.zeros(n, np.float32), np.zeros(n, np.float32), 1)
    assert int(rr[0]) == ref["root"]


@pytest.mark.parametrize("t", [1, 4])
def test_bf16_param_adamw_on_arbitrary_bit_patterns(t):
    """bf16 w as random 16-bit patterns (zeros, subnormals, infinities, NaNs), m, v, g as
    random 32-bit patterns: every result bit equals the oracle (NaNs by class)."""
    n = 2 * 4096 + 13
    rng = np.random.default_rng(700 + t)
    w16 = rng.integers(0, 2 ** 16, n, dtype=np.uint64).astype(np.uint16)
    bits = lambda: rng.integers(0, 2 ** 32, n, dtype=np.uint64).astype(np.uint32).view(np.float32)  # noqa: E731
    m, g = bits(), bits()
    v = rng.integers(0, 2 ** 31, n, dtype=np.uint64).astype(np.uint32).view(np.float32)
    plain = slice(None, None, 3)
    w16[plain] = U.bits16(torch.from_numpy(rng.standard_normal(len(w16[plain])).astype(np.float32)
                                           * 0.02).to(torch.bfloat16))
    m[plain] = rng.standard_normal(len(m[plain])).astype(np.float32) * 1e-4
    v[plain] = np.abs(rng.standard_normal(len(v[plain]))).astype(np.float32) * 1e-8
    g[plain] = rng.standard_normal(len(g[plain])).astype(np.float32) * 1e-3
    for a in (m, g):
        a[7::101] = -0.0
    w16[7::101] = 0x8000                                 # bf16 -0
    v[7::101] = 0.0
    hp = U.hp_for(t, clip=float("inf"))
    ctx = rs.Repstep(n, device=DEV, param_dtype=torch.bfloat16)
    W = torch.from_numpy(w16.view(np.int16).copy()).view(torch.bfloat16).to(DEV)
    M, V, G = (torch.from_numpy(a.copy()).to(DEV) for a in (m, v, g))
    ctx.reduce([G])
    ctx.clip(float("inf"))
    ctx.adamw(W, M, V, hp)
    ctx.sync()
    ow, om, ov = O.adamw_bf16w(w16, m, v, g, 1.0, U.HP["lr"], U.HP["beta1"], U.HP["beta2"],
                               U.HP["eps"], U.HP["wd"], np.float32(hp.bc1), np.float32(hp.bc2))
    U.assert_same_bf16(W, ow, "w")
    U.assert_same_f32(M, om, "m")
    U.assert_same_f32(V, ov, "v")


def test_bf16_param_standalone_hash_and_image(tmp_path):
    n = 3 * 4096 + 77
    ctx = rs.Repstep(n, device=DEV, param_dtype=torch.bfloat16)
    w, m, v = bf16_state(n)
    m.normal_(); v.uniform_()
    wide, mn, vn = widened(w), m.cpu().numpy(), v.cpu().numpy()
    r = torch.empty(1, dtype=torch.int64, device=DEV)
    ctx.hash(5, w, m, v, root_out=r)
    ctx.sync()
    assert U.root_of(r) == O.state_hash(5, wide, mn, vn)
    want = O.image(5, wide, mn, vn)
    img_d = torch.empty(rs.image_bytes(n), dtype=torch.uint8, device=DEV)
    img_h = torch.empty(rs.image_bytes(n), dtype=torch.uint8).pin_memory()
    ctx.image_write(5, w, m, v, img_d)
    ctx.image_write(5, w, m, v, img_h)
    ctx.sync()
    assert img_d.cpu().numpy().tobytes() == want
    assert img_h.numpy().tobytes() == want
    for src in (img_d, img_h):
        w2 = torch.zeros_like(w)
        m2, v2 = torch.empty_like(m), torch.empty_like(v)
        assert ctx.image_read(src, w2, m2, v2) == 5
        ctx.sync()
        U.assert_same_bf16(w2, U.bits16(w), "w read back")
        assert torch.equal(v2.view(torch.int32), v.view(torch.int32))
    # an image whose w holds a value that is not a bf16 exactly is rejected before any copy
    for src in (img_d.clone(), img_h.clone()):
        src[8 + 4 * 1000] ^= 1                   # low byte of w[1000]
        w3 = torch.zeros_like(w)
        m3 = torch.full_like(m, 7.0)
        with pytest.raises(rs.RepstepError) as ei:
            ctx.image_read(src, w3, m3, v)
        assert ei.value.code == 8
        assert torch.all(w3 == 0) and torch.all(m3 == 7.0)
    # checkpoint file: widened image bytes; load narrows; a non-bf16 word is rejected
    path = str(tmp_path / rs.checkpoint_name(5))
    ctx.save_checkpoint(path, 5, w, m, v)
    data = open(path, "rb").read()
    assert data == want and not os.path.exists(path + ".tmp")
    w4 = torch.zeros_like(w)
    m4, v4 = torch.empty_like(m), torch.empty_like(v)
    assert ctx.load_checkpoint(path, w4, m4, v4) == 5
    U.assert_same_bf16(w4, U.bits16(w), "w loaded")
    assert torch.equal(m4.view(torch.int32), m.view(torch.int32))
    bad = bytearray(data)
    bad[8 + 4 * (n - 1)] ^= 0x80                 # last w word
    open(path, "wb").write(bytes(bad))
    w5 = torch.zeros_like(w)
    m5 = torch.full_like(m, 7.0)
    with pytest.raises(rs.RepstepError) as ei:
        ctx.load_checkpoint(path, w5, m5, v4)
    assert ei.value.code == 8
    assert torch.all(w5 == 0) and torch.all(m5 == 7.0)


def test_bf16_param_dtype_mismatch_rejected_on_host():
    n = 4096
    ctx = rs.Repstep(n, device=DEV, param_dtype=torch.bfloat16)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)       # fp32 w: the binding refuses it
    with pytest.raises(ValueError):
        ctx.hash(0, w, m, v)
