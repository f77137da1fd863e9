"""GPU parity: the CUDA path through the C ABI against the CPU oracle, bit for bit (0 ulp),
on the same seeded inputs.  Sizes span several tiles and chunks with ragged tails."""
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


def run_steps(n, R, dtype=torch.float32, steps=3, scales=(1.0, 3000.0, 1.0), ctx_kw=None,
              nodes=1, check_intermediates=True, hash_mode=0):
    """Run `steps` fused steps on the GPU and in the oracle; assert every output bit."""
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, grad_dtype=dtype, device=dev, hash_mode=hash_mode, **(ctx_kw or {}))
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    ow, om, ov = w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    out = []
    for t in range(1, steps + 1):
        grads = U.gen_grads(n, R, t, dtype, scale=scales[(t - 1) % len(scales)])
        gnp = U.oracle_grads(grads)
        ctx.step(grads, w, m, v, U.hp_for(t), step=t, norm_out=norm, root_out=root, nodes=nodes)
        flags = ctx.sync()
        ref = U.oracle_step(gnp, ow, om, ov, t, nodes=nodes, hash_mode=hash_mode)
        ow, om, ov = ref["w"], ref["m"], ref["v"]
        if check_intermediates and n > 0:
            U.assert_same_f32(ctx.g_view(), O.reduce(gnp), f"g step {t}")
            _, chunks = O.norm(O.reduce(gnp), with_chunks=True)
            U.assert_same_f32(ctx.chunk_sums_view(), chunks, f"chunk sums step {t}")
            leaves = ctx.leaves_view().cpu().numpy().view(np.uint64)
            assert np.array_equal(leaves, O.leaves(t, ow, om, ov, hash_mode)), f"leaves step {t}"
        U.assert_same_f32(w, ow, f"w step {t}")
        U.assert_same_f32(m, om, f"m step {t}")
        U.assert_same_f32(v, ov, f"v step {t}")
        U.assert_same_f32(norm, np.array([ref["norm"]], np.float32), f"norm step {t}")
        assert U.root_of(root) == ref["root"], f"root step {t}"
        assert bool(flags & rs.FLAG_NONFINITE_NORM) == (not np.isfinite(ref["norm"]))
        out.append(dict(norm=float(ref["norm"]), root=ref["root"]))
    ctx.destroy()
    return out


@pytest.mark.parametrize("n,R,dtype", [
    (1, 1, torch.float32),
    (5, 3, torch.float32),
    (4095, 4, torch.float32),
    (4096, 8, torch.float32),
    (4097, 5, torch.float32),
    (3 * 4096 + 1234, 8, torch.bfloat16),
    (65536 + 7, 9, torch.float32),
    (100003, 16, torch.float32),
    (50001, 32, torch.float32),
    (200002, 2, torch.bfloat16),
    (123457, 12, torch.bfloat16),
    (40000, 33, torch.float32),
])
def test_step_matches_oracle(n, R, dtype):
    res = run_steps(n, R, dtype)
    if n >= 4096:
        assert any(r["norm"] > 1.0 for r in res)  # the clip was exercised


@pytest.mark.parametrize("n,R,dtype", [
    (1, 2, torch.float32),
    (33, 3, torch.float32),
    (4096, 8, torch.float32),
    (3 * 4096 + 1234, 8, torch.bfloat16),
    (100003, 16, torch.float32),
])
def test_audit_mode_step_matches_oracle(n, R, dtype):
    """Audit mode: BLAKE2b-64 leaves over the image bytes (short final blocks included)."""
    run_steps(n, R, dtype, hash_mode=rs.HASH_BLAKE2B)


def test_audit_mode_shards_and_standalone_hash():
    n = 8 * 37_501 + 5
    dev = torch.device("cuda", 0)
    a = rs.Repstep(n, device=dev, hash_mode=rs.HASH_BLAKE2B)
    b = rs.Repstep(n, device=dev, hash_mode=rs.HASH_BLAKE2B)
    wa, ma, va = I.gen_state(U.F32_WL, n=n, device=dev)
    wb, mb, vb = wa.clone(), ma.clone(), va.clone()
    r = torch.empty(3, dtype=torch.int64, device=dev)
    grads = U.gen_grads(n, 8, 1, scale=3000.0)
    hp = U.hp_for(1)
    a.step(grads, wa, ma, va, hp, step=1, root_out=r[0:1])
    for lo, hi in I.shard_ranges(n, 8):
        b.reduce(grads, begin=lo, count=hi - lo)
    b.clip(hp.clip)
    for lo, hi in I.shard_ranges(n, 8):
        b.adamw(wb, mb, vb, hp, begin=lo, count=hi - lo)
    b.root(1, root_out=r[1:2])
    b.hash(1, wb, mb, vb, root_out=r[2:3])
    a.sync(); b.sync()
    rr = r.cpu().numpy().view(np.uint64)
    want = O.state_hash(1, wa.cpu().numpy(), ma.cpu().numpy(), va.cpu().numpy(), hash_mode=1)
    assert rr[0] == rr[1] == rr[2] == want
    U.assert_same_f32(wb, wa.cpu().numpy(), "w")


@pytest.mark.parametrize("R,dp_shard,dtype", [
    (1, 1, torch.float32), (6, 2, torch.float32), (6, 3, torch.float32), (7, 1, torch.float32),
    (12, 4, torch.float32), (9, 9, torch.float32), (40, 8, torch.float32), (24, 3, torch.bfloat16),
    (8, 1, torch.float32),
])
def test_paper_exact_reduce_matches_oracle(R, dp_shard, dtype):
    """OPEN-1B Algorithm 1 order: g bit-identical to the oracle's restatement, then the
    rest of the step (norm, clip, AdamW, root) on that g."""
    n = 2 * 4096 + 333
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, grad_dtype=dtype, device=dev)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    ow, om, ov = w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    for t in (1, 2):
        grads = U.gen_grads(n, R, t, dtype, scale=3000.0 if t == 2 else 1.0)
        hp = U.hp_for(t)
        ctx.reduce_paper(grads, dp_shard)
        ctx.clip(hp.clip, norm_out=norm)
        ctx.adamw(w, m, v, hp)
        ctx.root(t, root_out=root)
        ctx.sync()
        g = O.reduce_alg1(U.oracle_grads(grads), dp_shard)
        U.assert_same_f32(ctx.g_view(), g, f"g step {t}")
        nv = O.norm(g)
        bc1, bc2 = O.bias_corrections(U.HP["beta1"], U.HP["beta2"], t)
        ow, om, ov = O.adamw(ow, om, ov, g, O.clip_scale(nv, U.HP["clip"]), U.HP["lr"],
                             U.HP["beta1"], U.HP["beta2"], U.HP["eps"], U.HP["wd"], bc1, bc2)
        assert np.float32(norm.item()) == nv
        U.assert_same_f32(w, ow, f"w step {t}")
        U.assert_same_f32(v, ov, f"v step {t}")
        assert U.root_of(root) == O.state_hash(t, ow, om, ov)
    if dp_shard == 1 and R & (R - 1) == 0:
        # one shard, power-of-two replicas: the canonical tree exactly
        b = rs.Repstep(n, grad_dtype=dtype, device=dev)
        b.reduce(grads)
        b.clip(1.0)
        b.sync()
        assert torch.equal(b.g_view().view(torch.int32), ctx.g_view().view(torch.int32))


@pytest.mark.parametrize("N,dp_shard,accum,dtype", [
    (1, 1, 1, torch.float32), (1, 1, 3, torch.float32), (6, 2, 2, torch.float32),
    (3, 3, 5, torch.float32), (12, 4, 4, torch.bfloat16), (7, 1, 6, torch.float32),
    (8, 2, 32, torch.float32), (64, 8, 4, torch.float32),
])
def test_paper_exact_reduce_with_accumulation(N, dp_shard, accum, dtype):
    """Algorithm 1 with its microbatch loop: N * accum microbatch gradients, rank-major;
    g and the chunk sums bit-identical to the oracle.  Signed zeros are planted so the
    +0 start of every rank's accumulation is exercised."""
    n = 2 * 4096 + 333
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, grad_dtype=dtype, device=dev)
    grads = U.gen_grads(n, N * accum, 1, dtype)
    for k, x in enumerate(grads):
        x[k % 97::97] = -0.0
    ctx.reduce_paper(grads, dp_shard, accum=accum)
    ctx.clip(1.0)
    ctx.sync()
    g = O.reduce_alg1_accum(U.oracle_grads(grads), dp_shard, accum)
    U.assert_same_f32(ctx.g_view(), g, "g")
    _, chunks = O.norm(g, with_chunks=True)
    U.assert_same_f32(ctx.chunk_sums_view(), chunks, "chunk sums")
    with pytest.raises(ValueError):
        ctx.reduce_paper(grads[:-1], dp_shard, accum=accum) if accum > 1 else \
            ctx.reduce_paper(grads, dp_shard, accum=0)


def test_paper_exact_reduce_in_ranges():
    n, R, dps = 50_000, 12, 4
    dev = torch.device("cuda", 0)
    a, b = rs.Repstep(n, device=dev), rs.Repstep(n, device=dev)
    grads = U.gen_grads(n, R, 3)
    a.reduce_paper(grads, dps)
    for lo, hi in [(0, 3), (3, 4100), (4100, 33_333), (33_333, n)]:
        b.reduce_paper(grads, dps, begin=lo, count=hi - lo)
    na, nb = (torch.empty(1, dtype=torch.float32, device=dev) for _ in range(2))
    a.clip(1.0, norm_out=na)
    b.clip(1.0, norm_out=nb)
    a.sync(); b.sync()
    assert torch.equal(a.g_view().view(torch.int32), b.g_view().view(torch.int32))
    assert na.item() == nb.item()
    with pytest.raises(rs.RepstepError) as ei:
        a.reduce_paper(grads, 5)            # 5 does not divide 12
    assert ei.value.code == 4


def test_empty_parameter_vector():
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(0, device=dev)
    z = torch.zeros(1, dtype=torch.float32, device=dev)
    grads = [torch.zeros(1, dtype=torch.float32, device=dev)] * 2
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    ctx.step(grads, z, z.clone(), z.clone(), U.hp_for(1), step=1, norm_out=norm, root_out=root)
    ctx.sync()
    e = np.zeros(0, np.float32)
    assert float(norm.item()) == 0.0
    assert U.root_of(root) == O.state_hash(1, e, e, e)
    ctx_a = rs.Repstep(0, device=dev, hash_mode=rs.HASH_BLAKE2B)
    ctx_a.step(grads, z, z.clone(), z.clone(), U.hp_for(1), step=1, norm_out=norm, root_out=root)
    ctx_a.sync()
    assert U.root_of(root) == O.state_hash(1, e, e, e, hash_mode=1)


@pytest.mark.parametrize("kw", [dict(param_dtype=torch.bfloat16), dict(subnormals=rs.SUBNORMALS_FTZ),
                                dict(hash_mode=rs.HASH_BLAKE2B, param_dtype=torch.bfloat16,
                                     subnormals=rs.SUBNORMALS_FTZ)])
def test_empty_parameter_vector_every_mode(kw):
    """n = 0 in the bf16-parameter, FTZ and audit modes, with a decay mask and the hash on
    a second stream: the root of the empty state, nothing launched over elements."""
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(0, device=dev, **kw)
    ctx.set_decay_mask(rs.decay_mask_from_segments(0, []).to(dev))
    ctx.set_hash_stream(torch.cuda.Stream(dev))
    pdt = kw.get("param_dtype", torch.float32)
    w = torch.zeros(1, dtype=pdt, device=dev)
    z = torch.zeros(1, dtype=torch.float32, device=dev)
    grads = [torch.zeros(1, dtype=torch.float32, device=dev)] * 3
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    ctx.step(grads, w, z.clone(), z.clone(), U.hp_for(1), step=1, norm_out=norm, root_out=root)
    ctx.sync()
    e = np.zeros(0, np.float32)
    assert float(norm.item()) == 0.0
    assert U.root_of(root) == O.state_hash(1, e, e, e, hash_mode=kw.get("hash_mode", 0))
    ctx.reduce_paper(grads, 1, accum=3)
    ctx.clip(1.0)
    ctx.sync()


@pytest.mark.parametrize("nt", [128, 256, 512])
def test_launch_shape_invariance(nt):
    n, R = 7 * 4096 * 5 + 333, 8
    c = (n + 4095) // 4096
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    base = None
    for grid in [1, 7, sm, 2 * sm + 1, c]:
        res = run_steps(n, R, steps=2, ctx_kw=dict(grid_blocks=grid, block_threads=nt),
                        check_intermediates=(grid == 7))
        if base is None:
            base = res
        assert res == base


def test_topologies_equal_flat_and_oracle():
    n, R = 20000, 32
    flat = run_steps(n, R, steps=2, check_intermediates=False)
    for nodes in [4, 8, 32, 2, 16]:
        assert run_steps(n, R, steps=2, nodes=nodes, check_intermediates=False) == flat


def test_topology_rejected():
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(1000, device=dev)
    grads = U.gen_grads(1000, 6, 1)
    with pytest.raises(rs.RepstepError) as ei:
        ctx.reduce(grads, nodes=2, gpus_per_node=3)
    assert ei.value.code == 4
    with pytest.raises(rs.RepstepError) as ei:
        ctx.reduce(grads, nodes=4, gpus_per_node=2)      # 4 x 2 != 6
    assert ei.value.code == 4


def _shard_run(n, R, ranges, dtype=torch.float32, steps=2):
    """Sharded reduce/AdamW calls vs one fused step: identical bits, and equal to the oracle."""
    dev = torch.device("cuda", 0)
    a = rs.Repstep(n, grad_dtype=dtype, device=dev)
    b = rs.Repstep(n, grad_dtype=dtype, device=dev)
    wa, ma, va = I.gen_state(U.F32_WL, n=n, device=dev)
    wb, mb, vb = wa.clone(), ma.clone(), va.clone()
    ow, om, ov = wa.cpu().numpy(), ma.cpu().numpy(), va.cpu().numpy()
    na = torch.empty(1, dtype=torch.float32, device=dev)
    nb = torch.empty(1, dtype=torch.float32, device=dev)
    ra = torch.empty(1, dtype=torch.int64, device=dev)
    rb = torch.empty(1, dtype=torch.int64, device=dev)
    for t in range(1, steps + 1):
        grads = U.gen_grads(n, R, t, dtype, scale=3000.0 if t == 1 else 1.0)
        hp = U.hp_for(t)
        a.step(grads, wa, ma, va, hp, step=t, norm_out=na, root_out=ra)
        for lo, hi in ranges:
            b.reduce(grads, begin=lo, count=hi - lo)
        b.clip(hp.clip, norm_out=nb)
        for lo, hi in reversed(ranges):
            b.adamw(wb, mb, vb, hp, begin=lo, count=hi - lo)
        b.root(t, root_out=rb)
        a.sync(); b.sync()
        ref = U.oracle_step(U.oracle_grads(grads), ow, om, ov, t)
        ow, om, ov = ref["w"], ref["m"], ref["v"]
        for x, y, name in [(wa, wb, "w"), (ma, mb, "m"), (va, vb, "v")]:
            U.assert_same_f32(y, x.cpu().numpy(), f"sharded {name}")
        U.assert_same_f32(wa, ow, "w vs oracle")
        assert float(na.item()) == float(nb.item()) == float(ref["norm"])
        assert U.root_of(ra) == U.root_of(rb) == ref["root"]


def test_shard_ranges_equal_unsharded():
    n = 8 * 37_501 + 5            # boundaries fall mid-chunk, not on 16-byte multiples
    _shard_run(n, 8, I.shard_ranges(n, 8))
    # ragged ranges, several inside one chunk
    _shard_run(50_000, 4, [(0, 3), (3, 4100), (4100, 4101), (4101, 12_289), (12_289, 50_000)])


def test_shard_ranges_bf16():
    n = 3 * 4096 * 8 + 17
    _shard_run(n, 8, I.shard_ranges(n, 8), dtype=torch.bfloat16)


def test_fused_equals_separate_calls_and_standalone_hash():
    n, R = 4096 * 9 + 100, 8
    dev = torch.device("cuda", 0)
    a = rs.Repstep(n, device=dev)
    b = rs.Repstep(n, device=dev)
    wa, ma, va = I.gen_state(U.F32_WL, n=n, device=dev)
    wb, mb, vb = wa.clone(), ma.clone(), va.clone()
    r = torch.empty(4, dtype=torch.int64, device=dev)
    nrm = torch.empty(2, dtype=torch.float32, device=dev)
    # hash of the initial state (step 0) equals the oracle's
    a.hash(0, wa, ma, va, root_out=r[3:])
    a.sync()
    assert U.root_of(r[3:]) == O.state_hash(0, wa.cpu().numpy(), ma.cpu().numpy(), va.cpu().numpy())
    for t in (1, 2):
        grads = U.gen_grads(n, R, t, scale=2000.0)
        hp = U.hp_for(t)
        a.step(grads, wa, ma, va, hp, step=t, norm_out=nrm[0:1], root_out=r[0:1])
        b.reduce(grads)
        b.clip(hp.clip, norm_out=nrm[1:2])
        b.adamw(wb, mb, vb, hp)
        b.root(t, root_out=r[1:2])
        b.hash(t, wb, mb, vb, root_out=r[2:3])
        a.sync(); b.sync()
        U.assert_same_f32(wb, wa.cpu().numpy(), "w")
        assert nrm[0].item() == nrm[1].item()
        rr = r.cpu().numpy().view(np.uint64)
        assert rr[0] == rr[1] == rr[2]


def test_call_order_is_enforced():
    n = 5000
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, device=dev)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    grads = U.gen_grads(n, 2, 1)
    with pytest.raises(rs.RepstepError) as ei:
        ctx.adamw(w, m, v, U.hp_for(1))           # no clip yet
    assert ei.value.code == 7
    ctx.reduce(grads, begin=0, count=1000)
    with pytest.raises(rs.RepstepError) as ei:
        ctx.clip(1.0)                             # only part of the range reduced
    assert ei.value.code == 7
    ctx.reduce(grads, begin=1000, count=n - 1000)
    ctx.clip(1.0)
    ctx.adamw(w, m, v, U.hp_for(1), begin=0, count=10)
    with pytest.raises(rs.RepstepError) as ei:
        ctx.root(1)                               # AdamW covered 10 of n elements
    assert ei.value.code == 7
    with pytest.raises(rs.RepstepError) as ei:
        ctx.reduce(grads, begin=n - 5, count=10)  # out of range
    assert ei.value.code == 1
    ctx.sync()


def test_misaligned_pointers_rejected():
    n = 1000
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, device=dev)
    buf = torch.zeros(n + 8, dtype=torch.float32, device=dev)
    grads = [buf[1:n + 1]]                        # 4-byte offset
    with pytest.raises(rs.RepstepError) as ei:
        ctx.reduce(grads)
    assert ei.value.code == 2


def test_image_round_trip_and_guards():
    n = 3 * 4096 + 77
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, device=dev)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    m.normal_(); v.uniform_()
    img_d = torch.empty(rs.image_bytes(n), dtype=torch.uint8, device=dev)
    img_h = torch.empty(rs.image_bytes(n), dtype=torch.uint8).pin_memory()
    ctx.image_write(7, w, m, v, img_d)
    ctx.image_write(7, w, m, v, img_h)
    ctx.sync()
    want = O.image(7, w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy())
    assert img_d.cpu().numpy().tobytes() == want
    assert img_h.numpy().tobytes() == want
    w2, m2, v2 = torch.empty_like(w), torch.empty_like(m), torch.empty_like(v)
    assert ctx.image_read(img_d, w2, m2, v2) == 7
    ctx.sync()
    assert torch.equal(w2.view(torch.int32), w.view(torch.int32))
    assert torch.equal(v2.view(torch.int32), v.view(torch.int32))
    # the image hash equals the state hash of its contents
    r = torch.empty(1, dtype=torch.int64, device=dev)
    ctx.hash(7, w2, m2, v2, root_out=r)
    ctx.sync()
    assert U.root_of(r) == O.state_hash(7, w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy())
    # a check that cannot fail is not a check: truncated, oversized, wrong header
    with pytest.raises(rs.RepstepError) as ei:
        ctx.image_read(img_h[:-4096], w2, m2, v2)
    assert ei.value.code == 8
    big = torch.zeros(rs.image_bytes(n) + 4, dtype=torch.uint8)
    with pytest.raises(rs.RepstepError):
        ctx.image_read(big, w2, m2, v2)
    bad = img_h.clone()
    bad[4] ^= 1                                   # header n off by one
    with pytest.raises(rs.RepstepError) as ei:
        ctx.image_read(bad, w2, m2, v2)
    assert ei.value.code == 8


def test_nonfinite_gradient_sets_flag():
    n = 9000
    dev = torch.device("cuda", 0)
    grads = U.gen_grads(n, 4, 1)
    grads[2][4321] = float("nan")
    ctx = rs.Repstep(n, device=dev)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    ow, om, ov = w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    ctx.step(grads, w, m, v, U.hp_for(1), step=1, norm_out=norm)
    flags = ctx.sync()
    assert flags & rs.FLAG_NONFINITE_NORM
    assert np.isnan(norm.item())
    ref = U.oracle_step(U.oracle_grads(grads), ow, om, ov, 1)
    U.assert_same_f32(w, ref["w"], "w with a NaN gradient")   # NaN slots compared by class


@pytest.mark.parametrize("t,bc_override", [(1, None), (2, None), (7, None), (3, (0.3, 1e-13)),
                                           (4, (-0.5, 3.0))])
def test_adamw_on_arbitrary_bit_patterns(t, bc_override):
    """w, m, v and g drawn as random 32-bit patterns (zeros, subnormals, huge values,
    infinities and NaNs included): every result bit equals the oracle (NaNs by class).
    Covers the fixed-divisor fast path's fallbacks and divisors outside its range."""
    n = 3 * 4096 + 11
    dev = torch.device("cuda", 0)
    rng = np.random.default_rng(100 + t)
    bits = lambda: rng.integers(0, 2 ** 32, n, dtype=np.uint64).astype(np.uint32).view(np.float32)  # noqa: E731
    w, m, g = bits(), bits(), bits()
    v = (rng.integers(0, 2 ** 31, n, dtype=np.uint64).astype(np.uint32)).view(np.float32)
    # plus plain values so most elements take the common path
    w[::3] = rng.standard_normal(len(w[::3])).astype(np.float32) * 0.02
    m[::3] = rng.standard_normal(len(m[::3])).astype(np.float32) * 1e-4
    v[::3] = np.abs(rng.standard_normal(len(v[::3]))).astype(np.float32) * 1e-8
    g[::3] = rng.standard_normal(len(g[::3])).astype(np.float32) * 1e-3
    # signed zeros where the sign of a zero quotient reaches w': w = m = g = -0, v = +0
    # gives u = -0 and w' = -0 - lr*(-0) = +0 (a quotient of +0 would leave -0)
    for a in (w, m, g):
        a[7::101] = -0.0
    v[7::101] = 0.0
    m[9::101] = -0.0                                     # -0 moments beside normal values
    hp = U.hp_for(t, clip=float("inf"))
    if bc_override:
        hp.bc1, hp.bc2 = bc_override
    ctx = rs.Repstep(n, device=dev)
    W, M, V, G = (torch.from_numpy(a.copy()).to(dev) for a in (w, m, v, g))
    ctx.reduce([G])
    ctx.clip(float("inf"))
    ctx.adamw(W, M, V, hp)
    ctx.sync()
    ow, om, ov = O.adamw(w, m, v, g, 1.0, U.HP["lr"], U.HP["beta1"], U.HP["beta2"], U.HP["eps"],
                         U.HP["wd"], np.float32(hp.bc1), np.float32(hp.bc2))
    U.assert_same_f32(W, ow, "w")
    U.assert_same_f32(M, om, "m")
    U.assert_same_f32(V, ov, "v")


def test_relaunch_is_deterministic():
    n, R = 77_777, 8
    a = run_steps(n, R, steps=2, check_intermediates=False)
    b = run_steps(n, R, steps=2, check_intermediates=False)
    assert a == b


def test_workload_flat1m_r4_full():
    wl = I.WORKLOADS["flat1m_r4"]
    res = run_steps(wl.n, wl.R, steps=wl.steps, scales=(1.0,))
    assert all(r["norm"] < 1.0 for r in res)       # N(0, 1e-3) grads over 1M params: no clip


def test_workload_flat12m8_student_t_full():
    """12.8M parameters, 8 Student-t(3) replicas, 10 steps; the 8 + 12n checkpoint image and
    its Merkle root every step, all bit-identical to the oracle."""
    wl = I.WORKLOADS["flat12m8_r8_student_t"]
    n, R = wl.n, wl.R
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, device=dev)
    w, m, v = I.gen_state(wl, device=dev)
    ow, om, ov = w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    img = torch.empty(rs.image_bytes(n), dtype=torch.uint8, device=dev)
    clipped = 0
    for t in range(1, wl.steps + 1):
        grads = [I.gen_grad(wl, t, r, device=dev) for r in range(R)]
        ctx.step(grads, w, m, v, U.hp_for(t), step=t, norm_out=norm, root_out=root)
        ctx.image_write(t, w, m, v, img)
        ctx.sync()
        ref = U.oracle_step(U.oracle_grads(grads), ow, om, ov, t)
        ow, om, ov = ref["w"], ref["m"], ref["v"]
        U.assert_same_f32(w, ow, f"w step {t}")
        U.assert_same_f32(m, om, f"m step {t}")
        U.assert_same_f32(v, ov, f"v step {t}")
        assert float(norm.item()) == float(ref["norm"])
        assert U.root_of(root) == ref["root"]
        assert img.cpu().numpy().tobytes() == O.image(t, ow, om, ov)
        clipped += ref["norm"] > 1.0
    assert img.numel() == 153_600_008


@pytest.mark.parametrize("hash_stream", [False, True])
def test_steps_beside_a_busy_stream(hash_stream):
    """The fp32 reduce and AdamW hand out chunks at run time, so which CTA sums which chunk
    depends on when each CTA starts.  Steps run while another stream keeps the SMs busy
    with matrix products; every output bit must still equal the oracle's."""
    n, R = 4_000_000 + 123, 8
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, device=dev)
    side = torch.cuda.Stream(dev)
    ctx.set_hash_stream(torch.cuda.Stream(dev) if hash_stream else None)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    ow, om, ov = w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
    a = torch.randn(4096, 4096, device=dev)
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    for t in (1, 2):
        grads = U.gen_grads(n, R, t)
        gnp = U.oracle_grads(grads)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(side):
            b = a
            for _ in range(6):
                b = b @ a
        ctx.step(grads, w, m, v, U.hp_for(t), step=t, norm_out=norm, root_out=root)
        ctx.sync()
        side.synchronize()
        ref = U.oracle_step(gnp, ow, om, ov, t)
        ow, om, ov = ref["w"], ref["m"], ref["v"]
        U.assert_same_f32(w, ow, f"w step {t}")
        U.assert_same_f32(m, om, f"m step {t}")
        U.assert_same_f32(v, ov, f"v step {t}")
        U.assert_same_f32(norm, np.array([ref["norm"]], np.float32), f"norm step {t}")
        assert U.root_of(root) == ref["root"], f"root step {t}"
    del b


def test_context_memory_is_recorded_on_every_stream_it_uses():
    """The workspace and the decay mask are marked as used on the creation stream, on each
    stream a call ran on, and on the hash stream, so that PyTorch's allocator does not hand
    them to a new tensor while a root is still pending there.  The step's bits do not
    depend on the stream."""
    n, R = 3 * 4096 + 17, 4
    dev = torch.device("cuda", 0)
    main = torch.cuda.current_stream(dev)
    side, hs = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ctx = rs.Repstep(n, device=dev)
    assert set(ctx._streams_used) == {main.cuda_stream}
    mask = rs.decay_mask_from_segments(n, [(0, False), (5000, True)]).to(dev)
    ctx.set_decay_mask(mask)
    ctx.set_hash_stream(hs)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    grads = U.gen_grads(n, R, 1)
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    side.wait_stream(main)
    with torch.cuda.stream(side):
        ctx.step(grads, w, m, v, U.hp_for(1), step=1, norm_out=norm, root_out=root)
        ctx.sync()
    assert set(ctx._streams_used) == {main.cuda_stream, side.cuda_stream, hs.cuda_stream}
    w2, m2, v2 = I.gen_state(U.F32_WL, n=n, device=dev)
    twin = rs.Repstep(n, device=dev)
    twin.set_decay_mask(mask)
    root2 = torch.empty(1, dtype=torch.int64, device=dev)
    twin.step(grads, w2, m2, v2, U.hp_for(1), step=1, root_out=root2)
    twin.sync()
    assert U.root_of(root) == U.root_of(root2)
    del ctx                           # its root is complete; freeing waits on all streams
    torch.cuda.synchronize(dev)
