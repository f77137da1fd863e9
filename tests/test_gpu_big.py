"""Full-size workloads on one GB300, in the launch configuration the benchmark times, with
every slot of every step compared with the oracle.

The oracle runs chunk-parallel on the host cores (tests/oracle_full.py; its functions are
unchanged and single-threaded per call) and follows its own trajectory from the same
initial state and the same gradients.  After each GPU step every slot of g, the chunk sums
of squares, w, m, v and the leaf digests is compared, and the pre-clip norm and the Merkle
root -- formed from the oracle's own chunk sums and leaves -- must be equal: 0 differing
slots and relFro 0, the statistics of "Cross-process reproducibility, settled by
measurement" (section "The measurement").  Each step's norm and root are also checked
against the fingerprints tests/golden/make_full_size_fingerprints.py wrote from the oracle
alone.  Invariances (launch shape, topology, shard ranges) are checked on the full arrays
by exact equality on the device.

Set REPSTEP_FULL_ORACLE_LOG to a file name to append one JSON line per compared step.
"""
import json
import os

import numpy as np
import pytest
import torch

from bitwise_reproducible_step_gb300 import inputs as I
from bitwise_reproducible_step_gb300 import repstep as rs
from tests import gpu_util as U
from tests import oracle_full as OF

pytestmark = [pytest.mark.gpu, pytest.mark.big]

CH = 4096
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "full_size_fingerprints.txt")


@pytest.fixture(scope="module", autouse=True)
def _built():
    U.ensure_built()
    torch.cuda.set_device(0)
    yield
    torch.cuda.empty_cache()


def fingerprints():
    """(workload, variant, step) -> (norm bits, root) from the committed golden file."""
    out = {}
    if not os.path.exists(GOLDEN):
        return out
    for line in open(GOLDEN):
        if not line.strip() or line.startswith("#"):
            continue
        wl, variant, t, norm, root = [x.strip() for x in line.split("|")]
        out[(wl, variant, int(t))] = (norm, root)
    return out


def record(rep, what):
    path = os.environ.get("REPSTEP_FULL_ORACLE_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(dict(what=what, **rep)) + "\n")


def check(rep, wl_name, variant, t):
    what = f"{wl_name}/{variant} step {t}"
    record(rep, what)
    OF.assert_identical(rep, what)
    fp = fingerprints().get((wl_name, variant, t))
    if fp is not None:
        assert (rep["norm"]["oracle"], rep["root"]["oracle"]) == fp, (what, fp)


def host_state(w, m, v):
    if w.dtype == torch.bfloat16:
        w_h = w.view(torch.int16).cpu().numpy().view(np.uint16)
    else:
        w_h = w.cpu().numpy()
    return w_h, m.cpu().numpy(), v.cpu().numpy()


def gpu_views(ctx, w, m, v, norm, root):
    return dict(g=ctx.g_view(), chunk_sums=ctx.chunk_sums_view(), leaves=ctx.leaves_view(),
                w=w, m=m, v=v, norm=norm, root=root)


def run_big(wl, steps, variant="default", ranges=None, compare_unsharded=False, hash_mode=0,
            single_pass=False):
    """single_pass: the benchmark's launch configuration -- repstep_step_fused with the two
    state buffers alternating and the root passes on a second stream; the single pass
    keeps g out of HBM, so g is not compared (the chunk sums, the state and every leaf
    are)."""
    n, R = wl.n, wl.R
    dev = torch.device("cuda", 0)
    gdt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
    ctx = rs.Repstep(n, grad_dtype=gdt, device=dev, hash_mode=hash_mode)
    w, m, v = I.gen_state(wl, device=dev)
    other = None
    if single_pass:
        ctx.set_hash_stream(torch.cuda.Stream(dev))
        other = tuple(torch.empty_like(x) for x in (w, m, v))
    fo = OF.FullOracle(n, R, *host_state(w, m, v), grad_dtype=wl.grad_dtype,
                       hash_mode=hash_mode)
    twin = None
    if compare_unsharded:
        twin = (rs.Repstep(n, grad_dtype=gdt, device=dev), w.clone(), m.clone(), v.clone())
    grads = [torch.empty(n, dtype=gdt, device=dev) for _ in range(R)]
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    reps = []
    for t in range(1, steps + 1):
        for r in range(R):
            I.gen_grad(wl, t, r, device=dev, out=grads[r])
        hp = U.hp_for(t)
        if ranges:
            for lo, hi in ranges:
                ctx.reduce(grads, begin=lo, count=hi - lo)
            ctx.clip(hp.clip, norm_out=norm)
            for lo, hi in ranges:
                ctx.adamw(w, m, v, hp, begin=lo, count=hi - lo)
            ctx.root(t, root_out=root)
        elif single_pass:
            ctx.step_fused(grads, w, m, v, *other, hp, step=t, norm_out=norm, root_out=root)
            (w, m, v), other = other, (w, m, v)
        else:
            ctx.step(grads, w, m, v, hp, step=t, norm_out=norm, root_out=root)
        assert ctx.sync() & ~rs.FLAG_NONFINITE_NORM == 0
        views = gpu_views(ctx, w, m, v, norm, root)
        if single_pass:
            del views["g"]
        rep = fo.step(grads, t, U.HP, views)
        check(rep, wl.name, variant, t)
        reps.append(rep)
        if twin is not None:
            tc, tw, tm, tv = twin
            tn = torch.empty(1, dtype=torch.float32, device=dev)
            tr = torch.empty(1, dtype=torch.int64, device=dev)
            tc.step(grads, tw, tm, tv, hp, step=t, norm_out=tn, root_out=tr)
            tc.sync()
            assert torch.equal(tw.view(torch.int32), w.view(torch.int32))
            assert torch.equal(tm.view(torch.int32), m.view(torch.int32))
            assert torch.equal(tv.view(torch.int32), v.view(torch.int32))
            assert tn.item() == norm.item() and U.root_of(tr) == U.root_of(root)
    fo.close()
    return [float(np.uint32(int(r["norm"]["oracle"], 16)).view(np.float32)) for r in reps]


def test_flat1200m_r8_segscale():
    """The benchmark workload: 1.2e9 parameters, R = 8, all 5 steps."""
    wl = I.WORKLOADS["flat1200m_r8_segscale"]
    norms = run_big(wl, steps=wl.steps)
    assert all(x < 1.0 for x in norms)              # tiny segment-scaled grads: no clip


def test_flat1200m_r8_segscale_single_pass():
    """The benchmark workload in the benchmark's launch configuration (the single-pass
    step, state buffers alternating, roots on a second stream), all 5 steps: every slot
    against the oracle, and the same fingerprints as the two-pass run."""
    wl = I.WORKLOADS["flat1200m_r8_segscale"]
    run_big(wl, steps=wl.steps, single_pass=True)


def test_flat1200m_r8_segscale_audit_mode():
    """The benchmark workload with BLAKE2b-64 audit-mode leaves, two steps."""
    wl = I.WORKLOADS["flat1200m_r8_segscale"]
    run_big(wl, steps=2, variant="audit", hash_mode=rs.HASH_BLAKE2B)


def test_flat3000m_r8_bf16_spiked_shards():
    """3e9 parameters, R = 8 bf16 gradients, all 3 steps reduced and updated as 8 contiguous
    shard ranges; equal to the unsharded run on the device and to the oracle everywhere."""
    wl = I.WORKLOADS["flat3000m_r8_bf16_spiked_shards"]
    norms = run_big(wl, steps=wl.steps, ranges=I.shard_ranges(wl.n, wl.shards),
                    compare_unsharded=True)
    assert all(x > 1.0 for x in norms)              # 1% spikes x 1e3 force the clip


def test_flat3000m_r8_bf16_single_pass():
    """3e9 parameters, R = 8 bf16 gradients, all 3 steps through the single-pass step
    (buffers alternating, roots on a second stream): step 1 speculates, clips and takes the
    second pass; steps 2 and 3 follow a clip and take the two passes at once.  Every slot
    against the oracle."""
    wl = I.WORKLOADS["flat3000m_r8_bf16_spiked_shards"]
    norms = run_big(wl, steps=wl.steps, single_pass=True)
    assert all(x > 1.0 for x in norms)


def test_flat268m_r32_three_steps_three_topologies():
    """268M parameters, R = 32: the workload's 3 steps, step t summed as the t-th staged
    topology (1 x 32, 4 x 8, 8 x 4 nodes x GPUs), against the oracle's staged sum."""
    wl = I.WORKLOADS["flat268m_r32_topologies"]
    n, R = wl.n, wl.R
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, device=dev)
    w, m, v = I.gen_state(wl, device=dev)
    fo = OF.FullOracle(n, R, *host_state(w, m, v))
    grads = [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(R)]
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    for t, (nodes, gpn) in zip(range(1, wl.steps + 1), wl.topologies):
        for r in range(R):
            I.gen_grad(wl, t, r, device=dev, out=grads[r])
        ctx.step(grads, w, m, v, U.hp_for(t), step=t, norm_out=norm, root_out=root,
                 nodes=nodes, gpus_per_node=gpn)
        assert ctx.sync() == 0
        rep = fo.step(grads, t, U.HP, gpu_views(ctx, w, m, v, norm, root), reducer="topology",
                      nodes=nodes, gpus_per_node=gpn)
        check(rep, wl.name, "topologies", t)
    fo.close()


def test_flat268m_r32_topologies_grids_blocks():
    """4 topologies x 5 grid sizes x 3 block sizes from a mid-run state: every output bit
    equal, and the default configuration equal to the oracle in every slot."""
    wl = I.WORKLOADS["flat268m_r32_topologies"]
    n, R = wl.n, wl.R
    dev = torch.device("cuda", 0)
    c = (n + CH - 1) // CH
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    grads = [I.gen_grad(wl, 1, r, device=dev) for r in range(R)]
    w0, m0, v0 = I.gen_state(wl, device=dev)
    m0.copy_(I.gen_grad(wl, 9, 0, device=dev))       # non-zero moments: a mid-run step
    v0.copy_(I.gen_grad(wl, 9, 1, device=dev).square())
    hp = U.hp_for(3)
    w, m, v = w0.clone(), m0.clone(), v0.clone()
    ref = None
    for nodes, gpn in wl.topologies:
        for grid in [0, 1, 7, sm, 2 * sm + 1, c]:
            for nt in ([128, 256, 512] if grid in (0, sm) else [256]):
                ctx = rs.Repstep(n, device=dev, grid_blocks=grid, block_threads=nt)
                w.copy_(w0); m.copy_(m0); v.copy_(v0)
                norm = torch.empty(1, dtype=torch.float32, device=dev)
                root = torch.empty(1, dtype=torch.int64, device=dev)
                ctx.step(grads, w, m, v, hp, step=3, norm_out=norm, root_out=root,
                         nodes=nodes, gpus_per_node=gpn)
                ctx.sync()
                if ref is None:
                    fo = OF.FullOracle(n, R, *host_state(w0, m0, v0))
                    rep = fo.step(grads, 3, U.HP, gpu_views(ctx, w, m, v, norm, root))
                    fo.close()
                    check(rep, wl.name, "mid_run_sweep_reference", 3)
                    ref = (w.clone(), m.clone(), v.clone(), norm.item(), U.root_of(root))
                else:
                    assert torch.equal(w.view(torch.int32), ref[0].view(torch.int32)), (nodes, grid, nt)
                    assert torch.equal(m.view(torch.int32), ref[1].view(torch.int32))
                    assert torch.equal(v.view(torch.int32), ref[2].view(torch.int32))
                    assert norm.item() == ref[3] and U.root_of(root) == ref[4]
                ctx.destroy()


def test_fixed_division_is_ieee_for_every_significand_pair():
    """The AdamW kernel divides by the step's bias corrections with Markstein's correction
    from a precomputed reciprocal; compare it with IEEE division for all 2^46 pairs."""
    assert rs.selftest_fixed_division(0, 1 << 23) == 0


def test_flat268m_r32_paper_exact_order():
    """OPEN-1B Algorithm 1 order on 268M parameters: 4 replicas x 8 shards (linear shard
    sums, TreeFold over replicas), every slot against the oracle's restatement."""
    wl = I.WORKLOADS["flat268m_r32_topologies"]
    n, R, dps = wl.n, wl.R, 8
    dev = torch.device("cuda", 0)
    grads = [I.gen_grad(wl, 1, r, device=dev) for r in range(R)]
    w, m, v = I.gen_state(wl, device=dev)
    fo = OF.FullOracle(n, R, *host_state(w, m, v))
    ctx = rs.Repstep(n, device=dev)
    hp = U.hp_for(1)
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    ctx.reduce_paper(grads, dps)
    ctx.clip(hp.clip, norm_out=norm)
    ctx.adamw(w, m, v, hp)
    ctx.root(1, root_out=root)
    ctx.sync()
    rep = fo.step(grads, 1, U.HP, gpu_views(ctx, w, m, v, norm, root), reducer="alg1",
                  dp_shard=dps)
    fo.close()
    check(rep, wl.name, "paper_exact_4x8", 1)


def bench_segments(n):
    """The decay segments of the benchmark's --decay-mask: no decay on a 5% embedding and
    on a 4096-element gain after every 16.7M-element block of matrices."""
    segs, e = [(0, False)], n // 20 | 1
    while e < n:
        segs.append((e, True))
        e += 16_777_216 + 3
        if e < n:
            segs.append((e, False))
            e += 4096
    return segs


def test_flat1200m_r8_bf16w_decay_mask_ftz():
    """The bench workload with all three optimizer variants at once -- bf16 parameters,
    the benchmark's decay segments and software flush-to-zero -- one mid-run step, every
    slot against the oracle's flush-to-zero functions."""
    wl = I.WORKLOADS["flat1200m_r8_segscale"]
    n, R = wl.n, wl.R
    dev = torch.device("cuda", 0)
    segs = bench_segments(n)
    ctx = rs.Repstep(n, device=dev, param_dtype=torch.bfloat16, subnormals=rs.SUBNORMALS_FTZ)
    ctx.set_decay_mask(rs.decay_mask_from_segments(n, segs).to(dev))
    w32, m, v = I.gen_state(wl, device=dev)
    w = w32.to(torch.bfloat16)
    del w32
    m.copy_(I.gen_grad(wl, 9, 0, device=dev))           # non-zero moments: a mid-run step
    v.copy_(I.gen_grad(wl, 9, 1, device=dev).square())
    fo = OF.FullOracle(n, R, *host_state(w, m, v), param_dtype="bf16", ftz=True,
                       segments=segs)
    grads = [I.gen_grad(wl, 3, r, device=dev) for r in range(R)]
    hp = U.hp_for(3)
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    ctx.step(grads, w, m, v, hp, step=3, norm_out=norm, root_out=root)
    assert ctx.sync() & ~rs.FLAG_NONFINITE_NORM == 0
    rep = fo.step(grads, 3, U.HP, gpu_views(ctx, w, m, v, norm, root))
    fo.close()
    check(rep, wl.name, "bf16w_decay_ftz_mid_run", 3)


@pytest.mark.parametrize("nt", [256, 512])
def test_repeated_steps_are_bit_identical(nt):
    """The same step, from the same state, 200 times: every output bit must repeat.  This
    caught a ring-refill race (a bulk copy overtaking a consumer's read of the previous
    tile) that hit about one run in 80 with 256-thread AdamW CTAs."""
    wl = I.WORKLOADS["flat268m_r32_topologies"]
    n, R = wl.n, wl.R
    dev = torch.device("cuda", 0)
    grads = [I.gen_grad(wl, 1, r, device=dev) for r in range(R)]
    w0, m0, v0 = I.gen_state(wl, device=dev)
    m0.copy_(I.gen_grad(wl, 9, 0, device=dev))
    v0.copy_(I.gen_grad(wl, 9, 1, device=dev).square())
    hp = U.hp_for(3)
    ctx = rs.Repstep(n, device=dev, block_threads=nt)
    w, m, v = w0.clone(), m0.clone(), v0.clone()
    root = torch.empty(1, dtype=torch.int64, device=dev)
    ref = None
    for _ in range(200):
        w.copy_(w0); m.copy_(m0); v.copy_(v0)
        ctx.step(grads, w, m, v, hp, step=3, root_out=root)
        assert ctx.sync() == 0
        if ref is None:
            ref = (w.clone(), m.clone(), v.clone(), U.root_of(root))
            continue
        assert U.root_of(root) == ref[3]
        assert torch.equal(w.view(torch.int32), ref[0].view(torch.int32))
    assert torch.equal(m.view(torch.int32), ref[1].view(torch.int32))
    assert torch.equal(v.view(torch.int32), ref[2].view(torch.int32))
